// merge_attn_states (vLLM Kimi-K3 MultiHeadLatentAttention page, the prefill
// path with chunked context): two attention results over disjoint key sets of
// the same query rows, each normalised by its own sum and carrying its
// log-sum-exp, combine into the result over the union of the keys.  A pure
// streaming op (two rows in, one row out per (token, head)): 16-byte loads and
// stores, fp32 arithmetic.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "kernel_args.h"
#include "ptx.cuh"
#include "xqa.h"
#include "xqa_internal.h"

namespace xqa {
namespace merge {

constexpr int kThreads = 256;

struct MergeArgs {
  uint16_t* out;
  const uint16_t* pre;
  const uint16_t* suf;
  float* out_lse;
  const float* pre_lse;
  const float* suf_lse;
  int64_t T, n_pre, chunks;  // chunks = T * H * (D / 8)
  int H, D;
  int64_t o_st, o_sh, p_st, p_sh, s_st, s_sh, l_st, l_sh;
};

// One thread per 8-element (16-byte) chunk of a row: the two log-sum-exps and
// both chunks are loaded together, so each thread keeps one round of DRAM
// latency in flight rather than two in a row.
template <bool kBf16>
__global__ void __launch_bounds__(kThreads) merge_kernel(const MergeArgs a) {
  const int64_t idx = int64_t(blockIdx.x) * kThreads + threadIdx.x;
  if (idx >= a.chunks) return;
  const int cpr = a.D >> 3;
  const int64_t row = idx / cpr;
  const int d = int(idx - row * cpr) << 3;
  const int64_t t = row / a.H;
  const int h = int(row - t * a.H);
  const int64_t li = t * a.l_st + h * a.l_sh;
  const bool has_pre = t < a.n_pre;
  const float ls = __ldg(a.suf_lse + li);
  const float lp = has_pre ? __ldg(a.pre_lse + li) : -INFINITY;
  const uint4 sv = __ldg(reinterpret_cast<const uint4*>(a.suf + t * a.s_st + h * a.s_sh + d));
  const uint4 pv = has_pre ? __ldg(reinterpret_cast<const uint4*>(a.pre + t * a.p_st + h * a.p_sh + d))
                           : make_uint4(0, 0, 0, 0);
  // weights of the two sides relative to the larger log-sum-exp; a side
  // with no visible key (-inf) weighs 0
  float wp = 0.f, ws = 1.f, M = ls;
  if (has_pre) {
    M = fmaxf(lp, ls);
    wp = M == -INFINITY ? 0.f : expf(lp - M);
    ws = M == -INFINITY ? 0.f : expf(ls - M);
  }
  const float z = wp + ws;
  const float fp = z == 0.f ? 0.f : wp / z;
  const float fs = z == 0.f ? 0.f : ws / z;
  uint32_t o4[4] = {sv.x, sv.y, sv.z, sv.w};  // bit-exact copy when the suffix stands alone
  if (fp != 0.f || fs != 1.f) {
    const uint32_t s4[4] = {sv.x, sv.y, sv.z, sv.w};
    const uint32_t p4[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 s2 = unpack_16x2(s4[k], kBf16);
      const float2 p2 = fp != 0.f ? unpack_16x2(p4[k], kBf16) : make_float2(0.f, 0.f);
      o4[k] = pack_f32x2(fs * s2.x + fp * p2.x, fs * s2.y + fp * p2.y, kBf16);
    }
  }
  *reinterpret_cast<uint4*>(a.out + t * a.o_st + h * a.o_sh + d) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
  if (a.out_lse && d == 0) a.out_lse[li] = z == 0.f ? -INFINITY : M + logf(z);
}

}  // namespace merge
}  // namespace xqa

namespace {

xqa_status merge_fail(xqa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  xqa::set_last_error(buf);
  return st;
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; }

}  // namespace

extern "C" xqa_status xqa_merge_attn_states(const xqa_merge_params* p, xqa_stream_t stream) {
  using namespace xqa::merge;
  if (!p) return merge_fail(XQA_ERR_INVALID_ARG, "params is NULL");
  if (p->dtype != XQA_F16 && p->dtype != XQA_BF16)
    return merge_fail(XQA_ERR_INVALID_ARG, "merge dtype must be fp16 or bf16");
  if (p->num_tokens < 0 || p->num_heads <= 0 || p->head_dim <= 0 || p->head_dim % 8)
    return merge_fail(XQA_ERR_INVALID_ARG, "need num_tokens >= 0, num_heads > 0, head_dim a positive multiple of 8");
  if (p->tokens_with_prefix < 0 || p->tokens_with_prefix > p->num_tokens)
    return merge_fail(XQA_ERR_INVALID_ARG, "tokens_with_prefix must lie in [0, num_tokens]");
  if (p->num_tokens == 0) return XQA_OK;
  const bool pre = p->tokens_with_prefix > 0;
  if (!p->output || !p->suffix_output || !p->suffix_lse || (pre && (!p->prefix_output || !p->prefix_lse)))
    return merge_fail(XQA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (misaligned(p->output) || misaligned(p->suffix_output) || (pre && misaligned(p->prefix_output)))
    return merge_fail(XQA_ERR_INVALID_ARG, "outputs must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(p->output_lse) | reinterpret_cast<uintptr_t>(p->suffix_lse) |
       reinterpret_cast<uintptr_t>(pre ? p->prefix_lse : nullptr)) & 3)
    return merge_fail(XQA_ERR_INVALID_ARG, "lse arrays must be 4-byte aligned");
  const int64_t st[6] = {p->out_stride_token,    p->out_stride_head,    p->suffix_stride_token,
                         p->suffix_stride_head,  p->prefix_stride_token, p->prefix_stride_head};
  for (int k = 0; k < (pre ? 6 : 4); ++k)
    if (st[k] < 0 || st[k] % 8)
      return merge_fail(XQA_ERR_INVALID_ARG, "output strides must be non-negative multiples of 8 elements");
  if (p->lse_stride_token < 0 || p->lse_stride_head < 0)
    return merge_fail(XQA_ERR_INVALID_ARG, "lse strides must be non-negative");
  MergeArgs a;
  a.out = static_cast<uint16_t*>(p->output);
  a.pre = static_cast<const uint16_t*>(pre ? p->prefix_output : p->suffix_output);
  a.suf = static_cast<const uint16_t*>(p->suffix_output);
  a.out_lse = p->output_lse;
  a.pre_lse = pre ? p->prefix_lse : p->suffix_lse;
  a.suf_lse = p->suffix_lse;
  a.T = p->num_tokens;
  a.n_pre = p->tokens_with_prefix;
  a.H = p->num_heads;
  a.D = p->head_dim;
  a.o_st = p->out_stride_token;
  a.o_sh = p->out_stride_head;
  a.p_st = pre ? p->prefix_stride_token : p->suffix_stride_token;
  a.p_sh = pre ? p->prefix_stride_head : p->suffix_stride_head;
  a.s_st = p->suffix_stride_token;
  a.s_sh = p->suffix_stride_head;
  a.l_st = p->lse_stride_token;
  a.l_sh = p->lse_stride_head;
  a.chunks = a.T * a.H * (a.D / 8);
  const int64_t blocks = (a.chunks + kThreads - 1) / kThreads;
  if (blocks > 0x7fffffffLL) return merge_fail(XQA_ERR_UNSUPPORTED, "too many rows for one launch");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (p->dtype == XQA_BF16)
    merge_kernel<true><<<unsigned(blocks), kThreads, 0, s>>>(a);
  else
    merge_kernel<false><<<unsigned(blocks), kThreads, 0, s>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return merge_fail(XQA_ERR_CUDA, "merge kernel launch: %s", cudaGetErrorString(e));
  return XQA_OK;
}
