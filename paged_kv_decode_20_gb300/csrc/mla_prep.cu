// Fused MLA decode prep (vLLM Kimi-K3 MultiHeadLatentAttention page,
// `_decode_concat_cache`, the launch right before forward_mqa): the absorbed
// query [ql_nope | rope(q_pe)] and the insert of each decode token's latent
// row [kv_c_normed | rope(k_pe)] into the paged cache at slot_mapping.  RoPE is
// the GPT-J (non-neox) pairing of get_rope(..., is_neox_style=False), computed
// in fp32 from the fp32 cos/sin table (the page's fused epilogues read that
// table directly in fp32).  A streaming op: one thread per 8-element output
// chunk, 16-byte loads and stores.  The fp8 variant (a plain per-tensor fp8
// cache takes an fp8 query, same page) multiplies each fp32 value by the
// query's or the cache's inverse scale and rounds it to e4m3 (8-byte stores).
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <cuda_fp8.h>

#include "ptx.cuh"
#include "xqa.h"
#include "xqa_internal.h"

namespace xqa {
namespace prep {

constexpr int kThreads = 256;

struct PrepArgs {
  const uint16_t* ql;
  const uint16_t* qpe;
  const uint16_t* kvc;
  const uint16_t* kpe;
  const int64_t* pos;
  const float* cs;
  const int64_t* slots;
  void* cache;   // bf16 or (fp8) e4m3 rows of W elements
  void* qout;
  uint32_t* err;
  const float* q_inv;      // fp8: device scalars multiplying the query and the cache row
  const float* cache_inv;
  int64_t ql_st, ql_sh, qpe_st, qpe_sh, kvc_st, kpe_st, max_pos, num_slots, T;
  int H, Lr, R, W;          // W = Lr + R
  int64_t q_chunks, chunks;  // query chunks, then cache chunks
};

// Rotates 8 consecutive rope elements starting at pair index p0 (even
// elements 2i, odd 2i+1 rotate by angle i).
__device__ __forceinline__ uint4 rope8(uint4 x, const float* cs, int R, int p0, bool rotate) {
  if (!rotate) return x;
  uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 v = unpack_16x2(w[k], true);
    const float c = __ldg(cs + p0 + k), s = __ldg(cs + R / 2 + p0 + k);
    w[k] = pack_f32x2(v.x * c - v.y * s, v.y * c + v.x * s, true);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The same rotation in fp32, all eight values returned (the e4m3 variant
// scales them before it rounds).
__device__ __forceinline__ void rope8f(uint4 x, const float* cs, int R, int p0, bool rotate, float* out) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 v = unpack_16x2(w[k], true);
    if (rotate) {
      const float c = __ldg(cs + p0 + k), s = __ldg(cs + R / 2 + p0 + k);
      out[2 * k] = v.x * c - v.y * s;
      out[2 * k + 1] = v.y * c + v.x * s;
    } else {
      out[2 * k] = v.x;
      out[2 * k + 1] = v.y;
    }
  }
}

// Eight fp32 values times `mul`, rounded to nearest even into e4m3 and
// saturated at +-448, as one 8-byte word (element k in byte k).
__device__ __forceinline__ uint2 to_e4m3x8(const float* v, float mul) {
  uint32_t w[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint32_t lo =
        __nv_cvt_float2_to_fp8x2(make_float2(v[4 * k] * mul, v[4 * k + 1] * mul), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi =
        __nv_cvt_float2_to_fp8x2(make_float2(v[4 * k + 2] * mul, v[4 * k + 3] * mul), __NV_SATFINITE, __NV_E4M3);
    w[k] = (lo & 0xffffu) | (hi << 16);
  }
  return make_uint2(w[0], w[1]);
}

template <bool F8>
__global__ void __launch_bounds__(kThreads) prep_kernel(const PrepArgs a) {
  const int64_t idx = int64_t(blockIdx.x) * kThreads + threadIdx.x;
  if (idx >= a.chunks) return;
  const int cpr = a.W >> 3;  // chunks per output row
  const bool is_q = idx < a.q_chunks;
  const int64_t rel = is_q ? idx : idx - a.q_chunks;
  const int64_t row = rel / cpr;
  const int e = int(rel - row * cpr) << 3;  // element offset in the row
  const int64_t t = is_q ? row / a.H : row;
  const int h = is_q ? int(row - t * a.H) : 0;
  // the token's rotation angles
  bool rotate = false;
  const float* cs = nullptr;
  if (e >= a.Lr && a.pos) {
    const int64_t p = a.pos[t];
    if (p >= 0 && p < a.max_pos) {
      rotate = true;
      cs = a.cs + p * a.R;
    } else if (a.err && (is_q ? h == 0 : true)) {
      atomicOr(a.err, 1u);
    }
  }
  if constexpr (F8) {
    int64_t dst_row = row;
    uint8_t* dst_base = static_cast<uint8_t*>(a.qout);
    if (!is_q) {
      const int64_t slot = a.slots[t];
      if (slot < 0) return;  // padding token: nothing to insert
      if (slot >= a.num_slots) {
        if (a.err && e == 0) atomicOr(a.err, 1u);
        return;
      }
      dst_row = slot;
      dst_base = static_cast<uint8_t*>(a.cache);
    }
    const uint4 x = e < a.Lr ? __ldg(reinterpret_cast<const uint4*>(is_q ? a.ql + t * a.ql_st + h * a.ql_sh + e
                                                                         : a.kvc + t * a.kvc_st + e))
                             : __ldg(reinterpret_cast<const uint4*>(
                                   is_q ? a.qpe + t * a.qpe_st + h * a.qpe_sh + (e - a.Lr)
                                        : a.kpe + t * a.kpe_st + (e - a.Lr)));
    float v[8];
    rope8f(x, cs, a.R, (e - a.Lr) >> 1, e >= a.Lr && rotate, v);
    *reinterpret_cast<uint2*>(dst_base + dst_row * a.W + e) = to_e4m3x8(v, __ldg(is_q ? a.q_inv : a.cache_inv));
    return;
  }
  if (is_q) {
    uint4 v;
    if (e < a.Lr)
      v = __ldg(reinterpret_cast<const uint4*>(a.ql + t * a.ql_st + h * a.ql_sh + e));
    else
      v = rope8(__ldg(reinterpret_cast<const uint4*>(a.qpe + t * a.qpe_st + h * a.qpe_sh + (e - a.Lr))), cs,
                a.R, (e - a.Lr) >> 1, rotate);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.qout) + row * a.W + e) = v;
  } else {
    const int64_t slot = a.slots[t];
    if (slot < 0) return;  // padding token: nothing to insert
    if (slot >= a.num_slots) {
      if (a.err && e == 0) atomicOr(a.err, 1u);
      return;
    }
    uint4 v;
    if (e < a.Lr)
      v = __ldg(reinterpret_cast<const uint4*>(a.kvc + t * a.kvc_st + e));
    else
      v = rope8(__ldg(reinterpret_cast<const uint4*>(a.kpe + t * a.kpe_st + (e - a.Lr))), cs, a.R,
                (e - a.Lr) >> 1, rotate);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.cache) + slot * a.W + e) = v;
  }
}

}  // namespace prep
}  // namespace xqa

namespace {

xqa_status prep_fail(xqa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  xqa::set_last_error(buf);
  return st;
}

bool bad16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; }

}  // namespace

extern "C" xqa_status xqa_mla_decode_prep(const xqa_mla_prep_params* p, xqa_stream_t stream) {
  using namespace xqa::prep;
  if (!p) return prep_fail(XQA_ERR_INVALID_ARG, "params is NULL");
  if (p->num_tokens < 0 || p->num_heads <= 0) return prep_fail(XQA_ERR_INVALID_ARG, "need num_tokens >= 0 and num_heads > 0");
  if (p->kv_lora_rank <= 0 || p->kv_lora_rank % 8 || p->rope_dim <= 0 || p->rope_dim % 8)
    return prep_fail(XQA_ERR_INVALID_ARG, "kv_lora_rank and rope_dim must be positive multiples of 8");
  if (p->num_tokens == 0) return XQA_OK;
  if (!p->ql_nope || !p->q_pe || !p->kv_c || !p->k_pe || !p->slot_mapping || !p->kv_cache || !p->q_out)
    return prep_fail(XQA_ERR_INVALID_ARG, "a required pointer is NULL");
  if (p->positions && (!p->cos_sin_cache || p->max_position <= 0))
    return prep_fail(XQA_ERR_INVALID_ARG, "positions need cos_sin_cache and max_position > 0");
  if (bad16(p->ql_nope) || bad16(p->q_pe) || bad16(p->kv_c) || bad16(p->k_pe) || bad16(p->kv_cache) ||
      bad16(p->q_out))
    return prep_fail(XQA_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
  if (p->cos_sin_cache && (reinterpret_cast<uintptr_t>(p->cos_sin_cache) & 3))
    return prep_fail(XQA_ERR_INVALID_ARG, "cos_sin_cache must be 4-byte aligned");
  if ((reinterpret_cast<uintptr_t>(p->positions) | reinterpret_cast<uintptr_t>(p->slot_mapping)) & 7)
    return prep_fail(XQA_ERR_INVALID_ARG, "positions and slot_mapping must be 8-byte aligned");
  if (reinterpret_cast<uintptr_t>(p->error_word) & 3)
    return prep_fail(XQA_ERR_INVALID_ARG, "error_word must be 4-byte aligned");
  if (p->fp8 && (!p->q_scale_inv || !p->cache_scale_inv))
    return prep_fail(XQA_ERR_INVALID_ARG, "the fp8 prep needs q_scale_inv and cache_scale_inv (device scalars)");
  if ((reinterpret_cast<uintptr_t>(p->q_scale_inv) | reinterpret_cast<uintptr_t>(p->cache_scale_inv)) & 3)
    return prep_fail(XQA_ERR_INVALID_ARG, "q_scale_inv and cache_scale_inv must be 4-byte aligned");
  const int64_t st[6] = {p->ql_stride_token, p->ql_stride_head, p->qpe_stride_token, p->qpe_stride_head,
                         p->kvc_stride_token, p->kpe_stride_token};
  for (int k = 0; k < 6; ++k)
    if (st[k] < 0 || st[k] % 8)
      return prep_fail(XQA_ERR_INVALID_ARG, "strides must be non-negative multiples of 8 elements");
  PrepArgs a;
  a.ql = static_cast<const uint16_t*>(p->ql_nope);
  a.qpe = static_cast<const uint16_t*>(p->q_pe);
  a.kvc = static_cast<const uint16_t*>(p->kv_c);
  a.kpe = static_cast<const uint16_t*>(p->k_pe);
  a.pos = p->positions;
  a.cs = p->cos_sin_cache;
  a.slots = p->slot_mapping;
  a.cache = p->kv_cache;
  a.qout = p->q_out;
  a.err = p->error_word;
  a.q_inv = p->q_scale_inv;
  a.cache_inv = p->cache_scale_inv;
  a.ql_st = p->ql_stride_token;
  a.ql_sh = p->ql_stride_head;
  a.qpe_st = p->qpe_stride_token;
  a.qpe_sh = p->qpe_stride_head;
  a.kvc_st = p->kvc_stride_token;
  a.kpe_st = p->kpe_stride_token;
  a.max_pos = p->max_position;
  a.num_slots = p->num_slots;
  a.T = p->num_tokens;
  a.H = p->num_heads;
  a.Lr = p->kv_lora_rank;
  a.R = p->rope_dim;
  a.W = a.Lr + a.R;
  a.q_chunks = a.T * a.H * (a.W / 8);
  a.chunks = a.q_chunks + a.T * (a.W / 8);
  const int64_t blocks = (a.chunks + kThreads - 1) / kThreads;
  if (blocks > 0x7fffffffLL) return prep_fail(XQA_ERR_UNSUPPORTED, "too many tokens for one launch");
  if (p->fp8)
    prep_kernel<true><<<unsigned(blocks), kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  else
    prep_kernel<false><<<unsigned(blocks), kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return prep_fail(XQA_ERR_CUDA, "prep kernel launch: %s", cudaGetErrorString(e));
  return XQA_OK;
}
