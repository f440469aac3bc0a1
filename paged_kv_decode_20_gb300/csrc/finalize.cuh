// Final normalisation of one query row, shared by the decode kernels.
#pragma once
#include <cuda_fp8.h>
#include <math.h>

#include "ptx.cuh"

#include "kernel_args.h"

namespace xqa {

constexpr float kLn2 = 0.6931471805599453f;

// A row's running state in the exp2 domain: maximum M (log2 units) and sum l
// of 2^(x - M) over its visible logits x; sig is the sink in log2 units (or
// -inf).  Returns the factor that turns the un-normalised output into the
// final one, (e^sink added to the normaliser once; API page, `sinks`), times
// out_mul (kv_scale * rcp_out_scale; API page, `kv_scale`, `rcp_out_scale`).
// When lse_dst is not null, also stores the row's log-sum-exp in natural-log
// units (the `lse` forward_mqa returns, vLLM Kimi-K3 MultiHeadLatentAttention
// page): ln(sum_t e^s_t + e^sink), -inf for a row with no visible logit and no
// sink.
__device__ __forceinline__ float finalize_row(float M, float l, float sig, float out_mul, float* lse_dst) {
  const float Mf = fmaxf(M, sig);
  float mul = 0.f, lse = -INFINITY;
  if (Mf != -INFINITY) {
    const float fm = (M == -INFINITY) ? 0.f : exp2f(M - Mf);
    const float den = l * fm + ((sig == -INFINITY) ? 0.f : exp2f(sig - Mf));
    mul = fm * out_mul / den;
    lse = (Mf + log2f(den)) * kLn2;
  }
  if (lse_dst) *lse_dst = lse;
  return mul;
}

// Index of row r (= spec token i * G + group member g) of kv head kvh of
// sequence b in an [B, qs, Hq] array.
__device__ __forceinline__ int64_t lse_index(const DecodeArgs& a, int b, int kvh, int r) {
  const int i = r / a.G, g = r % a.G;
  return (int64_t(b) * a.qs + i) * a.Hq + int64_t(kvh) * a.G + g;
}

// Stores four consecutive output elements at element index oi: 16-bit (the
// query's dtype) or E4M3 (round to nearest even, finite values beyond 448
// saturated, as the output scale rcp_out_scale is meant to prevent).
__device__ __forceinline__ void store_out4(const DecodeArgs& a, int64_t oi, float4 v) {
  if (a.out_e4m3) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v.x, v.y), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v.z, v.w), __NV_SATFINITE, __NV_E4M3);
    *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(a.out) + oi) = lo | (hi << 16);
  } else {
    const bool bf = a.q_bf16 != 0;
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + oi) =
        make_uint2(pack_f32x2(v.x, v.y, bf), pack_f32x2(v.z, v.w, bf));
  }
}

}  // namespace xqa
