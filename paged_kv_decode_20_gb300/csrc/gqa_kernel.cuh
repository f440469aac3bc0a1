// Grouped-query paged decode attention for sm_103a (the XQA-style call of the
// FlashInfer "flashinfer.xqa.xqa" API page).
//
// One CTA owns (sequence b, kv head kvh, row group rg, KV split).  Its rows are
// the q_seq_len x G query rows that share kv head kvh (speculative tokens and
// the GQA group stacked), padded to 16-row MMA blocks: RB blocks per consumer
// warp, and WR warp row groups (1, 2 or 4) that split the CTA's rows, so that
// up to 64 rows (D = 128) or 128 rows (D = 64) read each page of KV once.
//
//   warp 4 (producer, one lane): walks page_table and issues one TMA tile load
//     per (page, 128-byte column chunk) for K and for V into a ring of stages
//     (128 tokens when a row is one 128-byte chunk, else 64), each guarded by
//     a full/empty mbarrier pair.  NHD and HND differ only in the tensor map
//     and the coordinates.  TMA writes the rows with the 128-byte swizzle, so
//     ldmatrix reads are bank-conflict free.
//   warps 0-3 (consumers): warp w holds row group w % WR (RB 16-row blocks)
//     and takes the (w / WR)-th of 4 / WR equal token ranges of every stage
//     (WR = 1: a quarter of each stage, 16 or 32 tokens, i.e. two or four
//     independent 8-token MMA chains).
//     S = Q K^T with mma.sync m16n8k16 (rows on M, tokens on N), fp32 online
//     softmax in the exp2 domain with window / spec-mask / tail masking by
//     select, then O += P V (P re-used from the S accumulator registers).
//     fp8 K/V is widened to f16 in registers (cvt e4m3x2 -> f16x2, exact); a
//     consistent permutation of the contraction index lets each lane convert
//     whole 32-bit words, and a permutation of the V columns lets fp8 V be
//     read as words instead of transposed bytes.
//   epilogue: the four warps' (m, l, O) merge through shared memory.  With one
//     split the CTA finalises (sinks, scales) and writes the output; otherwise
//     it writes its partial to the workspace and takes a ticket on its
//     semaphore, and the last CTA to arrive merges every split (the same
//     log-sum-exp merge as merge_attn_states on the Kimi-K3 MLA page), writes
//     the output and resets the semaphore to zero.  No CTA ever waits on
//     another.
#pragma once
#include "finalize.cuh"
#include "kernel_args.h"
#include "ptx.cuh"

namespace xqa {

enum KvKind { kKvF16 = 0, kKvBf16 = 1, kKvE4m3 = 2 };

template <int KV, int D, int RB, int WR = 1>
struct GqaCfg {
  static constexpr bool kF8 = (KV == kKvE4m3);
  static constexpr int kElt = kF8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElt;  // 128 or 256
  static_assert(kRowBytes == 128 || kRowBytes == 256, "row must be 1 or 2 swizzle chunks");
  static constexpr int kChunks = kRowBytes / 128;
  // tokens per stage: 128 when a row is one 128-byte chunk and one 16-row
  // block suffices (four MMA chains per warp), else 64 (register budget)
  static constexpr int kTok = (kRowBytes == 128 && RB == 1 && WR == 1) ? 128 : 64;
  static constexpr int kTS = 4 / WR;  // warps sharing a row group (token splits)
  static_assert(WR == 1 || WR == 2 || WR == 4, "warp row groups");
  static constexpr int kTile = kTok * kRowBytes;           // K (or V) bytes per stage
  static constexpr int kStage = 2 * kTile;
  static constexpr int kNumStages = kStage >= 32768 ? 3 : 5;  // 96 KB or 80 KB per CTA
  static constexpr int kRows = 16 * RB * WR;
  static constexpr int kThreads = 160;
  // epilogue scratch: per token split O [kTS][rows][D], m and l [kTS][rows],
  // then per-row weights [rows][kTS] and the row's (max, sum) for a partial
  static constexpr int kScratch = kTS * kRows * D * 4 + 2 * kTS * kRows * 4 + (kTS + 2) * kRows * 4;
  static constexpr int kRing = kNumStages * kStage;
  static_assert(kScratch <= kRing, "epilogue scratch reuses the stage ring");
  static constexpr int kBarOff = kRing;
  static constexpr int kSmem = 1024 + kRing + 2 * kNumStages * 8 + 16;
};

__device__ __forceinline__ float load_scale(const float* dev, float host) {
  return dev ? __ldg(dev) : host;
}

template <int KV, int D, int RB, int WR>
__global__ void __launch_bounds__(160, 2)
    gqa_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const DecodeArgs a) {
  using C = GqaCfg<KV, D, RB, WR>;
  constexpr int TS = C::kTS;
  constexpr bool kF8 = C::kF8;
  constexpr bool kMmaBf16 = (KV == kKvBf16);
  constexpr int kKSteps = D / 16;
  constexpr int kDvTiles = D / 8;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* empty = full + C::kNumStages;
  int* flags = reinterpret_cast<int*>(empty + C::kNumStages);  // [0] abort, [1] last-CTA

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y / a.rg_count, rg = blockIdx.y % a.rg_count;
  // Inputs may come from the previous kernel in the stream: wait for it before
  // the first global access, then let the next decode call start launching.
  pdl_wait();
  pdl_launch_dependents();

  // Longest sequences first: CTAs launch in blockIdx order, so grid slot z
  // takes the sequence with the z-th most visible tokens (ties by index).
  // The long CTAs then start in the first wave instead of trailing the last
  // one.  Every CTA ranks the (at most 160) sequences itself from shared memory.
  // (Built only where it costs no registers in the main loop: 16-bit K/V
  // with one row block; the fp8 and two-row-block variants would spill.)
  int b = blockIdx.z;
  if (!kF8 && RB == 1 && WR == 1 && a.sort_b) {
    int* eff = reinterpret_cast<int*>(smem);  // the stage ring is unused until the first load
    const int64_t cap = int64_t(a.pps) * a.ps;
    if (tid < a.B) {
      int64_t e = a.seq_lens[tid];
      e = e < cap ? e : cap;
      if (a.win > 0) e = min(e, int64_t(a.win) + a.qs - 1);
      eff[tid] = int(e);
    }
    __syncthreads();
    if (tid < a.B) {
      const int mine = eff[tid];
      int rank = 0;
      for (int j = 0; j < a.B; ++j) {
        const int o = eff[j];
        rank += (o > mine) || (o == mine && j < tid);
      }
      if (rank == int(blockIdx.z)) eff[a.B] = tid;
    }
    __syncthreads();
    b = eff[a.B];
    __syncthreads();  // eff is stage memory: read before anyone reuses it
  }

  // ---- sequence geometry (identical in every CTA of this (b, kvh, rg))
  const int64_t max_len = int64_t(a.pps) * a.ps;
  const int64_t len_raw = a.seq_lens[b];
  const int L = int(len_raw < max_len ? len_raw : max_len);
  if (len_raw > max_len && a.err && tid == 0 && split == 0 && blockIdx.y == 0)
    atomicOr(a.err, kErrClamped);
  const int spec0 = L - a.qs;                       // first new (speculative) token
  const int t_lo_all = a.win > 0 ? max(0, spec0 - a.win + 1) : 0;
  const int pg_first = t_lo_all / a.ps;
  const int pg_last = (L + a.ps - 1) / a.ps;
  const int npages = max(0, pg_last - pg_first);
  const int nvalid = (npages + a.split_pages - 1) / a.split_pages;
  if (split >= max(nvalid, 1)) return;
  const int pg_lo = pg_first + split * a.split_pages;
  const int pg_hi = min(pg_lo + a.split_pages, pg_last);
  const int t_begin = pg_lo * a.ps;
  const int t_end = min(pg_hi * a.ps, L);
  const int nst = (nvalid == 0 || t_end <= t_begin) ? 0 : (t_end - t_begin + C::kTok - 1) / C::kTok;

  if (tid == 0) {
    for (int i = 0; i < C::kNumStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 4);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  const int unit = (b * a.Hkv + kvh) * a.rg_count + rg;
  float* scratch = reinterpret_cast<float*>(smem);  // epilogue: [TS][rows][D] O, then m, l
  float* sc_m = scratch + TS * C::kRows * D;
  float* sc_l = sc_m + TS * C::kRows;
  float* sc_w = sc_l + TS * C::kRows;  // [rows][TS] per-split weights (scales folded in)
  float* sc_ml = sc_w + TS * C::kRows;  // [rows][2] merged (max, sum) of a split partial

  if (warp == 4) {
    // ================= producer (whole warp fetches page indices, lane 0 issues TMA)
    if (nst > 0) {
      if (lane == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
      }
      const int32_t* pt = a.page_table + int64_t(b) * a.pps;
      const int box_rows = a.ps < C::kTok ? a.ps : C::kTok;
      const uint32_t box_bytes = uint32_t(box_rows) * 128u;
      constexpr int kChunkElems = 128 / C::kElt;
      // 32 consecutive page indices, one per lane, starting at win_base
      int win_base = pg_lo;
      auto fetch = [&](int base) {
        int pg = 0;
        if (base + lane < pg_hi) {
          pg = __ldg(pt + base + lane);
          if (pg < 0 || int64_t(pg) >= a.num_pages) pg = -1;  // out of the pool: TMA fills zeros
        }
        return pg;
      };
      int my_page = fetch(win_base);
      bool bad_page = false;
      int s = 0;
      for (; s < nst; ++s) {
        const int slot = s % C::kNumStages;
        const int round = s / C::kNumStages;
        int ok = 1;
        if (lane == 0 && s >= C::kNumStages) ok = mbar_wait(&empty[slot], (round & 1) ^ 1);
        if (!__shfl_sync(0xffffffffu, ok, 0)) {
          if (lane == 0) flags[0] = 1;
          break;
        }
        uint8_t* kdst = smem + slot * C::kStage;
        uint8_t* vdst = kdst + C::kTile;
        const int tok0 = t_begin + s * C::kTok;
        const int lp0 = tok0 / a.ps;
        const int sub = a.ps <= C::kTok ? 0 : tok0 % a.ps;
        const int n_piece = a.ps <= C::kTok ? min(C::kTok / a.ps, pg_hi - lp0) : 1;
        if (lp0 + n_piece > win_base + 32) {
          win_base = lp0;
          my_page = fetch(win_base);
        }
        if (lane == 0)
          mbar_arrive_expect_tx(&full[slot], uint32_t(n_piece) * box_bytes * 2u * C::kChunks);
        __syncwarp();
        // lane j issues the tile loads of page piece j (pieces are independent)
        const int page = __shfl_sync(0xffffffffu, my_page, (lp0 + lane - win_base) & 31);
        if (lane < n_piece) {
          bad_page |= page < 0;
          const int row_off = lane * box_rows;
          for (int c = 0; c < C::kChunks; ++c) {
            const int off = c * C::kTok * 128 + row_off * 128;
            if (a.hnd) {
              tma_load_3d(kdst + off, &tmK, &full[slot], c * kChunkElems, sub, page * a.Hkv + kvh);
              tma_load_3d(vdst + off, &tmV, &full[slot], c * kChunkElems, sub, page * a.Hkv + kvh);
            } else {
              tma_load_3d(kdst + off, &tmK, &full[slot], c * kChunkElems, kvh, page * a.ps + sub);
              tma_load_3d(vdst + off, &tmV, &full[slot], c * kChunkElems, kvh, page * a.ps + sub);
            }
          }
        }
      }
      bad_page = __any_sync(0xffffffffu, bad_page);
      if (lane == 0) {
        if (bad_page && a.err) atomicOr(a.err, kErrClamped);
        // Leave no copy in flight: wait (bounded) for the last stages issued.
        const int first = max(0, s - C::kNumStages);
        for (int t = first; t < s; ++t) {
          if (!mbar_wait(&full[t % C::kNumStages], (t / C::kNumStages) & 1)) flags[0] = 1;
        }
        if (flags[0] && a.err) atomicOr(a.err, kErrTimeout);
      }
    }
  } else {
    // ================= consumers =================
    const int g = lane >> 2, qd = lane & 3;
    const int wr = warp % WR, ts = warp / WR;  // this warp's row group and token split
    const int row0 = wr * RB * 16;             // its first row in the CTA's rows
    const float q_scale = load_scale(a.q_scale_dev, a.q_scale);
    const float kv_scale = load_scale(a.kv_scale_dev, a.kv_scale);
    float lscale = a.softmax_scale * q_scale * kv_scale * kLog2e;

    // ---- query fragments (A operand), rows of this CTA's row group
    uint32_t qa[RB][kKSteps][4];
    {
      const bool qbf = a.q_bf16 != 0;
      const uint16_t* q16 = static_cast<const uint16_t*>(a.q);
      float qv[RB][kKSteps][8];
      float amax = 0.f;
#pragma unroll
      for (int rb = 0; rb < RB; ++rb) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int r = rg * C::kRows + row0 + rb * 16 + g + 8 * hh;
          const bool ok = r < a.R;
          const int i = ok ? r / a.G : 0, gg = ok ? r % a.G : 0;
          const uint16_t* src =
              q16 + ((int64_t(b) * a.qs + i) * a.Hq + int64_t(kvh) * a.G + gg) * D;
#pragma unroll
          for (int kc = 0; kc < kKSteps; ++kc) {
            // element pairs of this lane: (d0, d0+1) and (d1, d1+1)
            int d0, d1;
            if (kF8) {
              d0 = 16 * kc + 4 * qd;
              d1 = d0 + 2;
            } else {
              d0 = 16 * kc + 2 * qd;
              d1 = d0 + 8;
            }
            uint32_t w0 = ok ? __ldg(reinterpret_cast<const uint32_t*>(src + d0)) : 0u;
            uint32_t w1 = ok ? __ldg(reinterpret_cast<const uint32_t*>(src + d1)) : 0u;
            float2 f0 = unpack_16x2(w0, qbf), f1 = unpack_16x2(w1, qbf);
            // fragment slots: [0,1] row g lo-k, [2,3] row g+8 lo-k, [4,5] row g hi-k, [6,7] row g+8 hi-k
            qv[rb][kc][2 * hh + 0] = f0.x;
            qv[rb][kc][2 * hh + 1] = f0.y;
            qv[rb][kc][4 + 2 * hh + 0] = f1.x;
            qv[rb][kc][4 + 2 * hh + 1] = f1.y;
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y))));
          }
        }
      }
      float qmul = 1.f;
      if (kF8 && qbf) {
        // bf16 q feeds an f16 MMA: rescale by a power of two (the largest |q|
        // of the CTA's rows lands in [2^14, 2^15)) and fold the inverse into
        // the logit scale.  Elements down to 2^-31 of that maximum convert
        // exactly (8 significant bits stay on the f16 grid); smaller ones round
        // to the f16 subnormal grid, an error below 2^-40 of the maximum.
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        int e = 0;
        if (amax > 0.f && amax < 3.0e38f) e = 14 - ilogbf(amax);
        e = max(-60, min(60, e));
        qmul = ldexpf(1.f, e);
        lscale *= ldexpf(1.f, -e);
      }
#pragma unroll
      for (int rb = 0; rb < RB; ++rb)
#pragma unroll
        for (int kc = 0; kc < kKSteps; ++kc)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (kF8 && qbf)
              qa[rb][kc][j] = pack_f32x2(qv[rb][kc][2 * j] * qmul, qv[rb][kc][2 * j + 1] * qmul, false);
            else
              qa[rb][kc][j] = pack_f32x2(qv[rb][kc][2 * j], qv[rb][kc][2 * j + 1], kMmaBf16);
          }
    }

    // ---- per-row metadata for the rows this lane holds (g and g+8 of each block)
    int row_lb[RB][2];       // first visible token (window), per row
    uint32_t row_mw[RB][2];  // spec-mask word of the row
#pragma unroll
    for (int rb = 0; rb < RB; ++rb)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int r = rg * C::kRows + row0 + rb * 16 + g + 8 * hh;
        const int i = r < a.R ? r / a.G : 0;
        row_lb[rb][hh] = a.win > 0 ? spec0 + i - a.win + 1 : INT_MIN;
        uint32_t mw = 0xffffffffu;
        if (a.mask) {
          const uint16_t* mrow = a.mask + (int64_t(b) * a.qs + i) * a.mask_words;
          mw = uint32_t(__ldg(mrow)) | (uint32_t(__ldg(mrow + 1)) << 16);
        }
        row_mw[rb][hh] = mw;
      }
    const int lb_max = a.win > 0 ? spec0 + a.qs - 1 - a.win + 1 : INT_MIN;

    float m_run[RB][2], l_run[RB][2];
    float o[RB][kDvTiles][4];
#pragma unroll
    for (int rb = 0; rb < RB; ++rb) {
      m_run[rb][0] = m_run[rb][1] = -INFINITY;
      l_run[rb][0] = l_run[rb][1] = 0.f;
#pragma unroll
      for (int j = 0; j < kDvTiles; ++j) o[rb][j][0] = o[rb][j][1] = o[rb][j][2] = o[rb][j][3] = 0.f;
    }

    constexpr int KB = C::kTok / (16 * TS);  // 16-token blocks per warp and stage
    constexpr int NT = 2 * KB;               // 8-token MMA n-tiles per warp and stage
    const int wt0 = 16 * KB * ts;            // this warp's first row of every stage
    const int mat = lane >> 3;
    for (int s = 0; s < nst; ++s) {
      const int slot = s % C::kNumStages;
      // voted, so the warp leaves together (its shuffles and ldmatrix are collective)
      if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], (s / C::kNumStages) & 1))) {
        flags[0] = 1;
        if (a.err && lane == 0) atomicOr(a.err, kErrTimeout);
        break;
      }
      const int ta = t_begin + s * C::kTok + wt0;  // this warp's first token
      if (ta < t_end) {
        const uint32_t kt = smem_u32(smem + slot * C::kStage);
        const uint32_t vt = kt + C::kTile;
        const bool edge = (ta + 16 * KB > t_end) || (ta < lb_max) || (a.mask && ta + 16 * KB > spec0);

        // ---- S = Q K^T over this warp's tokens (NT independent n-tile chains)
        float sacc[RB][NT][4];
#pragma unroll
        for (int rb = 0; rb < RB; ++rb)
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            sacc[rb][nt][0] = sacc[rb][nt][1] = sacc[rb][nt][2] = sacc[rb][nt][3] = 0.f;
        if constexpr (!kF8) {
#pragma unroll
          for (int kc = 0; kc < kKSteps; ++kc) {
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
              const int tr = wt0 + 16 * kb + (mat >> 1) * 8 + (lane & 7);
              const int u = 2 * kc + (mat & 1);
              const uint32_t addr =
                  kt + (u >> 3) * (C::kTok * 128) + tr * 128 + (((u & 7) ^ (tr & 7)) << 4);
              uint32_t r0, r1, r2, r3;
              ldsm_x4(addr, r0, r1, r2, r3);
#pragma unroll
              for (int rb = 0; rb < RB; ++rb) {
                mma16816<kMmaBf16>(sacc[rb][2 * kb], qa[rb][kc], r0, r1);
                mma16816<kMmaBf16>(sacc[rb][2 * kb + 1], qa[rb][kc], r2, r3);
              }
            }
          }
        } else {
#pragma unroll
          for (int kc2 = 0; kc2 < kKSteps / 2; ++kc2) {
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
              const int tr = wt0 + 16 * kb + (mat & 1) * 8 + (lane & 7);
              const int u = 2 * kc2 + (mat >> 1);
              const uint32_t addr = kt + tr * 128 + (((u & 7) ^ (tr & 7)) << 4);
              uint32_t r[4];
              ldsm_x4(addr, r[0], r[1], r[2], r[3]);
#pragma unroll
              for (int x = 0; x < 4; ++x) {
                const int nt = 2 * kb + (x & 1), kc = 2 * kc2 + (x >> 1);
                uint32_t b01, b23;
                e4m3x4_to_f16x2x2(r[x], b01, b23);
#pragma unroll
                for (int rb = 0; rb < RB; ++rb) mma16816<false>(sacc[rb][nt], qa[rb][kc], b01, b23);
              }
            }
          }
        }

        // ---- scale, mask, online softmax (exp2 domain)
        uint32_t pa[RB][KB][4];
        bool any_rescale = false;
        float corr[RB][2];
#pragma unroll
        for (int rb = 0; rb < RB; ++rb) {
          float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float x = sacc[rb][nt][e] * lscale;
              if (edge) {
                const int hh = e >> 1;
                const int t = ta + 8 * nt + 2 * qd + (e & 1);
                bool vis = t < t_end && t >= row_lb[rb][hh];
                if (a.mask && t >= spec0) vis = vis && ((row_mw[rb][hh] >> (t - spec0)) & 1u);
                x = vis ? x : -INFINITY;
              }
              sacc[rb][nt][e] = x;
              mx[e >> 1] = fmaxf(mx[e >> 1], x);
            }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 1));
            mx[hh] = fmaxf(mx[hh], __shfl_xor_sync(0xffffffffu, mx[hh], 2));
            const float m_new = fmaxf(m_run[rb][hh], mx[hh]);
            corr[rb][hh] = (m_new == -INFINITY) ? 1.f : exp2f(m_run[rb][hh] - m_new);
            any_rescale |= corr[rb][hh] != 1.f;
            m_run[rb][hh] = m_new;
          }
          // P rounded to the MMA's 16-bit type; the row sums use the rounded
          // values so that the output stays a convex combination of V.
          float rs[2] = {0.f, 0.f};
#pragma unroll
          for (int kb = 0; kb < KB; ++kb) {
            float p[2][4];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float mm = m_run[rb][e >> 1];
                p[h2][e] = (mm == -INFINITY) ? 0.f : ex2(sacc[rb][2 * kb + h2][e] - mm);
              }
            pa[rb][kb][0] = pack_f32x2(p[0][0], p[0][1], kMmaBf16);
            pa[rb][kb][1] = pack_f32x2(p[0][2], p[0][3], kMmaBf16);
            pa[rb][kb][2] = pack_f32x2(p[1][0], p[1][1], kMmaBf16);
            pa[rb][kb][3] = pack_f32x2(p[1][2], p[1][3], kMmaBf16);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 f = unpack_16x2(pa[rb][kb][k], kMmaBf16);
              rs[k & 1] += f.x + f.y;
            }
          }
          l_run[rb][0] = l_run[rb][0] * corr[rb][0] + rs[0];
          l_run[rb][1] = l_run[rb][1] * corr[rb][1] + rs[1];
        }
        if (__any_sync(0xffffffffu, any_rescale)) {
#pragma unroll
          for (int rb = 0; rb < RB; ++rb)
#pragma unroll
            for (int j = 0; j < kDvTiles; ++j) {
              o[rb][j][0] *= corr[rb][0];
              o[rb][j][1] *= corr[rb][0];
              o[rb][j][2] *= corr[rb][1];
              o[rb][j][3] *= corr[rb][1];
            }
        }

        // ---- O += P V
#pragma unroll
        for (int kb = 0; kb < KB; ++kb) {
          const int tb = ta + 16 * kb;  // first token of this 16-token block
          if constexpr (!kF8) {
            // V tokens held by this lane: (tb+2qd, +1) in r0/r2, (tb+8+2qd, +1) in r1/r3
            uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
            if (edge) {
              const int t0 = tb + 2 * qd, t1 = tb + 8 + 2 * qd;
              vm0 = ((t0 < t_end && t0 >= t_lo_all) ? 0x0000ffffu : 0u) |
                    ((t0 + 1 < t_end && t0 + 1 >= t_lo_all) ? 0xffff0000u : 0u);
              vm1 = ((t1 < t_end && t1 >= t_lo_all) ? 0x0000ffffu : 0u) |
                    ((t1 + 1 < t_end && t1 + 1 >= t_lo_all) ? 0xffff0000u : 0u);
            }
            const int tr = wt0 + 16 * kb + (mat & 1) * 8 + (lane & 7);
#pragma unroll
            for (int j2 = 0; j2 < kDvTiles / 2; ++j2) {
              const int u = 2 * j2 + (mat >> 1);
              const uint32_t addr =
                  vt + (u >> 3) * (C::kTok * 128) + tr * 128 + (((u & 7) ^ (tr & 7)) << 4);
              uint32_t r0, r1, r2, r3;
              ldsm_x4_t(addr, r0, r1, r2, r3);
              r0 &= vm0;
              r1 &= vm1;
              r2 &= vm0;
              r3 &= vm1;
#pragma unroll
              for (int rb = 0; rb < RB; ++rb) {
                mma16816<kMmaBf16>(o[rb][2 * j2], pa[rb][kb], r0, r1);
                mma16816<kMmaBf16>(o[rb][2 * j2 + 1], pa[rb][kb], r2, r3);
              }
            }
          } else {
            const int r0w = wt0 + 16 * kb;
            const int tl[4] = {r0w + 2 * qd, r0w + 2 * qd + 1, r0w + 8 + 2 * qd, r0w + 9 + 2 * qd};
            bool tv[4] = {true, true, true, true};
            if (edge) {
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const int t = t_begin + s * C::kTok + tl[k];
                tv[k] = t < t_end && t >= t_lo_all;
              }
            }
#pragma unroll
            for (int j4 = 0; j4 < D / 32; ++j4) {
              const int u = 2 * j4 + (g >> 2);
              uint32_t w[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint32_t addr = vt + tl[k] * 128 + (((u & 7) ^ (tl[k] & 7)) << 4) + 4 * (g & 3);
                uint32_t x;
                asm volatile("ld.shared.b32 %0, [%1];" : "=r"(x) : "r"(addr));
                w[k] = tv[k] ? x : 0u;
              }
#pragma unroll
              for (int cp = 0; cp < 2; ++cp) {
                // bytes (c, c) of tokens (0, 1) and of tokens (2, 3) for columns
                // c = 2cp and 2cp + 1: one permute feeds two conversions
                const uint32_t c0 = 2 * cp, c1 = 2 * cp + 1;
                const uint32_t sel = c0 | ((c0 + 4) << 4) | (c1 << 8) | ((c1 + 4) << 12);
                uint32_t b01_c0, b01_c1, b23_c0, b23_c1;
                e4m3x4_to_f16x2x2(prmt(w[0], w[1], sel), b01_c0, b01_c1);
                e4m3x4_to_f16x2x2(prmt(w[2], w[3], sel), b23_c0, b23_c1);
#pragma unroll
                for (int rb = 0; rb < RB; ++rb) {
                  mma16816<false>(o[rb][4 * j4 + c0], pa[rb][kb], b01_c0, b23_c0);
                  mma16816<false>(o[rb][4 * j4 + c1], pa[rb][kb], b01_c1, b23_c1);
                }
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // ---- row sums across the quad, then publish (m, l, O) of this warp
#pragma unroll
    for (int rb = 0; rb < RB; ++rb)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float v = l_run[rb][hh];
        v += __shfl_xor_sync(0xffffffffu, v, 1);
        v += __shfl_xor_sync(0xffffffffu, v, 2);
        l_run[rb][hh] = v;
      }
    named_bar(1, 128);  // every consumer is done with the stage ring
#pragma unroll
    for (int rb = 0; rb < RB; ++rb) {
#pragma unroll
      for (int j = 0; j < kDvTiles; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = row0 + rb * 16 + g + 8 * (e >> 1);
          const int n = 2 * qd + (e & 1);
          const int dv = kF8 ? (32 * (j >> 2) + 4 * n + (j & 3)) : (8 * j + n);
          scratch[(ts * C::kRows + row) * D + dv] = o[rb][j][e];
        }
      if (qd == 0) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int row = row0 + rb * 16 + g + 8 * hh;
          sc_m[ts * C::kRows + row] = m_run[rb][hh];
          sc_l[ts * C::kRows + row] = l_run[rb][hh];
        }
      }
    }
  }
  __syncthreads();
  // A wait gave up: the error word says so and nothing is written, but with
  // several splits the CTA still takes its ticket below, so that the last CTA
  // of the unit resets the semaphore and the next call starts from zero.
  const bool aborted = flags[0] != 0;
  if (aborted && nvalid <= 1) return;

  // ================= epilogue (all 160 threads) =================
  const float kv_scale = load_scale(a.kv_scale_dev, a.kv_scale);
  const float out_mul = kv_scale * a.rcp_out_scale;
  const bool single = nvalid <= 1;
  const int rows_here = min(C::kRows, a.R - rg * C::kRows);
  const int row_stride = D + 4;  // O, then m and l; padded so rows stay 16-byte aligned
  float* ws_unit = a.ws + (int64_t(unit) * a.nsplit) * C::kRows * row_stride;

  // phase 1: one thread per row folds the maxima of the warps holding it (and,
  // with one split, the sink and the output scales) into one weight per warp
  for (int row = aborted ? rows_here : tid; row < rows_here; row += C::kThreads) {
    float mw[TS], M = -INFINITY;
#pragma unroll
    for (int w = 0; w < TS; ++w) {
      mw[w] = sc_m[w * C::kRows + row];
      M = fmaxf(M, mw[w]);
    }
    float f[TS], l = 0.f;
#pragma unroll
    for (int w = 0; w < TS; ++w) {
      f[w] = (mw[w] == -INFINITY) ? 0.f : exp2f(mw[w] - M);
      l += f[w] * sc_l[w * C::kRows + row];
    }
    float mul = 1.f;
    if (single) {
      const int r = rg * C::kRows + row;
      const float sig = a.sinks ? __ldg(a.sinks + kvh * a.G + r % a.G) * kLog2e : -INFINITY;
      mul = finalize_row(M, l, sig, out_mul, a.lse ? a.lse + lse_index(a, b, kvh, r) : nullptr);
    } else {
      sc_ml[2 * row] = M;
      sc_ml[2 * row + 1] = l;
    }
#pragma unroll
    for (int w = 0; w < TS; ++w) sc_w[TS * row + w] = f[w] * mul;
  }
  __syncthreads();
  // phase 2: every (row, 4 columns) combines the warps' partial O
  for (int item = aborted ? rows_here * (D / 4) : tid; item < rows_here * (D / 4); item += C::kThreads) {
    const int row = item / (D / 4);
    const int dv = 4 * (item % (D / 4));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < TS; ++w) {
      const float f = sc_w[TS * row + w];
      const float4 v = *reinterpret_cast<const float4*>(scratch + (w * C::kRows + row) * D + dv);
      acc.x += f * v.x;
      acc.y += f * v.y;
      acc.z += f * v.z;
      acc.w += f * v.w;
    }
    if (single) {
      const int r = rg * C::kRows + row;
      const int i = r / a.G, gg = r % a.G;
      const int64_t oi = ((int64_t(b) * a.qs + i) * a.Hq + int64_t(kvh) * a.G + gg) * a.Dv + dv;
      store_out4(a, oi, acc);
    } else {
      float* dst = ws_unit + (int64_t(split) * C::kRows + row) * row_stride;
      *reinterpret_cast<float4*>(dst + dv) = acc;
      if (dv == 0) {
        dst[D] = sc_ml[2 * row];
        dst[D + 1] = sc_ml[2 * row + 1];
      }
    }
  }
  if (single) return;

  // ---- split-KV: the last CTA of this unit to finish merges every split
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t prev = atomicAdd(a.sems + unit, 1u);
    flags[1] = (prev == uint32_t(nvalid - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!flags[1]) return;
  if (aborted) {  // the last ticket: reset the semaphore, merge nothing
    if (tid == 0) a.sems[unit] = 0u;
    return;
  }
  __threadfence();
  // phase 1: one thread per row folds the split maxima, the sink and the
  // output scales into one weight per (row, split), staged in shared memory
  // (the stage ring is free again)
  float* wts = reinterpret_cast<float*>(smem);  // [rows][nvalid]
  if (tid < rows_here) {
    const int row = tid;
    float M = -INFINITY;
    for (int sp = 0; sp < nvalid; ++sp)
      M = fmaxf(M, __ldcg(ws_unit + (int64_t(sp) * C::kRows + row) * row_stride + D));
    float l = 0.f;
    for (int sp = 0; sp < nvalid; ++sp) {
      const float* src = ws_unit + (int64_t(sp) * C::kRows + row) * row_stride + D;
      const float ms = __ldcg(src);
      const float f = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      wts[row * nvalid + sp] = f;
      l += f * __ldcg(src + 1);
    }
    const int r = rg * C::kRows + row;
    const float sig = a.sinks ? __ldg(a.sinks + kvh * a.G + r % a.G) * kLog2e : -INFINITY;
    const float mul = finalize_row(M, l, sig, out_mul, a.lse ? a.lse + lse_index(a, b, kvh, r) : nullptr);
    for (int sp = 0; sp < nvalid; ++sp) wts[row * nvalid + sp] *= mul;
  }
  __syncthreads();
  // phase 2: every (row, 4-column group) sums the weighted partials
  const int64_t sstride = int64_t(C::kRows) * row_stride;
  for (int item = tid; item < rows_here * (D / 4); item += C::kThreads) {
    const int row = item / (D / 4);
    const int dv = 4 * (item % (D / 4));
    const float* w = wts + row * nvalid;
    const float* src = ws_unit + int64_t(row) * row_stride + dv;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int sp = 0;
    for (; sp + 4 <= nvalid; sp += 4) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = __ldcg(reinterpret_cast<const float4*>(src + (sp + u) * sstride));
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float f = w[sp + u];
        acc.x += f * v[u].x;
        acc.y += f * v[u].y;
        acc.z += f * v[u].z;
        acc.w += f * v[u].w;
      }
    }
    for (; sp < nvalid; ++sp) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(src + sp * sstride));
      const float f = w[sp];
      acc.x += f * v.x;
      acc.y += f * v.y;
      acc.z += f * v.z;
      acc.w += f * v.w;
    }
    const int r = rg * C::kRows + row;
    const int i = r / a.G, gg = r % a.G;
    const int64_t oi = ((int64_t(b) * a.qs + i) * a.Hq + int64_t(kvh) * a.G + gg) * a.Dv + dv;
    store_out4(a, oi, acc);
  }
  if (tid == 0) a.sems[unit] = 0u;
}

}  // namespace xqa
