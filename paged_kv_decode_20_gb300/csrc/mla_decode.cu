// MLA latent decode on the 5th-generation tensor cores (vLLM Kimi-K3
// MultiHeadLatentAttention page: the absorbed query [ql_nope | q_pe] of width
// kv_lora_rank + qk_rope_head_dim = 512 + 64 attends to one latent kv head of
// the same width through forward_mqa; V is the first kv_lora_rank = 512
// elements of each latent row; scale = qk_head_dim^-0.5 arrives as
// softmax_scale).
//
// The 128 query rows (heads x speculative tokens) form one M = 128 UMMA tile.
// Their fp32 output (128 x 512) alone fills a CTA's 512 tensor-memory
// columns, so a cluster of two CTAs shares each (sequence, KV split), each
// CTA holding half of the output columns:
//
//   CTA 0 ("master") owns latent dims [0, 256);
//   CTA 1 ("feeder") owns latent dims [256, 512) plus the rope dims [512, 576).
//   Each CTA streams only its dims of every latent row (TMA, 128-byte
//   swizzle, three-stage mbarrier ring) and computes the partial logits
//   S_c = Q_c K_c^T with tcgen05.mma (A = its latent query half held in
//   tensor memory, B = K from shared memory; CTA 1 adds the rope part with A
//   from shared memory).  CTA 1 ships S_1 (fp32) to CTA 0 with bulk copies
//   into distributed shared memory, a tile ahead of CTA 0's softmax.  CTA 0
//   adds it to S_0, runs the only online softmax, and ships P (bf16, already
//   in UMMA operand layout) with the per-row rescale factors back.  Both CTAs
//   accumulate O_c += P V_c in their own 256 tensor-memory columns, V_c being
//   the first four chunks of the K tile the CTA already holds.  Every latent
//   byte is read from HBM once; CTA 0's softmax waits on no round trip (the
//   feeder ships a tile's logits before the master needs them), while CTA 1's
//   P.V of a tile waits for one message back.
//
// Warp roles: 0 = TMA producer and tensor-memory allocator, 1 = MMA issuer,
// 2..9 = softmax (CTA 0) or logit shipping and O rescale (CTA 1), then the
// epilogue; warp w reaches TMEM lanes 32 (w % 4).. and two threads share a
// query row.  Split-KV partials merge exactly as in the grouped-query kernel:
// the last CTA of each column half to take a ticket merges every split.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "finalize.cuh"
#include "kernel_args.h"
#include "mla_launch.h"
#include "ptx.cuh"
#include "umma.cuh"

namespace xqa {
namespace mla {

constexpr int kRows = 128;       // UMMA M: query rows (heads x spec tokens)
constexpr int kLatent = 512;     // kv_lora_rank (= V width)
constexpr int kRope = 64;        // qk_rope_head_dim
constexpr int kDim = kLatent + kRope;
constexpr int kHalf = kLatent / 2;  // V columns per CTA
constexpr int kTok = 64;         // tokens per tile (UMMA N of QK, K of PV)
constexpr int kChunkBytes = kTok * 128;  // one 64-element column chunk of a tile
constexpr int kSoftWarps = 8;    // two threads per query row, 32 logit columns each
constexpr int kSoft = 32 * kSoftWarps;
constexpr int kSoftWarp0 = 2;    // softmax warps are 2..9: two per TMEM sub-partition
constexpr int kThreads = 32 * kSoftWarp0 + kSoft;

// ---- shared memory (offsets from the dynamic base, which is 1024-aligned:
// checked at run time).  Each CTA keeps two rings: K slots hold a tile's
// chunks until its QK is done; V slots hold the same latent chunks, fetched
// again (from L2, right after the QK) until its P.V is done.  Holding a stage
// only as long as its own use needs lets two slots of each kind cover the
// tile's whole exchange.  The barrier block sits at the same offset in both
// CTAs because each CTA signals barriers of its peer.
constexpr int kXBytes = kRows * kTok * 4;  // one fp32 logit tile
constexpr int kPBytes = kRows * kTok * 2;  // one bf16 P tile
constexpr int kFBytes = kRows * 4;         // one rescale factor per row
constexpr int kPMsg = kPBytes + kFBytes;   // P, then its factors (two copies)
constexpr int kVBytes = 4 * kChunkBytes;   // the four latent chunks of a tile
constexpr int kKBytes0 = 4 * kChunkBytes;  // CTA 0 K slot: 4 latent chunks
constexpr int kKBytes1 = 5 * kChunkBytes;  // CTA 1 K slot: 4 latent chunks + rope
// CTA 0: K x2 | V x2 | P x2 | factors x2 | logit receive slots x2
constexpr int kOffV0 = 2 * kKBytes0;
constexpr int kOffP0 = kOffV0 + 2 * kVBytes;
constexpr int kOffF0 = kOffP0 + 2 * kPBytes;
constexpr int kOffRecv = kOffF0 + 2 * kFBytes;
// CTA 1: K x2 | V x2 | rope query (128 x 64 bf16) | P x2 | factors x2 | send buffer
constexpr int kOffV1 = 2 * kKBytes1;
constexpr int kOffQRope = kOffV1 + 2 * kVBytes;
constexpr int kOffP1 = kOffQRope + kRows * 128;
constexpr int kOffF1 = kOffP1 + 2 * kPBytes;
constexpr int kOffSend = kOffF1 + 2 * kFBytes;
// both: [2][128] floats (CTA 0: row maxima / sums; CTA 1: the final m and l)
constexpr int kOffRowX = (kOffRecv + 2 * kXBytes) > (kOffSend + kXBytes) ? (kOffRecv + 2 * kXBytes)
                                                                         : (kOffSend + kXBytes);
constexpr int kOffBar = kOffRowX + 2 * kRows * 4;

enum BarIdx {
  kKFull = 0,                   // [2] a K slot's bytes landed
  kKEmpty = kKFull + 2,         // [2] the QK reading a K slot is done
  kVFull = kKEmpty + 2,         // [2] a V slot's bytes landed
  kVEmpty = kVFull + 2,         // [2] the P.V reading a V slot is done
  kQReady = kVEmpty + 2,        // the query is in tensor / shared memory
  kSFull = kQReady + 1,         // [2] S tile computed
  kSFree = kSFull + 2,          // [2] S tile read out of tensor memory
  kPFull = kSFree + 2,          // P (and any O rescale) ready for the P.V
  kPvDone = kPFull + 1,         // the last P.V issued is done
  kDrain = kPvDone + 1,         // every MMA this CTA issued is done
  kXFull = kDrain + 1,          // CTA 0 [2]: the peer's logit tile landed
  kXFree = kXFull + 2,          // CTA 1: CTA 0 received the previous logit tile
  kPIn = kXFree + 1,            // CTA 1 [2]: a P message landed
  kPSlotFree = kPIn + 2,        // CTA 0 [2]: CTA 1's P.V on that P slot is done
  kFin = kPSlotFree + 2,        // CTA 1: the final (m, l) rows landed
  kNumBars = kFin + 1
};
constexpr int kSmem = kOffBar + kNumBars * 8 + 32;
static_assert(kSmem <= 232448, "shared memory budget");
static_assert(kOffV0 % 1024 == 0 && kOffP0 % 1024 == 0 && kOffV1 % 1024 == 0 && kOffP1 % 1024 == 0 &&
                  kOffQRope % 1024 == 0 && kOffRecv % 16 == 0 && kOffSend % 16 == 0 && kOffF0 % 16 == 0 &&
                  kOffF1 % 16 == 0,
              "UMMA operands need 1024-byte alignment, bulk copies 16");
constexpr int kCopyPieces = 4;  // the logit tile and the P tile travel as this many bulk copies
static_assert(kPBytes % (16 * kCopyPieces) == 0 && kXBytes % (16 * kCopyPieces) == 0, "copy pieces");

// tensor memory columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;     // 256 fp32 columns: O half
constexpr uint32_t kColQ = 256;   // 128 columns: latent query half, bf16 pairs
constexpr uint32_t kColS = 384;   // 2 x 64 columns: logits double buffer

constexpr float kRescaleLog2 = 8.f;  // rescale O only when the max grows by > 2^8
constexpr int kMaxSplits = 64;       // merge weights [128][splits] fit in shared memory

struct MlaArgs {
  const uint16_t* q;  // [B, qs, Hq, 576]
  uint16_t* out;      // [B, qs, Hq, 512]
  const int32_t* page_table;
  const uint32_t* seq_lens;
  const float* sinks;
  const uint16_t* mask;
  const float* q_scale_dev;
  const float* kv_scale_dev;
  float* ws;
  uint32_t* sems;
  uint32_t* err;
  float* lse;  // optional [B, qs, Hq] natural-log log-sum-exp per row
  int64_t num_pages;
  int B, Hq, qs, ps, pps, win, nsplit, split_pages, mask_words;
  float q_scale, kv_scale, softmax_scale, rcp_out_scale;
  int q_bf16;
};

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t map_peer(uint32_t saddr, uint32_t peer) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(peer));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// One bulk copy of `bytes` from this CTA's shared memory into the peer's,
// completing that many transaction bytes on the peer's mbarrier.
__device__ __forceinline__ void bulk_to_peer(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes,
                                             uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst_cluster),
      "r"(src_cta), "r"(bytes), "r"(bar_cluster)
      : "memory");
}
// Tells the peer that this CTA has received what the peer sent.  The arrive
// carries no data of its own, so relaxed ordering suffices and avoids a
// cluster-scope release.
__device__ __forceinline__ void remote_arrive(uint32_t rbar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(rbar) : "memory");
}
// Arrives once on the barrier at the same offset in every CTA of `mask` when
// every MMA this thread issued so far is done.
__device__ __forceinline__ void commit_to(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ float ldscale(const float* dev, float host) { return dev ? __ldg(dev) : host; }

// 16-byte unit u (0..15) of row t of a 128 x 64 fp32 buffer, XOR-swizzled by row.
__device__ __forceinline__ int xunit(int t, int u) { return t * kTok + ((u ^ (t & 15)) & 15) * 4; }

// Multiplies this warp's 32 rows of O columns [128h, 128h + 128) by f.
__device__ __forceinline__ void rescale_o(uint32_t taddr, float f) {
#pragma unroll 1
  for (int part = 0; part < kHalf / 64; ++part) {
    float o[32];
    umma::tmem_ld32(taddr + 32u * part, o);
    umma::tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] *= f;
    umma::tmem_st32(taddr + 32u * part, reinterpret_cast<const uint32_t*>(o));
  }
  umma::tmem_st_wait();
}

// Zeroes V rows [r0, kTok) of a stage's four latent chunks: past a split's
// last token the rows hold stale or foreign data (possibly NaN), and P = 0
// there must not meet it in the P.V.
__device__ __forceinline__ void zero_v_tail(uint8_t* stage, int r0, int st) {
  for (int idx = st; idx < (kTok - r0) * 4 * 8; idx += kSoft) {
    const int r = r0 + idx / 32, k = (idx / 8) % 4, u = idx % 8;
    *reinterpret_cast<uint4*>(stage + k * kChunkBytes + r * 128 + u * 16) = make_uint4(0, 0, 0, 0);
  }
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmKV, const MlaArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] abort, [1] last CTA

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t c = cluster_rank();
  const uint32_t peer = c ^ 1u;
  const int split = blockIdx.x >> 1;
  const int b = blockIdx.z;

  // wait for the producer of our inputs, then let the next call start launching
  pdl_wait();
  pdl_launch_dependents();

  // ---- sequence geometry (identical in both CTAs and every split)
  const int64_t max_len = int64_t(a.pps) * a.ps;
  const int64_t len_raw = a.seq_lens[b];
  const int L = int(len_raw < max_len ? len_raw : max_len);
  if (len_raw > max_len && a.err && tid == 0 && blockIdx.x == 0) atomicOr(a.err, kErrClamped);
  const int spec0 = L - a.qs;
  const int t_lo_all = a.win > 0 ? max(0, spec0 - a.win + 1) : 0;
  const int pg_first = t_lo_all / a.ps;
  const int pg_last = (L + a.ps - 1) / a.ps;
  const int npages = max(0, pg_last - pg_first);
  const int nvalid = (npages + a.split_pages - 1) / a.split_pages;
  if (split >= max(nvalid, 1)) return;  // both CTAs of the cluster leave together
  const int pg_lo = pg_first + split * a.split_pages;
  const int pg_hi = min(pg_lo + a.split_pages, pg_last);
  const int t_begin = pg_lo * a.ps;
  const int t_end = min(pg_hi * a.ps, L);
  const int ntiles = (nvalid == 0 || t_end <= t_begin) ? 0 : (t_end - t_begin + kTok - 1) / kTok;
  const int nchunks = c == 0 ? 4 : 5;  // chunks of a K slot
  const int kbytes = c == 0 ? kKBytes0 : kKBytes1;
  const int off_v = c == 0 ? kOffV0 : kOffV1;
  const int off_p = c == 0 ? kOffP0 : kOffP1;
  // the layout assumes a 1024-aligned dynamic base (the 128-byte swizzle
  // atoms of the UMMA operands); both CTAs see the same base and leave together
  if (smem_u32(smem_raw) & 1023u) {
    if (tid == 0 && a.err) atomicOr(a.err, kErrTimeout);
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kKFull + i], 1);
      mbar_init(&bars[kKEmpty + i], 1);
      mbar_init(&bars[kVFull + i], 1);
      mbar_init(&bars[kVEmpty + i], 1);
    }
    mbar_init(&bars[kQReady], kSoftWarps);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bars[kSFull + k], 1);
      mbar_init(&bars[kSFree + k], kSoftWarps);
      mbar_init(&bars[kXFull + k], 1);      // own expect-tx arrival + the peer's bytes
      mbar_init(&bars[kPIn + k], 1);        // own expect-tx arrival + the peer's bytes
      mbar_init(&bars[kPSlotFree + k], 1);  // the peer's MMA completion
    }
    mbar_init(&bars[kPFull], kSoftWarps);
    mbar_init(&bars[kPvDone], 1);
    mbar_init(&bars[kDrain], 1);
    mbar_init(&bars[kXFree], 1);
    mbar_init(&bars[kFin], 1);
    flags[0] = flags[1] = 0;
    // the first two receive slots and the final rows are expected up front
    for (int k = 0; k < min(2, ntiles); ++k)
      mbar_arrive_expect_tx(&bars[c == 0 ? kXFull + k : kPIn + k], c == 0 ? kXBytes : kPMsg);
    if (c == 1) mbar_arrive_expect_tx(&bars[kFin], 2 * kRows * 4);
    fence_mbar_init();
  }
  if (warp == 0) {
    umma::tmem_alloc(tmem_slot, kTmemCols);
    umma::tmem_relinquish();
  }
  umma::fence_before_sync();
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before any remote access
  umma::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t peer_bars = map_peer(smem_u32(bars), peer);

  if (warp == 0) {
    // ================= TMA producer (lane 0 decides, lane j loads page piece j)
    // K(j) may load once the QK of tile j - 2 is done (its slot is free); V(j)
    // once the QK of tile j is done and the P.V of tile j - 2 has freed its V
    // slot.  Tests never block; the loop gives up after kWaitCycles idle.
    if (ntiles > 0) {
      if (lane == 0) prefetch_tensormap(&tmKV);
      const int32_t* pt = a.page_table + int64_t(b) * a.pps;
      const int box_rows = min(a.ps, kTok);
      const uint32_t box_bytes = uint32_t(box_rows) * 128u;
      bool bad_page = false;
      // all tile loads of tile j (nck chunks per page piece) into dst, on bar
      auto issue = [&](int j, uint8_t* dst, uint64_t* bar, int nck) {
        const int tok0 = t_begin + j * kTok;
        const int lp0 = tok0 / a.ps;
        const int sub = a.ps <= kTok ? 0 : tok0 % a.ps;
        const int n_piece = a.ps <= kTok ? min(kTok / a.ps, pg_hi - lp0) : 1;
        if (lane == 0) mbar_arrive_expect_tx(bar, uint32_t(n_piece) * box_bytes * nck);
        __syncwarp();
        if (lane < n_piece) {
          int page = __ldg(pt + lp0 + lane);
          if (page < 0 || int64_t(page) >= a.num_pages) {
            page = -1;  // the TMA fills zeros
            bad_page = true;
          }
          for (int k = 0; k < nck; ++k) {
            // chunk k: latent dims 256c + 64k (k < 4) or the rope dims
            const int x = k < 4 ? int(c) * kHalf + 64 * k : kLatent;
            tma_load_3d(dst + k * kChunkBytes + lane * box_rows * 128, &tmKV, bar, x, 0, page * a.ps + sub);
          }
        }
        __syncwarp();
      };
      // the tile two K loads ahead goes into L2 early, so that its own load
      // (issued only when a K slot frees) does not pay HBM latency
      auto prefetch = [&](int j) {
        if (j >= ntiles) return;
        const int tok0 = t_begin + j * kTok;
        const int lp0 = tok0 / a.ps;
        const int sub = a.ps <= kTok ? 0 : tok0 % a.ps;
        const int n_piece = a.ps <= kTok ? min(kTok / a.ps, pg_hi - lp0) : 1;
        if (lane < n_piece) {
          const int pg = __ldg(pt + lp0 + lane);
          if (pg >= 0 && int64_t(pg) < a.num_pages)
            for (int k = 0; k < nchunks; ++k)
              tma_prefetch_l2_3d(&tmKV, k < 4 ? int(c) * kHalf + 64 * k : kLatent, 0, pg * a.ps + sub);
        }
      };
      int nk = 0, nv = 0, seen = 0;  // K loads, V loads issued; QKs seen done (lane 0)
      long long t_idle = clock64();
      while (true) {
        int dec = 0;  // 1: load K(nk), 2: load V(nv), 3: finished, 4: gave up
        if (lane == 0) {
          if (seen < nk && mbar_test(&bars[kKEmpty + (seen & 1)], (seen >> 1) & 1)) {
            ++seen;
            t_idle = clock64();
          }
          if (nv >= ntiles)
            dec = 3;
          else if (nk < ntiles && nk < seen + 2)
            dec = 1;
          else if (nv < seen && (nv < 2 || mbar_test(&bars[kVEmpty + (nv & 1)], ((nv >> 1) - 1) & 1)))
            dec = 2;
          else if (clock64() - t_idle > kWaitCycles)
            dec = 4;
        }
        dec = __shfl_sync(0xffffffffu, dec, 0);
        if (dec == 3) break;
        if (dec == 4) {
          if (lane == 0) flags[0] = 1;
          break;
        }
        if (dec == 1) {
          issue(nk, smem + (nk & 1) * kbytes, &bars[kKFull + (nk & 1)], nchunks);
          prefetch(nk + 2);
          ++nk;
        } else if (dec == 2) {
          issue(nv, smem + off_v + (nv & 1) * kVBytes, &bars[kVFull + (nv & 1)], 4);
          ++nv;
        }
        if (dec && lane == 0) t_idle = clock64();
      }
      bad_page = __any_sync(0xffffffffu, bad_page);
      if (lane == 0) {
        if (bad_page && a.err) atomicOr(a.err, kErrClamped);
        // no load of this CTA may land after it exits
        for (int t = max(0, nk - 2); t < nk; ++t)
          if (!mbar_wait(&bars[kKFull + (t & 1)], (t >> 1) & 1)) flags[0] = 1;
        for (int t = max(0, nv - 2); t < nv; ++t)
          if (!mbar_wait(&bars[kVFull + (t & 1)], (t >> 1) & 1)) flags[0] = 1;
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    if (lane == 0 && ntiles > 0) {
      constexpr uint32_t kIdescQK = umma::idesc_f16(kRows, kTok, true, false, false);
      constexpr uint32_t kIdescPV = umma::idesc_f16(kRows, kHalf, true, false, true);
      const uint32_t kbase = smem_u32(smem);
      const uint32_t vbase = smem_u32(smem + off_v);
      const uint32_t pslot = smem_u32(smem + off_p);
      const uint32_t qrope = smem_u32(smem + kOffQRope);
      bool ok = mbar_wait(&bars[kQReady], 0);
      umma::fence_after_sync();
      auto issue_qk = [&](int j) {
        const uint32_t st = kbase + (j & 1) * kbytes;
        const uint32_t sd = tmem + kColS + 64u * uint32_t(j & 1);
        for (int k = 0; k < 4; ++k)
          for (int kk = 0; kk < 4; ++kk)
            umma::mma_ts(sd, tmem + kColQ + 32u * k + 8u * kk,
                         umma::smem_desc(st + k * kChunkBytes + 32 * kk, 16, 1024, umma::kSw128),
                         kIdescQK, (k | kk) != 0);
        if (c == 1)
          for (int kk = 0; kk < 4; ++kk)
            umma::mma_ss(sd, umma::smem_desc(qrope + 32 * kk, 16, 1024, umma::kSw128),
                         umma::smem_desc(st + 4 * kChunkBytes + 32 * kk, 16, 1024, umma::kSw128),
                         kIdescQK, 1u);
        umma::commit(&bars[kSFull + (j & 1)]);
        umma::commit(&bars[kKEmpty + (j & 1)]);  // the K slot may refill
      };
      auto issue_pv = [&](int j) {
        const uint32_t st = vbase + (j & 1) * kVBytes;
        const uint32_t pa = pslot + (j & 1) * kPBytes;
        for (int kk = 0; kk < 4; ++kk)
          umma::mma_ss(tmem + kColO, umma::smem_desc(pa + 32 * kk, 16, 1024, umma::kSw128),
                       umma::smem_desc(st + 2048 * kk, kChunkBytes, 1024, umma::kSw128), kIdescPV,
                       (j | kk) != 0);
        umma::commit(&bars[kVEmpty + (j & 1)]);
        umma::commit(&bars[kPvDone]);
        // the P slot may take CTA 0's next message once this P.V has read it
        if (c == 1) commit_to(&bars[kPSlotFree + (j & 1)], uint16_t(1u));
      };
      // Issue whichever is ready: the P.V of the oldest tile (it frees a V
      // slot) or the logits of the next one, so QK runs ahead of the round
      // trip that P takes.  Tests never block; the loop gives up after
      // kWaitCycles without progress.
      int nq = 0, np = 0;
      long long t_idle = clock64();
      while (ok && np < ntiles) {
        bool moved = false;
        // CTA 1's P arrives from the peer; CTA 0 wrote its own
        if (np < nq && mbar_test(&bars[kPFull], np & 1) &&
            mbar_test(&bars[kVFull + (np & 1)], (np >> 1) & 1) &&
            (c == 0 || mbar_test(&bars[kPIn + (np & 1)], (np >> 1) & 1))) {
          umma::fence_after_sync();
          issue_pv(np++);
          moved = true;
        }
        if (nq < ntiles && mbar_test(&bars[kKFull + (nq & 1)], (nq >> 1) & 1) &&
            (nq < 2 || mbar_test(&bars[kSFree + (nq & 1)], ((nq >> 1) - 1) & 1))) {
          umma::fence_after_sync();
          issue_qk(nq++);
          moved = true;
        }
        if (moved)
          t_idle = clock64();
        else if (clock64() - t_idle > kWaitCycles)
          ok = false;
      }
      if (!ok) flags[0] = 1;
      // nothing this thread issued may still run when tensor memory is freed
      umma::commit(&bars[kDrain]);
      if (!mbar_wait(&bars[kDrain], 0)) flags[0] = 1;
    }
  } else {
    // ================= softmax / logit shipping / epilogue =================
    // Warp w (2..9) reaches TMEM lanes 32 (w % 4) .. +31 (query rows); h = (w - 2) / 4
    // picks logit columns [32h, 32h + 32) of every tile and O columns [128h, 128h+128).
    const int q4 = warp & 3, h = (warp - kSoftWarp0) >> 2;
    const int t = 32 * q4 + lane;            // query row = TMEM lane
    const int st = tid - 32 * kSoftWarp0;    // 0 .. kSoft - 1
    const uint32_t lane_base = uint32_t(32 * q4) << 16;
    const uint32_t o_cols = tmem + lane_base + kColO + 128u * h;
    const int i = t / a.Hq, hd = t % a.Hq;  // row t = (spec token i, head hd)
    const float q_scale = ldscale(a.q_scale_dev, a.q_scale);
    const float kv_scale = ldscale(a.kv_scale_dev, a.kv_scale);
    const float lscale = a.softmax_scale * q_scale * kv_scale * kLog2e;
    float* rowx = reinterpret_cast<float*>(smem + kOffRowX);  // [2][128]
    constexpr unsigned kAll = 0xffffffffu;
    constexpr int kC = kTok / 2;  // logit columns per thread

    // ---- query: this thread's half of the row's latent half into tensor
    // memory; the rope part into shared memory (CTA 1)
    {
      const uint16_t* qrow = a.q + (int64_t(b) * a.qs * a.Hq + t) * kDim;
      const uint4* src = reinterpret_cast<const uint4*>(qrow + c * kHalf + 128 * h);
#pragma unroll
      for (int part = 0; part < 2; ++part) {  // 2 x 32 columns = 128 bf16
        uint32_t w[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = __ldg(src + part * 8 + v);
          w[4 * v + 0] = x.x;
          w[4 * v + 1] = x.y;
          w[4 * v + 2] = x.z;
          w[4 * v + 3] = x.w;
        }
        umma::tmem_st32(tmem + lane_base + kColQ + 64u * h + 32u * part, w);
      }
      if (c == 1) {
        const uint4* rsrc = reinterpret_cast<const uint4*>(qrow + kLatent);
        for (int u = 4 * h; u < 4 * h + 4; ++u)
          *reinterpret_cast<uint4*>(smem + kOffQRope + umma::sw128(t, u)) = __ldg(rsrc + u);
      }
      umma::tmem_st_wait();
      umma::fence_proxy_async_smem();
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kQReady]);
    }

    float m_ref = -INFINITY, l_half = 0.f;
    bool ok = true;
    // Control flow stays uniform across each warp (tcgen05.ld / st are
    // warp-collective) and across the eight softmax warps (named barrier 1):
    // waits are voted and loops are left collectively.
    if (c == 0) {
      // ---------------- CTA 0: full logits, online softmax, P for both CTAs
      const float* recv = reinterpret_cast<const float*>(smem + kOffRecv);
      const uint32_t pslot_peer = map_peer(smem_u32(smem + kOffP1), peer);
      const uint32_t fslot_peer = map_peer(smem_u32(smem + kOffF1), peer);
      const int row_lb = a.win > 0 ? spec0 + i - a.win + 1 : INT_MIN;
      uint32_t row_mw = 0xffffffffu;
      if (a.mask) {
        const uint16_t* mrow = a.mask + (int64_t(b) * a.qs + i) * a.mask_words;
        row_mw = uint32_t(__ldg(mrow)) | (uint32_t(__ldg(mrow + 1)) << 16);
      }
      for (int j = 0; j < ntiles; ++j) {
        const int sb = j & 1;
        const uint32_t par = (j >> 1) & 1;
        float s[kC];
        ok = __all_sync(kAll, mbar_wait(&bars[kSFull + sb], par));
        if (ok) {
          umma::fence_after_sync();
          umma::tmem_ld32(tmem + lane_base + kColS + 64u * sb + 32u * h, s);
          umma::tmem_ld_wait();
          umma::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kSFree + sb]);
          // the peer's partial logits of this tile
          ok = __all_sync(kAll, mbar_wait(&bars[kXFull + sb], par));
        }
        // received: the peer may refill its send buffer (and so this CTA's other
        // slot); after the last tile nobody waits for the signal, so none is sent
        if (ok && st == 0 && j + 1 < ntiles) remote_arrive(peer_bars + 8u * kXFree);
        const int tile0 = t_begin + j * kTok;
        float mx = -INFINITY;
        if (ok) {
          const float* rx = recv + sb * (kXBytes / 4);
#pragma unroll
          for (int v = 0; v < kC / 4; ++v) {
            const float4 p4 = *reinterpret_cast<const float4*>(rx + xunit(t, 8 * h + v));
            s[4 * v] += p4.x;
            s[4 * v + 1] += p4.y;
            s[4 * v + 2] += p4.z;
            s[4 * v + 3] += p4.w;
          }
          // visibility of this thread's 32 columns as one bit each (all set
          // away from the split's end, the window start and the spec tokens)
          const bool edge = tile0 + kTok > t_end || tile0 <= row_lb || (a.mask && tile0 + kTok > spec0);
          uint32_t vis = 0xffffffffu;
          if (edge) {
            vis = 0u;
#pragma unroll 1
            for (int k = 0; k < kC; ++k) {
              const int tt = tile0 + 32 * h + k;
              bool v = tt < t_end && tt >= row_lb;
              if (a.mask && tt >= spec0) v = v && ((row_mw >> (tt - spec0)) & 1u);
              vis |= uint32_t(v) << k;
            }
          }
#pragma unroll
          for (int k = 0; k < kC; ++k) {
            const float x = (vis >> k) & 1u ? s[k] * lscale : -INFINITY;
            s[k] = x;
            mx = fmaxf(mx, x);
          }
          rowx[h * kRows + t] = mx;
        }
        // both halves of every row published their maxima; the slot is consumed
        if (named_bar_or(1, kSoft, !ok)) {
          ok = false;
          break;
        }
        if (st == 0 && j + 2 < ntiles) mbar_arrive_expect_tx(&bars[kXFull + sb], kXBytes);
        mx = fmaxf(mx, rowx[(1 - h) * kRows + t]);
        // O may be rescaled once the previous P.V is done; P slot sb is free
        // once both CTAs' P.V of tile j - 2 are done (which also means its
        // copy to the peer has landed)
        if (j > 0) ok = __all_sync(kAll, mbar_wait(&bars[kPvDone], (j - 1) & 1));
        if (ok && j >= 2) ok = __all_sync(kAll, mbar_wait(&bars[kPSlotFree + sb], ((j >> 1) - 1) & 1));
        uint8_t* pbuf = smem + kOffP0 + sb * kPBytes;
        float* fbuf = reinterpret_cast<float*>(smem + kOffF0 + sb * kFBytes);
        if (ok) {
          umma::fence_after_sync();
          const float m_new = fmaxf(m_ref, mx);
          const bool need = m_new > m_ref + kRescaleLog2 || (m_ref == -INFINITY && m_new != -INFINITY);
          const float f = (need && m_ref != -INFINITY) ? exp2f(m_ref - m_new) : 1.f;
          if (need) {
            l_half *= f;
            m_ref = m_new;
          }
          // P (bf16) for this thread's 32 columns: units 4h..4h+3 of row t; the
          // row sum takes the rounded weights so O / l stays a convex combination
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float p0 = m_ref == -INFINITY ? 0.f : ex2(s[8 * u + 2 * e] - m_ref);
              const float p1 = m_ref == -INFINITY ? 0.f : ex2(s[8 * u + 2 * e + 1] - m_ref);
              w4[e] = pack_f32x2(p0, p1, true);
              const float2 r = unpack_16x2(w4[e], true);
              l_half += r.x + r.y;
            }
            *reinterpret_cast<uint4*>(pbuf + umma::sw128(t, 4 * h + u)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
          if (h == 0) fbuf[t] = f;
          // the split's last tile: its V slot must have landed before the tail is cleared
          if (tile0 + kTok > t_end) {
            ok = __all_sync(kAll, mbar_wait(&bars[kVFull + sb], (j >> 1) & 1));
            if (ok) zero_v_tail(smem + kOffV0 + sb * kVBytes, max(0, t_end - tile0), st);
          }
          // whole warp rescales its rows' O half-columns (factor 1 where unchanged)
          if (__any_sync(kAll, f != 1.f)) rescale_o(o_cols, f);
          umma::fence_proxy_async_smem();
          umma::fence_before_sync();
        }
        // every thread finished P, the factors and the V tail, or someone gave up
        if (named_bar_or(1, kSoft, !ok)) {
          ok = false;
          break;
        }
        if (lane == 0) mbar_arrive(&bars[kPFull]);
        // P in four copies from four warps, the factors in a fifth
        if ((st & 31) == 0 && st < 32 * kCopyPieces) {
          const uint32_t off = uint32_t(st >> 5) * (kPBytes / kCopyPieces);
          bulk_to_peer(pslot_peer + sb * kPBytes + off, smem_u32(pbuf) + off, kPBytes / kCopyPieces,
                       peer_bars + 8u * (kPIn + sb));
        } else if (st == 32 * kCopyPieces) {
          bulk_to_peer(fslot_peer + sb * kFBytes, smem_u32(fbuf), kFBytes, peer_bars + 8u * (kPIn + sb));
        }
      }
    } else {
      // ---------------- CTA 1: ship partial logits a tile ahead, apply P
      float* send = reinterpret_cast<float*>(smem + kOffSend);
      const uint32_t recv_peer = map_peer(smem_u32(smem + kOffRecv), peer);
      for (int j = 0; j <= ntiles; ++j) {
        if (j < ntiles) {
          const int sb = j & 1;
          float s[kC];
          ok = __all_sync(kAll, mbar_wait(&bars[kSFull + sb], (j >> 1) & 1));
          if (ok) {
            umma::fence_after_sync();
            umma::tmem_ld32(tmem + lane_base + kColS + 64u * sb + 32u * h, s);
            umma::tmem_ld_wait();
            umma::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kSFree + sb]);
            // the send buffer and the peer's slot sb are free once the peer
            // has received the previous tile
            if (j > 0 && st == 0) ok = mbar_wait(&bars[kXFree], (j - 1) & 1);
          }
          if (named_bar_or(1, kSoft, !ok)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int v = 0; v < kC / 4; ++v)
            *reinterpret_cast<float4*>(send + xunit(t, 8 * h + v)) =
                make_float4(s[4 * v], s[4 * v + 1], s[4 * v + 2], s[4 * v + 3]);
          umma::fence_proxy_async_smem();
          named_bar(1, kSoft);
          if ((st & 31) == 0 && st < 32 * kCopyPieces) {
            const uint32_t off = uint32_t(st >> 5) * (kXBytes / kCopyPieces);
            bulk_to_peer(recv_peer + sb * kXBytes + off, smem_u32(send) + off, kXBytes / kCopyPieces,
                         peer_bars + 8u * (kXFull + sb));
          }
        }
        if (j > 0) {
          // P of the previous tile: rescale O as the master did, then release the P.V
          const int jp = j - 1, kp = jp & 1;
          ok = __all_sync(kAll, mbar_wait(&bars[kPIn + kp], (jp >> 1) & 1));
          if (ok && jp > 0) ok = __all_sync(kAll, mbar_wait(&bars[kPvDone], (jp - 1) & 1));
          if (ok) {
            umma::fence_after_sync();
            const float f = reinterpret_cast<const float*>(smem + kOffF1 + kp * kFBytes)[t];
            if (__any_sync(kAll, f != 1.f)) rescale_o(o_cols, f);
            const int tile0 = t_begin + jp * kTok;
            if (tile0 + kTok > t_end) {
              ok = __all_sync(kAll, mbar_wait(&bars[kVFull + kp], (jp >> 1) & 1));
              if (ok) zero_v_tail(smem + kOffV1 + kp * kVBytes, max(0, t_end - tile0), st);
            }
            umma::fence_proxy_async_smem();
            umma::fence_before_sync();
          }
          // the slot's next message (tile jp + 2) is expected before its P.V frees it
          if (st == 0 && jp + 2 < ntiles) mbar_arrive_expect_tx(&bars[kPIn + kp], kPMsg);
          if (named_bar_or(1, kSoft, !ok)) {
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive(&bars[kPFull]);
        }
      }
    }
    if (!ok) flags[0] = 1;

    // ---- epilogue: wait for the last P.V, agree on (m, l), then finalise or
    // write the partial
    const bool have_o = ntiles > 0;
    if (have_o && ok && !__all_sync(kAll, mbar_wait(&bars[kPvDone], (ntiles - 1) & 1))) {
      flags[0] = 1;
      ok = false;
    }
    umma::fence_after_sync();
    float l_run;
    if (c == 0) {
      // the peer's completion signals for the last two P slots must land
      // before this CTA may exit
      for (int j = max(0, ntiles - 2); ok && j < ntiles; ++j)
        ok = __all_sync(kAll, mbar_wait(&bars[kPSlotFree + (j & 1)], (j >> 1) & 1));
      if (!ok) flags[0] = 1;
      rowx[h * kRows + t] = l_half;
      named_bar(1, kSoft);
      l_run = rowx[t] + rowx[kRows + t];
      named_bar(1, kSoft);
      if (h == 0) {
        rowx[t] = m_ref;
        rowx[kRows + t] = l_run;
      }
      umma::fence_proxy_async_smem();
      named_bar(1, kSoft);
      if (st == 0)
        bulk_to_peer(map_peer(smem_u32(rowx), peer), smem_u32(rowx), 2 * kRows * 4, peer_bars + 8u * kFin);
    } else {
      if (!__all_sync(kAll, mbar_wait(&bars[kFin], 0))) {
        flags[0] = 1;
        ok = false;
      }
      m_ref = rowx[t];
      l_run = rowx[kRows + t];
    }
    if (ok) {
      const bool single = nvalid <= 1;
      float mul = 0.f;
      const int64_t row_g = (int64_t(b) * a.qs + i) * a.Hq + hd;
      if (single) {
        const float sig = a.sinks ? __ldg(a.sinks + hd) * kLog2e : -INFINITY;
        mul = finalize_row(m_ref, l_run, sig, kv_scale * a.rcp_out_scale,
                           (a.lse && c == 0 && h == 0) ? a.lse + row_g : nullptr);
      }
      float* wrow = a.ws + ((int64_t(b) * a.nsplit + split) * kRows + t) * (kLatent + 4);
#pragma unroll
      for (int part = 0; part < kHalf / 64; ++part) {
        float o[32];
        if (have_o) {
          umma::tmem_ld32(o_cols + 32u * part, o);
          umma::tmem_ld_wait();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = 0.f;
        }
        const int col = int(c) * kHalf + 128 * h + 32 * part;
        if (single) {
          uint4* dst = reinterpret_cast<uint4*>(a.out + row_g * kLatent + col);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(pack_f32x2(o[8 * v] * mul, o[8 * v + 1] * mul, true),
                                pack_f32x2(o[8 * v + 2] * mul, o[8 * v + 3] * mul, true),
                                pack_f32x2(o[8 * v + 4] * mul, o[8 * v + 5] * mul, true),
                                pack_f32x2(o[8 * v + 6] * mul, o[8 * v + 7] * mul, true));
        } else {
          float4* dst = reinterpret_cast<float4*>(wrow + col);
#pragma unroll
          for (int v = 0; v < 8; ++v) dst[v] = make_float4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
        }
      }
      if (!single && h == 0) {
        wrow[kLatent + 2 * c] = m_ref;
        wrow[kLatent + 2 * c + 1] = l_run;
      }
    }
  }

  // ---- teardown: no tensor-memory or peer traffic may outlive this point
  umma::fence_before_sync();
  __syncthreads();
  cluster_sync();
  if (warp == 0) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
  if (flags[0]) {
    if (tid == 0 && a.err) atomicOr(a.err, kErrTimeout);
    return;
  }
  if (nvalid <= 1) return;

  // ---- split-KV: the last CTA of this column half merges every split
  __threadfence();
  __syncthreads();
  const int unit = b * 2 + int(c);
  if (tid == 0) {
    const uint32_t prev = atomicAdd(a.sems + unit, 1u);
    flags[1] = prev == uint32_t(nvalid - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!flags[1]) return;
  __threadfence();
  const float kv_scale = ldscale(a.kv_scale_dev, a.kv_scale);
  constexpr int kStride = kLatent + 4;
  const float* ws_b = a.ws + int64_t(b) * a.nsplit * kRows * kStride;
  // phase 1: one thread per row folds the split maxima, the sink and the
  // output scales into one weight per (row, split), staged in shared memory
  float* wts = reinterpret_cast<float*>(smem);  // [kRows][nvalid]
  if (tid < kRows) {
    const int row = tid;
    float M = -INFINITY;
    for (int sp = 0; sp < nvalid; ++sp)
      M = fmaxf(M, __ldcg(ws_b + (int64_t(sp) * kRows + row) * kStride + kLatent + 2 * c));
    float l = 0.f;
    for (int sp = 0; sp < nvalid; ++sp) {
      const float* src = ws_b + (int64_t(sp) * kRows + row) * kStride + kLatent + 2 * c;
      const float ms = __ldcg(src);
      const float f = ms == -INFINITY ? 0.f : exp2f(ms - M);
      wts[row * nvalid + sp] = f;
      l += f * __ldcg(src + 1);
    }
    const float sig = a.sinks ? __ldg(a.sinks + row % a.Hq) * kLog2e : -INFINITY;
    const int64_t row_g = (int64_t(b) * a.qs + row / a.Hq) * a.Hq + row % a.Hq;
    const float mul = finalize_row(M, l, sig, kv_scale * a.rcp_out_scale,
                                   (a.lse && c == 0) ? a.lse + row_g : nullptr);
    for (int sp = 0; sp < nvalid; ++sp) wts[row * nvalid + sp] *= mul;
  }
  __syncthreads();
  // phase 2: every (row, 4-column group) sums the weighted partials
  for (int item = tid; item < kRows * (kHalf / 4); item += kThreads) {
    const int row = item / (kHalf / 4);
    const int col = int(c) * kHalf + 4 * (item % (kHalf / 4));
    const float* w = wts + row * nvalid;
    const float* src = ws_b + int64_t(row) * kStride + col;
    const int64_t sstride = int64_t(kRows) * kStride;
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
    const int ii = row / a.Hq, hh = row % a.Hq;
    const int64_t oi = ((int64_t(b) * a.qs + ii) * a.Hq + hh) * kLatent + col;
    *reinterpret_cast<uint2*>(a.out + oi) =
        make_uint2(pack_f32x2(acc.x, acc.y, true), pack_f32x2(acc.z, acc.w, true));
  }
  if (tid == 0) a.sems[unit] = 0u;
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct Plan {
  int nsplit = 1, split_pages = 1;
  size_t ws_bytes = 0, nsems = 0;
};

const char* check_shape(const xqa_params* p, int v_head_dim) {
  if (p->num_kv_heads != 1) return "the MLA variant has one latent kv head (num_kv_heads must be 1)";
  if (p->head_dim != kDim || v_head_dim != kLatent)
    return "the MLA kernel is built for a 576-wide latent row (512 latent + 64 rope) with v_head_dim 512";
  if (p->num_q_heads * p->q_seq_len != kRows)
    return "the MLA kernel needs num_q_heads * q_seq_len == 128 (one UMMA tile of query rows)";
  if (p->q_dtype != XQA_BF16 || p->kv_dtype != XQA_BF16)
    return "the MLA kernel is built for bf16 query and latent cache";
  if (p->kv_layout != XQA_NHD && p->kv_layout != XQA_HND) return "bad kv_layout";
  return nullptr;
}

int sm_count_of(const xqa_params* p, int sm_count) {
  if (sm_count > 0) return sm_count;
  if (p->sm_count > 0) return p->sm_count;
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

bool plan(const xqa_params* p, int sm_count, Plan* pl) {
  int max_pages = p->pages_per_seq;
  if (p->sliding_win_size > 0) {
    const int64_t span = int64_t(p->sliding_win_size) + p->q_seq_len - 1;
    max_pages = int(std::min<int64_t>(max_pages, (span + p->page_size - 1) / p->page_size + 1));
  }
  const int sm = sm_count_of(p, sm_count);
  if (sm <= 0) return false;
  const int stage_pages = p->page_size <= kTok ? kTok / p->page_size : 1;
  // one cluster (2 CTAs, one per SM) per (sequence, split); aim for ~8 waves
  const int64_t pairs = int64_t(sm / 2) * 8;
  int64_t ns = (pairs + p->batch_size - 1) / p->batch_size;
  const int64_t by_tiles = (max_pages + stage_pages - 1) / stage_pages;
  const int64_t by_tokens = std::max<int64_t>(1, int64_t(max_pages) * p->page_size / 1024);
  ns = std::max<int64_t>(1, std::min(ns, std::min(by_tiles, by_tokens)));
  ns = std::min<int64_t>(ns, kMaxSplits);
  int sp = int((max_pages + ns - 1) / ns);
  sp = ((sp + stage_pages - 1) / stage_pages) * stage_pages;
  pl->split_pages = sp;
  pl->nsplit = (max_pages + sp - 1) / sp;
  pl->nsems = size_t(p->batch_size) * 2;
  pl->ws_bytes = pl->nsplit > 1 ? size_t(p->batch_size) * pl->nsplit * kRows * (kLatent + 4) * sizeof(float) : 0;
  return true;
}

}  // namespace mla

size_t mla_workspace_size(const xqa_params* p, int v_head_dim, int sm_count) {
  if (!p || mla::check_shape(p, v_head_dim)) return size_t(-1);
  mla::Plan pl;
  if (!mla::plan(p, sm_count, &pl)) return size_t(-1);
  return pl.ws_bytes;
}

size_t mla_semaphore_count(const xqa_params* p, int v_head_dim) {
  if (!p || mla::check_shape(p, v_head_dim)) return size_t(-1);
  return size_t(p->batch_size) * 2;
}

xqa_status mla_decode(const xqa_params* p, int v_head_dim, void* ws, size_t ws_bytes, uint32_t* sems,
                      cudaStream_t stream, char* err, size_t err_len) {
  using namespace mla;
  if (const char* why = check_shape(p, v_head_dim)) {
    snprintf(err, err_len, "%s", why);
    return XQA_ERR_UNSUPPORTED;
  }
  if (p->q_seq_len > 32) {
    snprintf(err, err_len, "q_seq_len > 32 is not supported");
    return XQA_ERR_UNSUPPORTED;
  }
  if ((reinterpret_cast<uintptr_t>(p->q) | reinterpret_cast<uintptr_t>(p->output)) & 15) {
    snprintf(err, err_len, "q and output must be 16-byte aligned for the MLA kernel");
    return XQA_ERR_INVALID_ARG;
  }
  Plan pl;
  if (!plan(p, 0, &pl)) {
    snprintf(err, err_len, "cannot query the SM count of the current device");
    return XQA_ERR_CUDA;
  }
  if (pl.ws_bytes > 0) {
    if (!ws || ws_bytes < pl.ws_bytes) {
      snprintf(err, err_len, "workspace needs %zu bytes, got %zu", pl.ws_bytes, ws ? ws_bytes : size_t(0));
      return XQA_ERR_WORKSPACE_TOO_SMALL;
    }
    if (!sems) {
      snprintf(err, err_len, "semaphores are required (%zu needed)", pl.nsems);
      return XQA_ERR_WORKSPACE_TOO_SMALL;
    }
    if (reinterpret_cast<uintptr_t>(ws) & 15) {
      snprintf(err, err_len, "workspace must be 16-byte aligned");
      return XQA_ERR_INVALID_ARG;
    }
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    snprintf(err, err_len, "cuTensorMapEncodeTiled is unavailable");
    return XQA_ERR_CUDA;
  }
  // NHD and HND coincide for one kv head: rows of 576 elements, token-major.
  CUtensorMap tm;
  cuuint64_t dims[3] = {cuuint64_t(kDim), 1, cuuint64_t(p->page_size) * cuuint64_t(p->num_pages)};
  cuuint64_t strides[2] = {cuuint64_t(kDim) * 2, cuuint64_t(kDim) * 2};
  cuuint32_t box[3] = {64, 1, cuuint32_t(std::min(p->page_size, kTok))};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p->k_cache), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(err, err_len, "cuTensorMapEncodeTiled failed (%d)", int(r));
    return XQA_ERR_CUDA;
  }
  MlaArgs a;
  memset(&a, 0, sizeof a);
  a.q = static_cast<const uint16_t*>(p->q);
  a.out = static_cast<uint16_t*>(p->output);
  a.page_table = p->page_table;
  a.seq_lens = p->seq_lens;
  a.sinks = p->sinks;
  a.mask = p->mask;
  a.q_scale_dev = p->q_scale_dev;
  a.kv_scale_dev = p->kv_scale_dev;
  a.ws = static_cast<float*>(ws);
  a.sems = sems;
  a.err = p->error_word;
  a.lse = p->lse;
  a.num_pages = p->num_pages;
  a.B = p->batch_size;
  a.Hq = p->num_q_heads;
  a.qs = p->q_seq_len;
  a.ps = p->page_size;
  a.pps = p->pages_per_seq;
  a.win = p->sliding_win_size;
  a.nsplit = pl.nsplit;
  a.split_pages = pl.split_pages;
  a.mask_words = ((p->q_seq_len + 31) / 32) * 2;
  a.q_scale = p->q_scale;
  a.kv_scale = p->kv_scale;
  a.softmax_scale = p->softmax_scale != 0.f ? p->softmax_scale : 1.0f / sqrtf(float(kDim));
  a.rcp_out_scale = p->rcp_out_scale;
  a.q_bf16 = 1;
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) {
    snprintf(err, err_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    return XQA_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pl.nsplit, 1, p->batch_size);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = p->enable_pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, mla_decode_kernel, tm, a);
  if (e != cudaSuccess) {
    snprintf(err, err_len, "MLA kernel launch: %s", cudaGetErrorString(e));
    return XQA_ERR_CUDA;
  }
  return XQA_OK;
}

}  // namespace xqa
