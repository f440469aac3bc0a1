// Grouped-query decode for large grouped tiles on the 5th-generation tensor
// cores (the XQA-style call of the FlashInfer "flashinfer.xqa.xqa" API page
// with q_seq_len x G > 16 query rows per kv head, e.g. speculative tokens on a
// large GQA group; 16-bit K/V).
//
// A unit is (sequence b, kv head kvh, row group rg, KV split).  Its rows
// (q_seq_len x G, up to 128, padded to one M = 128 UMMA tile with zero query
// rows that are never stored) are the A operand of S = Q K^T, held in tensor
// memory; every KV page is read once.  One CTA per unit, or (more unsplit
// units than CTA slots) one resident CTA per slot taking its units in turn:
// every role walks the same unit list, the barrier slots and phases run on
// across units, the next unit's query goes into tensor memory while the
// last one's epilogue reads O, and that unit's first P V waits for it.
//
//   warps 0 and 10 (producers of K and of V): walk page_table (32 page indices
//     per lane window) and issue a tile's TMA boxes, one per (page piece,
//     128-byte chunk), from as many lanes, into rings of 128-token K and V
//     tiles.  A K tile is freed by its Q K^T, a V tile by its P V, so the K
//     loads run ahead of the softmax.
//   warp 1 (one thread): S(j) = Q K(j)^T with N = 128 (D / 16 MMAs) into one
//     of two S buffers in tensor memory, then O += P(j - 1) V(j - 1) with
//     N = D into the O columns; commits free the tiles and the P buffer.
//   warps 2-9 (softmax, two threads per query row = tensor-memory lane, each
//     with half of the tile's tokens and half of O's columns): read S out of
//     tensor memory, scale / window / spec-mask / tail by select, run
//     the online softmax in the exp2 domain (O rescaled in place, only when a
//     row's maximum grew by more than 2^8, after the previous P V is done),
//     write P (16-bit, UMMA operand layout) and zero V rows past the split's
//     end; then the epilogue: O from tensor memory, normalised (sinks, scales)
//     or written as a split partial that the last CTA of the unit merges
//     (the log-sum-exp merge of merge_attn_states).
#include <cuda.h>
#include <cuda_runtime.h>
#include <string.h>

#include "finalize.cuh"
#include "kernel_args.h"
#include "ptx.cuh"
#include "umma.cuh"
#include "xqa.h"

namespace xqa {
namespace tc {

constexpr int kRows = 128;       // UMMA M: the CTA's query rows, padded
constexpr int kT = 128;          // tokens per tile (UMMA N of Q K^T, K of P V)
constexpr int kSoftWarp0 = 2;    // warps 2..9: two threads per query row
constexpr int kSoftWarps = 8;
constexpr int kSoft = 32 * kSoftWarps;
constexpr int kVWarp = kSoftWarp0 + kSoftWarps;  // the V producer
constexpr int kThreads = 32 * (kVWarp + 1);
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;    // 2 x 128 columns of logits
constexpr uint32_t kColO = 256;  // D fp32 columns of O
constexpr uint32_t kColQ = 384;  // D / 2 columns, the query as 16-bit pairs
constexpr float kRescaleLog2 = 8.f;  // rescale O only when the max grows by > 2^8

__device__ __forceinline__ float load_scale_tc(const float* dev, float host) { return dev ? __ldg(dev) : host; }

template <int D>
struct Cfg {
  static constexpr int kChunks = D / 64;             // 128-byte chunks of a K / V row
  static constexpr int kTileBytes = kT * D * 2;      // K (or V) of one tile: [chunk][128 rows][128 B]
  static constexpr int kKStages = D == 128 ? 3 : 4;
  static constexpr int kVStages = D == 128 ? 2 : 4;
  static constexpr int kPBytes = kRows * kT * 2;     // P of one tile: [64-token chunk][128 rows][128 B]
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKStages * kTileBytes;
  static constexpr int kOffP = kOffV + kVStages * kTileBytes;
  static constexpr int kOffRowX = kOffP + 2 * kPBytes;  // [2][128] row maxima / sums of the halves
  static constexpr int kOffOrd = kOffRowX + 2 * kRows * 4;  // [160] the sequences, longest first
  static constexpr int kOffBar = kOffOrd + 160 * 4;
  enum {
    kKFull = 0,                     // [kKStages] a K tile landed
    kKEmpty = kKFull + kKStages,    // [kKStages] the Q K^T reading it is done
    kVFull = kKEmpty + kKStages,    // [kVStages] a V tile landed
    kVEmpty = kVFull + kVStages,    // [kVStages] the P V reading it is done
    kSFull = kVEmpty + kVStages,    // [2] S(j) computed
    kSFree = kSFull + 2,            // [2] S(j) read out of tensor memory (8 warps)
    kPFull = kSFree + 2,            // [2] P(j) written, O rescaled, V tail zeroed (8 warps)
    kPVDone = kPFull + 2,           // [2] P(j) V(j) done
    kQReady = kPVDone + 2,          // a unit's query is in tensor memory (8 warps)
    kOFree = kQReady + 1,           // a unit's O was read out of tensor memory (8 warps)
    kDrain = kOFree + 1,            // every MMA is done
    kNumBars = kDrain + 1
  };
  static constexpr int kSmem = kOffBar + kNumBars * 8 + 16;
  static_assert(kSmem <= 232448 - 1024, "shared memory (with room to align the base)");
};

// Zeroes V rows [r0, kT) of a stage's V tile ([chunk][128 rows][128 B]): past a
// split's end the rows hold stale or foreign data (possibly NaN) that P = 0
// must not meet.  Threads st = 0..kSoft-1.
template <int D>
__device__ __forceinline__ void zero_v_rows(uint8_t* vtile, int r0, int st) {
  for (int idx = st; idx < (kT - r0) * 8 * Cfg<D>::kChunks; idx += kSoft) {
    const int u = idx & 7, rc = idx >> 3;
    const int r = r0 + rc / Cfg<D>::kChunks, c = rc % Cfg<D>::kChunks;
    *reinterpret_cast<uint4*>(vtile + c * kT * 128 + r * 128 + u * 16) = make_uint4(0, 0, 0, 0);
  }
}

// One unit of work: (sequence b, kv head kvh, row group rg, KV split) and
// the stretch of its tokens that the split covers.
struct Unit {
  int b, kvh, rg, split;
  int L, spec0, pg_hi, t_begin, t_end, ntiles, nvalid, rows_here;
};

// Unit k of this CTA; false past its last.  One CTA per unit (grid = splits x
// (kv heads x row groups) x sequences, slot z taking the sequence of rank z),
// or persistent CTAs (a.persist of them): CTA c takes the units of rank
// k G + c for even k and k G + G - 1 - c for odd k (G CTAs; units ranked by
// their sequence's length, longest first, then kv head and row group), so
// that the long and the short units even out across the CTAs.
__device__ __forceinline__ bool unit_at(const DecodeArgs& a, const int* ord, int k, Unit& u) {
  if (a.persist == 0) {
    if (k > 0) return false;
    u.split = blockIdx.x;
    u.kvh = blockIdx.y / a.rg_count;
    u.rg = blockIdx.y % a.rg_count;
    u.b = a.sort_b ? ord[blockIdx.z] : int(blockIdx.z);
  } else {
    const int G = int(gridDim.z), c = int(blockIdx.z);
    const int r = k * G + ((k & 1) ? G - 1 - c : c);
    const int per_seq = a.Hkv * a.rg_count;
    if (r >= a.B * per_seq) return false;
    u.b = ord[r / per_seq];
    const int rem = r % per_seq;
    u.kvh = rem / a.rg_count;
    u.rg = rem % a.rg_count;
    u.split = 0;
  }
  const int64_t max_len = int64_t(a.pps) * a.ps;
  const int64_t len_raw = a.seq_lens[u.b];
  u.L = int(len_raw < max_len ? len_raw : max_len);
  u.spec0 = u.L - a.qs;
  const int t_lo_all = a.win > 0 ? max(0, u.spec0 - a.win + 1) : 0;
  const int pg_first = t_lo_all / a.ps;
  const int pg_last = (u.L + a.ps - 1) / a.ps;
  const int npages = max(0, pg_last - pg_first);
  u.nvalid = (npages + a.split_pages - 1) / a.split_pages;
  const int pg_lo = pg_first + u.split * a.split_pages;
  u.pg_hi = min(pg_lo + a.split_pages, pg_last);
  u.t_begin = pg_lo * a.ps;
  u.t_end = min(u.pg_hi * a.ps, u.L);
  u.ntiles = (u.nvalid == 0 || u.t_end <= u.t_begin || u.split >= u.nvalid) ? 0 : (u.t_end - u.t_begin + kT - 1) / kT;
  u.rows_here = min(kRows, a.R - u.rg * kRows);
  return true;
}

template <bool kBf16, int D>
__global__ void __launch_bounds__(kThreads, 1)
    gqa_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeArgs a) {
  using C = Cfg<D>;
  constexpr unsigned kAll = 0xffffffffu;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);  // [0] abort, [1] last CTA

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int* ord = reinterpret_cast<int*>(smem + C::kOffOrd);
  pdl_wait();
  pdl_launch_dependents();

  // Longest sequences first: ord[z] is the sequence with the z-th most
  // visible tokens (ties by index).  With one CTA per unit, CTAs launch in
  // blockIdx order and grid slot z takes sequence ord[z], so the long CTAs
  // start in the first wave instead of trailing the last one; persistent
  // CTAs rank their units through it.  Every CTA ranks the (at most 160)
  // sequences itself (the K ring, unused until the first load, holds the
  // lengths).
  if (a.sort_b) {
    int* eff = reinterpret_cast<int*>(smem + C::kOffK);
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
      ord[rank] = tid;
    }
    __syncthreads();  // (read before anything else uses the ring)
  }

  // lengths past the page table's bound are clamped (and reported once)
  if (a.err && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
    for (int bb = tid; bb < a.B; bb += kThreads)
      if (int64_t(a.seq_lens[bb]) > int64_t(a.pps) * a.ps) atomicOr(a.err, kErrClamped);

  // a CTA past its unit's last split has nothing to do
  Unit u0;
  if (!unit_at(a, ord, 0, u0)) return;
  if (a.persist == 0 && u0.split >= max(u0.nvalid, 1)) return;

  if (tid == 0) {
    for (int s = 0; s < C::kKStages; ++s) {
      mbar_init(&bars[C::kKFull + s], 1);
      mbar_init(&bars[C::kKEmpty + s], 1);
    }
    for (int s = 0; s < C::kVStages; ++s) {
      mbar_init(&bars[C::kVFull + s], 1);
      mbar_init(&bars[C::kVEmpty + s], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&bars[C::kSFull + k], 1);
      mbar_init(&bars[C::kSFree + k], kSoftWarps);
      mbar_init(&bars[C::kPFull + k], kSoftWarps);
      mbar_init(&bars[C::kPVDone + k], 1);
    }
    mbar_init(&bars[C::kQReady], kSoftWarps);
    mbar_init(&bars[C::kOFree], kSoftWarps);
    mbar_init(&bars[C::kDrain], 1);
    flags[0] = flags[1] = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    umma::tmem_alloc(tmem_slot, kTmemCols);
    umma::tmem_relinquish();
  }
  umma::fence_before_sync();
  __syncthreads();
  umma::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  constexpr uint32_t kIdescQK = umma::idesc_f16(kRows, kT, kBf16, false, false);
  constexpr uint32_t kIdescPV = umma::idesc_f16(kRows, D, kBf16, false, true);

  if (warp == 0 || warp == kVWarp) {
    // ================= TMA producers: K (warp 0), V (warp 6) =================
    const bool is_v = warp == kVWarp;
    const int nst = is_v ? C::kVStages : C::kKStages;
    uint64_t* full = &bars[is_v ? C::kVFull : C::kKFull];
    uint64_t* empty = &bars[is_v ? C::kVEmpty : C::kKEmpty];
    const CUtensorMap* map = is_v ? &tmV : &tmK;
    uint8_t* ring = smem + (is_v ? C::kOffV : C::kOffK);
    const volatile int* vflags = flags;
    if (lane == 0) prefetch_tensormap(map);
    const int box_rows = min(a.ps, 64);
    const int pieces_max = kT / box_rows;  // page pieces of a full tile
    bool ok = true, bad = false;
    int g = 0;  // tiles issued, over all of this CTA's units (ring slot and phase)
    Unit u = u0;
    for (int k = 0; ok; ++k) {
      if (k > 0 && (vflags[0] || !unit_at(a, ord, k, u))) break;
      const int32_t* pt = a.page_table + int64_t(u.b) * a.pps;
      // lane l issues box l of the tile: page piece l / chunks, chunk l % chunks
      int win_base = -(1 << 30), my_page = 0;
      for (int j = 0; ok && j < u.ntiles; ++j, ++g) {
        const int s = g % nst, use = g / nst;
        if (use > 0) ok = __all_sync(kAll, mbar_wait(&empty[s], (use - 1) & 1));
        if (!ok) break;
        const int tok0 = u.t_begin + j * kT;
        const int n_piece = min(pieces_max, (u.pg_hi * a.ps - tok0 + box_rows - 1) / box_rows);
        const int first = tok0 / a.ps, last = (tok0 + n_piece * box_rows - 1) / a.ps;
        if (first < win_base || last >= win_base + 32) {  // refetch 32 page indices (warp-uniform)
          win_base = first;
          my_page = 0;
          if (win_base + lane < u.pg_hi) {
            const int pg = __ldg(pt + win_base + lane);
            my_page = (pg < 0 || int64_t(pg) >= a.num_pages) ? -1 : pg;  // out of the pool: TMA fills zeros
          }
        }
        const int l_piece = min(lane / C::kChunks, n_piece - 1);
        const int tk = tok0 + l_piece * box_rows;
        const int page = __shfl_sync(kAll, my_page, (tk / a.ps - win_base) & 31);
        if (lane == 0) mbar_arrive_expect_tx(&full[s], uint32_t(n_piece) * box_rows * 128u * C::kChunks);
        __syncwarp();
        if (lane < n_piece * C::kChunks) {
          bad |= page < 0;
          const int chunk = lane % C::kChunks;
          const int sub = tk % a.ps;
          uint8_t* dst = ring + s * C::kTileBytes + chunk * kT * 128 + l_piece * box_rows * 128;
          if (a.hnd)
            tma_load_3d(dst, map, &full[s], chunk * 64, sub, page * a.Hkv + u.kvh);
          else
            tma_load_3d(dst, map, &full[s], chunk * 64, u.kvh, page * a.ps + sub);
        }
        __syncwarp();
      }
    }
    bad = __any_sync(kAll, bad);
    if (lane == 0) {
      if (bad && a.err) atomicOr(a.err, kErrClamped);
      // no load of this CTA may land after it exits
      for (int j = max(0, g - nst); j < g; ++j)
        if (!mbar_wait(&full[j % nst], (j / nst) & 1)) ok = false;
      if (!ok) flags[0] = 1;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer (one thread) =================
    if (lane == 0) {
      const volatile int* vflags = flags;
      bool ok = true;
      const uint32_t k0 = smem_u32(smem + C::kOffK), v0 = smem_u32(smem + C::kOffV), p0 = smem_u32(smem + C::kOffP);
      int g = 0;   // tiles done, over all of this CTA's units (buffers and phases)
      int nq = 0;  // units with tiles done (the query's and O's barrier phases)
      bool any = false;  // an MMA was issued
      Unit u = u0;
      for (int k = 0; ok; ++k) {
        if (k > 0 && (vflags[0] || !unit_at(a, ord, k, u))) break;
        if (u.ntiles == 0) continue;
        ok = mbar_wait(&bars[C::kQReady], nq & 1);
        const int gb = g;
        // O += P(jj) V(jj) (tile jj of the unit): K = 128 tokens in steps of
        // 16; P chunks of 64 tokens 16 KB apart; V MN-major, 64-dim atoms
        // kT * 128 B apart, 8-token groups 1 KB apart.  The unit's first
        // P V overwrites O, once the previous unit's O has been read out.
        auto pv = [&](int jj) {
          const int gg = gb + jj;
          if (ok && jj == 0 && nq > 0) ok = mbar_wait(&bars[C::kOFree], (nq - 1) & 1);
          if (ok) ok = mbar_wait(&bars[C::kPFull + (gg & 1)], (gg >> 1) & 1);
          if (ok) ok = mbar_wait(&bars[C::kVFull + gg % C::kVStages], (gg / C::kVStages) & 1);
          if (!ok) return;
          umma::fence_after_sync();
          const uint32_t pa = p0 + (gg & 1) * C::kPBytes;
          const uint32_t va = v0 + (gg % C::kVStages) * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < kT / 16; ++kk)
            umma::mma_ss(tmem + kColO, umma::smem_desc(pa + (kk >> 2) * 16384 + 32 * (kk & 3), 16, 1024, umma::kSw128),
                         umma::smem_desc(va + 2048 * kk, kT * 128, 1024, umma::kSw128), kIdescPV, (jj | kk) != 0);
          umma::commit(&bars[C::kVEmpty + gg % C::kVStages]);
          umma::commit(&bars[C::kPVDone + (gg & 1)]);
        };
        for (int j = 0; ok && j < u.ntiles; ++j) {
          const int gg = gb + j, s = gg % C::kKStages;
          ok = mbar_wait(&bars[C::kKFull + s], (gg / C::kKStages) & 1);
          if (ok && gg >= 2) ok = mbar_wait(&bars[C::kSFree + (gg & 1)], ((gg >> 1) - 1) & 1);
          if (!ok) break;
          umma::fence_after_sync();
          any = true;
          // S(j) = Q K(j)^T: K = D in steps of 16 (32 bytes within a 128-byte chunk)
          const uint32_t ka = k0 + s * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            umma::mma_ts(tmem + kColS + 128u * uint32_t(gg & 1), tmem + kColQ + 8u * kk,
                         umma::smem_desc(ka + (kk >> 2) * (kT * 128) + 32 * (kk & 3), 16, 1024, umma::kSw128),
                         kIdescQK, kk != 0);
          umma::commit(&bars[C::kKEmpty + s]);
          umma::commit(&bars[C::kSFull + (gg & 1)]);
          if (j > 0) pv(j - 1);
        }
        if (ok) pv(u.ntiles - 1);
        g = gb + u.ntiles;
        ++nq;
      }
      if (!ok) flags[0] = 1;
      // nothing this thread issued may still run when tensor memory is read or freed
      if (any) {
        umma::commit(&bars[C::kDrain]);
        if (!mbar_wait(&bars[C::kDrain], 0)) flags[0] = 1;
      }
    }
    __syncwarp();
  } else {
    // ================= softmax: two threads per query row =================
    // Warp w (2..9) reaches tensor-memory lanes 32 (w % 4) .. +31 (query
    // rows); h = (w - 2) / 4 picks logit columns [64h, 64h + 64) of every
    // tile (its P chunk) and O columns [D/2 h, D/2 (h + 1)).
    const int q4 = warp & 3, h = (warp - kSoftWarp0) >> 2;
    const int t = 32 * q4 + lane;  // query row = tensor-memory lane
    const int st = tid - 32 * kSoftWarp0;  // 0 .. kSoft - 1
    const uint32_t lane_base = uint32_t(32 * q4) << 16;
    const float q_scale = load_scale_tc(a.q_scale_dev, a.q_scale);
    const float kv_scale = load_scale_tc(a.kv_scale_dev, a.kv_scale);
    const float lscale = a.softmax_scale * q_scale * kv_scale * kLog2e;
    float* rowx = reinterpret_cast<float*>(smem + C::kOffRowX);  // [2][128] the halves' row maxima
    constexpr int kC = kT / 2;  // logit columns per thread
    constexpr int kDh = D / 2;  // O columns per thread
    const volatile int* vflags = flags;
    bool ok = true;

    // ---- a unit's query rows into tensor memory: this thread's half of row t
    // (D / 2 values as D / 4 columns; zeros for padding rows)
    auto load_q = [&](const Unit& uq) {
      const int rq = uq.rg * kRows + t;
      const bool rl = t < uq.rows_here;
      const int iq = rl ? rq / a.G : a.qs - 1, gq = rl ? rq % a.G : 0;
      const uint16_t* qrow = static_cast<const uint16_t*>(a.q) +
                             ((int64_t(uq.b) * a.qs + iq) * a.Hq + int64_t(uq.kvh) * a.G + gq) * D + kDh * h;
      const uint4* src = reinterpret_cast<const uint4*>(qrow);
#pragma unroll
      for (int part = 0; part < kDh / 64; ++part) {
        uint32_t w[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = rl ? __ldg(src + part * 8 + v) : make_uint4(0, 0, 0, 0);
          w[4 * v + 0] = x.x;
          w[4 * v + 1] = x.y;
          w[4 * v + 2] = x.z;
          w[4 * v + 3] = x.w;
        }
        umma::tmem_st32(tmem + lane_base + kColQ + uint32_t(kDh / 2) * h + 32u * part, w);
      }
      if constexpr (kDh == 32) {  // D = 64: 32 values, 16 columns
        uint32_t w[16];
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          const uint4 x = rl ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
          w[4 * v + 0] = x.x;
          w[4 * v + 1] = x.y;
          w[4 * v + 2] = x.z;
          w[4 * v + 3] = x.w;
        }
        umma::tmem_st16(tmem + lane_base + kColQ + 16u * h, w);
      }
      umma::tmem_st_wait();
      umma::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::kQReady]);
    };

    // Unit by unit: the tiles' softmax; then the next unit's query (the last
    // Q K^T of this unit is done, so its columns are free, and the next
    // unit's first Q K^T overlaps this unit's epilogue); then the epilogue,
    // after which the next unit's first P V may overwrite O.  Barrier slots
    // and phases count tiles over all of the CTA's units (g).
    int g = 0;
    Unit u = u0;
    if (u.ntiles > 0) load_q(u);
    for (int k = 0;; ++k) {
      const int r = u.rg * kRows + t;  // row among the kv head's q_seq_len x G rows
      const bool real = t < u.rows_here;
      const int i = real ? r / a.G : a.qs - 1, gg = real ? r % a.G : 0;
      const int b = u.b, kvh = u.kvh, spec0 = u.spec0, t_begin = u.t_begin, t_end = u.t_end;
      const int row_lb = a.win > 0 ? spec0 + i - a.win + 1 : INT_MIN;
      uint32_t row_mw = 0xffffffffu;
      if (a.mask) {
        const uint16_t* mrow = a.mask + (int64_t(b) * a.qs + i) * a.mask_words;
        row_mw = uint32_t(__ldg(mrow)) | (uint32_t(__ldg(mrow + 1)) << 16);
      }
      // running maximum (log2 units, scale applied) and this half's sum
      float m_ref = -INFINITY, l_run = 0.f;
      const int gb = g;
      for (int j = 0; ok && j < u.ntiles; ++j) {
        const int gj = gb + j, sb = gj & 1;
        const int tile0 = t_begin + j * kT + kC * h;  // this thread's first token
        float x[kC];
        ok = __all_sync(kAll, mbar_wait(&bars[C::kSFull + sb], (gj >> 1) & 1));
        if (ok) {
          umma::fence_after_sync();
          umma::tmem_ld32(tmem + lane_base + kColS + 128u * sb + uint32_t(kC) * h, x);
          umma::tmem_ld32(tmem + lane_base + kColS + 128u * sb + uint32_t(kC) * h + 32u, x + 32);
          umma::tmem_ld_wait();
          umma::fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[C::kSFree + sb]);
        }
        // scale; window, spec mask and the split's end by select (never
        // multiply by 0); the maximum in four independent chains
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (ok) {
          const bool edge = tile0 + kC > t_end || tile0 <= row_lb || (a.mask && tile0 + kC > spec0);
          if (edge) {
#pragma unroll
            for (int c2 = 0; c2 < kC; ++c2) {
              const int tt = tile0 + c2;
              bool v = tt < t_end && tt >= row_lb;
              if (a.mask && tt >= spec0) v = v && ((row_mw >> (tt - spec0)) & 1u);
              x[c2] = v ? x[c2] * lscale : -INFINITY;
            }
          } else {
#pragma unroll
            for (int c2 = 0; c2 < kC; ++c2) x[c2] *= lscale;
          }
#pragma unroll
          for (int c2 = 0; c2 < kC; ++c2) mx4[c2 & 3] = fmaxf(mx4[c2 & 3], x[c2]);
          rowx[h * kRows + t] = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        }
        // both halves of every row published their maxima
        if (named_bar_or(1, kSoft, !ok)) {
          ok = false;
          break;
        }
        const float mx = fmaxf(rowx[t], rowx[kRows + t]);
        const float m_new = fmaxf(m_ref, mx);
        const bool need = m_new > m_ref + kRescaleLog2 || (m_ref == -INFINITY && m_new != -INFINITY);
        const float f = (need && m_ref != -INFINITY) ? exp2f(m_ref - m_new) : 1.f;
        if (need) {
          l_run *= f;
          m_ref = m_new;
        }
        // P buffer sb is free once P V of the tile two back is done
        if (gj >= 2) ok = __all_sync(kAll, mbar_wait(&bars[C::kPVDone + sb], ((gj >> 1) - 1) & 1));
        if (!ok) {
          named_bar_or(1, kSoft, true);  // (matched below: every half leaves together)
          break;
        }
        // P (16-bit, rounded; the row sum takes the rounded weights so O / l
        // stays a convex combination): this thread's 64 tokens are chunk h of
        // the [64-token chunk][128 rows][128 B] swizzled P tile
        uint8_t* prow = smem + C::kOffP + sb * C::kPBytes + h * 16384;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u8 = 0; u8 < kC / 8; ++u8) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float p0 = m_ref == -INFINITY ? 0.f : ex2(x[8 * u8 + 2 * e] - m_ref);
            const float p1 = m_ref == -INFINITY ? 0.f : ex2(x[8 * u8 + 2 * e + 1] - m_ref);
            w4[e] = pack_f32x2(p0, p1, kBf16);
            const float2 rr = unpack_16x2(w4[e], kBf16);
            ls[e] += rr.x + rr.y;
          }
          *reinterpret_cast<uint4*>(prow + umma::sw128(t, u8)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // O may change only once the previous tile's P V is done (whole
        // warps: the tensor-memory accesses are warp-collective); each half
        // scales its columns.  (f != 1 only past a unit's first tile.)
        if (__any_sync(kAll, f != 1.f)) {
          ok = __all_sync(kAll, mbar_wait(&bars[C::kPVDone + (sb ^ 1)], ((gj - 1) >> 1) & 1));
          if (ok) {
            umma::fence_after_sync();
#pragma unroll 1
            for (int q = 0; q < kDh / 16; ++q) {
              float o[16];
              umma::tmem_ld16(tmem + lane_base + kColO + uint32_t(kDh) * h + 16u * q, o);
              umma::tmem_ld_wait();
#pragma unroll
              for (int c2 = 0; c2 < 16; ++c2) o[c2] *= f;
              umma::tmem_st16(tmem + lane_base + kColO + uint32_t(kDh) * h + 16u * q,
                              reinterpret_cast<const uint32_t*>(o));
            }
            umma::tmem_st_wait();
          }
        }
        // a tile running past the split's end: its V rows past the end are zeroed
        const int vtile0 = t_begin + j * kT;
        if (ok && vtile0 + kT > t_end) {
          ok = __all_sync(kAll, mbar_wait(&bars[C::kVFull + gj % C::kVStages], (gj / C::kVStages) & 1));
          if (ok) zero_v_rows<D>(smem + C::kOffV + (gj % C::kVStages) * C::kTileBytes, t_end - vtile0, st);
        }
        if (named_bar_or(1, kSoft, !ok)) {
          ok = false;
          break;
        }
        umma::fence_proxy_async_smem();
        umma::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::kPFull + sb]);
      }
      g = gb + u.ntiles;
      // every half of every row takes the same decision on going on
      const bool stop = named_bar_or(1, kSoft, !ok || vflags[0] != 0);
      Unit nu;
      const bool has_next = !stop && unit_at(a, ord, k + 1, nu);
      if (has_next && nu.ntiles > 0) load_q(nu);
      // every P V of the unit is done (in order, so the last one's completion covers all)
      if (u.ntiles > 0 && ok) {
        ok = __all_sync(kAll, mbar_wait(&bars[C::kPVDone + ((g - 1) & 1)], ((g - 1) >> 1) & 1));
        umma::fence_after_sync();
      }
      if (!ok) flags[0] = 1;
      // the row's sum: both halves
      named_bar(1, kSoft);
      rowx[h * kRows + t] = l_run;
      named_bar(1, kSoft);
      const float l_row = rowx[t] + rowx[kRows + t];
      named_bar(1, kSoft);
      const bool aborted = vflags[0] != 0;
      const bool single = u.nvalid <= 1;
      const int unit = (b * a.Hkv + kvh) * a.rg_count + u.rg;
      float* ws_unit = a.ws + int64_t(unit) * a.nsplit * kRows * (D + 4);
      if (!aborted) {
        // ---- epilogue: this thread's half of O row t from tensor memory
        const float out_mul = kv_scale * a.rcp_out_scale;
        float mul = 1.f;
        if (single && real) {
          const float sig = a.sinks ? __ldg(a.sinks + kvh * a.G + gg) * kLog2e : -INFINITY;
          mul = finalize_row(m_ref, l_row, sig, out_mul,
                             (a.lse && h == 0) ? a.lse + lse_index(a, b, kvh, r) : nullptr);
        }
        float* wrow = ws_unit + (int64_t(u.split) * kRows + t) * (D + 4);
#pragma unroll 1
        for (int q = 0; q < kDh / 16; ++q) {
          float o[16];
          if (u.ntiles > 0) {
            umma::tmem_ld16(tmem + lane_base + kColO + uint32_t(kDh) * h + 16u * q, o);
            umma::tmem_ld_wait();
          } else {
#pragma unroll
            for (int c2 = 0; c2 < 16; ++c2) o[c2] = 0.f;
          }
          if (!real) continue;
          const int col = kDh * h + 16 * q;
          if (single) {
            const int64_t oi = ((int64_t(b) * a.qs + i) * a.Hq + int64_t(kvh) * a.G + gg) * a.Dv + col;
#pragma unroll
            for (int v = 0; v < 4; ++v)
              store_out4(a, oi + 4 * v, make_float4(o[4 * v] * mul, o[4 * v + 1] * mul, o[4 * v + 2] * mul,
                                                    o[4 * v + 3] * mul));
          } else {
#pragma unroll
            for (int v = 0; v < 4; ++v)
              reinterpret_cast<float4*>(wrow + col)[v] = make_float4(o[4 * v], o[4 * v + 1], o[4 * v + 2], o[4 * v + 3]);
          }
        }
        if (!single && real && h == 0) {
          wrow[D] = m_ref;
          wrow[D + 1] = l_row;
        }
      }
      // O has been read out: the next unit's first P V may overwrite it
      if (u.ntiles > 0) {
        umma::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::kOFree]);
      }
      if (!has_next) break;
      u = nu;
    }
  }

  // ---- teardown of tensor memory (every MMA is done or the call aborted)
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
  if (flags[0] && tid == 0 && a.err) atomicOr(a.err, kErrTimeout);
  // (persistent CTAs run unsplit units only)
  if (a.persist != 0 || u0.nvalid <= 1) return;
  const int nvalid = u0.nvalid, rows_here = u0.rows_here, b = u0.b, kvh = u0.kvh, rg = u0.rg;
  const int unit = (b * a.Hkv + kvh) * a.rg_count + rg;

  // ---- split-KV: the last CTA of the unit merges every split's partial (a
  // CTA whose wait gave up still takes its ticket, so the semaphore returns
  // to zero; the merge is skipped then)
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const uint32_t prev = atomicAdd(a.sems + unit, 1u);
    flags[1] = prev == uint32_t(nvalid - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!flags[1]) return;
  if (flags[0]) {
    if (tid == 0) a.sems[unit] = 0u;
    return;
  }
  __threadfence();
  const int row_stride = D + 4;
  float* ws_unit = a.ws + int64_t(unit) * a.nsplit * kRows * row_stride;
  const float kv_scale = load_scale_tc(a.kv_scale_dev, a.kv_scale);
  const float out_mul = kv_scale * a.rcp_out_scale;
  float* wts = reinterpret_cast<float*>(smem);  // [rows][nvalid] (the stage ring is free)
  for (int row = tid; row < rows_here; row += kThreads) {
    float M = -INFINITY;
    for (int sp = 0; sp < nvalid; ++sp)
      M = fmaxf(M, __ldcg(ws_unit + (int64_t(sp) * kRows + row) * row_stride + D));
    float l = 0.f;
    for (int sp = 0; sp < nvalid; ++sp) {
      const float* src = ws_unit + (int64_t(sp) * kRows + row) * row_stride + D;
      const float ms = __ldcg(src);
      const float f = (ms == -INFINITY) ? 0.f : exp2f(ms - M);
      wts[row * nvalid + sp] = f;
      l += f * __ldcg(src + 1);
    }
    const int rr = rg * kRows + row;
    const float sig = a.sinks ? __ldg(a.sinks + kvh * a.G + rr % a.G) * kLog2e : -INFINITY;
    const float mul = finalize_row(M, l, sig, out_mul, a.lse ? a.lse + lse_index(a, b, kvh, rr) : nullptr);
    for (int sp = 0; sp < nvalid; ++sp) wts[row * nvalid + sp] *= mul;
  }
  __syncthreads();
  const int64_t sstride = int64_t(kRows) * row_stride;
  for (int item = tid; item < rows_here * (D / 4); item += kThreads) {
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
    const int rr = rg * kRows + row;
    const int ii = rr / a.G, g2 = rr % a.G;
    store_out4(a, ((int64_t(b) * a.qs + ii) * a.Hq + int64_t(kvh) * a.G + g2) * a.Dv + dv, acc);
  }
  if (tid == 0) a.sems[unit] = 0u;
}

}  // namespace tc

// Launch (or, with launch == false, report the CTAs per SM of) the tensor-core
// grouped-query kernel for 16-bit K/V and head_dim 64 or 128.
cudaError_t gqa_tc_launch(bool bf16, int head_dim, bool launch, dim3 grid, const CUtensorMap* tk,
                          const CUtensorMap* tv, const DecodeArgs* args, cudaStream_t stream, int* ctas_per_sm) {
  const void* kern = nullptr;
  int smem = 0;
  if (bf16 && head_dim == 128) {
    kern = reinterpret_cast<const void*>(tc::gqa_tc_kernel<true, 128>);
    smem = tc::Cfg<128>::kSmem;
  } else if (bf16 && head_dim == 64) {
    kern = reinterpret_cast<const void*>(tc::gqa_tc_kernel<true, 64>);
    smem = tc::Cfg<64>::kSmem;
  } else if (!bf16 && head_dim == 128) {
    kern = reinterpret_cast<const void*>(tc::gqa_tc_kernel<false, 128>);
    smem = tc::Cfg<128>::kSmem;
  } else if (!bf16 && head_dim == 64) {
    kern = reinterpret_cast<const void*>(tc::gqa_tc_kernel<false, 64>);
    smem = tc::Cfg<64>::kSmem;
  } else {
    return cudaErrorInvalidValue;
  }
  smem += 1024;  // room to align the dynamic base to 1024 bytes
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (ctas_per_sm) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, kern, tc::kThreads, smem);
    if (e != cudaSuccess) return e;
  }
  if (!launch) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(tc::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = args->pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* kargs[] = {const_cast<CUtensorMap*>(tk), const_cast<CUtensorMap*>(tv), const_cast<DecodeArgs*>(args)};
  return cudaLaunchKernelExC(&cfg, kern, kargs);
}

}  // namespace xqa
