// MLA latent decode on the 5th-generation tensor cores (vLLM Kimi-K3
// MultiHeadLatentAttention page: the absorbed query [ql_nope | q_pe] of width
// kv_lora_rank + qk_rope_head_dim = 512 + 64 attends to one latent kv head of
// the same width through forward_mqa; V is the first kv_lora_rank = 512
// elements of each latent row; scale = qk_head_dim^-0.5 arrives as
// softmax_scale).
//
// The 128 query rows (heads x speculative tokens) form one M = 128 UMMA tile.
// Their fp32 output (128 x 512) alone fills a CTA's 512 tensor-memory
// columns, so a cluster of two CTAs shares each piece of a sequence and the
// two split the work by stage:
//
//   CTA 1 (the logit CTA) holds the whole query: the latent part in tensor
//   memory, the rope part in shared memory (bf16: the rows arrive in one TMA
//   box; the next piece's query loads while the previous piece's epilogue
//   runs).  It streams each 576-wide latent
//   row of the piece through a ring of three-chunk groups (128 tokens x 192
//   dims, TMA, 128-byte swizzle) and computes the logits S = Q K^T over
//   128-token tiles with tcgen05.mma, then runs the online softmax.  P (bf16,
//   already in UMMA operand layout) and one rescale factor per row travel into
//   CTA 0's shared memory by bulk copy, 64 tokens at a time.
//   CTA 0 (the output CTA) holds the whole fp32 output in tensor memory.  It
//   fetches the first 512 dims of each 64-token tile (V) again, from L2, and
//   accumulates O += P V with two N = 256 MMAs per 16 tokens.  Its eight spare
//   warps rescale O when the softmax raised a row maximum by more than 2^8,
//   clear V rows past the piece's end, and run the epilogue (O staged in
//   shared memory and stored by TMA).
//
// Only P crosses the cluster (16.5 KB per 64 tokens, one way), and every
// latent byte is read from HBM once.  Warp roles in both CTAs: 0 = TMA
// producer and tensor-memory allocator, 1 = MMA issuer, 2..9 = softmax
// (logit CTA) or rescale / epilogue (output CTA); warp w reaches TMEM lanes
// 32 (w % 4).., so two threads share each query row.
//
// Up to 256 sequences the clusters are persistent: cluster k runs, one after
// another, the pieces of the sequences that meet the k-th equal slice of the
// batch's pages (each sequence start charged a fixed piece cost), cut pieces
// first.  A sequence cut across clusters leaves one partial per piece, counted
// done on a per-sequence semaphore; a second kernel (mla_merge_kernel) merges
// each such sequence once its pieces are done.  Larger batches take one
// cluster per (sequence, fixed-size split), merged the same way.  In the bf16
// kernel the logit CTA starts a piece while the output CTA still writes the
// previous one out: it computes and stages the new piece's first tiles and
// sends them once the output CTA signals that its barriers are set up.
//
// The logit CTA is bound by its MMA instruction rate: an M = 128, N = 128,
// K = 16 tcgen05.mma accumulating into one tile takes ~140 cycles, and a
// 128-token logit tile is 36 of them.

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

constexpr int kRows = 128;       // UMMA M: query rows (heads x spec tokens), padded to 128
constexpr int kLatent = 512;     // kv_lora_rank (= V width)
constexpr int kRope = 64;        // qk_rope_head_dim
constexpr int kDim = kLatent + kRope;
constexpr int kHalf = kLatent / 2;  // output columns per epilogue thread and per merging CTA
constexpr int kTok = 64;         // tokens per P / V tile (UMMA K of PV)
constexpr int kTokQ = 2 * kTok;  // tokens per logit tile (UMMA N of QK)
constexpr int kChunkBytes = kTok * 128;    // one 128-byte column chunk of a V tile
constexpr int kChunkBytesQ = kTokQ * 128;  // one 128-byte column chunk of a logit tile
constexpr int kGroups = 3;       // K groups (ring slots) per logit tile
constexpr int kSoftWarps = 8;    // two threads per query row
constexpr int kSoft = 32 * kSoftWarps;
constexpr int kSoftWarp0 = 2;    // warps 2..9: two per TMEM sub-partition
constexpr int kThreads = 32 * kSoftWarp0 + kSoft;

// ---- messages from the logit CTA to the output CTA
constexpr int kPBytes = kRows * kTok * 2;  // one 16-bit P tile
constexpr int kFBytes = kRows * 4 + 16;    // one rescale factor per row, then a flag word
constexpr int kPMsg = kPBytes + kFBytes;
constexpr int kFinBytes = 2 * kRows * 4;   // the final row maxima and sums
// epilogue staging (in the output CTA's V ring and P slots, 224 KB): 28 KB per
// epilogue warp, 4 KB buffers of its 32 rows x 128 bytes (fp32 partial: 32
// columns, seven buffers; bf16 output: 64 columns, four buffers)
constexpr int kStageF32 = 7;
constexpr int kWarpStage = kStageF32 * 4096;
constexpr int kCopyPieces = 4;             // P travels as this many bulk copies

// ---- shared memory (offsets from the dynamic base, which is 1024-aligned:
// checked at run time), per element type of the latent cache.  The barrier
// block sits at the same offset in both CTAs because each CTA signals
// barriers of its peer.
// Tiles in shared memory are stored row group by row group: [8-row group]
// [128-byte column chunk][8 rows][128 bytes], so that one TMA box (a page
// piece's rows across several chunks) fills a contiguous run and every 8-row
// UMMA atom stays 1024-byte aligned.
//
// bf16 cache (a latent row is nine 64-dim chunks):
//   logit CTA: K ring of one logit tile, three slots of one 3-chunk group
//     (128 tokens x 192 dims, 48 KB) | rope query (128 x 64 bf16) | P staging x2
//     | factor staging x2 | row maxima [2 tiles][2 halves][128] | final rows
//   output CTA: V x3 (the 8 latent chunks of a 64-token tile, 64 KB) | P x2 |
//     factors x2 | final rows
// e4m3 cache (a latent row is four 128-dim chunks and a 64-byte rope part):
//   logit CTA: K ring of two logit tiles, each three slots: latent chunks 0-1,
//     latent chunks 2-3 (32 KB each) and the rope part (128 rows of 64 bytes,
//     64-byte swizzle, 8 KB) | rope query (128 x 64 e4m3, 64-byte swizzle) | the rest as bf16
//   output CTA: V x2 (e4m3, the 4 latent chunks of a 64-token tile, 32 KB) |
//     widened V x2 (f16, laid out as the bf16 V tile, 64 KB) | P x2 | factors x2 | final rows
template <bool F8>
struct Lay {
  static constexpr int kRingTiles = F8 ? 2 : 1;
  // The L2 prefetch of the latent rows is issued by the output CTA's
  // producer, this many 128-token tiles ahead of the V tile it loads (it
  // trails the logit CTA's loads by about a tile): a TMA instruction holds
  // its issuing thread for as long as the unit takes to generate the box's
  // requests, so the logit CTA's producer issues only its K loads.
  static constexpr int kPrefetchTilesOut = 2 * kRingTiles;
  static constexpr int kKSlots = kGroups * kRingTiles;
  static constexpr int kGroupChunks = F8 ? 2 : 3;       // 128-byte chunks per latent group
  static constexpr int kLatGroupBytes = kGroupChunks * kChunkBytesQ;
  static constexpr int kTileBytes = F8 ? 2 * kLatGroupBytes + kTokQ * 64 : 3 * kLatGroupBytes;
  // slot s of the ring (group s % 3 of a tile)
  __host__ __device__ static constexpr int slot_off(int s) {
    return (s / kGroups) * kTileBytes + (s % kGroups) * kLatGroupBytes;
  }
  __host__ __device__ static constexpr uint32_t slot_tx(int s, uint32_t rows) {  // bytes a slot receives
    return F8 && s % kGroups == 2 ? rows * 64u : rows * 128u * uint32_t(kGroupChunks);
  }
  static constexpr int kOffK = 0;
  static constexpr int kOffQRope = kOffK + kRingTiles * kTileBytes;
  static constexpr int kOffPS = kOffQRope + kRows * (F8 ? 64 : 128);
  static constexpr int kOffFS = kOffPS + 2 * kPBytes;
  static constexpr int kOffRowX = kOffFS + 2 * kFBytes;  // row maxima of the two threads of a row [2][128]
  static constexpr int kOffFinS = kOffRowX + 2 * kRows * 4;
  static constexpr int kLogitEnd = kOffFinS + kFinBytes;
  static constexpr int kVSlots = F8 ? 2 : 3;
  static constexpr int kVChunks = F8 ? 4 : 8;  // 128-byte chunks of a V tile row
  static constexpr int kVBytes = kVChunks * kChunkBytes;
  static constexpr int kHSlots = F8 ? 2 : 0;
  static constexpr int kHBytes = 8 * kChunkBytes;  // 512 f16 dims x 64 tokens
  static constexpr int kOffV = 0;
  static constexpr int kOffH = kOffV + kVSlots * kVBytes;
  static constexpr int kOffP = kOffH + kHSlots * kHBytes;
  static constexpr int kOffF = kOffP + 2 * kPBytes;
  static constexpr int kOffFin = kOffF + 2 * kFBytes;
  static constexpr int kOutEnd = kOffFin + kFinBytes;
  static constexpr int kOffBar = kLogitEnd > kOutEnd ? kLogitEnd : kOutEnd;
};

constexpr int kMaxKSlots = 6;
constexpr int kMaxVSlots = 3;
enum BarIdx {
  // logit CTA
  kKFull = 0,                      // [kKSlots] a group of K chunks landed
  kKEmpty = kKFull + kMaxKSlots,   // [kKSlots] the QK reading a group is done
  kSFull = kKEmpty + kMaxKSlots,   // [2] S tile computed
  kSFree = kSFull + 2,             // [2] S tile read out of tensor memory
  kQReady = kSFree + 2,            // the query is in tensor / shared memory
  kQLoad = kQReady + 1,            // bf16: the query's rows landed in the K ring (staging)
  kPSlotFree = kQLoad + 1,         // [2] the output CTA's P.V of that P slot is done
  // output CTA
  kVFull = kPSlotFree + 2,         // [kVSlots] a V slot landed
  kVEmpty = kVFull + kMaxVSlots,   // [kVSlots] the P.V (bf16) or the widening (e4m3) read a V slot
  kPFull = kVEmpty + kMaxVSlots,   // [2] own expect-tx arrival + the peer's P message
  kFin = kPFull + 2,               // own expect-tx arrival + the peer's final rows
  kReq = kFin + 1,                 // the MMA thread posted a request (bf16) / drained (e4m3)
  kOReady = kReq + 1,              // the warps served it
  kODone = kOReady + 1,            // every P.V issued so far is done
  kHFull = kODone + 1,             // [2] e4m3: the warps widened a V tile into an f16 slot
  kHEmpty = kHFull + 2,            // [2] e4m3: the P.V reading an f16 slot is done
  kDec = kHEmpty + 2,              // [2] e4m3: the MMA thread's rescale decision for a tile
  // both
  kDrain = kDec + 2,               // every MMA this CTA issued is done
  kNumBars = kDrain + 1,
  // bf16 logit CTA, set up once per kernel (in the slot of an e4m3-only
  // barrier): the output CTA has set up its barriers for the next piece (one
  // arrival per piece)
  kPeerReady = kDec
};
template <bool F8>
constexpr int smem_bytes() {
  return Lay<F8>::kOffBar + kNumBars * 8 + 32;
}
template <bool F8>
constexpr bool layout_ok() {
  using SL = Lay<F8>;
  return smem_bytes<F8>() <= 232448 && SL::kOffP % 1024 == 0 && SL::kOffH % 1024 == 0 && SL::kOffQRope % 1024 == 0 &&
         SL::kOffPS % 1024 == 0 && SL::kTileBytes % 1024 == 0 && SL::kLatGroupBytes % 1024 == 0 &&
         SL::kOffF % 16 == 0 && SL::kOffFS % 16 == 0 && SL::kOffFin % 16 == 0 && SL::kOffFinS % 16 == 0 &&
         SL::kOffBar % 8 == 0 && SL::kKSlots <= kMaxKSlots && SL::kVSlots <= kMaxVSlots;
}
static_assert(layout_ok<false>() && layout_ok<true>(),
              "shared memory budget; UMMA operands need 1024-byte alignment, bulk copies 16");
static_assert(kFBytes % 16 == 0 && kPBytes % (16 * kCopyPieces) == 0, "copy pieces");

// tensor memory columns
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 0;    // output CTA: 512 fp32 columns of O
constexpr uint32_t kColQ = 0;    // logit CTA: the latent query, 256 columns of bf16 pairs or 128 of e4m3 quads
constexpr uint32_t kColS = 256;  // logit CTA: 2 x 128 columns of logits

// requests from the output CTA's MMA thread to its warps
constexpr int kReqEnd = -1;
constexpr int kReqRescale = 1 << 30;  // multiply O rows by the tile's factors
constexpr int kReqTail = 1 << 29;     // zero the V rows past the split's end
constexpr int kReqTile = (1 << 29) - 1;

constexpr float kRescaleLog2 = 8.f;  // rescale O only when the max grows by > 2^8
constexpr int kOrderMaxB = 256;      // batches up to this size run on persistent clusters
constexpr int kMaxPieces = 128;      // persistent clusters (a sequence's pieces) at most
constexpr int kMaxSplits = 64;       // merge weights [128][splits] fit in shared memory
#ifndef XQA_MLA_WAVES
#define XQA_MLA_WAVES 3
#endif
constexpr int kWaves = XQA_MLA_WAVES;  // cluster waves the split plan aims for
#ifndef XQA_MLA_PIECE_TOKENS
#define XQA_MLA_PIECE_TOKENS 1024
#endif
// a persistent piece's fixed cost in KV tokens of streaming time: the
// pipeline fill and drain, the epilogue's stores and the barriers between
// pieces, all latency-bound while the other clusters stream the cache
// (measured on the latent workload: about 19 us, 1024 tokens)
constexpr int kPieceTokens = XQA_MLA_PIECE_TOKENS;

struct MlaArgs {
  const uint8_t* q;   // [B, qs, Hq, 576] bf16 or e4m3
  uint16_t* out;      // [B, qs, Hq, 512] bf16
  const int32_t* page_table;
  const uint32_t* seq_lens;
  const float* sinks;
  const uint16_t* mask;
  const float* q_scale_dev;
  const float* kv_scale_dev;
  float* ws;        // split partials: [slot][128 rows][512 + 4] fp32 (O, then m and l)
  uint32_t* sems;   // [2][B]: pieces of sequence b finished; its merge items done
  uint32_t* err;
  float* lse;  // optional [B, qs, Hq] natural-log log-sum-exp per row
  int64_t num_pages;
  int B, Hq, qs, ps, pps, win, nsplit, split_pages, mask_words;
  int R;    // real query rows Hq * qs (<= 128); rows R..127 of the tile are padding
  int ncl;  // persistent clusters
  int piece_cost;  // scheduled pages charged to each sequence start (a piece's fixed cost)
  float q_scale, kv_scale, softmax_scale, rcp_out_scale;
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
// Arrives once on the barrier at the same offset in every CTA of `mask` when
// every MMA this thread issued so far is done.
__device__ __forceinline__ void commit_to(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

// One arrival on a barrier of a peer CTA (its cluster address), ordered
// after this thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_peer(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

__device__ __forceinline__ float ldscale(const float* dev, float host) { return dev ? __ldg(dev) : host; }

// Multiplies this warp's 32 rows of O columns [256h, 256h + 256) by f.
__device__ __forceinline__ void rescale_o(uint32_t taddr, float f) {
#pragma unroll 1
  for (int part = 0; part < kHalf / 32; ++part) {
    float o[32];
    umma::tmem_ld32(taddr + 32u * part, o);
    umma::tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 32; ++k) o[k] *= f;
    umma::tmem_st32(taddr + 32u * part, reinterpret_cast<const uint32_t*>(o));
  }
  umma::tmem_st_wait();
}

// Zeroes V rows [r0, kTok) of a V slot's eight latent chunks ([row group]
// [chunk][8 rows][128 B]): past a split's last token the rows hold stale or
// foreign data (possibly NaN), and P = 0 there must not meet it in the P.V.
__device__ __forceinline__ void zero_v_tail(uint8_t* vslot, int r0, int st) {
  for (int idx = st; idx < (kTok - r0) * 8 * 8; idx += kSoft) {
    const int r = r0 + idx / 64, k = (idx / 8) % 8, u = idx % 8;
    *reinterpret_cast<uint4*>(vslot + ((r >> 3) * 8 + k) * 1024 + (r & 7) * 128 + u * 16) = make_uint4(0, 0, 0, 0);
  }
}

// Widens one e4m3 V tile (64 tokens x 512 dims, [row group][128-dim chunk][8
// rows][128 B], 128-byte swizzle) into the f16 V tile the P.V reads ([row
// group][64-dim chunk][8 rows][128 B], 128-byte swizzle); the cvt from e4m3 to
// f16 is exact.  Rows at or past `rows_valid` (past the split's end: stale,
// possibly NaN) are written as zeros.  Threads st = 0..kSoft-1.
__device__ __forceinline__ void widen_v(const uint8_t* v8, uint8_t* h16, int rows_valid, int st) {
#pragma unroll 4
  for (int idx = st; idx < kTok * 4 * 8; idx += kSoft) {
    const int u = idx & 7, r = (idx >> 3) & 7, c = (idx >> 6) & 3, rg = idx >> 8;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
    if (rg * 8 + r < rows_valid) {
      const uint4 x = *reinterpret_cast<const uint4*>(v8 + rg * 4096 + c * 1024 + r * 128 + ((u ^ r) << 4));
      e4m3x4_to_f16x2x2(x.x, lo.x, lo.y);
      e4m3x4_to_f16x2x2(x.y, lo.z, lo.w);
      e4m3x4_to_f16x2x2(x.z, hi.x, hi.y);
      e4m3x4_to_f16x2x2(x.w, hi.z, hi.w);
    }
    // dims 128c + 16u .. +15: units 2(u % 4) and 2(u % 4) + 1 of 64-dim chunk 2c + u / 4
    uint8_t* dst = h16 + rg * 8192 + (2 * c + (u >> 2)) * 1024 + r * 128;
    const int u2 = 2 * (u & 3);
    *reinterpret_cast<uint4*>(dst + ((u2 ^ r) << 4)) = lo;
    *reinterpret_cast<uint4*>(dst + (((u2 + 1) ^ r) << 4)) = hi;
  }
}

// One 4-D TMA box (row-group view of the latent rows) into shared memory.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// An L2 policy that keeps the lines it tags ahead of streamed data: a split
// partial is read back by the merge, up to a whole call later, while the
// other clusters stream the cache through L2.
__device__ __forceinline__ uint64_t l2_keep_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void st_keep4(float* dst, float x, float y, float z, float w, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst), "f"(x), "f"(y), "f"(z),
               "f"(w), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void st_keep2(float* dst, float x, float y, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(dst), "f"(x), "f"(y), "l"(pol) : "memory");
}
// One 2-D (3-D) TMA box from shared memory to global memory (a bulk
// async-group), optionally with an L2 cache policy.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
__device__ __forceinline__ void tma_store_2d_hint(const CUtensorMap* map, const void* src, int x, int y, uint64_t pol) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until every bulk group of this thread has completed (its global
// writes performed), then makes them visible device-wide.
__device__ __forceinline__ void bulk_wait_all_visible() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __threadfence();
}
// Bulk prefetch of `bytes` (a multiple of 16, 16-byte aligned) into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// The cluster whose slice of the persistent schedule holds scheduled page P
// (slice k = [tot * k / ncl, tot * (k + 1) / ncl)).
__device__ __forceinline__ int cluster_of(int64_t P, int64_t tot, int ncl) {
  int64_t k = P * ncl / tot;
  while (k + 1 < ncl && tot * (k + 1) / ncl <= P) ++k;
  while (k > 0 && tot * k / ncl > P) --k;
  return int(k);
}

// The pages sequence b's splits cover: a sliding window drops the pages
// before it; L is the length clamped to the page table's capacity.
struct SeqGeom {
  int L, pg_first, pg_last;
};
__device__ __forceinline__ SeqGeom seq_geom(const MlaArgs& a, int b) {
  const int64_t max_len = int64_t(a.pps) * a.ps;
  const int64_t len_raw = a.seq_lens[b];
  SeqGeom g;
  g.L = int(len_raw < max_len ? len_raw : max_len);
  const int t_lo_all = a.win > 0 ? max(0, g.L - a.qs - a.win + 1) : 0;
  g.pg_first = t_lo_all / a.ps;
  g.pg_last = (g.L + a.ps - 1) / a.ps;
  return g;
}

// Page indices of the piece a producer warp streams, 32 pages at a time in
// its registers: lane i holds the index of page base + i (-1 for an index
// outside the pool).  A tile's pieces then come from shuffles, and the page
// table is read once per 32 pages instead of on every tile, off the path
// from a freed ring slot to its next load.
struct PageWindow {
  int base = -(1 << 30), mine = 0;
  // Makes pages [first, last] (last < first + 32) available; whole warp.
  __device__ __forceinline__ void cover(const MlaArgs& a, const int32_t* pt, int first, int last, int pg_hi,
                                        int lane) {
    if (first >= base && last < base + 32) return;
    base = first;
    mine = 0;
    if (base + lane < pg_hi) {
      const int p = __ldg(pt + base + lane);
      mine = (p < 0 || int64_t(p) >= a.num_pages) ? -1 : p;
    }
  }
};

// The pieces of a tile of `tok` tokens starting at token tok0: boxes of
// min(page_size, 64) rows, piece l at tile row l * box.  Lane l < n loads
// piece l; `row` is its first row in the flattened [pages * page_size] row
// space (a negative row for a page index out of range: the TMA fills zeros
// there).  Pieces past the split's last page are not loaded.  Whole warp.
struct TilePieces {
  int n, row;
  bool bad;
};
__device__ __forceinline__ TilePieces tile_pieces(const MlaArgs& a, PageWindow& w, const int32_t* pt, int tok0,
                                                  int tok, int pg_hi, int lane) {
  TilePieces p;
  const int box = min(a.ps, kTok);
  const int split_end = pg_hi * a.ps;  // first token past the split's pages
  p.n = min(tok / box, (split_end - tok0 + box - 1) / box);
  p.bad = false;
  p.row = 0;
  if (p.n <= 0) return p;
  w.cover(a, pt, tok0 / a.ps, (tok0 + p.n * box - 1) / a.ps, pg_hi, lane);
  const int tk = tok0 + min(lane, p.n - 1) * box;
  const int page = __shfl_sync(0xffffffffu, w.mine, (tk / a.ps - w.base) & 31);
  if (lane < p.n) {
    p.bad = page < 0;
    p.row = page * a.ps + tk % a.ps;
  }
  return p;
}

template <bool F8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmKR,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmPF,
                      const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmWs,
                      const __grid_constant__ CUtensorMap tmO, const MlaArgs a) {
  using SL = Lay<F8>;
  // pieces overlap across the cluster (see the end of the piece loop)
  constexpr bool kDecoupled = !F8;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SL::kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + kNumBars);
  // [0] abort, [1] last CTA, [2] request word, [3] cluster abort, [4..5] rescale decisions (e4m3)
  int* flags = reinterpret_cast<int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t c = cluster_rank();
  const uint32_t peer = c ^ 1u;
  const bool logit_cta = c == 1;
  int split = blockIdx.x >> 1;
  int b = blockIdx.z;
  constexpr unsigned kAll = 0xffffffffu;

  // wait for the producer of our inputs, then let the next call start launching
  pdl_wait();
  pdl_launch_dependents();

  // the layout assumes a 1024-aligned dynamic base (the 128-byte swizzle
  // atoms of the UMMA operands); both CTAs see the same base and leave together
  if (smem_u32(smem_raw) & 1023u) {
    if (tid == 0 && a.err) atomicOr(a.err, kErrTimeout);
    return;
  }

  // ---- schedule.  Up to kOrderMaxB sequences the clusters are persistent:
  // cluster k takes the k-th of ncl equal slices of the batch's scheduled
  // pages laid end to end and runs the pieces of the sequences whose pages
  // meet its slice one after another.  A sequence schedules piece_cost
  // overhead pages and then its own pages (an empty sequence counts one page,
  // so that one cluster writes its output): a slice that starts more
  // sequences gets fewer pages, and a slice that covers only a sequence's
  // overhead takes no piece of it.  A sequence cut across clusters leaves one
  // fp32 partial per piece in workspace slot (cluster, 0) for the slice's
  // first sequence or (cluster, 1) for its last; the last CTA of each column
  // half to finish the sequence merges them.  A cluster runs its cut pieces
  // first (the slice's first sequence, then its last when that one runs on
  // past the slice), then the whole sequences between them: partials and
  // merges happen early, while the call's end is made of whole sequences.
  // Larger batches take one fixed split per cluster.
  const bool persistent = a.B <= kOrderMaxB;
  const int k_cl = int(blockIdx.x >> 1);
  int64_t tot = 1, s_lo = 0, s_hi = 0;  // all scheduled pages; this cluster's slice
  int ncl = a.ncl;                      // clusters with a non-empty slice
  int cur_b = b;                        // next sequence to look at (in order)
  int64_t cur_S = 0;                    // its first scheduled page
  int z_b = -1;                         // the slice's last sequence when it runs on past the slice
  int64_t z_S = 0;                      // (taken second), and its first scheduled page
  if (persistent) {
    int* sc = reinterpret_cast<int*>(smem);  // scratch: scheduled pages per sequence
    for (int bb = tid; bb < a.B; bb += kThreads) {
      const SeqGeom g = seq_geom(a, bb);
      sc[bb] = a.piece_cost + max(1, g.pg_last - g.pg_first);
    }
    __syncthreads();
    tot = 0;
    for (int bb = 0; bb < a.B; ++bb) tot += sc[bb];
    // fewer pages than clusters: the last clusters get no slice, every other
    // slice holds at least one page (so a sequence's pieces are exactly the
    // clusters from its first page's to its last page's)
    ncl = int(min(int64_t(a.ncl), tot));
    s_lo = k_cl < ncl ? tot * k_cl / ncl : tot;
    s_hi = k_cl < ncl ? tot * (k_cl + 1) / ncl : tot;
    cur_b = 0;
    while (cur_b < a.B && cur_S + sc[cur_b] <= s_lo) cur_S += sc[cur_b++];
    if (cur_b < a.B) {
      int bb = cur_b;
      int64_t S = cur_S;
      while (bb + 1 < a.B && S + sc[bb] + a.piece_cost < s_hi) S += sc[bb++];
      if (bb > cur_b && S + sc[bb] > s_hi) {
        z_b = bb;
        z_S = S;
      }
    }
    __syncthreads();  // the scratch is reused below
  }
  if (tid == 0) {
    flags[0] = flags[1] = flags[2] = flags[3] = 0;  // also for a cluster with no piece
    if (kDecoupled && logit_cta) {
      mbar_init(&bars[kPeerReady], 1);
      fence_mbar_init();
    }
  }
  if (warp == 0) {
    umma::tmem_alloc(tmem_slot, kTmemCols);
    umma::tmem_relinquish();
  }
  umma::fence_before_sync();
  __syncthreads();
  // bf16: the logit CTA's readiness barrier exists before the output CTA
  // signals it; from here on the two CTAs meet only through their barriers
  // (each sets up its own barriers for every piece, the output CTA then
  // signals the logit CTA, which sends nothing of the piece before that
  // signal) and once more before they exit
  if (kDecoupled) cluster_sync();
  umma::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t peer_bars = map_peer(smem_u32(bars), peer);
  const uint32_t box_rows = uint32_t(min(a.ps, kTok));
  // Q K^T: bf16 (kind::f16) or e4m3 (kind::f8f6f4); P V: bf16, or f16 when V is widened from e4m3
  constexpr uint32_t kIdescQK =
      F8 ? umma::idesc_e4m3(kRows, kTokQ, false, false) : umma::idesc_f16(kRows, kTokQ, true, false, false);
  constexpr uint32_t kIdescPV = umma::idesc_f16(kRows, kHalf, !F8, false, true);

  bool first_piece = true;
  int order = 0;      // pieces taken so far (persistent)
  int q_loaded = -1;  // logit CTA's softmax warps: the sequence whose query is in tensor memory
  int pend_b = -1;    // output CTA's first epilogue thread: the sequence whose partial is still being stored

  for (;;) {
  // ---- the piece: sequence b, pages [pg_lo, pg_hi), its index among the
  // sequence's nvalid pieces, and where its partial goes
  int nvalid, pg_lo, pg_hi, kf = 0;
  bool cl_first = true;  // the piece is its slice's first sequence (persistent)
  const bool z_now = persistent && order == 1 && z_b >= 0;  // the slice's last sequence, out of order
  int64_t S_b = 0;                                          // the sequence's first scheduled page
  if (persistent) {
    if (z_now) {
      b = z_b;
      S_b = z_S;
    } else {
      if (cur_b >= a.B || cur_S + a.piece_cost >= s_hi || cur_b == z_b) break;
      b = cur_b;
      S_b = cur_S;
    }
  }
  // ---- sequence geometry (identical in both CTAs and every split)
  const SeqGeom geo = seq_geom(a, b);
  const int L = geo.L;
  if (int64_t(a.seq_lens[b]) > int64_t(a.pps) * a.ps && a.err && tid == 0 && split == 0 && c == 0)
    atomicOr(a.err, kErrClamped);
  const int spec0 = L - a.qs;
  const int pg_first = geo.pg_first;
  const int pg_last = geo.pg_last;
  const int npages = max(0, pg_last - pg_first);
  const int nsched = max(1, npages);  // scheduled pages (persistent)
  if (persistent) {
    const int64_t S0 = S_b + a.piece_cost;  // the sequence's first own page
    const int64_t v_lo = max(s_lo, S0) - S0, v_hi = min(s_hi, S0 + nsched) - S0;
    pg_lo = pg_first + int(min(v_lo, int64_t(npages)));
    pg_hi = pg_first + int(min(v_hi, int64_t(npages)));
    kf = cluster_of(S0, tot, ncl);
    const int kl = cluster_of(S0 + nsched - 1, tot, ncl);
    nvalid = npages == 0 ? 0 : kl - kf + 1;
    split = k_cl - kf;
    cl_first = S0 <= s_lo;
  } else {
    nvalid = (npages + a.split_pages - 1) / a.split_pages;
    if (split >= max(nvalid, 1)) break;  // both CTAs of the cluster leave together
    pg_lo = pg_first + split * a.split_pages;
    pg_hi = min(pg_lo + a.split_pages, pg_last);
  }
  const int t_begin = pg_lo * a.ps;
  const int t_end = min(pg_hi * a.ps, L);
  const int ntiles = (nvalid == 0 || t_end <= t_begin) ? 0 : (t_end - t_begin + kTok - 1) / kTok;
  const int nqt = (ntiles + 1) / 2;  // logit tiles of 128 tokens
  // barriers are set up afresh for every piece (after the previous piece's
  // last wait, both CTAs having passed the cluster barrier that ends it)
  if (tid == 0) {
    // the barriers this CTA uses, with their arrival counts
    auto each_bar = [&](auto&& fn) {
      if (logit_cta) {
        for (int i = 0; i < SL::kKSlots; ++i) {
          fn(kKFull + i, 1);
          fn(kKEmpty + i, 1);
        }
        for (int k = 0; k < 2; ++k) {
          fn(kSFull + k, 1);
          fn(kSFree + k, kSoftWarps);
          fn(kPSlotFree + k, 1);  // the peer's MMA completion
        }
        fn(kQReady, kSoftWarps);
        fn(kQLoad, 1);
      } else {
        // an e4m3 V slot is freed by the eight warps that widen it, a bf16 one by the P.V
        for (int k = 0; k < SL::kVSlots; ++k) {
          fn(kVFull + k, 1);
          fn(kVEmpty + k, F8 ? kSoftWarps : 1);
        }
        for (int k = 0; k < 2; ++k) fn(kPFull + k, 1);
        fn(kFin, 1);
        fn(kReq, 1);
        fn(kOReady, kSoftWarps);
        fn(kODone, 1);
        if (F8)
          for (int k = 0; k < 2; ++k) {
            fn(kHFull + k, kSoftWarps);
            fn(kHEmpty + k, 1);
            fn(kDec + k, 1);
          }
      }
      fn(kDrain, 1);
    };
    if (!first_piece) each_bar([&](int i, int) { mbar_inval(&bars[i]); });
    each_bar([&](int i, int n) { mbar_init(&bars[i], uint32_t(n)); });
    if (!logit_cta) {
      // the first two P messages and the final rows are expected up front
      for (int k = 0; k < min(2, ntiles); ++k) mbar_arrive_expect_tx(&bars[kPFull + k], kPMsg);
      mbar_arrive_expect_tx(&bars[kFin], kFinBytes);
    }
    flags[0] = flags[1] = flags[2] = 0;
    fence_mbar_init();
    // the logit CTA may send this piece's messages now
    if (kDecoupled && !logit_cta) mbar_arrive_peer(map_peer(smem_u32(&bars[kPeerReady]), peer));
  }
  umma::fence_before_sync();
  __syncthreads();
  if (!kDecoupled) cluster_sync();  // the peer's barriers exist before any remote access
  umma::fence_after_sync();
  const int32_t* pt = a.page_table + int64_t(b) * a.pps;
  // this cluster's next sequence (persistent), whose query the logit CTA's
  // producer prefetches into L2 once it has issued this piece's last K load:
  // the query load at a piece's start is latency-bound while the other
  // clusters stream the cache
  int next_b = -1;
  if (persistent) {
    if (z_b >= 0 && order == 0)
      next_b = z_b;
    else if (z_now)
      next_b = cur_b < z_b ? cur_b : -1;
    else if (b + 1 < a.B && b + 1 != z_b && S_b + 2 * a.piece_cost + nsched < s_hi)
      next_b = b + 1;
  }

  if (warp == 0) {
    // ================= TMA producer =================
    // Logit CTA: every group of every logit tile, in order, into the K ring;
    // a slot refills once the QK that read it is done.  Output CTA: the latent
    // chunks of each 64-token tile into a V slot once the P.V (bf16) or the
    // widening (e4m3) of the tile kVSlots back is done.  Each wait gives up
    // after kWaitCycles.
    if (ntiles > 0) {
      if (lane == 0) {
        prefetch_tensormap(logit_cta ? &tmK : &tmV);
        prefetch_tensormap(&tmPF);
        if (logit_cta && F8) prefetch_tensormap(&tmKR);
      }
      bool ok = true, bad = false;
      int issued = 0;
      PageWindow win, win_pf;  // the tiles' pages; the L2-prefetched tiles' pages
      if (logit_cta) {
        // group gr of logit tile j (global group g = 3 j + gr) goes to ring
        // slot g % kKSlots: one wait, one expect-tx and one box per page piece
        TilePieces tp = {0, 0, false};
        // the query's loads go first (at the call's start every cluster loads
        // one at once; a piece after the first finds it loaded already)
        if (nqt > 0) ok = __all_sync(kAll, mbar_wait(&bars[kQReady], 0));
        for (int g = 0; ok && g < nqt * kGroups; ++g) {
          const int j = g / kGroups, gr = g - j * kGroups;
          const int slot = g % SL::kKSlots, use = g / SL::kKSlots;
          if (gr == 0) {
            tp = tile_pieces(a, win, pt, t_begin + j * kTokQ, kTokQ, pg_hi, lane);
            bad |= tp.bad;
          }
          if (use > 0) ok = __all_sync(kAll, mbar_wait(&bars[kKEmpty + slot], (use - 1) & 1));
          if (!ok) break;
          const uint32_t piece_bytes = SL::slot_tx(slot, box_rows);
          if (lane == 0) mbar_arrive_expect_tx(&bars[kKFull + slot], uint32_t(tp.n) * piece_bytes);
          __syncwarp();
          // one box per page piece (its rows across the group's chunks, or the
          // e4m3 rope part), one piece per lane: issuing a TMA instruction
          // holds its thread for hundreds of cycles
          if (lane < tp.n) {
            uint8_t* dst = smem + SL::kOffK + SL::slot_off(slot) + lane * int(piece_bytes);
            if (F8 && gr == 2)
              tma_load_3d(dst, &tmKR, &bars[kKFull + slot], 0, 0, tp.row >> 3);
            else
              tma_load_4d(dst, &tmK, &bars[kKFull + slot], 0, 0, SL::kGroupChunks * gr, tp.row >> 3);
          }
          __syncwarp();
          ++issued;
        }
        if (lane == 0 && next_b >= 0) {
          const int64_t qbytes = int64_t(a.qs) * a.Hq * kDim * (F8 ? 1 : 2);
          prefetch_l2_bulk(a.q + int64_t(next_b) * qbytes, uint32_t(qbytes));
        }
        // no load of this CTA may land after it exits
        if (lane == 0)
          for (int g = max(0, issued - SL::kKSlots); g < issued; ++g)
            if (!mbar_wait(&bars[kKFull + g % SL::kKSlots], (g / SL::kKSlots) & 1)) ok = false;
      } else {
        const uint32_t piece_bytes = uint32_t(box_rows) * 128u * SL::kVChunks;
        for (int j = 0; ok && j < ntiles; ++j) {
          const int slot = j % SL::kVSlots, use = j / SL::kVSlots;
          if (use > 0) ok = __all_sync(kAll, mbar_wait(&bars[kVEmpty + slot], (use - 1) & 1));
          if (!ok) break;
          const TilePieces tp = tile_pieces(a, win, pt, t_begin + j * kTok, kTok, pg_hi, lane);
          bad |= tp.bad;
          if (lane == 0) mbar_arrive_expect_tx(&bars[kVFull + slot], uint32_t(tp.n) * piece_bytes);
          __syncwarp();
          // one box per page piece: its rows across the latent chunks
          if (lane < tp.n)
            tma_load_4d(smem + SL::kOffV + slot * SL::kVBytes + lane * int(piece_bytes), &tmV, &bars[kVFull + slot],
                        0, 0, 0, tp.row >> 3);
          __syncwarp();
          // at the start of each 128-token logit tile, the latent rows of the
          // logit tile kPrefetchTilesOut ahead go into L2, so that the logit
          // CTA's loads (issued only as its ring slots free) do not pay HBM
          // latency; one box per page piece covers all 576 dims of its rows
          if ((j & 1) == 0 && j / 2 + SL::kPrefetchTilesOut < nqt) {
            const TilePieces pf =
                tile_pieces(a, win_pf, pt, t_begin + (j / 2 + SL::kPrefetchTilesOut) * kTokQ, kTokQ, pg_hi, lane);
            if (lane < pf.n && pf.row >= 0) tma_prefetch_l2_3d(&tmPF, 0, 0, pf.row);
          }
          ++issued;
        }
        if (lane == 0)
          for (int j = max(0, issued - SL::kVSlots); j < issued; ++j)
            if (!mbar_wait(&bars[kVFull + j % SL::kVSlots], (j / SL::kVSlots) & 1)) ok = false;
      }
      bad = __any_sync(kAll, bad);
      if (lane == 0) {
        if (bad && a.err) atomicOr(a.err, kErrClamped);
        if (!ok) flags[0] = 1;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ================= MMA issuer (one thread) =================
    if (lane == 0 && ntiles > 0) {
      bool ok = true;
      if (logit_cta) {
        // S(j) = Q K(j)^T over a 128-token tile into S buffer j % 2, one ring
        // slot (group) at a time.  bf16: 32 N = 128 MMAs (K = 16) with the
        // latent query from tensor memory and 4 with the rope query from
        // shared memory; e4m3: 16 (K = 32, kind::f8f6f4) and 2 over the
        // 64-byte rope rows.  Any shared-memory read (a barrier test included)
        // issued between MMAs costs the issuing thread ~100 cycles, so the
        // waits come once per group, not per chunk.
        const uint32_t kb = smem_u32(smem + SL::kOffK), qrope = smem_u32(smem + SL::kOffQRope);
        ok = mbar_wait(&bars[kQReady], 0);
        for (int j = 0; ok && j < nqt; ++j) {
          const int sb = j & 1;
          if (j >= 2) ok = mbar_wait(&bars[kSFree + sb], ((j >> 1) - 1) & 1);
          const uint32_t sd = tmem + kColS + 128u * uint32_t(sb);
#pragma unroll
          for (int gr = 0; gr < kGroups; ++gr) {
            const int g = kGroups * j + gr, slot = g % SL::kKSlots;
            if (ok) ok = mbar_wait(&bars[kKFull + slot], (g / SL::kKSlots) & 1);
            if (!ok) break;
            umma::fence_after_sync();
            const uint32_t sbase = kb + SL::slot_off(slot);
            if constexpr (F8) {
              if (gr < 2) {
#pragma unroll
                for (int dk = 0; dk < 2; ++dk) {
                  const int k = 2 * gr + dk;  // 128-dim chunk of the latent
#pragma unroll
                  for (int kk = 0; kk < 4; ++kk)
                    umma::mma_ts_f8(sd, tmem + kColQ + 32u * k + 8u * kk,
                                    umma::smem_desc(sbase + dk * 1024 + 32 * kk, 16, 2 * 1024, umma::kSw128),
                                    kIdescQK, (k | kk) != 0);
                }
              } else {
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)
                  umma::mma_ss_f8(sd, umma::smem_desc(qrope + 32 * kk, 16, 512, umma::kSw64),
                                  umma::smem_desc(sbase + 32 * kk, 16, 512, umma::kSw64), kIdescQK, 1u);
              }
            } else {
#pragma unroll
              for (int dk = 0; dk < 3; ++dk) {
                const int k = 3 * gr + dk;
                // chunk dk of the group: 8-row atoms every 3 KB
                const uint32_t st = sbase + dk * 1024;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  const uint64_t bdesc = umma::smem_desc(st + 32 * kk, 16, 3 * 1024, umma::kSw128);
                  if (k < 8)
                    umma::mma_ts(sd, tmem + kColQ + 32u * k + 8u * kk, bdesc, kIdescQK, (k | kk) != 0);
                  else
                    umma::mma_ss(sd, umma::smem_desc(qrope + 32 * kk, 16, 1024, umma::kSw128), bdesc, kIdescQK,
                                 1u);
                }
              }
            }
            umma::commit(&bars[kKEmpty + slot]);  // the group's slot may refill
          }
          if (!ok) break;
          umma::commit(&bars[kSFull + sb]);
        }
      } else if constexpr (F8) {
        // O += P(j) V(j) with the V tile the warps widened to f16: per 16
        // tokens, two N = 256 MMAs.  Each tile's rescale decision goes to the
        // warps through a two-slot ring (they read it before widening the tile
        // after next); a rescale waits for every earlier P.V and then for the
        // warps.
        const uint32_t hb = smem_u32(smem + SL::kOffH), pb = smem_u32(smem + SL::kOffP);
        const volatile uint32_t* fmsg = reinterpret_cast<const volatile uint32_t*>(smem + SL::kOffF);
        volatile int* dec = flags + 4;
        int nreq = 0, nod = 0;
        for (int j = 0; ok && j < ntiles; ++j) {
          const int p2 = j & 1;
          ok = mbar_wait(&bars[kPFull + p2], (j >> 1) & 1);
          if (!ok) break;
          // the slot's next message (tile j + 2) is sent only after this P.V
          if (j + 2 < ntiles) mbar_arrive_expect_tx(&bars[kPFull + p2], kPMsg);
          const bool resc = j > 0 && fmsg[p2 * (kFBytes / 4) + kRows] != 0u;
          if (resc) {  // O may change only once every earlier P.V is done
            umma::commit(&bars[kODone]);
            ok = mbar_wait(&bars[kODone], nod & 1);
            ++nod;
            if (!ok) break;
          }
          dec[p2] = resc ? 1 : 0;
          mbar_arrive(&bars[kDec + p2]);
          if (resc) {
            ok = mbar_wait(&bars[kOReady], nreq & 1);
            ++nreq;
            if (!ok) break;
          }
          ok = mbar_wait(&bars[kHFull + p2], (j >> 1) & 1);
          if (!ok) break;
          umma::fence_after_sync();
          const uint32_t pa = pb + p2 * kPBytes, va = hb + p2 * SL::kHBytes;
          for (int kk = 0; kk < 4; ++kk)
            for (int n = 0; n < 2; ++n)
              umma::mma_ss(tmem + kColO + uint32_t(kHalf * n),
                           umma::smem_desc(pa + 32 * kk, 16, 1024, umma::kSw128),
                           // V, MN-major: 64-dim atoms 1 KB apart, 8-row groups 8 KB apart
                           umma::smem_desc(va + 4 * n * 1024 + 2 * 8192 * kk, 1024, 8192, umma::kSw128),
                           kIdescPV, (j | kk) != 0);
          umma::commit(&bars[kHEmpty + p2]);
          // the logit CTA may stage and send the P of tile j + 2
          commit_to(&bars[kPSlotFree + p2], uint16_t(2u));
        }
      } else {
        // O += P(j) V(j): per 16 tokens, two N = 256 MMAs (O columns 0-255 and
        // 256-511).  A tile whose factors are not all 1, or whose V rows run
        // past the split's end, first goes to the warps (a request).
        const uint32_t vb = smem_u32(smem + SL::kOffV), pb = smem_u32(smem + SL::kOffP);
        const volatile uint32_t* fmsg = reinterpret_cast<const volatile uint32_t*>(smem + SL::kOffF);
        volatile int* req = flags + 2;
        int nreq = 0, nod = 0;
        for (int j = 0; ok && j < ntiles; ++j) {
          const int p2 = j & 1, vs = j % SL::kVSlots;
          ok = mbar_wait(&bars[kPFull + p2], (j >> 1) & 1);
          if (!ok) break;
          // the slot's next message (tile j + 2) is sent only after this P.V
          if (j + 2 < ntiles) mbar_arrive_expect_tx(&bars[kPFull + p2], kPMsg);
          const bool resc = j > 0 && fmsg[p2 * (kFBytes / 4) + kRows] != 0u;
          ok = mbar_wait(&bars[kVFull + vs], (j / SL::kVSlots) & 1);
          if (!ok) break;
          const bool tail = t_begin + (j + 1) * kTok > t_end;
          if (resc || tail) {
            if (resc) {  // O may change only once every earlier P.V is done
              umma::commit(&bars[kODone]);
              ok = mbar_wait(&bars[kODone], nod & 1);
              ++nod;
              if (!ok) break;
            }
            *req = j | (resc ? kReqRescale : 0) | (tail ? kReqTail : 0);
            mbar_arrive(&bars[kReq]);
            ok = mbar_wait(&bars[kOReady], nreq & 1);
            ++nreq;
            if (!ok) break;
          }
          umma::fence_after_sync();
          const uint32_t pa = pb + p2 * kPBytes, va = vb + vs * SL::kVBytes;
          for (int kk = 0; kk < 4; ++kk)
            for (int n = 0; n < 2; ++n)
              umma::mma_ss(tmem + kColO + uint32_t(kHalf * n),
                           umma::smem_desc(pa + 32 * kk, 16, 1024, umma::kSw128),
                           // V, MN-major: 64-dim atoms 1 KB apart, 8-row groups 8 KB apart
                           umma::smem_desc(va + 4 * n * 1024 + 2 * 8192 * kk, 1024, 8192, umma::kSw128),
                           kIdescPV, (j | kk) != 0);
          umma::commit(&bars[kVEmpty + vs]);
          // the logit CTA may stage and send the P of tile j + 2
          commit_to(&bars[kPSlotFree + p2], uint16_t(2u));
        }
      }
      if (!ok) flags[0] = 1;
      // nothing this thread issued may still run when tensor memory is read or freed
      umma::commit(&bars[kDrain]);
      if (!mbar_wait(&bars[kDrain], 0)) flags[0] = 1;
    }
    if (!logit_cta && lane == 0) {
      // the warps leave their request loop for the epilogue
      flags[2] = kReqEnd;
      mbar_arrive(&bars[kReq]);
    }
    // the other lanes wait here, not at the CTA barrier below: lanes parked at
    // a CTA barrier slow the MMA issue of their warp's active lane
    __syncwarp();
  } else if (logit_cta) {
    // ================= logit CTA: query load, online softmax, P shipping =====
    // Warp w (2..9) reaches TMEM lanes 32 (w % 4) .. +31 (query rows); h = (w - 2) / 4
    // picks logit columns [32h, 32h + 32) of every tile.
    const int q4 = warp & 3, h = (warp - kSoftWarp0) >> 2;
    const int t = 32 * q4 + lane;          // query row = TMEM lane
    const int st = tid - 32 * kSoftWarp0;  // 0 .. kSoft - 1
    const uint32_t lane_base = uint32_t(32 * q4) << 16;
    // row t = (spec token i, head t % Hq); rows at or past R are padding
    // (zero query, never stored): they take the last token's window and mask
    const bool real = t < a.R;
    const int i = min(t / a.Hq, a.qs - 1);
    const float q_scale = ldscale(a.q_scale_dev, a.q_scale);
    const float kv_scale = ldscale(a.kv_scale_dev, a.kv_scale);
    const float lscale = a.softmax_scale * q_scale * kv_scale * kLog2e;
    float* rowx = reinterpret_cast<float*>(smem + SL::kOffRowX);  // [2][128]
    constexpr int kC = kTok / 2;  // logit columns per thread

    // ---- query: this thread's half of the latent row into tensor memory
    // (bf16: dims [256h, 256h + 256) -> columns [128h, 128h + 128); e4m3: four
    // codes per column, columns [64h, 64h + 64)), half of its rope part into
    // shared memory (128- or 64-byte swizzled rows).  Loaded here for the
    // cluster's first piece; for the next ones at the end of the previous
    // piece, while the output CTA finishes its epilogue.
    int qload_n = 0;  // uses of the query-load barrier in this piece
    auto load_q = [&](int bq) {
      constexpr int kLB = F8 ? kLatent : 2 * kLatent;  // latent bytes of a query row
      constexpr int kRB = F8 ? kRope : 2 * kRope;      // rope bytes
      constexpr int kRU = kRB / 32;                    // rope 16-byte units per thread
      constexpr int kLU = kLB / 32;                    // latent 16-byte units per thread
      const uint4 zero = make_uint4(0, 0, 0, 0);
      uint4 rq[kRU];
      // latent units of this thread's half: from the staged rows (bf16) or
      // from registers loaded all at once (e4m3, half the bytes)
      uint4 xq[F8 ? kLU : 1];
      const uint8_t* row = smem + SL::kOffK + t * (kLB + kRB);
      auto unit = [&](int chunk, int u) {
        // an address's 16-byte unit is XORed with its bits 7-9 (128-byte swizzle)
        const uint32_t off = uint32_t(t * (kLB + kRB) + chunk * 128);
        return *reinterpret_cast<const uint4*>(row + chunk * 128 + ((u ^ int((off >> 7) & 7u)) << 4));
      };
      if constexpr (!F8) {
        // bf16: the sequence's 128 query rows in one TMA box ([row][9 chunks]
        // [128 B], 128-byte swizzle) into the free K ring; each thread then
        // reads its row's half (the swizzle spreads a warp's rows over the
        // banks)
        if (st == 0) {
          mbar_arrive_expect_tx(&bars[kQLoad], uint32_t(kRows * (kLB + kRB)));
          tma_load_3d(smem + SL::kOffK, &tmQ, &bars[kQLoad], 0, 0, bq * a.R);
        }
        const bool got = __all_sync(kAll, mbar_wait(&bars[kQLoad], qload_n & 1));
        ++qload_n;
        if (!got) flags[0] = 1;
#pragma unroll
        for (int u = 0; u < kRU; ++u) rq[u] = real ? unit(8, kRU * h + u) : zero;
      } else {
        const uint8_t* qrow = a.q + (int64_t(bq) * a.qs * a.Hq + min(t, a.R - 1)) * (kLB + kRB);
        const uint4* src = reinterpret_cast<const uint4*>(qrow + (kLB / 2) * h);
        const uint4* rsrc = reinterpret_cast<const uint4*>(qrow + kLB) + kRU * h;
#pragma unroll
        for (int u = 0; u < kRU; ++u) rq[u] = real ? __ldg(rsrc + u) : zero;
#pragma unroll
        for (int v = 0; v < kLU; ++v) xq[F8 ? v : 0] = real ? __ldg(src + v) : zero;
      }
#pragma unroll 1
      for (int half = 0; half < kLB / 512; ++half) {
        uint32_t w[64];
#pragma unroll
        for (int v = 0; v < 16; ++v) {
          const int vv = half * 16 + v;
          const uint4 x = F8 ? xq[F8 ? vv : 0] : (real ? unit(4 * h + vv / 8, vv % 8) : zero);
          w[4 * v + 0] = x.x;
          w[4 * v + 1] = x.y;
          w[4 * v + 2] = x.z;
          w[4 * v + 3] = x.w;
        }
        const uint32_t col = kColQ + uint32_t(kLB / 8) * uint32_t(h) + 64u * uint32_t(half);
        umma::tmem_st32(tmem + lane_base + col, w);
        umma::tmem_st32(tmem + lane_base + col + 32u, w + 32);
      }
#pragma unroll
      for (int u = 0; u < kRU; ++u)
        *reinterpret_cast<uint4*>(smem + SL::kOffQRope +
                                  (F8 ? umma::sw64(t, kRU * h + u) : umma::sw128(t, kRU * h + u))) = rq[u];
      umma::tmem_st_wait();
      umma::fence_proxy_async_smem();
    };
    if (q_loaded != b) load_q(b);
    umma::fence_before_sync();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[kQReady]);

    const uint32_t p_peer = map_peer(smem_u32(smem + SL::kOffP), peer);
    const uint32_t f_peer = map_peer(smem_u32(smem + SL::kOffF), peer);
    const int row_lb = a.win > 0 ? spec0 + i - a.win + 1 : INT_MIN;
    uint32_t row_mw = 0xffffffffu;
    if (a.mask) {
      const uint16_t* mrow = a.mask + (int64_t(b) * a.qs + i) * a.mask_words;
      row_mw = uint32_t(__ldg(mrow)) | (uint32_t(__ldg(mrow + 1)) << 16);
    }
    float m_ref = -INFINITY, l_half = 0.f;
    bool ok = true;
    // The output CTA signals once it has set up this piece's barriers: until
    // then this piece's tiles are computed and staged but not sent (the
    // output CTA may still be writing the previous piece out).
    bool peer_ready = false, peer_ok = false;
    auto wait_peer = [&]() {
      if (peer_ready) return;
      peer_ready = true;
      peer_ok = mbar_wait(&bars[kPeerReady], uint32_t(order) & 1u);
      if (!peer_ok) ok = false;
    };
    // Control flow stays uniform across each warp (tcgen05.ld is
    // warp-collective) and across the eight softmax warps (named barrier 1):
    // waits are voted and the loop is left collectively.
    // A 128-token logit tile holds two 64-token P tiles: both halves of this
    // thread's logits come out of tensor memory at once (the S buffer frees
    // early), then each half goes through the softmax and ships as its own
    // P message.
    for (int jq = 0; ok && jq < nqt; ++jq) {
      const int sb = jq & 1;
      const int nsub = min(2, ntiles - 2 * jq);
      float sv[2][kC];
      ok = __all_sync(kAll, mbar_wait(&bars[kSFull + sb], (jq >> 1) & 1));
      if (ok) {
        umma::fence_after_sync();
        umma::tmem_ld32(tmem + lane_base + kColS + 128u * uint32_t(sb) + 32u * h, sv[0]);
        if (nsub > 1) umma::tmem_ld32(tmem + lane_base + kColS + 128u * uint32_t(sb) + 64u + 32u * h, sv[1]);
        umma::tmem_ld_wait();
        umma::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kSFree + sb]);
      }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u >= nsub) break;
      const int j = 2 * jq + u, p2 = j & 1;
      float* s = sv[u];
      // staging slot p2 is free once the output CTA's P.V of tile j - 2 is
      // done (which also means its message landed)
      if (ok && j >= 2) ok = __all_sync(kAll, mbar_wait(&bars[kPSlotFree + p2], ((j >> 1) - 1) & 1));
      const int tile0 = t_begin + j * kTok;
      float mx = -INFINITY;
      if (ok) {
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
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // independent chains
#pragma unroll
        for (int k = 0; k < kC; ++k) {
          const float x = (vis >> k) & 1u ? s[k] * lscale : -INFINITY;
          s[k] = x;
          mx4[k & 3] = fmaxf(mx4[k & 3], x);
        }
        mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
        // (one buffer: the reads of the previous subtile's maxima precede
        // the barrier that ended it)
        rowx[h * kRows + t] = mx;
      }
      // both halves of every row published their maxima
      if (named_bar_or(1, kSoft, !ok)) {
        ok = false;
        break;
      }
      mx = fmaxf(mx, rowx[(1 - h) * kRows + t]);
      const float m_new = fmaxf(m_ref, mx);
      const bool need = m_new > m_ref + kRescaleLog2 || (m_ref == -INFINITY && m_new != -INFINITY);
      const float f = (need && m_ref != -INFINITY) ? exp2f(m_ref - m_new) : 1.f;
      if (need) {
        l_half *= f;
        m_ref = m_new;
      }
      // P (bf16, or f16 against a widened e4m3 V) for this thread's 32
      // columns: units 4h..4h+3 of row t; the row sum takes the rounded
      // weights so O / l stays a convex combination
      uint8_t* pstage = smem + SL::kOffPS + p2 * kPBytes;
      float* fstage = reinterpret_cast<float*>(smem + SL::kOffFS + p2 * kFBytes);
      float ls[4] = {0.f, 0.f, 0.f, 0.f};  // independent chains
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t w4[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float p0 = m_ref == -INFINITY ? 0.f : ex2(s[8 * u + 2 * e] - m_ref);
          const float p1 = m_ref == -INFINITY ? 0.f : ex2(s[8 * u + 2 * e + 1] - m_ref);
          w4[e] = pack_f32x2(p0, p1, !F8);
          if constexpr (F8) {
            // f16 keeps 11 significant bits: summing the unrounded weights
            // differs from the rounded ones by < 2^-12 of the sum
            ls[e] += p0 + p1;
          } else {
            const float2 r = unpack_16x2(w4[e], true);
            ls[e] += r.x + r.y;
          }
        }
        *reinterpret_cast<uint4*>(pstage + umma::sw128(t, 4 * h + u)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
      l_half += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      if (h == 0) fstage[t] = f;
      umma::fence_proxy_async_smem();
      // every thread wrote its P and factor; does any row need O rescaled?
      const bool resc = named_bar_or(1, kSoft, f != 1.f);
      if constexpr (kDecoupled) wait_peer();
      // P in four copies from four warps, the factors and the flag from a fifth
      if (kDecoupled && !ok) {
      } else if ((st & 31) == 0 && st < 32 * kCopyPieces) {
        const uint32_t off = uint32_t(st >> 5) * (kPBytes / kCopyPieces);
        bulk_to_peer(p_peer + p2 * kPBytes + off, smem_u32(pstage) + off, kPBytes / kCopyPieces,
                     peer_bars + 8u * (kPFull + p2));
      } else if (st == 32 * kCopyPieces) {
        reinterpret_cast<uint32_t*>(fstage)[kRows] = resc ? 1u : 0u;
        umma::fence_proxy_async_smem();
        bulk_to_peer(f_peer + p2 * kFBytes, smem_u32(fstage), kFBytes, peer_bars + 8u * (kPFull + p2));
      }
    }
    }
    if constexpr (kDecoupled) wait_peer();
    if (!ok) flags[0] = 1;
    // ---- the final row maxima and sums go to the output CTA (also when this
    // split saw no key: m = -inf, l = 0)
    float* fin = reinterpret_cast<float*>(smem + SL::kOffFinS);
    named_bar(1, kSoft);
    rowx[h * kRows + t] = l_half;
    named_bar(1, kSoft);
    if (h == 0) {
      fin[t] = m_ref;
      fin[kRows + t] = l_half + rowx[kRows + t];
    }
    umma::fence_proxy_async_smem();
    named_bar(1, kSoft);
    if (st == 0) {
      if (!kDecoupled || peer_ok)
        bulk_to_peer(map_peer(smem_u32(smem + SL::kOffFin), peer), smem_u32(fin), kFinBytes, peer_bars + 8u * kFin);
      // the peer's completion signals for the last two P slots must land
      // before this CTA may exit
      for (int j = max(0, ntiles - 2); ok && j < ntiles; ++j)
        if (!mbar_wait(&bars[kPSlotFree + (j & 1)], (j >> 1) & 1)) {
          flags[0] = 1;
          ok = false;
        }
    }
    // the next piece's query (every Q K^T of this piece is done: the softmax
    // read the last S tile, whose commit follows every earlier MMA)
    // (warp-uniform: the tensor-memory stores are warp-collective, and the
    // waits above ran on one lane)
    q_loaded = -1;
    if (__all_sync(kAll, ok) && next_b >= 0) {
      load_q(next_b);
      q_loaded = next_b;
    }
  } else {
    // ================= output CTA: requests, then the epilogue =================
    // Warp w (2..9) reaches TMEM lanes 32 (w % 4) .. +31; h = (w - 2) / 4 picks
    // O columns [256h, 256h + 256).
    const int q4 = warp & 3, h = (warp - kSoftWarp0) >> 2;
    const int t = 32 * q4 + lane;
    const int st = tid - 32 * kSoftWarp0;
    const uint32_t lane_base = uint32_t(32 * q4) << 16;
    const uint32_t o_cols = tmem + lane_base + kColO + uint32_t(kHalf * h);
    const bool real = t < a.R;  // rows at or past R are padding: computed, never stored
    const int i = min(t / a.Hq, a.qs - 1), hd = t % a.Hq;
    const float kv_scale = ldscale(a.kv_scale_dev, a.kv_scale);
    bool ok = true;
    // the previous piece's partial stores have had a piece's start to land:
    // count that piece done for the merge kernel (every warp's stores)
    if (pend_b >= 0) {
      if (lane == 0) bulk_wait_all_visible();
      named_bar(2, kSoft);
      if (st == 0) {
        __threadfence();
        atomicAdd(a.sems + pend_b, 1u);
      }
      pend_b = -1;
    }
    if constexpr (F8) {
      // Tile by tile: first the rescale decision for the previous tile (O is
      // multiplied by that tile's factors once every earlier P.V is done; the
      // MMA thread waits for it), then the e4m3 V tile widened to f16 (rows
      // past the split's end zeroed) into the f16 slot freed by the P.V of
      // the tile two back.  Then the end signal, which follows the drain.
      volatile int* dec = flags + 4;
      for (int j = 0; j <= ntiles; ++j) {
        if (j > 0) {
          const int jp = j - 1;
          ok = __all_sync(kAll, mbar_wait(&bars[kDec + (jp & 1)], (jp >> 1) & 1));
          if (!ok) break;
          if (dec[jp & 1]) {
            umma::fence_after_sync();
            const float f = reinterpret_cast<const float*>(smem + SL::kOffF + (jp & 1) * kFBytes)[t];
            if (__any_sync(kAll, f != 1.f)) rescale_o(o_cols, f);
            umma::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kOReady]);
          }
        }
        if (j == ntiles) break;
        ok = __all_sync(kAll, mbar_wait(&bars[kVFull + j % SL::kVSlots], (j / SL::kVSlots) & 1));
        if (ok && j >= 2) ok = __all_sync(kAll, mbar_wait(&bars[kHEmpty + (j & 1)], ((j >> 1) - 1) & 1));
        if (!ok) break;
        widen_v(smem + SL::kOffV + (j % SL::kVSlots) * SL::kVBytes, smem + SL::kOffH + (j & 1) * SL::kHBytes,
                t_end - (t_begin + j * kTok), st);
        umma::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars[kVEmpty + j % SL::kVSlots]);
          mbar_arrive(&bars[kHFull + (j & 1)]);
        }
      }
      if (ok) ok = __all_sync(kAll, mbar_wait(&bars[kReq], 0));
    } else {
      // Requests: rescale O by a tile's factors (every earlier P.V is done) and
      // / or zero the V rows past the split's end (the V slot has landed).  The
      // MMA thread waits for each request to be served before the next, so the
      // request word and the factor slot are stable while the warps read them.
      for (int k = 0;; ++k) {
        ok = __all_sync(kAll, mbar_wait(&bars[kReq], k & 1));
        if (!ok) break;
        const int r = *reinterpret_cast<volatile int*>(flags + 2);
        if (r == kReqEnd) break;
        const int j = r & kReqTile;
        umma::fence_after_sync();
        if (r & kReqRescale) {
          const float f = reinterpret_cast<const float*>(smem + SL::kOffF + (j & 1) * kFBytes)[t];
          if (__any_sync(kAll, f != 1.f)) rescale_o(o_cols, f);
        }
        if (r & kReqTail)
          zero_v_tail(smem + SL::kOffV + (j % SL::kVSlots) * SL::kVBytes, max(0, t_end - (t_begin + j * kTok)), st);
        umma::fence_proxy_async_smem();
        umma::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[kOReady]);
      }
    }
    if (!ok) flags[0] = 1;

    // ---- epilogue: the final (m, l) rows from the logit CTA, then finalise or
    // write the partial.  Every P.V is done (the end request follows the drain).
    if (!__all_sync(kAll, mbar_wait(&bars[kFin], 0))) {
      flags[0] = 1;
      ok = false;
    }
    umma::fence_after_sync();
    const float* fin = reinterpret_cast<const float*>(smem + SL::kOffFin);
    const float m_fin = fin[t], l_fin = fin[kRows + t];
    // (the staged stores below take named barriers: all eight warps decide together)
    ok = !named_bar_or(2, kSoft, !ok);
    if (ok) {
      const bool have_o = ntiles > 0;
      const bool single = nvalid <= 1;
      float mul = 0.f;
      const int64_t row_g = (int64_t(b) * a.qs + i) * a.Hq + hd;
      if (single) {
        const float sig = a.sinks ? __ldg(a.sinks + hd) * kLog2e : -INFINITY;
        mul = finalize_row(m_fin, l_fin, sig, kv_scale * a.rcp_out_scale,
                           (a.lse && h == 0 && real) ? a.lse + row_g : nullptr);
      }
      const int64_t slot = persistent ? 2 * int64_t(k_cl) + (cl_first ? 0 : 1) : int64_t(b) * a.nsplit + split;
      const uint64_t keep = l2_keep_policy();
      // O leaves through TMA stores that each warp issues for its own 32 rows
      // (no barrier between warps): a part is staged as [32 rows][128 B]
      // (128-byte swizzle) in the warp's 28 KB of the free V ring and P
      // slots, then stored by the warp's first lane.  bf16 output: four
      // 64-column pairs, each its own buffer, clipped at the sequence's R real
      // rows by the 3-D output view; fp32 partial: eight 32-column parts
      // through seven buffers.  The next part's columns come out of tensor
      // memory while the current one is staged.
      uint8_t* const wbuf = smem + SL::kOffV + (st >> 5) * kWarpStage;
      const bool store_rows = single ? 32 * q4 < a.R : true;
#pragma unroll 1
      for (int part = 0; part < kHalf / 32; ++part) {
        float cur[32];
        if (have_o) {
          umma::tmem_ld32(o_cols + 32u * part, cur);
          umma::tmem_ld_wait();
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) cur[k] = 0.f;
        }
        if (single) {
          // two parts (64 bf16 columns, 128 bytes) per staged row
          uint8_t* buf = wbuf + (part >> 1) * 4096;
#pragma unroll
          for (int v = 0; v < 4; ++v)
            *reinterpret_cast<uint4*>(buf + umma::sw128(lane, 4 * (part & 1) + v)) =
                make_uint4(pack_f32x2(cur[8 * v] * mul, cur[8 * v + 1] * mul, true),
                           pack_f32x2(cur[8 * v + 2] * mul, cur[8 * v + 3] * mul, true),
                           pack_f32x2(cur[8 * v + 4] * mul, cur[8 * v + 5] * mul, true),
                           pack_f32x2(cur[8 * v + 6] * mul, cur[8 * v + 7] * mul, true));
          if ((part & 1) == 0) continue;  // (the pair's second part stores both)
          umma::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && store_rows) {
            tma_store_3d(&tmO, buf, kHalf * h + 32 * (part - 1), 32 * q4, b);
            bulk_commit();
          }
        } else {
          // the buffer of the part kStageF32 back is free once its store read it
          if (part >= kStageF32) {
            if (lane == 0) bulk_wait_read<kStageF32 - 1>();
            __syncwarp();
          }
          uint8_t* buf = wbuf + (part % kStageF32) * 4096;
#pragma unroll
          for (int v = 0; v < 8; ++v)
            *reinterpret_cast<float4*>(buf + umma::sw128(lane, v)) =
                make_float4(cur[4 * v], cur[4 * v + 1], cur[4 * v + 2], cur[4 * v + 3]);
          umma::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d_hint(&tmWs, buf, kHalf * h + 32 * part, int(slot) * kRows + 32 * q4, keep);
            bulk_commit();
          }
        }
      }
      if (!single && h == 0) {
        float* wrow = a.ws + (slot * kRows + t) * (kLatent + 4);
        st_keep2(wrow + kLatent, m_fin, l_fin, keep);
      }
      // the staging is free again before the next piece loads V into it
      if (lane == 0) bulk_wait_read<0>();
      __syncwarp();
    }
    // a partial is counted done once its stores have landed (at the next
    // piece's start, or at the end); also after an abort, which the error
    // word reports, so that the merge does not wait out its time limit
    if (nvalid > 1) pend_b = b;
  }

  // ---- end of the piece in this CTA: no tensor-memory traffic outlives this
  // point, and none of the peer's: the output CTA has received every message
  // of the piece, the logit CTA every completion signal.  bf16: the logit CTA
  // goes on to the next piece while the output CTA still writes this one out;
  // a wait that gave up ends the loop for this CTA, and the peer's next wait
  // on it then gives up too.  e4m3 (bound by the output CTA, so that the
  // logit CTA gains nothing by running ahead): both CTAs pass two cluster
  // barriers, between which each reads the other's abort flag, and leave the
  // loop together.
  umma::fence_before_sync();
  __syncthreads();
  if constexpr (kDecoupled) {
    if (flags[0]) break;
  } else {
    cluster_sync();
    if (tid == 0) {
      uint32_t peer_abort;
      asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(peer_abort) : "r"(map_peer(smem_u32(flags), peer))
                   : "memory");
      flags[3] = flags[0] | int(peer_abort);
    }
    cluster_sync();
    if (flags[3]) break;
  }
  first_piece = false;
  if (!persistent) break;
  if (!z_now) {
    cur_S += a.piece_cost + nsched;
    ++cur_b;
  }
  ++order;
  }  // pieces
  // neither CTA leaves while the peer may still reach its shared memory
  // (e4m3: the last piece's cluster barriers did that)
  if (kDecoupled) cluster_sync();

  // ---- teardown
  if (pend_b >= 0) {  // (the output CTA's eight epilogue warps)
    if (lane == 0) bulk_wait_all_visible();
    named_bar(2, kSoft);
    if (tid == 32 * kSoftWarp0) {
      __threadfence();
      atomicAdd(a.sems + pend_b, 1u);
    }
  }
  umma::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    umma::fence_after_sync();
    umma::tmem_dealloc(tmem, kTmemCols);
  }
  if (flags[0] && tid == 0 && a.err) atomicOr(a.err, kErrTimeout);
}

// ---------------------------------------------------------------- split merge
// A second kernel in the same stream (programmatic dependent launch: its
// CTAs wait until every decode CTA has finished and its writes are visible)
// merges the partials of every sequence cut across clusters or splits with
// the log-sum-exp rule of merge_attn_states, adds the sinks and the output
// scales, and writes the bf16 rows (and their log-sum-exp).  It runs while
// the memory system is otherwise idle: merged at the end of the pieces that
// finish a sequence, the same loads compete with every cluster still
// streaming the cache, and the last ones end the call.
// Persistent: kMergeCtasPerSm CTAs per SM take the work items (sequence,
// column half, block of kMergeRows rows) in turn; each CTA first lays out the
// schedule of every sequence once (the decode kernel's integer arithmetic on
// the same lengths: pieces and partial slots).  Per item, the first pieces'
// partial rows are requested first; meanwhile one thread per row folds the
// pieces' maxima, the sink and the output scales into one weight per (row,
// piece) in shared memory (the merge_attn_states rule); then every thread
// sums its four rows x four columns.
constexpr int kMergeRows = 16;
constexpr int kMergeThreads = 256;
constexpr int kMergeChunk = 2;  // pieces of partial rows in flight per thread
constexpr int kMergeCtasPerSm = 3;
static_assert(kOrderMaxB <= kMergeThreads, "one sequence per thread in the schedule scan");

__global__ void __launch_bounds__(kMergeThreads, kMergeCtasPerSm) mla_merge_kernel(const MlaArgs a) {
  __shared__ int s_nvalid[kOrderMaxB], s_first[kOrderMaxB];  // per sequence (persistent schedule)
  __shared__ long long s_warp[kMergeThreads / 32];
  __shared__ float s_w[kMergeRows * kMaxPieces];  // per (row, piece): the maximum, then the weight
  __shared__ float s_l[kMergeRows * kMaxPieces];
  __shared__ bool s_ready;
  __shared__ int s_item;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool persistent = a.B <= kOrderMaxB;
  if (persistent) {
    // scheduled pages per sequence, their inclusive prefix sum over the batch
    long long sc = 0;
    int npages = 0;
    if (tid < a.B) {
      const SeqGeom g = seq_geom(a, tid);
      npages = max(0, g.pg_last - g.pg_first);
      sc = a.piece_cost + max(1, npages);
    }
    long long incl = sc;
    for (int o = 1; o < 32; o <<= 1) {
      const long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    long long before_warp = 0, tot = 0;
    for (int w = 0; w < kMergeThreads / 32; ++w) {
      if (w < warp) before_warp += s_warp[w];
      tot += s_warp[w];
    }
    if (tid < a.B) {
      const int64_t S0 = before_warp + incl - sc + a.piece_cost;
      const int ncl = int(min(int64_t(a.ncl), int64_t(tot)));
      const int kf = cluster_of(S0, tot, ncl);
      const int kl = cluster_of(S0 + max(1, npages) - 1, tot, ncl);
      s_nvalid[tid] = npages == 0 ? 0 : kl - kf + 1;
      // slot 2 kf, or 2 kf + 1 when the first piece starts inside cluster kf's slice
      s_first[tid] = 2 * kf + (S0 > tot * kf / ncl ? 1 : 0);
    }
    __syncthreads();
  }
  // (no griddepcontrol.wait: the CTAs are placed as decode CTAs exit and
  // merge each sequence as soon as its pieces are counted done, while the
  // last clusters still run; the next call's decode waits for this grid)
  pdl_launch_dependents();
  constexpr int kStride = kLatent + 4;
  constexpr int kQuads = kMergeThreads / (kHalf / 4);  // row groups of the CTA's threads
  constexpr int kRowsPer = kMergeRows / kQuads;
  constexpr int kBlocks = kRows / kMergeRows;
  const int c4 = tid % (kHalf / 4), rq = tid / (kHalf / 4);
  const float out_mul = ldscale(a.kv_scale_dev, a.kv_scale) * a.rcp_out_scale;
  const int items = a.B * 2 * kBlocks;
  // Items are handed out by a counter (semaphore 2B), so that the CTAs that
  // start first (on the SMs the first decode clusters leave) take most of
  // them and the last ones to start find the work done.
  uint32_t* const next_item = a.sems + 2 * a.B;
  for (;;) {
    if (tid == 0) s_item = int(atomicAdd(next_item, 1u));
    __syncthreads();
    const int item = s_item;
    __syncthreads();  // (s_item is rewritten for the next item)
    if (item >= items) break;
    const int b = item / (2 * kBlocks), c = (item / kBlocks) & 1, r0 = (item % kBlocks) * kMergeRows;
    if (r0 >= a.R) continue;
    // pieces; piece 0's slot, and piece sp >= 1's at slot1 + step (sp - 1):
    // slot 2 (kf + sp) of the persistent schedule, or split sp
    int nvalid, slot0, slot1, step;
    if (persistent) {
      nvalid = s_nvalid[b];
      slot0 = s_first[b];
      slot1 = (slot0 & ~1) + 2;
      step = 2;
    } else {
      const SeqGeom g = seq_geom(a, b);
      nvalid = (max(0, g.pg_last - g.pg_first) + a.split_pages - 1) / a.split_pages;
      slot0 = b * a.nsplit;
      slot1 = slot0 + 1;
      step = 1;
    }
    if (nvalid <= 1 || nvalid > kMaxPieces) continue;
    // every piece of the sequence is done and its partial visible
    if (tid == 0) {
      const long long t0 = clock64();
      uint32_t n;
      do {
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(n) : "l"(a.sems + b) : "memory");
      } while (n < uint32_t(nvalid) && clock64() - t0 < kWaitCycles);
      s_ready = n >= uint32_t(nvalid);
      if (!s_ready && a.err) atomicOr(a.err, kErrTimeout);
    }
    __syncthreads();
    const bool ready = s_ready;
    auto part_row = [&](int sp, int rr) {
      const int64_t slot = sp == 0 ? slot0 : slot1 + int64_t(step) * (sp - 1);
      return a.ws + (slot * kRows + r0 + rr) * kStride;
    };
    const int nrows = min(kMergeRows, a.R - r0);
    const int col = c * kHalf + 4 * c4;
    float4 v[kRowsPer][kMergeChunk];
    auto load_chunk = [&](int sp0) {
#pragma unroll
      for (int q = 0; q < kMergeChunk; ++q)
#pragma unroll
        for (int u = 0; u < kRowsPer; ++u) {
          const int rr = rq + kQuads * u;
          v[u][q] = (sp0 + q < nvalid && rr < nrows)
                        ? __ldcg(reinterpret_cast<const float4*>(part_row(sp0 + q, rr) + col))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    load_chunk(0);
    // (m, l) of every (row, piece), then one weight per (row, piece)
    for (int it = tid; it < nrows * nvalid; it += kMergeThreads) {
      const int rr = it / nvalid, sp = it - rr * nvalid;
      const float2 ml = __ldcg(reinterpret_cast<const float2*>(part_row(sp, rr) + kLatent));
      s_w[it] = ml.x;
      s_l[it] = ml.y;
    }
    __syncthreads();
    if (tid < nrows) {
      float* w = s_w + tid * nvalid;
      const float* lp = s_l + tid * nvalid;
      float M = -INFINITY;
      for (int sp = 0; sp < nvalid; ++sp) M = fmaxf(M, w[sp]);
      float l = 0.f;
      for (int sp = 0; sp < nvalid; ++sp) {
        const float f = w[sp] == -INFINITY ? 0.f : exp2f(w[sp] - M);
        w[sp] = f;
        l += f * lp[sp];
      }
      const int row = r0 + tid;
      const int64_t row_g = (int64_t(b) * a.qs + row / a.Hq) * a.Hq + row % a.Hq;
      const float sig = a.sinks ? __ldg(a.sinks + row % a.Hq) * kLog2e : -INFINITY;
      const float mul = finalize_row(M, l, sig, out_mul, (a.lse && c == 0) ? a.lse + row_g : nullptr);
      for (int sp = 0; sp < nvalid; ++sp) w[sp] *= mul;
    }
    __syncthreads();
    float4 acc[kRowsPer];
#pragma unroll
    for (int u = 0; u < kRowsPer; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp0 = 0; sp0 < nvalid; sp0 += kMergeChunk) {
      if (sp0 > 0) load_chunk(sp0);
#pragma unroll
      for (int q = 0; q < kMergeChunk; ++q)
#pragma unroll
        for (int u = 0; u < kRowsPer; ++u) {
          const int rr = rq + kQuads * u;
          const float f = (sp0 + q < nvalid && rr < nrows) ? s_w[rr * nvalid + sp0 + q] : 0.f;
          acc[u].x += f * v[u][q].x;
          acc[u].y += f * v[u][q].y;
          acc[u].z += f * v[u][q].z;
          acc[u].w += f * v[u][q].w;
        }
    }
#pragma unroll
    for (int u = 0; u < kRowsPer; ++u) {
      const int rr = rq + kQuads * u;
      if (rr >= nrows || !ready) continue;
      const int row = r0 + rr;
      const int64_t row_g = (int64_t(b) * a.qs + row / a.Hq) * a.Hq + row % a.Hq;
      *reinterpret_cast<uint2*>(a.out + row_g * kLatent + col) =
          make_uint2(pack_f32x2(acc[u].x, acc[u].y, true), pack_f32x2(acc[u].z, acc[u].w, true));
    }
    __syncthreads();  // the weights are rewritten by the next item
    // the last of the sequence's merge items zeroes both of its counters for
    // the next call (every other item has passed its wait)
    if (tid == 0) {
      const uint32_t items_b = 2u * uint32_t((a.R + kMergeRows - 1) / kMergeRows);
      if (atomicAdd(a.sems + a.B + b, 1u) == items_b - 1) {
        a.sems[b] = 0u;
        a.sems[a.B + b] = 0u;
      }
    }
  }
  // the last CTA to leave zeroes the item counter and its own count for the
  // next call (every CTA has drawn its last, out-of-range item by then)
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.sems + 2 * a.B + 1, 1u) == gridDim.x - 1) {
      *next_item = 0u;
      a.sems[2 * a.B + 1] = 0u;
    }
  }
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
  int nsplit = 1, split_pages = 1, ncl = 1;
  bool persistent = false;
  size_t ws_bytes = 0;   // split partials, then the per-sequence merge records
  size_t part_bytes = 0;  // the partials alone
};

const char* check_shape(const xqa_params* p, int v_head_dim) {
  if (p->num_kv_heads != 1) return "the MLA variant has one latent kv head (num_kv_heads must be 1)";
  if (p->head_dim != kDim || v_head_dim != kLatent)
    return "the MLA kernel is built for a 576-wide latent row (512 latent + 64 rope) with v_head_dim 512";
  if (int64_t(p->num_q_heads) * p->q_seq_len > kRows)
    return "the MLA kernel needs num_q_heads * q_seq_len <= 128 (one UMMA tile of query rows)";
  const bool bf16 = p->q_dtype == XQA_BF16 && p->kv_dtype == XQA_BF16;
  const bool e4m3 = p->q_dtype == XQA_E4M3 && p->kv_dtype == XQA_E4M3;
  if (!bf16 && !e4m3)
    return "the MLA kernel takes a bf16 query with a bf16 latent cache, or an e4m3 query with an e4m3 cache";
  if (p->out_dtype != XQA_BF16) return "the MLA kernel writes a bf16 output";
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
  // one cluster (2 CTAs, one per SM) per (sequence, split); aim for ~kWaves waves
  const int64_t pairs = int64_t(sm / 2) * kWaves;
  int64_t ns = (pairs + p->batch_size - 1) / p->batch_size;
  const int64_t by_tiles = (max_pages + stage_pages - 1) / stage_pages;
  const int64_t by_tokens = std::max<int64_t>(1, int64_t(max_pages) * p->page_size / 1024);
  ns = std::max<int64_t>(1, std::min(ns, std::min(by_tiles, by_tokens)));
  ns = std::min<int64_t>(ns, kMaxSplits);
  int sp = int((max_pages + ns - 1) / ns);
  sp = ((sp + stage_pages - 1) / stage_pages) * stage_pages;
  pl->split_pages = sp;
  pl->nsplit = (max_pages + sp - 1) / sp;
  pl->part_bytes = pl->nsplit > 1 ? size_t(p->batch_size) * pl->nsplit * kRows * (kLatent + 4) * sizeof(float) : 0;
  // up to kOrderMaxB sequences: persistent clusters, one per SM pair (at most
  // kMaxPieces, so that a sequence's merge weights fit in shared memory), two
  // partial slots each
  pl->persistent = p->batch_size <= kOrderMaxB;
  if (pl->persistent) {
    pl->ncl = std::max(1, std::min(sm / 2, kMaxPieces));
    pl->part_bytes = pl->ncl > 1 ? size_t(pl->ncl) * 2 * kRows * (kLatent + 4) * sizeof(float) : 0;
  }
  pl->ws_bytes = pl->part_bytes;
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
  // per sequence: finished pieces, finished merge items; then the merge
  // kernel's item counter and its count of finished CTAs
  return size_t(p->batch_size) * 2 + 2;
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
    if (reinterpret_cast<uintptr_t>(ws) & 15) {
      snprintf(err, err_len, "workspace must be 16-byte aligned");
      return XQA_ERR_INVALID_ARG;
    }
    if (!sems) {
      snprintf(err, err_len, "semaphores are required (%zu needed)", size_t(p->batch_size) * 2 + 2);
      return XQA_ERR_WORKSPACE_TOO_SMALL;
    }
    if (reinterpret_cast<uintptr_t>(sems) & 3) {
      snprintf(err, err_len, "semaphores must be 4-byte aligned");
      return XQA_ERR_INVALID_ARG;
    }
  }
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    snprintf(err, err_len, "cuTensorMapEncodeTiled is unavailable");
    return XQA_ERR_CUDA;
  }
  // NHD and HND coincide for one kv head: rows of 576 elements, token-major.
  // Row-group view (128 bytes, 8 rows, 128-byte chunks, row groups): a box of
  // one page piece's rows across several chunks lands as [row group][chunk]
  // [8 rows][128 B].  bf16: nine chunks of 64 dims; logit tiles take three
  // chunks per box, V tiles eight.  e4m3: four chunks of 128 latent dims
  // (logit tiles take two per box, V tiles four) and a separate 3-D view of
  // the 64-byte rope part (64-byte swizzle).
  const bool f8 = p->kv_dtype == XQA_E4M3;
  const cuuint64_t elt = f8 ? 1 : 2, row_bytes = cuuint64_t(kDim) * elt;
  const cuuint32_t box_rows = cuuint32_t(std::min(p->page_size, kTok));
  const cuuint64_t nrows = cuuint64_t(p->page_size) * cuuint64_t(p->num_pages);
  const CUtensorMapDataType dt = f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const cuuint32_t chunk_elems = cuuint32_t(128 / elt);
  const cuuint64_t nchunks = f8 ? kLatent / 128 : kDim / 64;
  cuuint64_t dims[4] = {chunk_elems, 8, nchunks, nrows / 8};
  cuuint64_t strides[3] = {row_bytes, 128, row_bytes * 8};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUtensorMap tk, tkr, tv;
  cuuint32_t kbox[4] = {chunk_elems, 8, cuuint32_t(f8 ? Lay<true>::kGroupChunks : Lay<false>::kGroupChunks),
                        box_rows / 8};
  cuuint32_t vbox[4] = {chunk_elems, 8, cuuint32_t(f8 ? Lay<true>::kVChunks : Lay<false>::kVChunks), box_rows / 8};
  CUresult r = enc(&tk, dt, 4, const_cast<void*>(p->k_cache), dims, strides, kbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS)
    r = enc(&tv, dt, 4, const_cast<void*>(p->k_cache), dims, strides, vbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r == CUDA_SUCCESS && f8) {
    // the rope part of each e4m3 row: (64 bytes, 8 rows, row groups) from byte 512 of the row
    cuuint64_t rdims[3] = {kRope, 8, nrows / 8};
    cuuint64_t rstrides[2] = {row_bytes, row_bytes * 8};
    cuuint32_t rbox[3] = {kRope, 8, box_rows / 8};
    r = enc(&tkr, dt, 3, static_cast<uint8_t*>(const_cast<void*>(p->k_cache)) + kLatent, rdims, rstrides, rbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    tkr = tk;  // unused by the bf16 kernel
  }
  if (r != CUDA_SUCCESS) {
    snprintf(err, err_len, "cuTensorMapEncodeTiled failed (%d)", int(r));
    return XQA_ERR_CUDA;
  }
  // L2 prefetch view of the same rows: (64 elements, 9 pieces, rows), so
  // that one box covers a page piece's rows across all 576 dims
  CUtensorMap tpf;
  cuuint64_t pdims[3] = {64, kDim / 64, nrows};
  cuuint64_t pstrides[2] = {64 * elt, row_bytes};
  cuuint32_t pbox[3] = {64, kDim / 64, box_rows};
  r = enc(&tpf, dt, 3, const_cast<void*>(p->k_cache), pdims, pstrides, pbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    snprintf(err, err_len, "cuTensorMapEncodeTiled (prefetch view) failed (%d)", int(r));
    return XQA_ERR_CUDA;
  }
  // bf16 query rows as (64 elements, 9 chunks, rows): one box is a
  // sequence's 128 query rows (rows past it are padding, never stored)
  CUtensorMap tq = tpf;  // unused by the e4m3 kernel
  if (!f8) {
    cuuint64_t qdims[3] = {64, kDim / 64, cuuint64_t(p->batch_size) * p->q_seq_len * p->num_q_heads};
    cuuint64_t qstrides[2] = {128, cuuint64_t(kDim) * 2};
    cuuint32_t qbox[3] = {64, kDim / 64, kRows};
    r = enc(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p->q), qdims, qstrides, qbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
      snprintf(err, err_len, "cuTensorMapEncodeTiled (query view) failed (%d)", int(r));
      return XQA_ERR_CUDA;
    }
  }
  // epilogue store views, one box per epilogue warp (its 32 rows): the
  // output (bf16, 512 per row, as [sequence][R rows][512]; a box is 64
  // columns of 32 rows, clipped at the R real rows) and the split partials
  // (fp32, 512 + 4 per row; a box is 32 columns of 32 rows of a slot)
  CUtensorMap to, tws = tpf;
  {
    const int R = p->num_q_heads * p->q_seq_len;
    cuuint64_t odims[3] = {kLatent, cuuint64_t(R), cuuint64_t(p->batch_size)};
    cuuint64_t ostrides[2] = {kLatent * 2, cuuint64_t(R) * kLatent * 2};
    cuuint32_t obox[3] = {64, cuuint32_t(std::min(R, 32)), 1};
    r = enc(&to, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p->output, odims, ostrides, obox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r == CUDA_SUCCESS && pl.ws_bytes > 0) {
      cuuint64_t wdims[2] = {kLatent + 4, cuuint64_t(pl.ws_bytes / ((kLatent + 4) * sizeof(float)))};
      cuuint64_t wstrides[1] = {(kLatent + 4) * sizeof(float)};
      cuuint32_t wbox[2] = {32, 32};
      r = enc(&tws, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ws, wdims, wstrides, wbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) {
      snprintf(err, err_len, "cuTensorMapEncodeTiled (epilogue views) failed (%d)", int(r));
      return XQA_ERR_CUDA;
    }
  }
  MlaArgs a;
  memset(&a, 0, sizeof a);
  a.q = static_cast<const uint8_t*>(p->q);
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
  a.ncl = pl.ncl;
  a.piece_cost = (kPieceTokens + p->page_size - 1) / p->page_size;
  a.mask_words = ((p->q_seq_len + 31) / 32) * 2;
  a.q_scale = p->q_scale;
  a.kv_scale = p->kv_scale;
  a.softmax_scale = p->softmax_scale != 0.f ? p->softmax_scale : 1.0f / sqrtf(float(kDim));
  a.rcp_out_scale = p->rcp_out_scale;
  a.R = p->num_q_heads * p->q_seq_len;
  const int smem = f8 ? smem_bytes<true>() : smem_bytes<false>();
  cudaError_t e = f8 ? cudaFuncSetAttribute(mla_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)
                     : cudaFuncSetAttribute(mla_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) {
    snprintf(err, err_len, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    return XQA_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = pl.persistent ? dim3(2 * pl.ncl, 1, 1) : dim3(2 * pl.nsplit, 1, p->batch_size);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = p->enable_pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = f8 ? cudaLaunchKernelEx(&cfg, mla_decode_kernel<true>, tk, tkr, tv, tpf, tq, tws, to, a)
         : cudaLaunchKernelEx(&cfg, mla_decode_kernel<false>, tk, tkr, tv, tpf, tq, tws, to, a);
  if (e != cudaSuccess) {
    snprintf(err, err_len, "MLA kernel launch: %s", cudaGetErrorString(e));
    return XQA_ERR_CUDA;
  }
  if (pl.ws_bytes > 0) {
    // the split merge, launched behind the decode kernel (its CTAs wait in
    // griddepcontrol.wait for the decode grid to finish)
    cudaLaunchConfig_t mcfg = {};
    const int sm = sm_count_of(p, 0);
    const int items = p->batch_size * 2 * (kRows / kMergeRows);
    mcfg.gridDim = dim3(std::max(1, std::min(items, sm * kMergeCtasPerSm)), 1, 1);
    mcfg.blockDim = dim3(kMergeThreads);
    mcfg.stream = stream;
    cudaLaunchAttribute mattr[1];
    mattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    mattr[0].val.programmaticStreamSerializationAllowed = 1;
    mcfg.attrs = mattr;
    mcfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&mcfg, mla_merge_kernel, a);
    if (e != cudaSuccess) {
      snprintf(err, err_len, "MLA merge kernel launch: %s", cudaGetErrorString(e));
      return XQA_ERR_CUDA;
    }
  }
  return XQA_OK;
}

}  // namespace xqa
