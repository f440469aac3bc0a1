// C ABI of the paged decode attention library (declared in include/xqa.h):
// argument validation, split-KV planning, TMA descriptor set-up and launch.
//
// Validation mirrors the XQA API page's stated constraints (FlashInfer
// "flashinfer.xqa.xqa": page_size in {16, 32, 64, 128}; K/V dtype equal to
// q's or float8_e4m3fn; page_table int32 [B, pages_per_seq]; sinks
// [num_kv_heads, head_group_ratio]; mask [B, q_seq_len,
// ((q_seq_len + 31) // 32) * 2]) and rejects before launching anything.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>

#include "gqa_launch.h"
#include "kernel_args.h"
#include "mla_launch.h"
#include "xqa.h"
#include "xqa_internal.h"

namespace {

thread_local char g_last_error[512] = "";

xqa_status fail(xqa_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return st;
}

xqa_status cuda_fail(cudaError_t e, const char* what) {
  return fail(XQA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// ---------------------------------------------------------------- driver entry
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// ---------------------------------------------------------------- device facts
constexpr int kMaxDevices = 64;
constexpr int kMaxSplits = 64;  // merge weights [rows][splits] fit in the kernel's shared memory

int device_sm_count(int dev) {
  static int cache[kMaxDevices] = {0};
  if (dev < 0 || dev >= kMaxDevices) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess) cache[dev] = n;
  }
  return cache[dev];
}

bool is_16bit(xqa_dtype t) { return t == XQA_F16 || t == XQA_BF16; }
int elt_bytes(xqa_dtype t) { return t == XQA_E4M3 ? 1 : 2; }

// ---------------------------------------------------------------- planning
struct Plan {
  bool mla = false;
  int D = 0, Dv = 0, G = 0, R = 0;
  int row_blocks = 1, warp_rows = 1, rows = 16, rg_count = 1;
  bool tc = false;  // the tensor-core kernel (large grouped tiles, 16-bit K/V)
  int nsplit = 1, split_pages = 1;
  int persist = 0;  // tensor-core kernel: persistent CTAs (0: one CTA per unit and split)
  int max_pages = 1;
  size_t ws_bytes = 0;
  size_t nsems = 0;
};

// mla: the latent variant, which also takes an e4m3 query with an e4m3 cache
// (vLLM Kimi-K3 MultiHeadLatentAttention page, `_decode_concat_cache`: an fp8
// cache takes an fp8 query) and then writes a bf16 output.
xqa_status validate_common(const xqa_params* p, bool mla = false) {
  if (!p) return fail(XQA_ERR_INVALID_ARG, "params is NULL");
  if (!p->q || !p->k_cache || !p->v_cache || !p->page_table || !p->seq_lens || !p->output)
    return fail(XQA_ERR_INVALID_ARG, "q, k_cache, v_cache, page_table, seq_lens and output are required");
  if (p->batch_size < 1) return fail(XQA_ERR_INVALID_ARG, "batch_size must be >= 1, got %d", p->batch_size);
  if (reinterpret_cast<uintptr_t>(p->lse) & 3) return fail(XQA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  if (p->num_q_heads < 1 || p->num_kv_heads < 1)
    return fail(XQA_ERR_INVALID_ARG, "num_q_heads and num_kv_heads must be >= 1");
  if (p->num_q_heads % p->num_kv_heads)
    return fail(XQA_ERR_INVALID_ARG, "num_q_heads (%d) must be a multiple of num_kv_heads (%d)",
                p->num_q_heads, p->num_kv_heads);
  if (p->page_size != 16 && p->page_size != 32 && p->page_size != 64 && p->page_size != 128)
    return fail(XQA_ERR_INVALID_ARG, "page_size must be one of 16, 32, 64, 128; got %d", p->page_size);
  if (p->pages_per_seq < 1) return fail(XQA_ERR_INVALID_ARG, "pages_per_seq must be >= 1");
  if (p->num_pages < 1) return fail(XQA_ERR_INVALID_ARG, "num_pages must be >= 1");
  if (p->q_seq_len < 1) return fail(XQA_ERR_INVALID_ARG, "q_seq_len must be >= 1");
  if (p->q_seq_len > 32)
    return fail(XQA_ERR_UNSUPPORTED, "q_seq_len > 32 is not supported (got %d)", p->q_seq_len);
  if (p->sliding_win_size < 0) return fail(XQA_ERR_INVALID_ARG, "sliding_win_size must be >= 0");
  if (mla && p->q_dtype == XQA_E4M3) {
    if (p->kv_dtype != XQA_E4M3) return fail(XQA_ERR_INVALID_ARG, "an e4m3 query needs an e4m3 latent cache");
    if (p->out_dtype != XQA_BF16)
      return fail(XQA_ERR_UNSUPPORTED, "the MLA decode of an e4m3 query writes a bf16 output");
  } else {
    if (!is_16bit(p->q_dtype))
      return fail(XQA_ERR_INVALID_ARG, mla ? "q dtype must be float16, bfloat16 or (with an e4m3 cache) e4m3"
                                           : "q dtype must be float16 or bfloat16");
    if (!(p->kv_dtype == p->q_dtype || p->kv_dtype == XQA_E4M3))
      return fail(XQA_ERR_INVALID_ARG, "kv dtype must match q's dtype or be float8_e4m3fn");
    // the output dtype matches the query, or the fp8 cache (API page, `output`)
    if (!(p->out_dtype == p->q_dtype || (p->out_dtype == XQA_E4M3 && p->kv_dtype == XQA_E4M3)))
      return fail(XQA_ERR_UNSUPPORTED,
                  "output dtype must equal the query dtype, or be float8_e4m3fn with an fp8 cache");
  }
  if (p->head_dim < 1) return fail(XQA_ERR_INVALID_ARG, "head_dim must be >= 1");
  const int64_t big = int64_t(1) << 31;
  if (p->num_pages * std::max(p->page_size, p->num_kv_heads) >= big ||
      int64_t(p->pages_per_seq) * p->page_size >= big)
    return fail(XQA_ERR_UNSUPPORTED, "cache too large for 32-bit TMA coordinates");
  if ((reinterpret_cast<uintptr_t>(p->k_cache) | reinterpret_cast<uintptr_t>(p->v_cache)) & 15)
    return fail(XQA_ERR_INVALID_ARG, "k_cache and v_cache must be 16-byte aligned");
  // the kernels read q as 32-bit element pairs and store four output elements
  // at once: one 8-byte store for a 16-bit output, one 4-byte store for e4m3
  if (reinterpret_cast<uintptr_t>(p->q) & 3) return fail(XQA_ERR_INVALID_ARG, "q must be 4-byte aligned");
  if (reinterpret_cast<uintptr_t>(p->output) & (p->out_dtype == XQA_E4M3 ? 3 : 7))
    return fail(XQA_ERR_INVALID_ARG, "output must be %d-byte aligned for its dtype",
                p->out_dtype == XQA_E4M3 ? 4 : 8);
  if ((reinterpret_cast<uintptr_t>(p->page_table) | reinterpret_cast<uintptr_t>(p->seq_lens) |
       reinterpret_cast<uintptr_t>(p->sinks) | reinterpret_cast<uintptr_t>(p->error_word) |
       reinterpret_cast<uintptr_t>(p->q_scale_dev) | reinterpret_cast<uintptr_t>(p->kv_scale_dev)) & 3)
    return fail(XQA_ERR_INVALID_ARG,
                "page_table, seq_lens, sinks, error_word and the device scales must be 4-byte aligned");
  if (p->mask && (reinterpret_cast<uintptr_t>(p->mask) & 1))
    return fail(XQA_ERR_INVALID_ARG, "mask must be 2-byte aligned");
  return XQA_OK;
}

int resolve_sm_count(const xqa_params* p, int sm_count) {
  if (sm_count > 0) return sm_count;
  if (p && p->sm_count > 0) return p->sm_count;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  return device_sm_count(dev);
}

// Pages a CTA set may have to read for one sequence: the whole table, or
// with a window the (window + q_seq_len - 1)-token span plus one page of
// misalignment.
int pages_bound(const xqa_params* p) {
  int n = p->pages_per_seq;
  if (p->sliding_win_size > 0) {
    int64_t span = int64_t(p->sliding_win_size) + p->q_seq_len - 1;
    n = int(std::min<int64_t>(n, (span + p->page_size - 1) / p->page_size + 1));
  }
  return n;
}

// Split count.  The kernels are HBM-bound and their CTAs go out in blockIdx
// order to sm_count x ctas_per_sm slots.  The count minimises a fluid model of
// the grid's makespan, taking every sequence at the page table's bound (the
// host does not read the lengths):
//   - n = units x splits CTAs of p = split tokens + a fixed per-CTA cost
//     (pipeline fill and drain, epilogue, merge) each;
//   - full waves share the memory system evenly, so k = n / slots of them take
//     k p;
//   - the r = n % slots CTAs of a last partial wave each run at most at twice
//     an even share, so they take p max(r / slots, 1/2).
// Fewer splits save the fixed costs; more splits fill the last wave.  Measured
// per-CTA costs, in tokens of streaming: mma.sync kernel ~128, tensor-core
// kernel ~1024 (its query into tensor memory and pipeline fill).  The choices
// on the measured workloads: Llama-3-8B-shaped (512 units) 1 split, 182 us
// against 192 and 197 us for 2 and 3; fp8 long context (1024 units of 32768
// tokens) 2 splits, 1.373 ms against 1.426 ms (1) and 1.398 ms (3); large
// group on the tensor-core kernel 1 split, 0.232 ms against 0.257 ms (2).
// Splits are whole pipeline stages and never below 256 tokens.
#ifndef XQA_GQA_CTA_COST_TOKENS
#define XQA_GQA_CTA_COST_TOKENS 128
#endif
#ifndef XQA_TC_CTA_COST_TOKENS
#define XQA_TC_CTA_COST_TOKENS 1024
#endif
void choose_splits(const xqa_params* p, Plan* pl, int sm_count, int ctas_per_sm, int stage_pages) {
  const int64_t units = int64_t(p->batch_size) * p->num_kv_heads * pl->rg_count;
  const int max_pages = pl->max_pages;
  const int64_t slots = int64_t(std::max(sm_count, 1)) * std::max(ctas_per_sm, 1);
  const int64_t cost = pl->tc ? XQA_TC_CTA_COST_TOKENS : XQA_GQA_CTA_COST_TOKENS;
  const int64_t by_stage = (max_pages + stage_pages - 1) / stage_pages;
  const int64_t by_tokens = std::max<int64_t>(1, (int64_t(max_pages) * p->page_size) / 256);
  const int ns_cap = int(std::max<int64_t>(1, std::min<int64_t>(kMaxSplits, std::min(by_stage, by_tokens))));
  int best_sp = 0, best_ns = 0;
  double best = 0.0;
  for (int ns = 1; ns <= ns_cap; ++ns) {
    int sp = (max_pages + ns - 1) / ns;
    sp = ((sp + stage_pages - 1) / stage_pages) * stage_pages;
    const int nsr = (max_pages + sp - 1) / sp;  // splits that stage rounding leaves
    if (nsr != ns) continue;
    const int64_t n = units * nsr;
    const double piece = double(int64_t(sp) * p->page_size + cost);
    const int64_t k = n / slots, r = n % slots;
    const double waves = double(k) + (r ? std::max(double(r) / double(slots), 0.5) : 0.0);
    const double m = waves * piece;
    if (best_ns == 0 || m < best * (1.0 - 1e-9)) {
      best = m;
      best_sp = sp;
      best_ns = nsr;
    }
  }
  if (best_ns == 0) {  // (ns = 1 always qualifies; kept for safety)
    best_sp = ((max_pages + stage_pages - 1) / stage_pages) * stage_pages;
    best_ns = 1;
  }
  pl->split_pages = std::max(best_sp, 1);
  pl->nsplit = (max_pages + pl->split_pages - 1) / pl->split_pages;
}

// Tokens per pipeline stage of the GQA kernel: 128 when a K row is one
// 128-byte swizzle chunk (fp8 D=128, 16-bit D=64) and one 16-row block holds
// the rows, else 64.  Must match GqaCfg::kTok.
int stage_tokens(const xqa_params* p, int row_blocks, int warp_rows) {
  return (p->head_dim * elt_bytes(p->kv_dtype) == 128 && row_blocks == 1 && warp_rows == 1) ? 128 : 64;
}

// Large grouped tiles with 16-bit K/V run on the tensor-core kernel: more
// than 16 rows per kv head at head_dim 128, more than 32 at head_dim 64 (the
// sizes the mma.sync kernel holds in one 16-row block per warp, or two).
bool use_tc(const xqa_params* p, int R) {
  return is_16bit(p->kv_dtype) && ((p->head_dim == 128 && R > 16) || (p->head_dim == 64 && R > 32));
}

// Rows of one CTA of the mma.sync kernel for R = q_seq_len x G query rows per
// kv head: 16-row blocks per consumer warp (row_blocks) and warp row groups
// (warp_rows), so that up to 64 rows share one pass over the KV pages (e4m3
// K/V; 16-bit K/V take the tensor-core kernel beyond one or two blocks).
void row_shape(int D, int R, int* row_blocks, int* warp_rows) {
  *row_blocks = 1;
  *warp_rows = 1;
  if (R <= 16) return;
  if (D == 64 && R <= 32) {
    *row_blocks = 2;  // two blocks per warp, the stage split four ways
    return;
  }
  *warp_rows = (D == 128 && R <= 32) ? 2 : 4;
}

xqa_status plan_gqa(const xqa_params* p, int sm_count_in, Plan* pl) {
  xqa_status st = validate_common(p);
  if (st != XQA_OK) return st;
  const int D = p->head_dim;
  if (p->kv_dtype == XQA_E4M3 ? D != 128 : (D != 64 && D != 128))
    return fail(XQA_ERR_UNSUPPORTED, "head_dim %d is not built for this KV dtype (16-bit KV: 64 or 128; fp8 KV: 128)", D);
  pl->D = pl->Dv = D;
  pl->G = p->num_q_heads / p->num_kv_heads;
  pl->R = p->q_seq_len * pl->G;
  pl->tc = use_tc(p, pl->R);
  row_shape(D, pl->R, &pl->row_blocks, &pl->warp_rows);
  pl->rows = pl->tc ? 128 : 16 * pl->row_blocks * pl->warp_rows;
  pl->rg_count = (pl->R + pl->rows - 1) / pl->rows;
  pl->max_pages = pages_bound(p);
  const int sm = resolve_sm_count(p, sm_count_in);
  if (sm <= 0) return fail(XQA_ERR_CUDA, "cannot query the SM count of the current device");
  int occ = 0;
  cudaError_t e;
  if (pl->tc)
    e = xqa::gqa_tc_launch(p->kv_dtype == XQA_BF16, D, false, dim3(), nullptr, nullptr, nullptr, nullptr, &occ);
  else if (p->kv_dtype == XQA_E4M3)
    e = xqa::gqa_launch_e4m3(D, pl->row_blocks, pl->warp_rows, false, dim3(), nullptr, nullptr, nullptr, nullptr,
                             &occ);
  else if (p->kv_dtype == XQA_BF16)
    e = xqa::gqa_launch_bf16(D, pl->row_blocks, pl->warp_rows, false, dim3(), nullptr, nullptr, nullptr, nullptr,
                             &occ);
  else
    e = xqa::gqa_launch_f16(D, pl->row_blocks, pl->warp_rows, false, dim3(), nullptr, nullptr, nullptr, nullptr,
                            &occ);
  if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
  const int tok = pl->tc ? 128 : stage_tokens(p, pl->row_blocks, pl->warp_rows);
  const int stage_pages = p->page_size <= tok ? tok / p->page_size : 1;
  choose_splits(p, pl, sm, occ, stage_pages);
  const int64_t units = int64_t(p->batch_size) * p->num_kv_heads * pl->rg_count;
  // More unsplit tensor-core units than CTA slots: the slots' CTAs stay
  // resident and take the units in turn (ranked longest first), so each unit
  // after a CTA's first starts its loads while the one before is finalised,
  // and no SM waits for the next CTA to be scheduled.  Needs the ranking
  // (2..160 sequences).
  const int64_t slots = int64_t(sm) * std::max(occ, 1);
  pl->persist = (pl->tc && pl->nsplit == 1 && p->batch_size > 1 && p->batch_size <= 160 && units > slots)
                    ? int(slots)
                    : 0;
  pl->nsems = size_t(units);
  pl->ws_bytes = pl->nsplit > 1 ? size_t(units) * pl->nsplit * pl->rows * (D + 4) * sizeof(float) : 0;
  return XQA_OK;
}

xqa_status make_maps(const xqa_params* p, int head_dim, int box_rows, CUtensorMap* tk, CUtensorMap* tv) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return fail(XQA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const int elt = elt_bytes(p->kv_dtype);
  CUtensorMapDataType dt = p->kv_dtype == XQA_E4M3   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                           : p->kv_dtype == XQA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const uint64_t D = uint64_t(head_dim), H = uint64_t(p->num_kv_heads), ps = uint64_t(p->page_size);
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3], estr[3] = {1, 1, 1};
  if (p->kv_layout == XQA_HND) {
    dims[0] = D;
    dims[1] = ps;
    dims[2] = H * uint64_t(p->num_pages);
    strides[0] = D * elt;
    strides[1] = ps * D * elt;
    box[0] = 128 / elt;
    box[1] = box_rows;
    box[2] = 1;
  } else {
    dims[0] = D;
    dims[1] = H;
    dims[2] = ps * uint64_t(p->num_pages);
    strides[0] = D * elt;
    strides[1] = H * D * elt;
    box[0] = 128 / elt;
    box[1] = 1;
    box[2] = box_rows;
  }
  const void* ptrs[2] = {p->k_cache, p->v_cache};
  CUtensorMap* maps[2] = {tk, tv};
  for (int i = 0; i < 2; ++i) {
    CUresult r = enc(maps[i], dt, 3, const_cast<void*>(ptrs[i]), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(XQA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  }
  return XQA_OK;
}

void fill_args(const xqa_params* p, const Plan& pl, void* ws, uint32_t* sems, xqa::DecodeArgs* a) {
  memset(a, 0, sizeof *a);
  a->q = p->q;
  a->out = p->output;
  a->page_table = p->page_table;
  a->seq_lens = p->seq_lens;
  a->sinks = p->sinks;
  a->mask = p->mask;
  a->q_scale_dev = p->q_scale_dev;
  a->kv_scale_dev = p->kv_scale_dev;
  a->ws = static_cast<float*>(ws);
  a->sems = sems;
  a->err = p->error_word;
  a->lse = p->lse;
  a->num_pages = p->num_pages;
  a->B = p->batch_size;
  a->Hq = p->num_q_heads;
  a->Hkv = p->num_kv_heads;
  a->G = pl.G;
  a->qs = p->q_seq_len;
  a->R = pl.R;
  a->ps = p->page_size;
  a->pps = p->pages_per_seq;
  a->win = p->sliding_win_size;
  a->nsplit = pl.nsplit;
  a->split_pages = pl.split_pages;
  a->rg_count = pl.rg_count;
  a->mask_words = ((p->q_seq_len + 31) / 32) * 2;
  a->Dv = pl.Dv;
  a->q_scale = p->q_scale;
  a->kv_scale = p->kv_scale;
  a->softmax_scale = p->softmax_scale != 0.f ? p->softmax_scale : 1.0f / sqrtf(float(pl.D));
  a->rcp_out_scale = p->rcp_out_scale;
  a->q_bf16 = p->q_dtype == XQA_BF16;
  a->out_e4m3 = p->out_dtype == XQA_E4M3;
  a->hnd = p->kv_layout == XQA_HND;
  a->pdl = p->enable_pdl != 0;
  a->sort_b = p->batch_size > 1 && p->batch_size <= 160;
  a->persist = pl.persist;
}

xqa_status check_buffers(const Plan& pl, void* ws, size_t ws_bytes, uint32_t* sems) {
  if (pl.ws_bytes > 0) {
    if (!ws || ws_bytes < pl.ws_bytes)
      return fail(XQA_ERR_WORKSPACE_TOO_SMALL, "workspace needs %zu bytes, got %zu", pl.ws_bytes,
                  ws ? ws_bytes : size_t(0));
    if (reinterpret_cast<uintptr_t>(ws) & 15)
      return fail(XQA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    if (!sems) return fail(XQA_ERR_WORKSPACE_TOO_SMALL, "semaphores are required (%zu needed)", pl.nsems);
  }
  return XQA_OK;
}

}  // namespace

namespace xqa {
void set_last_error(const char* msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }
}  // namespace xqa

extern "C" {

const char* xqa_status_string(xqa_status s) {
  switch (s) {
    case XQA_OK: return "XQA_OK";
    case XQA_ERR_INVALID_ARG: return "XQA_ERR_INVALID_ARG";
    case XQA_ERR_UNSUPPORTED: return "XQA_ERR_UNSUPPORTED";
    case XQA_ERR_WORKSPACE_TOO_SMALL: return "XQA_ERR_WORKSPACE_TOO_SMALL";
    case XQA_ERR_CUDA: return "XQA_ERR_CUDA";
  }
  return "XQA_ERR_UNKNOWN";
}

const char* xqa_last_error(void) { return g_last_error; }

size_t xqa_workspace_size(const xqa_params* p, int sm_count) {
  Plan pl;
  if (plan_gqa(p, sm_count, &pl) != XQA_OK) return size_t(-1);
  return pl.ws_bytes;
}

size_t xqa_semaphore_count(const xqa_params* p) {
  xqa_status st = validate_common(p);
  if (st != XQA_OK) return size_t(-1);
  const int G = p->num_q_heads / p->num_kv_heads;
  const int R = p->q_seq_len * G;
  int rb = 1, wr = 1;
  row_shape(p->head_dim, R, &rb, &wr);
  const int rows = use_tc(p, R) ? 128 : 16 * rb * wr;
  return size_t(p->batch_size) * p->num_kv_heads * ((R + rows - 1) / rows);
}

xqa_status xqa_decode(const xqa_params* p, void* ws, size_t ws_bytes, uint32_t* sems,
                      xqa_stream_t stream) {
  g_last_error[0] = 0;
  Plan pl;
  xqa_status st = plan_gqa(p, 0, &pl);
  if (st != XQA_OK) return st;
  st = check_buffers(pl, ws, ws_bytes, sems);
  if (st != XQA_OK) return st;
  CUtensorMap tk, tv;
  const int box_rows = std::min(p->page_size, pl.tc ? 64 : stage_tokens(p, pl.row_blocks, pl.warp_rows));
  st = make_maps(p, pl.D, box_rows, &tk, &tv);
  if (st != XQA_OK) return st;
  xqa::DecodeArgs a;
  fill_args(p, pl, ws, sems, &a);
  const dim3 grid = pl.persist ? dim3(1, 1, pl.persist) : dim3(pl.nsplit, p->num_kv_heads * pl.rg_count, p->batch_size);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (pl.tc)
    e = xqa::gqa_tc_launch(p->kv_dtype == XQA_BF16, pl.D, true, grid, &tk, &tv, &a, s, nullptr);
  else if (p->kv_dtype == XQA_E4M3)
    e = xqa::gqa_launch_e4m3(pl.D, pl.row_blocks, pl.warp_rows, true, grid, &tk, &tv, &a, s, nullptr);
  else if (p->kv_dtype == XQA_BF16)
    e = xqa::gqa_launch_bf16(pl.D, pl.row_blocks, pl.warp_rows, true, grid, &tk, &tv, &a, s, nullptr);
  else
    e = xqa::gqa_launch_f16(pl.D, pl.row_blocks, pl.warp_rows, true, grid, &tk, &tv, &a, s, nullptr);
  if (e != cudaSuccess) return cuda_fail(e, "decode kernel launch");
  return XQA_OK;
}

size_t xqa_mla_workspace_size(const xqa_params* p, int v_head_dim, int sm_count) {
  return xqa::mla_workspace_size(p, v_head_dim, sm_count);
}

size_t xqa_mla_semaphore_count(const xqa_params* p, int v_head_dim) {
  return xqa::mla_semaphore_count(p, v_head_dim);
}

xqa_status xqa_mla_decode(const xqa_params* p, int v_head_dim, void* ws, size_t ws_bytes,
                          uint32_t* sems, xqa_stream_t stream) {
  g_last_error[0] = 0;
  xqa_status st = validate_common(p, true);
  if (st != XQA_OK) return st;
  return xqa::mla_decode(p, v_head_dim, ws, ws_bytes, sems, reinterpret_cast<cudaStream_t>(stream),
                         g_last_error, sizeof g_last_error);
}

}  // extern "C"
