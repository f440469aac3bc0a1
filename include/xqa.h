/*
 * xqa.h — C ABI of the GB300 (sm_103a) paged-KV decode attention library.
 *
 * Operation (FlashInfer "flashinfer.xqa.xqa" API page: signature, parameter
 * list and the shape-inference note; beam_width is fixed to 1, the only width
 * that page supports): one or a few speculative query tokens per sequence
 * attend to a paged KV cache.  For batch b, query token i < q_seq_len and
 * query head h (kv head kvh = h / G, G = Hq / Hkv):
 *
 *   L = seq_lens[b] (it counts the q_seq_len new tokens), p = L - q_seq_len + i
 *   token t lives in page page_table[b][t / page_size], slot t % page_size
 *   visible(t): t < L, and t > p - sliding_win_size (window on), and for the
 *               new tokens t >= L - q_seq_len the mask bit (i, t - L + q_seq_len)
 *   s_t = softmax_scale * q_scale * kv_scale * <q[b,i,h,:], K[t,:]>
 *   out[b,i,h,:] = rcp_out_scale * kv_scale * sum_t e^{s_t - M} V[t,:] / Z
 *   with M = max(max_t s_t, sink) and Z = sum_t e^{s_t - M} + e^{sink - M};
 *   sink = sinks[kvh][h % G] (a logit, not scaled), absent when sinks is NULL.
 *   A row with nothing visible and no sink is written as zeros.
 *
 * The MLA latent variant (vLLM Kimi-K3 MultiHeadLatentAttention page:
 * head_size = kv_lora_rank + qk_rope_head_dim, scale = qk_head_dim^-0.5, and
 * the forward_mqa call on the absorbed query) is the same operation with one
 * kv head of width head_dim = kv_lora_rank + rope and V = the first v_head_dim
 * (= kv_lora_rank) elements of each latent row.
 *
 * Conventions
 *  - Every pointer is DEVICE memory owned by the caller; the library never
 *    allocates, frees or synchronises.  Calls are asynchronous on `stream`.
 *  - `output` is written in place (the API page: "modified in place").
 *  - Host-side validation returns a status before anything is launched; a
 *    launch failure returns XQA_ERR_CUDA.  Alignment: caches 16 bytes; q 4
 *    bytes; output 8 bytes (16-bit) or 4 bytes (e4m3); page_table, seq_lens,
 *    sinks, lse, error_word and the device scales 4 bytes; mask 2 bytes.
 *  - Device code never traps.  A page_table entry outside [0, num_pages)
 *    reads as zeros (TMA bounds fill) and a seq_len above
 *    pages_per_seq * page_size is clamped to it; both set bit 0 of
 *    `error_word` when the caller provides one.  Every pipeline wait is
 *    bounded (about a second); one that gives up sets bit 1 and the call's
 *    output is then undefined.
 */
#ifndef XQA_GB300_H
#define XQA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* xqa_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  XQA_OK = 0,
  XQA_ERR_INVALID_ARG = 1,         /* malformed argument (null pointer, bad shape, bad value) */
  XQA_ERR_UNSUPPORTED = 2,         /* well-formed but outside what the kernels implement */
  XQA_ERR_WORKSPACE_TOO_SMALL = 3, /* workspace_bytes < xqa_workspace_size(), or no semaphores */
  XQA_ERR_CUDA = 4                 /* a CUDA runtime call or kernel launch failed */
} xqa_status;

typedef enum { XQA_F16 = 0, XQA_BF16 = 1, XQA_E4M3 = 2 } xqa_dtype;

/* NHD: cache [num_pages, page_size, Hkv, head_dim]; HND: [num_pages, Hkv, page_size, head_dim]. */
typedef enum { XQA_NHD = 0, XQA_HND = 1 } xqa_layout;

typedef struct xqa_params {
  /* q [batch, q_seq_len, num_q_heads, head_dim], fp16 or bf16, contiguous. */
  const void* q;
  xqa_dtype q_dtype;
  /* K and V caches: kv_dtype is q_dtype or XQA_E4M3 (then "fp8 compute"),
     shared by both; both use kv_layout.  They may alias (MLA latent cache). */
  const void* k_cache;
  const void* v_cache;
  xqa_dtype kv_dtype;
  xqa_layout kv_layout;
  int64_t num_pages;
  /* int32 [batch, pages_per_seq], shared by K and V. */
  const int32_t* page_table;
  int32_t pages_per_seq;
  /* uint32 [batch]; max_seq_len = pages_per_seq * page_size. */
  const uint32_t* seq_lens;
  /* output [batch, q_seq_len, num_q_heads, v_head_dim]; out_dtype must equal q_dtype. */
  void* output;
  xqa_dtype out_dtype;
  int32_t batch_size;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t page_size;  /* 16, 32, 64 or 128 */
  int32_t q_seq_len;  /* >= 1; > 1 is speculative decoding */
  /* fp32 [num_kv_heads, num_q_heads / num_kv_heads] or NULL (no sinks). */
  const float* sinks;
  /* Scale factors for q and the KV cache.  A non-NULL *_dev pointer names one
     device float that replaces the host value (the "float or Tensor" form). */
  float q_scale;
  float kv_scale;
  const float* q_scale_dev;
  const float* kv_scale_dev;
  /* Logit scale; 0 means 1/sqrt(head_dim).  The API page's call has no such
     argument; the MLA variant needs (qk_nope + qk_rope)^-0.5. */
  float softmax_scale;
  int32_t sliding_win_size; /* 0 = no window */
  float rcp_out_scale;      /* reciprocal of the output scale; multiplies the output */
  /* uint16 [batch, q_seq_len, ((q_seq_len + 31) / 32) * 2], bit-packed in
     little-endian 32-bit words (bit j % 32 of word j / 32: may see new token j),
     or NULL (all new tokens visible). */
  const uint16_t* mask;
  int32_t sm_count;   /* SMs to plan for; 0 = the current device's count */
  int32_t enable_pdl; /* programmatic dependent launch; accepted, no numeric effect */
  uint32_t* error_word; /* optional device word; bit 0 = clamped length or bad page index */
  /* Optional fp32 [batch, q_seq_len, num_q_heads], or NULL: each row's
     log-sum-exp, the natural log of the normaliser its output was divided by
     (visible logits and the sink; -inf for a row with neither).  It is the
     `lse` that forward_mqa returns next to the latent output (vLLM Kimi-K3
     MultiHeadLatentAttention page, forward), in the units merge_attn_states
     takes (same page, the prefill path with chunked context). */
  float* lse;
} xqa_params;

/* Bytes of workspace xqa_decode needs for these parameters when planning for
   sm_count SMs (0 = current device).  0 means the call needs none.  Returns
   (size_t)-1 for parameters xqa_decode would reject. */
size_t xqa_workspace_size(const xqa_params* params, int sm_count);

/* Number of uint32 semaphores xqa_decode needs.  They must be zero on the
   first call; every call leaves them zero again (the last CTA to finish a
   split-KV reduction resets its counter), also a call whose pipeline wait
   gave up (bit 1 of error_word): its CTAs still take their tickets. */
size_t xqa_semaphore_count(const xqa_params* params);

/* Paged decode attention (the XQA-style call).  workspace: caller-owned device
   scratch of at least xqa_workspace_size() bytes (any contents); semaphores:
   xqa_semaphore_count() zeroed uint32.  Both may be NULL when their size is 0.
   Two calls that share workspace or semaphores must not overlap on the GPU. */
xqa_status xqa_decode(const xqa_params* params, void* workspace, size_t workspace_bytes,
                      uint32_t* semaphores, xqa_stream_t stream);

/* Same sizing queries for the MLA latent variant (num_kv_heads = 1).  The
   workspace holds the split partials (fp32); the semaphores (2 B + 2) count
   each sequence's finished pieces and finished merge items, then hand out the
   merge kernel's work items and count its finished CTAs. */
size_t xqa_mla_workspace_size(const xqa_params* params, int v_head_dim, int sm_count);
size_t xqa_mla_semaphore_count(const xqa_params* params, int v_head_dim);

/* MLA latent decode: params->num_kv_heads must be 1, head_dim the latent width
   (kv_lora_rank + rope) and v_head_dim the kv_lora_rank prefix used as V.
   k_cache and v_cache may be the same pointer (the latent cache).  q and
   output must be 16-byte aligned.  One or two kernel launches on `stream`:
   the decode, then (when the workspace size is not 0) the merge of the
   sequences cut across clusters or splits, launched with programmatic
   dependent launch: its CTAs take the SMs the decode CTAs leave and merge a
   sequence once the decode has counted all of its pieces done.  The
   semaphores (xqa_mla_semaphore_count uint32, 4-byte aligned; may be NULL
   when the workspace size is 0) must be zero on the first call; every call
   that runs to its end leaves them zero, also one that reported a timeout
   (bit 1 of error_word): a merge that gave up waiting still counts itself,
   and the last merge CTA to finish zeroes the work counter. */
xqa_status xqa_mla_decode(const xqa_params* params, int v_head_dim, void* workspace,
                          size_t workspace_bytes, uint32_t* semaphores, xqa_stream_t stream);

/* xqa_decode without caller-provided scratch.  The pages have no counterpart:
   the XQA call always takes workspace_buffer and semaphores from its caller.
   This variant is for callers that may not allocate device memory where they
   call decode attention (for example a runtime that has reserved the device's
   memory for its own KV-cache pool, or code whose allocator lives elsewhere):
   it uses a scratch array built into the library instead -- 64 MiB of split
   workspace and 16384 tickets, held on every GPU that loads the library until
   the process exits.  It never calls cudaMalloc or cudaFree.
   - The first call on a device looks up that device's scratch address
     (cudaGetSymbolAddress); make that first call before any stream capture.
     A lookup that fails returns XQA_ERR_CUDA and is tried again by the next
     call; a successful one is kept for the life of the process.
   - Problems whose workspace or ticket count exceed the built-in sizes are
     rejected with XQA_ERR_WORKSPACE_TOO_SMALL (see xqa_last_error) before
     anything is launched; use xqa_decode with your own buffers for them.
   - Every call on a device shares the one array.  Calls whose executions
     overlap on the GPU (different streams, different threads) race on it and
     produce wrong results; serialise them.  Each call clears the tickets it
     needs on `stream` before launching; the workspace keeps the last call's
     contents, which no call reads before writing. */
xqa_status xqa_decode_noalloc(const xqa_params* params, xqa_stream_t stream);

/* merge_attn_states (vLLM Kimi-K3 MultiHeadLatentAttention page, the prefill
   path with chunked context): two attention results over disjoint key sets of
   the same query rows, each normalised by its own sum, combine into the result
   over the union of the keys:
     M = max(lse_p, lse_s), w_p = e^(lse_p - M), w_s = e^(lse_s - M),
     out = (w_p out_p + w_s out_s) / (w_p + w_s), lse = M + ln(w_p + w_s).
   A side whose lse is -inf (no visible key) weighs 0; both -inf gives 0 and
   -inf.  Rows of tokens t >= tokens_with_prefix have no prefix and take the
   suffix unchanged (the page's prefill_tokens_with_context).
   Outputs are fp16 or bf16 [num_tokens, num_heads, head_dim] with element
   strides between tokens and between heads (head_dim contiguous; strides and
   pointers 16-byte aligned, head_dim a multiple of 8), so a prefix result wider
   than head_dim (a latent slice) is read in place.  lse arrays are fp32 with
   their own token and head strides, shared by the three of them.  output_lse
   may be NULL.  All memory is caller-owned device memory; the call is
   asynchronous on `stream`.  Returns XQA_ERR_INVALID_ARG for bad shapes,
   strides or alignment, before any launch. */
typedef struct xqa_merge_params {
  void* output;
  const void* prefix_output;
  const void* suffix_output;
  xqa_dtype dtype;            /* of all three outputs: XQA_F16 or XQA_BF16 */
  float* output_lse;          /* NULL: not written */
  const float* prefix_lse;
  const float* suffix_lse;
  int64_t num_tokens;
  int32_t num_heads;
  int32_t head_dim;
  int64_t tokens_with_prefix; /* 0 .. num_tokens */
  int64_t out_stride_token, out_stride_head;       /* elements */
  int64_t prefix_stride_token, prefix_stride_head; /* elements */
  int64_t suffix_stride_token, suffix_stride_head; /* elements */
  int64_t lse_stride_token, lse_stride_head;       /* floats */
} xqa_merge_params;

xqa_status xqa_merge_attn_states(const xqa_merge_params* params, xqa_stream_t stream);

/* Fused MLA decode prep (vLLM Kimi-K3 MultiHeadLatentAttention page,
   `_decode_concat_cache`, the launch right before forward_mqa), bf16:
     q_out[t, h] = [ql_nope[t, h] | rope(q_pe[t, h], positions[t])]
     kv_cache[slot_mapping[t]] = [kv_c[t] | rope(k_pe[t], positions[t])]
   rope is the GPT-J (non-neox) rotation: pair (2i, 2i+1) turns by angle i, with
   cos and sin read in fp32 from cos_sin_cache[positions[t]] = [cos_0..cos_{R/2-1} |
   sin_0..sin_{R/2-1}]; positions NULL means no rotation.  A negative slot is a
   padding token and inserts nothing.  A position outside [0, max_position) is
   not rotated and a slot >= num_slots is not written; both set bit 0 of
   error_word when one is given.
   Layouts: ql_nope [T, H, Lr], q_pe [T, H, R] with element strides per token and
   per head; kv_c [T, Lr], k_pe [T, R] with a token stride; kv_cache
   [num_slots, Lr + R] (num_pages * page_size rows of the latent cache, NHD);
   q_out [T, H, Lr + R] contiguous.  Lr and R multiples of 8, strides multiples
   of 8 elements, tensors 16-byte aligned.  Asynchronous on `stream`; returns
   XQA_ERR_INVALID_ARG before any launch for malformed arguments.
   fp8 != 0 is the plain per-tensor fp8 cache of the same page's
   `_decode_concat_cache` (an fp8 cache takes an fp8 query): q_out and kv_cache
   are then float8_e4m3fn, and every element written is x * q_scale_inv (query)
   or x * cache_scale_inv (cache row), x the fp32 value above, rounded to
   nearest even and saturated at +-448.  q_scale_inv and cache_scale_inv are
   device fp32 scalars (the reciprocals of q_scale and kv_scale), required
   then; the inputs stay bf16. */
typedef struct xqa_mla_prep_params {
  const void* ql_nope;
  int64_t ql_stride_token, ql_stride_head;
  const void* q_pe;
  int64_t qpe_stride_token, qpe_stride_head;
  const void* kv_c;
  int64_t kvc_stride_token;
  const void* k_pe;
  int64_t kpe_stride_token;
  const int64_t* positions;    /* [T] or NULL */
  const float* cos_sin_cache;  /* fp32 [max_position, R] */
  int64_t max_position;
  const int64_t* slot_mapping; /* [T] */
  void* kv_cache;
  int64_t num_slots;
  void* q_out;
  int64_t num_tokens;
  int32_t num_heads;
  int32_t kv_lora_rank;        /* Lr */
  int32_t rope_dim;            /* R */
  uint32_t* error_word;        /* optional */
  int32_t fp8;                 /* 0: bf16 q_out and cache; else e4m3 (see above) */
  const float* q_scale_inv;    /* device scalar, fp8 only */
  const float* cache_scale_inv; /* device scalar, fp8 only */
} xqa_mla_prep_params;

xqa_status xqa_mla_decode_prep(const xqa_mla_prep_params* params, xqa_stream_t stream);

/* A measurement aid, not part of the decode path: one launch that streams
   `bytes` of device memory at `buf` once (16-byte non-temporal loads, a
   grid-stride loop over 4 CTAs per SM, at most `sink_words` CTAs) and writes
   nothing but, with negligible probability, one word of `sink`.  Timed with
   events around it, it gives the device's read-only HBM rate that the decode
   kernels (which read the cache and write little) are set beside; the copy
   kernel's rate counts a write for every byte read.
   Errors: XQA_ERR_INVALID_ARG for a null buf or sink, bytes zero or not a
   multiple of 16, a buf not 16-byte aligned, or sink_words <= 0;
   XQA_ERR_CUDA for a failed device query or launch.  Asynchronous on
   `stream`; buf and sink are caller-owned device memory. */
xqa_status xqa_read_bandwidth_probe(const void* buf, size_t bytes, uint32_t* sink, int sink_words,
                                    xqa_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* xqa_status_string(xqa_status status);

/* Detail of the most recent non-OK status returned on the calling thread
   (static per-thread buffer; "" when none). */
const char* xqa_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* XQA_GB300_H */
