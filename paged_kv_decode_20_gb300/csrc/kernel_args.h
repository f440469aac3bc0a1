// Launch arguments shared by the host planner and the decode kernels.
#pragma once
#include <stdint.h>

namespace xqa {

constexpr float kLog2e = 1.4426950408889634f;

struct DecodeArgs {
  const void* q;               // [B, qs, Hq, D] f16/bf16
  void* out;                   // [B, qs, Hq, Dv] same dtype as q
  const int32_t* page_table;   // [B, pps]
  const uint32_t* seq_lens;    // [B]
  const float* sinks;          // [Hkv, G] or null
  const uint16_t* mask;        // [B, qs, mask_words] or null
  const float* q_scale_dev;    // optional device scalars
  const float* kv_scale_dev;
  float* ws;                   // split partials
  uint32_t* sems;              // one ticket counter per (b, kvh, row group)
  uint32_t* err;               // optional error word
  float* lse;                  // optional [B, qs, Hq] natural-log log-sum-exp per row
  int64_t num_pages;
  int B, Hq, Hkv, G, qs, R;    // R = qs * G rows per kv head
  int ps, pps, win;            // page size, pages per sequence, sliding window
  int nsplit;                  // splits per (b, kvh, row group) in the grid
  int split_pages;             // pages per split
  int rg_count;                // row groups per kv head
  int mask_words;              // uint16 per mask row
  int Dv;
  float q_scale, kv_scale, softmax_scale, rcp_out_scale;
  int q_bf16;                  // q (and a 16-bit out) are bf16 (else f16)
  int out_e4m3;                // out is float8_e4m3fn (rounded to nearest, saturated at +-448)
  int hnd;                     // cache layout HND (else NHD)
  int pdl;                     // launched with programmatic stream serialization
  int sort_b;                  // map grid slots to sequences longest first (B <= 160)
  int persist;                 // tensor-core kernel: this many persistent CTAs take the
                               // unsplit units in turn (0: one CTA per unit and split)
};

}  // namespace xqa
