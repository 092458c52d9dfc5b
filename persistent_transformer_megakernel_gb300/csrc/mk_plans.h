// Compile-time kernel plans of the decode megakernel (host and device).
//
// mk_create picks, for every GEMV phase, one of the fast layouts of
// mk_host.cu's table (staged or split-K, with its per-thread slice, rows per
// thread and tiles per batch) from the model's shape.  A kernel compiled for
// a plan has those five choices and the attention group size as constants: it
// runs every phase inline, with no device-function calls, only the code its
// model needs (a smaller instruction working set per forward) and no
// run-time dispatch.  Shapes whose choices match no plan run the general
// kernel, which dispatches at run time into out-of-line phase functions.
#pragma once

namespace mk {

// layout of one GEMV phase: {fast (1 staged, 2 split-K), KPT, RPT, BT}
struct PlanHidden1024 {
  // hidden 1024, 16 query / 8 KV heads of 128, MLP 3072 (the Qwen3-0.6B
  // dims, which the TTS talker mirrors): any vocabulary
  static constexpr bool fixed = true;
  static constexpr int hd = 128, grp = 2;
  static constexpr bool attn_blocks = true;     // attention in 8-position blocks per warp
  static constexpr int spec[5][4] = {{1, 32, 2, 2}, {2, 8, 8, 1}, {1, 32, 2, 2}, {2, 12, 4, 2}, {1, 32, 2, 2}};
};

struct PlanHidden2048 {
  // hidden 2048, 16 query / 8 KV heads of 128, MLP 6144 (the Qwen3-1.7B dims)
  static constexpr bool fixed = true;
  static constexpr int hd = 128, grp = 2;
  static constexpr bool attn_blocks = false;    // one position per warp (measured 4% faster at this shape)
  static constexpr int spec[5][4] = {{1, 64, 1, 4}, {2, 8, 8, 2}, {1, 64, 1, 4}, {2, 24, 2, 8}, {1, 64, 1, 4}};
};

struct PlanGeneral {
  static constexpr bool fixed = false;
  static constexpr int hd = 0, grp = 0;
  static constexpr bool attn_blocks = true;
  static constexpr int spec[5][4] = {};
};

}  // namespace mk
