// Batched prompt prefill (csrc/mk_prefill.cu): interface between the C ABI in
// mk_host.cu and the prefill kernels + tensor-core GEMMs (csrc/mk_gemm.cu).
#pragma once
#include <cstdint>
#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>
#include <vector>

#include "../../include/mk.h"
#include "mk_gemm.h"

namespace mkp {

constexpr int MK_PF_ERR_BAD_TOKEN = MK_ERR_BAD_TOKEN;
constexpr int MK_PF_ERR_NUMERIC = MK_ERR_NUMERIC;
constexpr int MK_PF_ERR_BAD_POSITION = MK_ERR_BAD_POSITION;

// the call-dependent fields, read by the kernels from a device copy so that a
// captured graph of the prefill can be replayed for another call
struct PfCall {
  const int32_t *ids;               // [n] prompt ids (device)
  const float *embeds;              // sentinel rows [n_embed_rows][H] fp32, or NULL
  int n_embed_rows;
  const int32_t *pos3;              // [3][n_pos] position streams, or NULL
  int n_pos, pos0;
  float *hidden;                    // [n][L+1][H] or NULL
  int32_t *out_ids;                 // [n] greedy ids, or NULL
  float *logits_out;                // [n][V], or NULL
  int *last_id;                     // the last token's greedy id (the handle's)
};

// everything a prefill kernel reads: shape, model, handle state, scratch, and
// the device copy of the call
struct PfArgs {
  int L, H, Hq, Hkv, d, I, V, vocab_in;
  float eps, inv_sqrt_d;
  int rope_mode, sec0, sec1, sec2, rope_len, max_seq;
  const uint16_t *embed;            // [vocab_in][H] bf16
  const float2 *rope;               // [rope_len][d/2] (cos, sin)
  uint16_t *kcache, *vcache;        // [L][Hkv][max_seq][d] bf16, the decode kernel's cache
  const PfCall *call;               // device copy of the call's fields
  int *err;                         // first error code (device)
  float *x, *qkv, *attn;            // chunk scratch (fp32): residual, normed q, attention output
  float *attn_part;                 // split-KV attention partials [PF_ATTN_SPLITS][tc][Hq][d + 2] (o, m, l)
  float *qkv_p, *y_p;               // GEMM outputs as split-K partials, qkv_stride / y_stride apart
  size_t qkv_stride, y_stride;
  int qkv_n;                        // partials of the QKV output of the current chunk
  uint16_t *hs;                     // GEMM input as three bf16 terms (hi, mid, lo), hs_stride apart
  size_t hs_stride;
};

// per-layer weights (borrowed device pointers, bf16)
struct PfLayer {
  const uint16_t *attn_norm, *wq, *wk, *wv, *q_norm, *k_norm, *wo, *mlp_norm, *w_gate, *w_up, *w_down;
};

// split-K partials the scratch holds per GEMM output (QKV and gate / up; O and down)
constexpr int PF_SPLITS_WIDE = 4;
constexpr int PF_SPLITS_NARROW = 8;
// position splits of one query tile's cached positions (long prompts: more CTAs per layer)
constexpr int PF_ATTN_SPLITS = 4;
constexpr int PF_ATTN_SPLIT_MIN = 512;   // chunks ending past this many prompt positions split
// captured prefill graphs kept per handle (least recently used replaced)
constexpr int PF_MAX_GRAPHS = 8;

// scratch and tensor maps, owned by an mk_handle
struct PfState {
  int tc = 0;                       // tokens per chunk the scratch holds
  int sms = 0;                      // multiprocessors (split-K sizing)
  float *x = nullptr, *qkv = nullptr, *attn = nullptr, *attn_part = nullptr;
  float *qkv_p = nullptr, *y_p = nullptr;  // [splits][tc][N] GEMM partials
  float *gu_p = nullptr;            // [splits][tc][2 I]: gate columns, then up columns
  float *logits = nullptr;          // [logit_rows][V], allocated on the first LM head
  int logit_rows = 0;
  float *pv = nullptr;              // argmax candidates [tc][blocks]
  int *pi = nullptr;
  uint16_t *hs = nullptr;           // [3][tc][kmax] bf16 input terms
  size_t kmax = 0;
  int *err = nullptr;
  PfCall *call = nullptr;           // device copy of the current call
  cudaStream_t cap = nullptr;       // capture stream
  // TMA tensor maps: per layer {wq, wk, wv}, {wo}, {w_gate, w_up}, {w_down},
  // then the LM head; the input terms per (K in H, Hq d, I) x (token block 32, 64, 128)
  std::vector<mkg::WMaps> wmaps;
  CUtensorMap xmaps[3][3];
  // the KV cache as K and V tensors [L * Hkv * max_seq][d] for the tensor-core attention
  CUtensorMap kmap, vmap;
  bool kv_maps = false;
  struct Graph {
    int n;
    bool all_logits;
    unsigned long long used;
    cudaGraph_t graph;
    cudaGraphExec_t exec;
  };
  std::vector<Graph> graphs;        // captured prefills, at most PF_MAX_GRAPHS
  unsigned long long clock = 0;
};

int pf_init(PfState &st, int tc, int H, int Hq, int Hkv, int d, int I);

// Tensor-core causal attention of a chunk (csrc/mk_pfattn.cu): the maps of the
// KV cache (made once per handle), and one launch per layer and chunk.
bool attn_tc_maps(const PfArgs &a, CUtensorMap *tk, CUtensorMap *tv);
int attn_tc_launch(const CUtensorMap &tk, const CUtensorMap &tv, const PfArgs &a, int layer, int t0, int nt,
                   cudaStream_t s);
void pf_free(PfState &st);

// Run n prompt forwards (positions call.pos0 ..): fills the KV cache, writes
// hidden / logits / out_ids when given, and the last token's greedy id to
// *call.last_id (device).  The launch sequence of a given (n, all ids or not)
// is captured as a CUDA graph on first use and replayed afterwards.  Returns
// MK_OK or an MK_ERR_* code (after the stream has completed).
int pf_run(PfState &st, PfArgs a, const PfLayer *layers, const uint16_t *final_norm, const uint16_t *lm_head,
           int n, const PfCall &call, cudaStream_t s);

}  // namespace mkp
