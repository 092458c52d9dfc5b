// Launch parameters and shared-memory layout shared by the host library and
// the device code.
#pragma once
#include <cstdint>

#ifndef MK_NCW
#define MK_NCW 8
#endif

#ifndef MK_KPT_MAX
#define MK_KPT_MAX 8
#endif

namespace mk {

constexpr int KPT_MAX = MK_KPT_MAX;  // longest per-thread input slice the GEMV geometry may pick
constexpr int NCW = MK_NCW;          // consumer warps per CTA
constexpr int NCT = NCW * 32;        // consumer threads
constexpr int NTHREADS = NCT + 32;   // + one TMA producer warp
constexpr int MAX_STAGES = 8;
constexpr int MAX_LAYERS = 64;
constexpr int MAX_OWN = 64;          // residual rows one CTA may own (H / grid, rounded up)
constexpr int RED_ROWS = 64;         // rows of one GEMV epilogue batch
constexpr int MAX_WPR = 8;           // warps that share one row (threads per row / 32)
constexpr int MAX_GRP_HD = 256;      // group size * head_dim handled by one attention unit
constexpr int MAX_POLL_CHUNKS = 8;    // split-KV chunk counts the chunk holding the new position merges by polling
constexpr int MAX_STAGE_K = 2048;    // widest GEMV input staged in shared memory
constexpr int STAGE_BYTES = 32 * 1024;   // one slot of the weight ring

// GEMV phases in the order of their geometry table
enum GemvKind { GV_QKV = 0, GV_O = 1, GV_GU = 2, GV_DOWN = 3, GV_LM = 4, GV_COUNT = 5 };

// How a GEMV phase maps rows and the input width onto the consumer threads:
// thread t owns KPT consecutive input elements (k-chunk t % TPR) of NG = NCT/TPR
// row groups; a tile holds RT rows (GU: RT gate/up row pairs).
//
// Two layouts of a thread's slice exist.  The general one (fast == 0) gives
// thread kc the KPT consecutive elements [kc*KPT, (kc+1)*KPT) and reduces one
// tile at a time.  The fast ones give thread kc chunks of CH consecutive
// elements, chunk c at c*TPR*CH + kc*CH (every shared-memory load of a warp
// covers consecutive bytes), accumulate the row partials of BT tiles in
// registers and reduce once per batch of tiles:
//   fast == 1 (staged): TPR = 32, one warp per row; the CTA polls the input
//             once into shared memory (natural order) and every warp reads
//             the whole vector from there -- used for the RMSNorm-fused
//             phases, whose norm needs the whole vector anyway;
//   fast == 2 (split-K): TPR = 256, all consumer threads share each row; each
//             thread polls its own slice directly (no CTA barrier before the
//             tiles) -- used for the wide inputs of the O and down projections.
struct GemvGeom {
  int K;        // input width
  int KPT;      // input elements per thread
  int TPR;      // threads per row (32, 64, 128, 256)
  int NG;       // row groups = NCT / TPR
  int RT;       // rows (pairs for GU) per ring tile
  int RPTP;     // rows per thread per tile (general: padded to a power of two, <= 16)
  int rows;     // total rows (pairs for GU) of the phase
  int fast;     // 0 general, 1 staged, 2 split-K (see above)
  int CH;       // fast layouts: consecutive elements per chunk (4 or 8)
  int BT;       // fast layouts: tiles per register batch
  int lgCH, lgSpan;   // split-K layout: log2 of CH and of TPR * CH
  int lgRT;     // log2 of RT when RT is a power of two, else -1
  float invK;   // 1 / K when K is a power of two (exact), else 0 (divide)
};

struct LayerPtrs {
  const uint16_t *attn_norm, *wq, *wk, *wv, *q_norm, *k_norm, *wo;
  const uint16_t *mlp_norm, *w_gate, *w_up, *w_down;
};

// Activations crossing CTAs travel as 64-bit words {float value, 32-bit tag};
// the tag names the forward that wrote them, so a reader polls a word until it
// carries the tag it expects.  One buffer per layer and kind, reused only by
// the next forward (after the grid barrier that closes every forward).
struct LLBuffers {
  unsigned long long *qkv;    // [L][(Hq + 2 Hkv) d]  raw q, k, v
  unsigned long long *attn;   // [L][Hq d]            attention output
  unsigned long long *xmid;   // [L][H]               residual after attention
  unsigned long long *u;      // [L][I]               SiLU(gate) * up
  unsigned long long *xout;   // [L][H]               residual after the MLP
  unsigned long long *part;   // [L][MAX_POLL_CHUNKS][Hq][d + 2]  chunk outputs, then running max and sum
};

// The call-dependent launch fields.  A replayed CUDA graph of the per-op path
// cannot change its kernels' parameters, so its launches read these from a
// device copy the host refreshes before each call; op_fwd advances by one
// after every forward of the graph.
struct CallBlock {
  const int32_t *in_ids;
  int32_t *out_ids;
  const float *embeds;
  const int32_t *pos3;
  float *logits, *hidden;
  unsigned long long *trace;
  int32_t *mbox_ids;
  int *mbox_count;
  long long spin_ns;
  const uint16_t *cb_books, *cb_text;
  const int32_t *cb_codes, *cb_text_ids;
  int cb_n, cb_rows, cb_text_rows, cb_n_rows;
  int n_in, n_fwd, pos0, n_embed_rows, chunks_override, op_fwd;
  unsigned tag0;
};

struct Params {
  // shape
  int L, H, Hq, Hkv, d, I, V, vocab_in, grp;
  float eps, inv_sqrt_d;
  int rope_mode, sec_b0, sec_b1;   // mode 2 (interleaved) uses sec1, sec2
  int sec1, sec2;   // pair i < sec_b0 -> stream 0, < sec_b1 -> 1, else 2
  int max_seq, rope_len, max_chunks;
  // weights (borrowed)
  const LayerPtrs *layers;
  const uint16_t *embed, *lm_head, *final_norm;
  // handle-owned state and scratch
  uint16_t *kcache, *vcache;       // [L][Hkv][max_seq][d]
  const float2 *rope;              // [rope_len][d/2] (cos, sin)
  LLBuffers ll;
  int ll_rep;                      // copies of every tagged buffer (readers spread over them)
  unsigned long long ll_cs;        // words between copies
  int poll_ns;                     // back-off between unsuccessful polls
  float *part, *cand_val;
  int *cand_idx;
  unsigned *tickets;               // [Hkv]
  unsigned *bar;                   // grid-barrier counter (zeroed before each launch)
  int *err;                        // first error code
  int *last_id;
  // this call
  const int32_t *in_ids;
  int n_in, n_fwd, pos0;
  unsigned tag0;                   // tag of forward 0 of this call (nonzero, increasing)
  int32_t *out_ids;
  const float *embeds;
  int n_embed_rows;
  const int32_t *pos3;
  float *logits, *hidden;
  unsigned long long *trace;
  int32_t *mbox_ids;               // streaming mailbox (host-mapped), or NULL
  int *mbox_count;
  // talker inputs summed in-kernel (negative ids select code rows), or cb_codes NULL
  const uint16_t *cb_books, *cb_text;
  const int32_t *cb_codes, *cb_text_ids;
  int cb_n, cb_rows, cb_text_rows, cb_n_rows;
  int chunks_override;
  int poll_cm;                     // chunk counts in (1, poll_cm] merge by polling; more: ticket merge
  int attn_ppc;                    // target cached positions per split-KV chunk (0: one chunk per CTA share)
  int attn_min_chunks;             // chunks of a short context (fewer than attn_ppc positions each)
  int attn_short_ppc;              // and at least ceil(ctx / this) chunks, up to poll_cm
  long long spin_ns;
  int fault_barrier;
  int G;                           // CTAs
  int stages, stage_bytes;
  // per-op path: one launch runs phase `op_phase` of forward `op_fwd`
  int per_op, op_fwd, op_phase;
  const CallBlock *blk;            // per-op graph replay: call fields come from here (else NULL)
  GemvGeom geo[GV_COUNT];
};

// flags shared inside a CTA between the consumer warps and the producer lane
enum SmemFlag { F_ABORT = 0, F_PROD_DONE = 1, F_FWD_DONE = 2, F_LAST = 3, F_COUNT = 8 };

// static part of the dynamic shared memory; the weight ring follows at RING_OFFSET
struct SmemCtl {
  Params prm;                            // launch parameters, copied at kernel start
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  LayerPtrs layers[MAX_LAYERS];          // pointer table copied at kernel start
  float red[2][RED_ROWS][MAX_WPR];       // per-warp row partials of one epilogue batch
  float misc[64];
  float xown[MAX_OWN];                   // residual rows this CTA owns
  int rr[GV_COUNT][2];                   // this CTA's row range of every GEMV phase
  int nt[GV_COUNT];                      // and its tile count (RT rows a tile)
  int flags[F_COUNT];
  float bestv[NCW];
  int besti[NCW];
  float qs[MAX_GRP_HD];                  // normed, rotated, scaled queries of one unit
  uint16_t kcur[128], vcur[128];         // this position's key / value (bf16, as cached)
  float ow[NCW][MAX_GRP_HD];             // per-warp unnormalised attention outputs
  float mw[NCW][8], lw[NCW][8];          // per-warp running max / sum per head
  alignas(16) float xs[MAX_STAGE_K];     // staged GEMV input (fast layout 1)
};

constexpr int RING_OFFSET = (int)((sizeof(SmemCtl) + 1023) / 1024 * 1024);

}  // namespace mk
