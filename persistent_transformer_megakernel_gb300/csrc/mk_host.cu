// Host side of libmk.so: the C ABI declared in include/mk.h.
//
// mk_create validates the shape, fixes the GEMV thread geometry of every phase,
// allocates the KV cache and scratch, builds the rotary cos/sin table on the
// host in double precision (page B = "I made a single CUDA kernel speak:
// streaming Qwen3-TTS at 50ms latency on an RTX 5090", section "So, What's the
// Catch with These Megakernels?": the rotary frequencies are host-built tables)
// and checks that one
// CTA per SM fits.  mk_decode runs all forwards of a call in one cooperative
// launch (page A = "Porting a 1,200-line persistent CUDA megakernel to
// Qwen3-TTS", section "The idea: one kernel that never exits"), or, with
// MK_DECODE_PER_OP, one ordinary launch per phase.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/mk.h"
#include "mk_launch.h"
#include "mk_prefill.h"
#include "mk_params.h"
#include "mk_plans.h"

namespace {

constexpr int kStageBytes = mk::STAGE_BYTES;
constexpr int kMaxStagesWanted = 6;
// split-KV: MAX_POLL_CHUNKS chunks up to MAX_POLL_CHUNKS * this many cached
// positions, one chunk per this many beyond
constexpr int kAttnPositionsPerChunk = 256;
// split-KV chunks of a short context: at least 4, and one per 48 positions up
// to the 8 that merge by polling (measured on the 0.6B shape, us/token with a
// fixed chunk count 1/2/3/4/6/8: 564/538/530/522/522/523 at 33..288 cached
// positions, -/579/552/540/533/532 at 33..544)
constexpr int kShortContextChunks = 4;
constexpr int kShortPositionsPerChunk = 48;
constexpr int kMinChunks = 64;
   // split-KV chunk capacity per kv head (at least grid / Hkv)

struct DeviceBuffers {
  std::vector<void *> owned;
  int alloc(void **p, size_t bytes) {
    if (bytes == 0) bytes = 16;
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) {
      cudaGetLastError();
      *p = nullptr;
      return e == cudaErrorMemoryAllocation ? MK_ERR_NO_MEMORY : MK_ERR_CUDA;
    }
    owned.push_back(*p);
    return MK_OK;
  }
  void free_all() {
    for (void *p : owned) cudaFree(p);
    owned.clear();
  }
};

// input elements per thread and threads per row of a GEMV with input width K:
// K = KPT * TPR with TPR a whole number of warps dividing the consumer threads;
// the largest KPT up to MK_KPT_MAX (fewer, longer per-thread dot products)
int choose_kpt(int K, int &kpt, int &tpr) {
  static const int kpts[] = {48, 32, 24, 16, 12, 8};
  auto ok = [&](int c) {
    if (K % c) return false;
    const int t = K / c;
    return t >= 32 && t <= mk::NCT && t % 32 == 0 && mk::NCT % t == 0;
  };
  for (int c : kpts)                       // widest slice allowed
    if (c <= mk::KPT_MAX && ok(c)) { kpt = c; tpr = K / c; return MK_OK; }
  for (int i = 5; i >= 0; --i)             // otherwise the narrowest that fits
    if (ok(kpts[i])) { kpt = kpts[i]; tpr = K / kpts[i]; return MK_OK; }
  return MK_ERR_UNSUPPORTED;
}

int pow2_at_least(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

// thread geometry of one GEMV phase: K input width, rows (pairs for gate/up)
int make_geom(int K, int rows, bool pairs, mk::GemvGeom &g) {
  int kpt, tpr;
  if (choose_kpt(K, kpt, tpr) != MK_OK) return MK_ERR_UNSUPPORTED;
  std::memset(&g, 0, sizeof(g));
  g.K = K;
  g.KPT = kpt;
  g.TPR = tpr;
  g.BT = 1;
  g.NG = mk::NCT / tpr;
  const int rows_fit = kStageBytes / (K * 2);
  if (pairs) {
    g.RT = std::min(rows_fit / 2, 8 * g.NG);
    if (g.RT < 1) return MK_ERR_UNSUPPORTED;
    g.RPTP = pow2_at_least((2 * g.RT + g.NG - 1) / g.NG);
  } else {
    g.RT = std::min(rows_fit, 16 * g.NG);
    if (g.RT < 1) return MK_ERR_UNSUPPORTED;
    g.RPTP = pow2_at_least((g.RT + g.NG - 1) / g.NG);
  }
  if (g.RPTP > 16 || g.KPT * g.RPTP > 128) {
    // too many rows per thread for this width: a smaller tile keeps the registers in bounds
    while (g.RPTP > 1 && g.KPT * g.RPTP > 128) {
      g.RPTP /= 2;
      g.RT = pairs ? std::min(g.RT, g.RPTP * g.NG / 2) : std::min(g.RT, g.RPTP * g.NG);
    }
    if (g.RT < 1 || g.KPT * g.RPTP > 128) return MK_ERR_UNSUPPORTED;
  }
  g.rows = rows;
  return MK_OK;
}

// The fast GEMV layouts compiled into the kernel (mk_device.cuh, gemv_dispatch):
// {layout, KPT, rows per thread per tile, tiles per register batch}
// The kernel for these layouts: a plan kernel whose compiled layouts and
// attention group size are exactly these, else the general kernel.
template <class PL>
bool plan_matches(int d, int grp, const mk::GemvGeom *geo) {
  if (PL::hd != d || PL::grp != grp) return false;
  for (int k = 0; k < mk::GV_COUNT; ++k) {
    const mk::GemvGeom &g = geo[k];
    if (g.fast != PL::spec[k][0] || g.KPT != PL::spec[k][1] || g.RPTP != PL::spec[k][2] || g.BT != PL::spec[k][3])
      return false;
  }
  return true;
}
// plan id (mk_info.plan): 1 PlanHidden1024, 2 PlanHidden2048, 0 the general kernel
int pick_plan(int d, int grp, const mk::GemvGeom *geo) {
  if (plan_matches<mk::PlanHidden1024>(d, grp, geo)) return 1;
  if (plan_matches<mk::PlanHidden2048>(d, grp, geo)) return 2;
  return 0;
}
const void *plan_kernel(int plan, int d) {
  if (plan == 1) return mk::kernel_hidden1024();
  if (plan == 2) return mk::kernel_hidden2048();
  return d == 64 ? mk::kernel_d64() : mk::kernel_d128();
}

// {fast (1 staged, 2 split-K), KPT, rows per thread per tile, tiles per
// batch}.  Tiles per batch set how much of the tile loop is unrolled: the
// staged layouts at width 1024 and 2048 were swept on the GB300 (0.6B: 1 and
// 2 equal, 4 slower by 9%; 1.7B: 4 fastest, 1/2/8 slower by 9/4/10%); the
// results do not depend on it.
struct FastCase { int fast, kpt, rpt, bt; };
const FastCase kFastCases[] = {{1, 32, 2, 2}, {1, 64, 1, 4}, {1, 16, 4, 2}, {1, 24, 2, 4}, {1, 8, 8, 1},
                               {2, 8, 8, 1},  {2, 8, 8, 2},  {2, 12, 4, 2}, {2, 24, 2, 8}};

// A fast layout for one GEMV phase, if one fits: the RMSNorm-fused phases
// (QKV, gate/up, LM head) take the staged layout (one warp per row, the input
// staged in shared memory), the O and down projections the split-K layout
// (all consumer threads per row).  Returns false to keep the general layout.
bool make_fast_geom(int kind, int K, int rows, int G, mk::GemvGeom &g) {
  const bool normed = kind == mk::GV_QKV || kind == mk::GV_GU || kind == mk::GV_LM;
  const bool pairs = kind == mk::GV_GU;
  const int per_cta = (rows + G - 1) / G;
  const FastCase *best = nullptr;
  for (const FastCase &c : kFastCases) {
    if (normed) {
      if (c.fast != 1 || K != 32 * c.kpt || K > mk::MAX_STAGE_K) continue;
      if (static_cast<long long>(mk::NCW) * c.rpt * K * 2 > kStageBytes) continue;   // 8 * RPT rows a tile
      best = &c;
      break;
    }
    if (c.fast != 2 || K != mk::NCT * c.kpt || c.kpt % 4) continue;
    if (static_cast<long long>(c.rpt) * K * 2 > kStageBytes) continue;              // RPT rows a tile
    // the fewest register slots that still hold every tile of a CTA, else the most
    const int tiles = (per_cta + c.rpt - 1) / c.rpt;
    if (!best) { best = &c; continue; }
    const bool fits = tiles <= c.bt, best_fits = (per_cta + best->rpt - 1) / best->rpt <= best->bt;
    if ((fits && (!best_fits || c.rpt * c.bt < best->rpt * best->bt)) ||
        (!fits && !best_fits && c.rpt * c.bt > best->rpt * best->bt))
      best = &c;
  }
  if (!best) return false;
  g.K = K;
  g.KPT = best->kpt;
  g.fast = best->fast;
  g.CH = (best->kpt % 8 == 0) ? 8 : 4;
  g.BT = best->bt;
  g.RPTP = best->rpt;
  g.rows = rows;
  if (best->fast == 1) {
    g.TPR = 32;
    g.NG = mk::NCW;
    g.RT = pairs ? mk::NCW * best->rpt / 2 : mk::NCW * best->rpt;
  } else {
    g.TPR = mk::NCT;
    g.NG = 1;
    g.RT = best->rpt;
  }
  return true;
}

// log2 of v when v is a power of two, else -1
int log2_exact(int v) {
  if (v <= 0 || (v & (v - 1))) return -1;
  int l = 0;
  while ((1 << l) < v) ++l;
  return l;
}

// the shift amounts the device code uses in place of divisions
void fill_shifts(mk::GemvGeom &g) {
  g.lgRT = log2_exact(g.RT);
  g.invK = log2_exact(g.K) >= 0 ? 1.0f / static_cast<float>(g.K) : 0.0f;
  g.lgCH = g.fast == 2 ? log2_exact(g.CH) : 0;
  g.lgSpan = g.fast == 2 ? log2_exact(g.TPR * g.CH) : 0;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

struct mk_handle {
  mk_config cfg;
  int device = 0;
  int G = 0;
  int smem = 0;
  int pos = 0;
  int max_chunks = 0;
  int stages = 0;
  int ll_rep = 1;             // copies of every tagged buffer; one measured fastest
  unsigned tag = 1;          // tag of the next forward's published activations
  size_t ll_words = 0;
  unsigned long long *ll_base = nullptr;
  int64_t weight_bytes = 0, kv_bytes = 0;
  const void *kernel = nullptr;
  DeviceBuffers buf;
  mk::Params base;      // call-independent launch parameters
  int *d_sync = nullptr;       // [0] barrier counter, [1] error word, [2] last id
  int32_t *d_ids_in = nullptr, *d_ids_out = nullptr;
  // batched prompt prefill: host copy of the layer pointers, scratch, GEMM handle
  std::vector<mkp::PfLayer> pf_layers;
  mkp::PfState pf;
  // streaming mailbox: host-mapped pinned ints, [0] count, ids from [32]
  int32_t *mbox = nullptr, *d_mbox = nullptr;
  // a launch started by mk_decode_start and not yet waited for
  int pending = 0, pending_fwd = 0;
  cudaStream_t pending_stream = nullptr;
  // per-op ablation under CUDA graph replay: one forward's launches, captured once
  mk::CallBlock *d_blk = nullptr;
  cudaStream_t cap = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t gexec = nullptr;
};

namespace {

// advances the replayed graph to the next forward
__global__ void mk_advance_forward(mk::CallBlock *b) { b->op_fwd += 1; }

// capture the per-op launches of one forward (every phase, then the advance)
int build_forward_graph(mk_handle *h) {
  if (h->gexec) return MK_OK;
  if (!h->cap && cudaStreamCreateWithFlags(&h->cap, cudaStreamNonBlocking) != cudaSuccess) return MK_ERR_CUDA;
  mk::Params p = h->base;
  p.per_op = 1;
  p.fault_barrier = -1;
  p.blk = h->d_blk;
  const int nph = 5 * p.L + 1;
  void *args[] = {&p};
  cudaError_t e = cudaStreamBeginCapture(h->cap, cudaStreamCaptureModeThreadLocal);
  for (int ph = 0; ph < nph && e == cudaSuccess; ++ph) {
    p.op_phase = ph;
    e = cudaLaunchKernel(h->kernel, dim3(h->G), dim3(mk::NTHREADS), args, h->smem, h->cap);
  }
  if (e == cudaSuccess) {
    mk_advance_forward<<<1, 1, 0, h->cap>>>(h->d_blk);
    e = cudaGetLastError();
  }
  cudaGraph_t g = nullptr;
  const cudaError_t e2 = cudaStreamEndCapture(h->cap, &g);
  if (e == cudaSuccess) e = e2;
  if (e == cudaSuccess) e = cudaGraphInstantiate(&h->gexec, g, 0);
  if (e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    h->gexec = nullptr;
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  h->graph = g;
  return MK_OK;
}

}  // namespace

// the shape checks of mk_create (everything but the weight pointers)
int check_shape(const mk_config &c) {
  if (c.n_layers < 1 || c.hidden < 1 || c.n_q_heads < 1 || c.n_kv_heads < 1 || c.head_dim < 1 ||
      c.intermediate < 1 || c.vocab < 1 || c.vocab_in < 1 || c.max_seq < 1 || c.rope_positions < 0 ||
      !(c.rms_eps >= 0.f) || !(c.rope_theta > 0.f) || c.flags != 0)
    return MK_ERR_INVALID_ARG;
  if (c.head_dim != 64 && c.head_dim != 128) return MK_ERR_UNSUPPORTED;
  if (c.n_q_heads % c.n_kv_heads) return MK_ERR_UNSUPPORTED;
  const int grp = c.n_q_heads / c.n_kv_heads;
  if (grp != 1 && grp != 2 && grp != 4 && grp != 8) return MK_ERR_UNSUPPORTED;
  if (grp * c.head_dim > mk::MAX_GRP_HD) return MK_ERR_UNSUPPORTED;
  if (c.n_layers > mk::MAX_LAYERS) return MK_ERR_UNSUPPORTED;
  if (c.rope_mode < 0 || c.rope_mode > 2) return MK_ERR_INVALID_ARG;
  if (c.rope_mode != 0) {
    if (c.mrope_sections[0] < 0 || c.mrope_sections[1] < 0 || c.mrope_sections[2] < 0 ||
        c.mrope_sections[0] + c.mrope_sections[1] + c.mrope_sections[2] != c.head_dim / 2)
      return MK_ERR_INVALID_ARG;
  }
  return MK_OK;
}

// the GEMV geometry of every phase for G CTAs: the general layouts, then a
// fast layout for each phase where one fits
int choose_geometry(const mk_config &c, int G, mk::GemvGeom *geo) {
  const int H = c.hidden, d = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads, I = c.intermediate;
  if (make_geom(H, (Hq + 2 * Hkv) * d, false, geo[mk::GV_QKV]) ||
      make_geom(Hq * d, H, false, geo[mk::GV_O]) ||
      make_geom(H, I, true, geo[mk::GV_GU]) ||
      make_geom(I, H, false, geo[mk::GV_DOWN]) ||
      make_geom(H, c.vocab, false, geo[mk::GV_LM]))
    return MK_ERR_UNSUPPORTED;
  // the residual stream is stored in the input layout of its readers (next
  // layer's QKV and the LM head): both must split H the same way
  if (geo[mk::GV_LM].fast != geo[mk::GV_QKV].fast || geo[mk::GV_LM].KPT != geo[mk::GV_QKV].KPT || geo[mk::GV_LM].TPR != geo[mk::GV_QKV].TPR)
    return MK_ERR_UNSUPPORTED;

  {
    // fast layouts where one fits (the general ones above stay otherwise)
    const int Ks[mk::GV_COUNT] = {H, Hq * d, H, I, H};
    const int rows[mk::GV_COUNT] = {(Hq + 2 * Hkv) * d, H, I, H, c.vocab};
    mk::GemvGeom fg[mk::GV_COUNT];
    bool ok[mk::GV_COUNT];
    for (int k = 0; k < mk::GV_COUNT; ++k) {
      std::memset(&fg[k], 0, sizeof(fg[k]));
      ok[k] = make_fast_geom(k, Ks[k], rows[k], G, fg[k]);
    }
    // the residual stream's layout is read by both the next layer's QKV and the
    // LM head: either both take the staged layout or neither does
    if (ok[mk::GV_QKV] != ok[mk::GV_LM]) ok[mk::GV_QKV] = ok[mk::GV_LM] = false;
    for (int k = 0; k < mk::GV_COUNT; ++k) {
      if (ok[k]) geo[k] = fg[k];
      fill_shifts(geo[k]);
      if (geo[k].fast == 2 && (geo[k].lgCH < 0 || geo[k].lgSpan < 0)) return MK_ERR_UNSUPPORTED;
    }
  }
  return MK_OK;
}

extern "C" {

const char *mk_error_string(int code) {
  switch (code) {
    case MK_OK: return "ok";
    case MK_ERR_INVALID_ARG: return "invalid argument";
    case MK_ERR_UNSUPPORTED: return "unsupported shape or launch geometry";
    case MK_ERR_KV_FULL: return "KV cache full";
    case MK_ERR_BAD_TOKEN: return "token id or sentinel row out of range";
    case MK_ERR_TIMEOUT: return "device wait timed out";
    case MK_ERR_NUMERIC: return "non-finite logit";
    case MK_ERR_CUDA: return "CUDA runtime error";
    case MK_ERR_NO_MEMORY: return "device out of memory";
    case MK_ERR_BAD_POSITION: return "position stream outside the rotary table";
    default: return "unknown error";
  }
}

int mk_create(const mk_config *cfg, const mk_weights *w, mk_handle **out) {
  if (!cfg || !w || !out) return MK_ERR_INVALID_ARG;
  *out = nullptr;
  const mk_config c = *cfg;
  if (int rc0 = check_shape(c)) return rc0;
  const int grp = c.n_q_heads / c.n_kv_heads;
  if (!w->embed || !w->final_norm || !w->layers) return MK_ERR_INVALID_ARG;
  if (!w->lm_head && c.vocab != c.vocab_in) return MK_ERR_INVALID_ARG;
  if (!aligned16(w->embed) || !aligned16(w->final_norm) || (w->lm_head && !aligned16(w->lm_head)))
    return MK_ERR_INVALID_ARG;
  for (int l = 0; l < c.n_layers; ++l) {
    const mk_layer_weights &L = w->layers[l];
    const void *ps[] = {L.attn_norm, L.wq, L.wk, L.wv, L.q_norm, L.k_norm, L.wo, L.mlp_norm, L.w_gate, L.w_up, L.w_down};
    for (const void *q : ps)
      if (!q || !aligned16(q)) return MK_ERR_INVALID_ARG;
  }
  const int H = c.hidden, d = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads, I = c.intermediate;

  mk::GemvGeom geo[mk::GV_COUNT];
  mk_handle *h = new (std::nothrow) mk_handle();
  if (!h) return MK_ERR_NO_MEMORY;
  h->cfg = c;
  int rc = MK_OK;
  auto fail = [&](int code) {
    h->buf.free_all();
    delete h;
    return code;
  };
  if (cudaGetDevice(&h->device) != cudaSuccess) return fail(MK_ERR_CUDA);
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, h->device) != cudaSuccess) return fail(MK_ERR_CUDA);
  int coop = 0;
  cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->device);
  if (!coop) return fail(MK_ERR_UNSUPPORTED);
  h->G = prop.multiProcessorCount;
  if (int rc1 = choose_geometry(c, h->G, geo)) return fail(rc1);
  h->kernel = plan_kernel(pick_plan(d, Hq / Hkv, geo), d);
  // residual rows owned per CTA, and rows of every phase, must fit the static buffers
  if ((H + h->G - 1) / h->G > mk::MAX_OWN) return fail(MK_ERR_UNSUPPORTED);
  for (int k = 0; k < mk::GV_COUNT; ++k) {
    const int trow = (k == mk::GV_GU) ? 2 * geo[k].RT : geo[k].RT;
    if (trow > mk::RED_ROWS || geo[k].TPR / 32 > mk::MAX_WPR) return fail(MK_ERR_UNSUPPORTED);
  }
  h->stages = std::min(kMaxStagesWanted,
                       (static_cast<int>(prop.sharedMemPerBlockOptin) - mk::RING_OFFSET) / kStageBytes);
  if (h->stages < 2) return fail(MK_ERR_UNSUPPORTED);
  h->smem = mk::RING_OFFSET + h->stages * kStageBytes;
  if (cudaFuncSetAttribute(h->kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, h->smem) != cudaSuccess) {
    cudaGetLastError();
    return fail(MK_ERR_CUDA);
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, h->kernel, mk::NTHREADS, h->smem) != cudaSuccess ||
      per_sm < 1) {
    cudaGetLastError();
    return fail(MK_ERR_UNSUPPORTED);
  }
  h->max_chunks = std::max(kMinChunks, h->G / Hkv);
  // one copy of the tagged activation buffers (more copies, read by CTA index,
  // measured slower: every producer then stores each word several times) and
  // no back-off in the polls (any sleep measured slower)
  h->ll_rep = 1;
  const int poll_ns = 0;
  const int attn_ppc = kAttnPositionsPerChunk;

  // ---- allocations ---------------------------------------------------------
  const int rope_len = c.rope_positions > 0 ? c.rope_positions : 2 * c.max_seq + 8;
  const size_t kv_elems = static_cast<size_t>(c.n_layers) * Hkv * c.max_seq * d;
  mk::LayerPtrs *d_layers = nullptr;
  uint16_t *kc = nullptr, *vc = nullptr;
  float2 *rope = nullptr;
  float *part = nullptr, *cand_val = nullptr;
  int *cand_idx = nullptr;
  unsigned *tickets = nullptr;
  if ((rc = h->buf.alloc((void **)&d_layers, sizeof(mk::LayerPtrs) * c.n_layers)) ||
      (rc = h->buf.alloc((void **)&kc, kv_elems * 2)) ||
      (rc = h->buf.alloc((void **)&vc, kv_elems * 2)) ||
      (rc = h->buf.alloc((void **)&rope, sizeof(float2) * static_cast<size_t>(rope_len) * (d / 2))) ||
      (rc = h->buf.alloc((void **)&h->ll_base, sizeof(unsigned long long) *
                         (h->ll_words = static_cast<size_t>(c.n_layers) *
                                        ((Hq + 2 * Hkv) * d + Hq * d + 2 * H + I +
                                         mk::MAX_POLL_CHUNKS * Hq * (d + 2))) *
                         h->ll_rep)) ||
      (rc = h->buf.alloc((void **)&part, sizeof(float) * static_cast<size_t>(Hq) * h->max_chunks * (d + 2))) ||
      (rc = h->buf.alloc((void **)&cand_val, sizeof(float) * h->G)) ||
      (rc = h->buf.alloc((void **)&cand_idx, sizeof(int) * h->G)) ||
      (rc = h->buf.alloc((void **)&tickets, sizeof(unsigned) * Hkv)) ||
      (rc = h->buf.alloc((void **)&h->d_sync, sizeof(int) * 4)) ||
      (rc = h->buf.alloc((void **)&h->d_ids_in, sizeof(int32_t) * c.max_seq)) ||
      (rc = h->buf.alloc((void **)&h->d_ids_out, sizeof(int32_t) * c.max_seq)) ||
      (rc = h->buf.alloc((void **)&h->d_blk, sizeof(mk::CallBlock))))
    return fail(rc);

  std::vector<mk::LayerPtrs> lp(c.n_layers);
  for (int l = 0; l < c.n_layers; ++l) {
    const mk_layer_weights &L = w->layers[l];
    lp[l] = mk::LayerPtrs{(const uint16_t *)L.attn_norm, (const uint16_t *)L.wq, (const uint16_t *)L.wk,
                          (const uint16_t *)L.wv, (const uint16_t *)L.q_norm, (const uint16_t *)L.k_norm,
                          (const uint16_t *)L.wo, (const uint16_t *)L.mlp_norm, (const uint16_t *)L.w_gate,
                          (const uint16_t *)L.w_up, (const uint16_t *)L.w_down};
  }
  h->pf_layers.resize(c.n_layers);
  for (int l = 0; l < c.n_layers; ++l)
    h->pf_layers[l] = mkp::PfLayer{lp[l].attn_norm, lp[l].wq, lp[l].wk, lp[l].wv, lp[l].q_norm, lp[l].k_norm,
                                   lp[l].wo, lp[l].mlp_norm, lp[l].w_gate, lp[l].w_up, lp[l].w_down};
  // rotary table: cos/sin(pos * theta^(-2i/d)) evaluated in double
  std::vector<float2> tab(static_cast<size_t>(rope_len) * (d / 2));
  for (int pos = 0; pos < rope_len; ++pos)
    for (int i = 0; i < d / 2; ++i) {
      const double omega = std::pow(static_cast<double>(c.rope_theta), -2.0 * i / d);
      const double phi = pos * omega;
      tab[static_cast<size_t>(pos) * (d / 2) + i] = make_float2(static_cast<float>(std::cos(phi)),
                                                                static_cast<float>(std::sin(phi)));
    }
  if (cudaMemcpy(d_layers, lp.data(), sizeof(mk::LayerPtrs) * c.n_layers, cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemcpy(rope, tab.data(), sizeof(float2) * tab.size(), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaMemset(tickets, 0, sizeof(unsigned) * Hkv) != cudaSuccess ||
      cudaMemset(h->d_sync, 0, sizeof(int) * 4) != cudaSuccess ||
      cudaMemset(kc, 0, kv_elems * 2) != cudaSuccess || cudaMemset(vc, 0, kv_elems * 2) != cudaSuccess ||
      cudaMemset(h->ll_base, 0, sizeof(unsigned long long) * h->ll_words * h->ll_rep) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return fail(MK_ERR_CUDA);
  }

  mk::Params &p = h->base;
  std::memset(&p, 0, sizeof(p));
  p.L = c.n_layers; p.H = H; p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.I = I; p.V = c.vocab; p.vocab_in = c.vocab_in;
  p.grp = grp;
  p.eps = c.rms_eps;
  p.inv_sqrt_d = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  p.rope_mode = c.rope_mode;
  p.sec_b0 = c.rope_mode ? c.mrope_sections[0] : d / 2;
  p.sec_b1 = c.rope_mode ? c.mrope_sections[0] + c.mrope_sections[1] : d / 2;
  p.sec1 = c.rope_mode ? c.mrope_sections[1] : 0;
  p.sec2 = c.rope_mode ? c.mrope_sections[2] : 0;
  p.max_seq = c.max_seq;
  p.rope_len = rope_len;
  p.max_chunks = h->max_chunks;
  p.layers = d_layers;
  p.embed = (const uint16_t *)w->embed;
  p.lm_head = (const uint16_t *)(w->lm_head ? w->lm_head : w->embed);
  p.final_norm = (const uint16_t *)w->final_norm;
  p.kcache = kc; p.vcache = vc; p.rope = rope;
  {
    unsigned long long *q = h->ll_base;
    const size_t Lc = static_cast<size_t>(c.n_layers);
    p.ll.qkv = q;  q += Lc * (Hq + 2 * Hkv) * d;
    p.ll.attn = q; q += Lc * Hq * d;
    p.ll.xmid = q; q += Lc * H;
    p.ll.u = q;    q += Lc * I;
    p.ll.xout = q; q += Lc * H;
    p.ll.part = q;
  }
  p.ll_rep = h->ll_rep;
  p.ll_cs = h->ll_words;
  p.poll_ns = poll_ns;
  p.attn_ppc = attn_ppc;
  p.poll_cm = mk::MAX_POLL_CHUNKS;
  p.attn_min_chunks = kShortContextChunks;
  p.attn_short_ppc = kShortPositionsPerChunk;
  p.part = part;
  p.cand_val = cand_val; p.cand_idx = cand_idx; p.tickets = tickets;
  p.bar = reinterpret_cast<unsigned *>(h->d_sync);
  p.err = h->d_sync + 1;
  p.last_id = h->d_sync + 2;
  p.G = h->G;
  p.stages = h->stages;
  p.stage_bytes = kStageBytes;
  for (int k = 0; k < mk::GV_COUNT; ++k) p.geo[k] = geo[k];

  const int64_t layer_params = static_cast<int64_t>(H) * (Hq + 2 * Hkv) * d + static_cast<int64_t>(Hq) * d * H +
                               3LL * H * I + 2LL * H + 2LL * d;
  h->weight_bytes = 2 * (layer_params * c.n_layers + static_cast<int64_t>(c.vocab) * H + H);
  h->kv_bytes = static_cast<int64_t>(kv_elems) * 4;
  if (cudaHostAlloc(reinterpret_cast<void **>(&h->mbox), sizeof(int32_t) * (32 + static_cast<size_t>(c.max_seq)),
                    cudaHostAllocMapped) != cudaSuccess) {
    cudaGetLastError();
    h->mbox = nullptr;
    return fail(MK_ERR_NO_MEMORY);
  }
  std::memset(h->mbox, 0, sizeof(int32_t) * (32 + static_cast<size_t>(c.max_seq)));
  if (cudaHostGetDevicePointer(reinterpret_cast<void **>(&h->d_mbox), h->mbox, 0) != cudaSuccess) {
    cudaGetLastError();
    cudaFreeHost(h->mbox);
    h->mbox = nullptr;
    return fail(MK_ERR_CUDA);
  }
  *out = h;
  return MK_OK;
}

int mk_reset_kv(mk_handle *h, mk_stream stream) {
  if (!h || h->pending) return MK_ERR_INVALID_ARG;
  h->pos = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(h->d_sync, 0, sizeof(int) * 4, s) != cudaSuccess ||
      cudaMemsetAsync(h->base.tickets, 0, sizeof(unsigned) * h->cfg.n_kv_heads, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  return MK_OK;
}

int mk_decode_start(mk_handle *h, const int32_t *d_in_ids, int32_t n_in, int32_t n_steps, int32_t *d_out_ids,
                    const mk_decode_opts *opts, mk_stream stream) {
  if (!h || h->pending || n_in < 0 || n_steps < 0) return MK_ERR_INVALID_ARG;
  // forwards counted in 64 bits: two int32 counts may not fit an int together
  if (static_cast<int64_t>(h->pos) + n_in + n_steps > h->cfg.max_seq) return MK_ERR_KV_FULL;
  const int n_fwd = n_in + n_steps;
  if (n_fwd == 0) {
    h->pending = 1;
    h->pending_fwd = 0;
    h->pending_stream = reinterpret_cast<cudaStream_t>(stream);
    return MK_OK;
  }
  if (!d_out_ids || (n_in > 0 && !d_in_ids)) return MK_ERR_INVALID_ARG;
  mk_decode_opts o;
  std::memset(&o, 0, sizeof(o));
  if (opts) o = *opts;
  if (o.fault_skip_barrier < 0) return MK_ERR_INVALID_ARG;
  if (o.n_embed_rows < 0 || o.attn_chunks < 0 || o.attn_chunks > h->max_chunks || o.spin_ns < 0 ||
      (o.flags & ~(MK_DECODE_PER_OP | MK_DECODE_PER_OP_GRAPH | MK_DECODE_STREAM)) ||
      (o.n_embed_rows > 0 && !o.embeds))
    return MK_ERR_INVALID_ARG;
  if (o.codes && (o.embeds || o.n_books < 0 || o.n_books > 64 || (o.n_books > 0 && (!o.books || o.book_rows < 1)) ||
                  !o.text || o.text_rows < 1 || !o.text_ids || o.n_code_rows < 0))
    return MK_ERR_INVALID_ARG;
  if (cudaSetDevice(h->device) != cudaSuccess) return MK_ERR_CUDA;

  mk::Params p = h->base;
  p.in_ids = d_in_ids;
  p.n_in = n_in;
  p.n_fwd = n_fwd;
  p.pos0 = h->pos;
  p.out_ids = d_out_ids;
  p.embeds = o.embeds;
  p.n_embed_rows = o.embeds ? o.n_embed_rows : 0;
  p.pos3 = o.pos3;
  p.logits = o.logits;
  p.hidden = o.hidden;
  p.trace = reinterpret_cast<unsigned long long *>(o.trace);
  p.chunks_override = o.attn_chunks;
  p.spin_ns = o.spin_ns > 0 ? o.spin_ns : 1000000000LL;
  p.fault_barrier = o.fault_skip_barrier - 1;   // forward index, -1 = off
  if (o.codes) {
    p.cb_books = static_cast<const uint16_t *>(o.books);
    p.cb_text = static_cast<const uint16_t *>(o.text);
    p.cb_codes = o.codes;
    p.cb_text_ids = o.text_ids;
    p.cb_n = o.n_books;
    p.cb_rows = o.book_rows;
    p.cb_text_rows = o.text_rows;
    p.cb_n_rows = o.n_code_rows;
  }
  if (o.flags & MK_DECODE_STREAM) {
    // an empty mailbox: the kernel raises the count as it publishes ids
    __atomic_store_n(&h->mbox[0], 0, __ATOMIC_RELEASE);
    p.mbox_count = h->d_mbox;
    p.mbox_ids = h->d_mbox + 32;
  }

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // every forward publishes its activations under a tag never used before
  if (h->tag > 0xF0000000u - static_cast<unsigned>(n_fwd)) {
    if (cudaMemsetAsync(h->ll_base, 0, sizeof(unsigned long long) * h->ll_words * h->ll_rep, s) != cudaSuccess) {
      cudaGetLastError();
      return MK_ERR_CUDA;
    }
    h->tag = 1;
  }
  p.tag0 = h->tag;
  h->tag += static_cast<unsigned>(n_fwd);
  // barrier counter, error word and merge tickets start at zero for every call
  if (cudaMemsetAsync(h->d_sync, 0, sizeof(int) * 2, s) != cudaSuccess ||
      cudaMemsetAsync(h->base.tickets, 0, sizeof(unsigned) * h->cfg.n_kv_heads, s) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  cudaError_t e = cudaSuccess;
  if (o.flags & MK_DECODE_PER_OP_GRAPH) {
    // the ablation as one replay of a captured graph per forward
    const int grc = build_forward_graph(h);
    if (grc != MK_OK) return grc;
    mk::CallBlock b;
    std::memset(&b, 0, sizeof(b));
    b.in_ids = p.in_ids; b.out_ids = p.out_ids; b.embeds = p.embeds; b.pos3 = p.pos3;
    b.logits = p.logits; b.hidden = p.hidden; b.trace = p.trace; b.spin_ns = p.spin_ns;
    b.n_in = p.n_in; b.n_fwd = p.n_fwd; b.pos0 = p.pos0; b.n_embed_rows = p.n_embed_rows;
    b.chunks_override = p.chunks_override; b.op_fwd = 0; b.tag0 = p.tag0;
    b.mbox_ids = p.mbox_ids; b.mbox_count = p.mbox_count;
    b.cb_books = p.cb_books; b.cb_text = p.cb_text; b.cb_codes = p.cb_codes; b.cb_text_ids = p.cb_text_ids;
    b.cb_n = p.cb_n; b.cb_rows = p.cb_rows; b.cb_text_rows = p.cb_text_rows; b.cb_n_rows = p.cb_n_rows;
    e = cudaMemcpyAsync(h->d_blk, &b, sizeof(b), cudaMemcpyHostToDevice, s);
    for (int f = 0; f < n_fwd && e == cudaSuccess; ++f) e = cudaGraphLaunch(h->gexec, s);
    if (e == cudaSuccess) {
      p.per_op = 1;
      p.fault_barrier = -1;
      p.op_fwd = n_fwd;
      p.op_phase = 5 * p.L + 1;   // final greedy selection
      void *args[] = {&p};
      e = cudaLaunchKernel(h->kernel, dim3(h->G), dim3(mk::NTHREADS), args, h->smem, s);
    }
  } else if (!(o.flags & MK_DECODE_PER_OP)) {
    p.per_op = 0;
    void *args[] = {&p};
    e = cudaLaunchCooperativeKernel(h->kernel, dim3(h->G), dim3(mk::NTHREADS), args, h->smem, s);
  } else {
    // the launch-overhead ablation: the same phases, one ordinary launch each
    p.per_op = 1;
    p.fault_barrier = -1;
    const int nph = 5 * p.L + 1;
    void *args[] = {&p};
    for (int f = 0; f < n_fwd && e == cudaSuccess; ++f)
      for (int ph = 0; ph < nph && e == cudaSuccess; ++ph) {
        p.op_fwd = f;
        p.op_phase = ph;
        e = cudaLaunchKernel(h->kernel, dim3(h->G), dim3(mk::NTHREADS), args, h->smem, s);
      }
    if (e == cudaSuccess) {
      p.op_fwd = n_fwd;
      p.op_phase = nph;      // final greedy selection
      e = cudaLaunchKernel(h->kernel, dim3(h->G), dim3(mk::NTHREADS), args, h->smem, s);
    }
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  h->pending = 1;
  h->pending_fwd = n_fwd;
  h->pending_stream = s;
  return MK_OK;
}

int mk_decode_wait(mk_handle *h) {
  if (!h || !h->pending) return MK_ERR_INVALID_ARG;
  h->pending = 0;
  if (h->pending_fwd == 0) return MK_OK;
  cudaStream_t s = h->pending_stream;
  int herr = 0;
  if (cudaSetDevice(h->device) != cudaSuccess ||
      cudaMemcpyAsync(&herr, h->d_sync + 1, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  if (herr != 0) return herr;
  h->pos += h->pending_fwd;
  return MK_OK;
}

int mk_decode(mk_handle *h, const int32_t *d_in_ids, int32_t n_in, int32_t n_steps, int32_t *d_out_ids,
              const mk_decode_opts *opts, mk_stream stream) {
  const int rc = mk_decode_start(h, d_in_ids, n_in, n_steps, d_out_ids, opts, stream);
  if (rc != MK_OK) return rc;
  return mk_decode_wait(h);
}

int mk_prefill(mk_handle *h, const int32_t *d_in_ids, int32_t n, int32_t *d_out_ids, const mk_decode_opts *opts,
               mk_stream stream) {
  if (!h || h->pending || n < 0) return MK_ERR_INVALID_ARG;
  if (n == 0) return MK_OK;
  if (!d_in_ids) return MK_ERR_INVALID_ARG;
  mk_decode_opts o;
  std::memset(&o, 0, sizeof(o));
  if (opts) o = *opts;
  if (o.flags || o.trace || o.codes || o.n_embed_rows < 0 || (o.n_embed_rows > 0 && !o.embeds))
    return MK_ERR_INVALID_ARG;
  if (static_cast<int64_t>(h->pos) + n > h->cfg.max_seq) return MK_ERR_KV_FULL;
  if (cudaSetDevice(h->device) != cudaSuccess) return MK_ERR_CUDA;
  const mk_config &c = h->cfg;
  int rc = mkp::pf_init(h->pf, std::min(256, c.max_seq), c.hidden, c.n_q_heads, c.n_kv_heads, c.head_dim,
                        c.intermediate);
  if (rc != MK_OK) return rc;
  const mk::Params &p = h->base;
  mkp::PfArgs a;
  std::memset(&a, 0, sizeof(a));
  a.L = p.L; a.H = p.H; a.Hq = p.Hq; a.Hkv = p.Hkv; a.d = p.d; a.I = p.I; a.V = p.V; a.vocab_in = p.vocab_in;
  a.eps = p.eps; a.inv_sqrt_d = p.inv_sqrt_d;
  a.rope_mode = p.rope_mode; a.sec0 = p.sec_b0; a.sec1 = p.sec1; a.sec2 = p.sec2;
  a.rope_len = p.rope_len; a.max_seq = p.max_seq;
  a.embed = p.embed; a.rope = p.rope; a.kcache = p.kcache; a.vcache = p.vcache;
  mkp::PfCall call;
  std::memset(&call, 0, sizeof(call));
  call.ids = d_in_ids; call.embeds = o.embeds; call.n_embed_rows = o.embeds ? o.n_embed_rows : 0;
  call.pos3 = o.pos3; call.n_pos = n; call.pos0 = h->pos; call.hidden = o.hidden;
  call.out_ids = d_out_ids; call.logits_out = o.logits; call.last_id = p.last_id;
  rc = mkp::pf_run(h->pf, a, h->pf_layers.data(), p.final_norm, p.lm_head, n, call,
                   reinterpret_cast<cudaStream_t>(stream));
  if (rc != MK_OK) return rc;
  h->pos += n;
  return MK_OK;
}

int mk_mailbox_read(mk_handle *h, int32_t *dst, int32_t cap, int32_t *n_out) {
  if (!h || !n_out || cap < 0 || (cap > 0 && !dst)) return MK_ERR_INVALID_ARG;
  const int32_t n = __atomic_load_n(&h->mbox[0], __ATOMIC_ACQUIRE);
  const int32_t m = n < cap ? n : cap;
  for (int32_t i = 0; i < m; ++i) dst[i] = __atomic_load_n(&h->mbox[32 + i], __ATOMIC_RELAXED);
  *n_out = n;
  return MK_OK;
}

int mk_decode_host(mk_handle *h, const int32_t *h_in_ids, int32_t n_in, int32_t n_steps, int32_t *h_out_ids,
                   const mk_decode_opts *opts, mk_stream stream) {
  if (!h || h->pending || n_in < 0 || n_steps < 0 || !h_out_ids || (n_in > 0 && !h_in_ids))
    return MK_ERR_INVALID_ARG;
  if (static_cast<int64_t>(h->pos) + n_in + n_steps > h->cfg.max_seq) return MK_ERR_KV_FULL;
  const int n_fwd = n_in + n_steps;
  if (n_fwd == 0) return MK_OK;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaSetDevice(h->device) != cudaSuccess) return MK_ERR_CUDA;
  if (n_in > 0 &&
      cudaMemcpyAsync(h->d_ids_in, h_in_ids, sizeof(int32_t) * n_in, cudaMemcpyHostToDevice, s) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  const int rc = mk_decode(h, h->d_ids_in, n_in, n_steps, h->d_ids_out, opts, stream);
  if (rc != MK_OK) return rc;
  if (cudaMemcpyAsync(h_out_ids, h->d_ids_out, sizeof(int32_t) * n_fwd, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  return MK_OK;
}

int mk_plan_for(const mk_config *cfg, int32_t n_sm, int32_t *plan) {
  if (!cfg || !plan || n_sm < 1) return MK_ERR_INVALID_ARG;
  if (int rc = check_shape(*cfg)) return rc;
  mk::GemvGeom geo[mk::GV_COUNT];
  std::memset(geo, 0, sizeof(geo));
  if (int rc = choose_geometry(*cfg, n_sm, geo)) return rc;
  *plan = pick_plan(cfg->head_dim, cfg->n_q_heads / cfg->n_kv_heads, geo);
  return MK_OK;
}

int mk_get_info(const mk_handle *h, mk_info *info) {
  if (!h || !info) return MK_ERR_INVALID_ARG;
  info->grid = h->G;
  info->threads = mk::NTHREADS;
  info->stages = h->stages;
  info->stage_bytes = kStageBytes;
  info->smem_bytes = h->smem;
  info->position = h->pos;
  info->max_chunks = h->max_chunks;
  info->weight_bytes = h->weight_bytes;
  info->kv_bytes = h->kv_bytes;
  info->plan = h->kernel == mk::kernel_hidden1024() ? 1 : h->kernel == mk::kernel_hidden2048() ? 2 : 0;
  return MK_OK;
}

int mk_destroy(mk_handle *h) {
  if (!h) return MK_OK;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  if (h->gexec) cudaGraphExecDestroy(h->gexec);
  if (h->graph) cudaGraphDestroy(h->graph);
  if (h->cap) cudaStreamDestroy(h->cap);
  if (h->mbox) cudaFreeHost(h->mbox);
  mkp::pf_free(h->pf);
  h->buf.free_all();
  delete h;
  return MK_OK;
}

}  // extern "C"
