// Device code of the persistent decode megakernel.
//
// One CTA per SM.  Warps 0..7 are consumers; warp 8 is the TMA producer, whose
// lane 0 walks the CTA's fixed tile schedule (weight rows of every GEMV phase,
// then KV-cache chunks of every attention phase, layer after layer, step after
// step) and streams it through a multi-stage shared-memory ring with 1-D bulk
// copies.  Weight streaming does not depend on the data, so the producer runs
// ahead across grid barriers and decode steps while the consumers wait.
//
// Per forward (one token), the phases are
//   per layer: QKV (RMSNorm fused) | attention (QK-norm, RoPE/MRoPE, KV append,
//              split-KV chunk states; up to 8 chunks the chunk holding the new
//              position polls the others and merges, more chunks: the
//              last-arriving CTA merges) | O-proj + residual
//              | RMSNorm + gate/up + SiLU*mul | down-proj + residual
//   then:      final RMSNorm + LM head + per-CTA argmax candidates, and the
//              forward's one grid barrier
// and the next forward's first phase reduces the candidates (greedy argmax,
// lowest index on ties) and feeds the id back in-kernel.  Between phases the
// activations travel as tagged words (value + forward tag) that each reader
// polls; there is no grid barrier inside a forward.
//
// page A = "Porting a 1,200-line persistent CUDA megakernel to Qwen3-TTS: ~25 ms
// to first audio chunk" (dev.to); page B = "I made a single CUDA kernel speak:
// streaming Qwen3-TTS at 50ms latency on an RTX 5090" (theaicatchup.com).
#pragma once
#include <cstdint>
#include <climits>
#include <cmath>

#include "mk_params.h"
#include "mk_plans.h"
#include "ptx.cuh"

namespace mk {

constexpr int CONS_BAR = 1;   // named barrier id used by the consumer warps
constexpr int MK_ERR_BAD_TOKEN_D = -4;
constexpr int MK_ERR_TIMEOUT_D = -5;
constexpr int MK_ERR_NUMERIC_D = -6;
constexpr int MK_ERR_BAD_POSITION_D = -9;

__device__ __forceinline__ void set_err(const Params &p, int code) { atomicCAS(p.err, 0, code); }

__device__ __forceinline__ volatile int &flag(SmemCtl &S, int i) {
  return reinterpret_cast<volatile int *>(S.flags)[i];
}

__device__ __forceinline__ void cons_sync() { named_bar_sync(CONS_BAR, NCT); }

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// round-to-nearest-even float -> bf16 bits (NaN kept quiet)
__device__ __forceinline__ uint16_t f2bf(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// 1 / sqrt(x), each step correctly rounded: the same value as 1.0f / sqrtf(x)
// under IEEE division and square root, without the general division's
// scaling path (about 300 cycles on the critical path of every norm)
__device__ __forceinline__ float inv_sqrt_rn(float x) { return __frcp_rn(__fsqrt_rn(x)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// position in the weight ring: fill index, its slot and the parity of the
// slot's mbarrier phase (advanced by one per tile, no division)
struct RingPos {
  uint32_t it = 0;
  int slot = 0;
  uint32_t par = 0;
  __device__ __forceinline__ void next(int stages) {
    ++it;
    if (++slot == stages) {
      slot = 0;
      par ^= 1u;
    }
  }
};

// the consumer's ring position and S.red buffer index, passed to and returned
// from the out-of-line GEMV phases by value (in registers, not through the
// caller's stack)
struct RingState {
  RingPos rp;
  int rb = 0;
};

// balanced contiguous split of `total` items over G CTAs
__device__ __forceinline__ void split_range(int total, int G, int cta, int &r0, int &r1) {
  r0 = static_cast<int>((static_cast<long long>(total) * cta) / G);
  r1 = static_cast<int>((static_cast<long long>(total) * (cta + 1)) / G);
}

// Reduce N row-partials held by every lane to one full sum per row: after the
// halving steps lane l holds row (l >> (5 - log2 N)), summed over the warp.
template <int N>
__device__ __forceinline__ float warp_multi_reduce(float (&v)[N], int lane) {
  constexpr int LOGN = (N >= 32) ? 5 : (N >= 16) ? 4 : (N >= 8) ? 3 : (N >= 4) ? 2 : (N >= 2) ? 1 : 0;
  static_assert(N == (1 << LOGN) && N <= 32, "slots: a power of two up to 32");
#pragma unroll
  for (int lvl = 0; lvl < LOGN; ++lvl) {
    const int o = 16 >> lvl;
    const int n = N >> lvl;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      float send = up ? v[i] : v[i + n / 2];
      float keep = up ? v[i + n / 2] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
#pragma unroll
  for (int o = 16 >> LOGN; o >= 1; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
  return v[0];
}

// ---------------------------------------------------------------------------
// waits (every wait has a time budget; on expiry the CTA is marked aborted and
// the caller carries on without blocking so that named barriers stay matched)
// ---------------------------------------------------------------------------
struct Deadline {
  unsigned long long start = 0;
  __device__ __forceinline__ bool expired(long long budget) {
    unsigned long long now = globaltimer();
    if (start == 0) { start = now; return false; }
    return static_cast<long long>(now - start) > budget;
  }
};

__device__ __forceinline__ void wait_full(const Params &p, SmemCtl &S, int slot, uint32_t parity) {
  if (mbar_try_wait(&S.full[slot], parity)) return;
  Deadline dl;
  int n = 0;
  while (!mbar_try_wait(&S.full[slot], parity)) {
    if ((++n & 63) == 0) {
      if (flag(S, F_ABORT)) return;
      if (dl.expired(p.spin_ns)) { set_err(p, MK_ERR_TIMEOUT_D); flag(S, F_ABORT) = 1; return; }
    }
  }
}

// grid-wide barrier over all CTAs (consumer threads only); returns false when
// the CTA must stop (timeout, or an error set by any CTA before arriving)
static __device__ bool grid_barrier(const Params &p, SmemCtl &S, unsigned &target, int bar_index, int cta) {
  cons_sync();
  if (threadIdx.x == 0) {
    target += static_cast<unsigned>(p.G);
    const bool skip = (p.fault_barrier == bar_index) && (cta == 0);   // test hook
    if (!skip) {
      __threadfence();
      red_release_add(p.bar, 1u);
    }
    if (!flag(S, F_ABORT)) {
      Deadline dl;
      int n = 0;
      while (ld_acquire(p.bar) < target) {
        if ((++n & 255) == 0 && dl.expired(p.spin_ns)) {
          set_err(p, MK_ERR_TIMEOUT_D);
          flag(S, F_ABORT) = 1;
          break;
        }
      }
    }
    if (ld_relaxed_i32(p.err) != 0) flag(S, F_ABORT) = 1;
  }
  cons_sync();
  return flag(S, F_ABORT) == 0;
}

// optional %globaltimer stamps of thread 0: trace[((gp * G) + cta) * 4 + k],
// k = 0 phase start, 1 input in registers, 2 tiles and epilogue done, 3 barrier passed
__device__ __forceinline__ void trace_mark(const Params &p, int gp, int cta, int k) {
  if (p.trace && threadIdx.x == 0) p.trace[(static_cast<size_t>(gp) * p.G + cta) * 4 + k] = globaltimer();
}

// ---------------------------------------------------------------------------
// tagged words: {float value (low 32 bits), tag (high 32 bits)} stored and
// loaded as single 64-bit accesses, so a reader that sees the tag it expects
// also sees the value written with it
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ll_store(unsigned long long *p, float v, unsigned tag) {
  const unsigned long long w = (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
// publish to every copy of a tagged buffer
__device__ __forceinline__ void ll_store_rep(const Params &p, unsigned long long *dst, float v, unsigned tag) {
  for (int r = 0; r < p.ll_rep; ++r) ll_store(dst + r * p.ll_cs, v, tag);
}
__device__ __forceinline__ unsigned long long ll_load(const unsigned long long *p) {
  unsigned long long w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}
__device__ __forceinline__ void ll_load2(const unsigned long long *p, unsigned long long &a,
                                         unsigned long long &b) {
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
__device__ __forceinline__ unsigned ll_tag(unsigned long long w) { return static_cast<unsigned>(w >> 32); }
__device__ __forceinline__ float ll_val(unsigned long long w) { return __uint_as_float(static_cast<unsigned>(w)); }

// Reload the stale words of w[] (word j at src + j * STRIDE) until all carry
// `tag`.  Gives up (values undefined) once the CTA is aborting, any CTA has
// reported an error, or the wait budget runs out.
template <int N, int STRIDE>
__device__ __forceinline__ void ll_settle(const Params &p, SmemCtl &S, const unsigned long long *src,
                                          unsigned tag, unsigned long long (&w)[N]) {
  bool ok = true;
#pragma unroll
  for (int j = 0; j < N; ++j) ok &= (ll_tag(w[j]) == tag);
  if (ok) return;
  Deadline dl;
  int n = 0;
  for (;;) {
#pragma unroll
    for (int j = 0; j < N; ++j)
      if (ll_tag(w[j]) != tag) w[j] = ll_load(src + j * STRIDE);
    ok = true;
#pragma unroll
    for (int j = 0; j < N; ++j) ok &= (ll_tag(w[j]) == tag);
    if (ok) return;
    if (p.poll_ns) __nanosleep(p.poll_ns);
    if ((++n & 15) == 0) {
      if (flag(S, F_ABORT) || ld_relaxed_i32(p.err) != 0) return;
      if (dl.expired(p.spin_ns)) {
        set_err(p, MK_ERR_TIMEOUT_D);
        flag(S, F_ABORT) = 1;
        return;
      }
    }
  }
}

// Where element k of a GEMV input vector lives in its tagged buffer.  Thread
// kc of the consuming phase owns elements [kc*KPT, (kc+1)*KPT); they are
// stored as KPT/2 word pairs, pair c of every thread side by side, so that
// each of the consumer's pair loads covers consecutive 16-byte slots of
// consecutive threads (a warp reads 512 contiguous bytes per load).
// A staged reader (fast layout 1) polls the vector in natural order.
__device__ __forceinline__ int ll_slot(const GemvGeom &g, int k) {
  if (g.fast == 1) return k;
  int kc, j;
  if (g.fast == 2) {
    const int c = k >> g.lgSpan, r = k - (c << g.lgSpan);
    kc = r >> g.lgCH;
    j = (c << g.lgCH) + (r - (kc << g.lgCH));
  } else {
    kc = k / g.KPT;
    j = k - kc * g.KPT;
  }
  return (j >> 1) * (2 * g.TPR) + 2 * kc + (j & 1);
}

// This thread's KPT tagged words -> floats (KPT even).  src points at the
// thread's first pair (16-byte aligned); pair c sits at src + c * stride.
// All loads are issued at once; only words that still carry an older tag are
// reloaded, tracked by a bit mask.
template <int KPT>
__device__ __forceinline__ void ll_poll_slice(const Params &p, SmemCtl &S, const unsigned long long *src,
                                              int stride, unsigned tag, float (&xr)[KPT]) {
  unsigned stale = 0;
#pragma unroll
  for (int c = 0; c < KPT / 2; ++c) {
    unsigned long long a, b;
    ll_load2(src + c * stride, a, b);
    xr[2 * c] = ll_val(a);
    xr[2 * c + 1] = ll_val(b);
    stale |= (ll_tag(a) != tag ? 1u : 0u) << (2 * c);
    stale |= (ll_tag(b) != tag ? 1u : 0u) << (2 * c + 1);
  }
  if (stale == 0) return;
  Deadline dl;
  int n = 0;
  for (;;) {
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      if (stale & (1u << j)) {
        const unsigned long long wj = ll_load(src + (j >> 1) * stride + (j & 1));
        if (ll_tag(wj) == tag) {
          xr[j] = ll_val(wj);
          stale &= ~(1u << j);
        }
      }
    }
    if (stale == 0) return;
    if (p.poll_ns) __nanosleep(p.poll_ns);
    if ((++n & 15) == 0) {
      if (flag(S, F_ABORT) || ld_relaxed_i32(p.err) != 0) return;
      if (dl.expired(p.spin_ns)) {
        set_err(p, MK_ERR_TIMEOUT_D);
        flag(S, F_ABORT) = 1;
        return;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// argmax helpers (largest value, lowest index among equals)
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// block-wide argmax over the consumer threads; every consumer gets the result
static __device__ void block_argmax(SmemCtl &S, float &v, int &i) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    float ov = __shfl_xor_sync(0xffffffffu, v, o);
    int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
  if (lane == 0) { S.bestv[w] = v; S.besti[w] = i; }
  cons_sync();
  v = S.bestv[0];
  i = S.besti[0];
  for (int k = 1; k < NCW; ++k)
    if (better(S.bestv[k], S.besti[k], v, i)) { v = S.bestv[k]; i = S.besti[k]; }
  cons_sync();
}

// reduce the per-CTA LM-head candidates of the previous forward -> greedy id
static __device__ int select_token(const Params &p, SmemCtl &S, int f_prev, int cta, bool final) {
  float v = -INFINITY;
  int i = INT_MAX;
  for (int c = threadIdx.x; c < p.G; c += NCT) {
    float cv = __ldcg(p.cand_val + c);
    int ci = __ldcg(p.cand_idx + c);
    if (better(cv, ci, v, i)) { v = cv; i = ci; }
  }
  block_argmax(S, v, i);
  if (threadIdx.x == 0 && cta == 0) {
    p.out_ids[f_prev] = i;
    if (final) *p.last_id = i;
    if (p.mbox_ids) {
      // streaming: the id reaches the host's mailbox before the count does
      *reinterpret_cast<volatile int32_t *>(p.mbox_ids + f_prev) = i;
      __threadfence_system();
      st_release_sys_i32(p.mbox_count, f_prev + 1);
    }
  }
  return i;
}

// ---------------------------------------------------------------------------
// GEMV phases
// ---------------------------------------------------------------------------
template <int KPT>
__device__ __forceinline__ void load_f32(const float *src, float (&xr)[KPT]) {
  const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
  for (int c = 0; c < KPT / 4; ++c) {
    float4 q = __ldcg(s4 + c);
    xr[4 * c] = q.x; xr[4 * c + 1] = q.y; xr[4 * c + 2] = q.z; xr[4 * c + 3] = q.w;
  }
}

template <int KPT>
__device__ __forceinline__ void load_bf16(const uint16_t *src, float (&xr)[KPT]) {
  const uint2 *s2 = reinterpret_cast<const uint2 *>(src);
#pragma unroll
  for (int c = 0; c < KPT / 4; ++c) {
    uint2 q = __ldg(s2 + c);
    xr[4 * c] = bf_lo(q.x); xr[4 * c + 1] = bf_hi(q.x);
    xr[4 * c + 2] = bf_lo(q.y); xr[4 * c + 3] = bf_hi(q.y);
  }
}

// dot of KPT bf16 weights in shared memory with the register slice
template <int KPT>
__device__ __forceinline__ float dot_row(const unsigned char *src, const float (&xr)[KPT]) {
  float s = 0.f;
  if constexpr (KPT % 8 == 0) {
#pragma unroll
    for (int c = 0; c < KPT / 8; ++c) {
      uint4 q = *reinterpret_cast<const uint4 *>(src + 16 * c);
      s = fmaf(bf_lo(q.x), xr[8 * c + 0], s);
      s = fmaf(bf_hi(q.x), xr[8 * c + 1], s);
      s = fmaf(bf_lo(q.y), xr[8 * c + 2], s);
      s = fmaf(bf_hi(q.y), xr[8 * c + 3], s);
      s = fmaf(bf_lo(q.z), xr[8 * c + 4], s);
      s = fmaf(bf_hi(q.z), xr[8 * c + 5], s);
      s = fmaf(bf_lo(q.w), xr[8 * c + 6], s);
      s = fmaf(bf_hi(q.w), xr[8 * c + 7], s);
    }
  } else {
#pragma unroll
    for (int c = 0; c < KPT / 4; ++c) {
      uint2 q = *reinterpret_cast<const uint2 *>(src + 8 * c);
      s = fmaf(bf_lo(q.x), xr[4 * c + 0], s);
      s = fmaf(bf_hi(q.x), xr[4 * c + 1], s);
      s = fmaf(bf_lo(q.y), xr[4 * c + 2], s);
      s = fmaf(bf_hi(q.y), xr[4 * c + 3], s);
    }
  }
  return s;
}

// Input row of forward f: a non-negative id reads the embedding table, a
// negative id -(r+1) row r of the caller's precomputed fp32 buffer (page B,
// "Why Does a Single Kernel Even Matter for TTS?", the sentinel) -- or, with
// code rows, the talker's sum of codebook rows and a text row, formed here in
// fp32 in table order (codebook 0 .. n-1, then text).
template <int KPT>
__device__ __forceinline__ void load_input_slice(const Params &p, int id, int k0, float (&xr)[KPT]) {
  if (id >= 0) {
    load_bf16<KPT>(p.embed + static_cast<size_t>(id) * p.H + k0, xr);
  } else if (p.cb_codes) {
    const int r = -id - 1;
#pragma unroll
    for (int i = 0; i < KPT; ++i) xr[i] = 0.f;
    for (int j = 0; j < p.cb_n; ++j) {
      const int c = p.cb_codes[static_cast<size_t>(r) * p.cb_n + j];
      float v[KPT];
      load_bf16<KPT>(p.cb_books + (static_cast<size_t>(j) * p.cb_rows + c) * p.H + k0, v);
#pragma unroll
      for (int i = 0; i < KPT; ++i) xr[i] += v[i];
    }
    float v[KPT];
    load_bf16<KPT>(p.cb_text + static_cast<size_t>(p.cb_text_ids[r]) * p.H + k0, v);
#pragma unroll
    for (int i = 0; i < KPT; ++i) xr[i] += v[i];
  } else {
    load_f32<KPT>(p.embeds + static_cast<size_t>(-id - 1) * p.H + k0, xr);
  }
}

// out of line: runs at layer 0 only, and its talker loop would otherwise sit
// in every copy of the QKV code
static __device__ __noinline__ float input_elem(const Params &p, int id, int k) {
  if (id >= 0) return bf2f(p.embed[static_cast<size_t>(id) * p.H + k]);
  if (!p.cb_codes) return p.embeds[static_cast<size_t>(-id - 1) * p.H + k];
  const int r = -id - 1;
  float acc = 0.f;
  for (int j = 0; j < p.cb_n; ++j)
    acc += bf2f(p.cb_books[(static_cast<size_t>(j) * p.cb_rows + p.cb_codes[static_cast<size_t>(r) * p.cb_n + j]) *
                               p.H + k]);
  return acc + bf2f(p.cb_text[static_cast<size_t>(p.cb_text_ids[r]) * p.H + k]);
}

// a negative id with code rows: the row and every id in it must be in range
__device__ __forceinline__ bool code_row_ok(const Params &p, int r) {
  if (r >= p.cb_n_rows) return false;
  for (int j = 0; j < p.cb_n; ++j) {
    const int c = p.cb_codes[static_cast<size_t>(r) * p.cb_n + j];
    if (c < 0 || c >= p.cb_rows) return false;
  }
  const int t = p.cb_text_ids[r];
  return t >= 0 && t < p.cb_text_rows;
}

// Epilogue of one batch of a GEMV phase: one thread per output row (pair)
// sums the warps' partials of rows a0 .. a0 + nout - 1 from S.red[rb] (pairs:
// gate rows of a tile, then its up rows) and applies the phase's epilogue:
// publish, residual add, SiLU(gate) * up, or logits plus a running argmax.
__device__ __forceinline__ void gemv_epilogue(const Params &p, SmemCtl &S, const GemvGeom &g, int kind, int layer,
                                              int f, int rb, int a0, int nout, unsigned tag, float &best_v,
                                              int &best_i) {
  const int t = threadIdx.x;
  const int wpr = g.TPR / 32;
  const int qkv_rows = (p.Hq + 2 * p.Hkv) * p.d;
  const int own0 = S.rr[kind][0];   // S.xown[0] is row own0 (O and down split H like the residual)
  // rows go to warps 1.. first: warp 0 shares its scheduler with the producer warp
  for (int q = (t + NCT - 32) % NCT; q < nout; q += NCT) {
    const int grow = a0 + q;
    float y = 0.f;
    if (kind == GV_GU) {
      const int qt = g.lgRT >= 0 ? (q >> g.lgRT) : q / g.RT;
      const int base = qt * 2 * g.RT + (q - qt * g.RT);
      float up = 0.f;
#pragma unroll
      for (int ww = 0; ww < MAX_WPR; ++ww)
        if (ww < wpr) { y += S.red[rb][base][ww]; up += S.red[rb][base + g.RT][ww]; }
      ll_store_rep(p, p.ll.u + static_cast<size_t>(layer) * p.I + ll_slot(p.geo[GV_DOWN], grow),
                   y / (1.0f + expf(-y)) * up, tag);
      continue;
    }
#pragma unroll
    for (int ww = 0; ww < MAX_WPR; ++ww)
      if (ww < wpr) y += S.red[rb][q][ww];
    switch (kind) {
      case GV_QKV: ll_store_rep(p, p.ll.qkv + static_cast<size_t>(layer) * qkv_rows + grow, y, tag); break;
      case GV_O: {
        const float xn = S.xown[grow - own0] + y;
        S.xown[grow - own0] = xn;
        ll_store_rep(p, p.ll.xmid + static_cast<size_t>(layer) * p.H + ll_slot(p.geo[GV_GU], grow), xn, tag);
        break;
      }
      case GV_DOWN: {
        const float xn = S.xown[grow - own0] + y;
        S.xown[grow - own0] = xn;
        ll_store_rep(p, p.ll.xout + static_cast<size_t>(layer) * p.H + ll_slot(p.geo[GV_QKV], grow), xn, tag);
        if (p.hidden) p.hidden[(static_cast<size_t>(f) * (p.L + 1) + layer + 1) * p.H + grow] = xn;
        break;
      }
      default: {  // LM head
        if (p.logits) p.logits[static_cast<size_t>(f) * p.V + grow] = y;
        if (!isfinite(y)) set_err(p, MK_ERR_NUMERIC_D);
        if (y > best_v) { best_v = y; best_i = grow; }
        break;
      }
    }
  }
}

// One GEMV phase of this CTA: y[r] = W[r,:] . in for the CTA's rows, with the
// RMSNorm of the input fused in (QKV, gate/up, LM head) and the phase's
// epilogue (publish, residual add, SiLU*mul, logits + argmax candidate).
// Tiles are consumed without a CTA-wide barrier; row partials collect in a
// batch buffer and one barrier per batch precedes the epilogue.
template <int KPT, int RPTP>
__device__ __noinline__ RingState gemv_phase(const Params &p, SmemCtl &S, unsigned char *ring, int kind, int layer,
                                             int f, int cta, int in_id, unsigned tag, RingState st, int gp) {
  RingPos &rp = st.rp;
  int &rb = st.rb;
  const GemvGeom g = p.geo[kind];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int kc = t % g.TPR, rg = t / g.TPR;
  const int k0 = kc * KPT;
  const bool norm = (kind == GV_QKV || kind == GV_GU || kind == GV_LM);

  // ---- gains (independent of the input: their latency overlaps the poll) ---
  float gn[KPT];
  if (norm) {
    const uint16_t *gain = kind == GV_QKV ? S.layers[layer].attn_norm
                         : kind == GV_GU  ? S.layers[layer].mlp_norm
                                          : p.final_norm;
    load_bf16<KPT>(gain + k0, gn);
  }
  // ---- input slice into registers ------------------------------------------
  float xr[KPT];
  if (kind == GV_QKV && layer == 0) {
    load_input_slice<KPT>(p, in_id, k0, xr);
  } else {
    const unsigned long long *src =
        kind == GV_QKV ? p.ll.xout + static_cast<size_t>(layer - 1) * p.H
      : kind == GV_O   ? p.ll.attn + static_cast<size_t>(layer) * p.Hq * p.d
      : kind == GV_GU  ? p.ll.xmid + static_cast<size_t>(layer) * p.H
      : kind == GV_DOWN ? p.ll.u + static_cast<size_t>(layer) * p.I
                        : p.ll.xout + static_cast<size_t>(p.L - 1) * p.H;
    ll_poll_slice<KPT>(p, S, src + (cta % p.ll_rep) * p.ll_cs + 2 * kc, 2 * g.TPR, tag, xr);
  }
  if (norm) {
    // RMSNorm fused into the GEMV: every CTA reduces mean(x^2) itself
    float ss = 0.f;
    if (rg == 0) {
#pragma unroll
      for (int j = 0; j < KPT; ++j) ss = fmaf(xr[j], xr[j], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) S.misc[w] = ss;
    cons_sync();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < NCW; ++i) tot += S.misc[i];
    const float ms = g.invK != 0.f ? tot * g.invK : tot / static_cast<float>(g.K);   // identical for 2^n
    const float rs = inv_sqrt_rn(ms + p.eps);
#pragma unroll
    for (int j = 0; j < KPT; ++j) xr[j] = xr[j] * rs * gn[j];
  }

  const int r0 = S.rr[kind][0], r1 = S.rr[kind][1];
  // the first layer's input also seeds the residual rows this CTA owns
  if (kind == GV_QKV && layer == 0) {
    const int o0 = S.rr[GV_O][0], o1 = S.rr[GV_O][1];
    for (int r = o0 + t; r < o1; r += NCT) {
      const float v = input_elem(p, in_id, r);
      S.xown[r - o0] = v;
      if (p.hidden) p.hidden[(static_cast<size_t>(f) * (p.L + 1)) * p.H + r] = v;
    }
  }
  trace_mark(p, gp, cta, 1);

  const int ntiles = (r1 - r0 + g.RT - 1) / g.RT;
  constexpr int LOGR = (RPTP >= 16) ? 4 : (RPTP >= 8) ? 3 : (RPTP >= 4) ? 2 : (RPTP >= 2) ? 1 : 0;
  const int wpr = g.TPR / 32;
  const int wg = w % wpr;                                   // warp within its row group
  const int trow = (kind == GV_GU) ? 2 * g.RT : g.RT;       // rows of a full tile
  const int bt = max(1, RED_ROWS / trow);                   // tiles per epilogue batch
  float best_v = -INFINITY;
  int best_i = INT_MAX;

  for (int tb = 0; tb < ntiles; tb += bt) {
    const int te = min(ntiles, tb + bt);
    for (int ti = tb; ti < te; ++ti) {
      const int a = r0 + ti * g.RT;
      const int nr = min(g.RT, r1 - a);
      const int rows_in_tile = (kind == GV_GU) ? 2 * nr : nr;
      const int slot = rp.slot;
      wait_full(p, S, slot, rp.par);
      const unsigned char *st = ring + static_cast<size_t>(slot) * STAGE_BYTES;
      // every row slot computes a dot product (slots past the tile's last row
      // re-read that row and are zeroed) so that no branch separates the rows
      // and their load/FMA chains interleave
      float acc[RPTP];
#pragma unroll
      for (int i = 0; i < RPTP; ++i) {
        const int row = rg + i * g.NG;
        const int rr = min(row, rows_in_tile - 1);
        const float dv = dot_row<KPT>(st + (static_cast<size_t>(rr) * g.K + k0) * 2, xr);
        acc[i] = row < rows_in_tile ? dv : 0.f;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[slot]);
      const float v = warp_multi_reduce<RPTP>(acc, lane);
      const int row = rg + (lane >> (5 - LOGR)) * g.NG;     // this lane's row inside the tile
      if ((lane & ((32 >> LOGR) - 1)) == 0 && row < rows_in_tile) {
        int brow;
        if (kind == GV_GU) brow = (ti - tb) * 2 * g.RT + (row < nr ? row : g.RT + (row - nr));
        else brow = (ti - tb) * g.RT + row;
        S.red[rb][brow][wg] = v;
      }
      rp.next(p.stages);
    }
    cons_sync();
    gemv_epilogue(p, S, g, kind, layer, f, rb, r0 + tb * g.RT, min(r1, r0 + te * g.RT) - (r0 + tb * g.RT), tag,
                  best_v, best_i);
    rb ^= 1;
  }
  // the warps without epilogue rows wait here instead of starting the next
  // phase's polls: the publishing stores leave sooner and the poll traffic
  // of every CTA is shorter (measured: 9% per token on the 0.6B shape)
  cons_sync();

  if (kind == GV_LM) {
    block_argmax(S, best_v, best_i);
    if (t == 0) {
      p.cand_val[cta] = best_v;
      p.cand_idx[cta] = best_i;
    }
  }
  trace_mark(p, gp, cta, 2);
  return st;
}

// ---------------------------------------------------------------------------
// fast GEMV layouts (GemvGeom::fast 1 and 2)
// ---------------------------------------------------------------------------
// dot of one bf16 row in shared memory with the thread's slice in the chunked
// layout: chunk c of thread kc holds the CH elements from c*SPAN + kc*CH, so
// every load of a warp covers consecutive bytes.  One accumulator per chunk;
// the chunk sums combine pairwise (a shallower tree than a running sum: the
// rounding error of long per-lane sums shows up at the 1.7B shape's fp32 noise
// floor).
template <int KPT, int CH, int SPAN>
__device__ __forceinline__ float dot_chunked(const unsigned char *row, int kc, const float (&xr)[KPT]) {
  constexpr int NCH = KPT / CH;
  float s[NCH];
#pragma unroll
  for (int c = 0; c < NCH; ++c) {
    const unsigned char *q = row + (c * SPAN + kc * CH) * 2;
    float a = 0.f;
    if constexpr (CH == 8) {
      const uint4 v = *reinterpret_cast<const uint4 *>(q);
      a = fmaf(bf_lo(v.x), xr[8 * c + 0], a);
      a = fmaf(bf_hi(v.x), xr[8 * c + 1], a);
      a = fmaf(bf_lo(v.y), xr[8 * c + 2], a);
      a = fmaf(bf_hi(v.y), xr[8 * c + 3], a);
      a = fmaf(bf_lo(v.z), xr[8 * c + 4], a);
      a = fmaf(bf_hi(v.z), xr[8 * c + 5], a);
      a = fmaf(bf_lo(v.w), xr[8 * c + 6], a);
      a = fmaf(bf_hi(v.w), xr[8 * c + 7], a);
    } else {
      const uint2 v = *reinterpret_cast<const uint2 *>(q);
      a = fmaf(bf_lo(v.x), xr[4 * c + 0], a);
      a = fmaf(bf_hi(v.x), xr[4 * c + 1], a);
      a = fmaf(bf_lo(v.y), xr[4 * c + 2], a);
      a = fmaf(bf_hi(v.y), xr[4 * c + 3], a);
    }
    s[c] = a;
  }
  float r;
  if constexpr (NCH == 8) r = ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
  else if constexpr (NCH == 4) r = (s[0] + s[1]) + (s[2] + s[3]);
  else if constexpr (NCH == 3) r = (s[0] + s[1]) + s[2];
  else if constexpr (NCH == 2) r = s[0] + s[1];
  else {
    static_assert(NCH == 1 || NCH == 6, "chunk counts of the compiled layouts");
    r = s[0];
#pragma unroll
    for (int c = 1; c < NCH; ++c) r += s[c];
  }
  return r;
}

// Poll n (<= MP) word pairs src[c * stride], src[c * stride + 1] until they
// carry `tag`; pairs c >= n read as zero.  Only stale words are reloaded.
template <int MP>
__device__ __forceinline__ void ll_poll_pairs(const Params &p, SmemCtl &S, const unsigned long long *src, int stride,
                                              int n, unsigned tag, float (&v)[2 * MP]) {
  unsigned stale = 0;
#pragma unroll
  for (int c = 0; c < MP; ++c) {
    v[2 * c] = v[2 * c + 1] = 0.f;
    if (c < n) {
      unsigned long long a, b;
      ll_load2(src + c * stride, a, b);
      v[2 * c] = ll_val(a);
      v[2 * c + 1] = ll_val(b);
      stale |= (ll_tag(a) != tag ? 1u : 0u) << (2 * c);
      stale |= (ll_tag(b) != tag ? 1u : 0u) << (2 * c + 1);
    }
  }
  if (stale == 0) return;
  Deadline dl;
  int k = 0;
  for (;;) {
#pragma unroll
    for (int j = 0; j < 2 * MP; ++j) {
      if (stale & (1u << j)) {
        const unsigned long long wj = ll_load(src + (j >> 1) * stride + (j & 1));
        if (ll_tag(wj) == tag) {
          v[j] = ll_val(wj);
          stale &= ~(1u << j);
        }
      }
    }
    if (stale == 0) return;
    if ((++k & 15) == 0) {
      if (flag(S, F_ABORT) || ld_relaxed_i32(p.err) != 0) return;
      if (dl.expired(p.spin_ns)) {
        set_err(p, MK_ERR_TIMEOUT_D);
        flag(S, F_ABORT) = 1;
        return;
      }
    }
  }
}

// One GEMV phase in a fast layout.  STAGED (layout 1): TPR = 32, row group =
// warp; the input vector is polled once per CTA into S.xs in natural order
// (thread t the word pairs at 2t + 512 m), its RMSNorm reduced on the way,
// and every warp then reads its chunks of the whole vector from S.xs.  Split-K
// (layout 2): TPR = 256, one row group; each thread polls its own chunks.
// Either way a thread keeps the partial dots of RPT rows of BT tiles in
// registers and the warp reduces them once per batch; the partials of the
// warps sharing a row (layout 2) meet in S.red before the epilogue.  Inlined
// into the plan kernels (kind a constant there); the general kernel calls the
// out-of-line copy below.
template <int KPT, int RPT, int BT, bool STAGED>
__device__ __forceinline__ void gemv_fast_body(const Params &p, SmemCtl &S, unsigned char *ring, int kind, int layer,
                                               int f, int cta, int in_id, unsigned tag, RingPos &rp, int &rb, int gp) {
  constexpr int CH = (KPT % 8 == 0) ? 8 : 4;
  constexpr int TPR = STAGED ? 32 : NCT;
  constexpr int NG = NCT / TPR;
  constexpr int SPAN = TPR * CH;
  constexpr int NS = RPT * BT;
  constexpr int LOGN = (NS >= 32) ? 5 : (NS >= 16) ? 4 : (NS >= 8) ? 3 : (NS >= 4) ? 2 : (NS >= 2) ? 1 : 0;
  static_assert((NS & (NS - 1)) == 0 && NS <= 32, "slots per batch: a power of two up to 32");
  const GemvGeom g = p.geo[kind];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int kc = t % TPR, rg = t / TPR;
  const int wg = w % (TPR / 32);

  float xr[KPT];
  if constexpr (STAGED) {
    // ---- gains of this lane's chunks (the loads overlap the poll) ----------
    const uint16_t *gain = kind == GV_QKV ? S.layers[layer].attn_norm
                         : kind == GV_GU  ? S.layers[layer].mlp_norm
                                          : p.final_norm;
    // kept as packed bf16 pairs across the poll (half the registers)
    uint32_t gw[KPT / 2];
#pragma unroll
    for (int c = 0; c < KPT / CH; ++c) {
#pragma unroll
      for (int j = 0; j < CH / 4; ++j) {
        const uint2 q = __ldg(reinterpret_cast<const uint2 *>(gain + c * SPAN + kc * CH) + j);
        gw[(c * CH) / 2 + 2 * j] = q.x;
        gw[(c * CH) / 2 + 2 * j + 1] = q.y;
      }
    }
    // ---- the input vector into S.xs, with its sum of squares ---------------
    constexpr int MP = (KPT * 32 + 511) / 512;   // word pairs per thread
    const int np = (g.K - 2 * t + 511) / 512;    // pairs of this thread inside the vector
    float v[2 * MP];
    if (kind == GV_QKV && layer == 0) {
#pragma unroll
      for (int c = 0; c < MP; ++c) {
        v[2 * c] = v[2 * c + 1] = 0.f;
        if (c < np) {
          v[2 * c] = input_elem(p, in_id, 2 * t + 512 * c);
          v[2 * c + 1] = input_elem(p, in_id, 2 * t + 512 * c + 1);
        }
      }
    } else {
      const unsigned long long *src =
          kind == GV_QKV ? p.ll.xout + static_cast<size_t>(layer - 1) * p.H
        : kind == GV_GU  ? p.ll.xmid + static_cast<size_t>(layer) * p.H
                         : p.ll.xout + static_cast<size_t>(p.L - 1) * p.H;
      ll_poll_pairs<MP>(p, S, src + (cta % p.ll_rep) * p.ll_cs + 2 * t, 512, np, tag, v);
    }
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < MP; ++c) {
      if (c < np) {
        *reinterpret_cast<float2 *>(&S.xs[2 * t + 512 * c]) = make_float2(v[2 * c], v[2 * c + 1]);
        ss = fmaf(v[2 * c], v[2 * c], ss);
        ss = fmaf(v[2 * c + 1], v[2 * c + 1], ss);
      }
    }
    ss = warp_sum(ss);
    if (lane == 0) S.misc[w] = ss;
    cons_sync();
    float tot = 0.f;
#pragma unroll
    for (int i = 0; i < NCW; ++i) tot += S.misc[i];
    const float ms = g.invK != 0.f ? tot * g.invK : tot / static_cast<float>(g.K);   // identical for 2^n
    const float rs = inv_sqrt_rn(ms + p.eps);
#pragma unroll
    for (int c = 0; c < KPT / CH; ++c) {
#pragma unroll
      for (int j = 0; j < CH; j += 4) {
        const float4 q = *reinterpret_cast<const float4 *>(&S.xs[c * SPAN + kc * CH + j]);
        const uint32_t g01 = gw[(c * CH + j) / 2], g23 = gw[(c * CH + j) / 2 + 1];
        xr[c * CH + j + 0] = q.x * rs * bf_lo(g01);
        xr[c * CH + j + 1] = q.y * rs * bf_hi(g01);
        xr[c * CH + j + 2] = q.z * rs * bf_lo(g23);
        xr[c * CH + j + 3] = q.w * rs * bf_hi(g23);
      }
    }
  } else {
    const unsigned long long *src = kind == GV_O ? p.ll.attn + static_cast<size_t>(layer) * p.Hq * p.d
                                                 : p.ll.u + static_cast<size_t>(layer) * p.I;
    ll_poll_slice<KPT>(p, S, src + (cta % p.ll_rep) * p.ll_cs + 2 * kc, 2 * TPR, tag, xr);
  }

  const int r0 = S.rr[kind][0], r1 = S.rr[kind][1];
  // the first layer's input also seeds the residual rows this CTA owns
  if (kind == GV_QKV && layer == 0) {
    const int o0 = S.rr[GV_O][0], o1 = S.rr[GV_O][1];
    for (int r = o0 + t; r < o1; r += NCT) {
      const float x0 = input_elem(p, in_id, r);
      S.xown[r - o0] = x0;
      if (p.hidden) p.hidden[(static_cast<size_t>(f) * (p.L + 1)) * p.H + r] = x0;
    }
  }
  trace_mark(p, gp, cta, 1);

  const int ntiles = S.nt[kind];
  const int trow = (kind == GV_GU) ? 2 * g.RT : g.RT;       // rows of a full tile
  const size_t rowb = static_cast<size_t>(g.K) * 2;
  float best_v = -INFINITY;
  int best_i = INT_MAX;
  for (int tb = 0; tb < ntiles; tb += BT) {
    const int te = min(ntiles, tb + BT);
    float acc[NS];
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      const int ti = tb + b;
      if (ti < te) {
        const int nr = min(g.RT, r1 - (r0 + ti * g.RT));
        const int rit = (kind == GV_GU) ? 2 * nr : nr;      // rows in this tile
        const int slot = rp.slot;
        wait_full(p, S, slot, rp.par);
        const unsigned char *st = ring + static_cast<size_t>(slot) * STAGE_BYTES;
        // row slots past the tile's last row re-read that row and are zeroed;
        // a paired gate/up tile holds gate rows at 0.. and up rows at RT..
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
          const int row = rg + i * NG;
          const bool paired = STAGED && RPT % 2 == 0 && kind == GV_GU;
          const bool ok = paired ? (row < g.RT ? row < nr : row - g.RT < nr) : row < rit;
          const int rr = paired ? row : min(row, rit - 1);
          const float dv = dot_chunked<KPT, CH, SPAN>(st + rr * rowb, kc, xr);
          acc[b * RPT + i] = ok ? dv : 0.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
        rp.next(p.stages);
      } else {
#pragma unroll
        for (int i = 0; i < RPT; ++i) acc[b * RPT + i] = 0.f;
      }
    }
    const float v = warp_multi_reduce<NS>(acc, lane);
    if constexpr (STAGED) {
      if (kind == GV_QKV || kind == GV_LM) {
        // a warp owns whole rows: the lane holding a row's sum publishes it
        // itself (no partials to combine, no batch barrier)
        const int sl = lane >> (5 - LOGN);
        const int b = sl / RPT, i = sl % RPT;
        const int ti = tb + b;
        if ((lane & ((32 >> LOGN) - 1)) == 0 && ti < te) {
          const int nr = min(g.RT, r1 - (r0 + ti * g.RT));
          const int row = rg + i * NG;
          if (row < nr) {
            const int grow = r0 + ti * g.RT + row;
            if (kind == GV_QKV) {
              ll_store_rep(p, p.ll.qkv + static_cast<size_t>(layer) * ((p.Hq + 2 * p.Hkv) * p.d) + grow, v, tag);
            } else {
              if (p.logits) p.logits[static_cast<size_t>(f) * p.V + grow] = v;
              if (!isfinite(v)) set_err(p, MK_ERR_NUMERIC_D);
              if (v > best_v || (v == best_v && grow < best_i)) { best_v = v; best_i = grow; }
            }
          }
        }
        continue;
      }
      if (RPT % 2 == 0 && kind == GV_GU) {
        // gate row r of a tile is the warp's slot i < RPT/2, its up row (r +
        // RT) slot i + RPT/2 of the same warp: the lane holding the gate sum
        // takes the up sum by one shuffle and publishes SiLU(gate) * up
        const float up = __shfl_down_sync(0xffffffffu, v, (RPT / 2) << (5 - LOGN));
        const int sl = lane >> (5 - LOGN);
        const int b = sl / RPT, i = sl % RPT;
        const int ti = tb + b;
        if ((lane & ((32 >> LOGN) - 1)) == 0 && i < RPT / 2 && ti < te) {
          const int nr = min(g.RT, r1 - (r0 + ti * g.RT));
          const int row = rg + i * NG;
          if (row < nr) {
            const int grow = r0 + ti * g.RT + row;
            float y = 0.f, u = 0.f;   // the same additions as the shared-buffer epilogue
            y += v;
            u += up;
            ll_store_rep(p, p.ll.u + static_cast<size_t>(layer) * p.I + ll_slot(p.geo[GV_DOWN], grow),
                         y / (1.0f + expf(-y)) * u, tag);
          }
        }
        continue;
      }
    }
    {
      const int sl = lane >> (5 - LOGN);                    // slot this lane holds
      const int b = sl / RPT, i = sl % RPT;
      const int ti = tb + b;
      if ((lane & ((32 >> LOGN) - 1)) == 0 && ti < te) {
        const int nr = min(g.RT, r1 - (r0 + ti * g.RT));
        const int rit = (kind == GV_GU) ? 2 * nr : nr;
        const int row = rg + i * NG;
        if (row < rit)
          S.red[rb][b * trow + ((kind == GV_GU && row >= nr) ? g.RT + (row - nr) : row)][wg] = v;
      }
    }
    cons_sync();
    gemv_epilogue(p, S, g, kind, layer, f, rb, r0 + tb * g.RT, min(r1, r0 + te * g.RT) - (r0 + tb * g.RT), tag,
                  best_v, best_i);
    rb ^= 1;
  }
  // warps without epilogue rows wait for the publishing ones (see gemv_phase)
  cons_sync();

  if (kind == GV_LM) {
    block_argmax(S, best_v, best_i);
    if (t == 0) {
      p.cand_val[cta] = best_v;
      p.cand_idx[cta] = best_i;
    }
  }
  trace_mark(p, gp, cta, 2);
}

// the out-of-line copy: the general kernel's dispatch, and the plan kernels'
// staged phases (QKV, gate/up and the LM head share one copy of the code)
template <int KPT, int RPT, int BT, bool STAGED>
__device__ __noinline__ RingState gemv_fast(const Params &p, SmemCtl &S, unsigned char *ring, int kind, int layer,
                                            int f, int cta, int in_id, unsigned tag, RingState st, int gp) {
  gemv_fast_body<KPT, RPT, BT, STAGED>(p, S, ring, kind, layer, f, cta, in_id, tag, st.rp, st.rb, gp);
  return st;
}

// dispatch on (KPT, RPTP) fixed at mk_create
static __device__ __noinline__ RingState gemv_dispatch(const Params &p, SmemCtl &S, unsigned char *ring, int kind,
                                                      int layer, int f, int cta, int in_id, unsigned tag, RingState st,
                                                      int gp) {
  const int kpt = p.geo[kind].KPT, r = p.geo[kind].RPTP;
  if (p.geo[kind].fast) {
    // the fast layouts mk_create may pick (KPT, rows per thread per tile, tiles per batch)
    const int bt = p.geo[kind].BT;
#define MK_FAST_CASE(ST, KP, RP, B) \
  if (p.geo[kind].fast == (ST ? 1 : 2) && kpt == KP && r == RP && bt == B) { \
    return gemv_fast<KP, RP, B, ST>(p, S, ring, kind, layer, f, cta, in_id, tag, st, gp); }
    MK_FAST_CASE(true, 32, 2, 2) MK_FAST_CASE(true, 64, 1, 4) MK_FAST_CASE(true, 16, 4, 2)
    MK_FAST_CASE(true, 24, 2, 4) MK_FAST_CASE(true, 8, 8, 1)
    MK_FAST_CASE(false, 8, 8, 1) MK_FAST_CASE(false, 8, 8, 2) MK_FAST_CASE(false, 12, 4, 2)
    MK_FAST_CASE(false, 24, 2, 8)
#undef MK_FAST_CASE
    return st;
  }
#define MK_GEMV_CASE(KP, RP) \
  if (kpt == KP && r == RP) return gemv_phase<KP, RP>(p, S, ring, kind, layer, f, cta, in_id, tag, st, gp);
  // every (KPT, RPTP) with KPT * RPTP <= 128 (mk_create rejects the others)
  MK_GEMV_CASE(8, 1) MK_GEMV_CASE(8, 2) MK_GEMV_CASE(8, 4) MK_GEMV_CASE(8, 8) MK_GEMV_CASE(8, 16)
  MK_GEMV_CASE(12, 1) MK_GEMV_CASE(12, 2) MK_GEMV_CASE(12, 4) MK_GEMV_CASE(12, 8)
  MK_GEMV_CASE(16, 1) MK_GEMV_CASE(16, 2) MK_GEMV_CASE(16, 4) MK_GEMV_CASE(16, 8)
  MK_GEMV_CASE(24, 1) MK_GEMV_CASE(24, 2) MK_GEMV_CASE(24, 4)
  if constexpr (KPT_MAX >= 32) { MK_GEMV_CASE(32, 1) MK_GEMV_CASE(32, 2) MK_GEMV_CASE(32, 4) }
  if constexpr (KPT_MAX >= 48) { MK_GEMV_CASE(48, 1) MK_GEMV_CASE(48, 2) }
#undef MK_GEMV_CASE
  return st;
}

// ---------------------------------------------------------------------------
// attention phase
// ---------------------------------------------------------------------------
struct AttnSched {
  int P, ctx, cs, C, units;
  int g0, c0;   // head and chunk of this CTA's first unit (unit = blockIdx.x)
};

__device__ __forceinline__ AttnSched attn_sched(const Params &p, int f) {
  AttnSched a;
  a.P = p.pos0 + f;
  a.ctx = a.P + 1;
  int cmax = p.chunks_override > 0 ? p.chunks_override : max(1, p.G / p.Hkv);
  // at least attn_min_chunks chunks, and one per attn_short_ppc positions up to
  // poll_cm chunks; beyond poll_cm * attn_ppc positions one per attn_ppc (up
  // to poll_cm chunks merge by polling, more by the last-arriving CTA)
  if (p.chunks_override <= 0 && p.attn_ppc > 0) {
    int want = max((a.ctx + p.attn_ppc - 1) / p.attn_ppc, min(p.attn_min_chunks, a.ctx));
    if (p.attn_short_ppc > 0) want = max(want, min(p.poll_cm, (a.ctx + p.attn_short_ppc - 1) / p.attn_short_ppc));
    cmax = min(cmax, want);
  }
  cmax = min(cmax, p.max_chunks);
  a.cs = (a.ctx + cmax - 1) / cmax;
  a.C = (a.ctx + a.cs - 1) / a.cs;
  a.units = p.Hkv * a.C;
  a.g0 = static_cast<int>(blockIdx.x) / a.C;
  a.c0 = static_cast<int>(blockIdx.x) - a.g0 * a.C;
  return a;
}

// rotary stream of pair i (page A, "Porting it to Qwen3-TTS-1.7B": MRoPE
// sections; contiguous runs of pair indices per position stream)
__device__ __forceinline__ int pair_stream(const Params &p, int i) {
  if (p.rope_mode == 0) return 0;
  if (p.rope_mode == 1) return i < p.sec_b0 ? 0 : (i < p.sec_b1 ? 1 : 2);
  // interleaved: streams take turns pair by pair until streams 1 and 2 have
  // their sections; the remaining pairs are stream 0
  const int r = i % 3;
  return ((r == 1 && i < 3 * p.sec1) || (r == 2 && i < 3 * p.sec2)) ? r : 0;
}

__device__ __forceinline__ int stream_pos(const Params &p, int f, int s, int P) {
  int pos = p.pos3 ? p.pos3[static_cast<size_t>(s) * p.n_fwd + f] : P;
  if (pos < 0 || pos >= p.rope_len) {
    set_err(p, MK_ERR_BAD_POSITION_D);
    pos = 0;
  }
  return pos;
}

// One warp normalises (RMS over head_dim, times gain) and rotates one head
// vector.  Lane l holds elements l + 32k so that the rotate-half partner of
// element i (i + d/2) sits in the same lane.
template <int HD>
__device__ __forceinline__ void norm_rope_head(const Params &p, float (&v)[HD / 32], const float (&gain)[HD / 32],
                                               const float2 (&cs)[HD / 64]) {
  static_assert((HD & (HD - 1)) == 0, "head_dim a power of two");
  constexpr int EPL = HD / 32;
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < EPL; ++k) ss = fmaf(v[k], v[k], ss);
  ss = warp_sum(ss);
  const float rs = inv_sqrt_rn(ss * (1.0f / static_cast<float>(HD)) + p.eps);   // HD a power of two: = ss / HD
#pragma unroll
  for (int k = 0; k < EPL; ++k) v[k] = v[k] * rs * gain[k];
#pragma unroll
  for (int k = 0; k < EPL / 2; ++k) {
    const float a = v[k], b = v[k + EPL / 2];
    v[k] = a * cs[k].x - b * cs[k].y;
    v[k + EPL / 2] = b * cs[k].x + a * cs[k].y;
  }
}

// the gain and rotary factors norm_rope_head needs for this lane (loaded
// before the head vector is polled, so their latency overlaps the wait)
template <int HD>
__device__ __forceinline__ void norm_rope_factors(const Params &p, const uint16_t *gain, int f, int P,
                                                  float (&g)[HD / 32], float2 (&cs)[HD / 64]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 0; k < HD / 32; ++k) g[k] = bf2f(gain[lane + 32 * k]);
#pragma unroll
  for (int k = 0; k < HD / 64; ++k) {
    const int i = lane + 32 * k;                         // pair index < d/2
    const int pos = stream_pos(p, f, pair_stream(p, i), P);
    cs[k] = p.rope[static_cast<size_t>(pos) * (HD / 2) + i];
  }
}

// Merge of split-KV chunk states for one output element (head j, dim i):
// chunks 0..C-2 were published as tagged words (o at pc + c*cstride + i, the
// chunk's running max m and sum l at + hd and + hd + 1); chunk C-1 is this
// CTA's own (o_own, m_own, l_own).  All loads of a round are issued before
// any is checked.  Returns sum_c e^(m_c - M) o_c / sum_c e^(m_c - M) l_c with
// M = max_c m_c, accumulated in chunk order.
static __device__ __noinline__ float merge_polled_chunks(const Params &p, SmemCtl &S, const unsigned long long *pc,
                                                         size_t cstride, int hd, int i, int C, float o_own,
                                                         float m_own, float l_own, unsigned tag) {
  constexpr int N = MAX_POLL_CHUNKS - 1;
  unsigned long long wo[N], wm[N], wl[N];
#pragma unroll
  for (int c = 0; c < N; ++c) {
    wo[c] = wm[c] = wl[c] = static_cast<unsigned long long>(tag) << 32;
    if (c < C - 1) {
      wo[c] = ll_load(pc + c * cstride + i);
      wm[c] = ll_load(pc + c * cstride + hd);
      wl[c] = ll_load(pc + c * cstride + hd + 1);
    }
  }
  Deadline dl;
  int n = 0;
  for (;;) {
    bool ok = true;
#pragma unroll
    for (int c = 0; c < N; ++c) ok &= (ll_tag(wo[c]) == tag) & (ll_tag(wm[c]) == tag) & (ll_tag(wl[c]) == tag);
    if (ok) break;
#pragma unroll
    for (int c = 0; c < N; ++c) {
      if (ll_tag(wo[c]) != tag) wo[c] = ll_load(pc + c * cstride + i);
      if (ll_tag(wm[c]) != tag) wm[c] = ll_load(pc + c * cstride + hd);
      if (ll_tag(wl[c]) != tag) wl[c] = ll_load(pc + c * cstride + hd + 1);
    }
    if ((++n & 15) == 0) {
      if (flag(S, F_ABORT) || ld_relaxed_i32(p.err) != 0) break;
      if (dl.expired(p.spin_ns)) {
        set_err(p, MK_ERR_TIMEOUT_D);
        flag(S, F_ABORT) = 1;
        break;
      }
    }
  }
  float M = -INFINITY;
#pragma unroll
  for (int c = 0; c < N + 1; ++c)
    if (c < C) M = fmaxf(M, c < C - 1 ? ll_val(wm[c < N ? c : 0]) : m_own);
  float os = 0.f, lsum = 0.f;
#pragma unroll
  for (int c = 0; c < N + 1; ++c) {
    if (c < C) {
      const bool own = (c == C - 1);
      const int k = c < N ? c : 0;
      const float mc = own ? m_own : ll_val(wm[k]);
      const float sc = expf(mc - M);
      os = fmaf(sc, own ? o_own : ll_val(wo[k]), os);
      lsum = fmaf(sc, own ? l_own : ll_val(wl[k]), lsum);
    }
  }
  return os / lsum;
}

// The last CTA of kv head g merges its C chunk states from p.part (the same
// arithmetic as merge_polled_chunks); out of line: only long contexts (more
// chunks than the polled merge takes) run it.
static __device__ __noinline__ void merge_ticket_chunks(const Params &p, unsigned long long *attn_ll, int g, int grp,
                                                        int hd, int C, unsigned tag) {
  for (int e = threadIdx.x; e < grp * hd; e += NCT) {
    const int h = e / hd, i = e - h * hd;
    const int j = g * grp + h;
    const float *src = p.part + static_cast<size_t>(j) * p.max_chunks * (hd + 2);
    float M = -INFINITY;
    for (int cc = 0; cc < C; ++cc) M = fmaxf(M, __ldcg(src + cc * (hd + 2) + hd));
    float os = 0.f, lsum = 0.f;
    for (int cc = 0; cc < C; ++cc) {
      const float sc = expf(__ldcg(src + cc * (hd + 2) + hd) - M);
      os = fmaf(sc, __ldcg(src + cc * (hd + 2) + i), os);
      lsum = fmaf(sc, __ldcg(src + cc * (hd + 2) + hd + 1), lsum);
    }
    ll_store_rep(p, attn_ll + ll_slot(p.geo[GV_O], j * hd + i), os / lsum, tag);
  }
}

// One attention phase: this CTA's (kv head, chunk) units.  BLOCKS picks the
// score loop: 8 positions per warp at a time with one multi-slot reduction
// (the default), or one position per warp with a warp sum per head (the
// 1.7B plan, whose staged GEMV allocates fewer registers next to it).  Both
// are the same online softmax; their summation orders differ.
template <int HD, int GRP, bool BLOCKS = true>
__device__ void attention_phase(const Params &p, SmemCtl &S, unsigned char *ring, int l, int f, int cta,
                                unsigned tag, RingPos &rp, int gp, const AttnSched &as) {
  constexpr int EPL = HD / 32;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int P = as.P;
  constexpr int TP = STAGE_BYTES / (4 * HD);   // positions per ring tile (K rows + V rows)
  // polled merge needs every unit on its own CTA (a CTA never waits for itself)
  const bool poll_merge = as.C > 1 && as.C <= p.poll_cm && as.units <= p.G;
  const LayerPtrs &LW = S.layers[l];
  const unsigned long long *qkv_ll = p.ll.qkv + static_cast<size_t>(l) * (p.Hq + 2 * p.Hkv) * HD +
                                     (cta % p.ll_rep) * p.ll_cs;
  unsigned long long *attn_ll = p.ll.attn + static_cast<size_t>(l) * p.Hq * HD;

  for (int u = cta; u < as.units; u += p.G) {
    // (a division costs hundreds of cycles here: the first unit's indices come with the schedule)
    const int g = u == cta ? as.g0 : u / as.C;
    const int c = u == cta ? as.c0 : u - g * as.C;
    const int a = c * as.cs, b = min(a + as.cs, as.ctx);
    const int pend = min(b, P);                // positions < P come through the ring
    const bool has_cur = (b == as.ctx);        // this chunk holds the new position P
    cons_sync();                               // shared scratch reuse across units

    // ---- QK-norm + RoPE of the group's queries; append K/V of position P ----
    const int njobs = GRP + (has_cur ? 2 : 0);
    for (int job = w; job < njobs; job += NCW) {
      // job < GRP: query head g*GRP + job; GRP: this position's key; GRP+1: its value
      const unsigned long long *src = job < GRP ? qkv_ll + (g * GRP + job) * HD
                                    : job == GRP ? qkv_ll + (p.Hq + g) * HD
                                                 : qkv_ll + (p.Hq + p.Hkv + g) * HD;
      float gv[EPL];
      float2 csv[EPL / 2];
      if (job <= GRP) norm_rope_factors<HD>(p, job < GRP ? LW.q_norm : LW.k_norm, f, P, gv, csv);
      unsigned long long wv[EPL];
#pragma unroll
      for (int k = 0; k < EPL; ++k) wv[k] = ll_load(src + lane + 32 * k);
      ll_settle<EPL, 32>(p, S, src + lane, tag, wv);
      float v[EPL];
#pragma unroll
      for (int k = 0; k < EPL; ++k) v[k] = ll_val(wv[k]);
      if (job <= GRP) norm_rope_head<HD>(p, v, gv, csv);
      if (job < GRP) {
#pragma unroll
        for (int k = 0; k < EPL; ++k) S.qs[job * HD + lane + 32 * k] = v[k] * p.inv_sqrt_d;
      } else {
        // this position's key (job GRP) or value, rounded to bf16 into the cache
        uint16_t *dst = (job == GRP ? p.kcache : p.vcache) +
                        ((static_cast<size_t>(l) * p.Hkv + g) * p.max_seq + P) * HD;
        uint16_t *cur = job == GRP ? S.kcur : S.vcur;
#pragma unroll
        for (int k = 0; k < EPL; ++k) {
          const uint16_t bb = f2bf(v[k]);
          dst[lane + 32 * k] = bb;
          cur[lane + 32 * k] = bb;
        }
        fence_proxy_async_global();
      }
    }
    cons_sync();
    trace_mark(p, gp, cta, 1);

    float q[GRP][EPL], o[GRP][EPL], m[GRP], ls[GRP];
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) { q[h][e] = S.qs[h * HD + lane * EPL + e]; o[h][e] = 0.f; }
      m[h] = -INFINITY;
      ls[h] = 0.f;
    }
    if constexpr (BLOCKS) {
    // ---- scores and online softmax, 8 positions per warp at a time -----------
    // Lane l holds dims l*EPL .. l*EPL+EPL-1 of q, of every key and value row
    // and of the output.  A block of 8 positions: per-lane partial scores of
    // the 8 x GRP (head, position) pairs, one multi-slot warp reduction (lane
    // holds slot (h * 8 + j) after it), the block's maximum and sum per head
    // by shuffles among the lanes of a head, then the rescaled output update.
    constexpr int NSL = 8 * GRP;
    constexpr int LPS = NSL >= 32 ? 0 : NSL >= 16 ? 1 : NSL >= 8 ? 2 : 3;   // log2 lanes per slot
    // positions j < nv of rows kb + j * HD (keys) and vb + j * HD (values)
    auto block = [&](const uint16_t *kb, const uint16_t *vb, int nv) {
      float sp[NSL], vv[8][EPL];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int jj = min(j, nv - 1);        // past the last position: re-read it, masked below
        float kk[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          kk[e] = bf2f(kb[jj * HD + lane * EPL + e]);
          vv[j][e] = bf2f(vb[jj * HD + lane * EPL + e]);
        }
#pragma unroll
        for (int h = 0; h < GRP; ++h) {
          float x = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) x = fmaf(q[h][e], kk[e], x);
          sp[h * 8 + j] = x;
        }
      }
      const float sv = warp_multi_reduce<NSL>(sp, lane);
      const int sl = lane >> LPS, hj = sl >> 3, jl = sl & 7;
      const bool valid = jl < nv;
      // block maximum of each head, then the new running maximum
      float bm = valid ? sv : -INFINITY;
#pragma unroll
      for (int off = 1 << LPS; off < (8 << LPS); off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
      float mn[GRP], sc[GRP];
      float m_own = 0.f;
#pragma unroll
      for (int h = 0; h < GRP; ++h) {
        mn[h] = fmaxf(m[h], __shfl_sync(0xffffffffu, bm, (h * 8) << LPS));
        sc[h] = expf(m[h] - mn[h]);
        if (hj == h) m_own = mn[h];
      }
      const float pe = valid ? expf(sv - m_own) : 0.f;
      float bs = pe;
#pragma unroll
      for (int off = 1 << LPS; off < (8 << LPS); off <<= 1) bs += __shfl_xor_sync(0xffffffffu, bs, off);
#pragma unroll
      for (int h = 0; h < GRP; ++h) {
        ls[h] = ls[h] * sc[h] + __shfl_sync(0xffffffffu, bs, (h * 8) << LPS);
        m[h] = mn[h];
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[h][e] *= sc[h];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float pj = __shfl_sync(0xffffffffu, pe, (h * 8 + j) << LPS);
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[h][e] = fmaf(pj, vv[j][e], o[h][e]);
        }
      }
    };
    for (int p0 = a; p0 < pend; p0 += TP) {
      const int np = min(TP, pend - p0);
      const int slot = rp.slot;
      wait_full(p, S, slot, rp.par);
      const uint16_t *kt = reinterpret_cast<const uint16_t *>(ring + static_cast<size_t>(slot) * STAGE_BYTES);
      const uint16_t *vt = kt + static_cast<size_t>(np) * HD;
      // warp w: positions 8w .. 8w+7 of every 8 * NCW
      for (int j0 = 8 * w; j0 < np; j0 += 8 * NCW) block(kt + j0 * HD, vt + j0 * HD, min(8, np - j0));
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[slot]);
      rp.next(p.stages);
    }
    if (has_cur && w == NCW - 1) block(S.kcur, S.vcur, 1);

    } else {
    // ---- (!BLOCKS) scores and online softmax, one warp per position ----------
    // score of one cached position for every head of the group (warp-reduced)
    auto score = [&](const float (&kk)[EPL], float (&sv)[GRP]) {
#pragma unroll
      for (int h = 0; h < GRP; ++h) {
        float x = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) x = fmaf(q[h][e], kk[e], x);
        sv[h] = warp_sum(x);
      }
    };
    // online-softmax update with one position's scores and value row
    auto update = [&](const float (&sv)[GRP], const float (&vv)[EPL]) {
#pragma unroll
      for (int h = 0; h < GRP; ++h) {
        const float mn = fmaxf(m[h], sv[h]);
        const float sc = expf(m[h] - mn);
        const float pe = expf(sv[h] - mn);
        ls[h] = ls[h] * sc + pe;
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[h][e] = fmaf(pe, vv[e], o[h][e] * sc);
        m[h] = mn;
      }
    };
    auto visit = [&](const float (&kk)[EPL], const float (&vv)[EPL]) {
      float sv[GRP];
      score(kk, sv);
      update(sv, vv);
    };
    for (int p0 = a; p0 < pend; p0 += TP) {
      const int np = min(TP, pend - p0);
      const int slot = rp.slot;
      wait_full(p, S, slot, rp.par);
      const unsigned char *st = ring + static_cast<size_t>(slot) * STAGE_BYTES;
      const uint16_t *kt = reinterpret_cast<const uint16_t *>(st) + lane * EPL;
      const uint16_t *vt = kt + static_cast<size_t>(np) * HD;
      // two positions at a time: their scores' warp reductions overlap; the
      // updates still run in position order (the same arithmetic as one by one)
      int i = w;
      for (; i + NCW < np; i += 2 * NCW) {
        float kk[2][EPL], vv[2][EPL], sv[2][GRP];
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            kk[j][e] = bf2f(kt[static_cast<size_t>(i + j * NCW) * HD + e]);
            vv[j][e] = bf2f(vt[static_cast<size_t>(i + j * NCW) * HD + e]);
          }
#pragma unroll
        for (int j = 0; j < 2; ++j) score(kk[j], sv[j]);
#pragma unroll
        for (int j = 0; j < 2; ++j) update(sv[j], vv[j]);
      }
      for (; i < np; i += NCW) {
        float kk[EPL], vv[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          kk[e] = bf2f(kt[static_cast<size_t>(i) * HD + e]);
          vv[e] = bf2f(vt[static_cast<size_t>(i) * HD + e]);
        }
        visit(kk, vv);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[slot]);
      rp.next(p.stages);
    }
    if (has_cur && w == NCW - 1) {
      float kk[EPL], vv[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) { kk[e] = bf2f(S.kcur[lane * EPL + e]); vv[e] = bf2f(S.vcur[lane * EPL + e]); }
      visit(kk, vv);
    }

    }

    // ---- merge the 8 warps, then the chunks ---------------------------------
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) S.ow[w][h * HD + lane * EPL + e] = o[h][e];
      if (lane == 0) { S.mw[w][h] = m[h]; S.lw[w][h] = ls[h]; }
    }
    cons_sync();
    for (int e = t; e < GRP * HD; e += NCT) {
      const int h = e / HD, i = e % HD;
      float M = -INFINITY;
      for (int ww = 0; ww < NCW; ++ww) M = fmaxf(M, S.mw[ww][h]);
      float os = 0.f, lsum = 0.f;
      for (int ww = 0; ww < NCW; ++ww) {
        const float sc = expf(S.mw[ww][h] - M);
        os = fmaf(sc, S.ow[ww][e], os);
        lsum = fmaf(sc, S.lw[ww][h], lsum);
      }
      const int j = g * GRP + h;
      if (as.C == 1) {
        ll_store_rep(p, attn_ll + ll_slot(p.geo[GV_O], j * HD + i), os / lsum, tag);
      } else if (poll_merge) {
        // chunks publish (o, m, l); the chunk holding the new position merges
        unsigned long long *pc = p.ll.part + (static_cast<size_t>(l) * MAX_POLL_CHUNKS * p.Hq + j) * (HD + 2);
        const size_t cstride = static_cast<size_t>(p.Hq) * (HD + 2);
        if (c < as.C - 1) {
          ll_store(pc + c * cstride + i, os, tag);
          if (i == 0) {
            ll_store(pc + c * cstride + HD, M, tag);
            ll_store(pc + c * cstride + HD + 1, lsum, tag);
          }
        } else {
          const float y = merge_polled_chunks(p, S, pc, cstride, HD, i, as.C, os, M, lsum, tag);
          ll_store_rep(p, attn_ll + ll_slot(p.geo[GV_O], j * HD + i), y, tag);
        }
      } else {
        float *dst = p.part + (static_cast<size_t>(j) * p.max_chunks + c) * (HD + 2);
        dst[i] = os;
        if (i == 0) { dst[HD] = M; dst[HD + 1] = lsum; }
      }
    }
    if (as.C > 1 && !poll_merge) {
      // the last CTA to finish a chunk of kv head g merges all C chunks
      cons_sync();
      if (t == 0) {
        __threadfence();
        const unsigned old = atomicAdd(p.tickets + g, 1u);
        const int last = (old == static_cast<unsigned>(as.C - 1)) ? 1 : 0;
        if (last) {
          atomicExch(p.tickets + g, 0u);
          __threadfence();
        }
        flag(S, F_LAST) = last;
      }
      cons_sync();
      if (flag(S, F_LAST)) merge_ticket_chunks(p, attn_ll, g, GRP, HD, as.C, tag);
    }
  }
  trace_mark(p, gp, cta, 2);
}

template <int HD>
__device__ void attention_dispatch(const Params &p, SmemCtl &S, unsigned char *ring, int l, int f, int cta,
                                   unsigned tag, RingPos &rp, int gp, const AttnSched &as) {
  switch (p.grp) {
    case 1: attention_phase<HD, 1>(p, S, ring, l, f, cta, tag, rp, gp, as); break;
    case 2: attention_phase<HD, 2>(p, S, ring, l, f, cta, tag, rp, gp, as); break;
    case 4: attention_phase<HD, 4>(p, S, ring, l, f, cta, tag, rp, gp, as); break;
    default: if constexpr (HD * 8 <= MAX_GRP_HD) attention_phase<HD, 8>(p, S, ring, l, f, cta, tag, rp, gp, as); break;
  }
}

// ---------------------------------------------------------------------------
// producer: walks the same tile schedule as the consumers
// ---------------------------------------------------------------------------
struct Producer {
  const Params &p;
  SmemCtl &S;
  unsigned char *ring;
  uint64_t pol_w, pol_kv;
  RingPos rp;
  bool stop = false;
  AttnSched as;
  int as_f = -1;

  __device__ Producer(const Params &pp, SmemCtl &SS, unsigned char *r) : p(pp), S(SS), ring(r) {
    pol_w = policy_evict_first();
    pol_kv = policy_evict_normal();
  }

  // claim the next ring slot (waits until the consumers released it)
  __device__ unsigned char *claim(int &slot) {
    slot = rp.slot;
    if (rp.it >= static_cast<uint32_t>(p.stages)) {
      const uint32_t par = rp.par ^ 1u;                       // the slot's previous fill

      if (!mbar_try_wait(&S.empty[slot], par)) {
        Deadline dl;
        int n = 0;
        while (!mbar_try_wait(&S.empty[slot], par)) {
          if ((++n & 63) == 0) {
            if (flag(S, F_ABORT)) { stop = true; return nullptr; }
            if (dl.expired(p.spin_ns)) { set_err(p, MK_ERR_TIMEOUT_D); stop = true; return nullptr; }
          }
        }
      }
    }
    if (flag(S, F_ABORT)) { stop = true; return nullptr; }
    return ring + static_cast<size_t>(slot) * STAGE_BYTES;
  }

  __device__ void gemv_tiles(int kind, int layer, int cta) {
    const GemvGeom g = p.geo[kind];
    const int r0 = S.rr[kind][0], r1 = S.rr[kind][1];
    const uint32_t rowb = static_cast<uint32_t>(g.K) * 2u;
    for (int a = r0; a < r1 && !stop; a += g.RT) {
      const int nr = min(g.RT, r1 - a);
      int slot;
      unsigned char *dst = claim(slot);
      if (!dst) return;
      const uint16_t *src[3];
      uint32_t bytes[3], offs[3] = {0, 0, 0};
      int n = 0;
      if (kind == GV_QKV) {
        const int qr = p.Hq * p.d, kr = p.Hkv * p.d;
        const int segs[4] = {0, qr, qr + kr, qr + 2 * kr};
        const uint16_t *mats[3] = {S.layers[layer].wq, S.layers[layer].wk, S.layers[layer].wv};
        for (int s = 0; s < 3; ++s) {
          const int lo = max(a, segs[s]), hi = min(a + nr, segs[s + 1]);
          if (lo < hi) {
            src[n] = mats[s] + static_cast<size_t>(lo - segs[s]) * g.K;
            bytes[n] = static_cast<uint32_t>(hi - lo) * rowb;
            ++n;
          }
        }
      } else if (kind == GV_GU) {
        src[0] = S.layers[layer].w_gate + static_cast<size_t>(a) * g.K;
        src[1] = S.layers[layer].w_up + static_cast<size_t>(a) * g.K;
        bytes[0] = bytes[1] = static_cast<uint32_t>(nr) * rowb;
        // up rows follow the gate rows; in the paired layout (staged, even
        // rows per thread) always at row RT, so that a warp holds the gate and
        // the up row of the same output in every tile, the last one included
        offs[1] = (g.fast == 1 && g.RPTP % 2 == 0) ? static_cast<uint32_t>(g.RT) * rowb : bytes[0];
        n = 2;
      } else {
        const uint16_t *base = kind == GV_O ? S.layers[layer].wo
                             : kind == GV_DOWN ? S.layers[layer].w_down
                                               : p.lm_head;
        src[0] = base + static_cast<size_t>(a) * g.K;
        bytes[0] = static_cast<uint32_t>(nr) * rowb;
        n = 1;
      }
      uint32_t total = 0;
      for (int i = 0; i < n; ++i) total += bytes[i];
      mbar_arrive_expect_tx(&S.full[slot], total);
      uint32_t off = 0;
      for (int i = 0; i < n; ++i) {
        if (i > 0) off = kind == GV_GU ? offs[i] : off + bytes[i - 1];
        bulk_load(dst + off, src[i], bytes[i], &S.full[slot], pol_w);
      }
      rp.next(p.stages);
    }
  }

  template <int HD>
  __device__ void kv_tiles(int l, int f, int cta) {
    if (as_f != f) {
      as = attn_sched(p, f);
      as_f = f;
    }
    constexpr int TP = STAGE_BYTES / (4 * HD);
    bool guarded = false;
    for (int u = cta; u < as.units && !stop; u += p.G) {
      const int g = u / as.C, c = u % as.C;
      const int a = c * as.cs, b = min(a + as.cs, as.ctx);
      const int pend = min(b, as.P);
      for (int p0 = a; p0 < pend && !stop; p0 += TP) {
        if (!guarded) {
          // positions up to P-1 were appended by earlier forwards of this
          // launch: wait until this CTA's consumers have passed the grid
          // barrier that closed forward f-1
          if (f > 0) {
            Deadline dl;
            int n = 0;
            while (ld_acquire_cta(&S.flags[F_FWD_DONE]) < f) {
              if ((++n & 63) == 0) {
                if (flag(S, F_ABORT)) { stop = true; return; }
                if (dl.expired(p.spin_ns)) { set_err(p, MK_ERR_TIMEOUT_D); stop = true; return; }
              }
            }
          }
          fence_proxy_async_global();
          guarded = true;
        }
        const int np = min(TP, pend - p0);
        int slot;
        unsigned char *dst = claim(slot);
        if (!dst) return;
        const size_t row0 = (static_cast<size_t>(l) * p.Hkv + g) * p.max_seq + p0;
        const uint32_t bytes = static_cast<uint32_t>(np) * HD * 2u;
        mbar_arrive_expect_tx(&S.full[slot], 2u * bytes);
        bulk_load(dst, p.kcache + row0 * HD, bytes, &S.full[slot], pol_kv);
        bulk_load(dst + bytes, p.vcache + row0 * HD, bytes, &S.full[slot], pol_kv);
        rp.next(p.stages);
      }
    }
  }

  // wait for every copy this producer issued (each slot's latest fill)
  __device__ void drain() {
    const uint32_t ns = static_cast<uint32_t>(p.stages);
    const uint32_t it = rp.it;
    const uint32_t used = it < ns ? it : ns;
    for (uint32_t s = 0; s < used; ++s) {
      const uint32_t last = ((it - 1 - s) / ns) * ns + s;     // largest fill index of slot s
      const uint32_t par = (last / ns) & 1u;
      Deadline dl;
      int n = 0;
      while (!mbar_try_wait(&S.full[s], par)) {
        if ((++n & 63) == 0 && dl.expired(p.spin_ns)) { set_err(p, MK_ERR_TIMEOUT_D); break; }
      }
    }
  }
};

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
// One GEMV phase.  Plan kernels: the split-K phases (O, down) inline, the
// staged ones through one shared out-of-line copy (the instruction working
// set of a forward is what limits the phase chain: three inline copies of the
// staged code measured 9% slower).  General kernel: run-time dispatch.
template <class PL, int KIND>
__device__ __forceinline__ void gemv_run(const Params &p, SmemCtl &S, unsigned char *ring, int layer, int f, int cta,
                                         int in_id, unsigned tag, RingState &st, int gp) {
  constexpr int fast = PL::spec[KIND][0], kpt = PL::spec[KIND][1], rpt = PL::spec[KIND][2], bt = PL::spec[KIND][3];
  if constexpr (PL::fixed && fast == 1) {
    st = gemv_fast<kpt, rpt, bt, true>(p, S, ring, KIND, layer, f, cta, in_id, tag, st, gp);
  } else if constexpr (PL::fixed) {
    gemv_fast_body<kpt, rpt, bt, fast == 1>(p, S, ring, KIND, layer, f, cta, in_id, tag, st.rp, st.rb, gp);
  } else {
    st = gemv_dispatch(p, S, ring, KIND, layer, f, cta, in_id, tag, st, gp);
  }
}

template <int HD, class PL>
__global__ void __launch_bounds__(NTHREADS, 1) mk_decode_kernel(const __grid_constant__ Params pg) {
  static_assert(!PL::fixed || PL::hd == HD, "a plan is compiled for its head_dim");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  SmemCtl &S = *reinterpret_cast<SmemCtl *>(smem_raw);
  unsigned char *ring = smem_raw + RING_OFFSET;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int cta = blockIdx.x;
  {
    // every phase reads the launch parameters: keep them in shared memory,
    // where a read never waits on a constant-cache refill
    const uint32_t *src = reinterpret_cast<const uint32_t *>(&pg);
    uint32_t *dst = reinterpret_cast<uint32_t *>(&S.prm);
    for (int i = tid; i < static_cast<int>(sizeof(Params) / 4); i += NTHREADS) dst[i] = src[i];
  }
  __syncthreads();
  if (pg.blk) {
    // a replayed per-op graph: the call's fields live in device memory
    if (tid == 0) {
      const CallBlock &b = *pg.blk;
      S.prm.in_ids = b.in_ids;
      S.prm.out_ids = b.out_ids;
      S.prm.embeds = b.embeds;
      S.prm.pos3 = b.pos3;
      S.prm.logits = b.logits;
      S.prm.hidden = b.hidden;
      S.prm.trace = b.trace;
      S.prm.mbox_ids = b.mbox_ids;
      S.prm.mbox_count = b.mbox_count;
      S.prm.cb_books = b.cb_books;
      S.prm.cb_text = b.cb_text;
      S.prm.cb_codes = b.cb_codes;
      S.prm.cb_text_ids = b.cb_text_ids;
      S.prm.cb_n = b.cb_n;
      S.prm.cb_rows = b.cb_rows;
      S.prm.cb_text_rows = b.cb_text_rows;
      S.prm.cb_n_rows = b.cb_n_rows;
      S.prm.spin_ns = b.spin_ns;
      S.prm.n_in = b.n_in;
      S.prm.n_fwd = b.n_fwd;
      S.prm.pos0 = b.pos0;
      S.prm.n_embed_rows = b.n_embed_rows;
      S.prm.chunks_override = b.chunks_override;
      S.prm.op_fwd = b.op_fwd;
      S.prm.tag0 = b.tag0;
    }
    __syncthreads();
  }
  const Params &p = S.prm;
  const int NPH = 5 * p.L + 1;

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], NCW);
    }
    fence_mbar_init();
    // this CTA's rows of every GEMV phase (the O and down ranges are also the
    // residual rows it owns), computed once instead of in every phase
    for (int k = 0; k < GV_COUNT; ++k) {
      split_range(p.geo[k].rows, p.G, cta, S.rr[k][0], S.rr[k][1]);
      S.nt[k] = (S.rr[k][1] - S.rr[k][0] + p.geo[k].RT - 1) / p.geo[k].RT;
    }
    flag(S, F_ABORT) = (p.per_op && ld_relaxed_i32(p.err) != 0) ? 1 : 0;
    flag(S, F_PROD_DONE) = 0;
    flag(S, F_FWD_DONE) = p.per_op ? INT_MAX : 0;
    flag(S, F_LAST) = 0;
  }
  {
    // the per-layer weight pointers, read by every phase, live in shared memory
    const unsigned long long *src = reinterpret_cast<const unsigned long long *>(p.layers);
    unsigned long long *dst = reinterpret_cast<unsigned long long *>(S.layers);
    const int n = p.L * static_cast<int>(sizeof(LayerPtrs) / sizeof(unsigned long long));
    for (int i = tid; i < n; i += NTHREADS) dst[i] = __ldg(src + i);
  }
  __syncthreads();
  if (flag(S, F_ABORT)) return;   // per-op launch after an earlier failure: nothing runs

  int gp_begin, gp_end;
  bool final_select;
  // (forward, phase) of gp_begin, advanced with gp (no division in the loop)
  int f0 = 0, ph0 = 0;
  if (p.per_op) {
    if (p.op_phase >= NPH) { gp_begin = gp_end = 0; final_select = true; }
    else {
      gp_begin = p.op_fwd * NPH + p.op_phase;
      gp_end = gp_begin + 1;
      final_select = false;
      f0 = p.op_fwd;
      ph0 = p.op_phase;
    }
  } else {
    gp_begin = 0;
    gp_end = p.n_fwd * NPH;
    final_select = true;
  }

  if (warp == NCW) {
    // ---------------- producer warp (lane 0 issues everything) ----------------
    if (lane == 0) {
      Producer pr(p, S, ring);
      int f = f0, ph = ph0;
      for (int gp = gp_begin; gp < gp_end && !pr.stop; ++gp) {
        if (ph == 5 * p.L) {
          pr.gemv_tiles(GV_LM, 0, cta);
        } else {
          const int l = ph / 5;
          switch (ph - 5 * l) {
            case 0: pr.gemv_tiles(GV_QKV, l, cta); break;
            case 1: pr.kv_tiles<HD>(l, f, cta); break;
            case 2: pr.gemv_tiles(GV_O, l, cta); break;
            case 3: pr.gemv_tiles(GV_GU, l, cta); break;
            default: pr.gemv_tiles(GV_DOWN, l, cta); break;
          }
        }
        if (++ph == NPH) { ph = 0; ++f; }
      }
      pr.drain();
      st_release_cta(&S.flags[F_PROD_DONE], 1);
    }
    return;
  }

  // -------------------------- consumer warps ----------------------------------
  // Phases hand their outputs to the next phase as tagged words (no barrier);
  // only the LM head ends with a grid barrier, which publishes the argmax
  // candidates and orders this forward's KV-cache writes before the next one.
  RingState st;
  RingPos &rp = st.rp;
  unsigned bar_target = 0;
  int in_id = 0;
  bool ok = true;
  AttnSched as;                 // the split-KV schedule of forward as_f (the same for all its layers)
  int as_f = -1;
  int f = f0, ph = ph0;
  for (int gp = gp_begin; gp < gp_end && ok; ++gp, (++ph == NPH) ? (ph = 0, ++f) : 0) {
    const unsigned tag = p.tag0 + static_cast<unsigned>(f);
    trace_mark(p, gp, cta, 0);
    if (ph == 5 * p.L) {
      gemv_run<PL, GV_LM>(p, S, ring, 0, f, cta, in_id, tag, st, gp);
      if (!p.per_op) {
        ok = grid_barrier(p, S, bar_target, f, cta);
        if (tid == 0) st_release_cta(&S.flags[F_FWD_DONE], f + 1);
      }
    } else {
      const int l = ph / 5, k = ph - 5 * l;
      if (k == 0 && l == 0) {
        // the token of this forward: teacher-forced input, or fed back in-kernel
        int prev = 0;
        if (f > 0) prev = select_token(p, S, f - 1, cta, false);
        int id;
        if (f < p.n_in) id = p.in_ids[f];
        else if (f > 0) id = prev;
        else id = *p.last_id;
        const bool bad = (id >= 0) ? (id >= p.vocab_in)
                       : p.cb_codes ? !code_row_ok(p, -(id + 1))
                                    : (p.embeds == nullptr || -(id + 1) >= p.n_embed_rows);
        if (bad) {
          if (tid == 0) set_err(p, MK_ERR_BAD_TOKEN_D);
          ok = false;
          break;
        }
        in_id = id;
      }
      if (k == 1 && as_f != f) {
        as = attn_sched(p, f);
        as_f = f;
      }
      switch (k) {
        case 0: gemv_run<PL, GV_QKV>(p, S, ring, l, f, cta, in_id, tag, st, gp); break;
        case 1:
          if constexpr (PL::fixed) attention_phase<HD, PL::grp, PL::attn_blocks>(p, S, ring, l, f, cta, tag, rp, gp, as);
          else attention_dispatch<HD>(p, S, ring, l, f, cta, tag, rp, gp, as);
          break;
        case 2: gemv_run<PL, GV_O>(p, S, ring, l, f, cta, in_id, tag, st, gp); break;
        case 3: gemv_run<PL, GV_GU>(p, S, ring, l, f, cta, in_id, tag, st, gp); break;
        default: gemv_run<PL, GV_DOWN>(p, S, ring, l, f, cta, in_id, tag, st, gp); break;
      }
    }
    trace_mark(p, gp, cta, 3);
    if (p.per_op) {
      cons_sync();
      ok = flag(S, F_ABORT) == 0;
    }
  }
  cons_sync();
  if (ok && final_select && flag(S, F_ABORT) == 0) select_token(p, S, p.n_fwd - 1, cta, true);

  // ---- shutdown: stop the producer and wait until its copies have landed ----
  cons_sync();
  if (tid == 0) {
    flag(S, F_ABORT) = 1;
    Deadline dl;
    int n = 0;
    while (ld_acquire_cta(&S.flags[F_PROD_DONE]) == 0) {
      if ((++n & 255) == 0 && dl.expired(2 * p.spin_ns)) { set_err(p, MK_ERR_TIMEOUT_D); break; }
    }
  }
  cons_sync();
}

}  // namespace mk
