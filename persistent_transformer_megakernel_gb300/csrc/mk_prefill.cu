// Batched prompt prefill: the n prompt forwards of a decode call computed all
// at once per layer.  The projections are dense contractions with M = prompt
// tokens and run on the tensor cores (csrc/mk_gemm.cu: tcgen05.mma, bf16
// operands staged by TMA, fp32 accumulators in tensor memory); every fp32
// activation enters them as three bf16 terms (hi + mid + lo, 24 significant
// bits, as many as fp32 holds), each term's products in their own fp32
// accumulator, so the products lose nothing to the bf16 operand format.  The
// causal GQA attention runs on the tensor cores too (csrc/mk_pfattn.cu).  The
// rest -- RMSNorm, QK-norm, RoPE / MRoPE, the bf16 KV append, attention over the cache, residual adds, SiLU * up, greedy argmax -- are the
// kernels below.  The KV cache it fills is the decode kernel's, so decoding
// continues from the prompt's last position (page A, "Porting a 1,200-line
// persistent CUDA megakernel to Qwen3-TTS": time to first chunk is what the
// listener waits for).
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "mk_gemm.h"
#include "mk_prefill.h"

namespace mkp {

constexpr int PF_THREADS = 256;

__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
// round-to-nearest-even float -> bf16 bits (NaN kept quiet)
__device__ __forceinline__ uint16_t f2bf(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x40u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// v = hi + mid + lo exactly up to fp32's 24 bits: each term is the bf16
// rounding of what the terms before it left
__device__ __forceinline__ void split3(float v, uint16_t &hi, uint16_t &mid, uint16_t &lo) {
  hi = f2bf(v);
  const float r1 = v - bf2f(hi);
  mid = f2bf(r1);
  lo = f2bf(r1 - bf2f(mid));
}

// a GEMM output element: the sum of its split-K partials (stride apart), in split order
__device__ __forceinline__ float sum_parts(const float *c, size_t stride, int n, size_t i) {
  float v = c[i];
  for (int s = 1; s < n; ++s) v += c[s * stride + i];
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// block-wide sum (PF_THREADS threads), every thread gets the result
__device__ __forceinline__ float block_sum(float v, float *red) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int i = 0; i < PF_THREADS / 32; ++i) t += red[i];
  return t;
}

// x[t] = input row of token t: embedding row (id >= 0) or the caller's fp32
// row -(id+1); hidden[t][0] = x[t] when requested
__global__ void pf_embed(const PfArgs a, int t0, int nt) {
  const int t = blockIdx.x;
  if (t >= nt) return;
  const PfCall &c = *a.call;
  const int id = c.ids[t0 + t];
  const bool bad = id >= 0 ? id >= a.vocab_in : (!c.embeds || -(id + 1) >= c.n_embed_rows);
  if (bad) {
    if (threadIdx.x == 0) atomicCAS(a.err, 0, MK_PF_ERR_BAD_TOKEN);
    return;
  }
  float *x = a.x + static_cast<size_t>(t) * a.H;
  for (int k = threadIdx.x; k < a.H; k += blockDim.x) {
    const float v = id >= 0 ? bf2f(a.embed[static_cast<size_t>(id) * a.H + k])
                            : c.embeds[static_cast<size_t>(-(id + 1)) * a.H + k];
    x[k] = v;
    if (c.hidden) c.hidden[(static_cast<size_t>(t0 + t) * (a.L + 1)) * a.H + k] = v;
  }
}

// Optionally x[t] += y[t] (a residual add) and record hidden[t][layer]; then
// h = x / sqrt(mean(x^2) + eps) * gain as three bf16 terms
__global__ void pf_add_norm_split(const PfArgs a, const float *y, int ny, const uint16_t *gain, int t0, int nt,
                                  int hidden_layer) {
  // y: ny split-K partials of the GEMM output, a.y_stride apart, or NULL
  __shared__ float red[PF_THREADS / 32];
  const int t = blockIdx.x;
  if (t >= nt) return;
  float *x = a.x + static_cast<size_t>(t) * a.H;
  float ss = 0.f;
  for (int k = threadIdx.x; k < a.H; k += blockDim.x) {
    float v = x[k];
    if (y) {
      v = v + sum_parts(y, a.y_stride, ny, static_cast<size_t>(t) * a.H + k);
      x[k] = v;
      if (a.call->hidden && hidden_layer >= 0)
        a.call->hidden[(static_cast<size_t>(t0 + t) * (a.L + 1) + hidden_layer) * a.H + k] = v;
    }
    ss = fmaf(v, v, ss);
  }
  const float tot = block_sum(ss, red);
  const float rs = 1.0f / sqrtf(tot / static_cast<float>(a.H) + a.eps);
  const size_t o = static_cast<size_t>(t) * a.H;
  for (int k = threadIdx.x; k < a.H; k += blockDim.x) {
    const float h = x[k] * rs * bf2f(gain[k]);
    split3(h, a.hs[o + k], a.hs[a.hs_stride + o + k], a.hs[2 * a.hs_stride + o + k]);
  }
}

// v (fp32, n per token) as three bf16 terms (the attention output before O)
__global__ void pf_split(const float *v, int n, int nt, uint16_t *hs, size_t hs_stride) {
  const size_t total = static_cast<size_t>(n) * nt;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    split3(v[i], hs[i], hs[hs_stride + i], hs[2 * hs_stride + i]);
}

// u = silu(gate) * up from the GEMM partials (nc of them, c_stride apart; row t
// holds the n gate columns, then the n up columns), as three bf16 terms
__global__ void pf_silu_mul_split(const float *gu, size_t c_stride, int nc, int n, int nt, uint16_t *hs,
                                  size_t hs_stride) {
  const size_t total = static_cast<size_t>(n) * nt;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const size_t t = i / n, c = i - t * n;
    const size_t gi = t * 2 * n + c;
    const float z = sum_parts(gu, c_stride, nc, gi);
    split3(z / (1.0f + expf(-z)) * sum_parts(gu, c_stride, nc, gi + n), hs[i], hs[hs_stride + i],
           hs[2 * hs_stride + i]);
  }
}


// rotary stream of pair i (the decode kernel's rule: contiguous sections, or
// the interleaved layout of rope_mode 2)
__device__ __forceinline__ int pf_pair_stream(const PfArgs &a, int i) {
  if (a.rope_mode == 0) return 0;
  if (a.rope_mode == 1) return i < a.sec0 ? 0 : (i < a.sec0 + a.sec1 ? 1 : 2);
  const int r = i % 3;
  return ((r == 1 && i < 3 * a.sec1) || (r == 2 && i < 3 * a.sec2)) ? r : 0;
}

// One warp per (token, head job): jobs 0..Hq-1 are query heads (RMSNorm over
// d with q_norm, rotary, times 1/sqrt(d), stored back in place); Hq..Hq+Hkv-1
// keys (RMSNorm with k_norm, rotary, rounded to bf16 into the cache at the
// token's slot); the rest values (rounded to bf16 into the cache).  Lane l
// holds elements l + 32k, so rotate-half partners share a lane.
template <int HD>
__global__ void pf_qk_rope_append(const PfArgs a, int layer, const uint16_t *q_norm, const uint16_t *k_norm,
                                  int t0, int nt) {
  constexpr int EPL = HD / 32;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  const int jobs = a.Hq + 2 * a.Hkv;
  if (warp >= nt * jobs) return;
  const int t = warp / jobs, job = warp % jobs;
  const PfCall &c = *a.call;
  const int P = c.pos0 + t0 + t;
  const int rows = (a.Hq + 2 * a.Hkv) * HD;
  const size_t base = static_cast<size_t>(t) * rows + static_cast<size_t>(job) * HD;
  float v[EPL];
#pragma unroll
  for (int k = 0; k < EPL; ++k) v[k] = sum_parts(a.qkv_p, a.qkv_stride, a.qkv_n, base + lane + 32 * k);
  if (job < a.Hq + a.Hkv) {
    const uint16_t *gain = job < a.Hq ? q_norm : k_norm;
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < EPL; ++k) ss = fmaf(v[k], v[k], ss);
    ss = warp_sum(ss);
    const float rs = 1.0f / sqrtf(ss / static_cast<float>(HD) + a.eps);
#pragma unroll
    for (int k = 0; k < EPL; ++k) v[k] = v[k] * rs * bf2f(gain[lane + 32 * k]);
#pragma unroll
    for (int k = 0; k < EPL / 2; ++k) {
      const int i = lane + 32 * k;
      const int s = pf_pair_stream(a, i);
      int pos = c.pos3 ? c.pos3[static_cast<size_t>(s) * c.n_pos + t0 + t] : P;
      if (pos < 0 || pos >= a.rope_len) {
        atomicCAS(a.err, 0, MK_PF_ERR_BAD_POSITION);
        pos = 0;
      }
      const float2 cs = a.rope[static_cast<size_t>(pos) * (HD / 2) + i];
      const float x0 = v[k], x1 = v[k + EPL / 2];
      v[k] = x0 * cs.x - x1 * cs.y;
      v[k + EPL / 2] = x1 * cs.x + x0 * cs.y;
    }
  }
  if (job < a.Hq) {
#pragma unroll
    for (int k = 0; k < EPL; ++k) a.qkv[base + lane + 32 * k] = v[k] * a.inv_sqrt_d;
  } else {
    const bool key = job < a.Hq + a.Hkv;
    const int g = key ? job - a.Hq : job - a.Hq - a.Hkv;
    uint16_t *dst = (key ? a.kcache : a.vcache) +
                    ((static_cast<size_t>(layer) * a.Hkv + g) * a.max_seq + P) * HD;
#pragma unroll
    for (int k = 0; k < EPL; ++k) dst[lane + 32 * k] = f2bf(v[k]);
  }
}

// Causal GQA attention of the chunk's tokens over the cache, tiled so that
// every cached K / V row read from memory serves many query rows.  A CTA owns
// one kv head g and PF_AR query rows (the GRP heads that read g, for
// PF_AR / GRP consecutive tokens); it walks the cache in tiles of PF_AP
// positions, slots 0 .. the last row's position, with an online softmax per
// row (running max m, sum l, output o).  A tile's K and V rows are widened to
// fp32 in shared memory; the scores q . k are formed in 2 x 4 register blocks
// (rows x positions), the weights e^(s - m) go through shared memory, and the
// output update o <- c o + sum_p w_p V[p] runs in 4-row register blocks.
// Position p of row r is masked (weight 0) when p exceeds r's own position.
// Loads of the next tile are issued before the current tile is computed.
constexpr int PF_AR = 32;                   // query rows per CTA
constexpr int PF_AP = 64;                   // cached positions per tile
constexpr int PF_KPAD = 4;                  // K / Q row padding (floats): conflict-free float4 reads
constexpr int PF_PPAD = 16;                 // weight row padding: the two rows of a warp in distinct banks

template <int HD>
constexpr size_t pf_attention_smem() {
  return sizeof(float) * (static_cast<size_t>(PF_AR) * (HD + PF_KPAD) + static_cast<size_t>(PF_AP) * (HD + PF_KPAD) +
                          static_cast<size_t>(PF_AP) * HD + static_cast<size_t>(PF_AR) * (PF_AP + PF_PPAD) + 2 * PF_AR);
}

template <int HD, int GRP>
__global__ void __launch_bounds__(PF_THREADS) pf_attention(const PfArgs a, int layer, int t0, int nt) {
  static_assert(PF_THREADS == 256 && PF_AR == 32 && PF_AP == 64, "thread mappings below assume these sizes");
  static_assert(PF_AR % GRP == 0, "a CTA holds whole tokens");
  constexpr int TT = PF_AR / GRP;           // tokens per CTA
  constexpr int QS = HD + PF_KPAD;          // row stride of Qs and Ks (floats)
  constexpr int PS = PF_AP + PF_PPAD;       // row stride of Ps
  constexpr int C8 = HD / 8;                // 16-byte pieces of a cached bf16 row
  constexpr int NLD = PF_AP * C8 / PF_THREADS;   // pieces per thread per tile (K and V each)
  constexpr int CPT = HD / 32;              // output columns per thread
  static_assert(NLD * PF_THREADS == PF_AP * C8, "tile pieces divide among the threads");
  extern __shared__ __align__(16) float sm[];
  float *Qs = sm;                           // [PF_AR][QS]
  float *Ks = Qs + PF_AR * QS;              // [PF_AP][QS]
  float *Vs = Ks + PF_AP * QS;              // [PF_AP][HD]
  float *Ps = Vs + PF_AP * HD;              // [PF_AR][PS]
  float *Cs = Ps + PF_AR * PS;              // [PF_AR] rescale factor of the tile
  float *Ls = Cs + PF_AR;                   // [PF_AR] final softmax sums

  const int tid = threadIdx.x;
  const int g = blockIdx.y;
  const int tok0 = blockIdx.x * TT;
  const int ntok = min(TT, nt - tok0);
  const int base_pos = a.call->pos0 + t0;
  const int pmax = base_pos + tok0 + ntok - 1;         // the CTA's last cached slot
  const int rows = (a.Hq + 2 * a.Hkv) * HD;

  // queries: row r = token tok0 + r / GRP, head g * GRP + r % GRP; rows past the
  // chunk hold zeros (and read slot 0 only; never stored)
  for (int e = tid; e < PF_AR * HD / 4; e += PF_THREADS) {
    const int r = e / (HD / 4), c4 = e % (HD / 4);
    const int tt = r / GRP, h = r % GRP;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tt < ntok)
      v = *reinterpret_cast<const float4 *>(a.qkv + static_cast<size_t>(tok0 + tt) * rows +
                                            static_cast<size_t>(g * GRP + h) * HD + 4 * c4);
    *reinterpret_cast<float4 *>(Qs + r * QS + 4 * c4) = v;
  }

  const uint16_t *kb = a.kcache + (static_cast<size_t>(layer) * a.Hkv + g) * a.max_seq * HD;
  const uint16_t *vb = a.vcache + (static_cast<size_t>(layer) * a.Hkv + g) * a.max_seq * HD;
  uint4 kreg[NLD], vreg[NLD];
  // a tile's rows past pmax are zeros: never read (they may hold stale or unset bits)
  auto load_tile = [&](int pb) {
#pragma unroll
    for (int u = 0; u < NLD; ++u) {
      const int e = tid + u * PF_THREADS;
      const int pp = pb + e / C8, c8 = e % C8;
      kreg[u] = make_uint4(0u, 0u, 0u, 0u);
      vreg[u] = kreg[u];
      if (pp <= pmax) {
        kreg[u] = *reinterpret_cast<const uint4 *>(kb + static_cast<size_t>(pp) * HD + 8 * c8);
        vreg[u] = *reinterpret_cast<const uint4 *>(vb + static_cast<size_t>(pp) * HD + 8 * c8);
      }
    }
  };
  auto store_tile = [&]() {
#pragma unroll
    for (int u = 0; u < NLD; ++u) {
      const int e = tid + u * PF_THREADS;
      const int pl = e / C8, c8 = e % C8;
      const uint4 k = kreg[u], v = vreg[u];
      float *kd = Ks + pl * QS + 8 * c8;
      float *vd = Vs + pl * HD + 8 * c8;
      *reinterpret_cast<float4 *>(kd) = make_float4(__uint_as_float(k.x << 16), __uint_as_float(k.x & 0xffff0000u),
                                                    __uint_as_float(k.y << 16), __uint_as_float(k.y & 0xffff0000u));
      *reinterpret_cast<float4 *>(kd + 4) = make_float4(__uint_as_float(k.z << 16), __uint_as_float(k.z & 0xffff0000u),
                                                        __uint_as_float(k.w << 16), __uint_as_float(k.w & 0xffff0000u));
      *reinterpret_cast<float4 *>(vd) = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u),
                                                    __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xffff0000u));
      *reinterpret_cast<float4 *>(vd + 4) = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xffff0000u),
                                                        __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xffff0000u));
    }
  };

  // score mapping: rows ty, ty + 16; positions tx + 16 j (a row's 16 threads are
  // one half-warp)
  const int ty = tid >> 4, tx = tid & 15;
  int prow[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int tt = (ty + 16 * i) / GRP;
    prow[i] = tt < ntok ? base_pos + tok0 + tt : 0;
  }
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  // output mapping: rows oy + 8 i, columns CPT * ox ..
  const int oy = tid >> 5, ox = tid & 31;
  float o[4][CPT];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int c = 0; c < CPT; ++c) o[i][c] = 0.f;

  const int ntiles = pmax / PF_AP + 1;
  load_tile(0);
  store_tile();
  __syncthreads();
  for (int ti = 0; ti < ntiles; ++ti) {
    const int pb = ti * PF_AP;
    if (ti + 1 < ntiles) load_tile(pb + PF_AP);
    // ---- scores of this tile ----------------------------------------------
    float s[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s[i][j] = 0.f;
#pragma unroll 8
    for (int k = 0; k < HD; k += 4) {
      const float4 q0 = *reinterpret_cast<const float4 *>(Qs + ty * QS + k);
      const float4 q1 = *reinterpret_cast<const float4 *>(Qs + (ty + 16) * QS + k);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 kv = *reinterpret_cast<const float4 *>(Ks + (tx + 16 * j) * QS + k);
        s[0][j] = fmaf(q0.x, kv.x, fmaf(q0.y, kv.y, fmaf(q0.z, kv.z, fmaf(q0.w, kv.w, s[0][j]))));
        s[1][j] = fmaf(q1.x, kv.x, fmaf(q1.y, kv.y, fmaf(q1.z, kv.z, fmaf(q1.w, kv.w, s[1][j]))));
      }
    }
    // ---- online softmax, per row over its half-warp -------------------------
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (pb + tx + 16 * j > prow[i]) s[i][j] = -INFINITY;
        mx = fmaxf(mx, s[i][j]);
      }
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      // slot 0 is in every row's range, so m is finite after the first tile
      const float mn = fmaxf(m[i], mx);
      const float c = expf(m[i] - mn);
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float w = s[i][j] == -INFINITY ? 0.f : expf(s[i][j] - mn);
        Ps[(ty + 16 * i) * PS + tx + 16 * j] = w;
        sum += w;
      }
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      l[i] = l[i] * c + sum;
      m[i] = mn;
      if (tx == 0) Cs[ty + 16 * i] = c;
    }
    __syncthreads();
    // ---- o <- c o + sum_p w_p V[p] ------------------------------------------
    float cr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) cr[i] = Cs[oy + 8 * i];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < CPT; ++c) o[i][c] *= cr[i];
#pragma unroll 2
    for (int p = 0; p < PF_AP; p += 4) {
      float4 w4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) w4[i] = *reinterpret_cast<const float4 *>(Ps + (oy + 8 * i) * PS + p);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        float v[CPT];
        if constexpr (CPT == 4) {
          const float4 t = *reinterpret_cast<const float4 *>(Vs + (p + qq) * HD + 4 * ox);
          v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
        } else {
          const float2 t = *reinterpret_cast<const float2 *>(Vs + (p + qq) * HD + 2 * ox);
          v[0] = t.x; v[1] = t.y;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float w = qq == 0 ? w4[i].x : qq == 1 ? w4[i].y : qq == 2 ? w4[i].z : w4[i].w;
#pragma unroll
          for (int c = 0; c < CPT; ++c) o[i][c] = fmaf(w, v[c], o[i][c]);
        }
      }
    }
    __syncthreads();
    if (ti + 1 < ntiles) {
      store_tile();
      __syncthreads();
    }
  }
  if (tx == 0) {
    Ls[ty] = l[0];
    Ls[ty + 16] = l[1];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = oy + 8 * i, tt = r / GRP, h = r % GRP;
    if (tt >= ntok) continue;
    const float inv = 1.0f / Ls[r];
    float *dst = a.attn + static_cast<size_t>(tok0 + tt) * a.Hq * HD + static_cast<size_t>(g * GRP + h) * HD + CPT * ox;
#pragma unroll
    for (int c = 0; c < CPT; ++c) dst[c] = o[i][c] * inv;
  }
}

// Greedy id of each token, in two stages: block (t, b) reads the logits of
// its slice of the vocabulary (storing them in logits_out when given) and
// keeps its best (largest value, lowest index among equals); then
// one warp per token reduces the blocks' candidates.  A non-finite logit is
// an error.
constexpr int PF_ARGMAX_BLOCKS = 64;

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

__global__ void pf_argmax_part(const float *lg, int V, int t_first, const PfCall *call, float *pv, int *pi,
                               int *err) {
  float *logits_out = call->logits_out;
  __shared__ float sv[PF_THREADS / 32];
  __shared__ int si[PF_THREADS / 32];
  const int t = blockIdx.y, b = blockIdx.x;
  const int per = (V + PF_ARGMAX_BLOCKS - 1) / PF_ARGMAX_BLOCKS;
  const int k0 = b * per, k1 = min(V, k0 + per);
  float v = -INFINITY;
  int i = 0x7fffffff;
  for (int k = k0 + threadIdx.x; k < k1; k += blockDim.x) {
    const float y = lg[static_cast<size_t>(t) * V + k];
    if (logits_out) logits_out[static_cast<size_t>(t_first + t) * V + k] = y;
    if (!isfinite(y)) atomicCAS(err, 0, MK_PF_ERR_NUMERIC);
    if (better(y, k, v, i)) { v = y; i = k; }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { sv[w] = v; si[w] = i; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < PF_THREADS / 32; ++k)
      if (better(sv[k], si[k], v, i)) { v = sv[k]; i = si[k]; }
    pv[t * PF_ARGMAX_BLOCKS + b] = v;
    pi[t * PF_ARGMAX_BLOCKS + b] = i;
  }
}

__global__ void pf_argmax_final(const float *pv, const int *pi, int t_first, const PfCall *call, int t_last) {
  const int t = blockIdx.x, lane = threadIdx.x;
  int32_t *out_ids = call->out_ids;
  int *last_id = call->last_id;
  float v = -INFINITY;
  int i = 0x7fffffff;
  for (int b = lane; b < PF_ARGMAX_BLOCKS; b += 32)
    if (better(pv[t * PF_ARGMAX_BLOCKS + b], pi[t * PF_ARGMAX_BLOCKS + b], v, i)) {
      v = pv[t * PF_ARGMAX_BLOCKS + b];
      i = pi[t * PF_ARGMAX_BLOCKS + b];
    }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (better(ov, oi, v, i)) { v = ov; i = oi; }
  }
  if (lane == 0) {
    if (out_ids) out_ids[t_first + t] = i;
    if (last_id && t_first + t == t_last) *last_id = i;
  }
}

}  // namespace mkp

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace mkp {
namespace {

template <typename T>
int dalloc(T **p, size_t n) {
  if (cudaMalloc(reinterpret_cast<void **>(p), sizeof(T) * (n ? n : 1)) != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return MK_ERR_NO_MEMORY;
  }
  return MK_OK;
}

int blocks_for(size_t n) { return static_cast<int>((n + PF_THREADS - 1) / PF_THREADS > 4096 ? 4096 : (n + PF_THREADS - 1) / PF_THREADS); }

int block_index(int bn) { return bn == 32 ? 0 : bn == 64 ? 1 : 2; }

// one projection: out[s][t][n] (n < N, t < nt) = W[n][:] . (three terms of token t_off + t)
int project(const PfState &st, const mkg::WMaps &w, int kidx, int N, int K, int nt, int t_off, int splits,
            float *out, size_t ldc, size_t part_stride, cudaStream_t s) {
  mkg::GemmCall c;
  c.N = N;
  c.K = K;
  c.nt = nt;
  c.t_off = t_off;
  c.splits = splits;
  c.out = out;
  c.ldc = ldc;
  c.part_stride = part_stride;
  c.err = st.err;
  return mkg::gemm_launch(w, st.xmaps[kidx][block_index(mkg::gemm_block_tokens(nt))], c, s);
}

}  // namespace

// one CTA per (kv head, PF_AR query rows); the dynamic shared memory above
// 48 KB is enabled once per instantiation by pf_attention_enable
template <int HD, int GRP>
void launch_attention(const PfArgs &a, int layer, int t0, int nt, cudaStream_t s) {
  constexpr int TT = PF_AR / GRP;
  pf_attention<HD, GRP><<<dim3((nt + TT - 1) / TT, a.Hkv), PF_THREADS, pf_attention_smem<HD>(), s>>>(a, layer, t0, nt);
}

template <int HD, int GRP>
bool attention_attr() {
  return cudaFuncSetAttribute(pf_attention<HD, GRP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(pf_attention_smem<HD>())) == cudaSuccess;
}

bool pf_attention_enable() {
  return attention_attr<64, 1>() && attention_attr<64, 2>() && attention_attr<64, 4>() && attention_attr<128, 1>() &&
         attention_attr<128, 2>();
}

int pf_init(PfState &st, int tc, int H, int Hq, int Hkv, int d, int I) {
  if (st.tc >= tc) return MK_OK;
  pf_free(st);
  if (H % 64 || (Hq * d) % 64 || I % 64) return MK_ERR_UNSUPPORTED;   // GEMM K blocks of 64
  const size_t rows = static_cast<size_t>(Hq + 2 * Hkv) * d;
  size_t kmax = H;
  if (static_cast<size_t>(Hq) * d > kmax) kmax = static_cast<size_t>(Hq) * d;
  if (static_cast<size_t>(I) > kmax) kmax = I;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  const size_t T = tc;
  int rc;
  if ((rc = dalloc(&st.x, T * H)) || (rc = dalloc(&st.qkv, T * rows)) || (rc = dalloc(&st.attn, T * Hq * d)) ||
      (rc = dalloc(&st.attn_part, static_cast<size_t>(PF_ATTN_SPLITS) * T * Hq * (d + 2))) ||
      (rc = dalloc(&st.qkv_p, PF_SPLITS_WIDE * T * rows)) || (rc = dalloc(&st.y_p, PF_SPLITS_NARROW * T * H)) ||
      (rc = dalloc(&st.gu_p, PF_SPLITS_WIDE * T * 2 * I)) ||
      (rc = dalloc(&st.hs, 3 * T * kmax)) || (rc = dalloc(&st.pv, T * PF_ARGMAX_BLOCKS)) ||
      (rc = dalloc(&st.pi, T * PF_ARGMAX_BLOCKS)) || (rc = dalloc(&st.err, 1)) || (rc = dalloc(&st.call, 1))) {
    pf_free(st);
    return rc;
  }
  st.tc = tc;
  st.kmax = kmax;
  // the input terms of tokens past a chunk's end are read (never stored): keep them finite
  if (cudaMemset(st.hs, 0, sizeof(uint16_t) * 3 * T * kmax) != cudaSuccess ||
      cudaStreamCreateWithFlags(&st.cap, cudaStreamNonBlocking) != cudaSuccess || !pf_attention_enable()) {
    cudaGetLastError();
    pf_free(st);
    return MK_ERR_CUDA;
  }
  // activation tensor maps: the three term matrices [tc][K] (rows K apart, as
  // the split kernels write them for a GEMM of input width K), T * kmax apart
  const int Ks[3] = {H, Hq * d, I};
  const int bns[3] = {32, 64, 128};
  for (int i = 0; i < 3; ++i)
    for (int b = 0; b < 3; ++b) {
      std::memset(&st.xmaps[i][b], 0, sizeof(CUtensorMap));
      if (!mkg::make_tmap(&st.xmaps[i][b], st.hs, Ks[i], T, static_cast<uint64_t>(Ks[i]) * 2, bns[b], 3,
                          T * kmax * 2)) {
        pf_free(st);
        return MK_ERR_CUDA;
      }
    }
  return MK_OK;
}

void pf_free(PfState &st) {
  for (PfState::Graph &g : st.graphs) {
    cudaGraphExecDestroy(g.exec);
    cudaGraphDestroy(g.graph);
  }
  if (st.cap) cudaStreamDestroy(st.cap);
  void *ps[] = {st.x, st.qkv, st.attn, st.attn_part, st.qkv_p, st.y_p, st.gu_p, st.logits, st.pv, st.pi, st.hs, st.err, st.call};
  for (void *p : ps)
    if (p) cudaFree(p);
  st = PfState();
}

// every launch of an n-token prefill, in order, on stream s
int pf_enqueue(PfState &st, const PfArgs &a, const PfLayer *layers, const uint16_t *final_norm,
               const uint16_t *lm_head, int n, bool all_logits, cudaStream_t s) {
  (void)lm_head;
  const int rows = (a.Hq + 2 * a.Hkv) * a.d;
  const int grp = a.Hq / a.Hkv;
  const int qd = a.Hq * a.d;
  const size_t T = st.tc;
  const size_t gu_stride = T * 2 * a.I;
  int rc = MK_OK;
  for (int t0 = 0; t0 < n && rc == MK_OK; t0 += st.tc) {
    const int nt = n - t0 < st.tc ? n - t0 : st.tc;
    // split-K counts of this chunk's projections (the readers sum that many partials)
    const int s_qkv = mkg::gemm_splits(rows, a.H, nt, st.sms, PF_SPLITS_WIDE);
    const int s_o = mkg::gemm_splits(a.H, qd, nt, st.sms, PF_SPLITS_NARROW);
    const int s_gu = mkg::gemm_splits(2 * a.I, a.H, nt, st.sms, PF_SPLITS_WIDE);
    const int s_dn = mkg::gemm_splits(a.H, a.I, nt, st.sms, PF_SPLITS_NARROW);
    PfArgs ac = a;
    ac.qkv_n = s_qkv;
    pf_embed<<<nt, PF_THREADS, 0, s>>>(ac, t0, nt);
    pf_add_norm_split<<<nt, PF_THREADS, 0, s>>>(ac, nullptr, 0, layers[0].attn_norm, t0, nt, -1);
    for (int l = 0; l < a.L && rc == MK_OK; ++l) {
      const PfLayer &w = layers[l];
      const mkg::WMaps *wm = &st.wmaps[static_cast<size_t>(l) * 4];
      // attention block: q, k and v columns of one [nt][rows] output, s_qkv partials
      if ((rc = project(st, wm[0], 0, rows, a.H, nt, 0, s_qkv, st.qkv_p, rows, a.qkv_stride, s))) break;
      const int jobs_warps = nt * (a.Hq + 2 * a.Hkv);
      const int wpb = PF_THREADS / 32;
      if (a.d == 64)
        pf_qk_rope_append<64><<<(jobs_warps + wpb - 1) / wpb, PF_THREADS, 0, s>>>(ac, l, w.q_norm, w.k_norm, t0, nt);
      else
        pf_qk_rope_append<128><<<(jobs_warps + wpb - 1) / wpb, PF_THREADS, 0, s>>>(ac, l, w.q_norm, w.k_norm, t0, nt);
      if (st.kv_maps) {
        // causal attention on the tensor cores
        if ((rc = attn_tc_launch(st.kmap, st.vmap, ac, l, t0, nt, s))) break;
      } else if (a.d == 64) {
        // groups mk_create accepts: group * head_dim <= 256
        switch (grp) {
          case 1: launch_attention<64, 1>(ac, l, t0, nt, s); break;
          case 2: launch_attention<64, 2>(ac, l, t0, nt, s); break;
          default: launch_attention<64, 4>(ac, l, t0, nt, s); break;
        }
      } else {
        switch (grp) {
          case 1: launch_attention<128, 1>(ac, l, t0, nt, s); break;
          default: launch_attention<128, 2>(ac, l, t0, nt, s); break;
        }
      }
      pf_split<<<blocks_for(static_cast<size_t>(nt) * qd), PF_THREADS, 0, s>>>(st.attn, qd, nt, st.hs, a.hs_stride);
      if ((rc = project(st, wm[1], 1, a.H, qd, nt, 0, s_o, st.y_p, a.H, a.y_stride, s))) break;
      pf_add_norm_split<<<nt, PF_THREADS, 0, s>>>(ac, st.y_p, s_o, w.mlp_norm, t0, nt, -1);
      // MLP block
      if ((rc = project(st, wm[2], 0, 2 * a.I, a.H, nt, 0, s_gu, st.gu_p, 2 * a.I, gu_stride, s))) break;
      pf_silu_mul_split<<<blocks_for(static_cast<size_t>(nt) * a.I), PF_THREADS, 0, s>>>(
          st.gu_p, gu_stride, s_gu, a.I, nt, st.hs, a.hs_stride);
      if ((rc = project(st, wm[3], 2, a.H, a.I, nt, 0, s_dn, st.y_p, a.H, a.y_stride, s))) break;
      pf_add_norm_split<<<nt, PF_THREADS, 0, s>>>(ac, st.y_p, s_dn, l + 1 < a.L ? layers[l + 1].attn_norm : final_norm,
                                                  t0, nt, l + 1);
    }
    if (rc != MK_OK) break;
    // LM head: every token of the chunk when ids or logits are wanted, else
    // only the prompt's last token (the first generated id)
    const bool has_last = (t0 + nt == n);
    if (all_logits || has_last) {
      const int first = all_logits ? 0 : nt - 1, m = all_logits ? nt : 1;
      if ((rc = project(st, st.wmaps[static_cast<size_t>(a.L) * 4], 0, a.V, a.H, m, first, 1, st.logits, a.V,
                        0, s)))
        break;
      pf_argmax_part<<<dim3(PF_ARGMAX_BLOCKS, m), PF_THREADS, 0, s>>>(st.logits, a.V, t0 + first, st.call, st.pv,
                                                                     st.pi, st.err);
      pf_argmax_final<<<m, 32, 0, s>>>(st.pv, st.pi, t0 + first, st.call, n - 1);
    }
  }
  if (cudaGetLastError() != cudaSuccess && rc == MK_OK) rc = MK_ERR_CUDA;
  return rc;
}

int pf_run(PfState &st, PfArgs a, const PfLayer *layers, const uint16_t *final_norm, const uint16_t *lm_head,
           int n, const PfCall &call, cudaStream_t s) {
  const int grp = a.Hq / a.Hkv;
  if ((a.d != 64 && a.d != 128) || a.Hq % a.Hkv || (grp != 1 && grp != 2 && grp != 4 && !(grp == 8 && a.d == 64)))
    return MK_ERR_UNSUPPORTED;
  const size_t T = st.tc;
  const bool all_logits = call.out_ids || call.logits_out;
  const int need_rows = all_logits ? st.tc : 1;
  if (st.logit_rows < need_rows) {
    if (st.logits) cudaFree(st.logits);
    st.logits = nullptr;
    st.logit_rows = 0;
    int rc = dalloc(&st.logits, static_cast<size_t>(need_rows) * a.V);
    if (rc) return rc;
    st.logit_rows = need_rows;
  }
  if (st.wmaps.empty()) {
    // weight tensor maps, made once per handle (the weights are borrowed for its lifetime)
    std::vector<mkg::WMaps> m(static_cast<size_t>(a.L) * 4 + 1);
    std::memset(m.data(), 0, sizeof(mkg::WMaps) * m.size());
    const int qd = a.Hq * a.d, kd = a.Hkv * a.d;
    // one stacked set of weight matrices per projection
    auto set = [](mkg::WMaps &w, int i, const void *base, int K, int rows) {
      w.rows[i] = rows;
      w.n = i + 1;
      return mkg::make_tmap(&w.map[i], base, K, rows, K * 2ull, 128);
    };
    bool ok = true;
    for (int l = 0; l < a.L && ok; ++l) {
      const PfLayer &w = layers[l];
      mkg::WMaps *q = &m[static_cast<size_t>(l) * 4];
      ok = set(q[0], 0, w.wq, a.H, qd) && set(q[0], 1, w.wk, a.H, kd) && set(q[0], 2, w.wv, a.H, kd) &&
           set(q[1], 0, w.wo, qd, a.H) && set(q[2], 0, w.w_gate, a.H, a.I) && set(q[2], 1, w.w_up, a.H, a.I) &&
           set(q[3], 0, w.w_down, a.I, a.H);
    }
    ok = ok && set(m[static_cast<size_t>(a.L) * 4], 0, lm_head, a.H, a.V);
    if (!ok) return MK_ERR_CUDA;
    st.wmaps.swap(m);
  }
  if (!st.kv_maps) st.kv_maps = attn_tc_maps(a, &st.kmap, &st.vmap);
  const int rows = (a.Hq + 2 * a.Hkv) * a.d;
  a.x = st.x; a.qkv = st.qkv; a.attn = st.attn; a.attn_part = st.attn_part;
  a.qkv_p = st.qkv_p; a.qkv_stride = T * rows;
  a.y_p = st.y_p; a.y_stride = T * a.H;
  a.hs = st.hs; a.hs_stride = T * st.kmax;
  a.call = st.call;
  a.err = st.err;
  // the call's fields, then the (captured once, replayed) launch sequence
  if (cudaMemcpyAsync(st.call, &call, sizeof(PfCall), cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemsetAsync(st.err, 0, sizeof(int), s) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  cudaGraphExec_t exec = nullptr;
  for (PfState::Graph &g : st.graphs)
    if (g.n == n && g.all_logits == all_logits) {
      exec = g.exec;
      g.used = ++st.clock;
    }
  int rc = MK_OK;
  if (!exec) {
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamBeginCapture(st.cap, cudaStreamCaptureModeThreadLocal);
    if (e == cudaSuccess) {
      rc = pf_enqueue(st, a, layers, final_norm, lm_head, n, all_logits, st.cap);
      const cudaError_t e2 = cudaStreamEndCapture(st.cap, &graph);
      if (rc == MK_OK && e2 == cudaSuccess) e = cudaGraphInstantiate(&exec, graph, 0);
      else e = e2 != cudaSuccess ? e2 : cudaErrorUnknown;
    }
    if (e == cudaSuccess && rc == MK_OK && exec) {
      if (static_cast<int>(st.graphs.size()) >= PF_MAX_GRAPHS) {
        // keep the cache bounded: replace the least recently used prompt length
        size_t lru = 0;
        for (size_t i = 1; i < st.graphs.size(); ++i)
          if (st.graphs[i].used < st.graphs[lru].used) lru = i;
        cudaGraphExecDestroy(st.graphs[lru].exec);
        cudaGraphDestroy(st.graphs[lru].graph);
        st.graphs.erase(st.graphs.begin() + static_cast<long>(lru));
      }
      st.graphs.push_back(PfState::Graph{n, all_logits, ++st.clock, graph, exec});
    } else {
      // not capturable here: run the same sequence directly
      if (graph) cudaGraphDestroy(graph);
      exec = nullptr;
      cudaGetLastError();
      rc = pf_enqueue(st, a, layers, final_norm, lm_head, n, all_logits, s);
    }
  }
  if (exec && cudaGraphLaunch(exec, s) != cudaSuccess) {
    cudaGetLastError();
    rc = MK_ERR_CUDA;
  }
  int herr = 0;
  if (cudaMemcpyAsync(&herr, st.err, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  if (rc != MK_OK) return rc;
  return herr;
}

}  // namespace mkp
