// Batched prompt prefill: the n prompt forwards of a decode call computed all
// at once per layer.  The projections are dense contractions with M = prompt
// tokens and run as bf16 tensor-core GEMMs with fp32 accumulation (cuBLAS);
// every fp32 activation enters them as three bf16 terms (hi + mid + lo, 24
// significant bits, as many as fp32 holds), so the products lose nothing to
// the bf16 operand format.  The
// rest -- RMSNorm, QK-norm, RoPE / MRoPE, the bf16 KV append, causal GQA
// attention over the cache, residual adds, SiLU * up, greedy argmax -- are the
// kernels below.  The KV cache it fills is the decode kernel's, so decoding
// continues from the prompt's last position (page A, "Porting a 1,200-line
// persistent CUDA megakernel to Qwen3-TTS": time to first chunk is what the
// listener waits for).
#include <cuda_runtime.h>
#include <cublas_v2.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>
#include <cstring>

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
  const int id = a.ids[t0 + t];
  const bool bad = id >= 0 ? id >= a.vocab_in : (!a.embeds || -(id + 1) >= a.n_embed_rows);
  if (bad) {
    if (threadIdx.x == 0) atomicCAS(a.err, 0, MK_PF_ERR_BAD_TOKEN);
    return;
  }
  float *x = a.x + static_cast<size_t>(t) * a.H;
  for (int k = threadIdx.x; k < a.H; k += blockDim.x) {
    const float v = id >= 0 ? bf2f(a.embed[static_cast<size_t>(id) * a.H + k])
                            : a.embeds[static_cast<size_t>(-(id + 1)) * a.H + k];
    x[k] = v;
    if (a.hidden) a.hidden[(static_cast<size_t>(t0 + t) * (a.L + 1)) * a.H + k] = v;
  }
}

// Optionally x[t] += y[t] (a residual add) and record hidden[t][layer]; then
// h = x / sqrt(mean(x^2) + eps) * gain as three bf16 terms
__global__ void pf_add_norm_split(const PfArgs a, const float *y, const uint16_t *gain, int t0, int nt,
                                  int hidden_layer) {
  __shared__ float red[PF_THREADS / 32];
  const int t = blockIdx.x;
  if (t >= nt) return;
  float *x = a.x + static_cast<size_t>(t) * a.H;
  float ss = 0.f;
  for (int k = threadIdx.x; k < a.H; k += blockDim.x) {
    float v = x[k];
    if (y) {
      v = v + y[static_cast<size_t>(t) * a.H + k];
      x[k] = v;
      if (a.hidden && hidden_layer >= 0)
        a.hidden[(static_cast<size_t>(t0 + t) * (a.L + 1) + hidden_layer) * a.H + k] = v;
    }
    ss = fmaf(v, v, ss);
  }
  const float tot = block_sum(ss, red);
  const float rs = 1.0f / sqrtf(tot / static_cast<float>(a.H) + a.eps);
  const size_t o = static_cast<size_t>(t) * a.H;
  for (int k = threadIdx.x; k < a.H; k += blockDim.x) {
    const float h = x[k] * rs * bf2f(gain[k]);
    split3(h, a.hh[o + k], a.hm[o + k], a.hl[o + k]);
  }
}

// v (fp32, n per token) as three bf16 terms (the attention output before O)
__global__ void pf_split(const float *v, int n, int nt, uint16_t *hi, uint16_t *mid, uint16_t *lo) {
  const size_t total = static_cast<size_t>(n) * nt;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    split3(v[i], hi[i], mid[i], lo[i]);
}

// u = silu(gate) * up, as three bf16 terms
__global__ void pf_silu_mul_split(const float *g, const float *u, int n, int nt, uint16_t *hi, uint16_t *mid,
                                  uint16_t *lo) {
  const size_t total = static_cast<size_t>(n) * nt;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float z = g[i];
    split3(z / (1.0f + expf(-z)) * u[i], hi[i], mid[i], lo[i]);
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
  const int P = a.pos0 + t0 + t;
  const int rows = (a.Hq + 2 * a.Hkv) * HD;
  float *src = a.qkv + static_cast<size_t>(t) * rows + static_cast<size_t>(job) * HD;
  float v[EPL];
#pragma unroll
  for (int k = 0; k < EPL; ++k) v[k] = src[lane + 32 * k];
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
      int pos = a.pos3 ? a.pos3[static_cast<size_t>(s) * a.n_pos + t0 + t] : P;
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
    for (int k = 0; k < EPL; ++k) src[lane + 32 * k] = v[k] * a.inv_sqrt_d;
  } else {
    const bool key = job < a.Hq + a.Hkv;
    const int g = key ? job - a.Hq : job - a.Hq - a.Hkv;
    uint16_t *dst = (key ? a.kcache : a.vcache) +
                    ((static_cast<size_t>(layer) * a.Hkv + g) * a.max_seq + P) * HD;
#pragma unroll
    for (int k = 0; k < EPL; ++k) dst[lane + 32 * k] = f2bf(v[k]);
  }
}

// Causal GQA attention of the chunk's tokens over the cache: one warp per
// (token, kv head) handles the GRP query heads that read that kv head, with
// an online softmax over slots 0..P (running max m, sum l, output o).
template <int HD, int GRP>
__global__ void pf_attention(const PfArgs a, int layer, int t0, int nt) {
  constexpr int EPL = HD / 32;
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= nt * a.Hkv) return;
  const int t = warp / a.Hkv, g = warp % a.Hkv;
  const int P = a.pos0 + t0 + t;
  const int rows = (a.Hq + 2 * a.Hkv) * HD;
  float q[GRP][EPL], o[GRP][EPL], m[GRP], l[GRP];
#pragma unroll
  for (int h = 0; h < GRP; ++h) {
    const float *qs = a.qkv + static_cast<size_t>(t) * rows + static_cast<size_t>(g * GRP + h) * HD;
#pragma unroll
    for (int e = 0; e < EPL; ++e) { q[h][e] = qs[lane + 32 * e]; o[h][e] = 0.f; }
    m[h] = -INFINITY;
    l[h] = 0.f;
  }
  const uint16_t *kb = a.kcache + (static_cast<size_t>(layer) * a.Hkv + g) * a.max_seq * HD;
  const uint16_t *vb = a.vcache + (static_cast<size_t>(layer) * a.Hkv + g) * a.max_seq * HD;
  for (int pos = 0; pos <= P; ++pos) {
    float kk[EPL], vv[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      kk[e] = bf2f(kb[static_cast<size_t>(pos) * HD + lane + 32 * e]);
      vv[e] = bf2f(vb[static_cast<size_t>(pos) * HD + lane + 32 * e]);
    }
#pragma unroll
    for (int h = 0; h < GRP; ++h) {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) s = fmaf(q[h][e], kk[e], s);
      s = warp_sum(s);
      const float mn = fmaxf(m[h], s);
      const float c = expf(m[h] - mn), w = expf(s - mn);
      l[h] = l[h] * c + w;
#pragma unroll
      for (int e = 0; e < EPL; ++e) o[h][e] = fmaf(w, vv[e], o[h][e] * c);
      m[h] = mn;
    }
  }
#pragma unroll
  for (int h = 0; h < GRP; ++h) {
    float *dst = a.attn + static_cast<size_t>(t) * a.Hq * HD + static_cast<size_t>(g * GRP + h) * HD;
#pragma unroll
    for (int e = 0; e < EPL; ++e) dst[lane + 32 * e] = o[h][e] / l[h];
  }
}

// greedy id of each token: the largest logit, the lowest index among equals;
// a non-finite logit is an error
__global__ void pf_argmax(const float *logits, int V, int nt, int t_first, int32_t *out_ids, int *last_id,
                          int t_last, int *err) {
  __shared__ float bv[PF_THREADS / 32];
  __shared__ int bi[PF_THREADS / 32];
  const int t = blockIdx.x;
  if (t >= nt) return;
  const float *row = logits + static_cast<size_t>(t) * V;
  float v = -INFINITY;
  int i = 0x7fffffff;
  for (int k = threadIdx.x; k < V; k += blockDim.x) {
    const float y = row[k];
    if (!isfinite(y)) atomicCAS(err, 0, MK_PF_ERR_NUMERIC);
    if (y > v || (y == v && k < i)) { v = y; i = k; }
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, i, o);
    if (ov > v || (ov == v && oi < i)) { v = ov; i = oi; }
  }
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) { bv[w] = v; bi[w] = i; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < PF_THREADS / 32; ++k)
      if (bv[k] > v || (bv[k] == v && bi[k] < i)) { v = bv[k]; i = bi[k]; }
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

// C[nt][N] (ldc) = (hi + mid + lo)[nt][K] . W[N][K]^T, fp32 accumulate on tensor
// cores: in column-major terms C^T (N x nt) = W (N x K, stored as K x N) . in^T
int gemm3(cublasHandle_t b, const uint16_t *hi, const uint16_t *mid, const uint16_t *lo, const uint16_t *W, int nt,
          int N, int K, float *C, int ldc) {
  const float one = 1.0f, zero = 0.0f;
  const uint16_t *terms[3] = {hi, mid, lo};
  cublasStatus_t st = CUBLAS_STATUS_SUCCESS;
  for (int i = 0; i < 3 && st == CUBLAS_STATUS_SUCCESS; ++i)
    st = cublasGemmEx(b, CUBLAS_OP_T, CUBLAS_OP_N, N, nt, K, &one, W, CUDA_R_16BF, K, terms[i], CUDA_R_16BF, K,
                      i == 0 ? &zero : &one, C, CUDA_R_32F, ldc, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
  return st == CUBLAS_STATUS_SUCCESS ? MK_OK : MK_ERR_CUDA;
}

int blocks_for(size_t n) { return static_cast<int>((n + PF_THREADS - 1) / PF_THREADS > 4096 ? 4096 : (n + PF_THREADS - 1) / PF_THREADS); }

}  // namespace

int pf_init(PfState &st, int tc, int H, int Hq, int Hkv, int d, int I) {
  if (st.tc >= tc) return MK_OK;
  pf_free(st);
  const size_t rows = static_cast<size_t>(Hq + 2 * Hkv) * d;
  size_t kmax = H;
  if (static_cast<size_t>(Hq) * d > kmax) kmax = static_cast<size_t>(Hq) * d;
  if (static_cast<size_t>(I) > kmax) kmax = I;
  cublasHandle_t b = nullptr;
  if (cublasCreate(&b) != CUBLAS_STATUS_SUCCESS) return MK_ERR_CUDA;
  st.blas = b;
  int rc;
  if ((rc = dalloc(&st.x, static_cast<size_t>(tc) * H)) || (rc = dalloc(&st.qkv, static_cast<size_t>(tc) * rows)) ||
      (rc = dalloc(&st.attn, static_cast<size_t>(tc) * Hq * d)) || (rc = dalloc(&st.y, static_cast<size_t>(tc) * H)) ||
      (rc = dalloc(&st.gate, static_cast<size_t>(tc) * I)) || (rc = dalloc(&st.up, static_cast<size_t>(tc) * I)) ||
      (rc = dalloc(&st.hh, static_cast<size_t>(tc) * kmax)) || (rc = dalloc(&st.hm, static_cast<size_t>(tc) * kmax)) ||
      (rc = dalloc(&st.hl, static_cast<size_t>(tc) * kmax)) ||
      (rc = dalloc(&st.err, 1))) {
    pf_free(st);
    return rc;
  }
  st.tc = tc;
  return MK_OK;
}

void pf_free(PfState &st) {
  void *ps[] = {st.x, st.qkv, st.attn, st.y, st.gate, st.up, st.logits, st.hh, st.hm, st.hl, st.err};
  for (void *p : ps)
    if (p) cudaFree(p);
  if (st.blas) cublasDestroy(static_cast<cublasHandle_t>(st.blas));
  st = PfState();
}

int pf_run(PfState &st, PfArgs a, const PfLayer *layers, const uint16_t *final_norm, const uint16_t *lm_head,
           int n, int32_t *out_ids, float *logits_out, int *last_id, cudaStream_t s) {
  cublasHandle_t b = static_cast<cublasHandle_t>(st.blas);
  if (cublasSetStream(b, s) != CUBLAS_STATUS_SUCCESS) return MK_ERR_CUDA;
  const bool all_logits = out_ids || logits_out;
  if (all_logits && !logits_out && !st.logits) {
    int rc = dalloc(&st.logits, static_cast<size_t>(st.tc) * a.V);
    if (rc) return rc;
  }
  a.x = st.x; a.qkv = st.qkv; a.attn = st.attn; a.y = st.y; a.gate = st.gate; a.up = st.up;
  a.hh = st.hh; a.hm = st.hm; a.hl = st.hl; a.err = st.err;
  if (cudaMemsetAsync(st.err, 0, sizeof(int), s) != cudaSuccess) return MK_ERR_CUDA;
  const int rows = (a.Hq + 2 * a.Hkv) * a.d;
  const int grp = a.Hq / a.Hkv;
  if ((a.d != 64 && a.d != 128) || a.Hq % a.Hkv || (grp != 1 && grp != 2 && grp != 4 && !(grp == 8 && a.d == 64)))
    return MK_ERR_UNSUPPORTED;
  int rc = MK_OK;
  for (int t0 = 0; t0 < n && rc == MK_OK; t0 += st.tc) {
    const int nt = n - t0 < st.tc ? n - t0 : st.tc;
    pf_embed<<<nt, PF_THREADS, 0, s>>>(a, t0, nt);
    pf_add_norm_split<<<nt, PF_THREADS, 0, s>>>(a, nullptr, layers[0].attn_norm, t0, nt, -1);
    for (int l = 0; l < a.L && rc == MK_OK; ++l) {
      const PfLayer &w = layers[l];
      // attention block
      if ((rc = gemm3(b, st.hh, st.hm, st.hl, w.wq, nt, a.Hq * a.d, a.H, st.qkv, rows)) ||
          (rc = gemm3(b, st.hh, st.hm, st.hl, w.wk, nt, a.Hkv * a.d, a.H, st.qkv + a.Hq * a.d, rows)) ||
          (rc = gemm3(b, st.hh, st.hm, st.hl, w.wv, nt, a.Hkv * a.d, a.H, st.qkv + (a.Hq + a.Hkv) * a.d, rows)))
        break;
      const int jobs_warps = nt * (a.Hq + 2 * a.Hkv), attn_warps = nt * a.Hkv;
      const int wpb = PF_THREADS / 32;
      if (a.d == 64) {
        pf_qk_rope_append<64><<<(jobs_warps + wpb - 1) / wpb, PF_THREADS, 0, s>>>(a, l, w.q_norm, w.k_norm, t0, nt);
        switch (grp) {
          case 1: pf_attention<64, 1><<<(attn_warps + wpb - 1) / wpb, PF_THREADS, 0, s>>>(a, l, t0, nt); break;
          case 2: pf_attention<64, 2><<<(attn_warps + wpb - 1) / wpb, PF_THREADS, 0, s>>>(a, l, t0, nt); break;
          case 4: pf_attention<64, 4><<<(attn_warps + wpb - 1) / wpb, PF_THREADS, 0, s>>>(a, l, t0, nt); break;
          default: pf_attention<64, 8><<<(attn_warps + wpb - 1) / wpb, PF_THREADS, 0, s>>>(a, l, t0, nt); break;
        }
      } else {
        pf_qk_rope_append<128><<<(jobs_warps + wpb - 1) / wpb, PF_THREADS, 0, s>>>(a, l, w.q_norm, w.k_norm, t0, nt);
        switch (grp) {
          case 1: pf_attention<128, 1><<<(attn_warps + wpb - 1) / wpb, PF_THREADS, 0, s>>>(a, l, t0, nt); break;
          case 2: pf_attention<128, 2><<<(attn_warps + wpb - 1) / wpb, PF_THREADS, 0, s>>>(a, l, t0, nt); break;
          default: pf_attention<128, 4><<<(attn_warps + wpb - 1) / wpb, PF_THREADS, 0, s>>>(a, l, t0, nt); break;
        }
      }
      pf_split<<<blocks_for(static_cast<size_t>(nt) * a.Hq * a.d), PF_THREADS, 0, s>>>(st.attn, a.Hq * a.d, nt,
                                                                                         st.hh, st.hm, st.hl);
      if ((rc = gemm3(b, st.hh, st.hm, st.hl, w.wo, nt, a.H, a.Hq * a.d, st.y, a.H))) break;
      pf_add_norm_split<<<nt, PF_THREADS, 0, s>>>(a, st.y, w.mlp_norm, t0, nt, -1);
      // MLP block
      if ((rc = gemm3(b, st.hh, st.hm, st.hl, w.w_gate, nt, a.I, a.H, st.gate, a.I)) ||
          (rc = gemm3(b, st.hh, st.hm, st.hl, w.w_up, nt, a.I, a.H, st.up, a.I)))
        break;
      pf_silu_mul_split<<<blocks_for(static_cast<size_t>(nt) * a.I), PF_THREADS, 0, s>>>(st.gate, st.up, a.I, nt,
                                                                                         st.hh, st.hm, st.hl);
      if ((rc = gemm3(b, st.hh, st.hm, st.hl, w.w_down, nt, a.H, a.I, st.y, a.H))) break;
      pf_add_norm_split<<<nt, PF_THREADS, 0, s>>>(a, st.y, l + 1 < a.L ? layers[l + 1].attn_norm : final_norm, t0,
                                                   nt, l + 1);
    }
    if (rc != MK_OK) break;
    // LM head: every token of the chunk when ids or logits are wanted, else
    // only the prompt's last token (the first generated id)
    const bool has_last = (t0 + nt == n);
    if (all_logits) {
      float *lg = logits_out ? logits_out + static_cast<size_t>(t0) * a.V : st.logits;
      if ((rc = gemm3(b, st.hh, st.hm, st.hl, lm_head, nt, a.V, a.H, lg, a.V))) break;
      pf_argmax<<<nt, PF_THREADS, 0, s>>>(lg, a.V, nt, t0, out_ids, last_id, n - 1, st.err);
    } else if (has_last) {
      if (!st.logits) {
        // one row suffices here
        if ((rc = dalloc(&st.logits, static_cast<size_t>(st.tc) * a.V))) break;
      }
      const size_t off = static_cast<size_t>(nt - 1) * a.H;
      if ((rc = gemm3(b, st.hh + off, st.hm + off, st.hl + off, lm_head, 1, a.V, a.H, st.logits, a.V))) break;
      pf_argmax<<<1, PF_THREADS, 0, s>>>(st.logits, a.V, 1, n - 1, nullptr, last_id, n - 1, st.err);
    }
  }
  if (cudaGetLastError() != cudaSuccess && rc == MK_OK) rc = MK_ERR_CUDA;
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
