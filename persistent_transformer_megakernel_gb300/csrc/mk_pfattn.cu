// Causal GQA attention of the batched prefill on the tensor cores (tcgen05).
//
// One CTA owns one kv head g and 128 query rows (row r = token tok0 + r / GRP,
// q head g * GRP + r % GRP) and walks the KV cache in tiles of 64 positions,
// slots 0 .. the last row's position.  Exact softmax in two passes over the
// tiles, so that the output accumulator never needs rescaling:
//   pass 1  S = Q K^T per tile (tensor cores, fp32 in tensor memory); each row
//           keeps its running maximum m over the unmasked positions;
//   pass 2  S again; p = exp(s - m) (0 where the position is past the row's
//           own), split into three bf16 terms (24 significant bits, what
//           fp32 holds) and written to shared memory; O += P V on the tensor
//           cores; l = sum of the p actually multiplied.  At the end o = O / l.
// Q (fp32, normed, rotated and scaled by 1/sqrt(d)) enters as three bf16
// terms as well; K and V are the bf16 cache as stored (exact).  With fewer
// terms the 0.6B prompt's last hidden state missed the parity bound (the
// score error, ~2^-17 of |q||k|, flips bf16 roundings of later keys).
// Operands follow the 128-byte swizzled layouts of csrc/mk_tc.cuh: Q, K and P
// K-major, V MN-major (positions x head_dim, as the cache holds it).
//
// Long prompts split the cached positions of a query tile over gridDim.z
// CTAs (blockIdx.z takes tiles [z * tps, (z + 1) * tps)); each writes its
// unnormalised output with its rows' maximum and sum, and pf_attn_merge
// combines the splits.
//
// Warp roles (352 threads): softmax warps 0-7, warp w owning TMEM lanes
// 32 (w % 4) .. + 31 (one query row per thread) and columns 32 (w / 4) .. + 31
// of every 64-position tile; warp 8 lane 0 issues the TMA loads of K and V
// tiles (two buffers each); warp 9 allocates tensor memory and its lane 0
// issues the S MMAs (two S buffers); warp 10 lane 0 issues the P V MMAs.
// Every wait is bounded; on expiry the CTA records MK_ERR_TIMEOUT, the MMA
// issuers still wait for what they issued, and tensor memory is freed.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/mk.h"
#include "mk_prefill.h"
#include "mk_tc.cuh"

namespace mkp {

using namespace mktc;

constexpr int AT_THREADS = 352;
constexpr int AT_SOFT_WARPS = 8;
constexpr int AT_TERMS = 3;         // bf16 terms of the fp32 Q and P
constexpr int AT_ROWS = 128;        // query rows per CTA (MMA M)
constexpr int AT_POS = 64;          // cached positions per tile
constexpr long long AT_WAIT_NS = 2000000000LL;

template <int HD>
struct AttnLayout {
  static constexpr int ATOMS = HD / 64;                       // 64-wide swizzle atoms along head_dim
  static constexpr uint32_t Q_TERM = ATOMS * AT_ROWS * 128;   // one bf16 term of Q
  static constexpr uint32_t KV_TILE = ATOMS * AT_POS * 128;   // one K or V tile
  static constexpr uint32_t P_TERM = AT_ROWS * 128;           // one bf16 term of P (64 positions)
  static constexpr uint32_t Q_OFF = 0;
  static constexpr uint32_t K_OFF = Q_OFF + AT_TERMS * Q_TERM;
  static constexpr uint32_t V_OFF = K_OFF + 2 * KV_TILE;
  static constexpr uint32_t P_OFF = V_OFF + 2 * KV_TILE;
  static constexpr uint32_t X_OFF = P_OFF + AT_TERMS * P_TERM;  // row max / sum exchange [2][2][128] fp32
  static constexpr uint32_t BYTES = X_OFF + 4 * AT_ROWS * 4;
  static constexpr size_t SMEM = 2048 + BYTES;                 // + control block and alignment slack
  static constexpr uint32_t TMEM_COLS = 256;                   // S0 [0, 64), S1 [64, 128), O [128, 128 + HD)
};

// byte offset of element (row, col) in a [rows x 64] bf16 tile, 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int row, int col) {
  return static_cast<uint32_t>(row) * 128u + ((static_cast<uint32_t>(col >> 3) ^ (row & 7)) << 4) +
         (static_cast<uint32_t>(col & 7) << 1);
}


// MN-major operand descriptor (128-byte swizzle): lbo = bytes between 64-wide
// atoms along N, sbo = bytes between 8-row groups along K
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>(lbo >> 4) << 16) |
         (static_cast<uint64_t>(sbo >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// two fp32 -> two bf16 (round to nearest even) packed: e0 in the low half
__device__ __forceinline__ uint32_t bf16x2_rn(float e0, float e1) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(e1), "f"(e0));
  return d;
}
__device__ __forceinline__ float bf16_lo_val(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_val(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 8 fp32 values -> three packed bf16 terms (each the rounding of what the
// terms before it left) as three 16-byte words
__device__ __forceinline__ void split3x8(const float (&v)[8], uint4 &t0, uint4 &t1, uint4 &t2) {
  uint32_t a[4], b[4], c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float x0 = v[2 * i], x1 = v[2 * i + 1];
    a[i] = bf16x2_rn(x0, x1);
    const float r0 = x0 - bf16_lo_val(a[i]), r1 = x1 - bf16_hi_val(a[i]);
    b[i] = bf16x2_rn(r0, r1);
    c[i] = bf16x2_rn(r0 - bf16_lo_val(b[i]), r1 - bf16_hi_val(b[i]));
  }
  t0 = make_uint4(a[0], a[1], a[2], a[3]);
  t1 = make_uint4(b[0], b[1], b[2], b[3]);
  t2 = make_uint4(c[0], c[1], c[2], c[3]);
}
// the value of a packed three-term word group, element e
__device__ __forceinline__ float term_sum(const uint4 &t0, const uint4 &t1, const uint4 &t2, int e) {
  const uint32_t w0 = e < 2 ? t0.x : e < 4 ? t0.y : e < 6 ? t0.z : t0.w;
  const uint32_t w1 = e < 2 ? t1.x : e < 4 ? t1.y : e < 6 ? t1.z : t1.w;
  const uint32_t w2 = e < 2 ? t2.x : e < 4 ? t2.y : e < 6 ? t2.z : t2.w;
  return (e & 1) ? (bf16_hi_val(w0) + bf16_hi_val(w1)) + bf16_hi_val(w2)
                 : (bf16_lo_val(w0) + bf16_lo_val(w1)) + bf16_lo_val(w2);
}

template <int HD, int GRP>
__global__ void __launch_bounds__(AT_THREADS, 1)
    pf_attn_tc(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv, const PfArgs a,
               int layer, int t0, int nt) {
  using LY = AttnLayout<HD>;
  constexpr int TT = AT_ROWS / GRP;                     // tokens per CTA
  extern __shared__ unsigned char smraw[];
  unsigned char *sm = smraw + ((1024u - (smem_addr(smraw) & 1023u)) & 1023u);
  // control block
  uint64_t *kfull = reinterpret_cast<uint64_t *>(sm);   // [2]
  uint64_t *kfree = kfull + 2, *vfull = kfull + 4, *vfree = kfull + 6;
  uint64_t *sfull = kfull + 8, *sfree = kfull + 10;     // [2] each
  uint64_t *pfull = kfull + 12, *pfree = kfull + 13, *ofull = kfull + 14, *sdone = kfull + 15;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(kfull + 16);
  unsigned char *buf = sm + 1024;
  unsigned char *Qs = buf + LY::Q_OFF, *Ks = buf + LY::K_OFF, *Vs = buf + LY::V_OFF, *Ps = buf + LY::P_OFF;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y;
  const int tok0 = blockIdx.x * TT;
  const int ntok = min(TT, nt - tok0);
  const int base_pos = a.call->pos0 + t0;
  const int pmax = base_pos + tok0 + ntok - 1;          // the CTA's last cached slot
  // position split z: tiles [jb, jb + nT) of this query tile's 0 .. pmax / AT_POS
  const int ns = gridDim.z;
  const int tps = ns > 1 ? ((base_pos + nt - 1) / AT_POS + ns) / ns : 0;   // the chunk's tiles / ns, rounded up
  const int jb = ns > 1 ? static_cast<int>(blockIdx.z) * tps : 0;
  const int nT = ns > 1 ? max(0, min(pmax / AT_POS + 1, jb + tps) - jb) : pmax / AT_POS + 1;   // tiles per pass
  const int qrows = a.Hq * HD;
  if (nT == 0) {
    // no cached position of this split reaches these rows: an empty state (l = 0)
    if (threadIdx.x < AT_ROWS) {
      const int r = threadIdx.x, tt = r / GRP, h = r % GRP;
      if (tt < ntok) {
        float *dst = a.attn_part + ((static_cast<size_t>(blockIdx.z) * nt + tok0 + tt) * a.Hq + g * GRP + h) * (HD + 2);
        dst[HD] = -INFINITY;
        dst[HD + 1] = 0.f;
      }
    }
    return;
  }
  (void)qrows;
  const int rows = (a.Hq + 2 * a.Hkv) * HD;
  const int kv_row0 = (layer * a.Hkv + g) * a.max_seq;  // first cache row of (layer, g)

  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&kfree[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&vfree[i], 1);
      mbar_init(&sfull[i], 1);
      mbar_init(&sfree[i], AT_SOFT_WARPS);
    }
    mbar_init(pfull, AT_SOFT_WARPS);
    mbar_init(pfree, 1);
    mbar_init(ofull, 1);
    mbar_init(sdone, 1);
    fence_mbar_init();
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
  }
  if (warp == 9) tmem_alloc(tslot, LY::TMEM_COLS);

  // ---- Q (fp32) -> three bf16 terms in shared memory, K-major swizzled -----
  if (warp < AT_SOFT_WARPS) {
    const int r = 32 * (warp & 3) + lane;               // the query row; the two warps of a row split head_dim
    const int tt = r / GRP, h = r % GRP;
    const float *q = a.qkv + static_cast<size_t>(tok0 + tt) * rows + static_cast<size_t>(g * GRP + h) * HD;
#pragma unroll 1
    for (int c8 = (warp >> 2) * (HD / 16); c8 < ((warp >> 2) + 1) * (HD / 16); ++c8) {
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = tt < ntok ? q[c8 * 8 + e] : 0.f;
      uint4 t0, t1, t2;
      split3x8(v, t0, t1, t2);
      const uint32_t off = (c8 >> 3) * (AT_ROWS * 128) + sw128(r, (c8 & 7) * 8);
      *reinterpret_cast<uint4 *>(Qs + off) = t0;
      *reinterpret_cast<uint4 *>(Qs + LY::Q_TERM + off) = t1;
      *reinterpret_cast<uint4 *>(Qs + 2 * LY::Q_TERM + off) = t2;
    }
    fence_proxy_async_smem();                           // generic writes -> tensor-core reads
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const int total = 2 * nT;                             // S tiles over both passes

  if (warp == 8) {
    // ---------------- TMA: K tiles (both passes), V tiles (pass 2) ----------------
    if (lane == 0) {
      const uint64_t keep = l2_evict_last();
      int nk = 0, nv = 0;                               // loads issued
      for (int u = 0; u < total; ++u) {
        const int j = u < nT ? u : u - nT;
        const int kb = u & 1;
        if (u >= 2 && !mbar_wait(&kfree[kb], ((u >> 1) - 1) & 1, AT_WAIT_NS)) {
          atomicCAS(a.err, 0, MK_ERR_TIMEOUT);
          break;
        }
        mbar_expect_tx(&kfull[kb], LY::KV_TILE);
#pragma unroll
        for (int at = 0; at < LY::ATOMS; ++at)
          tma_load_2d_hint(Ks + kb * LY::KV_TILE + at * (AT_POS * 128), &tk, at * 64, kv_row0 + (jb + j) * AT_POS,
                           &kfull[kb], keep);
        ++nk;
        if (u >= nT) {
          const int vb = j & 1;
          if (j >= 2 && !mbar_wait(&vfree[vb], ((j >> 1) - 1) & 1, AT_WAIT_NS)) {
            atomicCAS(a.err, 0, MK_ERR_TIMEOUT);
            break;
          }
          mbar_expect_tx(&vfull[vb], LY::KV_TILE);
#pragma unroll
          for (int at = 0; at < LY::ATOMS; ++at)
            tma_load_2d_hint(Vs + vb * LY::KV_TILE + at * (AT_POS * 128), &tv, at * 64, kv_row0 + (jb + j) * AT_POS,
                             &vfull[vb], keep);
          ++nv;
        }
      }
      // no copy may still be landing when the CTA exits (they all land, also on
      // the error path: the last fill of each buffer is waited for)
      for (int u = nk - 2 < 0 ? 0 : nk - 2; u < nk; ++u) mbar_wait(&kfull[u & 1], (u >> 1) & 1, AT_WAIT_NS);
      for (int j = nv - 2 < 0 ? 0 : nv - 2; j < nv; ++j) mbar_wait(&vfull[j & 1], (j >> 1) & 1, AT_WAIT_NS);
    }
  } else if (warp == 9) {
    // ---------------- S = Q K^T (M 128, N 64, K head_dim, three Q terms) -------------
    if (lane == 0) {
      constexpr uint32_t IDS = idesc_bf16_f32(AT_ROWS, AT_POS);
      const uint32_t qa = smem_addr(Qs), ka = smem_addr(Ks);
      for (int u = 0; u < total; ++u) {
        const int sb = u & 1;
        if (!mbar_wait(&kfull[sb], (u >> 1) & 1, AT_WAIT_NS) ||
            (u >= 2 && !mbar_wait(&sfree[sb], ((u >> 1) - 1) & 1, AT_WAIT_NS))) {
          atomicCAS(a.err, 0, MK_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t d = tbase + static_cast<uint32_t>(sb * AT_POS);
#pragma unroll
        for (int term = 0; term < AT_TERMS; ++term)
#pragma unroll
          for (int s = 0; s < HD / 16; ++s) {
            const uint32_t within = static_cast<uint32_t>((s & 3) * 32);
            const uint64_t ad = desc_sw128(qa + term * LY::Q_TERM + (s >> 2) * (AT_ROWS * 128) + within);
            const uint64_t bd = desc_sw128(ka + sb * LY::KV_TILE + (s >> 2) * (AT_POS * 128) + within);
            mma_bf16(d, ad, bd, IDS, (term | s) != 0);
          }
        mma_commit(&sfull[sb]);
        mma_commit(&kfree[sb]);
      }
      mma_commit(sdone);                                // all S MMAs of this CTA finished
      mbar_wait(sdone, 0, AT_WAIT_NS);
    }
  } else if (warp == 10) {
    // ---------------- O += P V (M 128, N head_dim, K 64 positions, three P terms) -------
    if (lane == 0) {
      constexpr uint32_t IDO = idesc_bf16_f32(AT_ROWS, HD) | (1u << 16);   // B (V) MN-major
      const uint32_t pa = smem_addr(Ps), va = smem_addr(Vs);
      const uint32_t dO = tbase + 2 * AT_POS;
      for (int j = 0; j < nT; ++j) {
        const int vb = j & 1;
        if (!mbar_wait(pfull, j & 1, AT_WAIT_NS) || !mbar_wait(&vfull[vb], (j >> 1) & 1, AT_WAIT_NS)) {
          atomicCAS(a.err, 0, MK_ERR_TIMEOUT);
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int term = 0; term < AT_TERMS; ++term)
#pragma unroll
          for (int s = 0; s < AT_POS / 16; ++s) {
            const uint64_t ad = desc_sw128(pa + term * LY::P_TERM + s * 32);
            const uint64_t bd = desc_mn_sw128(va + vb * LY::KV_TILE + s * 2048, AT_POS * 128, 1024);
            mma_bf16(dO, ad, bd, IDO, (j | term | s) != 0);
          }
        mma_commit(pfree);
        mma_commit(&vfree[vb]);
      }
      mma_commit(ofull);                                // the accumulator is final (or abandoned)
    }
  } else {
    // ---------------- softmax warps: one query row per thread, half the columns ----------
    const int qd = warp & 3, hf = warp >> 2;            // TMEM lane quarter, column half
    const int r = 32 * qd + lane;
    const int tt = r / GRP;
    const int prow = tt < ntok ? base_pos + tok0 + tt : pmax;   // the row's own position
    const uint32_t tl = tbase + (static_cast<uint32_t>(32 * qd) << 16);
    float *xm = reinterpret_cast<float *>(buf + LY::X_OFF);      // [2 halves][128 rows] maxima, then sums
    float m = -INFINITY;
    bool ok = true;
    // pass 1: the row maximum over the unmasked positions of this half
    for (int u = 0; u < nT && ok; ++u) {
      const int sb = u & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&sfull[sb], (u >> 1) & 1, AT_WAIT_NS))) {   // warp-uniform
        if (lane == 0) atomicCAS(a.err, 0, MK_ERR_TIMEOUT);
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < AT_POS / 2; c0 += 16) {
        const int col = hf * (AT_POS / 2) + c0;
        float v[16];
        tmem_ld16(tl + static_cast<uint32_t>(sb * AT_POS + col), v);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if ((jb + u) * AT_POS + col + i <= prow) m = fmaxf(m, v[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfree[sb]);
    }
    // the two halves' maxima meet in shared memory (all softmax warps pass here)
    xm[hf * AT_ROWS + r] = m;
    asm volatile("bar.sync 1, %0;" ::"r"(AT_SOFT_WARPS * 32) : "memory");
    m = fmaxf(xm[r], xm[AT_ROWS + r]);
    // pass 2: p = exp(s - m) as three bf16 terms, l = sum of the p multiplied
    float l = 0.f;
    for (int j = 0; j < nT && ok; ++j) {
      const int u = nT + j, sb = u & 1;
      const bool ready = mbar_wait(&sfull[sb], (u >> 1) & 1, AT_WAIT_NS) &&
                         (j == 0 || mbar_wait(pfree, (j - 1) & 1, AT_WAIT_NS));
      if (!__all_sync(0xffffffffu, ready)) {
        if (lane == 0) atomicCAS(a.err, 0, MK_ERR_TIMEOUT);
        ok = false;
        break;
      }
      tc_fence_after();
      float lt = 0.f;                                   // this tile's sum, then added to l
#pragma unroll
      for (int c0 = 0; c0 < AT_POS / 2; c0 += 16) {
        const int col = hf * (AT_POS / 2) + c0;
        float v[16];
        tmem_ld16(tl + static_cast<uint32_t>(sb * AT_POS + col), v);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float pv[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int c = col + half * 8 + e;
            pv[e] = ((jb + j) * AT_POS + c <= prow) ? __expf(v[half * 8 + e] - m) : 0.f;
          }
          uint4 t0, t1, t2;
          split3x8(pv, t0, t1, t2);
#pragma unroll
          for (int e = 0; e < 8; ++e) lt += term_sum(t0, t1, t2, e);
          const uint32_t off = sw128(r, col + half * 8);
          *reinterpret_cast<uint4 *>(Ps + off) = t0;
          *reinterpret_cast<uint4 *>(Ps + LY::P_TERM + off) = t1;
          *reinterpret_cast<uint4 *>(Ps + 2 * LY::P_TERM + off) = t2;
        }
      }
      l += lt;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sfree[sb]);
        mbar_arrive(pfull);
      }
    }
    // o = O / l for the rows of real tokens (each half of a row stores half of head_dim)
    xm[2 * AT_ROWS + hf * AT_ROWS + r] = l;
    asm volatile("bar.sync 1, %0;" ::"r"(AT_SOFT_WARPS * 32) : "memory");
    l = xm[2 * AT_ROWS + r] + xm[3 * AT_ROWS + r];
    const bool done = __all_sync(0xffffffffu, mbar_wait(ofull, 0, AT_WAIT_NS));
    tc_fence_after();
    if (!done) {
      if (lane == 0) atomicCAS(a.err, 0, MK_ERR_TIMEOUT);
    } else if (ok) {
      // one split: o = O / l; several: this split's O with the row's m and l
      const float inv = ns > 1 ? 1.0f : 1.0f / l;
      const int h = r % GRP;
      float *dst = ns > 1 ? a.attn_part + ((static_cast<size_t>(blockIdx.z) * nt + tok0 + tt) * a.Hq + g * GRP + h) *
                                              (HD + 2)
                          : a.attn + static_cast<size_t>(tok0 + tt) * a.Hq * HD + static_cast<size_t>(g * GRP + h) * HD;
      if (ns > 1 && hf == 0 && tt < ntok) {
        dst[HD] = l > 0.f ? m : -INFINITY;
        dst[HD + 1] = l;
      }
#pragma unroll 1
      for (int c0 = hf * (HD / 2); c0 < (hf + 1) * (HD / 2); c0 += 16) {
        float v[16];
        tmem_ld16(tl + static_cast<uint32_t>(2 * AT_POS + c0), v);
        if (tt < ntok) {
#pragma unroll
          for (int i = 0; i < 16; i += 2)
            *reinterpret_cast<float2 *>(dst + c0 + i) = make_float2(v[i] * inv, v[i + 1] * inv);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) tmem_dealloc(tbase, LY::TMEM_COLS);
}

// The position splits of one (token, q head): o = sum_s e^(m_s - M) O_s /
// sum_s e^(m_s - M) l_s with M the largest m_s of the non-empty splits, in
// split order.  One warp per (token, head), lane l dims l, l + 32, ...
template <int HD>
__global__ void pf_attn_merge(const PfArgs a, int nt, int ns) {
  const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (wid >= nt * a.Hq) return;
  const int tok = wid / a.Hq, head = wid - tok * a.Hq;
  const size_t stride = static_cast<size_t>(nt) * a.Hq * (HD + 2);
  const float *src = a.attn_part + (static_cast<size_t>(tok) * a.Hq + head) * (HD + 2);
  float M = -INFINITY;
  for (int z = 0; z < ns; ++z)
    if (src[z * stride + HD + 1] > 0.f) M = fmaxf(M, src[z * stride + HD]);
  float L = 0.f, o[HD / 32];
#pragma unroll
  for (int k = 0; k < HD / 32; ++k) o[k] = 0.f;
  for (int z = 0; z < ns; ++z) {
    const float lz = src[z * stride + HD + 1];
    if (lz > 0.f) {
      const float w = expf(src[z * stride + HD] - M);
      L = fmaf(w, lz, L);
#pragma unroll
      for (int k = 0; k < HD / 32; ++k) o[k] = fmaf(w, src[z * stride + lane + 32 * k], o[k]);
    }
  }
  float *dst = a.attn + (static_cast<size_t>(tok) * a.Hq + head) * HD;
#pragma unroll
  for (int k = 0; k < HD / 32; ++k) dst[lane + 32 * k] = o[k] / L;
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

template <int HD, int GRP>
int launch_tc(const CUtensorMap &tk, const CUtensorMap &tv, const PfArgs &a, int layer, int t0, int nt,
              cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(pf_attn_tc<HD, GRP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(AttnLayout<HD>::SMEM)) != cudaSuccess) {
      cudaGetLastError();
      return MK_ERR_CUDA;
    }
    attr = true;
  }
  constexpr int TT = AT_ROWS / GRP;
  // prompts reaching past PF_ATTN_SPLIT_MIN positions (from the chunk's first
  // token at slot pos0 = 0) split their positions over PF_ATTN_SPLITS CTAs
  const int ns = (t0 + nt > PF_ATTN_SPLIT_MIN) ? PF_ATTN_SPLITS : 1;
  pf_attn_tc<HD, GRP><<<dim3((nt + TT - 1) / TT, a.Hkv, ns), AT_THREADS, AttnLayout<HD>::SMEM, s>>>(tk, tv, a, layer,
                                                                                                      t0, nt);
  if (ns > 1) {
    const int warps = nt * a.Hq;
    pf_attn_merge<HD><<<(warps + 7) / 8, 256, 0, s>>>(a, nt, ns);
  }
  return cudaGetLastError() == cudaSuccess ? MK_OK : MK_ERR_CUDA;
}

}  // namespace

bool attn_tc_maps(const PfArgs &a, CUtensorMap *tk, CUtensorMap *tv) {
  const uint64_t rows = static_cast<uint64_t>(a.L) * a.Hkv * a.max_seq;
  return mkg::make_tmap(tk, a.kcache, a.d, rows, a.d * 2ull, AT_POS) &&
         mkg::make_tmap(tv, a.vcache, a.d, rows, a.d * 2ull, AT_POS);
}

int attn_tc_launch(const CUtensorMap &tk, const CUtensorMap &tv, const PfArgs &a, int layer, int t0, int nt,
                   cudaStream_t s) {
  const int grp = a.Hq / a.Hkv;
  if (a.d == 128) {
    switch (grp) {
      case 1: return launch_tc<128, 1>(tk, tv, a, layer, t0, nt, s);
      case 2: return launch_tc<128, 2>(tk, tv, a, layer, t0, nt, s);
      default: return MK_ERR_UNSUPPORTED;
    }
  }
  switch (grp) {
    case 1: return launch_tc<64, 1>(tk, tv, a, layer, t0, nt, s);
    case 2: return launch_tc<64, 2>(tk, tv, a, layer, t0, nt, s);
    case 4: return launch_tc<64, 4>(tk, tv, a, layer, t0, nt, s);
    default: return MK_ERR_UNSUPPORTED;
  }
}

}  // namespace mkp
