// Tensor-core GEMM of the batched prompt prefill (csrc/mk_gemm.cu):
//
//   out[s][t][n] = sum over k in split s of  W[n][k] * (hi + mid + lo)[t][k]
//
// W is a bf16 weight matrix [N][K] (row-major, nn.Linear layout); the fp32
// activation of token t enters as three bf16 terms hi, mid, lo (each the bf16
// rounding of what the terms before it left, so hi + mid + lo holds fp32's 24
// significant bits), stored as three bf16 matrices [tokens][K], one per term
// (a 3-D tensor: K, token, term).  Each term's products accumulate into its own
// fp32 accumulator in tensor memory (tcgen05.mma kind::f16, bf16 x bf16 ->
// fp32) and the three sums are added once at the end; operands reach shared
// memory through TMA tensor loads.  K may be split
// over `splits` CTAs per output tile; split s writes its own fp32 partial at
// out + s * part_stride and the reader sums the partials in split order.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mkg {

// A bf16 tensor map over rows of `inner` elements (`row_bytes` apart, a
// multiple of 16), `outer` rows, read in boxes of 64 x box_rows with the
// 128-byte swizzle; with planes > 1 a 3-D map of `planes` such matrices
// `plane_bytes` apart (box depth 1).  Returns false when the driver rejects it.
bool make_tmap(CUtensorMap *map, const void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
               uint32_t box_rows, uint64_t planes = 1, uint64_t plane_bytes = 0);

// Up to three weight matrices whose rows are stacked along the output: matrix
// i fills output columns [off_i, off_i + rows[i]) with off_0 = 0 and off_i =
// off_{i-1} + rows[i-1] (one launch for the q, k and v projections, or for
// gate and up).
struct WMaps {
  CUtensorMap map[3];
  int rows[3];
  int n;
};

struct GemmCall {
  int N, K, nt;            // output rows (all matrices), input width, tokens
  int t_off;               // first token read (output token t reads token t_off + t of each term)
  int splits;              // CTAs sharing one output tile's K range
  float *out;              // fp32, token-major: out[s * part_stride + t * ldc + n]
  size_t ldc, part_stride;
  int *err;                // set (first error wins) when a device wait times out
};

// Token block (MMA N) the launcher uses for nt tokens: 32, 64 or 128.
int gemm_block_tokens(int nt);

// The activation map (3-D: K, token, term) must have been made with box_rows
// = gemm_block_tokens(nt); the weight map (2-D) with box_rows = 128.  Enqueues one
// launch; MK_OK or MK_ERR_INVALID_ARG / MK_ERR_CUDA.
int gemm_launch(const WMaps &w, const CUtensorMap &x_map, const GemmCall &c, cudaStream_t s);

// splits for an N x K output with nt tokens: enough CTAs to cover the GPU's
// SMs, at least 4 K blocks of 64 per split, at most max_splits
int gemm_splits(int N, int K, int nt, int sms, int max_splits);

}  // namespace mkg
