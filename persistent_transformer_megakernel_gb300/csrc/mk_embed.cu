// Talker input rows for the negative-id sentinel: the sum of the codebook
// embeddings and the text embedding of each step (page B = "I made a single
// CUDA kernel speak: streaming Qwen3-TTS at 50ms latency on an RTX 5090",
// section "Why Does a Single Kernel Even Matter for TTS?": each talker input is
// that 17-way sum).  One CTA per row, fp32 accumulation in table
// order (codebook 0 .. n_books-1, then text).
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/mk.h"

namespace {

__global__ void embed_sum_kernel(const uint16_t *books, int n_books, int book_rows, const uint16_t *text,
                                 int text_rows, int H, const int32_t *codes, const int32_t *text_ids,
                                 float *out, int *err) {
  const int r = blockIdx.x;
  for (int k = threadIdx.x; k < H; k += blockDim.x) {
    float acc = 0.f;
    bool bad = false;
    for (int j = 0; j < n_books; ++j) {
      const int id = codes[static_cast<size_t>(r) * n_books + j];
      if (id < 0 || id >= book_rows) { bad = true; break; }
      acc += __uint_as_float(static_cast<uint32_t>(books[(static_cast<size_t>(j) * book_rows + id) * H + k]) << 16);
    }
    const int tid_ = text_ids[r];
    if (tid_ < 0 || tid_ >= text_rows) bad = true;
    if (bad) {
      atomicCAS(err, 0, 1);
      return;
    }
    acc += __uint_as_float(static_cast<uint32_t>(text[static_cast<size_t>(tid_) * H + k]) << 16);
    out[static_cast<size_t>(r) * H + k] = acc;
  }
}

}  // namespace

extern "C" int mk_embed_sum(const void *books, int32_t n_books, int32_t book_rows, const void *text,
                            int32_t text_rows, int32_t hidden, const int32_t *codes, const int32_t *text_ids,
                            int32_t n, float *out, mk_stream stream) {
  if (n < 0 || n_books < 0 || book_rows < 1 || text_rows < 1 || hidden < 1) return MK_ERR_INVALID_ARG;
  if (n == 0) return MK_OK;
  if ((n_books > 0 && (!books || !codes)) || !text || !text_ids || !out) return MK_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int *d_err = nullptr;
  if (cudaMallocAsync(&d_err, sizeof(int), s) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_NO_MEMORY;
  }
  cudaMemsetAsync(d_err, 0, sizeof(int), s);
  embed_sum_kernel<<<n, 256, 0, s>>>(static_cast<const uint16_t *>(books), n_books, book_rows,
                                     static_cast<const uint16_t *>(text), text_rows, hidden, codes, text_ids,
                                     out, d_err);
  int herr = 0;
  cudaError_t e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaMemcpyAsync(&herr, d_err, sizeof(int), cudaMemcpyDeviceToHost, s);
  cudaFreeAsync(d_err, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  return herr ? MK_ERR_BAD_TOKEN : MK_OK;
}

// ---------------------------------------------------------------------------
// mk_embed_sum_noalloc: the same sum for callers that must not allocate device
// memory (see include/mk.h).  Its scratch -- one status word per output row --
// lives in a fixed file-scope device array instead of a per-call allocation.
// ---------------------------------------------------------------------------
#include <mutex>

namespace {

constexpr int kNoAllocMaxRows = 4096;   // 16 KB of status words on every device using the library
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) int g_noalloc_status[kNoAllocMaxRows];

std::mutex g_noalloc_mu;                              // serialises calls (shared scratch)
int *g_noalloc_dev_ptr[kNoAllocMaxDevices] = {};      // device address of the array, per device
int g_noalloc_host[kNoAllocMaxRows];                  // host copy of the status words

// one CTA per row; a bad id marks status[r] instead of a shared error word
__global__ void embed_sum_status_kernel(const uint16_t *books, int n_books, int book_rows, const uint16_t *text,
                                        int text_rows, int H, const int32_t *codes, const int32_t *text_ids,
                                        float *out, int *status) {
  const int r = blockIdx.x;
  for (int k = threadIdx.x; k < H; k += blockDim.x) {
    float acc = 0.f;
    bool bad = false;
    for (int j = 0; j < n_books; ++j) {
      const int id = codes[static_cast<size_t>(r) * n_books + j];
      if (id < 0 || id >= book_rows) { bad = true; break; }
      acc += __uint_as_float(static_cast<uint32_t>(books[(static_cast<size_t>(j) * book_rows + id) * H + k]) << 16);
    }
    const int tid_ = text_ids[r];
    if (tid_ < 0 || tid_ >= text_rows) bad = true;
    if (bad) {
      status[r] = 1;
      return;
    }
    acc += __uint_as_float(static_cast<uint32_t>(text[static_cast<size_t>(tid_) * H + k]) << 16);
    out[static_cast<size_t>(r) * H + k] = acc;
  }
}

}  // namespace

extern "C" int mk_embed_sum_noalloc(const void *books, int32_t n_books, int32_t book_rows, const void *text,
                                    int32_t text_rows, int32_t hidden, const int32_t *codes,
                                    const int32_t *text_ids, int32_t n, float *out, mk_stream stream) {
  if (n < 0 || n_books < 0 || book_rows < 1 || text_rows < 1 || hidden < 1) return MK_ERR_INVALID_ARG;
  if (n > kNoAllocMaxRows) return MK_ERR_INVALID_ARG;      // more rows than the static scratch holds
  if (n == 0) return MK_OK;
  if ((n_books > 0 && (!books || !codes)) || !text || !text_ids || !out) return MK_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  if (dev < 0 || dev >= kNoAllocMaxDevices) return MK_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_dev_ptr[dev]) {
    // first call on this device (current now): look up the array's device address
    int *ptr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void **>(&ptr), g_noalloc_status) != cudaSuccess || !ptr) {
      cudaGetLastError();
      return MK_ERR_CUDA;
    }
    g_noalloc_dev_ptr[dev] = ptr;
  }
  int *status = g_noalloc_dev_ptr[dev];
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int) * n, s);   // the previous call's words remain
  if (e == cudaSuccess) {
    embed_sum_status_kernel<<<n, 256, 0, s>>>(static_cast<const uint16_t *>(books), n_books, book_rows,
                                              static_cast<const uint16_t *>(text), text_rows, hidden, codes,
                                              text_ids, out, status);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) e = cudaMemcpyAsync(g_noalloc_host, status, sizeof(int) * n, cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MK_ERR_CUDA;
  }
  for (int r = 0; r < n; ++r)
    if (g_noalloc_host[r]) return MK_ERR_BAD_TOKEN;
  return MK_OK;
}
