// Offline weight packer: int8 codes (n, k) -> 4-bit or 2-bit storage.
//
// The BitBLAS guide ("BitBLAS自定义操作开发指南", section 实际应用案例 案例2)
// stores 4-bit weights as an (N, K//2) uint8 matrix.  The plain layout keeps
// the lowest k in the lowest bits; the interleaved layout permutes fields
// inside every 32-bit word (even elements in the low 16 bits, odd elements in
// the high 16 bits, each in order) so that the GEMM kernels turn one masked
// word half into an in-order fp16 pair without any shuffle.
#include "bq_internal.h"

namespace bq {

namespace {

// One output byte per thread: plain layout.
__global__ void pack_plain_kernel(const int8_t* __restrict__ q, int64_t n, int64_t k, int bits,
                                  uint8_t* __restrict__ out) {
  const int per = 8 / bits;
  const int64_t row_bytes = k / per;
  const int64_t total = n * row_bytes;
  const uint32_t mask = (1u << bits) - 1u;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / row_bytes;
    const int64_t jb = i - r * row_bytes;
    const int8_t* src = q + r * k + jb * per;
    uint32_t byte = 0;
    for (int t = 0; t < per; ++t) byte |= ((uint32_t)(uint8_t)src[t] & mask) << (t * bits);
    out[i] = (uint8_t)byte;
  }
}

// One output 32-bit word per thread: interleaved layout.
__global__ void pack_inter_kernel(const int8_t* __restrict__ q, int64_t n, int64_t k, int bits,
                                  uint32_t* __restrict__ out) {
  const int e_per_word = 32 / bits;
  const int64_t row_words = k / e_per_word;
  const int64_t total = n * row_words;
  const uint32_t mask = (1u << bits) - 1u;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / row_words;
    const int64_t jw = i - r * row_words;
    const int8_t* src = q + r * k + jw * e_per_word;
    uint32_t w = 0;
    for (int e = 0; e < e_per_word; ++e) {
      const int pos = (e & 1) ? (e_per_word / 2 + (e >> 1)) : (e >> 1);
      w |= ((uint32_t)(uint8_t)src[e] & mask) << (pos * bits);
    }
    out[i] = w;
  }
}

}  // namespace

cudaError_t launch_pack(const int8_t* q, int64_t n, int64_t k, int bits, int layout, uint8_t* packed,
                        cudaStream_t stream) {
  if (n == 0 || k == 0) return cudaSuccess;
  if (bits == 8) return cudaMemcpyAsync(packed, q, (size_t)(n * k), cudaMemcpyDeviceToDevice, stream);
  const int threads = 256;
  int64_t work = layout == BQ_LAYOUT_PLAIN ? n * k * bits / 8 : n * k * bits / 32;
  int64_t blocks = (work + threads - 1) / threads;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (layout == BQ_LAYOUT_PLAIN) {
    pack_plain_kernel<<<(unsigned)blocks, threads, 0, stream>>>(q, n, k, bits, packed);
  } else {
    pack_inter_kernel<<<(unsigned)blocks, threads, 0, stream>>>(q, n, k, bits, reinterpret_cast<uint32_t*>(packed));
  }
  return cudaGetLastError();
}

}  // namespace bq
