// Pieces shared by the tensor-core GEMM kernels: host helpers, the weight-tile
// conversion into the 128B-swizzled K-major fp16 layout that tcgen05.mma
// reads, and a warp-uniform bounded mbarrier wait.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "bq_device.cuh"

namespace bq {

// 2-D tensor map over a row-major matrix of `rows` rows of `row_elems`
// elements (uint8, fp16 when elem == 2, int32 when elem == 4); box = box_x
// elements x box_rows rows; out-of-range elements read as zero and are not
// written by stores.
cudaError_t make_map(CUtensorMap* map, const void* base, int elem, uint64_t row_elems, uint64_t rows, uint32_t box_x,
                     uint32_t box_rows, CUtensorMapSwizzle swz);
// The same over `batch` matrices `item_stride` bytes apart: always a 3-D map
// (third coordinate = batch item, box depth 1), also for one item, so that a
// kernel's 3-D copies may use it; load and store only with 3-D copies.
cudaError_t make_map3(CUtensorMap* map, const void* base, int elem, uint64_t row_elems, uint64_t rows, uint64_t batch,
                      uint64_t item_stride, uint32_t box_x, uint32_t box_rows, CUtensorMapSwizzle swz);
// Streaming multiprocessors of the current device.
int sm_count();
// Split-K factor the single-CTA kernel uses for `tiles` 128-row tiles of nkb
// k-blocks (1 when the grid fills the GPU).
int choose_split(long long tiles, int nkb);

// Swizzle mode of a raw TMA box whose rows are box_x bytes (128, 64 or 32).
inline CUtensorMapSwizzle raw_swizzle(int box_x) {
  return box_x == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : (box_x == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

namespace {

// Position of 16-byte chunk `chunk` of row r inside a raw box with rows of
// BOX_X bytes, as the box's swizzle placed it (bits 4.. of the address XOR
// bits 7..: 128B swizzle 3 bits, 64B 2 bits, 32B 1 bit).
template <int BOX_X>
__device__ __forceinline__ int raw_chunk_pos(int chunk, int r) {
  static_assert(BOX_X == 128 || BOX_X == 64 || BOX_X == 32, "raw box row width");
  if constexpr (BOX_X == 128) return chunk ^ (r & 7);
  else if constexpr (BOX_X == 64) return chunk ^ ((r >> 1) & 3);
  else return chunk ^ ((r >> 2) & 1);
}

// Store one 16-byte fp16 chunk (logical chunk lc = 8 k values) of row r into a
// 128B-swizzled K-major tile (chunk c of row r lives at position c ^ (r & 7)).
__device__ __forceinline__ void st_chunk(uint8_t* tile, int r, int lc, uint4 v) {
  *reinterpret_cast<uint4*>(tile + r * 128 + ((lc ^ (r & 7)) << 4)) = v;
}

// Convert one 16-byte raw weight piece (row r, piece sub) and store it.
// UNS (4-bit only): the nibbles are unsigned codes u in [0, 15]; flipping
// their top bits makes them the two's-complement codes of u - 8.
template <int BBITS, bool INTER, bool UNS = false>
__device__ __forceinline__ void convert_b_piece(uint8_t* tb, int r, int sub, const uint4& v) {
  static_assert(!UNS || BBITS == 4, "unsigned codes are 4-bit");
  constexpr uint32_t FLIP = UNS ? 0x88888888u : 0u;
  const uint32_t wv[4] = {v.x ^ FLIP, v.y ^ FLIP, v.z ^ FLIP, v.w ^ FLIP};
  if constexpr (BBITS == 8) {
    uint4 o0, o1;
    cvt_i8x4_f16(wv[0], o0.x, o0.y);
    cvt_i8x4_f16(wv[1], o0.z, o0.w);
    cvt_i8x4_f16(wv[2], o1.x, o1.y);
    cvt_i8x4_f16(wv[3], o1.z, o1.w);
    st_chunk(tb, r, 2 * sub, o0);
    st_chunk(tb, r, 2 * sub + 1, o1);
  } else if constexpr (BBITS == 4) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t h[4];
      cvt_i4x8_f16(INTER ? wv[j] : plain_to_inter_i4(wv[j]), h);
      st_chunk(tb, r, 4 * sub + j, make_uint4(h[0], h[1], h[2], h[3]));
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t h[8];
      cvt_i2x16_f16(INTER ? wv[j] : plain_to_inter_i2(wv[j]), h);
      st_chunk(tb, r, 8 * sub + 2 * j, make_uint4(h[0], h[1], h[2], h[3]));
      st_chunk(tb, r, 8 * sub + 2 * j + 1, make_uint4(h[4], h[5], h[6], h[7]));
    }
  }
}

// Zero-point epilogue term for 32 consecutive output columns of one row:
// v[i] + (8 - z[ncol + i]) * rsum, one fp32 fma each.  v is the accumulated
// sum over x * (u - 8) (the unsigned 4-bit codes u converted as u - 8), so the
// result is the sum over x * (u - z) before the column scale.
__device__ __forceinline__ void add_zero_point(float* v, const __half* zero_point, int ncol, float rsum) {
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const __half2 z2 = *reinterpret_cast<const __half2*>(zero_point + ncol + 2 * i);
    v[2 * i] = __fmaf_rn(__fsub_rn(8.0f, __low2float(z2)), rsum, v[2 * i]);
    v[2 * i + 1] = __fmaf_rn(__fsub_rn(8.0f, __high2float(z2)), rsum, v[2 * i + 1]);
  }
}

// Wait on an mbarrier phase with every lane of the warp; true only if all
// lanes saw it complete (a warp-uniform decision).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns, int* status) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, timeout_ns, status));
}

}  // namespace
}  // namespace bq
