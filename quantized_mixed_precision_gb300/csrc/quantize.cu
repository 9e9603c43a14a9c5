// Symmetric per-row quantisation (row absmax -> fp16 scale -> rounded codes),
// fused into one pass over x.
//
// Follows "BMINF的後訓練量化實現", section 實現代碼分析2: the scale is
// abs(row absmax) / D stored as fp16, and the codes are nearbyint(x / scale)
// computed from that stored scale (quantize_copy_float), or with the quotient
// first rounded to fp16 (quantize_copy_half).  The page runs a reduction
// kernel and then an elementwise kernel, reading x twice; here one block keeps
// its row in registers so x is read from HBM once.
#include <cuda_fp16.h>

#include "bq_device.cuh"
#include "bq_internal.h"
#include "gemm_common.cuh"
#include "quant_math.cuh"

namespace bq {

namespace {

__device__ __forceinline__ int qmax_of(int bits) { return bits == 8 ? 127 : (bits == 4 ? 7 : 1); }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// fp16 rows with cols % 8 == 0 and cols <= 1024 * VPT: 128-thread blocks walk
// the rows b, b + gridDim.x, ...; a row lives in registers as VPT 16-byte
// vectors per thread (x is read from HBM exactly once), and the next row's
// loads are issued before the current row is reduced and coded, so the
// arithmetic of one row overlaps the memory latency of the next.
constexpr int QT = 128;
constexpr int Q_BLOCKS_PER_SM = 8;

template <int VPT, int MODE>
__global__ void __launch_bounds__(QT, Q_BLOCKS_PER_SM) quantize_rows_f16_kernel(const __half* __restrict__ x,
                                                                                int64_t rows, int64_t cols,
                                                                                int64_t ld_x, int bits,
                                                                                int8_t* __restrict__ q,
                                                                                __half* __restrict__ scale) {
  __shared__ float red[2][QT / 32];
  const int tid = threadIdx.x;
  const int nvec = (int)(cols >> 3);
  const int d = qmax_of(bits);
  const float fd = (float)d;
  int64_t row = blockIdx.x;
  if (row >= rows) return;
  uint4 v[VPT], vn[VPT];
  {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * ld_x);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int idx = tid + QT * i;
      v[i] = idx < nvec ? __ldcs(xr + idx) : make_uint4(0, 0, 0, 0);   // streamed once
    }
  }
#pragma unroll 1
  for (int it = 0; row < rows; row += gridDim.x, ++it) {
    const int64_t nrow = row + gridDim.x;
    if (nrow < rows) {
      const uint4* xn = reinterpret_cast<const uint4*>(x + nrow * ld_x);
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int idx = tid + QT * i;
        vn[i] = idx < nvec ? __ldcs(xn + idx) : make_uint4(0, 0, 0, 0);
      }
    }
    // |x| and max are exact in fp16: reduce packed pairs, convert once
    __half2 m2 = __float2half2_rn(0.0f);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const __half2* h = reinterpret_cast<const __half2*>(&v[i]);
#pragma unroll
      for (int j = 0; j < 4; ++j) m2 = __hmax2(m2, __habs2(h[j]));
    }
    float amax = fmaxf(__low2float(m2), __high2float(m2));
    amax = warp_max(amax);
    float* rb = red[it & 1];   // alternate buffers: one barrier per row suffices
    if ((tid & 31) == 0) rb[tid >> 5] = amax;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < QT / 32; ++w) amax = fmaxf(amax, rb[w]);
    const __half sh = __float2half_rn(__fdiv_rn(amax, fd));
    const float s = __half2float(sh);
    const float rcp = s == 0.0f ? 0.0f : __frcp_rn(s);
    const bool normal_scale = s >= 6.103515625e-05f;   // 2**-14, the smallest normal fp16
    if (tid == 0) scale[row] = sh;
    uint2* qr = reinterpret_cast<uint2*>(q + row * cols);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int idx = tid + QT * i;
      if (idx < nvec) {
        const __half2* h = reinterpret_cast<const __half2*>(&v[i]);
        float f[8], m[8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 p = __half22float2(h[j]);
          f[2 * j] = p.x;
          f[2 * j + 1] = p.y;
        }
        if (MODE == BQ_ROUND_F32DIV && normal_scale) {
          // |x / s| <= d (1 + 2**-11) for a normal scale: no code needs
          // clamping, and the division-free form gives the code exactly
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            float r0, r1;
            code2_fast(f[e], f[e + 1], s, rcp, m[e], m[e + 1], r0, r1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) m[e] = code_exact(f[e], s, fd, MODE);
        }
        // low bytes of the codes -> two words
        uint32_t packed[2];
#pragma unroll
        for (int j = 0; j < 2; ++j)
          packed[j] = __byte_perm(__byte_perm(code_byte(m[4 * j]), code_byte(m[4 * j + 1]), 0x0040),
                                  __byte_perm(code_byte(m[4 * j + 2]), code_byte(m[4 * j + 3]), 0x0040), 0x5410);
        __stcs(qr + idx, make_uint2(packed[0], packed[1]));
      }
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) v[i] = vn[i];
  }
}

// Any element type / shape: one 256-thread block per row, two passes
// (the second pass reads the row again, normally from L2).
template <typename T>
__device__ __forceinline__ float load_as_float(const T* p);
template <>
__device__ __forceinline__ float load_as_float<__half>(const __half* p) {
  return __half2float(*p);
}
template <>
__device__ __forceinline__ float load_as_float<float>(const float* p) {
  return *p;
}

template <typename T>
__global__ void __launch_bounds__(256) quantize_rows_generic_kernel(const T* __restrict__ x, int64_t rows,
                                                                    int64_t cols, int64_t ld_x, int bits,
                                                                    int mode, int8_t* __restrict__ q,
                                                                    __half* __restrict__ scale) {
  __shared__ float red[8];
  const int64_t row = blockIdx.x;
  if (row >= rows) return;
  const T* xr = x + row * ld_x;
  float amax = 0.0f;
  for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) amax = fmaxf(amax, fabsf(load_as_float(xr + c)));
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
    v = warp_max(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  amax = red[0];
  const int d = qmax_of(bits);
  const __half sh = __float2half_rn(__fdiv_rn(amax, (float)d));
  const float s = __half2float(sh);
  if (threadIdx.x == 0) scale[row] = sh;
  int8_t* qr = q + row * cols;
  for (int64_t c = threadIdx.x; c < cols; c += blockDim.x)
    qr[c] = (int8_t)(uint8_t)(code_byte(code_exact(load_as_float(xr + c), s, (float)d, mode)) & 0xffu);
}

template <int VPT>
cudaError_t launch_rows_f16(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int bits, int mode, int8_t* q,
                            uint16_t* scale, cudaStream_t stream) {
  // as many rows per block as the resident blocks need, and then as few blocks
  // as carry that many rows each, so that no block walks one row more than
  // the others (4096 rows: 1024 blocks of 4, not 1216 blocks of 3 or 4)
  const int64_t blocks = (int64_t)sm_count() * Q_BLOCKS_PER_SM;
  const int64_t per = (rows + blocks - 1) / blocks;
  const unsigned grid = (unsigned)((rows + per - 1) / per);
  if (mode == BQ_ROUND_BMINF_HALF)
    quantize_rows_f16_kernel<VPT, BQ_ROUND_BMINF_HALF><<<grid, QT, 0, stream>>>(
        static_cast<const __half*>(x), rows, cols, ld_x, bits, q, reinterpret_cast<__half*>(scale));
  else
    quantize_rows_f16_kernel<VPT, BQ_ROUND_F32DIV><<<grid, QT, 0, stream>>>(
        static_cast<const __half*>(x), rows, cols, ld_x, bits, q, reinterpret_cast<__half*>(scale));
  return cudaGetLastError();
}

// Scales only (int8 codes, D = 127), for the fused quantised linear whose
// GEMM quantises the activations itself: one warp per fp16 row of `cols`
// elements (a multiple of 8, 16-byte aligned rows), the same absmax and fp16
// scale as the quantiser kernel.  x is read with ordinary caching so that the
// GEMM that follows finds it in L2.
constexpr int RS_WARPS = 8;

__global__ void __launch_bounds__(RS_WARPS * 32) row_scale_f16_kernel(const __half* __restrict__ x, int64_t rows,
                                                                     int64_t cols, __half* __restrict__ scale) {
  const int64_t row = (int64_t)blockIdx.x * RS_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * cols);
  const int nvec = (int)(cols >> 3);
  __half2 m2[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) m2[u] = __float2half2_rn(0.0f);
  int i = lane;
  for (; i + 96 < nvec; i += 128) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = xr[i + 32 * u];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const __half2* h = reinterpret_cast<const __half2*>(&v[u]);
#pragma unroll
      for (int j = 0; j < 4; ++j) m2[u] = __hmax2(m2[u], __habs2(h[j]));
    }
  }
  for (; i < nvec; i += 32) {
    const uint4 v = xr[i];
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int j = 0; j < 4; ++j) m2[0] = __hmax2(m2[0], __habs2(h[j]));
  }
  const __half2 m = __hmax2(__hmax2(m2[0], m2[1]), __hmax2(m2[2], m2[3]));
  float amax = fmaxf(__low2float(m), __high2float(m));
  amax = warp_max(amax);
  if (lane == 0) scale[row] = __float2half_rn(__fdiv_rn(amax, 127.0f));
}

// Row sums for the zero-point epilogue: one warp per row, each lane sums its
// 16-byte chunks in fp32 in k order, then a fixed butterfly across the warp.
__global__ void __launch_bounds__(RS_WARPS * 32) row_sum_f16_kernel(const __half* __restrict__ x, int64_t rows,
                                                                   int64_t cols, float* __restrict__ sum) {
  const int64_t row = (int64_t)blockIdx.x * RS_WARPS + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * cols);
  const int nvec = (int)(cols >> 3);
  float acc = 0.0f;
  for (int i = lane; i < nvec; i += 32) {
    const uint4 v = xr[i];
    const __half2* h = reinterpret_cast<const __half2*>(&v);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 p = __half22float2(h[j]);
      acc = __fadd_rn(__fadd_rn(acc, p.x), p.y);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
  if (lane == 0) sum[row] = acc;
}

}  // namespace

cudaError_t launch_row_sum_f16(const void* x, int64_t rows, int64_t cols, float* sum, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  if (cols == 0) return cudaMemsetAsync(sum, 0, (size_t)rows * sizeof(float), stream);
  const int64_t blocks = (rows + RS_WARPS - 1) / RS_WARPS;
  if (blocks > 0x7fffffffLL || cols % 8 != 0) return cudaErrorInvalidValue;
  row_sum_f16_kernel<<<(unsigned)blocks, RS_WARPS * 32, 0, stream>>>(static_cast<const __half*>(x), rows, cols, sum);
  return cudaGetLastError();
}

cudaError_t launch_row_scale_f16(const void* x, int64_t rows, int64_t cols, uint16_t* scale, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  if (cols == 0) return cudaMemsetAsync(scale, 0, (size_t)rows * sizeof(uint16_t), stream);
  const int64_t blocks = (rows + RS_WARPS - 1) / RS_WARPS;
  if (blocks > 0x7fffffffLL || cols % 8 != 0) return cudaErrorInvalidValue;
  row_scale_f16_kernel<<<(unsigned)blocks, RS_WARPS * 32, 0, stream>>>(static_cast<const __half*>(x), rows, cols,
                                                                       reinterpret_cast<__half*>(scale));
  return cudaGetLastError();
}

cudaError_t launch_quantize(const void* x, int xtype, int64_t rows, int64_t cols, int64_t ld_x, int bits, int mode,
                            int8_t* q, uint16_t* scale, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  if (cols == 0) {
    // absmax of an empty row is 0: scale 0, no codes
    return cudaMemsetAsync(scale, 0, (size_t)rows * sizeof(uint16_t), stream);
  }
  if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
  const bool vec_ok = xtype == BQ_F16 && (cols % 8) == 0 && (ld_x % 8) == 0 && cols <= 4096 &&
                      (reinterpret_cast<uintptr_t>(x) % 16) == 0 && (reinterpret_cast<uintptr_t>(q) % 8) == 0;
  if (vec_ok) {
    if (cols <= 1024) return launch_rows_f16<1>(x, rows, cols, ld_x, bits, mode, q, scale, stream);
    if (cols <= 2048) return launch_rows_f16<2>(x, rows, cols, ld_x, bits, mode, q, scale, stream);
    return launch_rows_f16<4>(x, rows, cols, ld_x, bits, mode, q, scale, stream);
  }
  if (rows > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (xtype == BQ_F16) {
    quantize_rows_generic_kernel<__half><<<(unsigned)rows, 256, 0, stream>>>(
        static_cast<const __half*>(x), rows, cols, ld_x, bits, mode, q, reinterpret_cast<__half*>(scale));
  } else {
    quantize_rows_generic_kernel<float><<<(unsigned)rows, 256, 0, stream>>>(
        static_cast<const float*>(x), rows, cols, ld_x, bits, mode, q, reinterpret_cast<__half*>(scale));
  }
  return cudaGetLastError();
}

}  // namespace bq
