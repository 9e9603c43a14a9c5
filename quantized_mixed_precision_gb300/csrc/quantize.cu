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

namespace bq {

namespace {

__device__ __forceinline__ int qmax_of(int bits) { return bits == 8 ? 127 : (bits == 4 ? 7 : 1); }

// Code for one element from the stored fp16 scale s (as float) and its
// reciprocal rcp = RN(1 / s) (0 when s == 0, which yields code 0).  In F32DIV
// mode the code is rne(RN(x / s)).  RN(x * rcp) differs from RN(x / s) by
// less than 2**-14 for |x / s| < 256, so both round to the same integer
// unless the product lies within 2**-12 of a half-integer; only then is the
// IEEE division evaluated.
__device__ __forceinline__ int quant_one(float x, float s, float rcp, int d, int mode) {
  float r;
  if (mode == BQ_ROUND_BMINF_HALF) {
    r = s == 0.0f ? 0.0f : rintf(__half2float(__float2half_rn(__fdiv_rn(x, s))));
  } else {
    const float t = __fmul_rn(x, rcp);
    r = rintf(t);                                     // nearest integer, ties to even
    if (fabsf(t - r) > 0.5f - 2.44140625e-4f) r = rintf(__fdiv_rn(x, s));
  }
  const int q = __float2int_rn(r);
  return q > d ? d : (q < -d ? -d : q);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One 128-thread block per row; the row (fp16, cols % 8 == 0,
// cols <= 1024 * VPT) lives in registers as VPT 16-byte vectors per thread,
// so x is read from HBM exactly once.
constexpr int QT = 128;

template <int VPT>
__global__ void __launch_bounds__(QT) quantize_rows_f16_kernel(const __half* __restrict__ x, int64_t rows,
                                                               int64_t cols, int64_t ld_x, int bits, int mode,
                                                               int8_t* __restrict__ q, __half* __restrict__ scale) {
  __shared__ float red[QT / 32];
  const int tid = threadIdx.x;
  const int64_t row = blockIdx.x;
  const int nvec = (int)(cols >> 3);
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * ld_x);
  uint4 v[VPT];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = tid + QT * i;
    v[i] = idx < nvec ? __ldcs(xr + idx) : make_uint4(0, 0, 0, 0);   // streamed once
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
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
#pragma unroll
  for (int w = 0; w < QT / 32; ++w) amax = fmaxf(amax, red[w]);
  const int d = qmax_of(bits);
  const __half sh = __float2half_rn(__fdiv_rn(amax, (float)d));
  const float s = __half2float(sh);
  const float rcp = s == 0.0f ? 0.0f : __frcp_rn(s);
  if (tid == 0) scale[row] = sh;
  uint2* qr = reinterpret_cast<uint2*>(q + row * cols);
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int idx = tid + QT * i;
    if (idx < nvec) {
      const __half2* h = reinterpret_cast<const __half2*>(&v[i]);
      uint32_t packed[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float2 f0 = __half22float2(h[2 * j]);
        const float2 f1 = __half22float2(h[2 * j + 1]);
        const uint32_t b0 = (uint32_t)quant_one(f0.x, s, rcp, d, mode);
        const uint32_t b1 = (uint32_t)quant_one(f0.y, s, rcp, d, mode);
        const uint32_t b2 = (uint32_t)quant_one(f1.x, s, rcp, d, mode);
        const uint32_t b3 = (uint32_t)quant_one(f1.y, s, rcp, d, mode);
        // low bytes of the four codes -> one word
        packed[j] = __byte_perm(__byte_perm(b0, b1, 0x0040), __byte_perm(b2, b3, 0x0040), 0x5410);
      }
      __stcs(qr + idx, make_uint2(packed[0], packed[1]));
    }
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
  const float rcp = s == 0.0f ? 0.0f : __frcp_rn(s);
  if (threadIdx.x == 0) scale[row] = sh;
  int8_t* qr = q + row * cols;
  for (int64_t c = threadIdx.x; c < cols; c += blockDim.x)
    qr[c] = (int8_t)quant_one(load_as_float(xr + c), s, rcp, d, mode);
}

template <int VPT>
cudaError_t launch_rows_f16(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int bits, int mode, int8_t* q,
                            uint16_t* scale, cudaStream_t stream) {
  quantize_rows_f16_kernel<VPT><<<(unsigned)rows, QT, 0, stream>>>(
      static_cast<const __half*>(x), rows, cols, ld_x, bits, mode, q, reinterpret_cast<__half*>(scale));
  return cudaGetLastError();
}

}  // namespace

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
