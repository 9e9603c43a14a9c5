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

namespace bq {

namespace {

__device__ __forceinline__ int qmax_of(int bits) { return bits == 8 ? 127 : (bits == 4 ? 7 : 1); }

constexpr float RNE_MAGIC = 12582912.0f;   // 1.5 * 2**23: adding it rounds |t| < 2**22 to an integer (ties to even)

// Code for one element from the stored fp16 scale s (as float) and its
// reciprocal rcp = RN(1 / s) (0 when s == 0, which yields code 0), returned
// as a float that carries the code in its low byte (two's complement).  In
// F32DIV mode the code is rne(RN(x / s)) clamped to [-d, d].  RN(x * rcp)
// differs from RN(x / s) by less than 2**-14 for |x / s| < 256, so both round
// to the same integer unless the product lies within 2**-12 of a
// half-integer; only then is the IEEE division evaluated.  The rounding is
// t + 1.5 * 2**23 in fp32 (round to nearest even), whose low mantissa bits are
// then the integer, so no float -> int conversion is needed; clamping before
// the rounding equals clamping after it, the bounds being integers.
__device__ __forceinline__ float code_exact(float x, float s, float fd, int mode) {
  float t = s == 0.0f ? 0.0f : __fdiv_rn(x, s);
  if (mode == BQ_ROUND_BMINF_HALF) t = __half2float(__float2half_rn(t));
  return __fadd_rn(fminf(fmaxf(t, -fd), fd), RNE_MAGIC);
}

// Fast form for F32DIV: the code of x, and whether the product was too close
// to a half-integer for it to be trusted (then code_exact decides).
__device__ __forceinline__ float code_fast(float x, float rcp, float fd, bool& unsure) {
  const float tc = fminf(fmaxf(__fmul_rn(x, rcp), -fd), fd);
  const float m = __fadd_rn(tc, RNE_MAGIC);
  unsure = fabsf(tc - __fsub_rn(m, RNE_MAGIC)) > 0.5f - 2.44140625e-4f;
  return m;
}

__device__ __forceinline__ float quant_one(float x, float s, float rcp, float fd, int mode) {
  if (mode == BQ_ROUND_BMINF_HALF) return code_exact(x, s, fd, mode);
  bool unsure;
  const float m = code_fast(x, rcp, fd, unsure);
  return unsure ? code_exact(x, s, fd, mode) : m;
}

__device__ __forceinline__ uint32_t code_byte(float m) { return __float_as_uint(m); }

// Fast F32DIV form for two elements with packed fp32x2 arithmetic (each lane
// of a packed op is an ordinary IEEE round-to-nearest operation): the codes
// m = RN(x * rcp) + 1.5 * 2**23 and the distances |RN(x * rcp) - rne(.)|.
__device__ __forceinline__ void code_fast2(float x0, float x1, float rcp, float& m0, float& m1, float& d0,
                                           float& d1) {
  asm("{\n\t.reg .b64 x, c, g, t, m, r, d;\n\t"
      "mov.b64 x, {%4, %5};\n\t"
      "mov.b64 c, {%6, %6};\n\t"
      "mov.b64 g, {%7, %7};\n\t"
      "mul.rn.f32x2 t, x, c;\n\t"
      "add.rn.f32x2 m, t, g;\n\t"
      "sub.rn.f32x2 r, m, g;\n\t"
      "sub.rn.f32x2 d, t, r;\n\t"
      "mov.b64 {%0, %1}, m;\n\t"
      "mov.b64 {%2, %3}, d;\n\t}"
      : "=f"(m0), "=f"(m1), "=f"(d0), "=f"(d1)
      : "f"(x0), "f"(x1), "f"(rcp), "f"(RNE_MAGIC));
}

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
          // |x / s| <= d (1 + 2**-11) for a normal scale, so no code needs clamping
          float dev = 0.0f;
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            float d0, d1;
            code_fast2(f[e], f[e + 1], rcp, m[e], m[e + 1], d0, d1);
            dev = fmaxf(dev, fmaxf(fabsf(d0), fabsf(d1)));
          }
          if (dev > 0.5f - 2.44140625e-4f) {   // rare: a product within 2**-12 of a half-integer
#pragma unroll
            for (int e = 0; e < 8; ++e) m[e] = quant_one(f[e], s, rcp, fd, MODE);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) m[e] = quant_one(f[e], s, rcp, fd, MODE);
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
  const float rcp = s == 0.0f ? 0.0f : __frcp_rn(s);
  if (threadIdx.x == 0) scale[row] = sh;
  int8_t* qr = q + row * cols;
  for (int64_t c = threadIdx.x; c < cols; c += blockDim.x)
    qr[c] = (int8_t)(uint8_t)(code_byte(quant_one(load_as_float(xr + c), s, rcp, (float)d, mode)) & 0xffu);
}

template <int VPT>
cudaError_t launch_rows_f16(const void* x, int64_t rows, int64_t cols, int64_t ld_x, int bits, int mode, int8_t* q,
                            uint16_t* scale, cudaStream_t stream) {
  const int64_t blocks = (int64_t)sm_count() * Q_BLOCKS_PER_SM;
  const unsigned grid = (unsigned)(rows < blocks ? rows : blocks);
  if (mode == BQ_ROUND_BMINF_HALF)
    quantize_rows_f16_kernel<VPT, BQ_ROUND_BMINF_HALF><<<grid, QT, 0, stream>>>(
        static_cast<const __half*>(x), rows, cols, ld_x, bits, q, reinterpret_cast<__half*>(scale));
  else
    quantize_rows_f16_kernel<VPT, BQ_ROUND_F32DIV><<<grid, QT, 0, stream>>>(
        static_cast<const __half*>(x), rows, cols, ld_x, bits, q, reinterpret_cast<__half*>(scale));
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
