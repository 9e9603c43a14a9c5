// Skinny-M GEMM (M <= 16): one pass over the packed weights.
//
// The work is bound by reading the weights from HBM once (the decode-step
// use of the quantised linear in "BMINF的後訓練量化實現", 實現代碼分析2, runs
// with M = batch).  Each warp owns 16 weight rows and a share of K; every
// thread issues 16-byte loads of two weight rows, turns the 4- or 2-bit
// codes into fp16 pairs in registers (exact) and feeds them straight into
// mma.sync m16n8k16 as the A fragment, so weights never touch shared memory.
// The activations (at most 16 rows) sit in shared memory as fp16 (int8
// activations are converted exactly on the way in).  Accumulation is fp32;
// for integer operands every partial sum stays below 2**24 (checked on the
// host), so it is exact.
//
// K-permutation: inside one MMA the hardware pairs A column k with B row k.
// Thread t of a quad loads weight bytes [16t, 16t + 16) of a step; its fp16
// pairs are assigned to the MMA's k slots in load order, and the B fragment
// is read from the activation columns of exactly those k, so the contraction
// covers every k once with matching operands.
#include <cuda_fp16.h>

#include "bq_device.cuh"
#include "bq_internal.h"

namespace bq {

namespace {

constexpr int GEMV_WARPS = 8;

template <int BBITS>
struct GemvCfg {
  static constexpr int E16 = 128 / BBITS;             // codes per 16-byte load
  static constexpr int STEP = 4 * E16;                // k per step (4 threads of a quad)
  static constexpr int PAIRS = E16 / 2;               // fp16 pairs per 16-byte load
  static constexpr int MMAS = PAIRS / 2;              // m16n8k16 per step
  static constexpr int CH_PER_T = E16 / 8;            // 16-byte activation chunks per thread per step
  static constexpr int PAD = BBITS == 4 ? 16 : 64;    // row pad: conflict-free fragment loads
  // chunk position swizzle inside an activation row
  __device__ __forceinline__ static int swz(int c) {
    return BBITS == 4 ? (c ^ (((c >> 3) & 1) << 1)) : (c ^ ((c >> 3) & 7));
  }
};

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int BBITS, bool INTER>
__device__ __forceinline__ void convert_load(const uint4& v, uint32_t (&h)[GemvCfg<BBITS>::PAIRS]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BBITS == 4) {
      uint32_t t[4];
      cvt_i4x8_f16(INTER ? w[i] : plain_to_inter_i4(w[i]), t);
#pragma unroll
      for (int j = 0; j < 4; ++j) h[4 * i + j] = t[j];
    } else {
      uint32_t t[8];
      cvt_i2x16_f16(INTER ? w[i] : plain_to_inter_i2(w[i]), t);
#pragma unroll
      for (int j = 0; j < 8; ++j) h[8 * i + j] = t[j];
    }
  }
}

template <int BBITS, int ACT, int NB, bool INTER, int UNROLL>
__global__ void __launch_bounds__(GEMV_WARPS * 32) gemv_mma_kernel(const void* __restrict__ act,
                                                                   const uint8_t* __restrict__ w, int M, int N,
                                                                   int K, const __half* __restrict__ row_scale,
                                                                   const __half* __restrict__ col_scale, int epi,
                                                                   void* __restrict__ out) {
  using C = GemvCfg<BBITS>;
  extern __shared__ __align__(16) uint8_t smem[];
  const int rs = 2 * K + C::PAD;                      // activation row stride (bytes)
  float* red = reinterpret_cast<float*>(smem + (size_t)M * rs);  // [warps][NB][4][32]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t = lane & 3;

  // ---- stage activations (M rows) into shared memory as swizzled fp16 ----
  const int chunks_per_row = K >> 3;
  for (int idx = tid; idx < M * chunks_per_row; idx += blockDim.x) {
    const int m = idx / chunks_per_row, c = idx - m * chunks_per_row;
    uint4 v;
    if constexpr (ACT == ACT_F16) {
      v = __ldg(reinterpret_cast<const uint4*>(static_cast<const __half*>(act) + (size_t)m * K) + c);
    } else {
      const uint2 raw = __ldg(reinterpret_cast<const uint2*>(static_cast<const int8_t*>(act) + (size_t)m * K) + c);
      cvt_i8x4_f16(raw.x, v.x, v.y);
      cvt_i8x4_f16(raw.y, v.z, v.w);
    }
    *reinterpret_cast<uint4*>(smem + (size_t)m * rs + C::swz(c) * 16) = v;
  }
  __syncthreads();

  const int n0 = blockIdx.x * 16;
  const size_t row_bytes = (size_t)K * BBITS / 8;
  const uint8_t* w0 = w + (size_t)(n0 + g) * row_bytes + 16 * t;
  const uint8_t* w1 = w0 + 8 * row_bytes;
  const int nsteps = (K + C::STEP - 1) / C::STEP;

  float d[NB][4];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int i = 0; i < 4; ++i) d[nb][i] = 0.0f;

  for (int s0 = warp; s0 < nsteps; s0 += GEMV_WARPS * UNROLL) {
    uint4 v0[UNROLL], v1[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int s = s0 + u * GEMV_WARPS;
      const bool ok = s < nsteps && (s * C::STEP + t * C::E16) < K;
      if (ok) {
        const size_t off = (size_t)s * (C::STEP * BBITS / 8);
        v0[u] = __ldcs(reinterpret_cast<const uint4*>(w0 + off));
        v1[u] = __ldcs(reinterpret_cast<const uint4*>(w1 + off));
      } else {
        v0[u] = make_uint4(0, 0, 0, 0);
        v1[u] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int s = s0 + u * GEMV_WARPS;
      if (s >= nsteps) continue;                        // warp-uniform
      // Threads whose k range lies past K (a ragged last step) hold zero
      // codes and read zero activations; mma.sync needs the whole warp.
      const bool kin = (s * C::STEP + t * C::E16) < K;
      uint32_t h0[C::PAIRS], h1[C::PAIRS];
      convert_load<BBITS, INTER>(v0[u], h0);
      convert_load<BBITS, INTER>(v1[u], h1);
      const int cbase = (s * C::STEP + t * C::E16) >> 3;  // first activation chunk of this thread
#pragma unroll
      for (int jc = 0; jc < C::CH_PER_T; ++jc) {
        uint4 xb[NB];
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          const int m = nb * 8 + g;
          if (m < M && kin) {
            xb[nb] = *reinterpret_cast<const uint4*>(smem + (size_t)m * rs + C::swz(cbase + jc) * 16);
          } else {
            xb[nb] = make_uint4(0, 0, 0, 0);
          }
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const int j = 2 * jc + half;                  // MMA index inside the step
          const uint32_t a[4] = {h0[2 * j], h1[2 * j], h0[2 * j + 1], h1[2 * j + 1]};
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const uint32_t b0 = half ? xb[nb].z : xb[nb].x;
            const uint32_t b1 = half ? xb[nb].w : xb[nb].y;
            mma_16816(d[nb], a, b0, b1);
          }
        }
      }
    }
  }

  // ---- reduce the warps' K shares, then the epilogue ----
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[((warp * NB + nb) * 4 + i) * 32 + lane] = d[nb][i];
  __syncthreads();
  if (warp < NB) {
    const int nb = warp;
    float acc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float sacc = 0.0f;
#pragma unroll
      for (int ww = 0; ww < GEMV_WARPS; ++ww) sacc += red[((ww * NB + nb) * 4 + i) * 32 + lane];
      acc[i] = sacc;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int n = n0 + g + (i >= 2 ? 8 : 0);
      const int m = nb * 8 + 2 * t + (i & 1);
      if (m >= M) continue;
      const size_t o = (size_t)m * N + n;
      if (epi == EPI_I32) {
        static_cast<int32_t*>(out)[o] = __float2int_rn(acc[i]);
      } else {
        float v = __fmul_rn(acc[i], __half2float(col_scale[n]));
        if (epi == EPI_F16_ROWCOL) v = __fmul_rn(v, __half2float(row_scale[m]));
        static_cast<__half*>(out)[o] = __float2half_rn(v);
      }
    }
  }
}

template <int BBITS, int ACT, int NB, bool INTER>
cudaError_t launch_t(const GemmArgs& g, cudaStream_t stream) {
  using C = GemvCfg<BBITS>;
  const size_t smem = (size_t)g.M * (2 * g.K + C::PAD) + (size_t)GEMV_WARPS * NB * 4 * 32 * sizeof(float);
  auto kern = gemv_mma_kernel<BBITS, ACT, NB, INTER, 4>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)(g.N / 16), GEMV_WARPS * 32, smem, stream>>>(
      g.a, static_cast<const uint8_t*>(g.b), (int)g.M, (int)g.N, (int)g.K,
      reinterpret_cast<const __half*>(g.row_scale), reinterpret_cast<const __half*>(g.col_scale), g.epi, g.c);
  return cudaGetLastError();
}

template <int BBITS, int ACT>
cudaError_t launch_bits_act(const GemmArgs& g, cudaStream_t stream) {
  const bool inter = g.layout == BQ_LAYOUT_INTERLEAVED;
  if (g.M <= 8) return inter ? launch_t<BBITS, ACT, 1, true>(g, stream) : launch_t<BBITS, ACT, 1, false>(g, stream);
  return inter ? launch_t<BBITS, ACT, 2, true>(g, stream) : launch_t<BBITS, ACT, 2, false>(g, stream);
}

}  // namespace

cudaError_t launch_gemv_mma(const GemmArgs& g, cudaStream_t stream) {
  if (g.M < 1 || g.M > 16) return cudaErrorInvalidValue;
  if (g.bbits == 4) {
    return g.act == ACT_F16 ? launch_bits_act<4, ACT_F16>(g, stream) : launch_bits_act<4, ACT_I8>(g, stream);
  }
  if (g.bbits == 2) {
    return g.act == ACT_F16 ? launch_bits_act<2, ACT_F16>(g, stream) : launch_bits_act<2, ACT_I8>(g, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bq
