// Skinny-M GEMM (M <= 16): one pass over the packed weights.
//
// The work is bound by reading the weights from HBM once (the decode-step
// use of the quantised linear in "BMINF的後訓練量化實現", 實現代碼分析2, runs
// with M = batch).  A block of 4 warps owns 16 weight rows; each warp takes a
// quarter of K.  Every thread first issues all of its 16-byte weight loads
// (two rows, up to UNITS steps: ~8 KB per warp in flight).  The activations
// (at most 16 rows) are staged into shared memory with asynchronous copies
// issued before the weight loads, so they never queue behind them; int8
// activations are staged as bytes and converted exactly to fp16 when the
// MMA operand is built.  The
// codes are then turned into fp16 pairs in registers (exact) and fed straight
// into mma.sync m16n8k16 as the A fragment, so weights never touch shared
// memory.  Accumulation is fp32; for integer operands every partial sum stays
// below 2**24 (bounded on the host), so it is exact.
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

constexpr int GEMV_WARPS = 4;
constexpr int UNITS = 8;   // steps whose loads a warp keeps in flight

template <int BBITS>
struct GemvCfg {
  static constexpr int E16 = 128 / BBITS;             // codes per 16-byte load
  static constexpr int STEP = 4 * E16;                // k per step (4 threads of a quad)
  static constexpr int PW = 16 / BBITS;               // fp16 pairs per 32-bit word
  static constexpr int KW = 32 / BBITS;               // k per 32-bit word
  static constexpr int PAD = BBITS == 4 ? 16 : 64;    // staged fp16 activation row pad (bytes)
  // Chunk position inside a staged activation row.  Thread t of a quad reads
  // chunks [t * E16 / 8, (t + 1) * E16 / 8) of a step; with this swizzle and
  // the row pad the 8 threads of a quarter warp (2 rows x 4 quads) hit 8
  // different 16-byte bank groups.
  __device__ __forceinline__ static int swz(int c) {
    return BBITS == 4 ? (c ^ (((c >> 3) & 1) << 1)) : (c ^ ((c >> 3) & 7));
  }
};

// Staged activation row stride: fp16 rows with the swizzle pad, or int8 rows
// padded by 8 bytes (conflict-free 8-byte fragment loads).
template <int BBITS, int ACT>
__host__ __device__ constexpr int gemv_row_stride(int K) {
  return ACT == ACT_F16 ? 2 * K + GemvCfg<BBITS>::PAD : K + 8;
}

__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int BBITS, bool INTER>
__device__ __forceinline__ void convert_word(uint32_t w, uint32_t (&h)[GemvCfg<BBITS>::PW]) {
  if constexpr (BBITS == 4) {
    cvt_i4x8_f16(INTER ? w : plain_to_inter_i4(w), h);
  } else {
    cvt_i2x16_f16(INTER ? w : plain_to_inter_i2(w), h);
  }
}

template <int BBITS, int ACT, int NB, bool INTER>
__global__ void __launch_bounds__(GEMV_WARPS * 32, 5) gemv_mma_kernel(const void* __restrict__ act,
                                                                      const uint8_t* __restrict__ w, int M, int N,
                                                                      int K, const __half* __restrict__ row_scale,
                                                                      const __half* __restrict__ col_scale, int epi,
                                                                      void* __restrict__ out) {
  using C = GemvCfg<BBITS>;
  __shared__ float red[GEMV_WARPS][NB][4][32];
  extern __shared__ __align__(16) uint8_t xs[];       // M staged activation rows
  const int rs = gemv_row_stride<BBITS, ACT>(K);

  // ---- stage the activations asynchronously (they are small and L2 resident) ----
  if constexpr (ACT == ACT_F16) {
    const int chunks_per_row = K >> 3;                // 16-byte chunks of 8 fp16
    for (int idx = threadIdx.x; idx < M * chunks_per_row; idx += blockDim.x) {
      const int m = idx / chunks_per_row, c = idx - m * chunks_per_row;
      cp_async_16(xs + (size_t)m * rs + C::swz(c) * 16, static_cast<const __half*>(act) + (size_t)m * K + 8 * c);
    }
  } else {
    const int chunks_per_row = K >> 3;                // 8-byte chunks of 8 int8
    for (int idx = threadIdx.x; idx < M * chunks_per_row; idx += blockDim.x) {
      const int m = idx / chunks_per_row, c = idx - m * chunks_per_row;
      cp_async_8(xs + (size_t)m * rs + 8 * c, static_cast<const int8_t*>(act) + (size_t)m * K + 8 * c);
    }
  }

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int n0 = blockIdx.x * 16;
  const size_t row_bytes = (size_t)K * BBITS / 8;
  const uint8_t* w0 = w + (size_t)(n0 + g) * row_bytes + 16 * t;
  const uint8_t* w1 = w0 + 8 * row_bytes;
  const int nsteps = (K + C::STEP - 1) / C::STEP;
  const int s_begin = (warp * nsteps) / GEMV_WARPS;
  const int s_end = ((warp + 1) * nsteps) / GEMV_WARPS;

  float d[NB][4];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int i = 0; i < 4; ++i) d[nb][i] = 0.0f;

  // The first iteration always runs (every warp takes part in the staging
  // barrier, even one with no steps of its own).
  for (int s0 = s_begin, first = 1; s0 < s_end || first; s0 += UNITS, first = 0) {
    uint4 v0[UNITS], v1[UNITS];
#pragma unroll
    for (int u = 0; u < UNITS; ++u) {
      const int s = s0 + u;
      if (s < s_end && (s * C::STEP + t * C::E16) < K) {
        const size_t off = (size_t)s * (C::STEP * BBITS / 8);
        v0[u] = __ldcs(reinterpret_cast<const uint4*>(w0 + off));
        v1[u] = __ldcs(reinterpret_cast<const uint4*>(w1 + off));
      } else {
        // zero words convert to zero codes
        v0[u] = make_uint4(0, 0, 0, 0);
        v1[u] = make_uint4(0, 0, 0, 0);
      }
    }
    if (first) {
      cp_async_wait_all();
      __syncthreads();
    }
#pragma unroll
    for (int u = 0; u < UNITS; ++u) {
      const int s = s0 + u;
      if (s >= s_end) break;                                  // warp-uniform
      // a ragged last step: threads past K hold zero codes and read zero
      // activations (mma.sync needs the whole warp)
      const int kbase = s * C::STEP + t * C::E16;
      const bool kin = kbase < K;
      const uint32_t wa[4] = {v0[u].x, v0[u].y, v0[u].z, v0[u].w};
      const uint32_t wb[4] = {v1[u].x, v1[u].y, v1[u].z, v1[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t ha[C::PW], hb[C::PW];
        convert_word<BBITS, INTER>(wa[i], ha);
        convert_word<BBITS, INTER>(wb[i], hb);
#pragma unroll
        for (int c = 0; c < C::PW / 4; ++c) {
          const int chunk = (kbase >> 3) + i * (C::KW / 8) + c;
          uint4 xb[NB];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const int m = nb * 8 + g;
            if (m < M && kin) {
              if constexpr (ACT == ACT_F16) {
                xb[nb] = *reinterpret_cast<const uint4*>(xs + (size_t)m * rs + C::swz(chunk) * 16);
              } else {
                const uint2 raw = *reinterpret_cast<const uint2*>(xs + (size_t)m * rs + 8 * chunk);
                cvt_i8x4_f16(raw.x, xb[nb].x, xb[nb].y);
                cvt_i8x4_f16(raw.y, xb[nb].z, xb[nb].w);
              }
            } else {
              xb[nb] = make_uint4(0, 0, 0, 0);
            }
          }
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            mma_16816(d[nb], ha[4 * c + 0], hb[4 * c + 0], ha[4 * c + 1], hb[4 * c + 1], xb[nb].x, xb[nb].y);
            mma_16816(d[nb], ha[4 * c + 2], hb[4 * c + 2], ha[4 * c + 3], hb[4 * c + 3], xb[nb].z, xb[nb].w);
          }
        }
      }
    }
  }

  // ---- reduce the warps' K shares, then the epilogue ----
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[warp][nb][i][lane] = d[nb][i];
  __syncthreads();
  if (warp < NB) {
    const int nb = warp;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float acc = 0.0f;
#pragma unroll
      for (int ww = 0; ww < GEMV_WARPS; ++ww) acc += red[ww][nb][i][lane];
      const int n = n0 + g + (i >= 2 ? 8 : 0);
      const int m = nb * 8 + 2 * t + (i & 1);
      if (m >= M) continue;
      const size_t o = (size_t)m * N + n;
      if (epi == EPI_I32) {
        static_cast<int32_t*>(out)[o] = __float2int_rn(acc);
      } else {
        float v = __fmul_rn(acc, __half2float(col_scale[n]));
        if (epi == EPI_F16_ROWCOL) v = __fmul_rn(v, __half2float(row_scale[m]));
        static_cast<__half*>(out)[o] = __float2half_rn(v);
      }
    }
  }
}

template <int BBITS, int ACT, int NB, bool INTER>
cudaError_t launch_t(const GemmArgs& g, cudaStream_t stream) {
  const int smem = (int)g.M * gemv_row_stride<BBITS, ACT>((int)g.K);
  auto kern = gemv_mma_kernel<BBITS, ACT, NB, INTER>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
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

bool gemv_fits(int64_t M, int64_t K, int bbits) {
  const int64_t bytes = M * (2 * K + (bbits == 4 ? 16 : 64));
  return M >= 1 && M <= 16 && bytes <= 200 * 1024;
}

cudaError_t launch_gemv_mma(const GemmArgs& g, cudaStream_t stream) {
  if (!gemv_fits(g.M, g.K, g.bbits)) return cudaErrorInvalidValue;
  if (g.bbits == 4) {
    return g.act == ACT_F16 ? launch_bits_act<4, ACT_F16>(g, stream) : launch_bits_act<4, ACT_I8>(g, stream);
  }
  if (g.bbits == 2) {
    return g.act == ACT_F16 ? launch_bits_act<2, ACT_F16>(g, stream) : launch_bits_act<2, ACT_I8>(g, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bq
