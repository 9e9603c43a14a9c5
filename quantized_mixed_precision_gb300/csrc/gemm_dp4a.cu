// int8 x int8 GEMM with exact int32 accumulation on the CUDA cores (dp4a).
//
// This is the igemm of "BMINF的後訓練量化實現" (實現代碼分析2: int8 operands,
// int32 result, alpha = 1, beta = 0) for the cases the tensor-core path
// cannot make exact: skinny M, and int32 results with K beyond the sliced
// tensor-core accumulation.  64 x 64 output tile per block, 256 threads, each
// thread 4 x 4 outputs; K advances 64 bytes at a time through shared memory
// stored k-word-major so every thread reads its four A rows and four B rows
// as one 16-byte vector each.
#include <cuda_fp16.h>

#include "bq_device.cuh"
#include "bq_internal.h"

namespace bq {

namespace {

constexpr int T = 64;   // tile edge (outputs)
constexpr int KW = 16;  // 32-bit words of K per step (64 int8)
constexpr int LDS = T + 4;

__global__ void __launch_bounds__(256) gemm_dp4a_kernel(const int8_t* __restrict__ A, const int8_t* __restrict__ B,
                                                        int M, int N, int K, const __half* __restrict__ row_scale,
                                                        const __half* __restrict__ col_scale, int epi,
                                                        void* __restrict__ out) {
  const int actfn = epi >> 4;
  epi &= 15;
  __shared__ __align__(16) int As[KW][LDS];
  __shared__ __align__(16) int Bs[KW][LDS];
  const int tid = threadIdx.x;
  const int ty = tid >> 4, tx = tid & 15;
  const int m0 = blockIdx.y * T, n0 = blockIdx.x * T;
  const int lr = tid >> 2, lq = tid & 3;  // loader: row 0..63, 16-byte quarter 0..3

  int acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0;

  for (int k0 = 0; k0 < K; k0 += 4 * KW) {
    int4 av = make_int4(0, 0, 0, 0), bv = make_int4(0, 0, 0, 0);
    if (m0 + lr < M) av = __ldg(reinterpret_cast<const int4*>(A + (size_t)(m0 + lr) * K + k0) + lq);
    if (n0 + lr < N) bv = __ldg(reinterpret_cast<const int4*>(B + (size_t)(n0 + lr) * K + k0) + lq);
    As[4 * lq + 0][lr] = av.x;
    As[4 * lq + 1][lr] = av.y;
    As[4 * lq + 2][lr] = av.z;
    As[4 * lq + 3][lr] = av.w;
    Bs[4 * lq + 0][lr] = bv.x;
    Bs[4 * lq + 1][lr] = bv.y;
    Bs[4 * lq + 2][lr] = bv.z;
    Bs[4 * lq + 3][lr] = bv.w;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < KW; ++w) {
      const int4 a4 = *reinterpret_cast<const int4*>(&As[w][4 * ty]);
      const int4 b4 = *reinterpret_cast<const int4*>(&Bs[w][4 * tx]);
      const int a[4] = {a4.x, a4.y, a4.z, a4.w};
      const int b[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = __dp4a(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + 4 * ty + i;
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + 4 * tx + j;
      if (n >= N) continue;
      const size_t o = (size_t)m * N + n;
      if (epi == EPI_I32) {
        static_cast<int32_t*>(out)[o] = acc[i][j];
      } else {
        float v = __fmul_rn(__int2float_rn(acc[i][j]), __half2float(col_scale[n]));
        if (epi == EPI_F16_ROWCOL) v = __fmul_rn(v, __half2float(row_scale[m]));
        v = apply_act(v, actfn);
        static_cast<__half*>(out)[o] = __float2half_rn(v);
      }
    }
  }
}

}  // namespace

cudaError_t launch_gemm_dp4a(const GemmArgs& g, cudaStream_t stream) {
  dim3 grid((unsigned)((g.N + T - 1) / T), (unsigned)((g.M + T - 1) / T));
  gemm_dp4a_kernel<<<grid, 256, 0, stream>>>(static_cast<const int8_t*>(g.a), static_cast<const int8_t*>(g.b),
                                              (int)g.M, (int)g.N, (int)g.K,
                                              reinterpret_cast<const __half*>(g.row_scale),
                                              reinterpret_cast<const __half*>(g.col_scale), epi_arg(g), g.c);
  return cudaGetLastError();
}

}  // namespace bq
