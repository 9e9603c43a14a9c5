// Tensor-core GEMM for small M with the weights as the MMA's A operand
// (tcgen05, sm_103a): D[n, m] = sum_k W[n, k] * X[m, k], stored as Y[m, n].
//
// The forms are those of the BitBLAS guide ("BitBLAS自定义操作开发指南",
// 混合精度算子开发实战 2 and 实际应用案例 案例2: fp16 activations times 4-bit
// (or 2-bit) weights, fp32 accumulation, per-output-channel scale) at the
// small, dynamic M of decoding.
//
// With M activation rows (M <= 128) a weight-by-activation product is a
// 128 x MN x 64 MMA per k-block, MN = M rounded up to 16, so the tensor core
// is nearly idle and the cost is streaming and converting the weights.  Each
// CTA owns 128 weight rows (the MMA's M = the TMEM lanes) and all of K:
//   producer warps  one thread: TMA of the raw packed weight rows into a
//                   ring of RKB k-blocks per stage, as far ahead as the ring
//                   allows and from before griddepcontrol.wait, so a chain of
//                   layers streams the next layer's weights early; another
//                   (after griddepcontrol.wait): TMA of each k-block's fp16
//                   activation tile (MN rows, 128B swizzle, the MMA's B
//                   operand) into a ring of its own.
//   converter groups of 4 warps take the k-blocks in turn: thread = weight
//                   row = TMEM lane; its 64 codes become 32 fp16 pairs in
//                   registers and go to a TMEM stage with tcgen05.st, so the
//                   weights never pass through shared memory as fp16.
//   MMA warp        one elected lane issues tcgen05.mma (A from TMEM, B from
//                   shared memory) into a 128 x MN fp32 accumulator.
// Epilogue (converter group 0): tcgen05.ld, scale, and for each activation
// row m a store of the 32 consecutive outputs of a warp (coalesced).
// Every wait is bounded in time; a wait that gives up records
// BQ_ERR_TIMEOUT and the CTA abandons the tile.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "bq_device.cuh"
#include "bq_internal.h"
#include "gemm_common.cuh"

namespace bq {
namespace {

constexpr int SW_N = 128;                // weight rows per CTA (TMEM lanes)
constexpr int SW_K = 64;                 // k per block
constexpr int SW_NG = 2;                 // converter groups (4 warps each)
constexpr uint64_t SW_DRAIN_NS = 4000000000ull;
// M range served here: below it the skinny kernel streams the weights faster
// (bulk copies of whole row segments), above it the CTA-pair kernel
constexpr int64_t SWAP_MIN_M = 16;
constexpr int64_t SWAP_MAX_M = 128;

template <int BBITS, int MN>
struct SwapCfg {
  static constexpr int CONV_WARPS = 4 * SW_NG;
  static constexpr int MMA_WARP = CONV_WARPS;
  static constexpr int PRODUCER_WARP = MMA_WARP + 1;          // weights
  static constexpr int X_WARP = PRODUCER_WARP + 1;             // activations
  static constexpr int THREADS = (X_WARP + 1) * 32;
  static constexpr int RKB = 4;                                // k-blocks per raw weight stage
  static constexpr int RST = 3;                                // raw weight stages
  static constexpr int W_ROW = SW_K * BBITS / 8;               // packed bytes per row per k-block
  static constexpr int W_BOX_X = RKB * W_ROW;                  // 128 (4-bit) or 64 (2-bit) bytes
  static constexpr int W_RAW = SW_N * W_BOX_X;
  static constexpr int X_TILE = MN * 128;                      // fp16 activation tile (64 k per row)
  // activation stages: their own ring, deep enough to hide the load latency
  static constexpr int SX = 32768 / X_TILE >= 16 ? 16 : (32768 / X_TILE >= 4 ? 32768 / X_TILE : 4);
  static constexpr int A_COLS = SW_K / 2;                      // TMEM columns of one weight stage
  // Two accumulator slices (the two halves of K, summed in the epilogue:
  // shorter fp32 chains) and, in the remaining columns, the TMEM weight
  // stages.  The MMAs per k-block are tiny, so the ring spans the whole
  // latency from a converter's tcgen05.st to the commit that frees a stage.
  // 256 columns (two CTAs per SM) up to MN = 64, else 512.
  static constexpr int NCOLS = 2 * MN + 4 * A_COLS <= 256 ? 256 : 512;
  static constexpr int ST = (NCOLS - 2 * MN) / A_COLS > 8 ? 8 : (NCOLS - 2 * MN) / A_COLS;
  static constexpr int OFF_X = RST * W_RAW;
  static constexpr int OFF_BAR = OFF_X + SX * X_TILE;
  static constexpr size_t SMEM = (size_t)OFF_BAR + 512 + 1024;
  static_assert(MN % 16 == 0 && MN >= 16 && MN <= 128, "MMA N");
  static_assert(W_RAW % 1024 == 0 && X_TILE % 1024 == 0, "stage alignment");
  static_assert(SW_NG <= ST, "converter groups per stage ring");
  static_assert(SMEM <= 232448, "shared memory");
};

// ZP (4-bit): unsigned weight codes with a per-column zero point; the
// epilogue adds (8 - zero_point[n]) * row_sum[m] before the column scale.
template <int BBITS, int MN, bool INTER, bool ZP = false>
__global__ void __launch_bounds__(SwapCfg<BBITS, MN>::THREADS, 1)
    gemm_swap_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_x, int M,
                     int N, int K, const __half* __restrict__ row_scale, const __half* __restrict__ col_scale,
                     const __half* __restrict__ zero_point, const float* __restrict__ row_sum, int epi,
                     void* __restrict__ out, uint64_t timeout_ns, int* status) {
  using C = SwapCfg<BBITS, MN>;
  static_assert(!ZP || BBITS == 4, "zero points are for 4-bit weights");
  constexpr uint32_t FLIP = ZP ? 0x88888888u : 0u;   // unsigned codes u -> two's-complement u - 8
  const int actfn = epi >> 4;
  epi &= 15;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);   // TMEM weight stage written
  uint64_t* empty_bar = full_bar + C::ST;                                 // MMAs done with a TMEM weight stage
  uint64_t* rfull_bar = empty_bar + C::ST;                               // raw weight stage landed
  uint64_t* rempty_bar = rfull_bar + C::RST;                             // raw weight stage read
  uint64_t* xfull_bar = rempty_bar + C::RST;                             // activation stage landed
  uint64_t* xempty_bar = xfull_bar + C::SX;                              // MMAs done with an activation stage
  uint64_t* accum_bar = xempty_bar + C::SX;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum_bar + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * SW_N;
  const int nkb = K / SW_K;
  const uint32_t rzero = (uint32_t)K >> 30;   // 0 (K <= 65536), not known to the compiler
  // k-blocks [0, kb_half) accumulate into slice 0, the rest into slice 1
  const int kb_half = nkb >= 2 ? (nkb + 1) / 2 : nkb;
  const bool two_slices = kb_half < nkb;

  if (tid == 0) {
    for (int s = 0; s < C::ST; ++s) {
      mbar_init(&full_bar[s], 4);   // one converter group, one arrival per warp
      mbar_init(&empty_bar[s], 1);
    }
    for (int s = 0; s < C::SX; ++s) {
      mbar_init(&xfull_bar[s], 1);
      mbar_init(&xempty_bar[s], 1);
    }
    for (int s = 0; s < C::RST; ++s) {
      mbar_init(&rfull_bar[s], 1);
      mbar_init(&rempty_bar[s], (SW_NG < C::RKB ? SW_NG : C::RKB) * 4 * 32);
    }
    mbar_init(accum_bar, 1);
    mbar_fence_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(tmem_slot, C::NCOLS);
    tmem_relinquish();
  }
  if (warp == C::PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tmap_w);
    tma_prefetch_desc(&tmap_x);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == C::PRODUCER_WARP || warp == C::X_WARP) {
    // ------------------------------------------------------------ TMA producers (one warp each, so
    // neither waits behind the other's polling)
    if (warp == C::PRODUCER_WARP && lane == 0) {
      // raw weights: read-only, independent of any earlier kernel; as far
      // ahead as the raw ring allows
      const int nrg = (nkb + C::RKB - 1) / C::RKB;
      int wg = 0;
      for (; wg < nrg; ++wg) {
        const int rs = wg % C::RST;
        if (wg >= C::RST && !mbar_wait(&rempty_bar[rs], ((wg / C::RST) & 1) ^ 1, timeout_ns, status)) break;
        mbar_arrive_expect_tx(&rfull_bar[rs], C::W_RAW);
        tma_load_2d(smem + rs * C::W_RAW, &tmap_w, wg * C::W_BOX_X, n0, &rfull_bar[rs]);
        if (wg + 1 == C::RST || wg + 1 == nrg) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
      }
      // no TMA write may land after the CTA has exited
      for (int g = wg > C::RST ? wg - C::RST : 0; g < wg; ++g)
        mbar_wait(&rfull_bar[g % C::RST], (g / C::RST) & 1, SW_DRAIN_NS, status);
    } else if (warp == C::X_WARP && lane == 0) {
      // activations: written by the kernel before this one
      asm volatile("griddepcontrol.wait;" ::: "memory");
      int kb = 0;
      for (; kb < nkb; ++kb) {
        const int sx = kb % C::SX;
        if (!mbar_wait(&xempty_bar[sx], ((kb / C::SX) & 1) ^ 1, timeout_ns, status)) break;
        mbar_arrive_expect_tx(&xfull_bar[sx], C::X_TILE);
        tma_load_2d(smem + C::OFF_X + sx * C::X_TILE, &tmap_x, kb * SW_K, 0, &xfull_bar[sx]);
      }
      for (int k2 = kb > C::SX ? kb - C::SX : 0; k2 < kb; ++k2)
        mbar_wait(&xfull_bar[k2 % C::SX], (k2 / C::SX) & 1, SW_DRAIN_NS, status);
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
    const uint32_t smem_base = __shfl_sync(0xffffffffu, smem_u32(smem), 0);
    const uint32_t idesc = idesc_f16_f32(SW_N, MN);
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % C::ST, sx = kb % C::SX;
      if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[s], (kb / C::ST) & 1, timeout_ns, status) &&
                                       mbar_wait(&xfull_bar[sx], (kb / C::SX) & 1, timeout_ns, status)))
        break;
      tc_fence_after();
      const uint32_t a_tm = tm + (uint32_t)(2 * MN + s * C::A_COLS);
      const bool second = kb >= kb_half;
      const uint32_t d = tm + (second ? (uint32_t)MN : 0u);
      const uint64_t bdesc = smem_desc_sw128(smem_base + C::OFF_X + sx * C::X_TILE);
      if (elect_one()) {
#pragma unroll
        for (int kk = 0; kk < SW_K / 16; ++kk)
          tc_mma_f16_ts(d, a_tm + 8 * kk, bdesc + 2 * kk, idesc, ((kb != 0 && kb != kb_half) || kk > 0) ? 1u : 0u);
        tc_commit(&empty_bar[s]);
        tc_commit(&xempty_bar[sx]);
      }
      __syncwarp();
    }
    if (elect_one()) tc_commit(accum_bar);
    __syncwarp();
    mbar_wait(accum_bar, 0, SW_DRAIN_NS, status);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ weights -> TMEM (and the epilogue)
    const int q = warp & 3;                               // TMEM lane quadrant
    const int r = q * 32 + lane;                          // weight row in the tile == TMEM lane
    const int grp = warp >> 2;
    bool ok = true;
    for (int kb = grp; kb < nkb; kb += SW_NG) {
      const int wg = kb / C::RKB, rs = wg % C::RST;
      if (kb % C::RKB < SW_NG && !warp_wait(&rfull_bar[rs], (wg / C::RST) & 1, timeout_ns, status)) {
        ok = false;
        break;
      }
      // this row's W_ROW bytes of k-block kb inside the swizzled raw box row
      const uint8_t* rowp = smem + rs * C::W_RAW + r * C::W_BOX_X;
      uint32_t h[32];
      if constexpr (BBITS == 4) {
        const int c0 = (kb % C::RKB) * 2;                 // two 16-byte chunks of a 128-byte row
        const uint4 v0 = *reinterpret_cast<const uint4*>(rowp + ((c0 ^ (r & 7)) << 4));
        const uint4 v1 = *reinterpret_cast<const uint4*>(rowp + (((c0 + 1) ^ (r & 7)) << 4));
        if ((kb % C::RKB) + SW_NG >= C::RKB || kb + SW_NG >= nkb)
          mbar_arrive_after_loads(&rempty_bar[rs], fold4(v0) ^ fold4(v1), rzero);
        const uint32_t wv[8] = {v0.x ^ FLIP, v0.y ^ FLIP, v0.z ^ FLIP, v0.w ^ FLIP,
                                v1.x ^ FLIP, v1.y ^ FLIP, v1.z ^ FLIP, v1.w ^ FLIP};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint32_t t4[4];
          cvt_i4x8_f16(INTER ? wv[j] : plain_to_inter_i4(wv[j]), t4);
          h[4 * j] = t4[0];
          h[4 * j + 1] = t4[1];
          h[4 * j + 2] = t4[2];
          h[4 * j + 3] = t4[3];
        }
      } else {
        const int c0 = kb % C::RKB;                       // one 16-byte chunk of a 64-byte row (64B swizzle)
        const uint4 v0 = *reinterpret_cast<const uint4*>(rowp + ((c0 ^ ((r >> 1) & 3)) << 4));
        if ((kb % C::RKB) + SW_NG >= C::RKB || kb + SW_NG >= nkb)
          mbar_arrive_after_loads(&rempty_bar[rs], fold4(v0), rzero);
        const uint32_t wv[4] = {v0.x, v0.y, v0.z, v0.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint32_t t8[8];
          cvt_i2x16_f16(INTER ? wv[j] : plain_to_inter_i2(wv[j]), t8);
#pragma unroll
          for (int e = 0; e < 8; ++e) h[8 * j + e] = t8[e];
        }
      }
      const int s = kb % C::ST;
      if (!warp_wait(&empty_bar[s], ((kb / C::ST) & 1) ^ 1, timeout_ns, status)) {
        ok = false;
        break;
      }
      tc_fence_after();   // the store follows the MMAs that released the stage
      tmem_st_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(2 * MN + s * C::A_COLS), h);
      tmem_st_wait_tied(h);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full_bar[s]);
    }
    // ---------------------------------------------------------- epilogue (group 0)
    if (grp == 0) {
      const bool acc_ok = warp_wait(accum_bar, 0, ok ? timeout_ns : 0, status);
      tc_fence_after();
      const int n = n0 + r;
      if (acc_ok) {
        const float cs = (epi != EPI_I32 && n < N) ? __half2float(col_scale[n]) : 0.0f;
        const float zc = (ZP && n < N) ? __fsub_rn(8.0f, __half2float(zero_point[n])) : 0.0f;
#pragma unroll 1
        for (int c = 0; c < MN / 32 + (MN % 32 ? 1 : 0); ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(32 * c), v);
          tmem_ld_wait_tied(v);
          if (two_slices) {
            uint32_t v2[32];
            tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(MN + 32 * c), v2);
            tmem_ld_wait_tied(v2);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(v2[i]));
          }
          if (n >= N) continue;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int m = 32 * c + i;
            if (m >= M) break;
            float acc = __uint_as_float(v[i]);
            if constexpr (ZP) acc = __fmaf_rn(zc, row_sum[m], acc);
            const size_t o = (size_t)m * N + n;
            if (epi == EPI_I32) {
              static_cast<int32_t*>(out)[o] = __float2int_rn(acc);
            } else {
              float y = __fmul_rn(acc, cs);
              if (epi == EPI_F16_ROWCOL) y = __fmul_rn(y, __half2float(row_scale[m]));
              y = apply_act(y, actfn);
              static_cast<__half*>(out)[o] = __float2half_rn(y);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::NCOLS);
  }
}

template <int BBITS, int MN, bool INTER, bool ZP = false>
cudaError_t launch_swap_t(const GemmArgs& g, cudaStream_t stream) {
  using C = SwapCfg<BBITS, MN>;
  int* status = nullptr;
  cudaError_t e = device_status_ptr(&status);
  if (e != cudaSuccess) return e;
  CUtensorMap mw, mx;
  e = make_map(&mw, g.b, 1, (uint64_t)g.K * BBITS / 8, (uint64_t)g.N, C::W_BOX_X, SW_N,
               C::W_BOX_X == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
  if (e != cudaSuccess) return e;
  e = make_map(&mx, g.a, 2, (uint64_t)g.K, (uint64_t)g.M, SW_K, MN, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  auto kern = gemm_swap_kernel<BBITS, MN, INTER, ZP>;
  e = set_smem_once(kern, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((g.N + SW_N - 1) / SW_N));
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int M = (int)g.M, N = (int)g.N, K = (int)g.K;
  const __half* rsc = reinterpret_cast<const __half*>(g.row_scale);
  const __half* csc = reinterpret_cast<const __half*>(g.col_scale);
  const int epi = epi_arg(g);
  void* out = g.c;
  const uint64_t to = (uint64_t)wait_timeout_ns();
  const __half* zp = reinterpret_cast<const __half*>(g.zero_point);
  const float* rsum = g.row_sum;
  e = cudaLaunchKernelEx(&cfg, kern, mw, mx, M, N, K, rsc, csc, zp, rsum, epi, out, to, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BBITS, int MN>
cudaError_t launch_swap_layout(const GemmArgs& g, cudaStream_t stream) {
  if constexpr (BBITS == 4) {
    if (g.zero_point) {
      if (g.layout == BQ_LAYOUT_PLAIN) return launch_swap_t<4, MN, false, true>(g, stream);
      return launch_swap_t<4, MN, true, true>(g, stream);
    }
  }
  if (g.layout == BQ_LAYOUT_PLAIN) return launch_swap_t<BBITS, MN, false>(g, stream);
  return launch_swap_t<BBITS, MN, true>(g, stream);
}

template <int BBITS>
cudaError_t launch_swap_bits(const GemmArgs& g, cudaStream_t stream) {
  if (g.M <= 16) return launch_swap_layout<BBITS, 16>(g, stream);
  if (g.M <= 32) return launch_swap_layout<BBITS, 32>(g, stream);
  if (g.M <= 64) return launch_swap_layout<BBITS, 64>(g, stream);
  return launch_swap_layout<BBITS, 128>(g, stream);
}

}  // namespace

bool gemm_swap_applies(const GemmArgs& g) {
  return SWAP_ENABLED && g.act == ACT_F16 && (g.bbits == 4 || g.bbits == 2) && g.M > SWAP_MIN_M &&
         g.M <= SWAP_MAX_M && g.K >= SW_K;
}

cudaError_t launch_gemm_swap(const GemmArgs& g, cudaStream_t stream) {
  return g.bbits == 4 ? launch_swap_bits<4>(g, stream) : launch_swap_bits<2>(g, stream);
}

}  // namespace bq
