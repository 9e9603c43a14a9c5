// Tensor-core GEMM for the quantised linear (larger M), sm_103a.
//
// C[i, j] = sum_k A[i, k] * B[j, k] with A = activations (int8 or fp16,
// (M, K) row-major) and B = weights (int8 or packed 4-/2-bit codes, (N, K)),
// followed by the fused epilogue (int32 store, or the fp16 dequantisation
// with per-column and optional per-row scales).  The forms are those of the
// BitBLAS guide ("BitBLAS自定义操作开发指南", 混合精度算子开发实战 1 and 2,
// 实际应用案例 案例1 and 案例2) and the BMINF linear ("BMINF的後訓練量化實現",
// 實現代碼分析2: igemm then elementwise_copy_scale).
//
// sm_103a has no integer tcgen05 MMA, so every operand is converted exactly to
// fp16 (int8, int4 and int2 values are fp16 integers) and multiplied with
// tcgen05.mma kind::f16 into an fp32 accumulator in tensor memory.  Integer
// products are exact and every partial sum is an integer; while those stay
// below 2**24 the fp32 accumulation is exact too (the host guarantees that for
// the int32 paths by bounding K, or by splitting K into separately
// accumulated slices that are summed as integers in the epilogue).
//
// CTA organisation (one 128 x BN output tile per CTA):
//   warps 0-7  converters: 16-byte global loads of the raw A / B k-blocks into
//              registers (PF k-blocks ahead), exact conversion to fp16, stores
//              into a STAGES-deep ring of 128-byte-swizzled K-major tiles;
//              afterwards the epilogue (TMEM -> registers -> global).
//   warp 8     allocates tensor memory; lane 0 issues the MMAs (4 per 64-wide
//              k-block) and commits each stage back to the converters.
// Every mbarrier wait is bounded in time; a wait that gives up records
// BQ_ERR_TIMEOUT, the CTA abandons the tile, waits (bounded) for MMAs it
// issued, frees tensor memory and exits.
#include <cuda_fp16.h>

#include "bq_device.cuh"
#include "bq_internal.h"

namespace bq {

// First error recorded by a bounded wait of this kernel (BQ_OK if none).
__device__ int g_tc_status = 0;

cudaError_t device_status_ptr(int** out) {
  // The address differs per device; look it up on the current one.
  static int* cached[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!cached[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_tc_status);
    if (e != cudaSuccess) return e;
    cached[dev] = static_cast<int*>(p);
  }
  *out = cached[dev];
  return cudaSuccess;
}

cudaError_t read_device_status(int* status_out, bool reset) {
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return e;
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_tc_status, sizeof(int));
  if (e != cudaSuccess) return e;
  if (reset && v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int));
    if (e != cudaSuccess) return e;
  }
  *status_out = v;
  return cudaSuccess;
}

namespace {

constexpr int BM = 128;
constexpr int BK = 64;               // fp16 elements per 128-byte swizzle row
constexpr int CONV_WARPS = 8;
constexpr int CONV_THREADS = CONV_WARPS * 32;
constexpr int TC_THREADS = CONV_THREADS + 32;
constexpr uint64_t DRAIN_TIMEOUT_NS = 4000000000ull;

template <int ACT, int BBITS, int BN, int NACC, bool INTER, int STAGES>
struct TcCfg {
  static constexpr int A_ROW_BYTES = ACT == ACT_F16 ? BK * 2 : BK;      // raw bytes per A row per k-block
  static constexpr int B_ROW_BYTES = BK * BBITS / 8;                     // raw bytes per B row per k-block
  static constexpr int A_PIECES_ROW = A_ROW_BYTES / 16;
  static constexpr int B_PIECES_ROW = B_ROW_BYTES / 16;
  static constexpr int A_PIECES = BM * A_PIECES_ROW;
  static constexpr int B_PIECES = BN * B_PIECES_ROW;
  static constexpr int NPA = (A_PIECES + CONV_THREADS - 1) / CONV_THREADS;
  static constexpr int NPB = (B_PIECES + CONV_THREADS - 1) / CONV_THREADS;
  static constexpr int A_TILE = BM * 128;                                // fp16 tile bytes
  static constexpr int B_TILE = BN * 128;
  static constexpr int STAGE_BYTES = A_TILE + B_TILE;
  static constexpr int NCOLS = NACC * BN;                                // TMEM columns
  static constexpr int PF = 3;                                           // register prefetch depth
  static constexpr size_t SMEM = (size_t)STAGES * STAGE_BYTES + 1024 + 256;
  static_assert(NCOLS <= 512 && (NCOLS & (NCOLS - 1)) == 0, "TMEM columns must be a power of two <= 512");
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN");
};

struct RawPiece {
  uint4 v;
};

// Store one 16-byte fp16 chunk (logical chunk lc, 8 k values) of row r into a
// 128B-swizzled K-major tile.
__device__ __forceinline__ void st_chunk(uint8_t* tile, int r, int lc, uint4 v) {
  *reinterpret_cast<uint4*>(tile + r * 128 + ((lc ^ (r & 7)) << 4)) = v;
}

template <int ACT, int BBITS, int BN, int NACC, bool INTER, int STAGES>
__global__ void __launch_bounds__(TC_THREADS, 1)
    gemm_tc_kernel(const void* __restrict__ a_ptr, const uint8_t* __restrict__ b_ptr, int M, int N, int K,
                   const __half* __restrict__ row_scale, const __half* __restrict__ col_scale, int epi,
                   void* __restrict__ out, uint64_t timeout_ns, int* status) {
  using C = TcCfg<ACT, BBITS, BN, NACC, INTER, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* accum_bar = empty_bar + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum_bar + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.y * BM;
  const int n0 = blockIdx.x * BN;
  const int nkb = K / BK;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], CONV_THREADS);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(accum_bar, 1);
    mbar_fence_init();
  }
  if (warp == CONV_WARPS) {
    tmem_alloc(tmem_slot, C::NCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < CONV_WARPS) {
    // ------------------------------------------------------------------ converters
    const int c = tid;
    const size_t a_row_stride = (size_t)K * (ACT == ACT_F16 ? 2 : 1);
    const size_t b_row_stride = (size_t)K * BBITS / 8;
    const uint8_t* a_bytes = static_cast<const uint8_t*>(a_ptr);

    RawPiece ra[C::PF][C::NPA], rb[C::PF][C::NPB];

    auto load_kb = [&](int kb, RawPiece (&pa)[C::NPA], RawPiece (&pb)[C::NPB]) {
#pragma unroll
      for (int i = 0; i < C::NPA; ++i) {
        const int pi = c + i * CONV_THREADS;
        const int r = pi / C::A_PIECES_ROW, sub = pi % C::A_PIECES_ROW;
        if (pi < C::A_PIECES && m0 + r < M) {
          pa[i].v = __ldg(reinterpret_cast<const uint4*>(a_bytes + (size_t)(m0 + r) * a_row_stride +
                                                          (size_t)kb * C::A_ROW_BYTES + sub * 16));
        } else {
          pa[i].v = make_uint4(0, 0, 0, 0);
        }
      }
#pragma unroll
      for (int i = 0; i < C::NPB; ++i) {
        const int pi = c + i * CONV_THREADS;
        const int r = pi / C::B_PIECES_ROW, sub = pi % C::B_PIECES_ROW;
        if (pi < C::B_PIECES && n0 + r < N) {
          pb[i].v = __ldg(reinterpret_cast<const uint4*>(b_ptr + (size_t)(n0 + r) * b_row_stride +
                                                          (size_t)kb * C::B_ROW_BYTES + sub * 16));
        } else {
          // zero codes: 0 for int8, and a zero word converts to zero for 4 / 2 bits
          pb[i].v = make_uint4(0, 0, 0, 0);
        }
      }
    };

    auto store_kb = [&](uint8_t* stage, const RawPiece (&pa)[C::NPA], const RawPiece (&pb)[C::NPB]) {
      uint8_t* ta = stage;
      uint8_t* tb = stage + C::A_TILE;
#pragma unroll
      for (int i = 0; i < C::NPA; ++i) {
        const int pi = c + i * CONV_THREADS;
        if (pi >= C::A_PIECES) continue;
        const int r = pi / C::A_PIECES_ROW, sub = pi % C::A_PIECES_ROW;
        if constexpr (ACT == ACT_F16) {
          st_chunk(ta, r, sub, pa[i].v);
        } else {
          uint4 o0, o1;
          cvt_i8x4_f16(pa[i].v.x, o0.x, o0.y);
          cvt_i8x4_f16(pa[i].v.y, o0.z, o0.w);
          cvt_i8x4_f16(pa[i].v.z, o1.x, o1.y);
          cvt_i8x4_f16(pa[i].v.w, o1.z, o1.w);
          st_chunk(ta, r, 2 * sub, o0);
          st_chunk(ta, r, 2 * sub + 1, o1);
        }
      }
#pragma unroll
      for (int i = 0; i < C::NPB; ++i) {
        const int pi = c + i * CONV_THREADS;
        if (pi >= C::B_PIECES) continue;
        const int r = pi / C::B_PIECES_ROW, sub = pi % C::B_PIECES_ROW;
        const uint32_t wv[4] = {pb[i].v.x, pb[i].v.y, pb[i].v.z, pb[i].v.w};
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
    };

#pragma unroll
    for (int p = 0; p < C::PF; ++p)
      if (p < nkb) load_kb(p, ra[p], rb[p]);

    bool ok = true;
    for (int kb0 = 0; kb0 < nkb && ok; kb0 += C::PF) {
#pragma unroll
      for (int p = 0; p < C::PF; ++p) {
        const int kb = kb0 + p;
        if (kb < nkb && ok) {
          const int s = kb % STAGES;
          const uint32_t par = ((kb / STAGES) & 1) ^ 1;
          const bool w_ok = mbar_wait(&empty_bar[s], par, timeout_ns, status);
          if (!__all_sync(0xffffffffu, w_ok)) {
            ok = false;
          } else {
            store_kb(smem + s * C::STAGE_BYTES, ra[p], rb[p]);
            fence_proxy_async_smem();
            mbar_arrive(&full_bar[s]);
            if (kb + C::PF < nkb) load_kb(kb + C::PF, ra[p], rb[p]);
          }
        }
      }
    }

    // ------------------------------------------------------------------ epilogue
    const bool acc_ok = __all_sync(0xffffffffu, mbar_wait(accum_bar, 0, ok ? timeout_ns : 0, status));
    tc_fence_after();
    if (acc_ok) {
      const int q = warp & 3;                 // TMEM lane quadrant of this warp
      const int chalf = warp >> 2;            // column half
      const int row = m0 + 32 * q + lane;
      const bool row_ok = row < M;
      float rsc = 1.0f;
      if (epi == EPI_F16_ROWCOL && row_ok) rsc = __half2float(row_scale[row]);
#pragma unroll 1
      for (int cc = 0; cc < BN / 64; ++cc) {
        const int col = chalf * (BN / 2) + cc * 32;
        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)col;
        uint32_t r[32];
        float v[32];
        int iv[32];
#pragma unroll
        for (int a = 0; a < NACC; ++a) {
          tmem_ld_32x32b_x32(taddr + a * BN, r);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float f = __uint_as_float(r[i]);
            if (a == 0) {
              v[i] = f;
              iv[i] = __float2int_rn(f);
            } else {
              v[i] += f;
              iv[i] += __float2int_rn(f);
            }
          }
        }
        const int ncol = n0 + col;
        if (row_ok && ncol < N) {
          if (epi == EPI_I32) {
            int4* dst = reinterpret_cast<int4*>(static_cast<int32_t*>(out) + (size_t)row * N + ncol);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_int4(iv[4 * i], iv[4 * i + 1], iv[4 * i + 2], iv[4 * i + 3]);
          } else {
            uint32_t hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float x0 = __fmul_rn(v[2 * i], __half2float(col_scale[ncol + 2 * i]));
              float x1 = __fmul_rn(v[2 * i + 1], __half2float(col_scale[ncol + 2 * i + 1]));
              if (epi == EPI_F16_ROWCOL) {
                x0 = __fmul_rn(x0, rsc);
                x1 = __fmul_rn(x1, rsc);
              }
              const __half2 h2 = __halves2half2(__float2half_rn(x0), __float2half_rn(x1));
              hv[i] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(out) + (size_t)row * N + ncol);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(BM, BN);
      const uint32_t smem_base = smem_u32(smem);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % STAGES;
        if (!mbar_wait(&full_bar[s], (kb / STAGES) & 1, timeout_ns, status)) break;
        tc_fence_after();
        const int slice = (int)(((long long)kb * NACC) / nkb);
        const bool first = kb == 0 || slice != (int)(((long long)(kb - 1) * NACC) / nkb);
        const uint32_t d = tmem + (uint32_t)(slice * BN);
        const uint32_t sa = smem_base + s * C::STAGE_BYTES;
        const uint64_t adesc = smem_desc_sw128(sa);
        const uint64_t bdesc = smem_desc_sw128(sa + C::A_TILE);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // +32 bytes along K per 16-element step = +2 in the descriptor's address field
          tc_mma_f16(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, (first && kk == 0) ? 0u : 1u);
        }
        tc_commit(&empty_bar[s]);
      }
      tc_commit(accum_bar);
      // make sure no MMA is still in flight before the tensor memory is freed
      mbar_wait(accum_bar, 0, DRAIN_TIMEOUT_NS, status);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == CONV_WARPS) {
    tc_fence_after();
    tmem_dealloc(tmem, C::NCOLS);
  }
}

// ---------------------------------------------------------------------------
// Variant with the int8 activations in tensor memory ("TA").  Converting A
// into shared memory costs a store and an MMA read of every A element; here
// 4 warps (one thread per tile row, which is exactly the TMEM lane that row
// occupies) convert their row's 64 codes of a k-block to 32 fp16 pairs and
// write them with tcgen05.st into a TMEM stage; the MMA reads A from TMEM
// (the [a_tmem] operand form) and only B passes through shared memory.
//   warps 0-3   A converters (TMEM writers)
//   warps 4-11  B converters (swizzled shared-memory tiles), then the epilogue
//   warp 12     tensor-memory allocation and the MMA issuer (lane 0)
// ---------------------------------------------------------------------------
constexpr int TA_A_WARPS = 4;
constexpr int TA_B_WARPS = 8;
constexpr int TA_B_THREADS = TA_B_WARPS * 32;
constexpr int TA_THREADS = (TA_A_WARPS + TA_B_WARPS + 1) * 32;

template <int BBITS, int BN, int STAGES>
struct TaCfg {
  static constexpr int B_ROW_BYTES = BK * BBITS / 8;
  static constexpr int B_PIECES_ROW = B_ROW_BYTES / 16;
  static constexpr int B_PIECES = BN * B_PIECES_ROW;
  static constexpr int NPB = (B_PIECES + TA_B_THREADS - 1) / TA_B_THREADS;
  static constexpr int B_TILE = BN * 128;
  static constexpr int A_COLS = BK / 2;                    // TMEM columns per A stage
  static constexpr int NCOLS = 512;
  static constexpr int PF = 4;
  static constexpr size_t SMEM = (size_t)STAGES * B_TILE + 1024 + 256;
  static_assert(BN + STAGES * A_COLS <= NCOLS, "TMEM budget");
};

template <int BBITS, int BN, bool INTER, int STAGES>
__global__ void __launch_bounds__(TA_THREADS, 1)
    gemm_tc_ta_kernel(const int8_t* __restrict__ a_ptr, const uint8_t* __restrict__ b_ptr, int M, int N, int K,
                      const __half* __restrict__ row_scale, const __half* __restrict__ col_scale, int epi,
                      void* __restrict__ out, uint64_t timeout_ns, int* status) {
  using C = TaCfg<BBITS, BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + STAGES * C::B_TILE);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* accum_bar = empty_bar + STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum_bar + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.y * BM;
  const int n0 = blockIdx.x * BN;
  const int nkb = K / BK;
  constexpr int MMA_WARP = TA_A_WARPS + TA_B_WARPS;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full_bar[s], TA_A_WARPS * 32 + TA_B_THREADS);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(accum_bar, 1);
    mbar_fence_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(tmem_slot, C::NCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < TA_A_WARPS) {
    // ------------------------------------------------------------ A -> TMEM
    const int row = m0 + warp * 32 + lane;
    const bool row_ok = row < M;
    const uint4* arow = reinterpret_cast<const uint4*>(a_ptr + (size_t)(row_ok ? row : 0) * K);
    uint4 ra[C::PF][4];
    auto load_a = [&](int kb, uint4 (&v)[4]) {
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = row_ok ? __ldg(arow + kb * 4 + j) : make_uint4(0, 0, 0, 0);
    };
#pragma unroll
    for (int p = 0; p < C::PF; ++p)
      if (p < nkb) load_a(p, ra[p]);
    bool ok = true;
    for (int kb0 = 0; kb0 < nkb && ok; kb0 += C::PF) {
#pragma unroll
      for (int p = 0; p < C::PF; ++p) {
        const int kb = kb0 + p;
        if (kb < nkb && ok) {
          uint32_t h[32];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            cvt_i8x4_f16(ra[p][j].x, h[8 * j + 0], h[8 * j + 1]);
            cvt_i8x4_f16(ra[p][j].y, h[8 * j + 2], h[8 * j + 3]);
            cvt_i8x4_f16(ra[p][j].z, h[8 * j + 4], h[8 * j + 5]);
            cvt_i8x4_f16(ra[p][j].w, h[8 * j + 6], h[8 * j + 7]);
          }
          if (kb + C::PF < nkb) load_a(kb + C::PF, ra[p]);
          const int s = kb % STAGES;
          const bool w_ok = mbar_wait(&empty_bar[s], ((kb / STAGES) & 1) ^ 1, timeout_ns, status);
          if (!__all_sync(0xffffffffu, w_ok)) {
            ok = false;
          } else {
            tmem_st_32x32b_x32(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(BN + s * C::A_COLS), h);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&full_bar[s]);
          }
        }
      }
    }
  } else if (warp < MMA_WARP) {
    // ------------------------------------------------------------ B -> smem
    const int c = tid - TA_A_WARPS * 32;
    const size_t b_row_stride = (size_t)K * BBITS / 8;
    uint4 rb[C::PF][C::NPB];
    auto load_b = [&](int kb, uint4 (&v)[C::NPB]) {
#pragma unroll
      for (int i = 0; i < C::NPB; ++i) {
        const int pi = c + i * TA_B_THREADS;
        const int r = pi / C::B_PIECES_ROW, sub = pi % C::B_PIECES_ROW;
        v[i] = (pi < C::B_PIECES && n0 + r < N)
                   ? __ldg(reinterpret_cast<const uint4*>(b_ptr + (size_t)(n0 + r) * b_row_stride +
                                                          (size_t)kb * C::B_ROW_BYTES + sub * 16))
                   : make_uint4(0, 0, 0, 0);
      }
    };
    auto store_b = [&](uint8_t* tb, const uint4 (&v)[C::NPB]) {
#pragma unroll
      for (int i = 0; i < C::NPB; ++i) {
        const int pi = c + i * TA_B_THREADS;
        if (pi >= C::B_PIECES) continue;
        const int r = pi / C::B_PIECES_ROW, sub = pi % C::B_PIECES_ROW;
        const uint32_t wv[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
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
    };
#pragma unroll
    for (int p = 0; p < C::PF; ++p)
      if (p < nkb) load_b(p, rb[p]);
    bool ok = true;
    for (int kb0 = 0; kb0 < nkb && ok; kb0 += C::PF) {
#pragma unroll
      for (int p = 0; p < C::PF; ++p) {
        const int kb = kb0 + p;
        if (kb < nkb && ok) {
          const int s = kb % STAGES;
          const bool w_ok = mbar_wait(&empty_bar[s], ((kb / STAGES) & 1) ^ 1, timeout_ns, status);
          if (!__all_sync(0xffffffffu, w_ok)) {
            ok = false;
          } else {
            store_b(smem + s * C::B_TILE, rb[p]);
            fence_proxy_async_smem();
            mbar_arrive(&full_bar[s]);
            if (kb + C::PF < nkb) load_b(kb + C::PF, rb[p]);
          }
        }
      }
    }

    // ------------------------------------------------------------ epilogue
    const bool acc_ok = __all_sync(0xffffffffu, mbar_wait(accum_bar, 0, ok ? timeout_ns : 0, status));
    tc_fence_after();
    if (acc_ok) {
      const int q = warp & 3;                       // TMEM lane quadrant of this warp
      const int chalf = (warp - TA_A_WARPS) >> 2;   // column half
      const int row = m0 + 32 * q + lane;
      const bool row_ok = row < M;
      float rsc = 1.0f;
      if (epi == EPI_F16_ROWCOL && row_ok) rsc = __half2float(row_scale[row]);
#pragma unroll 1
      for (int cc = 0; cc < BN / 64; ++cc) {
        const int col = chalf * (BN / 2) + cc * 32;
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)col, r);
        tmem_ld_wait();
        const int ncol = n0 + col;
        if (row_ok && ncol < N) {
          if (epi == EPI_I32) {
            int4* dst = reinterpret_cast<int4*>(static_cast<int32_t*>(out) + (size_t)row * N + ncol);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_int4(__float2int_rn(__uint_as_float(r[4 * i])), __float2int_rn(__uint_as_float(r[4 * i + 1])),
                                 __float2int_rn(__uint_as_float(r[4 * i + 2])),
                                 __float2int_rn(__uint_as_float(r[4 * i + 3])));
          } else {
            uint32_t hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float x0 = __fmul_rn(__uint_as_float(r[2 * i]), __half2float(col_scale[ncol + 2 * i]));
              float x1 = __fmul_rn(__uint_as_float(r[2 * i + 1]), __half2float(col_scale[ncol + 2 * i + 1]));
              if (epi == EPI_F16_ROWCOL) {
                x0 = __fmul_rn(x0, rsc);
                x1 = __fmul_rn(x1, rsc);
              }
              const __half2 h2 = __halves2half2(__float2half_rn(x0), __float2half_rn(x1));
              hv[i] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(out) + (size_t)row * N + ncol);
#pragma unroll
            for (int i = 0; i < 4; ++i) dst[i] = make_uint4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(BM, BN);
      const uint32_t smem_base = smem_u32(smem);
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % STAGES;
        if (!mbar_wait(&full_bar[s], (kb / STAGES) & 1, timeout_ns, status)) break;
        tc_fence_after();
        const uint64_t bdesc = smem_desc_sw128(smem_base + s * C::B_TILE);
        const uint32_t a_tm = tmem + (uint32_t)(BN + s * C::A_COLS);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // 16 k = 8 TMEM columns of A; 32 bytes along K in the swizzled B tile
          tc_mma_f16_ts(tmem, a_tm + 8 * kk, bdesc + 2 * kk, idesc, (kb == 0 && kk == 0) ? 0u : 1u);
        }
        tc_commit(&empty_bar[s]);
      }
      tc_commit(accum_bar);
      mbar_wait(accum_bar, 0, DRAIN_TIMEOUT_NS, status);
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::NCOLS);
  }
}

template <int BBITS, int BN, bool INTER>
cudaError_t launch_ta(const GemmArgs& g, cudaStream_t stream) {
  constexpr int STAGES = 4;
  using C = TaCfg<BBITS, BN, STAGES>;
  int* status = nullptr;
  cudaError_t se = device_status_ptr(&status);
  if (se != cudaSuccess) return se;
  auto kern = gemm_tc_ta_kernel<BBITS, BN, INTER, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((g.N + BN - 1) / BN), (unsigned)((g.M + BM - 1) / BM));
  kern<<<grid, TA_THREADS, C::SMEM, stream>>>(static_cast<const int8_t*>(g.a), static_cast<const uint8_t*>(g.b),
                                              (int)g.M, (int)g.N, (int)g.K,
                                              reinterpret_cast<const __half*>(g.row_scale),
                                              reinterpret_cast<const __half*>(g.col_scale), g.epi, g.c,
                                              (uint64_t)wait_timeout_ns(), status);
  return cudaGetLastError();
}

template <int BBITS, int BN>
cudaError_t launch_ta_layout(const GemmArgs& g, cudaStream_t stream) {
  if (BBITS != 8 && g.layout == BQ_LAYOUT_PLAIN) return launch_ta<BBITS, BN, false>(g, stream);
  return launch_ta<BBITS, BN, true>(g, stream);
}

template <int ACT, int BBITS, int BN, int NACC, bool INTER>
cudaError_t launch_t(const GemmArgs& g, cudaStream_t stream) {
  constexpr int STAGES = 4;
  int* status = nullptr;
  cudaError_t se = device_status_ptr(&status);
  if (se != cudaSuccess) return se;
  using C = TcCfg<ACT, BBITS, BN, NACC, INTER, STAGES>;
  auto kern = gemm_tc_kernel<ACT, BBITS, BN, NACC, INTER, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((g.N + BN - 1) / BN), (unsigned)((g.M + BM - 1) / BM));
  kern<<<grid, TC_THREADS, C::SMEM, stream>>>(g.a, static_cast<const uint8_t*>(g.b), (int)g.M, (int)g.N, (int)g.K,
                                              reinterpret_cast<const __half*>(g.row_scale),
                                              reinterpret_cast<const __half*>(g.col_scale), g.epi, g.c,
                                              (uint64_t)wait_timeout_ns(), status);
  return cudaGetLastError();
}

template <int ACT, int BBITS, int BN, int NACC>
cudaError_t launch_layout(const GemmArgs& g, cudaStream_t stream) {
  if (BBITS != 8 && g.layout == BQ_LAYOUT_PLAIN) return launch_t<ACT, BBITS, BN, NACC, false>(g, stream);
  return launch_t<ACT, BBITS, BN, NACC, true>(g, stream);
}

}  // namespace

cudaError_t launch_gemm_tc(const GemmArgs& g, cudaStream_t stream) {
  const int nkb = (int)(g.K / BK);
  if (g.act == ACT_I8 && g.bbits == 8) {
    // int32 output: slices of at most 1024 k keep every partial sum < 2**24 exactly
    if (g.epi == EPI_I32) {
      if (nkb <= 16) return launch_layout<ACT_I8, 8, 256, 1>(g, stream);
      if (nkb <= 32) return launch_layout<ACT_I8, 8, 256, 2>(g, stream);
      if (nkb <= 64) return launch_layout<ACT_I8, 8, 128, 4>(g, stream);
      return cudaErrorInvalidValue;
    }
    return launch_ta_layout<8, 256>(g, stream);
  }
  // int8 activations with 4- / 2-bit weights: every partial sum < 2**24 (host-bounded K)
  if (g.act == ACT_I8 && g.bbits == 4) return launch_ta_layout<4, 256>(g, stream);
  if (g.act == ACT_I8 && g.bbits == 2) return launch_ta_layout<2, 256>(g, stream);
  // fp16 activations: the accumulator is not an exact integer, so K is split
  // into two separately accumulated halves (shorter fp32 accumulation chains
  // in the tensor core), summed in fp32 in the epilogue.
  if (g.act == ACT_F16 && g.bbits == 4) {
    if (nkb >= 2) return launch_layout<ACT_F16, 4, 256, 2>(g, stream);
    return launch_layout<ACT_F16, 4, 256, 1>(g, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bq
