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
  static constexpr int CPT = E16 / 8;                 // 8-value activation chunks per thread per step
  static constexpr int PAD = BBITS == 4 ? 16 : 64;    // staged fp16 activation row pad (bytes)
  // Position of 16-byte chunk j (0 <= j < CPT) of quad thread t inside one
  // step of a staged fp16 row.  The XOR depends only on t, so every thread
  // precomputes its offsets once; with the row pad, the 8 threads of a
  // quarter warp (2 rows x 4 quad threads) hit 8 different bank groups.
  __device__ __forceinline__ static int chunk_pos(int t, int j) {
    const int c = t * CPT + j;
    return BBITS == 4 ? (c ^ ((t >> 1) << 1)) : (c ^ t);
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

// UNS: unsigned 4-bit codes u, converted as u - 8 (top bits flipped).
template <int BBITS, bool INTER, bool UNS = false>
__device__ __forceinline__ void convert_word(uint32_t w, uint32_t (&h)[GemvCfg<BBITS>::PW]) {
  if constexpr (BBITS == 4) {
    if constexpr (UNS) w ^= 0x88888888u;
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
  const int actfn = epi >> 4;
  epi &= 15;
  __shared__ float red[GEMV_WARPS][NB][4][32];
  extern __shared__ __align__(16) uint8_t xs[];       // M staged activation rows, then 16 zero bytes
  const int rs = gemv_row_stride<BBITS, ACT>(K);
  // 16 zero bytes after the rows, 16-byte aligned (int8 rows have an 8-byte stride)
  uint8_t* const zero_chunk = xs + (((size_t)M * rs + 15) & ~(size_t)15);

  // ---- stage the activations asynchronously (they are small and L2 resident) ----
  const int chunks_per_row = K >> 3;
  if constexpr (ACT == ACT_F16) {
    for (int idx = threadIdx.x; idx < M * chunks_per_row; idx += blockDim.x) {
      const int m = idx / chunks_per_row, c = idx - m * chunks_per_row;
      const int sstep = c / (C::STEP / 8), cin = c - sstep * (C::STEP / 8);   // step, chunk within the step
      const int pos = C::chunk_pos(cin / C::CPT, cin % C::CPT);
      cp_async_16(xs + (size_t)m * rs + (size_t)sstep * (C::STEP * 2) + pos * 16,
                  static_cast<const __half*>(act) + (size_t)m * K + 8 * c);
    }
  } else {
    for (int idx = threadIdx.x; idx < M * chunks_per_row; idx += blockDim.x) {
      const int m = idx / chunks_per_row, c = idx - m * chunks_per_row;
      cp_async_8(xs + (size_t)m * rs + 8 * c, static_cast<const int8_t*>(act) + (size_t)m * K + 8 * c);
    }
  }
  if (threadIdx.x == 0) *reinterpret_cast<uint4*>(zero_chunk) = make_uint4(0, 0, 0, 0);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int n0 = blockIdx.x * 16;
  const size_t row_bytes = (size_t)K * BBITS / 8;
  const uint8_t* w0 = w + (size_t)(n0 + g) * row_bytes + 16 * t;
  const uint8_t* w1 = w0 + 8 * row_bytes;
  const int nsteps = (K + C::STEP - 1) / C::STEP;
  const int s_begin = (warp * nsteps) / GEMV_WARPS;
  const int s_end = ((warp + 1) * nsteps) / GEMV_WARPS;

  // Per-thread activation fragment addressing: rows past M read the zero chunk.
  const uint8_t* xrow[NB];
  uint32_t xmask[NB];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int m = nb * 8 + g;
    xrow[nb] = m < M ? xs + (size_t)m * rs : zero_chunk;
    xmask[nb] = m < M ? 0xffffffffu : 0u;
  }
  uint32_t xoff[C::CPT];        // byte offset of chunk j of this thread inside a step
#pragma unroll
  for (int j = 0; j < C::CPT; ++j)
    xoff[j] = ACT == ACT_F16 ? (uint32_t)(C::chunk_pos(t, j) * 16) : (uint32_t)((t * C::CPT + j) * 8);
  constexpr uint32_t STEP_BYTES = ACT == ACT_F16 ? C::STEP * 2 : C::STEP;

  // Two independent accumulator chains per output block (even / odd words).
  float d[2][NB][4];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) d[a][nb][i] = 0.0f;

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
      // a ragged last step: threads past K hold zero codes and read the zero
      // chunk (mma.sync needs the whole warp)
      const bool kin = (s * C::STEP + t * C::E16) < K;
      const uint32_t sbase = (uint32_t)s * STEP_BYTES;
      const uint32_t wa[4] = {v0[u].x, v0[u].y, v0[u].z, v0[u].w};
      const uint32_t wb[4] = {v1[u].x, v1[u].y, v1[u].z, v1[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t ha[C::PW], hb[C::PW];
        convert_word<BBITS, INTER>(wa[i], ha);
        convert_word<BBITS, INTER>(wb[i], hb);
#pragma unroll
        for (int c = 0; c < C::PW / 4; ++c) {
          const int j = i * (C::PW / 4) + c;                  // chunk of this thread in the step
          uint4 xb[NB];
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            const uint8_t* p = kin ? xrow[nb] + ((sbase + xoff[j]) & xmask[nb]) : zero_chunk;
            if constexpr (ACT == ACT_F16) {
              xb[nb] = *reinterpret_cast<const uint4*>(p);
            } else {
              const uint2 raw = *reinterpret_cast<const uint2*>(p);
              cvt_i8x4_f16(raw.x, xb[nb].x, xb[nb].y);
              cvt_i8x4_f16(raw.y, xb[nb].z, xb[nb].w);
            }
          }
#pragma unroll
          for (int nb = 0; nb < NB; ++nb) {
            float (&dd)[4] = d[i & 1][nb];
            mma_16816(dd, ha[4 * c + 0], hb[4 * c + 0], ha[4 * c + 1], hb[4 * c + 1], xb[nb].x, xb[nb].y);
            mma_16816(dd, ha[4 * c + 2], hb[4 * c + 2], ha[4 * c + 3], hb[4 * c + 3], xb[nb].z, xb[nb].w);
          }
        }
      }
    }
  }

  // ---- reduce the chains and the warps' K shares, then the epilogue ----
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[warp][nb][i][lane] = d[0][nb][i] + d[1][nb][i];
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
        v = apply_act(v, actfn);
        static_cast<__half*>(out)[o] = __float2half_rn(v);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Bulk-copy variant (the common case: 16 rows of packed weights fit in shared
// memory).  Each warp owns a quarter of K and an mbarrier: its lane 0 arms
// the barrier with the byte count and lanes 0-15 each issue one
// cp.async.bulk of that quarter of one weight row, so the block keeps ~32 KB
// in flight without holding registers and every warp starts as soon as its
// own quarter has landed.  The activations (at most 16 rows) are read as
// MMA fragments straight from global memory (L1 resident) at the start of
// each step, so they never queue behind the weight stream.  The kernel
// supports programmatic dependent launch: the weights (read-only) are
// requested before griddepcontrol.wait, the activations are read and the
// outputs written only after it, so a chain of layer GEMVs streams the next
// layer's weights while the previous one finishes.
// ---------------------------------------------------------------------------
constexpr int WROW_PAD = 64;     // bytes between staged weight rows

template <int BBITS>
__host__ __device__ constexpr int gemv_bulk_smem(int K) {
  return 16 * (K * BBITS / 8 + WROW_PAD);
}

// Activation bytes of all M rows (staged in shared memory when at most GEMV_XS_MAX).
template <int ACT>
constexpr int gemv_x_bytes(int64_t M, int64_t K) {
  return (int)(M * K * (ACT == ACT_F16 ? 2 : 1));
}

// Largest activation block (all M rows) staged in shared memory next to the
// weights; beyond it the activations are read from global memory.
constexpr int GEMV_XS_MAX = 8 * 1024;

// 8 activation values (k0 .. k0+7) of one row (row pointer xr, in shared
// memory when XS, else global) as 4 fp16x2 words.
// A lane with live == false loads nothing and returns zeros (the conversion
// runs unpredicated, so the branch covers only the load).
template <int ACT, bool XS>
__device__ __forceinline__ uint4 load_x8(const uint8_t* xr, int k0, bool live) {
  if constexpr (ACT == ACT_F16) {
    if (!live) return make_uint4(0, 0, 0, 0);
    if constexpr (XS) return *reinterpret_cast<const uint4*>(xr + 2 * k0);
    return __ldg(reinterpret_cast<const uint4*>(xr + 2 * k0));
  } else {
    uint2 raw = make_uint2(0, 0);
    if (live) raw = XS ? *reinterpret_cast<const uint2*>(xr + k0) : __ldg(reinterpret_cast<const uint2*>(xr + k0));
    uint4 v;
    cvt_i8x4_f16(raw.x, v.x, v.y);
    cvt_i8x4_f16(raw.y, v.z, v.w);
    return v;
  }
}

// FULL: K is a multiple of the step, so no thread ever reaches past K.
// XS: the activations (M * K elements, at most GEMV_XS_MAX bytes) are staged
// in shared memory after the weights: each warp copies its K range of every
// row once (one bulk copy per row), instead of every warp of every SM
// re-reading the same few L2 lines at each step.
// ZP (fp16 x 4-bit): unsigned weight codes with a per-column zero point; the
// epilogue adds (8 - zero_point[n]) * row_sum[m] before the column scale.
// Every block forms the row sums itself: beside each product MMA, one with an
// all-ones A fragment sums the same activation fragment over k into fp32
// (every row of that accumulator holds the sums); the block adds the warps'
// shares in warp order, the same in every block, and block 0 also writes
// them to row_sum.
template <int BBITS, int ACT, int NB, bool INTER, bool FULL, bool XS, bool ZP = false>
__global__ void __launch_bounds__(GEMV_WARPS * 32) gemv_bulk_kernel(const void* __restrict__ act,
                                                                    const uint8_t* __restrict__ w, int M, int N, int K,
                                                                    const __half* __restrict__ row_scale,
                                                                    const __half* __restrict__ col_scale,
                                                                    const __half* __restrict__ zero_point,
                                                                    float* __restrict__ row_sum, int epi,
                                                                    void* __restrict__ out, uint64_t timeout_ns,
                                                                    int* status) {
  static_assert(!ZP || (BBITS == 4 && ACT == ACT_F16), "zero points are for fp16 x 4-bit");
  using C = GemvCfg<BBITS>;
  const int actfn = epi >> 4;
  epi &= 15;
  __shared__ float red[GEMV_WARPS][NB][4][32];
  __shared__ float rs_part[ZP ? GEMV_WARPS : 1][ZP ? NB * 8 : 1];   // ZP: the warps' shares of the row sums
  __shared__ __align__(8) uint64_t wbar[GEMV_WARPS];
  __shared__ __align__(8) uint64_t xbar[GEMV_WARPS];
  extern __shared__ __align__(16) uint8_t wsm[];         // 16 staged weight rows, then (XS) the activations
  constexpr int XB = ACT == ACT_F16 ? 2 : 1;             // activation bytes per element
  const int rb = K * BBITS / 8;                          // packed bytes per weight row
  const int ws = rb + WROW_PAD;
  const int n0 = blockIdx.x * 16;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nsteps = (K + C::STEP - 1) / C::STEP;
  const int s_begin = (warp * nsteps) / GEMV_WARPS;
  const int s_end = ((warp + 1) * nsteps) / GEMV_WARPS;
  constexpr int STEP_W = C::STEP * BBITS / 8;            // packed bytes of one step (64)
  const int seg_off = s_begin * STEP_W;
  const int seg = min((s_end - s_begin) * STEP_W, rb - seg_off);   // this warp's bytes per row

  // this warp's activation bytes of each row: [x0, x1)
  const int x0 = s_begin * C::STEP * XB, x1 = min(s_end * C::STEP, K) * XB;
  uint8_t* const xsm = wsm + 16 * ws;

  if (lane == 0) {
    mbar_init(&wbar[warp], 1);
    if (XS) mbar_init(&xbar[warp], 1);
    mbar_fence_init();
  }
  __syncwarp();
  // ---- weights first (read-only, independent of any earlier kernel) ----
  if (seg > 0) {
    if (lane == 0) mbar_arrive_expect_tx(&wbar[warp], 16u * (uint32_t)seg);
    __syncwarp();
    if (lane < 16)
      bulk_load(wsm + lane * ws + seg_off, w + (size_t)(n0 + lane) * rb + seg_off, (uint32_t)seg, &wbar[warp]);
  }
  // let a dependent kernel start its own weight prefetch; then wait for the
  // kernel that produced the activations before reading them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (XS && x1 > x0) {
    if (lane == 0) mbar_arrive_expect_tx(&xbar[warp], (uint32_t)(M * (x1 - x0)));
    __syncwarp();
    if (lane < M)
      bulk_load(xsm + (size_t)lane * K * XB + x0, static_cast<const uint8_t*>(act) + (size_t)lane * K * XB + x0,
                (uint32_t)(x1 - x0), &xbar[warp]);
  }

  // Each warp waits for its own quarter; on a timeout it still waits
  // (bounded) for its copies before it may exit, and skips the math.
  bool w_ok = true;
  if (seg > 0) {
    w_ok = mbar_wait(&wbar[warp], 0, timeout_ns, status);
    if (!w_ok) mbar_wait(&wbar[warp], 0, 4000000000ull, status);
  }
  if (XS && x1 > x0) {
    const bool x_ok = mbar_wait(&xbar[warp], 0, timeout_ns, status);
    if (!x_ok) mbar_wait(&xbar[warp], 0, 4000000000ull, status);
    w_ok = w_ok && x_ok;
  }
  w_ok = __all_sync(0xffffffffu, w_ok);

  const int g = lane >> 2, t = lane & 3;
  const int s_stop = w_ok ? s_end : s_begin;
  const uint8_t* wr0 = wsm + g * ws + 16 * t;
  const uint8_t* wr1 = wr0 + 8 * ws;
  // Activation row of each MMA column.  Lanes whose column is past M load
  // nothing and feed zeros (those columns are never stored): with M = 1 only
  // the 4 lanes of column 0 read activations, so a fragment load moves 64
  // bytes through the shared-memory / L1 data path instead of 512.
  const uint8_t* xr[NB];
  bool xv[NB];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int m = nb * 8 + g;
    xv[nb] = m < M;
    xr[nb] = (XS ? xsm : static_cast<const uint8_t*>(act)) + (size_t)(m < M ? m : 0) * K * XB;
  }

  float d[2][NB][4];
#pragma unroll
  for (int a = 0; a < 2; ++a)
#pragma unroll
    for (int nb = 0; nb < NB; ++nb)
#pragma unroll
      for (int i = 0; i < 4; ++i) d[a][nb][i] = 0.0f;
  float dz[ZP ? NB : 1][4];   // ZP: sums of the activations over this warp's k
#pragma unroll
  for (int nb = 0; nb < (ZP ? NB : 1); ++nb)
#pragma unroll
    for (int i = 0; i < 4; ++i) dz[nb][i] = 0.0f;
  constexpr uint32_t ONES = 0x3C003C00u;   // two fp16 ones

#pragma unroll 2
  for (int s = s_begin; s < s_stop; ++s) {
    const int kbase = s * C::STEP + t * C::E16;          // first k of this thread's 16 bytes
    // a ragged last step: threads past K read zero weights and activations
    // of the warp's own first step (staged, finite); ZP: zero activations,
    // which the row sums also take
    const bool kin = FULL || kbase < K;
    const int kx = kin ? kbase : s_begin * C::STEP;
    // activation fragments first, overlapping the conversion
    uint4 xb[C::CPT][NB];
#pragma unroll
    for (int j = 0; j < C::CPT; ++j)
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) xb[j][nb] = load_x8<ACT, XS>(xr[nb], kx + 8 * j, xv[nb] && (!ZP || kin));
    const uint32_t woff = (uint32_t)s * STEP_W;
    uint4 va = *reinterpret_cast<const uint4*>(wr0 + (kin ? woff : 0));
    uint4 vb = *reinterpret_cast<const uint4*>(wr1 + (kin ? woff : 0));
    if (!FULL && !kin) {
      va = make_uint4(0, 0, 0, 0);
      vb = make_uint4(0, 0, 0, 0);
    }
    const uint32_t wa[4] = {va.x, va.y, va.z, va.w};
    const uint32_t wb[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t ha[C::PW], hb[C::PW];
      convert_word<BBITS, INTER, ZP>(wa[i], ha);
      convert_word<BBITS, INTER, ZP>(wb[i], hb);
#pragma unroll
      for (int c = 0; c < C::PW / 4; ++c) {
        const int j = i * (C::PW / 4) + c;
#pragma unroll
        for (int nb = 0; nb < NB; ++nb) {
          float (&dd)[4] = d[i & 1][nb];
          mma_16816(dd, ha[4 * c + 0], hb[4 * c + 0], ha[4 * c + 1], hb[4 * c + 1], xb[j][nb].x, xb[j][nb].y);
          mma_16816(dd, ha[4 * c + 2], hb[4 * c + 2], ha[4 * c + 3], hb[4 * c + 3], xb[j][nb].z, xb[j][nb].w);
          if constexpr (ZP) {
            mma_16816(dz[nb], ONES, ONES, ONES, ONES, xb[j][nb].x, xb[j][nb].y);
            mma_16816(dz[nb], ONES, ONES, ONES, ONES, xb[j][nb].z, xb[j][nb].w);
          }
        }
      }
    }
  }

  if constexpr (ZP) {
    // accumulator row g = 0 (lanes 0..3): columns m = 8 nb + 2 t and 8 nb + 2 t + 1
    if (g == 0) {
#pragma unroll
      for (int nb = 0; nb < NB; ++nb) {
        rs_part[warp][nb * 8 + 2 * t] = dz[nb][0];
        rs_part[warp][nb * 8 + 2 * t + 1] = dz[nb][1];
      }
    }
  }
#pragma unroll
  for (int nb = 0; nb < NB; ++nb)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[warp][nb][i][lane] = d[0][nb][i] + d[1][nb][i];
  const bool ok = __syncthreads_and(w_ok ? 1 : 0) != 0;
  if constexpr (ZP) {
    if (blockIdx.x == 0 && (int)threadIdx.x < M) {
      float r = 0.0f;
#pragma unroll
      for (int ww = 0; ww < GEMV_WARPS; ++ww) r = __fadd_rn(r, rs_part[ww][threadIdx.x]);
      row_sum[threadIdx.x] = r;
    }
  }
  if (warp < NB && ok) {
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
        if constexpr (ZP) {
          float r = 0.0f;
#pragma unroll
          for (int ww = 0; ww < GEMV_WARPS; ++ww) r = __fadd_rn(r, rs_part[ww][m]);
          acc = __fmaf_rn(__fsub_rn(8.0f, __half2float(zero_point[n])), r, acc);
        }
        float v = __fmul_rn(acc, __half2float(col_scale[n]));
        if (epi == EPI_F16_ROWCOL) v = __fmul_rn(v, __half2float(row_scale[m]));
        v = apply_act(v, actfn);
        static_cast<__half*>(out)[o] = __float2half_rn(v);
      }
    }
  }
}

template <int BBITS, int ACT, int NB, bool INTER, bool FULL, bool XS, bool ZP = false>
cudaError_t launch_bulk(const GemmArgs& g, cudaStream_t stream) {
  int* status = nullptr;
  cudaError_t e = device_status_ptr(&status);
  if (e != cudaSuccess) return e;
  const int smem = gemv_bulk_smem<BBITS>((int)g.K) + (XS ? gemv_x_bytes<ACT>(g.M, g.K) : 0);
  auto kern = gemv_bulk_kernel<BBITS, ACT, NB, INTER, FULL, XS, ZP>;
  if (smem > 48 * 1024) {
    e = set_smem_once(kern, smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(g.N / 16));
  cfg.blockDim = dim3(GEMV_WARPS * 32);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const void* a = g.a;
  const uint8_t* b = static_cast<const uint8_t*>(g.b);
  int M = (int)g.M, N = (int)g.N, K = (int)g.K;
  const __half* rsc = reinterpret_cast<const __half*>(g.row_scale);
  const __half* csc = reinterpret_cast<const __half*>(g.col_scale);
  int epi = epi_arg(g);
  void* c = g.c;
  uint64_t to = (uint64_t)wait_timeout_ns();
  const __half* zp = reinterpret_cast<const __half*>(g.zero_point);
  float* rsum = const_cast<float*>(g.row_sum);   // ZP: written by block 0
  e = cudaLaunchKernelEx(&cfg, kern, a, b, M, N, K, rsc, csc, zp, rsum, epi, c, to, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BBITS, int ACT, int NB, bool INTER>
cudaError_t launch_t(const GemmArgs& g, cudaStream_t stream) {
  const int smem = (((int)g.M * gemv_row_stride<BBITS, ACT>((int)g.K) + 15) & ~15) + 16;
  auto kern = gemv_mma_kernel<BBITS, ACT, NB, INTER>;
  if (smem > 48 * 1024) {
    cudaError_t e = set_smem_once(kern, smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)(g.N / 16), GEMV_WARPS * 32, smem, stream>>>(
      g.a, static_cast<const uint8_t*>(g.b), (int)g.M, (int)g.N, (int)g.K,
      reinterpret_cast<const __half*>(g.row_scale), reinterpret_cast<const __half*>(g.col_scale), epi_arg(g), g.c);
  return cudaGetLastError();
}

// fp16 x unsigned 4-bit with zero points: the bulk variant only (gemv_zp_fits)
cudaError_t launch_bulk_zp(const GemmArgs& g, cudaStream_t stream) {
  const bool inter = g.layout == BQ_LAYOUT_INTERLEAVED;
  const bool full = g.K % GemvCfg<4>::STEP == 0;
  if (g.M <= 8 && gemv_x_bytes<ACT_F16>(g.M, g.K) <= GEMV_XS_MAX) {   // activations staged in shared memory
    if (full) return inter ? launch_bulk<4, ACT_F16, 1, true, true, true, true>(g, stream)
                           : launch_bulk<4, ACT_F16, 1, false, true, true, true>(g, stream);
    return inter ? launch_bulk<4, ACT_F16, 1, true, false, true, true>(g, stream)
                 : launch_bulk<4, ACT_F16, 1, false, false, true, true>(g, stream);
  }
  if (g.M <= 8) {
    if (full) return inter ? launch_bulk<4, ACT_F16, 1, true, true, false, true>(g, stream)
                           : launch_bulk<4, ACT_F16, 1, false, true, false, true>(g, stream);
    return inter ? launch_bulk<4, ACT_F16, 1, true, false, false, true>(g, stream)
                 : launch_bulk<4, ACT_F16, 1, false, false, false, true>(g, stream);
  }
  if (full) return inter ? launch_bulk<4, ACT_F16, 2, true, true, false, true>(g, stream)
                         : launch_bulk<4, ACT_F16, 2, false, true, false, true>(g, stream);
  return inter ? launch_bulk<4, ACT_F16, 2, true, false, false, true>(g, stream)
               : launch_bulk<4, ACT_F16, 2, false, false, false, true>(g, stream);
}

template <int BBITS, int ACT>
cudaError_t launch_bits_act(const GemmArgs& g, cudaStream_t stream) {
  const bool inter = g.layout == BQ_LAYOUT_INTERLEAVED;
  if (gemv_bulk_smem<BBITS>((int)g.K) <= 64 * 1024) {
    const bool full = g.K % GemvCfg<BBITS>::STEP == 0;
    if (g.M <= 8 && gemv_x_bytes<ACT>(g.M, g.K) <= GEMV_XS_MAX) {
      if (full)
        return inter ? launch_bulk<BBITS, ACT, 1, true, true, true>(g, stream)
                     : launch_bulk<BBITS, ACT, 1, false, true, true>(g, stream);
      return inter ? launch_bulk<BBITS, ACT, 1, true, false, true>(g, stream)
                   : launch_bulk<BBITS, ACT, 1, false, false, true>(g, stream);
    }
    if (g.M <= 8) {
      if (full)
        return inter ? launch_bulk<BBITS, ACT, 1, true, true, false>(g, stream)
                     : launch_bulk<BBITS, ACT, 1, false, true, false>(g, stream);
      return inter ? launch_bulk<BBITS, ACT, 1, true, false, false>(g, stream)
                   : launch_bulk<BBITS, ACT, 1, false, false, false>(g, stream);
    }
    if (full)
      return inter ? launch_bulk<BBITS, ACT, 2, true, true, false>(g, stream)
                   : launch_bulk<BBITS, ACT, 2, false, true, false>(g, stream);
    return inter ? launch_bulk<BBITS, ACT, 2, true, false, false>(g, stream)
                 : launch_bulk<BBITS, ACT, 2, false, false, false>(g, stream);
  }
  if (g.M <= 8) return inter ? launch_t<BBITS, ACT, 1, true>(g, stream) : launch_t<BBITS, ACT, 1, false>(g, stream);
  return inter ? launch_t<BBITS, ACT, 2, true>(g, stream) : launch_t<BBITS, ACT, 2, false>(g, stream);
}

}  // namespace

bool gemv_fits(int64_t M, int64_t K, int bbits) {
  const int64_t bytes = M * (2 * K + (bbits == 4 ? 16 : 64)) + 32;
  return M >= 1 && M <= 16 && bytes <= 200 * 1024;
}

bool gemv_zp_fits(int64_t M, int64_t K) {
  return M >= 1 && M <= 16 && gemv_bulk_smem<4>((int)K) <= 64 * 1024;
}

cudaError_t launch_gemv_mma(const GemmArgs& g, cudaStream_t stream) {
  if (g.zero_point) {
    if (g.act != ACT_F16 || g.bbits != 4 || !gemv_zp_fits(g.M, g.K)) return cudaErrorInvalidValue;
    return launch_bulk_zp(g, stream);
  }
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
