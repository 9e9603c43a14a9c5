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
// below 2**24 the fp32 accumulation is exact too.  The host guarantees that
// for every integer path by bounding K, or (int8 x int8) by keeping every
// chain at most 1024 k long: separately accumulated TMEM slices, or split-K
// ranges of at most 16 k-blocks.  Slices and split-K partials of integer
// operands are rounded to int32 and summed as integers before the epilogue,
// so the fp16 dequantisation starts from the exact sum as well.  fp16
// activations accumulate in two slices (shorter fp32 chains).
//
// One 128 x BN output tile per CTA; warp roles:
//   producer warp  one thread issues 2-D TMA loads (cp.async.bulk.tensor) of
//                  the raw codes of B (and of A) into a ring of RST raw stages
//                  of RKB k-blocks each (128-byte box rows, swizzled); rows
//                  past M / N and columns past K arrive zero-filled.
//   A warps (4/group) int8 activations only: thread = tile row = TMEM lane; reads
//                  its 64 raw codes (128B-swizzled, conflict-free), converts
//                  them to 32 fp16 pairs and writes them with tcgen05.st into
//                  a TMEM stage that the MMA reads as its A operand.
//                  fp16 activations need no conversion: the producer loads
//                  them with TMA straight into the 128B-swizzled MMA layout.
//   B warps (8/group) read raw weight codes, convert them to fp16 and store the
//                  128B-swizzled K-major tile the MMA reads; after the
//                  mainloop they run the epilogue (TMEM -> registers -> HBM).
//   MMA warp       allocates tensor memory; lane 0 issues 4 MMAs per 64-wide
//                  k-block and commits each stage back to its producers.
// Every mbarrier wait is bounded in time; a wait that gives up records
// BQ_ERR_TIMEOUT, the CTA abandons the tile, waits (bounded) for the TMA
// loads and MMAs it issued, frees tensor memory and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "bq_device.cuh"
#include "bq_internal.h"
#include "gemm_common.cuh"
#include "quant_math.cuh"

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

// ---------------------------------------------------------------------------
// Host helpers shared by the tensor-core kernels: tensor maps, SM count,
// split-K choice
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D map over a row-major matrix of `rows` rows of `row_elems` elements
// (uint8, fp16 when elem == 2, int32 when elem == 4); box = box_x elements x
// box_rows rows.  Out-of-range elements read as zero and are not written.
cudaError_t make_map(CUtensorMap* map, const void* base, int elem, uint64_t row_elems, uint64_t rows, uint32_t box_x,
                     uint32_t box_rows, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {row_elems, rows};
  const cuuint64_t strides[1] = {row_elems * (uint64_t)elem};
  const cuuint32_t box[2] = {box_x, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = elem == 4   ? CU_TENSOR_MAP_DATA_TYPE_INT32
                                 : elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = fn(map, dt, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_map3(CUtensorMap* map, const void* base, int elem, uint64_t row_elems, uint64_t rows, uint64_t batch,
                      uint64_t item_stride, uint32_t box_x, uint32_t box_rows, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const uint64_t row_bytes = row_elems * (uint64_t)elem;
  if (batch <= 1) item_stride = (rows * row_bytes + 15) / 16 * 16;   // one item: any valid stride
  const cuuint64_t dims[3] = {row_elems, rows, batch < 1 ? 1 : batch};
  const cuuint64_t strides[2] = {row_bytes, item_stride};
  const cuuint32_t box[3] = {box_x, box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = elem == 4   ? CU_TENSOR_MAP_DATA_TYPE_INT32
                                 : elem == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int sm_count() {
  static int n[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (!n[dev] && cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) n[dev] = 148;
  return n[dev];
}

// Split-K factor for a grid of `tiles` output tiles of nkb k-blocks each: the
// largest of 2, 3, 4, 8 that keeps the grid within one wave (tiles x split <=
// SMs) and leaves every CTA at least 4 k-blocks; 1 if none does.
int choose_split(long long tiles, int nkb) {
  const long long sms = sm_count();
  int best = 1;
  for (int s : {2, 3, 4, 8})
    if (tiles * s <= sms && nkb >= 4 * s) best = s;
  return best;
}

namespace {

constexpr int BM = 128;
constexpr int BK = 64;                 // k per block: one 128-byte fp16 swizzle row
constexpr int B_THREADS = 256;         // one weight-converter group (8 warps) per k-block
constexpr uint64_t DRAIN_TIMEOUT_NS = 4000000000ull;

// A_I8_TMEM: int8 codes, converted into TMEM stages.  A_F16_SMEM: fp16
// values loaded straight into the MMA's shared-memory layout.  A_Q_TMEM: fp16
// values quantised per row to int8 codes (row scales given) by the same
// converters, which then store the codes into TMEM stages as with A_I8_TMEM.
// A_F16_ZP: as A_F16_SMEM, with unsigned 4-bit weight codes and a per-column
// zero point (the epilogue adds (8 - z) times the activation row sum).
enum AMode : int { A_I8_TMEM = 0, A_F16_SMEM = 1, A_Q_TMEM = 2, A_F16_ZP = 3 };

// Converter groups per CTA.
constexpr int TC_NG = 1;

// NG converter groups take the k-blocks in turn (group g converts k-blocks
// kb = g (mod NG)), so conversion of consecutive k-blocks overlaps.
template <int AMODE, int BBITS, int BN, int NACC, int ST, int RST, int NG, int MINB = 1>
struct Cfg {
  static constexpr bool A_SMEM = AMODE == A_F16_SMEM || AMODE == A_F16_ZP;   // fp16 A straight to the MMA
  static constexpr bool A_TMEM = !A_SMEM;                      // A converted into TMEM stages
  static constexpr int A_WARPS = A_TMEM ? 4 * NG : 0;
  static constexpr int B_WARPS = 8 * NG;
  static constexpr int MMA_WARP = A_WARPS + B_WARPS;
  static constexpr int PRODUCER_WARP = MMA_WARP + 1;
  static constexpr int THREADS = (PRODUCER_WARP + 1) * 32;
  // A raw stage holds RKB k-blocks, so every TMA box row is 128 bytes (64
  // for 2-bit weights): the TMA engine moves a box row by row, and narrow
  // rows waste its request rate.  Quantised fp16 activations take 128 bytes
  // per row per k-block already, and keep raw stages of 2 k-blocks.
  static constexpr int RKB = (BBITS == 8 || AMODE == A_Q_TMEM) ? 2 : 4;
  static constexpr int B_RAW_ROW = BK * BBITS / 8;            // raw weight bytes per row per k-block
  static constexpr int B_BOX_X = RKB * B_RAW_ROW;             // bytes per raw weight box row (128, 64 or 32)
  static constexpr int B_PIECES_ROW = B_RAW_ROW / 16;         // 16-byte pieces per row per k-block
  static constexpr int B_PIECES = BN * B_PIECES_ROW;
  static constexpr int NPB = (B_PIECES + B_THREADS - 1) / B_THREADS;
  static constexpr int B_RAW = BN * B_BOX_X;                  // raw weight bytes per raw stage
  static constexpr int A_BOX = BM * 128;                      // one int8 A box: 2 k-blocks x 128 rows
  static constexpr int A_KB = BM * 128;                       // one fp16 A box: 1 k-block x 128 rows
  static constexpr int A_RAW = AMODE == A_I8_TMEM   ? A_BOX * (RKB / 2)          // raw A per raw stage
                               : AMODE == A_Q_TMEM ? A_KB * RKB
                                                   : 0;
  static constexpr int A_TILE = A_SMEM ? BM * 128 : 0;        // fp16 A tile in the MMA stage
  static constexpr int B_TILE = BN * 128;
  static constexpr int STAGE = A_TILE + B_TILE;
  static constexpr int RSTAGE = (A_RAW + B_RAW + 1023) / 1024 * 1024;
  static constexpr int A_COLS = BK / 2;                        // TMEM columns of one A stage
  static constexpr int ACC_COLS = NACC * BN;
  static constexpr int USED_COLS = ACC_COLS + (A_TMEM ? ST * A_COLS : 0);
  static constexpr int NCOLS = USED_COLS <= 128 ? 128 : (USED_COLS <= 256 ? 256 : 512);
  static constexpr int OFF_RAW = ST * STAGE;
  static constexpr int OFF_BAR = OFF_RAW + RST * RSTAGE;
  static constexpr size_t SMEM = (size_t)OFF_BAR + 256 + 1024;
  static_assert(USED_COLS <= 512 / MINB, "tensor memory budget (MINB CTAs per SM)");
  static_assert(MINB * (SMEM + 1024) <= 233472 && SMEM <= 232448, "shared memory budget");
  static_assert(STAGE % 1024 == 0 && A_RAW % 1024 == 0, "stage alignment");
  static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
  static_assert((BN / (2 * NG)) % 32 == 0, "epilogue column parts are whole 32-column chunks");
};

template <int AMODE, int BBITS, int BN, int NACC, bool INTER, int ST, int RST, int NG, int MINB>
__global__ void __launch_bounds__(Cfg<AMODE, BBITS, BN, NACC, ST, RST, NG, MINB>::THREADS, MINB)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b, int M,
                   int N, int K, const __half* __restrict__ row_scale, const __half* __restrict__ col_scale,
                   const __half* __restrict__ zero_point, const float* __restrict__ row_sum, int epi,
                   void* __restrict__ out, uint64_t timeout_ns, int* status) {
  using C = Cfg<AMODE, BBITS, BN, NACC, ST, RST, NG, MINB>;
  const int actfn = epi >> 4;
  epi &= 15;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);   // MMA stage ready
  uint64_t* empty_bar = full_bar + ST;                                   // MMA stage consumed
  uint64_t* rfull_bar = empty_bar + ST;                                  // raw stage landed
  uint64_t* rempty_bar = rfull_bar + RST;                                // raw stage read
  uint64_t* accum_bar = rempty_bar + RST;
  uint64_t* ready_bar = accum_bar + 1;                                   // split-K: peers' pipelines done
  uint64_t* recv_bar = ready_bar + 1;                                    // split-K: peers' partials landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(recv_bar + 1);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.y * BM;
  const int n0 = blockIdx.x * BN;
  // Split-K: the gridDim.z CTAs of a cluster share one output tile and take
  // consecutive ranges of k-blocks; kb below counts within this CTA's range.
  const int S = gridDim.z;
  const int kb_lo = (int)(((long long)blockIdx.z * (K / BK)) / S);
  const int nkb = (int)(((long long)(blockIdx.z + 1) * (K / BK)) / S) - kb_lo;
  const uint32_t rzero = (uint32_t)K >> 30;      // 0 (K <= 65536), not known to the compiler
  // threads that consume one k-block: one A group (4 warps) and one B group (8 warps)
  constexpr int CONSUMERS = (C::A_WARPS / NG + 8) * 32;

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      // fp16 A: the producer's expect-tx arrival plus the B converters
      mbar_init(&full_bar[s], C::A_SMEM ? 1 + B_THREADS : CONSUMERS);
      mbar_init(&empty_bar[s], 1);
    }
    for (int s = 0; s < RST; ++s) {
      mbar_init(&rfull_bar[s], 1);
      mbar_init(&rempty_bar[s], CONSUMERS * NG);   // every group releases each raw stage once
    }
    mbar_init(accum_bar, 1);
    mbar_init(ready_bar, S > 1 ? S - 1 : 1);
    mbar_init(recv_bar, S * B_THREADS);
    mbar_fence_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(tmem_slot, C::NCOLS);
    tmem_relinquish();
  }
  if (warp == C::PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // peers may arrive on this CTA's barriers only once they are initialised
  if (S > 1) cluster_sync_all();

  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued_groups = 0, issued_kb = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        if (kb % C::RKB == 0) {
          // raw stage for k-blocks [kb, kb + RKB): boxes past K read as zero
          const int grp = kb / C::RKB;
          const int rs = grp % RST;
          if (!mbar_wait(&rempty_bar[rs], ((grp / RST) & 1) ^ 1, timeout_ns, status)) break;
          uint8_t* raw = smem + C::OFF_RAW + rs * C::RSTAGE;
          mbar_arrive_expect_tx(&rfull_bar[rs], C::A_RAW + C::B_RAW);
          if constexpr (AMODE == A_I8_TMEM) {
#pragma unroll
            for (int b = 0; b < C::RKB / 2; ++b)
              tma_load_2d(raw + b * C::A_BOX, &tmap_a, (kb_lo + kb + 2 * b) * BK, m0, &rfull_bar[rs]);
          } else if constexpr (AMODE == A_Q_TMEM) {
#pragma unroll
            for (int b = 0; b < C::RKB; ++b)
              tma_load_2d(raw + b * C::A_KB, &tmap_a, (kb_lo + kb + b) * BK, m0, &rfull_bar[rs]);
          }
          tma_load_2d(raw + C::A_RAW, &tmap_b, (kb_lo + kb) * C::B_RAW_ROW, n0, &rfull_bar[rs]);
          issued_groups = grp + 1;
        }
        if constexpr (C::A_SMEM) {
          const int s = kb % ST;
          if (!mbar_wait(&empty_bar[s], ((kb / ST) & 1) ^ 1, timeout_ns, status)) break;
          mbar_arrive_expect_tx(&full_bar[s], BM * BK * 2);
          tma_load_2d(smem + s * C::STAGE, &tmap_a, (kb_lo + kb) * BK, m0, &full_bar[s]);
        }
        issued_kb = kb + 1;
      }
      // no TMA write may land after the CTA has exited
      for (int grp = issued_groups > RST ? issued_groups - RST : 0; grp < issued_groups; ++grp)
        mbar_wait(&rfull_bar[grp % RST], (grp / RST) & 1, DRAIN_TIMEOUT_NS, status);
      if constexpr (C::A_SMEM) {
        for (int kb = issued_kb > ST ? issued_kb - ST : 0; kb < issued_kb; ++kb)
          mbar_wait(&full_bar[kb % ST], (kb / ST) & 1, DRAIN_TIMEOUT_NS, status);
      }
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop, so the operand addresses are warp-uniform;
    // one elected lane issues the MMAs and their commits.
    const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
    const uint32_t smem_base = __shfl_sync(0xffffffffu, smem_u32(smem), 0);
    const uint32_t idesc = idesc_f16_f32(BM, BN);
    // accumulator slice j takes the k-blocks [ceil(j nkb / NACC), ceil((j + 1) nkb / NACC))
    int slice = 0, next_b = NACC > 1 ? (nkb + NACC - 1) / NACC : nkb;
    for (int kb = 0; kb < nkb; ++kb) {
      const int s = kb % ST;
      if (!__all_sync(0xffffffffu, mbar_wait(&full_bar[s], (kb / ST) & 1, timeout_ns, status))) break;
      tc_fence_after();
      bool first = kb == 0;
      while (kb == next_b && slice + 1 < NACC) {
        ++slice;
        first = true;
        next_b = ((slice + 1) * nkb + NACC - 1) / NACC;
      }
      const uint32_t d = tm + (uint32_t)(slice * BN);
      const uint64_t bdesc = smem_desc_sw128(smem_base + s * C::STAGE + C::A_TILE);
      if (elect_one()) {
        if constexpr (C::A_SMEM) {
          const uint64_t adesc = smem_desc_sw128(smem_base + s * C::STAGE);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)   // +32 bytes along K = +2 in the address field
            tc_mma_f16(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, (first && kk == 0) ? 0u : 1u);
        } else {
          const uint32_t a_tm = tm + (uint32_t)(C::ACC_COLS + s * C::A_COLS);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)   // 16 k = 8 TMEM columns of A
            tc_mma_f16_ts(d, a_tm + 8 * kk, bdesc + 2 * kk, idesc, (first && kk == 0) ? 0u : 1u);
        }
        tc_commit(&empty_bar[s]);
      }
      __syncwarp();
    }
    if (elect_one()) tc_commit(accum_bar);
    __syncwarp();
    // no MMA may still be running when the tensor memory is freed
    mbar_wait(accum_bar, 0, DRAIN_TIMEOUT_NS, status);
    __syncwarp();
  } else if (warp < C::A_WARPS) {
    // ------------------------------------------------------------ int8 A -> TMEM
    const int q = warp & 3;                               // TMEM lane quadrant
    const int r = q * 32 + lane;                          // tile row == TMEM lane
    RowQuant rq{};
    if constexpr (AMODE == A_Q_TMEM) rq = row_quant(m0 + r < M ? __half2float(row_scale[m0 + r]) : 0.0f);
    for (int kb = warp >> 2; kb < nkb; kb += NG) {
      const int grp = kb / C::RKB, rs = grp % RST;
      if (!warp_wait(&rfull_bar[rs], (grp / RST) & 1, timeout_ns, status)) break;
      uint32_t h[32];
      if constexpr (AMODE == A_Q_TMEM) {
        // this k-block is one 128-byte box row of fp16 values (chunk c of row r at c ^ (r & 7))
        const uint8_t* box = smem + C::OFF_RAW + rs * C::RSTAGE + (kb % C::RKB) * C::A_KB + r * 128;
        quant64_f16_codes(box, r, rq, h);
        // the codes depend on every value read, so the release follows those reads
        if ((kb % C::RKB) + NG >= C::RKB || kb + NG >= nkb) {   // group's last use
          uint32_t dep = 0;
#pragma unroll
          for (int i = 0; i < 32; ++i) dep ^= h[i];
          mbar_arrive_after_loads(&rempty_bar[rs], dep, rzero);
        }
      } else {
        // this k-block is half of a 128-byte box row (128B swizzle: chunk c of row r at c ^ (r & 7))
        const uint8_t* box = smem + C::OFF_RAW + rs * C::RSTAGE + ((kb % C::RKB) >> 1) * C::A_BOX + r * 128;
        const int c0 = (kb & 1) * 4;
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = *reinterpret_cast<const uint4*>(box + (((c0 + j) ^ (r & 7)) << 4));
        if ((kb % C::RKB) + NG >= C::RKB || kb + NG >= nkb)   // group's last use
          mbar_arrive_after_loads(&rempty_bar[rs], fold4(v[0]) ^ fold4(v[1]) ^ fold4(v[2]) ^ fold4(v[3]), rzero);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          cvt_i8x4_f16(v[j].x, h[8 * j + 0], h[8 * j + 1]);
          cvt_i8x4_f16(v[j].y, h[8 * j + 2], h[8 * j + 3]);
          cvt_i8x4_f16(v[j].z, h[8 * j + 4], h[8 * j + 5]);
          cvt_i8x4_f16(v[j].w, h[8 * j + 6], h[8 * j + 7]);
        }
      }
      const int s = kb % ST;
      if (!warp_wait(&empty_bar[s], ((kb / ST) & 1) ^ 1, timeout_ns, status)) break;
      tc_fence_after();   // the store follows the MMAs that released the stage
      tmem_st_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(C::ACC_COLS + s * C::A_COLS), h);
      tmem_st_wait_tied(h);
      tc_fence_before();
      mbar_arrive(&full_bar[s]);
    }
  } else {
    // ------------------------------------------------------------ weights -> fp16 smem
    const int bw = warp - C::A_WARPS;                     // 0 .. 8 * NG - 1
    const int c = (bw & 7) * 32 + lane;                   // thread within its group
    bool ok = true;
    for (int kb = bw >> 3; kb < nkb; kb += NG) {
      const int grp = kb / C::RKB, rs = grp % RST;
      if (!warp_wait(&rfull_bar[rs], (grp / RST) & 1, timeout_ns, status)) {
        ok = false;
        break;
      }
      const uint8_t* raw = smem + C::OFF_RAW + rs * C::RSTAGE + C::A_RAW;
      // piece pi is (row pi % BN, piece pi / BN): a quarter warp reads 8 rows,
      // whose swizzled chunk positions differ (conflict-free)
      uint4 v[C::NPB];
#pragma unroll
      for (int i = 0; i < C::NPB; ++i) {
        const int pi = c + i * B_THREADS;
        const int r = pi % BN, sub = pi / BN;
        const int chunk = (kb % C::RKB) * C::B_PIECES_ROW + sub;
        const int pos = raw_chunk_pos<C::B_BOX_X>(chunk, r);
        v[i] = pi < C::B_PIECES ? *reinterpret_cast<const uint4*>(raw + r * C::B_BOX_X + (pos << 4))
                                : make_uint4(0, 0, 0, 0);
      }
      if ((kb % C::RKB) + NG >= C::RKB || kb + NG >= nkb) {   // group's last use
        uint32_t dep = 0;
#pragma unroll
        for (int i = 0; i < C::NPB; ++i) dep ^= fold4(v[i]);
        mbar_arrive_after_loads(&rempty_bar[rs], dep, rzero);
      }
      const int s = kb % ST;
      if (!warp_wait(&empty_bar[s], ((kb / ST) & 1) ^ 1, timeout_ns, status)) {
        ok = false;
        break;
      }
      uint8_t* tb = smem + s * C::STAGE + C::A_TILE;
#pragma unroll
      for (int i = 0; i < C::NPB; ++i) {
        const int pi = c + i * B_THREADS;
        if (pi < C::B_PIECES) convert_b_piece<BBITS, INTER, AMODE == A_F16_ZP>(tb, pi % BN, pi / BN, v[i]);
      }
      fence_proxy_async_smem();
      mbar_arrive(&full_bar[s]);
    }

    // ------------------------------------------------------------ epilogue
    // (with split-K the epilogue runs after the cluster reduction below)
    const bool acc_ok = S == 1 && warp_wait(accum_bar, 0, ok ? timeout_ns : 0, status);
    tc_fence_after();
    if (acc_ok) {
      // 2 * NG warps share each TMEM lane quadrant; each takes a column part
      const int q = warp & 3;                           // TMEM lane quadrant of this warp
      const int cpart = bw >> 2;                        // 0 .. 2 * NG - 1
      constexpr int PART = BN / (2 * NG);
      const int row = m0 + 32 * q + lane;
      const bool row_ok = row < M;
      float rsc = 1.0f;
      if (epi == EPI_F16_ROWCOL && row_ok) rsc = __half2float(row_scale[row]);
#pragma unroll 1
      for (int cc = 0; cc < PART / 32; ++cc) {
        const int col = cpart * PART + cc * 32;
        const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)col;
        uint32_t r[32];
        float v[32];
        int iv[32];
#pragma unroll
        for (int a = 0; a < NACC; ++a) {
          tmem_ld_32x32b_x32(taddr + a * BN, r);
          tmem_ld_wait_tied(r);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float f = __uint_as_float(r[i]);
            v[i] = a == 0 ? f : v[i] + f;
            iv[i] = a == 0 ? __float2int_rn(f) : iv[i] + __float2int_rn(f);
          }
        }
        const int ncol = n0 + col;
        // integer operands: the dequantisation starts from the exact integer sum of the slices
        if (C::A_TMEM && NACC > 1) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __int2float_rn(iv[i]);
        }
        if constexpr (AMODE == A_F16_ZP) {
          if (row_ok && ncol < N) add_zero_point(v, zero_point, ncol, row_sum[row]);
        }
        if (row_ok && ncol < N) {
          if (epi == EPI_I32) {
            int4* dst = reinterpret_cast<int4*>(static_cast<int32_t*>(out) + (size_t)row * N + ncol);
#pragma unroll
            for (int i = 0; i < 8; ++i) dst[i] = make_int4(iv[4 * i], iv[4 * i + 1], iv[4 * i + 2], iv[4 * i + 3]);
          } else {
            uint32_t hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const __half2 sc2 = *reinterpret_cast<const __half2*>(col_scale + ncol + 2 * i);
              float x0 = __fmul_rn(v[2 * i], __low2float(sc2));
              float x1 = __fmul_rn(v[2 * i + 1], __high2float(sc2));
              if (epi == EPI_F16_ROWCOL) {
                x0 = __fmul_rn(x0, rsc);
                x1 = __fmul_rn(x1, rsc);
              }
              x0 = apply_act(x0, actfn);
              x1 = apply_act(x1, actfn);
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
  }

  tc_fence_before();
  __syncthreads();

  if (S > 1) {
    // ------------------------------------------------------------ split-K reduction
    // Every CTA's pipeline is idle now (MMAs, TMA loads and converters are
    // done), so its pipeline buffers become a receive area.  The tile's BN/32
    // column chunks are owned round-robin (chunk c by CTA c % S); each CTA
    // sends every chunk of its partial accumulator into its owner's area
    // (distributed shared memory, slot [sender][c / S], rows 128B-swizzled),
    // arrives on every CTA's receive barrier, and then reduces and stores the
    // chunks it owns.  All handshakes are mbarriers with bounded waits.
    if constexpr (NACC == 1) {   // split-K runs with one accumulator slice
    constexpr int NCH = BN / 32;
    const int rank = (int)cluster_ctarank();
    const int slots = (NCH + S - 1) / S;
    const uint32_t recv_base = smem_u32(smem);
    if (tid == 0) {
      for (int p = 0; p < S; ++p)
        if (p != rank) mbar_arrive_cluster(mapa_shared(smem_u32(ready_bar), (uint32_t)p));
    }
    if (warp >= C::A_WARPS && warp < C::A_WARPS + 8) {
      const int bw = warp - C::A_WARPS;
      const int q = warp & 3, chalf = bw >> 2;
      const int r = 32 * q + lane;                          // tile row (TMEM lane)
      bool ok = __all_sync(0xffffffffu, mbar_wait(accum_bar, 0, DRAIN_TIMEOUT_NS, status));
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(ready_bar, 0, DRAIN_TIMEOUT_NS, status)) && ok;
      tc_fence_after();
      if (ok) {
        for (int cc = 0; cc < NCH / 2; ++cc) {
          const int c = chalf * (NCH / 2) + cc;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(32 * c), v);
          tmem_ld_wait_tied(v);
          const uint32_t owner = (uint32_t)(c % S);
          const uint32_t row_addr = recv_base + (uint32_t)(((rank * slots + c / S) * BM + r) * 128);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            st_cluster_v4(mapa_shared(row_addr + (uint32_t)((j ^ (r & 7)) << 4), owner),
                          make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
        }
      }
      // one arrival per thread on every CTA's receive barrier (also on error,
      // so no peer waits in vain)
      for (int p = 0; p < S; ++p) mbar_arrive_cluster(mapa_shared(smem_u32(recv_bar), (uint32_t)p));
      ok = __all_sync(0xffffffffu, mbar_wait_cluster(recv_bar, 0, DRAIN_TIMEOUT_NS, status)) && ok;
      if (ok) {
        const int row = m0 + r;
        const bool row_ok = row < M;
        float rsc = 1.0f;
        if (epi == EPI_F16_ROWCOL && row_ok) rsc = __half2float(row_scale[row]);
        const int owned = (NCH - rank + S - 1) / S;
        for (int slot = chalf; slot < owned; slot += 2) {
          const int c = rank + slot * S;
          // integer operands: every partial is an exact integer below 2**24, summed as int32
          // (its float value for the fp16 epilogue is one rounding of the exact sum)
          float acc[32];
          int iacc[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            acc[i] = 0.0f;
            iacc[i] = 0;
          }
          for (int src = 0; src < S; ++src) {
            const uint8_t* rowp = smem + ((src * slots + slot) * BM + r) * 128;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const uint4 w4 = *reinterpret_cast<const uint4*>(rowp + ((j ^ (r & 7)) << 4));
              const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                if constexpr (C::A_TMEM) iacc[4 * j + e] += __float2int_rn(__uint_as_float(w[e]));
                else acc[4 * j + e] += __uint_as_float(w[e]);
              }
            }
          }
          if constexpr (C::A_TMEM) {
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[i] = __int2float_rn(iacc[i]);
          }
          const int ncol = n0 + 32 * c;
          if constexpr (AMODE == A_F16_ZP) {
            if (row_ok && ncol < N) add_zero_point(acc, zero_point, ncol, row_sum[row]);
          }
          if (row_ok && ncol < N) {
            if (epi == EPI_I32) {
              int4* dst = reinterpret_cast<int4*>(static_cast<int32_t*>(out) + (size_t)row * N + ncol);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                if constexpr (C::A_TMEM)
                  dst[i] = make_int4(iacc[4 * i], iacc[4 * i + 1], iacc[4 * i + 2], iacc[4 * i + 3]);
                else
                  dst[i] = make_int4(__float2int_rn(acc[4 * i]), __float2int_rn(acc[4 * i + 1]),
                                     __float2int_rn(acc[4 * i + 2]), __float2int_rn(acc[4 * i + 3]));
              }
            } else {
              uint32_t hv[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const __half2 sc2 = *reinterpret_cast<const __half2*>(col_scale + ncol + 2 * i);
                float x0 = __fmul_rn(acc[2 * i], __low2float(sc2));
                float x1 = __fmul_rn(acc[2 * i + 1], __high2float(sc2));
                if (epi == EPI_F16_ROWCOL) {
                  x0 = __fmul_rn(x0, rsc);
                  x1 = __fmul_rn(x1, rsc);
                }
                x0 = apply_act(x0, actfn);
                x1 = apply_act(x1, actfn);
                const __half2 h2 = __halves2half2(__float2half_rn(x0), __float2half_rn(x1));
                hv[i] = *reinterpret_cast<const uint32_t*>(&h2);
              }
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(out) + (size_t)row * N + ncol);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(hv[4 * i], hv[4 * i + 1], hv[4 * i + 2], hv[4 * i + 3]);
            }
          }
        }
      }
    }
    }  // NACC == 1
    tc_fence_before();
    __syncthreads();
  }

  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::NCOLS);
  }
}

// ---------------------------------------------------------------------------
// Host side: launch
// ---------------------------------------------------------------------------
template <int AMODE, int BBITS, int BN, int NACC, bool INTER, int ST, int RST, int NG, int MINB>
cudaError_t launch_t(const GemmArgs& g, int split, cudaStream_t stream) {
  using C = Cfg<AMODE, BBITS, BN, NACC, ST, RST, NG, MINB>;
  // the split-K receive area (split x slots x 16 KB) must fit in the pipeline buffers
  if (NACC != 1 || split < 1 || split * ((BN / 32 + split - 1) / split) * BM * 128 > C::OFF_BAR) split = 1;
  int* status = nullptr;
  cudaError_t e = device_status_ptr(&status);
  if (e != cudaSuccess) return e;
  CUtensorMap ma, mb;
  if (AMODE != A_I8_TMEM) {   // fp16 rows, one k-block per box
    e = make_map(&ma, g.a, 2, (uint64_t)g.K, (uint64_t)g.M, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    e = make_map(&ma, g.a, 1, (uint64_t)g.K, (uint64_t)g.M, 2 * BK, BM, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (e != cudaSuccess) return e;
  e = make_map(&mb, g.b, 1, (uint64_t)g.K * BBITS / 8, (uint64_t)g.N, C::B_BOX_X, BN, raw_swizzle(C::B_BOX_X));
  if (e != cudaSuccess) return e;
  auto kern = gemm_tc_kernel<AMODE, BBITS, BN, NACC, INTER, ST, RST, NG, MINB>;
  e = set_smem_once(kern, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((g.N + BN - 1) / BN), (unsigned)((g.M + BM - 1) / BM), (unsigned)split);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = (unsigned)split;
  cfg.attrs = attr;
  cfg.numAttrs = split > 1 ? 1 : 0;
  const int M = (int)g.M, N = (int)g.N, K = (int)g.K;
  const __half* rsc = reinterpret_cast<const __half*>(g.row_scale);
  const __half* csc = reinterpret_cast<const __half*>(g.col_scale);
  const int epi = epi_arg(g);
  void* out = g.c;
  const uint64_t to = (uint64_t)wait_timeout_ns();
  const __half* zp = reinterpret_cast<const __half*>(g.zero_point);
  const float* rsum = g.row_sum;
  e = cudaLaunchKernelEx(&cfg, kern, ma, mb, M, N, K, rsc, csc, zp, rsum, epi, out, to, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int AMODE, int BBITS, int BN, int NACC, int ST, int RST, int NG = TC_NG, int MINB = 1>
cudaError_t launch_layout(const GemmArgs& g, cudaStream_t stream) {
  const long long tiles = ((g.N + BN - 1) / BN) * ((g.M + BM - 1) / BM);
  const int split = NACC == 1 ? choose_split(tiles, (int)(g.K / BK)) : 1;
  if (BBITS != 8 && g.layout == BQ_LAYOUT_PLAIN)
    return launch_t<AMODE, BBITS, BN, NACC, false, ST, RST, NG, MINB>(g, split, stream);
  return launch_t<AMODE, BBITS, BN, NACC, true, ST, RST, NG, MINB>(g, split, stream);
}

// int8 x int8 on the single-CTA kernel: the chains of at most 16 k-blocks
// that keep the fp32 accumulation exact.  Returns the TMEM slices to use (1:
// 256-wide tiles, K split over a cluster so that no CTA's range exceeds 16
// k-blocks), or 0 when no configuration fits (K beyond 64 k-blocks).
int tc_i8_slices(const GemmArgs& g) {
  const int nkb = (int)(g.K / BK);
  const long long tiles = ((g.N + 255) / 256) * ((g.M + BM - 1) / BM);
  const int split = choose_split(tiles, nkb);
  if ((nkb + split - 1) / split <= 16) return 1;
  if (nkb <= 32) return 2;
  if (nkb <= 64) return 4;
  return 0;
}

}  // namespace

bool gemm_tc_i8_exact(const GemmArgs& g) { return gemm_pair_bn(g) != 0 || tc_i8_slices(g) != 0; }

cudaError_t launch_gemm_tc(const GemmArgs& g, cudaStream_t stream) {
  if (const int bn = gemm_pair_bn(g)) return launch_gemm_pair(g, bn, stream);
  const int nkb = (int)(g.K / BK);
  if (g.act == ACT_I8 && g.bbits == 8) {
    // every fp32 chain at most 1024 k long: each partial sum < 2**24, exact
    switch (tc_i8_slices(g)) {
      case 1: return launch_layout<A_I8_TMEM, 8, 256, 1, 4, 2>(g, stream);
      case 2: return launch_layout<A_I8_TMEM, 8, 128, 2, 4, 2>(g, stream);
      case 4: return launch_layout<A_I8_TMEM, 8, 64, 4, 4, 2, 1>(g, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (g.act == ACT_Q8) {
    // fp16 activations quantised in the converters: the int8 paths' chains
    if (g.bbits == 8) {
      switch (tc_i8_slices(g)) {
        case 1: return launch_layout<A_Q_TMEM, 8, 256, 1, 3, 2>(g, stream);
        case 2: return launch_layout<A_Q_TMEM, 8, 128, 2, 4, 2>(g, stream);
        case 4: return launch_layout<A_Q_TMEM, 8, 64, 4, 4, 2, 1>(g, stream);
        default: return cudaErrorInvalidValue;
      }
    }
    if (g.bbits == 4) return launch_layout<A_Q_TMEM, 4, 256, 1, 3, 2>(g, stream);
    if (g.bbits == 2) return launch_layout<A_Q_TMEM, 2, 256, 1, 4, 2>(g, stream);
    return cudaErrorInvalidValue;
  }
  // int8 activations with 4- / 2-bit weights: every partial sum < 2**24 (host-bounded K)
  if (g.act == ACT_I8 && g.bbits == 4) return launch_layout<A_I8_TMEM, 4, 256, 1, 3, 2>(g, stream);
  if (g.act == ACT_I8 && g.bbits == 2) return launch_layout<A_I8_TMEM, 2, 256, 1, 4, 2>(g, stream);
  if (g.act == ACT_F16 && g.bbits == 4) {
    // fp32 chains of at most about half of K: two TMEM slices, or split-K
    const long long tiles = ((g.N + 255) / 256) * ((g.M + BM - 1) / BM);
    if (g.zero_point) {
      if (nkb < 2 || choose_split(tiles, nkb) > 1) return launch_layout<A_F16_ZP, 4, 256, 1, 3, 2>(g, stream);
      return launch_layout<A_F16_ZP, 4, 256, 2, 3, 2>(g, stream);
    }
    if (nkb < 2 || choose_split(tiles, nkb) > 1) return launch_layout<A_F16_SMEM, 4, 256, 1, 3, 2>(g, stream);
    return launch_layout<A_F16_SMEM, 4, 256, 2, 3, 2>(g, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bq
