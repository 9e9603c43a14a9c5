// Tensor-core GEMM on CTA pairs (tcgen05 cta_group::2), sm_103a.
//
// Same products and epilogues as the single-CTA kernel in gemm_tc.cu (int8
// activations times int8 / 4-bit / 2-bit weights, every code converted
// exactly to fp16, fp32 accumulation in tensor memory, fused dequantisation),
// for the forms of the BitBLAS guide ("BitBLAS自定义操作开发指南",
// 混合精度算子开发实战 1 and 2) and the BMINF linear ("BMINF的後訓練量化實現",
// 實現代碼分析2).
//
// A 256 x BN output tile is computed by the two CTAs of a cluster with pair
// MMAs (M = 256).  CTA r of the pair holds tile rows 128r .. 128r + 127: their
// int8 activations, converted into its tensor memory, and their accumulators.
// It also holds weight rows r*BN/2 .. (r+1)*BN/2 - 1 of the tile, converted
// into its shared memory.  Each SM thus converts and stores only half of the
// tile's weights per k-block while its tensor core does a full 128 x BN x 64
// share of the MMA work: the weight conversion and the shared-memory traffic
// per MMA flop are half of what one CTA per 128 x BN tile needs.
//
// Warp roles per CTA.  The converters come in groups that take the k-blocks
// in turn (group g of n converts kb = g mod n), so the fixed cost of each
// k-block's waits and arrivals overlaps across groups:
//   NA groups of 4 warps      A: int8 activation row (thread = row = TMEM
//                             lane) -> 32 fp16 pairs -> tcgen05.st into a
//                             TMEM stage (AQ: fp16 activation row ->
//                             int8 codes as fp16 pairs, the same way).
//   NB groups of P_BW warps   B: raw weight codes -> fp16 128B-swizzled
//                             K-major tile in shared memory.
//   next warp                 allocates tensor memory (collectively with the
//                             peer CTA); in the even CTA one elected lane
//                             issues the pair MMAs.
//   last warp                 producer: one thread issues the TMA loads of
//                             this CTA's raw activation and weight codes into
//                             a ring of raw stages.
// After the mainloop the converter warps store this CTA's 128 rows of the tile.
//
// Handshakes: raw stages are local (TMA complete_tx -> consumers -> producer).
// An MMA stage is ready once one A group and one B group of each CTA have
// arrived on the even CTA's full barrier (one arrival per warp); the commit of the pair MMAs arrives
// on both CTAs' empty barriers (multicast), and at the end on both
// accumulator barriers.  Every wait is bounded in time; a wait that gives up
// records BQ_ERR_TIMEOUT and the CTA leaves the tile.
//
// One CTA per SM (the shared-memory footprint guarantees it), so a CTA's
// collective tensor-memory allocation never waits on another pair that holds
// the same SM's tensor memory.
//
// Chunked accumulation (DR, int8 x int8 with K > 1024).  A product of two
// int8 codes lies in [-128 * 127, 128 * 128], so an fp32 chain longer than
// 16 k-blocks of 64 may pass 2**24, where odd integers are no longer
// representable.  In DR mode K is cut into chunks of CH_KB = 16 k-blocks that
// accumulate alternately into two TMEM accumulators (the int8 activations then
// go to shared memory as fp16 tiles, like fp16 activations, to leave tensor
// memory to the accumulators).  When chunk c is done, four drain warps (one
// per TMEM lane quadrant) read its accumulator D (exact) while chunk c + 1
// runs in the other one, split it as D = 8192 h + L with h = ceil(D / 8192),
// write L (-8192 < L <= 0) back and arrive.  Chunk c + 2 accumulates on top
// of L: its partial sums stay in [-8191 - 1024 * 16256, 1024 * 16384], inside
// +-2**24, so every value the accumulator takes is an exact integer.  The
// high parts h add up as integers in the output's own bytes (int16 per
// element for fp16 outputs, int32 for int32 outputs; every element belongs to
// one drain thread of one CTA), and the epilogue forms
// Cint = 8192 * sum(h) + D0 + D1 exactly before the dequantisation.  The
// splits use full-rate fp32 and integer arithmetic only (split_high, exact_sum).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include "bq_device.cuh"
#include "bq_internal.h"
#include "gemm_common.cuh"
#include "quant_math.cuh"

namespace bq {
namespace {

constexpr int PM = 128;                  // tile rows per CTA (256 per pair)
constexpr int PK = 64;                   // k per block: one 128-byte fp16 swizzle row
constexpr int P_NA = 2;                  // activation converter groups (4 warps each)
constexpr int P_NA_Q = 4;                // the same, quantising fp16 activations
constexpr int P_NB_Q = 4;                // weight converter groups beside them
constexpr int P_NB_DR = 4;               // weight converter groups with chunked accumulation
constexpr int ST_DR = 4;                 // MMA stages with chunked accumulation (fp16 A and B tiles)
constexpr int P_NB_I8 = 6;               // weight converter groups, int8 activations
constexpr int P_NB_F16 = 6;              // weight converter groups, fp16 activations
constexpr int P_BW = 2;                  // warps per weight converter group
constexpr int P_B_THREADS = P_BW * 32;   // weight converters per group
constexpr uint64_t P_DRAIN_NS = 4000000000ull;
constexpr int CH_KB = 16;                // k-blocks per accumulation chunk (DR mode)
constexpr float H_UNIT = 8192.0f;        // weight of one high-part unit (2**13)

// AF16: fp16 activations, loaded by TMA straight into the MMA's 128B-swizzled
// K-major layout (no activation converters, A read from shared memory), and
// two accumulator slices of half of K each (shorter fp32 chains).  Otherwise
// int8 activations, converted into tensor memory, one accumulator; with AQ
// the activations arrive as fp16 and the activation converters quantise them
// to int8 codes (the row scales given) before storing them the same way.
template <int BBITS, int BN, int ST, int RST, bool AF16, bool AQ = false, bool DR = false>
struct PairCfg {
  static constexpr int HB = BN / 2;                            // weight rows per CTA
  // quantising converters (AQ) do several times the work of an int8 conversion: more of them
  static constexpr int NA = AF16 ? 0 : ((AQ && !DR) ? P_NA_Q : P_NA);  // activation converter groups
  static constexpr int A_WARPS = 4 * NA;
  static constexpr int NB = AF16 ? P_NB_F16 : (DR ? P_NB_DR : (AQ ? P_NB_Q : P_NB_I8));   // weight converter groups
  static constexpr int CONSUMER_WARPS = A_WARPS + NB * P_BW;
  // DR: one warp per TMEM lane quadrant drains the chunks in the background
  static constexpr int DRAIN_WARPS = DR ? 4 : 0;
  static constexpr int MMA_WARP = CONSUMER_WARPS + DRAIN_WARPS;
  static constexpr int PRODUCER_WARP = MMA_WARP + 1;
  static constexpr int THREADS = (PRODUCER_WARP + 1) * 32;
  // a raw stage holds RKB k-blocks so that every TMA box row is 128 bytes (64
  // for 2-bit weights); fp16 activations to quantise fill 128-byte rows with
  // one k-block, and keep raw stages of 2 k-blocks (weight rows of 64 or 32
  // bytes for 4- and 2-bit weights)
  static constexpr int RKB = (BBITS == 8 || AQ) ? 2 : 4;
  static constexpr int B_RAW_ROW = PK * BBITS / 8;             // raw weight bytes per row per k-block
  static constexpr int B_BOX_X = RKB * B_RAW_ROW;
  static constexpr int B_PIECES_ROW = B_RAW_ROW / 16;          // 16-byte pieces per row per k-block
  static constexpr int B_PIECES = HB * B_PIECES_ROW;
  static constexpr int NPB = (B_PIECES + P_B_THREADS - 1) / P_B_THREADS;
  static constexpr int B_RAW = HB * B_BOX_X;
  static constexpr int A_BOX = PM * 128;                       // int8 activations: 2 k-blocks x 128 rows
  static constexpr int A_KB = PM * 128;                        // fp16 activations: 1 k-block x 128 rows
  static constexpr int A_RAW = AF16 ? 0 : (AQ ? A_KB * RKB : A_BOX * (RKB / 2));
  static constexpr bool A_SMEM = AF16 || DR;                   // A read by the MMA from shared memory
  static constexpr int A_TILE = A_SMEM ? PM * 128 : 0;         // fp16 activation tile of one MMA stage
  static constexpr int B_TILE = HB * 128;                      // fp16 weight tile of one MMA stage
  static constexpr int STAGE = A_TILE + B_TILE;
  static constexpr int RSTAGE = (A_RAW + B_RAW + 1023) / 1024 * 1024;
  static constexpr int NACC = (AF16 || DR) ? 2 : 1;            // accumulators (halves of K; DR: chunks in turn)
  static constexpr int A_COLS = PK / 2;                        // TMEM columns of one activation stage
  static constexpr int ACC_COLS = NACC * BN;
  static constexpr int USED_COLS = ACC_COLS + (A_SMEM ? 0 : ST * A_COLS);
  static constexpr int NCOLS = USED_COLS <= 256 ? 256 : 512;
  static constexpr int OFF_RAW = ST * STAGE;
  static constexpr int STG_BYTES = 32 * 32 * 4;                // epilogue staging box per warp (int32)
  // threads that read one (full) raw stage: a stage of RKB k-blocks is read by
  // min(groups, RKB) groups of each kind
  static constexpr int RAW_READERS =
      (NA < RKB ? NA : RKB) * 4 * 32 + (NB < RKB ? NB : RKB) * P_B_THREADS;
  // arrivals that fill an MMA stage: one warp per arrival, one A and one B group of each CTA
  static constexpr int FULL_ARRIVALS = 2 * ((AF16 ? 0 : 4) + P_BW);
  static constexpr int OFF_BAR = OFF_RAW + RST * RSTAGE;
  static constexpr size_t SMEM = (size_t)OFF_BAR + 256 + 1024;
  static_assert(USED_COLS <= 512, "tensor memory budget");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(SMEM > 116 * 1024, "one CTA per SM");
  static_assert(STAGE % 1024 == 0 && RSTAGE % 1024 == 0 && A_RAW % 1024 == 0, "stage alignment");
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "pair MMA N and 32-column epilogue chunks");
  static_assert(CONSUMER_WARPS % 4 == 0 && THREADS <= 1024, "warp roles");
  static_assert(!AF16 || BBITS == 4, "fp16 activations pair with 4-bit weights");
  static_assert(!(AF16 && AQ), "one activation form");
  // A group that has finished k-block kb - n (n groups) knows that the MMAs of
  // kb - n - ST are done; its wait for the stage of kb must not pass on the
  // parity of a phase two behind, which needs n <= ST.
  static_assert(NA <= ST && NB <= ST, "converter groups per stage ring");
  static_assert(CONSUMER_WARPS * STG_BYTES <= OFF_BAR, "epilogue staging fits in the pipeline buffers");
  static_assert((3 * ST + 2 * RST + 5) * 8 + 4 <= 256, "barrier area");
};

// Batched launch (grid z = item): element strides of the scales, the byte
// stride of the output, and whether A and B have one matrix per item (else
// every item reads item 0's; their tensor maps then hold one item).
struct PairBatch {
  int64_t srs, scs, sc;
  int za_on, zb_on;
  int on;   // batched: 3-D tensor maps; otherwise the 2-D maps of one matrix
};

// A tile load through a 2-D map, or a 3-D map at batch item z.
__device__ __forceinline__ void tma_load_item(void* dst, const void* tmap, int x, int y, int z, bool b3,
                                              uint64_t* bar) {
  if (b3) tma_load_3d(dst, tmap, x, y, z, bar);
  else tma_load_2d(dst, tmap, x, y, bar);
}

// True if the 32 consecutive output elements at element offset `off` lie
// inside the M x N output; otherwise records BQ_DIAG_RANGE (a self-check of
// the chunked accumulation's bookkeeping) and the caller skips the access.
__device__ __forceinline__ bool out_span_ok(size_t off, int M, int N, int* status) {
  if (off % 32 == 0 && off + 32 <= (size_t)M * (size_t)N) return true;
  record_error(status, BQ_DIAG_RANGE);
  return false;
}

// Split of an accumulator value D (an integer, |D| < 2**24) as D = 8192 h + L
// without conversion instructions, which issue at a quarter of the FMA rate:
// u = D / 8192 + 1.5 * 2**23, rounded once, lies in [2**23, 2**24) where fp32
// steps by 1, so u = 1.5 * 2**23 + h with h = rint(D / 8192) (ties to even),
// and the bit pattern of u is 0x4B400000 + h (|h| < 2**22).
constexpr uint32_t RNE_MAGIC_BITS = 0x4B400000u;   // bit pattern of 1.5 * 2**23
__device__ __forceinline__ float split_high(float d) { return __fmaf_rn(d, 1.0f / H_UNIT, RNE_MAGIC); }
// The same with h = ceil(D / 8192) (the sum rounded toward +infinity), so
// that L = D - 8192 h lies in (-8192, 0]
__device__ __forceinline__ float split_high_up(float d) { return __fmaf_ru(d, 1.0f / H_UNIT, RNE_MAGIC); }
// h as an int32, from u = split_high(D)
__device__ __forceinline__ int split_h(float u) { return (int)(__float_as_uint(u) - RNE_MAGIC_BITS); }
// L = D - 8192 h, exact (|L| <= 4096; -8192 < L <= 0 after split_high_up)
__device__ __forceinline__ float split_low(float d, float u) {
  return __fmaf_rn(-H_UNIT, __fsub_rn(u, RNE_MAGIC), d);
}

// D0 + D1 + 8192 hd exactly, for accumulator values D0 and D1 (integers,
// |D| <= 2**24) and an integer hd: returns the pattern of H + 1.5 * 2**23 for
// H = h0 + h1 + hd (|H| < 2**22) and sets l = L0 + L1 (exact, |l| <= 8192), so
// that the sum is 8192 H + l.  Unsigned arithmetic: the two patterns together
// pass the int32 range before the subtraction brings them back.
__device__ __forceinline__ int exact_sum(float d0, float d1, int hd, float& l) {
  const float u0 = split_high(d0), u1 = split_high(d1);
  l = __fadd_rn(split_low(d0, u0), split_low(d1, u1));
  return (int)(__float_as_uint(u0) + __float_as_uint(u1) - RNE_MAGIC_BITS + (uint32_t)hd);
}

// DR: drain warp q's share of chunk c (k-blocks CH_KB c .. CH_KB (c + 1) - 1,
// accumulated in accumulator c & 1): TMEM lane quadrant q (tile rows
// 32q .. 32q + 31), every 32-column chunk of the tile.  Each accumulator value
// is split as D = 8192 h + L (h = ceil(D / 8192), so -8192 < L <= 0), L is
// written back, and h is added to the running high parts in the output's
// bytes (int16 for fp16 outputs, int32 for int32 outputs; the first drain
// writes them); then the warp arrives on the even CTA's drained barrier of
// that accumulator.  If the chunk's barrier wait
// gives up, the warp still arrives (the MMA issuer then finds the status).
template <int BN>
__device__ __forceinline__ void pair_drain(int c, uint32_t tmem, uint64_t* chunk_bar, uint64_t* drained_bar, int q,
                                           int lane, int m0, int n0, int M, int N, int epi, void* out,
                                           uint64_t timeout_ns, int* status) {
  const int row0 = m0 + 32 * q, row = row0 + lane;
  const int acc = c & 1;
  const bool ready =
      __all_sync(0xffffffffu, mbar_wait(&chunk_bar[acc], (uint32_t)((c >> 1) & 1), timeout_ns, status));
  tc_fence_after();
  // chunks whose columns start inside N, for a quadrant with rows inside M (warp-uniform)
  int nch = 0;
  if (ready && row0 < M) {
    nch = (N - n0 + 31) / 32;
    if (nch > BN / 32) nch = BN / 32;
  }
#pragma unroll 1
  for (int ch = 0; ch < nch; ++ch) {
    const uint32_t ta = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN + 32 * ch);
    const size_t off = (size_t)row * N + n0 + 32 * ch;
    const bool mine = row < M && out_span_ok(off, M, N, status);
    // fp16 outputs: the running high parts (int16) of this row's 32 columns
    // are loaded first, so that their latency overlaps the tensor-memory work
    uint32_t old[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) old[i] = 0;
    if (mine && c > 0 && epi != EPI_I32) {
      const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(out) + off);
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        const uint4 o = p[v];
        old[4 * v] = o.x;
        old[4 * v + 1] = o.y;
        old[4 * v + 2] = o.z;
        old[4 * v + 3] = o.w;
      }
    }
    uint32_t r[32];
    uint32_t hp[16];   // high parts, two int16 per word
    tmem_ld_32x32b_x32(ta, r);
    tmem_ld_wait_tied(r);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      // D = 8192 h + L exactly, with h = ceil(D / 8192) and -8192 < L <= 0, in
      // full-rate arithmetic only (no conversion instructions): see split_high
      const float f0 = __uint_as_float(r[2 * i]), f1 = __uint_as_float(r[2 * i + 1]);
      const float u0 = split_high_up(f0), u1 = split_high_up(f1);
      r[2 * i] = __float_as_uint(split_low(f0, u0));
      r[2 * i + 1] = __float_as_uint(split_low(f1, u1));
      // the low 16 bits of u's pattern are h modulo 2**16
      hp[i] = __vadd2(__byte_perm(__float_as_uint(u0), __float_as_uint(u1), 0x5410), old[i]);
    }
    tmem_st_32x32b_x32(ta, r);
    tmem_st_wait_tied(r);
    if (mine) {
      if (epi == EPI_I32) {   // int32 running sums (they may pass the int16 range at long K)
        int4* p = reinterpret_cast<int4*>(static_cast<int32_t*>(out) + off);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint32_t w0 = hp[2 * v], w1 = hp[2 * v + 1];
          int4 h = make_int4((int)(int16_t)(w0 & 0xffffu), (int)w0 >> 16, (int)(int16_t)(w1 & 0xffffu),
                             (int)w1 >> 16);
          if (c > 0) {
            const int4 o = p[v];
            h.x += o.x;
            h.y += o.y;
            h.z += o.z;
            h.w += o.w;
          }
          p[v] = h;
        }
      } else {
        uint4* p = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + off);
#pragma unroll
        for (int v = 0; v < 4; ++v) p[v] = make_uint4(hp[4 * v], hp[4 * v + 1], hp[4 * v + 2], hp[4 * v + 3]);
      }
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&drained_bar[acc]), 0));
}

// ACTV: the fp16 epilogue applies the activation in bits 4.. of `epi` (a
// separate instantiation, so the kernel without one carries no trace of it).
// DR: chunked accumulation (int8 x int8, K > 1024); `out` is the output
// (also the home of the running high parts), used only in that mode.
// ZP (fp16 activations): unsigned 4-bit weight codes with a per-column zero
// point; the epilogue adds (8 - zero_point[j]) * row_sum[i].
template <int BBITS, int BN, bool INTER, int ST, int RST, bool AF16, bool AQ, bool ACTV, bool DR, bool ZP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<BBITS, BN, ST, RST, AF16, AQ, DR>::THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                     const __grid_constant__ CUtensorMap tmap_c, int M, int N, int K,
                     const __half* __restrict__ row_scale, const __half* __restrict__ col_scale,
                     const __half* __restrict__ zero_point, const float* __restrict__ row_sum, int epi,
                     void* out, const PairBatch bt, uint64_t timeout_ns, int* status) {
  using C = PairCfg<BBITS, BN, ST, RST, AF16, AQ, DR>;
  static_assert(!DR || (BBITS == 8 && !AF16), "chunked accumulation is for int8 x int8");
  static_assert(!ZP || (AF16 && BBITS == 4), "zero points are for fp16 x 4-bit");
  const int actfn = epi >> 4;
  epi &= 15;
  extern __shared__ uint8_t smem_raw[];
  // same offset in both CTAs: the pair MMA addresses the peer's tile by this CTA's offsets
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);   // even CTA: stage filled by both
  uint64_t* empty_bar = full_bar + ST;                                   // MMAs done with a stage
  uint64_t* rfull_bar = empty_bar + ST;                                  // raw stage landed
  uint64_t* rempty_bar = rfull_bar + RST;                                // raw stage read
  uint64_t* accum_bar = rempty_bar + RST;                                // all MMAs done
  uint64_t* afull_bar = accum_bar + 1;                                   // fp16 activation tile landed
  uint64_t* chunk_bar = afull_bar + ST;                                  // DR: MMAs of a chunk done (per accumulator)
  uint64_t* drained_bar = chunk_bar + 2;                                 // DR (even CTA): chunk drained (per accumulator)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drained_bar + 2);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  // batch item: its scales and output; A and B through the third map coordinate
  const int z = (int)blockIdx.z;
  const int za = bt.za_on ? z : 0, zb = bt.zb_on ? z : 0;
  if (row_scale) row_scale += z * bt.srs;
  if (col_scale) col_scale += z * bt.scs;
  out = static_cast<uint8_t*>(out) + z * bt.sc;
  const int m0 = (int)(blockIdx.x >> 1) * (2 * PM) + (int)rank * PM;   // this CTA's tile rows
  const int n0 = blockIdx.y * BN;                                      // the pair's output columns
  const int nb0 = n0 + (int)rank * C::HB;                              // this CTA's weight rows
  const int nkb = K / PK;
  // DR: chunks of CH_KB k-blocks; chunk c is drained when chunk c + 2 will reuse its accumulator
  const int nchunks = DR ? (nkb + CH_KB - 1) / CH_KB : 1;
  const int ndrain = nchunks > 2 ? nchunks - 2 : 0;
  const uint32_t rzero = (uint32_t)K >> 30;      // 0 (K <= 65536), not known to the compiler

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&full_bar[s], C::FULL_ARRIVALS);
      mbar_init(&empty_bar[s], 1);
      mbar_init(&afull_bar[s], 1);
    }
    for (int s = 0; s < RST; ++s) {
      mbar_init(&rfull_bar[s], 1);
      mbar_init(&rempty_bar[s], C::RAW_READERS);   // every group that reads a raw stage releases it once
    }
    mbar_init(accum_bar, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&chunk_bar[i], 1);
      // one arrival per drain warp of each CTA (a count of 0 is not a valid
      // mbarrier; without DR the barrier is unused)
      mbar_init(&drained_bar[i], C::DRAIN_WARPS > 0 ? 2 * C::DRAIN_WARPS : 1);
    }
    mbar_fence_init();
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc_pair(tmem_slot, C::NCOLS);
    tmem_relinquish_pair();
  }
  if (warp == C::PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tmap_a);
    tma_prefetch_desc(&tmap_b);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the peer arrives on this CTA's barriers only once they are initialised
  cluster_sync_all();

  bool ok = true;
  // DR: the drain warps and the consumer warps meet here before the epilogue
  // reads the high parts the drains stored
  constexpr int DRAIN_SYNC_THREADS = (C::CONSUMER_WARPS + C::DRAIN_WARPS) * 32;
  if (warp == C::PRODUCER_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0, issued_a = 0;
      for (int kb = 0; kb < nkb; ++kb) {
        if (kb % C::RKB == 0) {
          // raw stage for k-blocks [kb, kb + RKB): boxes past K read as zero
          const int grp = kb / C::RKB, rs = grp % RST;
          if (!mbar_wait(&rempty_bar[rs], ((grp / RST) & 1) ^ 1, timeout_ns, status)) break;
          uint8_t* raw = smem + C::OFF_RAW + rs * C::RSTAGE;
          mbar_arrive_expect_tx(&rfull_bar[rs], C::A_RAW + C::B_RAW);
          if constexpr (AQ) {
#pragma unroll
            for (int b = 0; b < C::RKB; ++b)
              tma_load_item(raw + b * C::A_KB, &tmap_a, (kb + b) * PK, m0, za, bt.on, &rfull_bar[rs]);
          } else if constexpr (!AF16) {
#pragma unroll
            for (int b = 0; b < C::RKB / 2; ++b)
              tma_load_item(raw + b * C::A_BOX, &tmap_a, (kb + 2 * b) * PK, m0, za, bt.on, &rfull_bar[rs]);
          }
          tma_load_item(raw + C::A_RAW, &tmap_b, kb * C::B_RAW_ROW, nb0, zb, bt.on, &rfull_bar[rs]);
          issued = grp + 1;
        }
        if constexpr (AF16) {
          // fp16 activations straight into the MMA stage, once the MMAs are done with it
          const int s = kb % ST;
          if (!mbar_wait(&empty_bar[s], ((kb / ST) & 1) ^ 1, timeout_ns, status)) break;
          mbar_arrive_expect_tx(&afull_bar[s], C::A_TILE);
          tma_load_item(smem + s * C::STAGE, &tmap_a, kb * PK, m0, za, bt.on, &afull_bar[s]);
          issued_a = kb + 1;
        }
      }
      // no TMA write may land after the CTA has exited
      for (int grp = issued > RST ? issued - RST : 0; grp < issued; ++grp)
        mbar_wait(&rfull_bar[grp % RST], (grp / RST) & 1, P_DRAIN_NS, status);
      for (int kb = issued_a > ST ? issued_a - ST : 0; kb < issued_a; ++kb)
        mbar_wait(&afull_bar[kb % ST], (kb / ST) & 1, P_DRAIN_NS, status);
    }
    __syncwarp();
  } else if (warp == C::MMA_WARP) {
    // ------------------------------------------------------------ pair MMA issuer (even CTA)
    // The whole warp runs the loop, so the operand addresses are warp-uniform;
    // one elected lane issues the MMAs and their commits.
    if (rank == 0) {
      const uint32_t tm = __shfl_sync(0xffffffffu, tmem, 0);
      const uint32_t smem_base = __shfl_sync(0xffffffffu, smem_u32(smem), 0);
      const uint32_t idesc = idesc_f16_f32(2 * PM, BN);
      // fp16 activations: k-blocks [0, kb_half) accumulate into slice 0, the rest into slice 1
      const int kb_half = C::NACC == 2 ? (nkb + 1) / 2 : nkb;
      for (int kb = 0; kb < nkb; ++kb) {
        const int s = kb % ST;
        const int chunk = kb / CH_KB;
        if (DR && kb % CH_KB == 0 && chunk >= 2) {
          // chunk c adds on top of what the drain of chunk c - 2 left in the same accumulator
          if (!__all_sync(0xffffffffu,
                          mbar_wait_cluster(&drained_bar[chunk & 1], ((chunk - 2) >> 1) & 1, timeout_ns, status)))
            break;
        }
        if (!__all_sync(0xffffffffu, mbar_wait_cluster(&full_bar[s], (kb / ST) & 1, timeout_ns, status))) break;
        tc_fence_after();
        // DR: accumulator chunk & 1, fresh for chunks 0 and 1; otherwise slices of halves of K
        const int slice = DR ? (chunk & 1) : (kb < kb_half ? 0 : 1);
        const bool first = DR ? (kb % CH_KB == 0 && chunk < 2) : (kb == 0 || kb == kb_half);
        const uint32_t d = tm + (uint32_t)(slice * BN);
        const uint64_t bdesc = smem_desc_sw128(smem_base + s * C::STAGE + C::A_TILE);
        if (elect_one()) {
          if constexpr (C::A_SMEM) {
            const uint64_t adesc = smem_desc_sw128(smem_base + s * C::STAGE);
#pragma unroll
            for (int kk = 0; kk < PK / 16; ++kk)   // +32 bytes along K = +2 in the address field
              tc_mma_f16_pair(d, adesc + 2 * kk, bdesc + 2 * kk, idesc, (first && kk == 0) ? 0u : 1u);
          } else {
            const uint32_t a_tm = tm + (uint32_t)(C::ACC_COLS + s * C::A_COLS);
#pragma unroll
            for (int kk = 0; kk < PK / 16; ++kk)   // 16 k = 8 TMEM columns of A = +32 bytes of B
              tc_mma_f16_ts_pair(d, a_tm + 8 * kk, bdesc + 2 * kk, idesc, (first && kk == 0) ? 0u : 1u);
          }
          tc_commit_pair(&empty_bar[s], 0x3);
          // DR: the last k-block of a chunk whose accumulator a later chunk reuses: let the drain warps take it
          if (DR && (kb + 1) % CH_KB == 0 && chunk < ndrain) tc_commit_pair(&chunk_bar[chunk & 1], 0x3);
        }
        __syncwarp();
      }
      if (elect_one()) tc_commit_pair(accum_bar, 0x3);
      __syncwarp();
      // no MMA may still be running when either CTA frees its tensor memory or exits
      mbar_wait(accum_bar, 0, P_DRAIN_NS, status);
    }
    __syncwarp();
  } else if (warp < C::A_WARPS) {
    // ------------------------------------------------------------ int8 activations -> TMEM
    // A group g (warps 4g .. 4g + 3) converts the k-blocks kb = g (mod NA)
    const int q = warp & 3;                               // TMEM lane quadrant
    const int r = q * 32 + lane;                          // tile row == TMEM lane
    RowQuant rq{};
    if constexpr (AQ) rq = row_quant(m0 + r < M ? __half2float(row_scale[m0 + r]) : 0.0f);
    for (int kb = warp >> 2; kb < nkb; kb += C::NA) {
      const int grp = kb / C::RKB, rs = grp % RST;
      // the group's first k-block of a raw stage waits for it to land
      if (kb % C::RKB < C::NA && !warp_wait(&rfull_bar[rs], (grp / RST) & 1, timeout_ns, status)) {
        ok = false;
        break;
      }
      const bool last_use = (kb % C::RKB) + C::NA >= C::RKB || kb + C::NA >= nkb;   // the group's last use
      uint32_t h[32];
      if constexpr (AQ) {
        // this k-block is one 128-byte box row of fp16 values (chunk c of row r at c ^ (r & 7))
        const uint8_t* box = smem + C::OFF_RAW + rs * C::RSTAGE + (kb % C::RKB) * C::A_KB + r * 128;
        quant64_f16_codes(box, r, rq, h);
        // the codes depend on every value read, so the release follows those reads
        if (last_use) {
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
        if (last_use)
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
      if (!warp_wait(&empty_bar[s], ((kb / ST) & 1) ^ 1, timeout_ns, status)) {
        ok = false;
        break;
      }
      if constexpr (C::A_SMEM) {
        // DR: the row's 64 fp16 values into the stage's 128B-swizzled K-major tile
        uint8_t* ta = smem + s * C::STAGE;
#pragma unroll
        for (int j = 0; j < 8; ++j) st_chunk(ta, r, j, make_uint4(h[4 * j], h[4 * j + 1], h[4 * j + 2], h[4 * j + 3]));
        fence_proxy_async_smem();   // generic stores -> visible to the tensor core (async proxy)
      } else {
        // order the store after the MMAs whose completion the barrier reported:
        // without the fence it may overwrite the stage while they still read it
        tc_fence_after();
        tmem_st_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(C::ACC_COLS + s * C::A_COLS), h);
        tmem_st_wait_tied(h);
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&full_bar[s]), 0));
    }
  } else if (warp < C::CONSUMER_WARPS) {
    // ------------------------------------------------------------ weights -> fp16 smem
    // B group g (warps A_WARPS + g * P_BW ..) converts the k-blocks kb = g (mod NB)
    const int bw = warp - C::A_WARPS;
    const int c = (bw % P_BW) * 32 + lane;                // converter thread within its group
    for (int kb = bw / P_BW; kb < nkb; kb += C::NB) {
      const int grp = kb / C::RKB, rs = grp % RST;
      if (kb % C::RKB < C::NB && !warp_wait(&rfull_bar[rs], (grp / RST) & 1, timeout_ns, status)) {
        ok = false;
        break;
      }
      const uint8_t* raw = smem + C::OFF_RAW + rs * C::RSTAGE + C::A_RAW;
      // piece pi is (row pi % HB, piece pi / HB): a quarter warp reads 8 rows,
      // whose swizzled chunk positions differ (conflict-free)
      uint4 v[C::NPB];
#pragma unroll
      for (int i = 0; i < C::NPB; ++i) {
        const int pi = c + i * P_B_THREADS;
        const int r = pi % C::HB, sub = pi / C::HB;
        const int chunk = (kb % C::RKB) * C::B_PIECES_ROW + sub;
        const int pos = raw_chunk_pos<C::B_BOX_X>(chunk, r);
        v[i] = pi < C::B_PIECES ? *reinterpret_cast<const uint4*>(raw + r * C::B_BOX_X + (pos << 4))
                                : make_uint4(0, 0, 0, 0);
      }
      if ((kb % C::RKB) + C::NB >= C::RKB || kb + C::NB >= nkb) {   // group's last use
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
        const int pi = c + i * P_B_THREADS;
        if (pi < C::B_PIECES) convert_b_piece<BBITS, INTER, ZP>(tb, pi % C::HB, pi / C::HB, v[i]);
      }
      fence_proxy_async_smem();   // generic stores -> visible to the tensor core (async proxy)
      // fp16 activations: this CTA's half of the stage is complete once its tile has landed
      if (AF16 && !warp_wait(&afull_bar[s], (kb / ST) & 1, timeout_ns, status)) {
        ok = false;
        break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&full_bar[s]), 0));
    }
  } else if constexpr (DR) {
    // ------------------------------------------------------------ drain warps (DR)
    // warp CONSUMER_WARPS + q owns TMEM lane quadrant q; chunk c is drained
    // while chunk c + 1 is multiplied, before chunk c + 2 reuses the accumulator
    const int q = warp & 3;
#pragma unroll 1
    for (int c = 0; c < ndrain; ++c)
      pair_drain<BN>(c, tmem, chunk_bar, drained_bar, q, lane, m0, n0, M, N, epi, out, timeout_ns, status);
    __threadfence_block();   // the high parts' stores, before the consumers read them
    asm volatile("bar.sync 1, %0;" ::"n"(DRAIN_SYNC_THREADS) : "memory");
  }

  // ------------------------------------------------------------ epilogue (consumer warps)
  if (warp < C::CONSUMER_WARPS) {
    const bool acc_ok = warp_wait(accum_bar, 0, ok ? timeout_ns : 0, status);
    tc_fence_after();
    // DR: every consumer thread waits for every drain warp's high parts (exactly once, whatever happened)
    if constexpr (DR) asm volatile("bar.sync 1, %0;" ::"n"(DRAIN_SYNC_THREADS) : "memory");
    if (acc_ok) {
      // CONSUMER_WARPS / 4 warps share each TMEM lane quadrant; each takes
      // every such 32-column chunk.  The pipeline buffers are idle now: each
      // warp stages its 32 x 32 output boxes in its own 4 KB of them (rows
      // swizzled like the tensor map) and stores them with TMA.
      const int q = warp & 3;
      const int part = warp >> 2;
      const int row0 = m0 + 32 * q;
      const int row = row0 + lane;
      float rsc = 1.0f;
      if (epi == EPI_F16_ROWCOL && row < M) rsc = __half2float(row_scale[row]);
      uint8_t* stg = smem + warp * C::STG_BYTES;
#pragma unroll 1
      for (int ch = part; ch < BN / 32 && row0 < M; ch += C::CONSUMER_WARPS / 4) {
        const int col = ch * 32;
        const int ncol = n0 + col;
        if (ncol >= N) break;
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)col, r);
        tmem_ld_wait_tied(r);
        if constexpr (C::NACC == 2 && !DR) {
          uint32_t r2[32];
          tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(col + BN), r2);
          tmem_ld_wait_tied(r2);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + __uint_as_float(r2[i]));
        }
        if constexpr (ZP) {
          if (row < M) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
            add_zero_point(v, zero_point, ncol, row_sum[row]);
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(v[i]);
          }
        }
        // exact integer sums, in r as int32 patterns for int32 outputs: rint(D0);
        // DR: D0 + D1 + 8192 times the drained high parts (for fp16 outputs that
        // sum rounded once to fp32, in r as a float)
        if constexpr (!DR) {
          if (epi == EPI_I32) {
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = (uint32_t)__float2int_rn(__uint_as_float(r[i]));
          }
        } else {
          const size_t off = (size_t)row * N + ncol;
          const bool with_h = ndrain > 0 && row < M && out_span_ok(off, M, N, status);
          // D1 in two halves of 16 columns (fewer live registers)
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            uint32_t r2[16];
            if (nchunks >= 2) {
              tmem_ld_32x32b_x16(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(col + BN + 16 * hf), r2);
              tmem_ld_wait_tied(r2);
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j) r2[j] = 0u;
            }
            if (epi == EPI_I32) {
              const int4* p = reinterpret_cast<const int4*>(static_cast<const int32_t*>(out) + off) + 4 * hf;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const int4 h = with_h ? p[v] : make_int4(0, 0, 0, 0);
                const int hd[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  const int j = 4 * v + e, i = 16 * hf + j;
                  float l;
                  const int hm = exact_sum(__uint_as_float(r[i]), __uint_as_float(r2[j]), hd[e], l);
                  r[i] = (uint32_t)((hm - (int)RNE_MAGIC_BITS) * (int)H_UNIT + split_h(__fadd_rn(l, RNE_MAGIC)));
                }
              }
            } else {
              const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(out) + off) + 2 * hf;
#pragma unroll
              for (int v = 0; v < 2; ++v) {
                const uint4 h = with_h ? p[v] : make_uint4(0, 0, 0, 0);
                const uint32_t w[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  const int j = 8 * v + e, i = 16 * hf + j;
                  const int hd = (e & 1) ? ((int)w[e >> 1] >> 16) : (int)(int16_t)(w[e >> 1] & 0xffffu);
                  float l;
                  const int hm = exact_sum(__uint_as_float(r[i]), __uint_as_float(r2[j]), hd, l);
                  // 8192 H + L rounded once (H: its pattern less that of 1.5 * 2**23)
                  r[i] = __float_as_uint(__fmaf_rn(H_UNIT, __fsub_rn(__int_as_float(hm), RNE_MAGIC), l));
                }
              }
            }
          }
        }
        if (lane == 0) bulk_wait_read_all();   // the previous box has left the staging buffer
        __syncwarp();
        if (epi == EPI_I32) {
          // row `lane`: 32 int32 = 8 chunks of 16 bytes; 128B swizzle (chunk j at j ^ (lane & 7))
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<int4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_int4((int)r[4 * j], (int)r[4 * j + 1], (int)r[4 * j + 2], (int)r[4 * j + 3]);
        } else {
          uint32_t hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __half2 sc2 = *reinterpret_cast<const __half2*>(col_scale + ncol + 2 * i);
            float x0 = __fmul_rn(__uint_as_float(r[2 * i]), __low2float(sc2));
            float x1 = __fmul_rn(__uint_as_float(r[2 * i + 1]), __high2float(sc2));
            if (epi == EPI_F16_ROWCOL) {
              x0 = __fmul_rn(x0, rsc);
              x1 = __fmul_rn(x1, rsc);
            }
            if constexpr (ACTV) {
              x0 = apply_act(x0, actfn);
              x1 = apply_act(x1, actfn);
            }
            const __half2 h2 = __halves2half2(__float2half_rn(x0), __float2half_rn(x1));
            hv[i] = *reinterpret_cast<const uint32_t*>(&h2);
          }
          // row `lane`: 32 fp16 = 4 chunks of 16 bytes; 64B swizzle (chunk j at j ^ ((lane >> 1) & 3))
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                make_uint4(hv[4 * j], hv[4 * j + 1], hv[4 * j + 2], hv[4 * j + 3]);
        }
        fence_proxy_async_smem();   // generic stores -> visible to the TMA engine
        // DR: this box's high parts were written and read through the generic
        // proxy; order those accesses before the TMA store of the same bytes
        if constexpr (DR) asm volatile("fence.proxy.async.global;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          if (bt.on) tma_store_3d(&tmap_c, stg, ncol, row0, z);   // rows past M are not written
          else tma_store_2d(&tmap_c, stg, ncol, row0);
          bulk_commit_group();
        }
      }
      // the staging buffers must outlive the TMA engine's reads of them; the
      // global writes themselves are complete when the grid is
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  // the peer no longer reads this CTA's shared memory or arrives on its barriers
  cluster_sync_all();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::NCOLS);
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
template <int BBITS, int BN, bool INTER, int ST, int RST, bool AF16, bool AQ, bool ACTV, bool DR, bool ZP = false>
cudaError_t launch_pair_t(const GemmArgs& g, cudaStream_t stream) {
  using C = PairCfg<BBITS, BN, ST, RST, AF16, AQ, DR>;
  int* status = nullptr;
  cudaError_t e = device_status_ptr(&status);
  if (e != cudaSuccess) return e;
  CUtensorMap ma, mb, mc;
  // A batched launch copies with 3-D instructions through 3-D maps for all
  // three operands (the batch item as the third coordinate; a broadcast
  // operand's map holds one item); a single call uses 2-D maps and copies.
  // The rank of every map must match bt.on, the kernel's choice of copy.
  const uint64_t nb = (uint64_t)(g.batch < 1 ? 1 : g.batch);
  const bool b3 = nb > 1;
  const uint64_t na = g.sa ? nb : 1, nbw = g.sb ? nb : 1;
  auto map = [&](CUtensorMap* m, const void* base, int elem, uint64_t row_elems, uint64_t rows, uint64_t items,
                 int64_t stride, uint32_t bx, uint32_t by, CUtensorMapSwizzle swz) {
    return b3 ? make_map3(m, base, elem, row_elems, rows, items, (uint64_t)stride, bx, by, swz)
              : make_map(m, base, elem, row_elems, rows, bx, by, swz);
  };
  if (AF16 || AQ)   // one k-block of fp16 rows: 128 bytes, the MMA's (or the converters') 128B swizzle
    e = map(&ma, g.a, 2, (uint64_t)g.K, (uint64_t)g.M, na, g.sa, PK, PM, CU_TENSOR_MAP_SWIZZLE_128B);
  else        // two k-blocks of int8 rows
    e = map(&ma, g.a, 1, (uint64_t)g.K, (uint64_t)g.M, na, g.sa, 2 * PK, PM, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  e = map(&mb, g.b, 1, (uint64_t)g.K * BBITS / 8, (uint64_t)g.N, nbw, g.sb, C::B_BOX_X, C::HB,
          raw_swizzle(C::B_BOX_X));
  if (e != cudaSuccess) return e;
  // output boxes of 32 x 32: int32 rows of 128 bytes, fp16 rows of 64 bytes
  if (g.epi == EPI_I32)
    e = map(&mc, g.c, 4, (uint64_t)g.N, (uint64_t)g.M, nb, g.sc, 32, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  else
    e = map(&mc, g.c, 2, (uint64_t)g.N, (uint64_t)g.M, nb, g.sc, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
  if (e != cudaSuccess) return e;
  const PairBatch bt{g.srs / 2, g.scs / 2, g.sc, g.sa != 0, g.sb != 0, b3 ? 1 : 0};
  auto kern = gemm_pair_kernel<BBITS, BN, INTER, ST, RST, AF16, AQ, ACTV, DR, ZP>;
  e = set_smem_once(kern, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid((unsigned)(2 * ((g.M + 2 * PM - 1) / (2 * PM))), (unsigned)((g.N + BN - 1) / BN), (unsigned)nb);
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(ma, mb, mc, (int)g.M, (int)g.N, (int)g.K,
                                              reinterpret_cast<const __half*>(g.row_scale),
                                              reinterpret_cast<const __half*>(g.col_scale),
                                              reinterpret_cast<const __half*>(g.zero_point), g.row_sum, epi_arg(g), g.c,
                                              bt, (uint64_t)wait_timeout_ns(), status);
  return cudaGetLastError();
}

template <int BBITS, int BN, int ST, int RST, bool AF16, bool AQ, bool ACTV>
cudaError_t launch_pair_act(const GemmArgs& g, cudaStream_t stream) {
  if constexpr (BBITS == 8 && !AF16) {
    // int8 x int8 beyond 16 k-blocks: chunked accumulation keeps the sums exact
    // (fp16 A and B tiles in ST_DR stages, four drain warps; fp16 activations to quantise need wider raw stages)
    if (g.K > 16 * PK) return launch_pair_t<8, BN, true, ST_DR, AQ ? 2 : 3, false, AQ, ACTV, true>(g, stream);
    return launch_pair_t<8, BN, true, ST, RST, false, AQ, ACTV, false>(g, stream);
  } else if constexpr (AF16) {
    if (g.zero_point) {
      if (g.layout == BQ_LAYOUT_PLAIN) return launch_pair_t<BBITS, BN, false, ST, RST, AF16, AQ, ACTV, false, true>(g, stream);
      return launch_pair_t<BBITS, BN, true, ST, RST, AF16, AQ, ACTV, false, true>(g, stream);
    }
    if (g.layout == BQ_LAYOUT_PLAIN) return launch_pair_t<BBITS, BN, false, ST, RST, AF16, AQ, ACTV, false>(g, stream);
    return launch_pair_t<BBITS, BN, true, ST, RST, AF16, AQ, ACTV, false>(g, stream);
  } else {
    if (BBITS != 8 && g.layout == BQ_LAYOUT_PLAIN)
      return launch_pair_t<BBITS, BN, false, ST, RST, AF16, AQ, ACTV, false>(g, stream);
    return launch_pair_t<BBITS, BN, true, ST, RST, AF16, AQ, ACTV, false>(g, stream);
  }
}

template <int BBITS, int BN, int ST, int RST, bool AF16 = false, bool AQ = false>
cudaError_t launch_pair_layout(const GemmArgs& g, cudaStream_t stream) {
  if (g.actfn != BQ_ACT_NONE) return launch_pair_act<BBITS, BN, ST, RST, AF16, AQ, true>(g, stream);
  return launch_pair_act<BBITS, BN, ST, RST, AF16, AQ, false>(g, stream);
}

cudaError_t launch_pair_f16(const GemmArgs& g, int bn, cudaStream_t stream) {
  switch (bn) {
    case 256: return launch_pair_layout<4, 256, 6, 2, true>(g, stream);
    case 224: return launch_pair_layout<4, 224, 6, 3, true>(g, stream);
    case 192: return launch_pair_layout<4, 192, 6, 3, true>(g, stream);
    case 160: return launch_pair_layout<4, 160, 6, 3, true>(g, stream);
    default: return cudaErrorInvalidValue;
  }
}

// fp16 activations quantised in the converters: raw stages of 2 k-blocks
// with twice the activation bytes, so fewer of them fit
template <int BBITS>
cudaError_t launch_pair_q(const GemmArgs& g, int bn, cudaStream_t stream) {
  switch (bn) {
    case 256: return launch_pair_layout<BBITS, 256, 6, BBITS == 8 ? 2 : 3, false, true>(g, stream);
    case 224: return launch_pair_layout<BBITS, 224, 6, 3, false, true>(g, stream);
    case 192: return launch_pair_layout<BBITS, 192, 6, 3, false, true>(g, stream);
    case 160: return launch_pair_layout<BBITS, 160, 6, 3, false, true>(g, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int BBITS>
cudaError_t launch_pair_bits(const GemmArgs& g, int bn, cudaStream_t stream) {
  constexpr int RST = BBITS == 8 ? 4 : 3;
  switch (bn) {
    case 256: return launch_pair_layout<BBITS, 256, 6, BBITS == 4 ? 2 : RST>(g, stream);
    case 224: return launch_pair_layout<BBITS, 224, 6, RST>(g, stream);
    case 192: return launch_pair_layout<BBITS, 192, 6, RST>(g, stream);
    case 160: return launch_pair_layout<BBITS, 160, 6, RST>(g, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

int gemm_pair_bn(const GemmArgs& g) {
  if (g.M <= 0 || g.N <= 0 || g.K < PK) return 0;
  // fp16 activations accumulate two halves of K separately: at least two k-blocks
  if (g.act == ACT_F16 && (g.bbits != 4 || g.K < 2 * PK)) return 0;
  // int8 x int8 beyond K = 1024 runs with chunked accumulation, whose running
  // high parts live in the output: as int16 for fp16 outputs, where
  // |sum of high parts| <= 2K + 2048 must stay below 2**15
  if (g.bbits == 8 && g.epi != EPI_I32 && g.K > 8192) return 0;
  if (g.bbits != 8 && g.bbits != 4 && g.bbits != 2) return 0;
  // grids smaller than the GPU go to the single-CTA kernel, which splits K over clusters
  const long long tiles1 = ((g.N + 255) / 256) * ((g.M + 127) / 128);
  if (choose_split(tiles1, (int)(g.K / PK)) > 1) return 0;
  // the tile width that finishes in the fewest waves of pairs, weighting a wave by its width
  const long long pairs = sm_count() / 2;
  const long long mp = (g.M + 2 * PM - 1) / (2 * PM);
  int best = 0;
  long long best_cost = 0;
  for (int bn : {256, 224, 192, 160}) {
    const long long waves = (mp * ((g.N + bn - 1) / bn) + pairs - 1) / pairs;
    const long long cost = waves * (bn + 32);
    if (best == 0 || cost < best_cost) {
      best = bn;
      best_cost = cost;
    }
  }
  return best;
}

cudaError_t launch_gemm_pair(const GemmArgs& g, int bn, cudaStream_t stream) {
  if (g.act == ACT_F16) return launch_pair_f16(g, bn, stream);
  if (g.act == ACT_Q8) {
    if (g.bbits == 4) return launch_pair_q<4>(g, bn, stream);
    if (g.bbits == 2) return launch_pair_q<2>(g, bn, stream);
    if (g.bbits == 8) return launch_pair_q<8>(g, bn, stream);
    return cudaErrorInvalidValue;
  }
  if (g.bbits == 4) return launch_pair_bits<4>(g, bn, stream);
  if (g.bbits == 2) return launch_pair_bits<2>(g, bn, stream);
  if (g.bbits == 8) return launch_pair_bits<8>(g, bn, stream);
  return cudaErrorInvalidValue;
}

}  // namespace bq
