// Device-side helpers shared by the bq kernels: fp16 conversions of packed
// integer codes, mbarrier waits with a time limit, and thin inline-PTX
// wrappers for the sm_100-family tensor-core instructions (tcgen05.*).
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

#include "bq_internal.h"

namespace bq {

// ---------------------------------------------------------------------------
// Device status word: the first error recorded by a kernel (BQ_OK if none).
// The word lives in the tensor-core GEMM's translation unit; kernels receive
// its address as an argument.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void record_error(int* status, int code) {
  atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// Exact integer -> fp16 conversions by exponent-bias ("magic number")
// arithmetic: a field value u in [0, 2^b) OR'ed into the low mantissa bits of
// 1024.0 (0x6400) gives the fp16 number 1024 + u exactly; subtracting
// 1024 + bias yields the signed value.  Two's-complement fields are made
// offset-binary by flipping their top bit, so u = v + bias; for sub-byte
// fields the flip, the mask and the OR happen in one LOP3.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// fp16x2 constants (low half, high half equal)
constexpr uint32_t H2_MAGIC = 0x64006400u;      // 1024.0
constexpr uint32_t H2_1032 = 0x64086408u;       // 1024 + 8
constexpr uint32_t H2_1152 = 0x64806480u;       // 1024 + 128
constexpr uint32_t H2_1026 = 0x64026402u;       // 1024 + 2
constexpr uint32_t H2_INV16 = 0x2c002c00u;      // 1/16
constexpr uint32_t H2_NEG72 = 0xd480d480u;      // -(64 + 8)
constexpr uint32_t H2_INV4 = 0x34003400u;       // 1/4
constexpr uint32_t H2_NEG258 = 0xdc08dc08u;     // -(256 + 2)
constexpr uint32_t H2_NEG66 = 0xd420d420u;      // -(64 + 2)
constexpr uint32_t H2_INV64 = 0x24002400u;      // 1/64
constexpr uint32_t H2_NEG18 = 0xcc80cc80u;      // -(16 + 2)

// 4 int8 (one 32-bit word, k order 0..3) -> 2 fp16x2 words: (k0,k1), (k2,k3).
__device__ __forceinline__ void cvt_i8x4_f16(uint32_t w, uint32_t& h01, uint32_t& h23) {
  const uint32_t u = w ^ 0x80808080u;            // offset binary: u = v + 128
  // bytes {u.b0, 0x64, u.b1, 0x64} and {u.b2, 0x64, u.b3, 0x64}
  h01 = hsub2_u32(prmt(u, 0x64646464u, 0x5140u), H2_1152);
  h23 = hsub2_u32(prmt(u, 0x64646464u, 0x5342u), H2_1152);
}

// (a & mask) ^ (c & mask) | (c & ~mask): with c = magic | (sign bits inside
// the mask) this flips the top bit of every masked field (two's complement
// -> offset binary) and ORs in the magic exponent in a single LOP3.
__device__ __forceinline__ uint32_t lop3_flip_or(uint32_t a, uint32_t mask, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(r) : "r"(a), "r"(mask), "r"(c));
  return r;
}

// One interleaved 4-bit word (8 codes) -> 4 fp16x2 words in k order.
// Field positions 0..3 hold k = 0, 2, 4, 6 and positions 4..7 hold k = 1, 3, 5, 7.
__device__ __forceinline__ void cvt_i4x8_f16(uint32_t w, uint32_t (&h)[4]) {
  const uint32_t y = w >> 8;
  h[0] = hsub2_u32(lop3_flip_or(w, 0x000f000fu, 0x64086408u), H2_1032);                 // k0, k1
  h[1] = hfma2_u32(lop3_flip_or(w, 0x00f000f0u, 0x64806480u), H2_INV16, H2_NEG72);      // k2, k3
  h[2] = hsub2_u32(lop3_flip_or(y, 0x000f000fu, 0x64086408u), H2_1032);                 // k4, k5
  h[3] = hfma2_u32(lop3_flip_or(y, 0x00f000f0u, 0x64806480u), H2_INV16, H2_NEG72);      // k6, k7
}

// One interleaved 2-bit word (16 codes) -> 8 fp16x2 words in k order.
// Field positions 0..7 hold k = 0, 2, ..., 14 and positions 8..15 hold k = 1, 3, ..., 15.
__device__ __forceinline__ void cvt_i2x16_f16(uint32_t w, uint32_t (&h)[8]) {
  const uint32_t y = w >> 8;
  h[0] = hsub2_u32(lop3_flip_or(w, 0x00030003u, 0x64026402u), H2_1026);
  h[1] = hfma2_u32(lop3_flip_or(w, 0x000c000cu, 0x64086408u), H2_INV4, H2_NEG258);
  h[2] = hfma2_u32(lop3_flip_or(w, 0x00300030u, 0x64206420u), H2_INV16, H2_NEG66);
  h[3] = hfma2_u32(lop3_flip_or(w, 0x00c000c0u, 0x64806480u), H2_INV64, H2_NEG18);
  h[4] = hsub2_u32(lop3_flip_or(y, 0x00030003u, 0x64026402u), H2_1026);
  h[5] = hfma2_u32(lop3_flip_or(y, 0x000c000cu, 0x64086408u), H2_INV4, H2_NEG258);
  h[6] = hfma2_u32(lop3_flip_or(y, 0x00300030u, 0x64206420u), H2_INV16, H2_NEG66);
  h[7] = hfma2_u32(lop3_flip_or(y, 0x00c000c0u, 0x64806480u), H2_INV64, H2_NEG18);
}

// Plain-layout sub-byte word -> interleaved word (register permutation), so
// the same converters serve both layouts.
__device__ __forceinline__ uint32_t plain_to_inter_i4(uint32_t w) {
  // plain nibble i holds k = i.  Want positions 0..3 <- k0,k2,k4,k6 and 4..7 <- k1,k3,k5,k7.
  uint32_t even = 0, odd = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    even |= ((w >> (8 * i)) & 0xfu) << (4 * i);
    odd |= ((w >> (8 * i + 4)) & 0xfu) << (4 * i);
  }
  return even | (odd << 16);
}

__device__ __forceinline__ uint32_t plain_to_inter_i2(uint32_t w) {
  uint32_t even = 0, odd = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    even |= ((w >> (4 * i)) & 0x3u) << (2 * i);
    odd |= ((w >> (4 * i + 2)) & 0x3u) << (2 * i);
  }
  return even | (odd << 16);
}

// Activation of the fused epilogue (a bq_activation) on the fp32 dequantised
// value, before its rounding to fp16.  GELU uses the erf form v * Phi(v),
// written with erfc so that negative v loses nothing to cancellation.
__device__ __forceinline__ float apply_act(float v, int actfn) {
  if (actfn == BQ_ACT_RELU) return fmaxf(v, 0.0f);
  if (actfn == BQ_ACT_GELU) return 0.5f * v * erfcf(-v * 0.70710678118654752f);
  return v;
}

// ---------------------------------------------------------------------------
// Shared-memory mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}

// One blocking poll: try_wait may suspend the thread until the phase
// completes, for up to a hardware-defined time.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// One non-blocking poll: has the phase with the given parity completed?
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed, or give up after
// timeout_ns nanoseconds: records BQ_ERR_TIMEOUT in *status, returns false.
// The first poll does not block and the deadline is checked before every
// blocking poll, so a zero limit gives up unless the phase had completed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t timeout_ns, int* status) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (globaltimer_ns() - t0 >= timeout_ns) {
      record_error(status, BQ_ERR_TIMEOUT);
      return false;
    }
    if (mbar_try_wait(bar, parity)) return true;
  }
}

// Arrive once and add `bytes` to the transaction count the phase waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// 2-D tiled TMA load of the box at (x, y) (x in elements of the innermost
// dimension, a multiple of 16 bytes) into shared memory; completion is
// signalled on `bar` as transaction bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 3-D tensor load (x, y, and the batch item z) into this CTA's shared memory.
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
      : "memory");
}

// 3-D tensor store shared -> global (bulk-group completion), as tma_store_2d
// with the batch item z.
__device__ __forceinline__ void tma_store_3d(const void* tmap, const void* src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
               : "memory");
}

// 2-D tensor store shared -> global (bulk-group completion).  Elements of the
// box outside the tensor are not written.  The x coordinate times the element
// size must be a multiple of 16 bytes, and x, y must not be negative.
__device__ __forceinline__ void tma_store_2d(const void* tmap, const void* src, int x, int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y), "r"(smem_u32(src))
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until the shared-memory sources of all committed bulk stores have been read.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Wait until all committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Contiguous bulk copy global -> shared (size and both addresses multiples of
// 16 bytes); completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// Asynchronous global -> shared copies (no registers); complete with cp_async_wait_all().
__device__ __forceinline__ void cp_async_16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_8(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Thread-block cluster helpers (distributed shared memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared::cluster address of the same shared-memory location in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t local_saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_saddr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t caddr, uint4 v) {
  asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(caddr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// Arrive on an mbarrier of a peer CTA (release at cluster scope: this thread's
// earlier shared::cluster stores are visible to whoever observes the phase).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t remote_bar_caddr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar_caddr) : "memory");
}

// Arrive on an mbarrier of a CTA of this cluster with the default semantics
// (release at CTA scope): orders this thread's earlier writes to its own
// CTA's shared and tensor memory before the arrival, without the cost of a
// cluster-scope release (which waits for the thread's outstanding memory
// operations to become visible cluster-wide: about a microsecond).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t remote_bar_caddr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(remote_bar_caddr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait (acquire at cluster scope) for arrivals made by peer CTAs;
// same polling as mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint64_t timeout_ns, int* status) {
  if (mbar_test_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (globaltimer_ns() - t0 >= timeout_ns) {
      record_error(status, BQ_ERR_TIMEOUT);
      return false;
    }
    if (mbar_try_wait_cluster(bar, parity)) return true;
  }
}

// All threads of all CTAs of the cluster (used once, right after set-up,
// where every thread is guaranteed to arrive).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Release a TMA-filled shared-memory stage right after reading it with
// ordinary loads, without a fence: `dep` folds every word the thread loaded
// from the stage and `zero` is a run-time zero the compiler cannot see
// through, so the arrival count 1 + (dep & zero) is a data dependency of the
// arrive on every load.  The arrive cannot issue before all of them have
// returned their data, so the TMA refill it allows cannot overtake them (an
// mbarrier release alone does not order generic-proxy reads before an
// async-proxy write).
__device__ __forceinline__ void mbar_arrive_after_loads(uint64_t* bar, uint32_t dep, uint32_t zero) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
               "r"(1u + (dep & zero))
               : "memory");
}

// XOR of the four words of a 16-byte value (folded into `dep` above).
__device__ __forceinline__ uint32_t fold4(const uint4& v) { return v.x ^ v.y ^ v.z ^ v.w; }


// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core) wrappers, cta_group::1
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// One lane of a fully active warp (the same lane every time) gets true.  An
// elected-lane branch keeps the values computed by the whole warp uniform, so
// the tcgen05.mma operands stay in uniform registers instead of being moved
// into them at every issue.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "elect.sync _|P, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (fp16 or bf16 operands, fp32 accumulator).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16.  A occupies 128 lanes (one per
// row); each 32-bit column holds two consecutive k (lower k in the low half).
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 wrappers, cta_group::2 (a CTA pair of a cluster shares one MMA).
// A kernel uses one cta_group for all its tcgen05 instructions.  Allocation
// and deallocation are collective: one warp of each CTA of the pair issues
// them, and both CTAs receive the same tensor-memory columns.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Pair MMA issued by the even CTA: D (M = 256: rows 0-127 in the even CTA's
// tensor memory, 128-255 in the odd CTA's) (+)= A[tmem] * B[smem]^T, where A's
// rows split the same way and B's N rows are split in halves, the first half
// in the even CTA's shared memory and the second in the odd CTA's, both at
// the same offsets as the addresses given here.
__device__ __forceinline__ void tc_mma_f16_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                   uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Pair MMA with both operands in shared memory: A's 256 rows split like D
// (rows 0-127 in the even CTA's shared memory, 128-255 in the odd CTA's), B as
// for the tensor-memory form; all at the same offsets in both CTAs.
__device__ __forceinline__ void tc_mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier at the same shared-memory offset in every CTA
// of cta_mask when all pair MMAs issued so far by this thread complete.
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns from registers: thread i of the
// warp writes lane (base + i).
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}


// Arrive once on an mbarrier when all previously issued tcgen05 ops of this thread complete.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp receives lane (base + i).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// 32 lanes x 16 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

// tcgen05.ld and tcgen05.st are asynchronous: the load writes its destination
// registers, and the store reads its source registers, some time after issue.
// Every wait below names those registers as operands, so that the compiler
// neither reads the destinations before the load has written them nor
// reuses the sources' physical registers while the store may still read
// them (an untied wait left both open, and stores then read registers the
// compiler had already reassigned).
//
// Wait for this thread's tcgen05.ld and tie the 32 destination registers to
// the wait, so that no use of them (nor any reuse of their physical
// registers) is scheduled before the asynchronous load has written them.
__device__ __forceinline__ void tmem_ld_wait_tied(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
        "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
        "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}

// The same for a 16-register load.
__device__ __forceinline__ void tmem_ld_wait_tied(uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
        "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
      :
      : "memory");
}

// Wait for this thread's tcgen05.st with its 32 source registers as inputs of
// the wait: they stay allocated, unchanged, until the store has read them.
__device__ __forceinline__ void tmem_st_wait_tied(const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::st.sync.aligned;" ::"r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
      "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored in the
// 128-byte swizzle layout: rows of 128 bytes (64 fp16 along K), 8-row groups
// of 1024 bytes; inside a group, 16-byte chunk c of row r sits at chunk
// position c ^ r.  The tile base must be 1024-byte aligned.  Advancing K by
// 16 elements inside the 128-byte row is done by adding 32 bytes to the
// start address (the swizzle is applied on absolute address bits).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3ffffu) >> 4);            // start address
  d |= (uint64_t)1 << 16;                              // leading byte offset (unused for swizzled K-major)
  d |= (uint64_t)(1024 >> 4) << 32;                    // stride byte offset: 8-row group pitch
  d |= (uint64_t)1 << 46;                              // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                              // swizzle mode: 128B
  return d;
}

// Instruction descriptor, kind::f16: fp16 A and B (K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n) {
  return (1u << 4)                         // D format: f32
         | (0u << 7) | (0u << 10)          // A, B format: f16
         | ((uint32_t)(n >> 3) << 17)      // N / 8
         | ((uint32_t)(m >> 4) << 24);     // M / 16
}

}  // namespace bq
