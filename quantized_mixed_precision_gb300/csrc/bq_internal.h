// Internal launchers behind the C ABI (include/bq.h).  Every launcher takes
// already validated arguments and enqueues work on `stream`; it returns the
// CUDA error of the launch.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "bq.h"

namespace bq {

// Streaming multiprocessors of the current device.
int sm_count();
// Time limit of bounded device-side waits (nanoseconds).
int64_t wait_timeout_ns();
// Address (on the current device) of the status word the bounded waits write.
cudaError_t device_status_ptr(int** out);
// Synchronise the device, read the status word and optionally clear it.
cudaError_t read_device_status(int* status_out, bool reset);

cudaError_t launch_quantize(const void* x, int xtype, int64_t rows, int64_t cols, int64_t ld_x, int bits,
                            int mode, int8_t* q, uint16_t* scale, cudaStream_t stream);

// Per-row int8 scales (D = 127) of an fp16 matrix with contiguous rows of
// `cols` elements (cols % 8 == 0): the scales bq_quantize_sym would store.
cudaError_t launch_row_scale_f16(const void* x, int64_t rows, int64_t cols, uint16_t* scale, cudaStream_t stream);

// fp32 row sums of an fp16 matrix with contiguous rows of `cols` elements
// (cols % 8 == 0), each summed in a fixed order.
cudaError_t launch_row_sum_f16(const void* x, int64_t rows, int64_t cols, float* sum, cudaStream_t stream);

cudaError_t launch_pack(const int8_t* q, int64_t n, int64_t k, int bits, int layout, uint8_t* packed,
                        cudaStream_t stream);

// Device status recorded by a failed internal self-check (a library defect,
// not a caller error): an output span outside the output's bounds.
constexpr int BQ_DIAG_RANGE = 64;

// Epilogue kinds shared by the GEMM kernels.
enum EpiKind : int { EPI_I32 = 0, EPI_F16_COL = 1, EPI_F16_ROWCOL = 2 };
// Activation operand kinds: int8 codes; fp16 values multiplied as fp16; fp16
// values quantised per row to int8 codes inside the GEMM (with the row scales
// passed as row_scale, already computed).
enum ActKind : int { ACT_I8 = 0, ACT_F16 = 1, ACT_Q8 = 2 };

struct GemmArgs {
  const void* a;          // activations (M, K): int8 or fp16
  const void* b;          // weights (N, K): int8 or packed 4/2-bit
  int act;                // ActKind
  int bbits;              // 8, 4, 2
  int layout;             // bq_layout of b (sub-byte only)
  int64_t M, N, K;
  const uint16_t* row_scale;  // fp16 (M) or null
  const uint16_t* col_scale;  // fp16 (N) or null
  int epi;                // EpiKind
  void* c;                // int32 or fp16 (M, N)
  int actfn = BQ_ACT_NONE;  // bq_activation applied before the fp16 rounding
  // 4-bit weights with a zero point (fp16 activations only): the weights are
  // unsigned codes u, zero_point is fp16 (N) and row_sum holds the fp32 row
  // sums of the activations; the epilogue adds (8 - z[j]) * row_sum[i] to the
  // accumulated sum over x * (u - 8) before the column scale.
  const uint16_t* zero_point = nullptr;
  const float* row_sum = nullptr;
  // Batched launch on the CTA-pair kernel (grid z = item): byte strides
  // between items (0 broadcasts an operand); batch 1 is an ordinary call.
  int64_t batch = 1;
  int64_t sa = 0, sb = 0, srs = 0, scs = 0, sc = 0;
};

// The epilogue argument the GEMM kernels take: the EpiKind in bits 0-3 and
// the bq_activation above them (each kernel splits it on entry).
inline int epi_arg(const GemmArgs& g) { return g.epi | (g.actfn << 4); }

// Raise a kernel's dynamic shared-memory limit once per (device, kernel), so
// that later launches make no attribute call (e.g. inside a stream capture).
cudaError_t set_smem_once_ptr(const void* kern, int bytes);

template <typename Kernel>
cudaError_t set_smem_once(Kernel kern, int bytes) {
  return set_smem_once_ptr(reinterpret_cast<const void*>(kern), bytes);
}

// Skinny-M path (M <= 16): one pass over the weights, legacy mma.sync fp16.
// gemv_fits tells whether its staged activations fit in shared memory.
bool gemv_fits(int64_t M, int64_t K, int bbits);
// The same for fp16 x 4-bit weights with zero points (bulk variant only).
bool gemv_zp_fits(int64_t M, int64_t K);
cudaError_t launch_gemv_mma(const GemmArgs& g, cudaStream_t stream);
// int8 x int8 with exact int32 dp4a accumulation (any M).
cudaError_t launch_gemm_dp4a(const GemmArgs& g, cudaStream_t stream);
// Tensor-core (tcgen05) GEMM for larger M.
cudaError_t launch_gemm_tc(const GemmArgs& g, cudaStream_t stream);
// Whether launch_gemm_tc has an exact configuration for int8 x int8 (CTA
// pairs with chunked accumulation, or single-CTA chains of <= 16 k-blocks).
bool gemm_tc_i8_exact(const GemmArgs& g);
// CTA-pair tensor-core kernel (int8 activations): the tile width it would use
// for this problem, or 0 when the single-CTA kernel is the better fit.
int gemm_pair_bn(const GemmArgs& g);
cudaError_t launch_gemm_pair(const GemmArgs& g, int bn, cudaStream_t stream);
// Small-M tensor-core kernel with the weights as the MMA's A operand.
constexpr bool SWAP_ENABLED = true;
bool gemm_swap_applies(const GemmArgs& g);
cudaError_t launch_gemm_swap(const GemmArgs& g, cudaStream_t stream);

}  // namespace bq
