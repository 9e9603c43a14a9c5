/*
 * bq.h -- C ABI of the quantized mixed-precision GEMM library (libbq.so).
 *
 * One GB300 (sm_103a).  Every entry point takes plain pointers and sizes,
 * launches asynchronously on the caller's CUDA stream, allocates nothing,
 * and returns a bq_status.  Arguments are validated on the host before any
 * launch; an invalid call returns an error code and launches nothing.
 *
 * Conventions shared by all calls
 *   - Pointers named x, q, scale, A, B, Bp, Wp, C, X, Y and *_scale are DEVICE
 *     pointers owned by the caller; the library never frees or retains them.
 *   - Matrices are row-major and contiguous unless a leading dimension is
 *     given.  Weights are stored "NT": B is (N, K) and every GEMM contracts
 *     the K axis of both operands, C[i, j] = sum_k A[i, k] * B[j, k].
 *   - fp16 values travel as uint16_t bit patterns (IEEE binary16).
 *   - stream is a cudaStream_t (NULL = the legacy default stream).
 *   - Pointers must be 16-byte aligned (BQ_ERR_ALIGNMENT otherwise).
 *   - M, N or rows == 0 is a valid empty call (BQ_OK, nothing launched).
 *
 * Pages followed (by title and section):
 *   [BitBLAS] "BitBLAS自定义操作开发指南：使用DSL扩展新的混合精度算子",
 *             sections 混合精度算子开发实战 1 (INT8 x INT4, int32 accumulation),
 *             2 添加反量化支持 (per-column fp16 dequantisation), 实际应用案例
 *             案例1 (INT8 x INT2) and 案例2 (fp16 x 4-bit, fp32 accumulation),
 *             高级功能 动态形状支持 (dynamic M in [1, 1024]).
 *   [BMINF]   "BMINF的後訓練量化實現", section 實現代碼分析2 (quantize:
 *             fp16 scale = absmax / 127, codes = nearbyint(x / scale);
 *             elementwise_copy_scale: int32 * w_scale * x_scale -> fp16;
 *             igemm: int8 x int8 -> int32).
 *   [Pallas]  "JAX Pallas 在 TPU 上编写高效矩阵乘法内核：从分块算法、性能建模到
 *             算子融合", section 模板化矩阵乘法 / 融合激活函数 (the activation
 *             acts on the f32 result of the last step, before the one downcast).
 *   [DISC]    "全面支持 PyTorch 2.0：BladeDISC 5 月~11 月新功能发布", section
 *             Ongoing Work / CUTLASS Gemm CodeGen (GEMM + GELU fusion).
 */
#ifndef BQ_H_
#define BQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bq_status {
  BQ_OK = 0,
  BQ_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad enum value      */
  BQ_ERR_UNSUPPORTED = 2, /* valid but outside the supported shapes / ranges  */
  BQ_ERR_ALIGNMENT = 3,   /* a pointer or leading dimension is misaligned     */
  BQ_ERR_CUDA = 4,        /* the CUDA runtime reported an error at launch     */
  BQ_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (see below)   */
} bq_status;

typedef enum bq_ftype { BQ_F16 = 0, BQ_F32 = 1 } bq_ftype;
typedef enum bq_layout { BQ_LAYOUT_PLAIN = 0, BQ_LAYOUT_INTERLEAVED = 1 } bq_layout;
typedef enum bq_round { BQ_ROUND_F32DIV = 0, BQ_ROUND_BMINF_HALF = 1 } bq_round;
typedef enum bq_activation { BQ_ACT_NONE = 0, BQ_ACT_RELU = 1, BQ_ACT_GELU = 2 } bq_activation;

/* Human-readable name of a status code (static string, never NULL). */
const char* bq_status_string(int status);

/*
 * bq_quantize_sym -- symmetric per-row quantisation, one fused pass.
 *   [BMINF 實現代碼分析2, PartialAttention.quantize and its quantize()]
 *
 *   scale[r] = fp16_rne( max_c |x[r, c]| / D )        D = 127, 7, 1 for bits 8, 4, 2
 *   q[r, c]  = clamp( rne( x[r, c] / float(scale[r]) ), -D, D )
 *
 *   The division producing the scale is IEEE fp32 and is rounded once to
 *   fp16; codes are computed from the stored fp16 scale.  mode
 *   BQ_ROUND_F32DIV rounds the fp32 quotient to the nearest integer (ties to
 *   even); BQ_ROUND_BMINF_HALF first rounds the quotient to fp16, as the
 *   page's quantize_copy_half does.  A row whose scale is 0 (all zeros, or an
 *   absmax so small that absmax / D underflows fp16) gets all-zero codes.
 *   NaN / Inf inputs are not supported.
 *
 *   x      device, xtype elements, rows x cols with leading dimension ld_x
 *          (elements, ld_x >= cols)
 *   q      device int8, rows x cols, leading dimension cols (one code per byte;
 *          pack 4- and 2-bit codes with bq_pack_weights)
 *   scale  device fp16, rows
 *   Errors: INVALID_ARG (null, negative sizes, ld_x < cols, bits not 8/4/2,
 *   bad xtype/mode), ALIGNMENT (x, q or scale not 16-byte aligned),
 *   UNSUPPORTED (cols > 1 << 24), CUDA.
 */
bq_status bq_quantize_sym(const void* x, int xtype, int64_t rows, int64_t cols, int64_t ld_x,
                          int bits, int mode, int8_t* q, uint16_t* scale, void* stream);

/*
 * bq_packed_size -- bytes of the packed (n, k) code matrix: n * k * bits / 8.
 *   Returns 0 for invalid arguments (bits not 8/4/2, negative sizes, or
 *   k * bits not a multiple of 32 for the interleaved layout / 8 for plain).
 */
size_t bq_packed_size(int64_t n, int64_t k, int bits, int layout);

/*
 * bq_pack_weights -- pack int8 codes (n, k) into sub-byte storage.
 *   [BitBLAS 案例2 stores 4-bit weights as (N, K // 2) uint8]
 *
 *   Row r of the output occupies k * bits / 8 consecutive bytes.  Each code
 *   contributes its low `bits` bits (two's complement).
 *   BQ_LAYOUT_PLAIN: element k sits in byte k * bits / 8 at bit offset
 *     (k mod (8 / bits)) * bits -- the lowest k in the lowest bits (for 4 bits:
 *     low nibble = even k).
 *   BQ_LAYOUT_INTERLEAVED: the plain row cut into 32-bit little-endian words
 *     (8 elements per word for 4 bits, 16 for 2 bits), and inside each word
 *     the even-indexed elements fill the low 16 bits in order and the odd-
 *     indexed elements the high 16 bits in order.  One mask per 16-bit half
 *     then yields the consecutive pair (k, k+1) -- the layout the GEMM
 *     kernels convert from without shuffles.  For 8 bits both layouts are
 *     the plain int8 matrix.
 *   q       device int8, n x k (leading dimension k)
 *   packed  device, bq_packed_size(n, k, bits, layout) bytes
 *   Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED (k not a multiple of 32 / bits
 *   for the interleaved layout, of 8 / bits for plain), CUDA.
 */
bq_status bq_pack_weights(const int8_t* q, int64_t n, int64_t k, int bits, int layout,
                          uint8_t* packed, void* stream);

/*
 * Integer GEMMs with int32 accumulation and an optional fused dequantisation.
 *   [BitBLAS 混合精度算子开发实战 1 and 2; 案例1; BMINF igemm and
 *    elementwise_copy_scale]
 *
 *   Cint[i, j] = sum_k int(A[i, k]) * int(B[j, k])        (exact, on every path)
 *   If row_scale == NULL and col_scale == NULL:  C is int32 (M, N), C = Cint.
 *   Otherwise C is fp16 (M, N):
 *     C[i, j] = fp16_rne( float(Cint[i, j]) * float(col_scale[j]) [* float(row_scale[i])] )
 *   evaluated as IEEE fp32 products in that order (a missing scale is
 *   omitted).  row_scale given without col_scale is INVALID_ARG.
 *
 *   A          device int8 (M, K), leading dimension K
 *   B / Bp     device: int8 (N, K) for i8xi8; packed 4-bit / 2-bit codes
 *              (bq_pack_weights layout `layout`) for i8xi4 / i8xi2
 *   row_scale  device fp16 (M) or NULL;  col_scale device fp16 (N) or NULL
 *   C          device int32 or fp16 (M, N), leading dimension N
 *   Limits (UNSUPPORTED otherwise): K % 64 == 0, N % 64 == 0, K <= 65536;
 *   i8xi4 additionally needs K <= 16384 (|a * b| <= 1024, so every partial
 *   sum stays within 2**24 and the fp32 tensor-core accumulation is exact;
 *   for i8xi2 |a * b| <= 256 and K <= 65536 already guarantees that).
 *   With K == 0 the output is all zeros and A / B may be NULL.
 *   The tensor cores multiply exact fp16 images of the codes into fp32
 *   accumulators, which hold integers exactly up to 2**24: every fp32 chain
 *   is kept within that bound, so the fp16 epilogue starts from the exact
 *   Cint as well.  int8 x int8 products reach 2**14, so its fresh chains
 *   are at most 1024 k long: CTA pairs cut K into chunks of 16 k-blocks and
 *   drain each finished chunk's accumulator while the next chunk runs (its
 *   high part collects as an integer in the output's own bytes before the
 *   epilogue overwrites them; the remainder, in (-8192, 0], stays in the
 *   accumulator under the chunk after next), the single-CTA kernel uses
 *   separate TMEM slices or split-K ranges of at most 16 k-blocks summed as
 *   integers.
 *   Any M >= 0.  Dispatch: M <= 16 runs the skinny kernel (one pass over the
 *   weights; int8 x int8 uses an exact dp4a kernel there), larger M the
 *   tensor-core GEMM: 256-row tiles on CTA pairs when the grid fills the GPU,
 *   128-row tiles with K split over a cluster otherwise.  int8 x int8 shapes
 *   with no exact tensor-core configuration (fp16 output with K > 8192 on
 *   CTA pairs, K > 4096 on grids smaller than the GPU) run the dp4a kernel.
 *   Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED, CUDA.
 */
bq_status bq_gemm_i8xi8(const int8_t* A, const int8_t* B, int64_t M, int64_t N, int64_t K,
                        const uint16_t* row_scale, const uint16_t* col_scale, void* C,
                        void* stream);
bq_status bq_gemm_i8xi4(const int8_t* A, const uint8_t* Bp, int layout, int64_t M, int64_t N,
                        int64_t K, const uint16_t* row_scale, const uint16_t* col_scale, void* C,
                        void* stream);
bq_status bq_gemm_i8xi2(const int8_t* A, const uint8_t* Bp, int layout, int64_t M, int64_t N,
                        int64_t K, const uint16_t* row_scale, const uint16_t* col_scale, void* C,
                        void* stream);

/*
 * bq_gemm_f16xi4 -- fp16 activations times 4-bit weights, fp32 accumulation.
 *   [BitBLAS 案例2 (fp16 x dequantised 4-bit, fp32 accumulate) and
 *    高级功能 动态形状支持 (M dynamic in [1, 1024])]
 *
 *   Y[i, j] = fp16_rne( float(col_scale[j]) * sum_k float(X[i, k]) * q[j, k] )
 *   The per-channel scale is applied once, after the accumulation.
 *   X          device fp16 (M, K), leading dimension K
 *   Wp         device packed 4-bit codes (N, K) in layout `layout`
 *   col_scale  device fp16 (N), required
 *   Y          device fp16 (M, N)
 *   Limits: K % 64 == 0, N % 64 == 0, K <= 65536 (UNSUPPORTED otherwise).
 *   Dispatch: M <= 16 runs the skinny kernel, 16 < M <= 128 a tensor-core
 *   kernel with the weights as the MMA's A operand, larger M the tensor-core
 *   GEMM on CTA pairs (or with K split over a cluster for small grids).
 *   Errors: INVALID_ARG, ALIGNMENT, UNSUPPORTED, CUDA.
 */
bq_status bq_gemm_f16xi4(const uint16_t* X, const uint8_t* Wp, int layout, int64_t M, int64_t N,
                         int64_t K, const uint16_t* col_scale, uint16_t* Y, void* stream);

/*
 * GEMMs with a fused activation epilogue.  [Pallas 融合激活函数; DISC GEMM +
 * GELU]
 *
 *   Same operands, limits, dispatch and errors as the call without "_act";
 *   the output must be fp16 (col_scale required).  The activation acts on
 *   the fp32 dequantised value v (after every scale product) and the result
 *   is rounded once to fp16:
 *     C[i, j] = fp16_rne( act(v[i, j]) )
 *   activation  BQ_ACT_NONE  act(v) = v
 *               BQ_ACT_RELU  act(v) = max(v, 0)
 *               BQ_ACT_GELU  act(v) = v * Phi(v) = 0.5 * v * erfc(-v / sqrt(2))
 *                            (the erf form; evaluated in fp32 with erfcf, which
 *                            has no cancellation for negative v)
 *   Errors: INVALID_ARG also for an unknown activation or a NULL col_scale.
 */
bq_status bq_gemm_i8xi8_act(const int8_t* A, const int8_t* B, int64_t M, int64_t N, int64_t K,
                            const uint16_t* row_scale, const uint16_t* col_scale, int activation,
                            void* C, void* stream);
bq_status bq_gemm_i8xi4_act(const int8_t* A, const uint8_t* Bp, int layout, int64_t M, int64_t N,
                            int64_t K, const uint16_t* row_scale, const uint16_t* col_scale,
                            int activation, void* C, void* stream);
bq_status bq_gemm_i8xi2_act(const int8_t* A, const uint8_t* Bp, int layout, int64_t M, int64_t N,
                            int64_t K, const uint16_t* row_scale, const uint16_t* col_scale,
                            int activation, void* C, void* stream);
bq_status bq_gemm_f16xi4_act(const uint16_t* X, const uint8_t* Wp, int layout, int64_t M, int64_t N,
                             int64_t K, const uint16_t* col_scale, int activation, uint16_t* Y,
                             void* stream);

/*
 * Batched GEMMs with broadcast operands.  [BMINF 實現代碼分析2: igemm takes
 * (batch, rows, k) operands, and an operand whose batch is 1 is shared by
 * every item (stride 0); the fused QKV projection multiplies one block of
 * activations by the three stacked weight matrices, w_project_qkv (3, N, K)]
 *
 *   For every b in [0, batch):
 *     C + b*stride_c = the unbatched call on A + b*stride_a, B + b*stride_b,
 *                      row_scale + b*stride_rs, col_scale + b*stride_cs
 *   with that call's semantics, limits, dispatch and activation.  Strides
 *   count elements of each array (bytes for packed weights); a stride of 0
 *   broadcasts the operand.  stride_c must be at least M * N when batch > 1
 *   (outputs never overlap).  Every item's pointers must be 16-byte aligned,
 *   i.e. aligned bases and strides whose byte size is a multiple of 16.
 *   All items are validated before the first launch; they are launched in
 *   order on `stream`, one after another.
 *   Errors: as the unbatched call; INVALID_ARG also for batch < 0, a
 *   negative stride or overlapping outputs.
 */
bq_status bq_gemm_i8xi8_batched(const int8_t* A, int64_t stride_a, const int8_t* B, int64_t stride_b,
                                int64_t batch, int64_t M, int64_t N, int64_t K,
                                const uint16_t* row_scale, int64_t stride_rs, const uint16_t* col_scale,
                                int64_t stride_cs, int activation, void* C, int64_t stride_c, void* stream);
bq_status bq_gemm_i8xi4_batched(const int8_t* A, int64_t stride_a, const uint8_t* Bp, int64_t stride_b,
                                int layout, int64_t batch, int64_t M, int64_t N, int64_t K,
                                const uint16_t* row_scale, int64_t stride_rs, const uint16_t* col_scale,
                                int64_t stride_cs, int activation, void* C, int64_t stride_c, void* stream);
bq_status bq_gemm_i8xi2_batched(const int8_t* A, int64_t stride_a, const uint8_t* Bp, int64_t stride_b,
                                int layout, int64_t batch, int64_t M, int64_t N, int64_t K,
                                const uint16_t* row_scale, int64_t stride_rs, const uint16_t* col_scale,
                                int64_t stride_cs, int activation, void* C, int64_t stride_c, void* stream);
bq_status bq_gemm_f16xi4_batched(const uint16_t* X, int64_t stride_x, const uint8_t* Wp, int64_t stride_w,
                                 int layout, int64_t batch, int64_t M, int64_t N, int64_t K,
                                 const uint16_t* col_scale, int64_t stride_cs, int activation, uint16_t* Y,
                                 int64_t stride_y, void* stream);

/*
 * bq_quantized_linear -- the quantised linear layer with fp16 activations:
 * per-row int8 quantisation of X, the integer GEMM against pre-quantised
 * weights and the two-scale dequantisation, with no int8 copy of X in memory.
 *   [BMINF 實現代碼分析2: one decode step runs quantize(h) -> igemm ->
 *   elementwise_copy_scale; Pallas 小结与实践路线: fusing the input's
 *   preprocessing into the matrix-multiply kernel]
 *
 *   x_scale[i] = fp16_rne( max_k |X[i, k]| / 127 )
 *   q[i, k]    = the bq_quantize_sym codes (bits 8, BQ_ROUND_F32DIV) of X
 *   Y[i, j]    = fp16_rne( act( fp32( fp32( float(Cint[i, j]) * float(w_scale[j]) )
 *                                      * float(x_scale[i]) ) ) )
 *   Cint[i, j] = sum_k q[i, k] * W[j, k]   (exact)
 *   So x_scale equals bq_quantize_sym's scale and Y equals bq_gemm_*_act on
 *   its codes with row_scale = x_scale and col_scale = w_scale, bit for bit.
 *
 *   X        device fp16, M x K, contiguous rows (read twice: a pass for the
 *            row scales, then by the GEMM, which quantises each tile of X as
 *            it converts it for the tensor cores)
 *   W        device weights (N, K): int8 codes (bits 8) or packed 4- / 2-bit
 *            codes in `layout` (bq_pack_weights), N * K * bits / 8 bytes
 *   w_scale  device fp16, N (per output column)
 *   x_scale  device fp16, M: OUTPUT, the activation scales
 *   Y        device fp16, M x N: OUTPUT
 *   activation  a bq_activation, as in the "_act" calls
 *   M == 0 is an empty call.  N == 0 still writes x_scale; K == 0 writes
 *   x_scale = 0 and Y = 0.
 *   Limits: K % 64 == 0, N % 64 == 0; K <= 8192 (bits 8), 16384 (4), 65536
 *   (2).  Runs on the tensor-core kernels for every M (CTA pairs, or K split
 *   over a cluster for grids smaller than the GPU).  int8 weights with
 *   K > 4096 need every fp32 chain to stay exact: K split 8 ways into ranges
 *   of at most 1024 (grids of at most 18 tiles of 128 x 256) or CTA pairs
 *   with chunked accumulation (grids that fill the GPU); the shapes between
 *   return UNSUPPORTED.
 *   Errors: INVALID_ARG (null pointers where data is needed, negative sizes,
 *   bits not 8/4/2, bad layout or activation), ALIGNMENT (any pointer not
 *   16-byte aligned), UNSUPPORTED, CUDA.
 */
bq_status bq_quantized_linear(const uint16_t* X, int64_t M, int64_t K, const void* W, int bits, int layout,
                              int64_t N, const uint16_t* w_scale, int activation, uint16_t* x_scale,
                              uint16_t* Y, void* stream);

/*
 * bq_gemm_f16xu4_zp -- fp16 activations times 4-bit weights with a per-column
 * scale and zero point.  [BitBLAS 实际应用案例 案例2: fp16 A (M, K), packed
 * weights (N, K // 2) uint8, scale (N,) and zero_point (N,) fp16, fp32
 * accumulation of the products with the dequantised weights]
 *
 *   w[j, k]  = col_scale[j] * (u[j, k] - zero_point[j])   u in [0, 15] unsigned
 *   Y[i, j]  = fp16_rne( act( sum_k X[i, k] * w[j, k] ) )
 *   The codes u are packed like the signed 4-bit codes (bq_pack_weights of
 *   the values 0..15, either layout); zero_point need not be an integer.
 *   Evaluated as col_scale[j] * (S[i, j] + (8 - zero_point[j]) * row_sum[i])
 *   with S the fp32 sum over X * (u - 8) of the fp16 x int4 kernels (the
 *   same chains) and the activation applied to that fp32 value.
 *
 *   X          device fp16, M x K
 *   Wp         device packed unsigned 4-bit codes, N x K / 2 bytes
 *   col_scale, zero_point  device fp16, N
 *   row_sum    device fp32, M: OUTPUT, row_sum[i] = sum_k X[i, k] in fp32
 *              (a fixed order), used by the epilogue (M <= 16: formed inside
 *              the skinny kernel, no extra launch)
 *   Y          device fp16, M x N: OUTPUT
 *   Limits: K % 64 == 0, N % 64 == 0, K <= 65536.  Dispatch as bq_gemm_f16xi4
 *   (M <= 16 the skinny kernel while 16 staged weight rows fit in 64 KB,
 *   16 < M <= 128 the kernel with the weights as the MMA's A operand, else
 *   the CTA-pair or split-K tensor-core kernels).  M == 0 is an empty call;
 *   N == 0 still writes row_sum.
 *   Errors: INVALID_ARG (null pointers, bad layout or activation),
 *   ALIGNMENT, UNSUPPORTED, CUDA.
 */
bq_status bq_gemm_f16xu4_zp(const uint16_t* X, const uint8_t* Wp, int layout, int64_t M, int64_t N, int64_t K,
                            const uint16_t* col_scale, const uint16_t* zero_point, int activation, float* row_sum,
                            uint16_t* Y, void* stream);

/*
 * Device-side wait status.  Every wait inside the tensor-core kernels and the
 * skinny kernel (on a shared-memory mbarrier) is bounded in time.  A wait that gives up records
 * BQ_ERR_TIMEOUT in a device status word, abandons the tile, waits (again
 * bounded) for the tensor-core work it issued, frees its tensor memory and
 * returns, leaving the CUDA context usable.  The launch itself still
 * reports BQ_OK because it is asynchronous.
 *
 * bq_device_status: synchronises the device, returns the recorded status in
 *   *status_out (BQ_OK if none) and clears it when reset != 0.  A value of
 *   64 records a failed internal self-check (an output span outside the
 *   output, skipped rather than accessed): a library defect, not a caller
 *   error.
 * bq_set_wait_timeout_ns: sets the time limit of those waits for later
 *   launches (default 2 s).  Returns the previous value.  Intended for tests
 *   that make a wait run out: with a limit of 0 every wait whose phase has
 *   not completed at its first (non-blocking) poll gives up.
 */
bq_status bq_device_status(int* status_out, int reset);
int64_t bq_set_wait_timeout_ns(int64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* BQ_H_ */
