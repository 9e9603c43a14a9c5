// C ABI of libbq.so (declared in include/bq.h): host-side validation and the
// M-bucket dispatch between the skinny-M kernels and the tensor-core GEMM.
// Nothing here allocates device memory.
#include <atomic>
#include <cstdint>

#include "bq_internal.h"

namespace bq {

namespace {
std::atomic<int64_t> g_wait_timeout_ns{2000000000LL};

constexpr int64_t MAX_K = 65536;
constexpr int64_t MAX_DIM = 1LL << 24;
constexpr int64_t SKINNY_M = 16;
constexpr int64_t MAX_STRIDE = 1LL << 46;   // bytes; with MAX_BATCH, every item offset stays below 2**62
constexpr int64_t MAX_BATCH = 1LL << 16;

// A stride in elements as bytes: negative stays negative (rejected), a huge
// one saturates above MAX_STRIDE (rejected) instead of overflowing.
inline int64_t stride_bytes(int64_t s, int64_t elem) {
  if (s < 0) return -1;
  return s > MAX_STRIDE ? MAX_STRIDE + 16 : s * elem;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bq_status from_cuda(cudaError_t e) { return e == cudaSuccess ? BQ_OK : BQ_ERR_CUDA; }

inline bool valid_bits(int bits) { return bits == 8 || bits == 4 || bits == 2; }

inline bool valid_layout(int layout) { return layout == BQ_LAYOUT_PLAIN || layout == BQ_LAYOUT_INTERLEAVED; }

// An activation needs the fp16 output (col_scale given); NONE is always valid.
inline bool valid_activation(int activation, const void* col_scale) {
  if (activation == BQ_ACT_NONE) return true;
  return (activation == BQ_ACT_RELU || activation == BQ_ACT_GELU) && col_scale != nullptr;
}

// Shared checks of the GEMM entry points.  max_k bounds K so that every
// partial sum of the integer paths stays below 2**24 (exact fp32 accumulation).
bq_status check_gemm(const void* a, const void* b, int64_t M, int64_t N, int64_t K, const void* row_scale,
                     const void* col_scale, const void* c, int64_t max_k) {
  if (M < 0 || N < 0 || K < 0) return BQ_ERR_INVALID_ARG;
  if (row_scale && !col_scale) return BQ_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return BQ_OK;
  // with K == 0 the operands hold no elements and may be null
  if (!c || (K > 0 && (!a || !b))) return BQ_ERR_INVALID_ARG;
  if (K % 64 != 0 || N % 64 != 0 || K > max_k || M > MAX_DIM || N > MAX_DIM) return BQ_ERR_UNSUPPORTED;
  if (!aligned16(c) || (K > 0 && (!aligned16(a) || !aligned16(b)))) return BQ_ERR_ALIGNMENT;
  if ((row_scale && !aligned16(row_scale)) || (col_scale && !aligned16(col_scale))) return BQ_ERR_ALIGNMENT;
  return BQ_OK;
}

bq_status run_gemm(GemmArgs g, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (g.M == 0 || g.N == 0) return BQ_OK;
  g.epi = g.col_scale ? (g.row_scale ? EPI_F16_ROWCOL : EPI_F16_COL) : EPI_I32;
  if (g.K == 0) {
    const size_t bytes = (size_t)g.M * (size_t)g.N * (g.epi == EPI_I32 ? 4 : 2);
    return from_cuda(cudaMemsetAsync(g.c, 0, bytes, s));
  }
  cudaError_t e;
  if (g.act == ACT_Q8) {
    // fp16 activations quantised inside the GEMM: the tensor-core kernels only
    e = launch_gemm_tc(g, s);
  } else if (g.zero_point) {
    // 4-bit weights with a zero point: the same M buckets as fp16 x int4
    if (g.M <= SKINNY_M && gemv_zp_fits(g.M, g.K)) e = launch_gemv_mma(g, s);
    else if (gemm_swap_applies(g)) e = launch_gemm_swap(g, s);
    else e = launch_gemm_tc(g, s);
  } else if (g.act == ACT_I8 && g.bbits == 8) {
    // skinny M, and shapes with no exact tensor-core configuration, use dp4a
    const bool tc_ok = g.M > SKINNY_M && gemm_tc_i8_exact(g);
    e = tc_ok ? launch_gemm_tc(g, s) : launch_gemm_dp4a(g, s);
  } else if (gemm_swap_applies(g)) {
    e = launch_gemm_swap(g, s);
  } else if (g.M <= SKINNY_M && gemv_fits(g.M, g.K, g.bbits)) {
    e = launch_gemv_mma(g, s);
  } else {
    e = launch_gemm_tc(g, s);
  }
  return from_cuda(e);
}

// Whether run_gemm sends this (unbatched) problem, its epilogue kind already
// set, to the CTA-pair kernel.
bool routes_to_pair(const GemmArgs& g) {
  if (g.act == ACT_Q8 || g.zero_point || g.M <= 0 || g.N <= 0 || g.K <= 0) return false;
  if (g.act == ACT_I8 && g.bbits == 8) return g.M > SKINNY_M && gemm_pair_bn(g) != 0;
  if (gemm_swap_applies(g)) return false;
  if (g.M <= SKINNY_M && gemv_fits(g.M, g.K, g.bbits)) return false;
  return gemm_pair_bn(g) != 0;
}

// Batched calls: item b uses every pointer advanced by b times its stride
// (in bytes here; 0 broadcasts).  Validates once for all items -- the items
// differ from the first only by offsets that are multiples of 16 bytes --
// then launches them: as one grid on the CTA-pair kernel where that kernel
// serves the shape, else one after another.
bq_status run_batched(const GemmArgs& g, int64_t batch, int64_t sa, int64_t sb, int64_t srs, int64_t scs,
                      int64_t sc, int64_t max_k, void* stream) {
  if (batch < 0 || sa < 0 || sb < 0 || srs < 0 || scs < 0 || sc < 0) return BQ_ERR_INVALID_ARG;
  if (batch == 0) return BQ_OK;
  bq_status st = check_gemm(g.a, g.b, g.M, g.N, g.K, g.row_scale, g.col_scale, g.c, max_k);
  if (st != BQ_OK) return st;
  if (g.M == 0 || g.N == 0) return BQ_OK;
  if (batch > 1) {
    const int64_t out_bytes = g.M * g.N * (g.col_scale ? 2 : 4);
    if (sc < out_bytes) return BQ_ERR_INVALID_ARG;   // outputs would overlap
    if ((sa | sb | srs | scs | sc) % 16 != 0) return BQ_ERR_ALIGNMENT;
    if (sa > MAX_STRIDE || sb > MAX_STRIDE || srs > MAX_STRIDE || scs > MAX_STRIDE || sc > MAX_STRIDE ||
        batch > MAX_BATCH)
      return BQ_ERR_UNSUPPORTED;
  }
  // Items that run on the CTA-pair kernel share one launch (grid z = item) when
  // every strided operand's items do not overlap (3-D tensor maps).
  GemmArgs gb = g;
  gb.epi = g.col_scale ? (g.row_scale ? EPI_F16_ROWCOL : EPI_F16_COL) : EPI_I32;
  if (batch > 1 && g.K > 0 && routes_to_pair(gb)) {
    const int64_t a_bytes = g.M * g.K * (g.act == ACT_F16 ? 2 : 1);
    const int64_t b_bytes = g.N * g.K * g.bbits / 8;
    if ((sa == 0 || sa >= a_bytes) && (sb == 0 || sb >= b_bytes)) {
      gb.batch = batch;
      gb.sa = sa;
      gb.sb = sb;
      gb.srs = g.row_scale ? srs : 0;
      gb.scs = g.col_scale ? scs : 0;
      gb.sc = sc;
      return from_cuda(launch_gemm_pair(gb, gemm_pair_bn(gb), static_cast<cudaStream_t>(stream)));
    }
  }
  for (int64_t b = 0; b < batch; ++b) {
    GemmArgs gi = g;
    gi.a = static_cast<const uint8_t*>(g.a) + b * sa;
    gi.b = static_cast<const uint8_t*>(g.b) + b * sb;
    if (g.row_scale) gi.row_scale = reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(g.row_scale) + b * srs);
    if (g.col_scale) gi.col_scale = reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(g.col_scale) + b * scs);
    gi.c = static_cast<uint8_t*>(g.c) + b * sc;
    st = run_gemm(gi, stream);
    if (st != BQ_OK) return st;
  }
  return BQ_OK;
}

}  // namespace

int64_t wait_timeout_ns() { return g_wait_timeout_ns.load(); }

cudaError_t set_smem_once_ptr(const void* kern, int bytes) {
  struct Entry {
    const void* kern;
    int dev;
    int bytes;
  };
  static Entry table[256];
  static std::atomic<int> used{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int n = used.load();
  for (int i = 0; i < n && i < 256; ++i)
    if (table[i].kern == kern && table[i].dev == dev && table[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  const int slot = used.fetch_add(1);
  if (slot < 256) table[slot] = Entry{kern, dev, bytes};
  return cudaSuccess;
}

}  // namespace bq

using namespace bq;

extern "C" {

const char* bq_status_string(int status) {
  switch (status) {
    case BQ_OK: return "BQ_OK";
    case BQ_ERR_INVALID_ARG: return "BQ_ERR_INVALID_ARG";
    case BQ_ERR_UNSUPPORTED: return "BQ_ERR_UNSUPPORTED";
    case BQ_ERR_ALIGNMENT: return "BQ_ERR_ALIGNMENT";
    case BQ_ERR_CUDA: return "BQ_ERR_CUDA";
    case BQ_ERR_TIMEOUT: return "BQ_ERR_TIMEOUT";
    default: return "BQ_ERR_UNKNOWN";
  }
}

bq_status bq_quantize_sym(const void* x, int xtype, int64_t rows, int64_t cols, int64_t ld_x, int bits, int mode,
                          int8_t* q, uint16_t* scale, void* stream) {
  if (rows < 0 || cols < 0 || ld_x < cols) return BQ_ERR_INVALID_ARG;
  if (!valid_bits(bits) || (xtype != BQ_F16 && xtype != BQ_F32)) return BQ_ERR_INVALID_ARG;
  if (mode != BQ_ROUND_F32DIV && mode != BQ_ROUND_BMINF_HALF) return BQ_ERR_INVALID_ARG;
  if (rows == 0) return BQ_OK;
  if (!x || !q || !scale) return BQ_ERR_INVALID_ARG;
  if (cols > MAX_DIM || rows > (1LL << 31) - 1) return BQ_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(q) || !aligned16(scale)) return BQ_ERR_ALIGNMENT;
  return from_cuda(launch_quantize(x, xtype, rows, cols, ld_x, bits, mode, q, scale,
                                   static_cast<cudaStream_t>(stream)));
}

size_t bq_packed_size(int64_t n, int64_t k, int bits, int layout) {
  if (n < 0 || k < 0 || !valid_bits(bits) || !valid_layout(layout)) return 0;
  const int64_t unit = (layout == BQ_LAYOUT_INTERLEAVED && bits != 8) ? 32 / bits : 8 / bits;
  if (k % unit != 0) return 0;
  return (size_t)n * (size_t)k * (size_t)bits / 8;
}

bq_status bq_pack_weights(const int8_t* q, int64_t n, int64_t k, int bits, int layout, uint8_t* packed,
                          void* stream) {
  if (n < 0 || k < 0 || !valid_bits(bits) || !valid_layout(layout)) return BQ_ERR_INVALID_ARG;
  if (n == 0 || k == 0) return BQ_OK;
  if (!q || !packed) return BQ_ERR_INVALID_ARG;
  if (bq_packed_size(n, k, bits, layout) == 0) return BQ_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(packed)) return BQ_ERR_ALIGNMENT;
  return from_cuda(launch_pack(q, n, k, bits, layout, packed, static_cast<cudaStream_t>(stream)));
}

bq_status bq_gemm_i8xi8(const int8_t* A, const int8_t* B, int64_t M, int64_t N, int64_t K,
                        const uint16_t* row_scale, const uint16_t* col_scale, void* C, void* stream) {
  return bq_gemm_i8xi8_act(A, B, M, N, K, row_scale, col_scale, BQ_ACT_NONE, C, stream);
}

bq_status bq_gemm_i8xi8_act(const int8_t* A, const int8_t* B, int64_t M, int64_t N, int64_t K,
                            const uint16_t* row_scale, const uint16_t* col_scale, int activation, void* C,
                            void* stream) {
  if (!valid_activation(activation, col_scale)) return BQ_ERR_INVALID_ARG;
  bq_status st = check_gemm(A, B, M, N, K, row_scale, col_scale, C, MAX_K);
  if (st != BQ_OK) return st;
  GemmArgs g{A, B, ACT_I8, 8, BQ_LAYOUT_PLAIN, M, N, K, row_scale, col_scale, EPI_I32, C, activation};
  return run_gemm(g, stream);
}

static bq_status gemm_sub_byte(const int8_t* A, const uint8_t* Bp, int layout, int bits, int64_t M, int64_t N,
                               int64_t K, const uint16_t* row_scale, const uint16_t* col_scale, int activation,
                               void* C, void* stream) {
  if (!valid_layout(layout) || !valid_activation(activation, col_scale)) return BQ_ERR_INVALID_ARG;
  // |a * b| <= 128 * 8 (4 bits) or 128 * 2 (2 bits): K <= 2**24 / that keeps sums exact
  const int64_t max_k = bits == 4 ? 16384 : MAX_K;
  bq_status st = check_gemm(A, Bp, M, N, K, row_scale, col_scale, C, max_k);
  if (st != BQ_OK) return st;
  GemmArgs g{A, Bp, ACT_I8, bits, layout, M, N, K, row_scale, col_scale, EPI_I32, C, activation};
  return run_gemm(g, stream);
}

bq_status bq_gemm_i8xi4(const int8_t* A, const uint8_t* Bp, int layout, int64_t M, int64_t N, int64_t K,
                        const uint16_t* row_scale, const uint16_t* col_scale, void* C, void* stream) {
  return gemm_sub_byte(A, Bp, layout, 4, M, N, K, row_scale, col_scale, BQ_ACT_NONE, C, stream);
}

bq_status bq_gemm_i8xi4_act(const int8_t* A, const uint8_t* Bp, int layout, int64_t M, int64_t N, int64_t K,
                            const uint16_t* row_scale, const uint16_t* col_scale, int activation, void* C,
                            void* stream) {
  return gemm_sub_byte(A, Bp, layout, 4, M, N, K, row_scale, col_scale, activation, C, stream);
}

bq_status bq_gemm_i8xi2(const int8_t* A, const uint8_t* Bp, int layout, int64_t M, int64_t N, int64_t K,
                        const uint16_t* row_scale, const uint16_t* col_scale, void* C, void* stream) {
  return gemm_sub_byte(A, Bp, layout, 2, M, N, K, row_scale, col_scale, BQ_ACT_NONE, C, stream);
}

bq_status bq_gemm_i8xi2_act(const int8_t* A, const uint8_t* Bp, int layout, int64_t M, int64_t N, int64_t K,
                            const uint16_t* row_scale, const uint16_t* col_scale, int activation, void* C,
                            void* stream) {
  return gemm_sub_byte(A, Bp, layout, 2, M, N, K, row_scale, col_scale, activation, C, stream);
}

bq_status bq_gemm_f16xi4(const uint16_t* X, const uint8_t* Wp, int layout, int64_t M, int64_t N, int64_t K,
                         const uint16_t* col_scale, uint16_t* Y, void* stream) {
  return bq_gemm_f16xi4_act(X, Wp, layout, M, N, K, col_scale, BQ_ACT_NONE, Y, stream);
}

bq_status bq_gemm_f16xi4_act(const uint16_t* X, const uint8_t* Wp, int layout, int64_t M, int64_t N, int64_t K,
                             const uint16_t* col_scale, int activation, uint16_t* Y, void* stream) {
  if (!valid_layout(layout)) return BQ_ERR_INVALID_ARG;
  if (M > 0 && N > 0 && !col_scale) return BQ_ERR_INVALID_ARG;
  if (!valid_activation(activation, col_scale)) return BQ_ERR_INVALID_ARG;
  bq_status st = check_gemm(X, Wp, M, N, K, nullptr, col_scale, Y, MAX_K);
  if (st != BQ_OK) return st;
  GemmArgs g{X, Wp, ACT_F16, 4, layout, M, N, K, nullptr, col_scale, EPI_F16_COL, Y, activation};
  return run_gemm(g, stream);
}

bq_status bq_gemm_i8xi8_batched(const int8_t* A, int64_t stride_a, const int8_t* B, int64_t stride_b, int64_t batch,
                                int64_t M, int64_t N, int64_t K, const uint16_t* row_scale, int64_t stride_rs,
                                const uint16_t* col_scale, int64_t stride_cs, int activation, void* C,
                                int64_t stride_c, void* stream) {
  if (!valid_activation(activation, col_scale)) return BQ_ERR_INVALID_ARG;
  GemmArgs g{A, B, ACT_I8, 8, BQ_LAYOUT_PLAIN, M, N, K, row_scale, col_scale, EPI_I32, C, activation};
  return run_batched(g, batch, stride_bytes(stride_a, 1), stride_bytes(stride_b, 1), stride_bytes(stride_rs, 2),
                     stride_bytes(stride_cs, 2), stride_bytes(stride_c, col_scale ? 2 : 4), MAX_K, stream);
}

static bq_status sub_byte_batched(const int8_t* A, int64_t stride_a, const uint8_t* Bp, int64_t stride_b, int layout,
                                  int bits, int64_t batch, int64_t M, int64_t N, int64_t K,
                                  const uint16_t* row_scale, int64_t stride_rs, const uint16_t* col_scale,
                                  int64_t stride_cs, int activation, void* C, int64_t stride_c, void* stream) {
  if (!valid_layout(layout) || !valid_activation(activation, col_scale)) return BQ_ERR_INVALID_ARG;
  const int64_t max_k = bits == 4 ? 16384 : MAX_K;
  GemmArgs g{A, Bp, ACT_I8, bits, layout, M, N, K, row_scale, col_scale, EPI_I32, C, activation};
  return run_batched(g, batch, stride_bytes(stride_a, 1), stride_bytes(stride_b, 1), stride_bytes(stride_rs, 2),
                     stride_bytes(stride_cs, 2), stride_bytes(stride_c, col_scale ? 2 : 4), max_k, stream);
}

bq_status bq_gemm_i8xi4_batched(const int8_t* A, int64_t stride_a, const uint8_t* Bp, int64_t stride_b, int layout,
                                int64_t batch, int64_t M, int64_t N, int64_t K, const uint16_t* row_scale,
                                int64_t stride_rs, const uint16_t* col_scale, int64_t stride_cs, int activation,
                                void* C, int64_t stride_c, void* stream) {
  return sub_byte_batched(A, stride_a, Bp, stride_b, layout, 4, batch, M, N, K, row_scale, stride_rs, col_scale,
                          stride_cs, activation, C, stride_c, stream);
}

bq_status bq_gemm_i8xi2_batched(const int8_t* A, int64_t stride_a, const uint8_t* Bp, int64_t stride_b, int layout,
                                int64_t batch, int64_t M, int64_t N, int64_t K, const uint16_t* row_scale,
                                int64_t stride_rs, const uint16_t* col_scale, int64_t stride_cs, int activation,
                                void* C, int64_t stride_c, void* stream) {
  return sub_byte_batched(A, stride_a, Bp, stride_b, layout, 2, batch, M, N, K, row_scale, stride_rs, col_scale,
                          stride_cs, activation, C, stride_c, stream);
}

bq_status bq_gemm_f16xi4_batched(const uint16_t* X, int64_t stride_x, const uint8_t* Wp, int64_t stride_w, int layout,
                                 int64_t batch, int64_t M, int64_t N, int64_t K, const uint16_t* col_scale,
                                 int64_t stride_cs, int activation, uint16_t* Y, int64_t stride_y, void* stream) {
  if (!valid_layout(layout)) return BQ_ERR_INVALID_ARG;
  if (M > 0 && N > 0 && !col_scale) return BQ_ERR_INVALID_ARG;
  if (!valid_activation(activation, col_scale)) return BQ_ERR_INVALID_ARG;
  GemmArgs g{X, Wp, ACT_F16, 4, layout, M, N, K, nullptr, col_scale, EPI_F16_COL, Y, activation};
  return run_batched(g, batch, stride_bytes(stride_x, 2), stride_bytes(stride_w, 1), 0, stride_bytes(stride_cs, 2),
                     stride_bytes(stride_y, 2), MAX_K, stream);
}

bq_status bq_quantized_linear(const uint16_t* X, int64_t M, int64_t K, const void* W, int bits, int layout,
                              int64_t N, const uint16_t* w_scale, int activation, uint16_t* x_scale,
                              uint16_t* Y, void* stream) {
  if (M < 0 || N < 0 || K < 0) return BQ_ERR_INVALID_ARG;
  if (!valid_bits(bits) || !valid_layout(layout)) return BQ_ERR_INVALID_ARG;
  if (activation != BQ_ACT_NONE && activation != BQ_ACT_RELU && activation != BQ_ACT_GELU)
    return BQ_ERR_INVALID_ARG;
  if (M == 0) return BQ_OK;
  if (!x_scale || (K > 0 && !X)) return BQ_ERR_INVALID_ARG;
  if (N > 0 && (!Y || !w_scale || (K > 0 && !W))) return BQ_ERR_INVALID_ARG;
  const int64_t max_k = bits == 8 ? 8192 : (bits == 4 ? 16384 : MAX_K);
  if (K % 64 != 0 || N % 64 != 0 || K > max_k || M > MAX_DIM || N > MAX_DIM) return BQ_ERR_UNSUPPORTED;
  if (!aligned16(x_scale) || (K > 0 && !aligned16(X))) return BQ_ERR_ALIGNMENT;
  if (N > 0 && (!aligned16(Y) || !aligned16(w_scale) || (K > 0 && !aligned16(W)))) return BQ_ERR_ALIGNMENT;
  GemmArgs g{X, W, ACT_Q8, bits, layout, M, N, K, x_scale, w_scale, EPI_F16_ROWCOL, Y, activation};
  // int8 weights: every fp32 chain must stay exact (decided before any launch)
  if (bits == 8 && N > 0 && K > 0 && !gemm_tc_i8_exact(g)) return BQ_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = launch_row_scale_f16(X, M, K, x_scale, s);
  if (e != cudaSuccess) return BQ_ERR_CUDA;
  if (N == 0) return BQ_OK;
  return run_gemm(g, stream);
}

bq_status bq_gemm_f16xu4_zp(const uint16_t* X, const uint8_t* Wp, int layout, int64_t M, int64_t N, int64_t K,
                            const uint16_t* col_scale, const uint16_t* zero_point, int activation, float* row_sum,
                            uint16_t* Y, void* stream) {
  if (!valid_layout(layout)) return BQ_ERR_INVALID_ARG;
  if (activation != BQ_ACT_NONE && activation != BQ_ACT_RELU && activation != BQ_ACT_GELU)
    return BQ_ERR_INVALID_ARG;
  if (M > 0 && N > 0 && (!col_scale || !zero_point)) return BQ_ERR_INVALID_ARG;
  if (M > 0 && !row_sum) return BQ_ERR_INVALID_ARG;
  bq_status st = check_gemm(X, Wp, M, N, K, nullptr, col_scale, Y, MAX_K);
  if (st != BQ_OK) return st;
  if (M == 0) return BQ_OK;
  if (!aligned16(row_sum) || (zero_point && !aligned16(zero_point))) return BQ_ERR_ALIGNMENT;
  if (K > 0 && !X) return BQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the skinny kernel (the route run_gemm takes for these shapes) forms the
  // row sums itself and writes them; every other route reads them
  const bool sums_in_gemv = N > 0 && K > 0 && M <= SKINNY_M && gemv_zp_fits(M, K);
  if (!sums_in_gemv && launch_row_sum_f16(X, M, K, row_sum, s) != cudaSuccess) return BQ_ERR_CUDA;
  if (N == 0) return BQ_OK;
  GemmArgs g{X, Wp, ACT_F16, 4, layout, M, N, K, nullptr, col_scale, EPI_F16_COL, Y, activation};
  g.zero_point = zero_point;
  g.row_sum = row_sum;
  return run_gemm(g, stream);
}

bq_status bq_device_status(int* status_out, int reset) {
  if (!status_out) return BQ_ERR_INVALID_ARG;
  return from_cuda(read_device_status(status_out, reset != 0));
}

int64_t bq_set_wait_timeout_ns(int64_t ns) {
  if (ns < 0) ns = 0;
  return g_wait_timeout_ns.exchange(ns);
}

}  // extern "C"
