// Arithmetic of the symmetric per-row quantiser, shared by the quantiser
// kernel and the GEMM converters that quantise fp16 activations in place, so
// that both produce the same codes bit for bit.
//
// "BMINF的後訓練量化實現", section 實現代碼分析2: the scale is the row absmax
// divided by D (127 for int8) and stored as fp16; the codes are
// nearbyint(x / scale) from that stored scale (quantize_copy_float), or with
// the quotient first rounded to fp16 (quantize_copy_half).
#pragma once
#include <cuda_fp16.h>
#include <cstdint>

#include "bq.h"

namespace bq {
namespace {

constexpr float RNE_MAGIC = 12582912.0f;   // 1.5 * 2**23: adding it rounds |t| < 2**22 to an integer (ties to even)
// The fast form of the code rne(RN(x / s)) for fp16 x and a normal fp16
// scale s (|x / s| <= 127 (1 + 2**-11)), without a division: t1 = RN(x * rcp)
// with rcp = RN(1 / s), the residual e = x - t1 s (exact in one fma), and
// t2 = RN(t1 + e rcp), which lies within 2**-40 of x / s before its rounding.
// Why that decides the integer: x / s is either a half-integer or at least
// 2**-12 away from every half-integer (x - h s is a nonzero multiple of
// 2**(e_s - 11); checked exhaustively over all such pairs), so rne(t2) =
// rne(x / s) away from ties, and at a tie x / s = h exactly, t2 = h, and the
// rounding below takes the even neighbour as the definition does.

// Code for one element from the stored fp16 scale s (as float), by the
// definition: rne(RN(x / s)) (F32DIV) or rne(fp16(RN(x / s))) (BMINF_HALF),
// clamped to [-d, d]; s == 0 yields code 0.  Returned as a float that carries
// the code in its low byte (two's complement): the rounding is
// t + 1.5 * 2**23 in fp32 (round to nearest even), whose low mantissa bits are
// then the integer; clamping before the rounding equals clamping after it, the
// bounds being integers.  Used for the rows whose scale is 0 or an fp16
// subnormal, where the fast form's error bound does not hold, and for
// BMINF_HALF.
__device__ __forceinline__ float code_exact(float x, float s, float fd, int mode) {
  float t = s == 0.0f ? 0.0f : __fdiv_rn(x, s);
  if (mode == BQ_ROUND_BMINF_HALF) t = __half2float(__float2half_rn(t));
  return __fadd_rn(fminf(fmaxf(t, -fd), fd), RNE_MAGIC);
}

__device__ __forceinline__ uint32_t code_byte(float m) { return __float_as_uint(m); }

// Fast form for two elements with packed fp32x2 arithmetic (each lane of a
// packed op is an ordinary IEEE round-to-nearest operation, fma with one
// rounding): m = RN(t2 + 1.5 * 2**23), whose low mantissa bits hold the code,
// and r = m - 1.5 * 2**23, the code as an integer-valued float.
__device__ __forceinline__ void code2_fast(float x0, float x1, float s, float rcp, float& m0, float& m1, float& r0,
                                           float& r1) {
  asm("{\n\t.reg .b64 x, ns, c, g, t, e, u, m, r;\n\t"
      "mov.b64 x, {%4, %5};\n\t"
      "mov.b64 ns, {%6, %6};\n\t"
      "mov.b64 c, {%7, %7};\n\t"
      "mov.b64 g, {%8, %8};\n\t"
      "mul.rn.f32x2 t, x, c;\n\t"
      "fma.rn.f32x2 e, t, ns, x;\n\t"
      "fma.rn.f32x2 u, e, c, t;\n\t"
      "add.rn.f32x2 m, u, g;\n\t"
      "sub.rn.f32x2 r, m, g;\n\t"
      "mov.b64 {%0, %1}, m;\n\t"
      "mov.b64 {%2, %3}, r;\n\t}"
      : "=f"(m0), "=f"(m1), "=f"(r0), "=f"(r1)
      : "f"(x0), "f"(x1), "f"(-s), "f"(rcp), "f"(RNE_MAGIC));
}

// Per-row constants of the int8 quantiser (D = 127, F32DIV) for the stored
// fp16 scale s: its reciprocal, and whether s is a normal fp16 (then
// |x / s| <= 127 (1 + 2**-11) for every x of the row and no code needs
// clamping).
struct RowQuant {
  float s, rcp;
  bool normal;
};

__device__ __forceinline__ RowQuant row_quant(float s) {
  return RowQuant{s, s == 0.0f ? 0.0f : __frcp_rn(s), s >= 6.103515625e-05f};
}

// int8 codes (D = 127, F32DIV) of a row's 64 fp16 values of one k-block, as
// 32 fp16 pairs (low half = even k) -- the form a kind::f16 tensor-core
// operand takes -- bit-identical to the codes the quantiser kernel stores.
// `row` is the row's 128 bytes in a 128B-swizzled shared-memory box (16-byte
// chunk c at position c ^ (r & 7)).
__device__ __forceinline__ uint32_t pack_codes(float c0, float c1) {
  const __half2 p = __floats2half2_rn(c0, c1);   // integers |c| <= 127: exact
  return *reinterpret_cast<const uint32_t*>(&p);
}

__device__ __forceinline__ void quant64_f16_codes(const uint8_t* row, int r, const RowQuant& rq, uint32_t (&h)[32]) {
  if (rq.normal) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint4 v = *reinterpret_cast<const uint4*>(row + ((j ^ (r & 7)) << 4));
      const __half2* x2 = reinterpret_cast<const __half2*>(&v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 p = __half22float2(x2[i]);
        float m0, m1, c0, c1;
        code2_fast(p.x, p.y, rq.s, rq.rcp, m0, m1, c0, c1);
        h[4 * j + i] = pack_codes(c0, c1);
      }
    }
  } else {   // scale 0 or an fp16 subnormal: the definition
#pragma unroll 1
    for (int j = 0; j < 8; ++j) {
      const uint4 v = *reinterpret_cast<const uint4*>(row + ((j ^ (r & 7)) << 4));
      const __half2* x2 = reinterpret_cast<const __half2*>(&v);
      uint32_t w[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 p = __half22float2(x2[i]);
        w[i] = pack_codes(__fsub_rn(code_exact(p.x, rq.s, 127.0f, BQ_ROUND_F32DIV), RNE_MAGIC),
                          __fsub_rn(code_exact(p.y, rq.s, 127.0f, BQ_ROUND_F32DIV), RNE_MAGIC));
      }
      // (dynamic j: the codes go through a small local array only on this rare path)
      h[4 * j] = w[0];
      h[4 * j + 1] = w[1];
      h[4 * j + 2] = w[2];
      h[4 * j + 3] = w[3];
    }
  }
}

}  // namespace
}  // namespace bq
