"""CPU oracle for the quantize -> pack -> mixed-precision GEMM hot path.

TEST INFRASTRUCTURE ONLY.  This module is the plain, slow, obviously correct
statement of what the CUDA library computes.  It shares no code, table or
helper with the library and imports nothing from it.  Only the test suite,
the smoke check and the benchmark's CPU-baseline leg may import it; the
product path never does.

Pages this follows (cited by title and section):

* [BitBLAS] "BitBLAS自定义操作开发指南：使用DSL扩展新的混合精度算子"
  (BitBLAS guide to custom mixed-precision operators), sections
  "混合精度算子开发实战 1. 创建混合精度矩阵乘法" (INT8xINT4 GEMM with int32
  accumulation, B stored (N, K)), "2. 添加反量化支持" (per-column fp16
  dequantisation), "实际应用案例 案例1" (INT8xINT2, BitNet-b1.58) and
  "案例2" (fp16 activations times dequantised 4-bit weights, fp32
  accumulation, weights stored (N, K//2) uint8).
* [BMINF] "BMINF的後訓練量化實現" (BMINF post-training quantisation),
  section "實現代碼分析2": the ``quantize`` docstring of
  ``PartialAttention`` (row-absmax scale ``abs(max)/127`` stored as fp16,
  codes ``nearbyintf(x / scale)``), and ``elementwise_copy_scale``
  (``out0 = in0 * in1 * in2``: int32 times weight scale times activation
  scale, fp16 result).
* [Pallas] "JAX Pallas 在 TPU 上编写高效矩阵乘法内核", section "块矩阵乘法"
  (the block identity z_ij = sum_k x_ik y_kj) and the note that int8/int4
  inputs accumulate in int32.

Readings taken where the pages are silent or ambiguous (each is listed in
the design notes with its reason):

* Q1  the scale division runs in fp32 and is rounded once to fp16 (RNE); the
      codes are computed from the STORED fp16 scale.
* Q2  default rounding divides in fp32 and rounds to nearest-even; the
      BMINF "half" variant first rounds the quotient to fp16.
* Q4  codes saturate to [-D, D] (only matters for fp16-subnormal scales).
* Q5  a row whose scale is 0 gets all-zero codes.
* Q6  2-bit codes use D = 1 (absmax), i.e. {-1, 0, 1}.  Parity unpinned
      beyond the invariants: the pages never quantise to 2 bits.
* Q7  sub-byte codes are two's complement; "plain" packing puts the lowest
      k in the lowest bits; the "interleaved" packing is defined below.
* Q10 dequantisation multiplies in fp32 in the order int32 * w_scale *
      x_scale and rounds once to fp16 (the literal fp16(int32) cast
      overflows for |C| >= 65520; ``dequant_literal_fp16`` reports that).
* Q11 fp16 x int4 applies the per-channel scale after an exact (float64)
      accumulation.
* Q16 4-bit weights with a zero point hold unsigned codes u in [0, 15] (the
      same bit fields as the signed codes) and dequantise as s * (u - z).
* Q15 a fused activation acts on the dequantised value (after every scale
      product, as the Pallas page applies it to the f32 result of the last
      step before the one downcast) and the result is rounded once to fp16;
      GELU is the erf form v * Phi(v) (the BladeDISC page names GELU without
      a formula).

A fused activation follows [Pallas] section "模板化矩阵乘法 / 融合激活函数"
and [DISC] "全面支持 PyTorch 2.0：BladeDISC 5 月~11 月新功能发布", section
"Ongoing Work / CUTLASS Gemm CodeGen" (GEMM + GELU).
"""

from __future__ import annotations

import math

import numpy as np

# Symmetric code range per bit width: D such that codes lie in [-D, D].
# [BMINF 實現代碼分析2] divides the absmax by 127 for int8; the 4-bit value 7
# follows the int4 range [-8, 7] kept symmetric; 2 bits use 1 (reading Q6).
QMAX = {8: 127, 4: 7, 2: 1}


# ---------------------------------------------------------------------------
# a1 + a2: symmetric per-row quantisation  [BMINF 實現代碼分析2, quantize]
# ---------------------------------------------------------------------------
def quantize_scale(x: np.ndarray, bits: int = 8) -> np.ndarray:
    """Per-row scale s[r] = fp16(max_c |x[r, c]| / D).

    The page's reduction keeps the element of largest magnitude and stores
    ``abs(value) / 127`` into an fp16 buffer: the division happens in fp32
    and the store rounds to nearest-even (reading Q1).
    """
    if x.dtype not in (np.float16, np.float32):
        raise TypeError("x must be float16 or float32")
    if x.ndim != 2:
        raise ValueError("x must be 2-D (rows, cols)")
    d = np.float32(QMAX[bits])
    if x.shape[1] == 0:
        return np.zeros(x.shape[0], dtype=np.float16)
    absmax = np.abs(x).max(axis=1).astype(np.float32)   # exact
    return (absmax / d).astype(np.float16)               # fp32 divide, one RNE


def quantize_codes(x: np.ndarray, scale_f16: np.ndarray, bits: int = 8,
                   mode: str = "f32div") -> np.ndarray:
    """Codes q[r, c] = sat(nearbyint(x[r, c] / s[r])) from the stored fp16 s.

    mode "f32div": the quotient is an fp32 division rounded to nearest-even
    (the page's ``quantize_copy_float``).  mode "bminf_half": the quotient is
    first rounded to fp16 (``quantize_copy_half``), then to an integer.
    Saturation to [-D, D] is reading Q4; rows with s == 0 give 0 (Q5).
    """
    d = QMAX[bits]
    xs = x.astype(np.float32)
    s = scale_f16.astype(np.float32)[:, None]
    zero_row = (s == 0)
    with np.errstate(divide="ignore", invalid="ignore"):
        quot = xs / np.where(zero_row, np.float32(1), s)
    if mode == "bminf_half":
        with np.errstate(over="ignore"):
            quot = quot.astype(np.float16).astype(np.float32)
    elif mode != "f32div":
        raise ValueError("mode must be 'f32div' or 'bminf_half'")
    q = np.rint(quot)                                     # ties to even
    q = np.clip(q, -d, d)
    q = np.where(zero_row, 0, q)
    return q.astype(np.int8)


def quantize_sym(x: np.ndarray, bits: int = 8, mode: str = "f32div"):
    """Fused a1 + a2: returns (codes int8 (R, C), scale fp16 (R,))."""
    s = quantize_scale(x, bits)
    return quantize_codes(x, s, bits, mode), s


# ---------------------------------------------------------------------------
# a3: packed sub-byte storage
# ---------------------------------------------------------------------------
def packed_row_bytes(k: int, bits: int) -> int:
    """Bytes per packed row: K*bits/8 ([BitBLAS 案例2] stores 4-bit (N, K//2))."""
    return k * bits // 8


def pack_plain(q: np.ndarray, bits: int) -> np.ndarray:
    """Plain packing: element k of a row sits in byte k*bits//8, at bit
    offset (k mod (8/bits))*bits, two's complement (low nibble = even k)."""
    q = np.asarray(q)
    n, k = q.shape
    if bits == 8:
        return q.astype(np.int8).view(np.uint8).copy()
    per = 8 // bits
    if k % per:
        raise ValueError("K must be a multiple of 8/bits")
    mask = (1 << bits) - 1
    out = np.zeros((n, k // per), dtype=np.uint8)
    for t in range(per):
        field = (q[:, t::per].astype(np.int64) & mask).astype(np.uint8)
        out |= (field << (t * bits)).astype(np.uint8)
    return out


def unpack_plain(p: np.ndarray, k: int, bits: int) -> np.ndarray:
    """Inverse of ``pack_plain``: sign-extends every field to int8."""
    p = np.asarray(p, dtype=np.uint8)
    n = p.shape[0]
    if bits == 8:
        return p.view(np.int8).copy()
    per = 8 // bits
    mask = (1 << bits) - 1
    half = 1 << (bits - 1)
    q = np.zeros((n, k), dtype=np.int8)
    for t in range(per):
        field = ((p >> (t * bits)) & mask).astype(np.int16)
        q[:, t::per] = np.where(field >= half, field - (1 << bits), field)
    return q


def interleave_order(bits: int) -> list[int]:
    """Position of each element inside one 32-bit little-endian word of the
    interleaved layout.

    A word holds E = 32/bits consecutive k.  Element e (0 <= e < E) is stored
    in field position p(e): even e fill the low 16 bits in order
    (p = e/2), odd e fill the high 16 bits in order (p = E/2 + (e-1)/2).
    Masking one field from each 16-bit half then yields the pair (e, e+1).
    For 8-bit codes the interleaved layout is the plain layout.
    """
    if bits == 8:
        return [0, 1, 2, 3]
    e_per_word = 32 // bits
    return [e // 2 if e % 2 == 0 else e_per_word // 2 + e // 2
            for e in range(e_per_word)]


def pack_interleaved(q: np.ndarray, bits: int) -> np.ndarray:
    """Interleaved packing: a permutation of fields inside every 32-bit word
    of a plain-packed row (rows and words keep their order)."""
    q = np.asarray(q)
    n, k = q.shape
    if bits == 8:
        return pack_plain(q, 8)
    e_per_word = 32 // bits
    if k % e_per_word:
        raise ValueError("K must be a multiple of 32/bits")
    order = interleave_order(bits)
    mask = (1 << bits) - 1
    words = np.zeros((n, k // e_per_word), dtype=np.uint64)
    for e in range(e_per_word):
        field = (q[:, e::e_per_word].astype(np.int64) & mask).astype(np.uint64)
        words |= field << np.uint64(order[e] * bits)
    return words.astype("<u4").view(np.uint8).reshape(n, k * bits // 8)


def unpack_interleaved(p: np.ndarray, k: int, bits: int) -> np.ndarray:
    """Inverse of ``pack_interleaved``."""
    p = np.ascontiguousarray(p, dtype=np.uint8)
    n = p.shape[0]
    if bits == 8:
        return unpack_plain(p, k, 8)
    e_per_word = 32 // bits
    order = interleave_order(bits)
    mask = (1 << bits) - 1
    half = 1 << (bits - 1)
    words = p.view("<u4").astype(np.int64)
    q = np.zeros((n, k), dtype=np.int8)
    for e in range(e_per_word):
        field = (words >> (order[e] * bits)) & mask
        q[:, e::e_per_word] = np.where(field >= half, field - (1 << bits), field)
    return q


def unpack(p: np.ndarray, k: int, bits: int, layout: str) -> np.ndarray:
    if layout == "plain":
        return unpack_plain(p, k, bits)
    if layout == "interleaved":
        return unpack_interleaved(p, k, bits)
    raise ValueError(layout)


def pack(q: np.ndarray, bits: int, layout: str) -> np.ndarray:
    if layout == "plain":
        return pack_plain(q, bits)
    if layout == "interleaved":
        return pack_interleaved(q, bits)
    raise ValueError(layout)


# ---------------------------------------------------------------------------
# a5: integer GEMM  [BitBLAS 混合精度算子开发实战 1; 案例1]
# ---------------------------------------------------------------------------
INT32_MIN, INT32_MAX = -(1 << 31), (1 << 31) - 1


def gemm_int(a: np.ndarray, b_codes: np.ndarray) -> np.ndarray:
    """C[i, j] = sum_k int(A[i, k]) * int(B[j, k]) as int32.

    A is (M, K) int8, B is the (N, K) matrix of unpacked codes (NT form, the
    contraction runs over both operands' second axis).  A float64 matmul is
    used as the library step: every product and partial sum is an integer
    below 2**53, so it is exact.  The result must fit int32 (the page's
    accumulator type); otherwise OverflowError.
    """
    a = np.asarray(a)
    b_codes = np.asarray(b_codes)
    if a.shape[1] != b_codes.shape[1]:
        raise ValueError("K mismatch")
    k = a.shape[1]
    if k and k * 128 * 128 >= (1 << 53):
        raise ValueError("K too large for an exact float64 accumulation")
    c = np.rint(a.astype(np.float64) @ b_codes.astype(np.float64).T).astype(np.int64)
    if c.size and (c.min() < INT32_MIN or c.max() > INT32_MAX):
        raise OverflowError("int32 accumulator overflow")
    return c.astype(np.int32)


# ---------------------------------------------------------------------------
# a6: fused dequantisation  [BitBLAS 2. 添加反量化支持; BMINF elementwise_copy_scale]
# ---------------------------------------------------------------------------
def activation(v: np.ndarray, kind: str = "none") -> np.ndarray:
    """The fused activation, in float64 (reading Q15).

    "none": v;  "relu": max(v, 0);  "gelu": v * Phi(v) with Phi the standard
    normal distribution function, Phi(v) = erfc(-v / sqrt(2)) / 2.
    """
    v = np.asarray(v, dtype=np.float64)
    if kind == "none":
        return v
    if kind == "relu":
        return np.where(v > 0.0, v, 0.0)
    if kind == "gelu":
        phi = np.vectorize(lambda t: 0.5 * math.erfc(-t / math.sqrt(2.0)), otypes=[np.float64])
        return v * phi(v) if v.size else v
    raise ValueError(kind)


def dequant(c: np.ndarray, col_scale: np.ndarray,
            row_scale: np.ndarray | None = None, act: str = "none") -> np.ndarray:
    """D[i, j] = fp16( act( (float(C[i, j]) * float(sw[j])) * float(sx[i]) ) ).

    All products in IEEE fp32 (each rounded to nearest-even), one final
    rounding to fp16 (reading Q10).  Without a row scale the second product
    is omitted.  The activation (reading Q15) acts on that fp32 value.
    """
    cf = np.asarray(c, dtype=np.int32).astype(np.float32)
    out = cf * col_scale.astype(np.float32)[None, :]
    if row_scale is not None:
        out = out * row_scale.astype(np.float32)[:, None]
    if act != "none":
        out = activation(out, act)
    with np.errstate(over="ignore"):
        return out.astype(np.float16)


def dequant_literal_fp16(c: np.ndarray, col_scale: np.ndarray) -> np.ndarray:
    """The page's literal form fp16(C_int32) * scale evaluated in fp16.

    Used only to count how many entries overflow to inf under that reading.
    """
    with np.errstate(over="ignore"):
        return (np.asarray(c).astype(np.float16) * col_scale.astype(np.float16)[None, :])


# ---------------------------------------------------------------------------
# a7 / a8: fp16 activations x 4-bit weights  [BitBLAS 案例2; 高级功能 动态形状]
# ---------------------------------------------------------------------------
def gemm_f16xq(x: np.ndarray, w_codes: np.ndarray, scale: np.ndarray, act: str = "none") -> np.ndarray:
    """Y[i, j] = fp16( act( s[j] * sum_k float(X[i, k]) * q[j, k] ) ).

    The sum is a float64 matmul (library step).  For fp16 X and 4-bit codes
    every product is exact (at most 15 significant bits); the sum is exact
    too while the products' exponents span less than 53 - 15 - log2(K) bits,
    and otherwise rounds at 2**-53 relative to the largest partial sum, far
    inside the fp16 tolerance.  The per-channel scale is applied after it
    (reading Q11), then the activation (reading Q15).
    """
    acc = np.asarray(x, dtype=np.float64) @ np.asarray(w_codes, dtype=np.float64).T
    v = acc * scale.astype(np.float64)[None, :]
    if act != "none":
        v = activation(v, act)
    with np.errstate(over="ignore"):
        return v.astype(np.float16)


def gemm_f16xq_acc(x: np.ndarray, w_codes: np.ndarray) -> np.ndarray:
    """The exact unscaled float64 accumulator of ``gemm_f16xq``."""
    return np.asarray(x, dtype=np.float64) @ np.asarray(w_codes, dtype=np.float64).T


# ---------------------------------------------------------------------------
# 4-bit weights with a per-column zero point  [BitBLAS 实际应用案例 案例2]
# ---------------------------------------------------------------------------
def unpack_unsigned(p: np.ndarray, k: int, bits: int, layout: str) -> np.ndarray:
    """Unsigned codes 0 .. 2**bits - 1 of a packed matrix: the same fields as
    ``unpack`` reads, taken without sign extension (reading Q16)."""
    q = unpack(p, k, bits, layout)
    return (q.astype(np.int16) & ((1 << bits) - 1)).astype(np.uint8)


def gemm_f16xu4_zp(x: np.ndarray, u_codes: np.ndarray, scale: np.ndarray, zero_point: np.ndarray,
                   act: str = "none") -> np.ndarray:
    """Y[i, j] = fp16( act( sum_k X[i, k] * w[j, k] ) ),  w[j, k] = s[j] * (u[j, k] - z[j]).

    The page's NF4 example takes fp16 activations (M, K), packed weights
    (N, K // 2) uint8, and a per-column fp16 ``scale`` and ``zero_point``,
    with fp32 accumulation of the products of the dequantised weights.  Reading
    Q16: the weight codes are unsigned 4-bit values u in [0, 15] and the
    dequantisation is the affine w = s * (u - z) with the fp16 zero point z
    (not necessarily an integer).  Every w is exact in float64, and the sum is
    a float64 matmul (library step), one rounding to fp16 at the end.
    """
    w = scale.astype(np.float64)[:, None] * (np.asarray(u_codes, dtype=np.float64)
                                             - zero_point.astype(np.float64)[:, None])
    v = np.asarray(x, dtype=np.float64) @ w.T
    if act != "none":
        v = activation(v, act)
    with np.errstate(over="ignore"):
        return v.astype(np.float16)


# ---------------------------------------------------------------------------
# The whole quantised linear of one configuration
# ---------------------------------------------------------------------------
def quantized_linear(x: np.ndarray, w_codes: np.ndarray, w_scale: np.ndarray, act: str = "none"):
    """Quantised linear with fp16 activations and pre-quantised weights.

    The chain of [BMINF 實現代碼分析2] for one decode step: ``quantize`` the
    activations per row to int8 (``quantize_sym`` with D = 127, fp32
    division), ``igemm`` with int32 accumulation against the weight codes
    (8-, 4- or 2-bit values, unpacked, (N, K)), then
    ``elementwise_copy_scale`` with the weight scale per output column and the
    activation scale per row (``dequant``, reading Q10), and the optional
    activation (reading Q15).  Returns (Y fp16 (M, N), x_scale fp16 (M,)).
    """
    xq, sx = quantize_sym(np.asarray(x), 8, "f32div")
    c = gemm_int(xq, w_codes)
    return dequant(c, w_scale, sx, act), sx


def quantized_linear_i8(x: np.ndarray, w: np.ndarray):
    """Quantise activations X (M, K) and weights W (N, K) per row to int8,
    multiply in int32 and dequantise with both scales, in the order of
    [BMINF 實現代碼分析2]: quantize -> igemm -> elementwise_copy_scale."""
    xq, sx = quantize_sym(x, 8)
    wq, sw = quantize_sym(w, 8)
    c = gemm_int(xq, wq)
    return dequant(c, sw, sx), (xq, sx, wq, sw, c)
