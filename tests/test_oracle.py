"""Pins for the CPU oracle: checks against things other than the oracle itself.

Every check here uses hand-worked values from tests/golden/, closed forms,
invariants, or brute force written with different primitives (pure-Python
integers, ``struct``'s IEEE half/single rounding, ``math.fsum``), so that a
dropped term, a wrong sign, index or rounding in the oracle fails one of them.
"""

import math
import struct

import numpy as np
import pytest

from oracle import bq_oracle as O
from quantized_mixed_precision_gb300 import roofline, workloads as W
from tests.golden_io import load


# --------------------------------------------------------------------------
# Independent scalar rounding helpers (Python struct: IEEE binary16 / binary32,
# round-half-to-even).
# --------------------------------------------------------------------------
def f16(v: float) -> float:
    try:
        return struct.unpack("<e", struct.pack("<e", v))[0]
    except OverflowError:
        return math.copysign(math.inf, v)


def f32(v: float) -> float:
    return struct.unpack("<f", struct.pack("<f", v))[0]


def brute_quantize_row(row, bits, mode="f32div"):
    d = {8: 127, 4: 7, 2: 1}[bits]
    a = max(abs(float(v)) for v in row)
    s = f16(f32(a / d))           # fp32 quotient (correctly rounded), then fp16
    q = []
    for v in row:
        if s == 0:
            q.append(0)
            continue
        t = f32(float(v) / s)
        if mode == "bminf_half":
            t = f16(t)
        r = round(t)              # Python rounds half to even
        q.append(max(-d, min(d, r)))
    return q, s


# --------------------------------------------------------------------------
# Quantiser
# --------------------------------------------------------------------------
def test_quantize_hand_example():
    g = load("quantize_hand_example.txt")
    x = np.array([[float(v) for v in g["x"].split()]], dtype=np.float16)
    q, s = O.quantize_sym(x, int(g["bits"]))
    assert float(s[0]) == float(g["scale"])
    assert q[0].tolist() == [int(v) for v in g["q"].split()]


@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("mode", ["f32div", "bminf_half"])
def test_quantize_brute_force(bits, mode):
    rng = np.random.default_rng(1)
    x = W.normal_f16(rng, (6, 37), 0.3)
    x[2] = 0                                   # all-zero row (reading Q5)
    x[3, :] = np.float16(0.5) * np.sign(x[3])  # ties everywhere
    q, s = O.quantize_sym(x, bits, mode)
    for r in range(x.shape[0]):
        bq, bs = brute_quantize_row(x[r].tolist(), bits, mode)
        assert float(s[r]) == bs
        assert q[r].tolist() == bq


def test_quantize_float32_input_brute_force():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((4, 50)) * 3).astype(np.float32)
    q, s = O.quantize_sym(x, 8)
    for r in range(4):
        bq, bs = brute_quantize_row(x[r].tolist(), 8)
        assert float(s[r]) == bs and q[r].tolist() == bq


@pytest.mark.parametrize("bits", [8, 4, 2])
def test_quantize_invariants(bits):
    d = O.QMAX[bits]
    rng = np.random.default_rng(3)
    x = W.normal_f16(rng, (64, 1000), 0.02)
    q, s = O.quantize_sym(x, bits)
    assert np.abs(q.astype(int)).max() <= d
    # every (non-zero, normal-scale) row reaches +-D
    assert (np.abs(q.astype(int)).max(axis=1) == d).all()
    # reconstruction error at most half a step (plus an fp32 ulp of slack)
    err = np.abs(x.astype(np.float64) - q.astype(np.float64) * s.astype(np.float64)[:, None])
    bound = s.astype(np.float64)[:, None] * (0.5 + 2.0 ** -20)
    assert (err <= bound).all()


def test_quantize_half_mode_bound():
    rng = np.random.default_rng(4)
    x = W.normal_f16(rng, (64, 1000), 1.0)
    q, s = O.quantize_sym(x, 8, "bminf_half")
    err = np.abs(x.astype(np.float64) - q.astype(np.float64) * s.astype(np.float64)[:, None])
    assert (err <= s.astype(np.float64)[:, None] * (0.5 + 2.0 ** -5)).all()


def test_quantize_double_rounding_example():
    # x / s = 101.47 rounds to fp16 101.5 and then to 102 in the BMINF half
    # mode, but to 101 with an fp32 quotient (reading Q2).
    s = np.float16(1.0)
    x = np.array([[127.0, 101.47]], dtype=np.float32)
    assert float(O.quantize_scale(x, 8)[0]) == 1.0
    assert O.quantize_codes(x, np.array([s]), 8, "f32div")[0, 1] == 101
    assert O.quantize_codes(x, np.array([s]), 8, "bminf_half")[0, 1] == 102


def test_quantize_subnormal_scale_saturates():
    # absmax = 178 * 2^-24 (an fp16 subnormal); 178/127 * 2^-24 rounds to the
    # scale 2^-24, so absmax / s = 178 would exceed 127 without saturation.
    a = np.float16(178 * 2.0 ** -24)
    x = np.array([[a, -a, np.float16(0)]], dtype=np.float16)
    q, s = O.quantize_sym(x, 8)
    assert float(s[0]) == 2.0 ** -24
    assert q[0].tolist() == [127, -127, 0]


def test_quantize_zero_row():
    q, s = O.quantize_sym(np.zeros((2, 8), np.float16), 4)
    assert (s == 0).all() and (q == 0).all()


# --------------------------------------------------------------------------
# Packing
# --------------------------------------------------------------------------
def _codes(txt):
    return np.array([[int(v) for v in txt.split()]], dtype=np.int8)


def _bytes(txt):
    return [int(v, 16) for v in txt.split()]


def test_pack_hand_bytes():
    g = load("pack_hand_bytes.txt")
    assert O.pack_plain(_codes(g["int4_plain_codes"]), 4)[0].tolist() == _bytes(g["int4_plain_bytes"])
    assert O.pack_plain(_codes(g["int2_plain_codes"]), 2)[0].tolist() == _bytes(g["int2_plain_bytes"])
    c4 = _codes(g["int4_inter_codes"])
    assert O.pack_interleaved(c4, 4)[0].tolist() == _bytes(g["int4_inter_bytes"])
    assert O.pack_plain(c4, 4)[0].tolist() == _bytes(g["int4_plain_bytes_same"])
    c2 = _codes(g["int2_word_codes"])
    assert O.pack_plain(c2, 2)[0].tolist() == _bytes(g["int2_word_plain_bytes"])
    assert O.pack_interleaved(c2, 2)[0].tolist() == _bytes(g["int2_word_inter_bytes"])


@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("layout", ["plain", "interleaved"])
def test_pack_round_trip(bits, layout):
    rng = np.random.default_rng(5)
    lo = -(1 << (bits - 1))
    q = rng.integers(lo, -lo, size=(7, 64), dtype=np.int8)
    p = O.pack(q, bits, layout)
    assert p.shape == (7, O.packed_row_bytes(64, bits))
    assert (O.unpack(p, 64, bits, layout) == q).all()


def test_pack_plain_bitwise_brute_force():
    rng = np.random.default_rng(6)
    for bits in (4, 2):
        q = rng.integers(-(1 << (bits - 1)), 1 << (bits - 1), size=(3, 32), dtype=np.int8)
        p = O.pack_plain(q, bits)
        per = 8 // bits
        for r in range(3):
            for k in range(32):
                field = (int(p[r, k // per]) >> ((k % per) * bits)) & ((1 << bits) - 1)
                assert field == (int(q[r, k]) + (1 << bits)) % (1 << bits)


# --------------------------------------------------------------------------
# Integer GEMM
# --------------------------------------------------------------------------
def brute_gemm(a, b):
    m, k = a.shape
    n = b.shape[0]
    al, bl = a.astype(int).tolist(), b.astype(int).tolist()
    return [[sum(al[i][t] * bl[j][t] for t in range(k)) for j in range(n)] for i in range(m)]


@pytest.mark.parametrize("m,n,k", [(1, 1, 1), (3, 5, 7), (17, 2, 9), (4, 16, 33)])
@pytest.mark.parametrize("bbits", [8, 4, 2])
def test_gemm_brute_force(m, n, k, bbits):
    rng = np.random.default_rng(m * 100 + n * 10 + k)
    a = W.int8_uniform(rng, (m, k))
    lo = -(1 << (bbits - 1))
    b = rng.integers(lo, -lo, size=(n, k), dtype=np.int8)
    assert O.gemm_int(a, b).tolist() == brute_gemm(a, b)


def test_gemm_matches_int64_matmul():
    rng = np.random.default_rng(7)
    a = W.int8_uniform(rng, (96, 320))
    b = W.int8_uniform(rng, (80, 320))
    assert (O.gemm_int(a, b) == (a.astype(np.int64) @ b.astype(np.int64).T)).all()


def test_gemm_closed_forms():
    k = 4096
    a = np.full((3, k), 127, np.int8)
    b = np.full((5, k), -8, np.int8)
    assert (O.gemm_int(a, b) == -1016 * k).all()
    rng = np.random.default_rng(8)
    a = W.int8_uniform(rng, (9, 64))
    eye = np.eye(64, dtype=np.int8)
    assert (O.gemm_int(a, eye) == a).all()
    # extreme int8 product: (-128) * (-128) * 4096 = 2**26 (beyond fp32's exact range)
    a = np.full((2, 4096), -128, np.int8)
    assert (O.gemm_int(a, a) == 1 << 26).all()


def test_gemm_overflow_detected():
    a = np.full((1, 131072), -128, np.int8)
    with pytest.raises(OverflowError):
        O.gemm_int(a, a)


@pytest.mark.parametrize("bm,bn,bk", [(8, 8, 8), (16, 4, 32), (32, 32, 64)])
def test_gemm_block_identity(bm, bn, bk):
    # JAX Pallas TPU matmul tutorial, section 块矩阵乘法: z_ij = sum_k x_ik y_kj
    rng = np.random.default_rng(9)
    m, n, k = 32, 32, 64
    a = W.int8_uniform(rng, (m, k))
    b = W.int4_uniform(rng, (n, k))
    z = np.zeros((m, n), np.int64)
    for i in range(0, m, bm):
        for j in range(0, n, bn):
            for t in range(0, k, bk):
                z[i:i + bm, j:j + bn] += O.gemm_int(a[i:i + bm, t:t + bk], b[j:j + bn, t:t + bk])
    assert (z == O.gemm_int(a, b)).all()


# --------------------------------------------------------------------------
# Dequantisation
# --------------------------------------------------------------------------
def test_dequant_power_of_two_scales_exact():
    rng = np.random.default_rng(10)
    c = rng.integers(-300000, 300000, size=(5, 6)).astype(np.int32)
    c[0, 0] = 65519 * 64
    sw = np.array([2.0 ** -e for e in (4, 6, 7, 9, 10, 12)], np.float16)
    sx = np.array([2.0 ** -e for e in (0, 1, 3, 5, 8)], np.float16)
    d = O.dequant(c, sw, sx)
    for i in range(5):
        for j in range(6):
            exact = float(c[i, j]) * float(sw[j]) * float(sx[i])   # exact in double
            if abs(int(c[i, j])) < (1 << 24):
                assert float(d[i, j]) == f16(exact)


def test_dequant_brute_force_fp32_order():
    rng = np.random.default_rng(11)
    c = rng.integers(-(1 << 26), 1 << 26, size=(4, 7)).astype(np.int32)
    sw = W.uniform_f16(rng, (7,), 1e-3, 1e-2)
    sx = W.uniform_f16(rng, (4,), 1e-4, 1e-3)
    d = O.dequant(c, sw, sx)
    d1 = O.dequant(c, sw)
    for i in range(4):
        for j in range(7):
            cf = f32(float(int(c[i, j])))
            p1 = f32(cf * float(sw[j]))
            assert float(d1[i, j]) == f16(p1)
            assert float(d[i, j]) == f16(f32(p1 * float(sx[i])))


def test_dequant_literal_reading_overflows():
    # reading Q10: fp16(C_int32) is inf once |C| >= 65520
    c = np.array([[65519, 65520, -70000]], np.int32)
    lit = O.dequant_literal_fp16(c, np.array([1e-3, 1e-3, 1e-3], np.float16))
    assert np.isfinite(lit[0, 0]) and np.isinf(lit[0, 1]) and np.isinf(lit[0, 2])
    ours = O.dequant(c, np.array([1e-3, 1e-3, 1e-3], np.float16))
    assert np.isfinite(ours).all()


# --------------------------------------------------------------------------
# fp16 x 4-bit weights
# --------------------------------------------------------------------------
def test_f16xq_brute_force_fsum():
    rng = np.random.default_rng(12)
    x = W.normal_f16(rng, (3, 40), 1.0)
    q = W.int4_uniform(rng, (6, 40))
    s = W.uniform_f16(rng, (6,), 0.008, 0.016)
    y = O.gemm_f16xq(x, q, s)
    acc = O.gemm_f16xq_acc(x, q)
    for i in range(3):
        for j in range(6):
            exact = math.fsum(float(x[i, t]) * int(q[j, t]) for t in range(40))
            assert acc[i, j] == exact
            assert float(y[i, j]) == f16(exact * float(s[j]))


def test_f16xq_scale_unit_and_identity():
    x = np.array([[1.5, -2.25, 0.0, 3.0]], np.float16)
    eye = np.eye(4, dtype=np.int8)
    assert (O.gemm_f16xq(x, eye, np.ones(4, np.float16)) == x).all()


# --------------------------------------------------------------------------
# Whole quantised linear (workload with two scales)
# --------------------------------------------------------------------------
def test_quantized_linear_small():
    rng = np.random.default_rng(13)
    x = W.normal_f16(rng, (5, 64), 1.0)
    w = W.normal_f16(rng, (7, 64), 0.02)
    y, (xq, sx, wq, sw, c) = O.quantized_linear_i8(x, w)
    assert c.tolist() == brute_gemm(xq, wq)
    ref = x.astype(np.float64) @ w.astype(np.float64).T
    # quantisation error of an int8 linear stays within a few percent of the output scale
    assert np.abs(y.astype(np.float64) - ref).max() < 0.05 * np.abs(ref).max()


def test_quantized_linear_hand_example():
    g = load("quantized_linear_hand_example.txt")
    x = np.array([[float(v) for v in g["x"].split()]], np.float16)
    wq = np.array([[int(v) for v in row.split()] for row in g["w_codes"].split(";")], np.int8)
    sw = np.array([float(v) for v in g["w_scale"].split()], np.float16)
    y, sx = O.quantized_linear(x, wq, sw)
    assert float(sx[0]) == float(g["x_scale"])
    assert [float(v) for v in y[0]] == [float(v) for v in g["y"].split()]
    y_relu, _ = O.quantized_linear(x, wq, sw, "relu")
    assert [float(v) for v in y_relu[0]] == [float(v) for v in g["y_relu"].split()]


def brute_quantized_linear(x, wq, sw, act="none"):
    """Pure-Python chain: per-row quantisation with struct rounding, integer
    sums, then the fp32 products in the order int32 * w_scale * x_scale."""
    out, scales = [], []
    for row in x:
        q, s = brute_quantize_row([float(v) for v in row], 8)
        scales.append(s)
        yrow = []
        for j in range(wq.shape[0]):
            c = sum(int(a) * int(b) for a, b in zip(q, wq[j]))
            v = f32(f32(f32(float(c)) * float(sw[j])) * s)
            if act == "relu":
                v = max(v, 0.0)
            yrow.append(f16(v))
        out.append(yrow)
    return out, scales


@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("act", ["none", "relu"])
def test_quantized_linear_brute_force(bits, act):
    rng = np.random.default_rng(14 + bits)
    x = W.normal_f16(rng, (4, 96), 1.0)
    x[2] *= np.float16(1e-3)                          # a row with a small scale
    x[3] = 0                                          # a zero row: scale 0, codes 0
    d = {8: 127, 4: 7, 2: 1}[bits]
    wq = rng.integers(-d - (bits != 2), d + 1, size=(6, 96)).astype(np.int8)
    sw = W.uniform_f16(rng, (6,), 1e-3, 1e-2)
    y, sx = O.quantized_linear(x, wq, sw, act)
    ref, ref_s = brute_quantized_linear(x, wq, sw, act)
    assert [float(v) for v in sx] == ref_s
    assert y.astype(np.float64).tolist() == ref


def test_quantized_linear_lossless_activations():
    # rows that are exactly integer codes times a power of two, absmax 127 x 2**-e:
    # the scale is 2**-e exactly, the codes are the integers, and the result is
    # the float64 product of X itself with the weights, rounded twice (fp32, fp16)
    rng = np.random.default_rng(15)
    m, n, k = 5, 7, 128
    exps = [3, 6, 8, 10, 12]
    q = rng.integers(-127, 128, size=(m, k))
    q[:, 5] = 127
    x = np.array([q[i] * 2.0 ** -exps[i] for i in range(m)], np.float16)
    wq = rng.integers(-128, 128, size=(n, k)).astype(np.int8)
    sw = W.uniform_f16(rng, (n,), 1e-3, 1e-2)
    y, sx = O.quantized_linear(x, wq, sw)
    assert [float(v) for v in sx] == [2.0 ** -e for e in exps]
    exact = x.astype(np.float64) @ wq.astype(np.float64).T        # = C * 2**-e, exact in float64
    for i in range(m):
        for j in range(n):
            c = exact[i, j] * 2.0 ** exps[i]
            assert c == int(c)
            assert float(y[i, j]) == f16(f32(f32(c) * float(sw[j])) * 2.0 ** -exps[i])
            ulp = 2.0 ** (math.floor(math.log2(abs(float(y[i, j])))) - 10) if y[i, j] != 0 else 2.0 ** -24
            assert abs(float(y[i, j]) - exact[i, j] * float(sw[j])) <= ulp


# --------------------------------------------------------------------------
# 4-bit weights with a per-column zero point
# --------------------------------------------------------------------------
def _rows(txt, conv=float):
    return [[conv(v) for v in row.split()] for row in txt.split(";")]


def test_zero_point_hand_example():
    g = load("zero_point_hand_example.txt")
    x = np.array(_rows(g["x"]), np.float16)
    u = np.array(_rows(g["u"], int), np.uint8)
    s = np.array([float(v) for v in g["scale"].split()], np.float16)
    z = np.array([float(v) for v in g["zero_point"].split()], np.float16)
    assert O.gemm_f16xu4_zp(x, u, s, z).astype(np.float64).tolist() == _rows(g["y"])
    assert O.gemm_f16xu4_zp(x, u, s, z, "relu").astype(np.float64).tolist() == _rows(g["y_relu"])


def test_zero_point_brute_force_fsum():
    rng = np.random.default_rng(16)
    x = W.normal_f16(rng, (3, 48), 1.0)
    u = rng.integers(0, 16, size=(5, 48)).astype(np.uint8)
    s = W.uniform_f16(rng, (5,), 1e-3, 1e-2)
    z = np.array([0, 7.5, 8, 15, 3.3], np.float16)             # integer and fractional zero points
    y = O.gemm_f16xu4_zp(x, u, s, z)
    for i in range(3):
        for j in range(5):
            # every product is exact in double (at most 11 + 11 + 28 significant bits); fsum rounds once
            exact = math.fsum(float(x[i, t]) * (float(s[j]) * (int(u[j, t]) - float(z[j]))) for t in range(48))
            assert float(y[i, j]) == f16(exact)


def test_zero_point_eight_is_the_symmetric_form():
    # u = v + 8 with zero point 8 is the signed 4-bit code v: the symmetric fp16 x int4 product
    rng = np.random.default_rng(17)
    x = W.normal_f16(rng, (4, 64), 1.0)
    v = W.int4_uniform(rng, (6, 64))
    s = W.uniform_f16(rng, (6,), 1e-3, 1e-2)
    y = O.gemm_f16xu4_zp(x, (v + 8).astype(np.uint8), s, np.full(6, 8, np.float16))
    assert (y.view(np.uint16) == O.gemm_f16xq(x, v, s).view(np.uint16)).all()


@pytest.mark.parametrize("layout", ["plain", "interleaved"])
def test_unsigned_codes_round_trip(layout):
    rng = np.random.default_rng(18)
    u = rng.integers(0, 16, size=(5, 64)).astype(np.uint8)
    p = O.pack(u.astype(np.int16).astype(np.int8), 4, layout)   # the low four bits of each code
    assert (O.unpack_unsigned(p, 64, 4, layout) == u).all()
    # the fields are the codes' bits: code 15 in the lowest field of a plain byte is 0x0f
    if layout == "plain":
        assert O.pack(np.array([[15, 0]], np.int8), 4, "plain")[0, 0] == 0x0F


# --------------------------------------------------------------------------
# Roofline accounting helper
# --------------------------------------------------------------------------
def test_roofline_helper_printed_numbers():
    g = load("pallas_roofline_numbers.txt")
    m, k, n = int(g["m"]), int(g["k"]), int(g["n"])
    bits = 8 * int(g["itemsize"])
    assert roofline.matmul_ops(m, k, n) == int(g["flops"])
    assert roofline.matmul_min_bytes(m, k, n, bits, bits, bits) == int(g["membw_bytes"])
    # packed 4-bit weights count half a byte per element
    assert roofline.matmul_min_bytes(4096, 4096, 4096, 8, 4, 16) == (16 + 8 + 32) * 2 ** 20


# ---------------------------------------------------------------------------
# fused activation (reading Q15): pinned to tabulated values of the standard
# normal distribution function and to identities, not to the formula itself
# ---------------------------------------------------------------------------
def test_gelu_tabulated_values():
    # Phi(1) = 0.8413447460685429 and Phi(3) = 0.9986501019683699 (standard
    # normal table), so GELU(1) = Phi(1) and GELU(-3) = -3 * (1 - Phi(3)).
    g = O.activation(np.array([1.0, -3.0, 0.0]), "gelu")
    assert g[0] == pytest.approx(0.8413447460685429, rel=1e-15)
    assert g[1] == pytest.approx(-3.0 * (1.0 - 0.9986501019683699), rel=1e-12)
    assert g[2] == 0.0


def test_gelu_odd_part_and_limits():
    # Phi(v) + Phi(-v) = 1  =>  GELU(v) - GELU(-v) = v  (a sign or argument slip breaks it)
    v = np.linspace(-6.0, 6.0, 97)
    g = O.activation(v, "gelu")
    gm = O.activation(-v, "gelu")
    assert np.allclose(g - gm, v, rtol=0, atol=1e-14)
    # far tails: identity for large v, vanishing (and negative) for very negative v
    assert O.activation(np.array([40.0]), "gelu")[0] == 40.0
    tail = O.activation(np.array([-12.0]), "gelu")[0]
    assert -1e-30 < tail < 0.0
    # monotone from its minimum near v = -0.75 on
    w = np.linspace(-0.7, 5.0, 200)
    assert (np.diff(O.activation(w, "gelu")) > 0).all()


def test_relu_and_none():
    v = np.array([-2.5, -0.0, 0.0, 1e-8, 3.0])
    assert O.activation(v, "relu").tolist() == [0.0, 0.0, 0.0, 1e-8, 3.0]
    assert O.activation(v, "none").tolist() == v.tolist()
    with pytest.raises(ValueError):
        O.activation(v, "tanh")


def test_dequant_relu_commutes_with_rounding():
    # RNE to fp16 is monotone and maps 0 to 0, so ReLU before the rounding
    # equals clamping the rounded value; a dropped activation, or min taken
    # for max, fails this.
    rng = np.random.default_rng(5)
    c = rng.integers(-40000, 40000, size=(7, 64)).astype(np.int32)
    sw = W.uniform_f16(rng, (64,), 1e-3, 1e-2)
    sx = W.uniform_f16(rng, (7,), 1e-3, 1e-1)
    base = O.dequant(c, sw, sx).astype(np.float64)
    assert (O.dequant(c, sw, sx, act="relu").astype(np.float64) == np.maximum(base, 0.0)).all()
    assert (O.dequant(c, sw, sx, act="none") == O.dequant(c, sw, sx)).all()


def test_f16xq_gelu_positive_scale_preserves_sign_of_dequant():
    rng = np.random.default_rng(6)
    x = W.normal_f16(rng, (3, 128), 1.0)
    q = W.int4_uniform(rng, (32, 128))
    s = W.uniform_f16(rng, (32,), 0.008, 0.016)
    y = O.gemm_f16xq(x, q, s).astype(np.float64)
    yg = O.gemm_f16xq(x, q, s, act="gelu").astype(np.float64)
    # GELU(v) has the sign of v, |GELU(v)| <= |v|, and GELU(v) >= v / 2 for v >= 0
    assert (np.sign(yg) * np.sign(y) >= 0).all()
    assert (np.abs(yg) <= np.abs(y) + 1e-3).all()
    pos = y > 0.05
    assert (yg[pos] >= 0.5 * y[pos] - 1e-3).all()
