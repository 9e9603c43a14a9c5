"""C-ABI checks that need no GPU: the library loads, exports every function
the header declares, and rejects invalid calls on the host before any launch.

Only calls that fail validation are made here (fake but aligned pointers are
never dereferenced because validation returns first)."""

import ctypes
import os

import pytest

import quantized_mixed_precision_gb300 as bq


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(bq.LIB_PATH):
        from quantized_mixed_precision_gb300 import build
        build.build()
    return bq.lib()


EXPECTED = sorted([
    "bq_status_string", "bq_quantize_sym", "bq_packed_size", "bq_pack_weights", "bq_gemm_i8xi8",
    "bq_gemm_i8xi4", "bq_gemm_i8xi2", "bq_gemm_f16xi4", "bq_device_status", "bq_set_wait_timeout_ns",
    "bq_gemm_i8xi8_act", "bq_gemm_i8xi4_act", "bq_gemm_i8xi2_act", "bq_gemm_f16xi4_act",
    "bq_gemm_i8xi8_batched", "bq_gemm_i8xi4_batched", "bq_gemm_i8xi2_batched", "bq_gemm_f16xi4_batched",
    "bq_quantized_linear", "bq_gemm_f16xu4_zp",
])

FAKE = ctypes.c_void_p(0x10000)     # aligned, never dereferenced
FAKE_ODD = ctypes.c_void_p(0x10008)  # 8-byte aligned only


def test_header_lists_expected_functions():
    assert bq.header_functions() == EXPECTED


def test_every_declared_symbol_is_exported(lib):
    for name in bq.header_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert bq.bq_status_string(0) == "BQ_OK"
    assert bq.bq_status_string(5) == "BQ_ERR_TIMEOUT"
    assert bq.bq_status_string(99) == "BQ_ERR_UNKNOWN"


def test_packed_size(lib):
    assert bq.bq_packed_size(11008, 4096, 4, "interleaved") == 22544384
    assert bq.bq_packed_size(8192, 8192, 2, "plain") == 16 * 2 ** 20
    assert bq.bq_packed_size(4, 6, 4, "plain") == 12
    assert bq.bq_packed_size(4, 12, 4, "interleaved") == 0      # needs k % 8
    assert bq.bq_packed_size(4, 16, 3, "plain") == 0
    assert bq.bq_packed_size(-1, 16, 4, "plain") == 0


def test_quantize_validation(lib):
    f = lib.bq_quantize_sym
    assert f(None, 0, 4, 8, 8, 8, 0, FAKE, FAKE, None) == bq.BQ_ERR_INVALID_ARG
    assert f(FAKE, 0, 4, 8, 4, 8, 0, FAKE, FAKE, None) == bq.BQ_ERR_INVALID_ARG     # ld_x < cols
    assert f(FAKE, 0, 4, 8, 8, 3, 0, FAKE, FAKE, None) == bq.BQ_ERR_INVALID_ARG     # bits
    assert f(FAKE, 2, 4, 8, 8, 8, 0, FAKE, FAKE, None) == bq.BQ_ERR_INVALID_ARG     # xtype
    assert f(FAKE, 0, 4, 8, 8, 8, 7, FAKE, FAKE, None) == bq.BQ_ERR_INVALID_ARG     # mode
    assert f(FAKE_ODD, 0, 4, 8, 8, 8, 0, FAKE, FAKE, None) == bq.BQ_ERR_ALIGNMENT
    assert f(FAKE, 0, 4, 1 << 25, 1 << 25, 8, 0, FAKE, FAKE, None) == bq.BQ_ERR_UNSUPPORTED
    assert f(None, 0, 0, 8, 8, 8, 0, None, None, None) == bq.BQ_OK                  # empty


def test_pack_validation(lib):
    f = lib.bq_pack_weights
    assert f(None, 4, 64, 4, 1, FAKE, None) == bq.BQ_ERR_INVALID_ARG
    assert f(FAKE, 4, 64, 5, 1, FAKE, None) == bq.BQ_ERR_INVALID_ARG
    assert f(FAKE, 4, 64, 4, 2, FAKE, None) == bq.BQ_ERR_INVALID_ARG
    assert f(FAKE, 4, 12, 4, 1, FAKE, None) == bq.BQ_ERR_UNSUPPORTED
    assert f(FAKE, 4, 64, 4, 1, FAKE_ODD, None) == bq.BQ_ERR_ALIGNMENT
    assert f(FAKE, 0, 64, 4, 1, FAKE, None) == bq.BQ_OK


@pytest.mark.parametrize("name", ["bq_gemm_i8xi4", "bq_gemm_i8xi2"])
def test_packed_gemm_validation(lib, name):
    f = getattr(lib, name)
    ok = dict(A=FAKE, B=FAKE, L=1, M=32, N=64, K=64, rs=None, cs=FAKE, C=FAKE)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["A"], a["B"], a["L"], a["M"], a["N"], a["K"], a["rs"], a["cs"], a["C"], None)

    assert call(A=None) == bq.BQ_ERR_INVALID_ARG
    assert call(C=None) == bq.BQ_ERR_INVALID_ARG
    assert call(L=5) == bq.BQ_ERR_INVALID_ARG
    assert call(M=-1) == bq.BQ_ERR_INVALID_ARG
    assert call(rs=FAKE, cs=None) == bq.BQ_ERR_INVALID_ARG
    assert call(K=96) == bq.BQ_ERR_UNSUPPORTED
    assert call(N=96) == bq.BQ_ERR_UNSUPPORTED
    assert call(K=1 << 17) == bq.BQ_ERR_UNSUPPORTED
    assert call(A=FAKE_ODD) == bq.BQ_ERR_ALIGNMENT
    assert call(cs=FAKE_ODD) == bq.BQ_ERR_ALIGNMENT
    assert call(M=0) == bq.BQ_OK
    assert call(N=0, C=None) == bq.BQ_OK


def test_i8xi4_exactness_bound(lib):
    # 128 * 8 * K must stay <= 2**24: K = 16384 is accepted by validation,
    # 16448 is not (the i8xi2 bound is 65536).
    f = lib.bq_gemm_i8xi4
    assert f(FAKE, FAKE, 1, 32, 64, 16448, None, None, FAKE, None) == bq.BQ_ERR_UNSUPPORTED
    g = lib.bq_gemm_i8xi2
    assert g(FAKE, FAKE, 1, 32, 64, 65600, None, None, FAKE, None) == bq.BQ_ERR_UNSUPPORTED


def test_i8xi8_and_f16xi4_validation(lib):
    f = lib.bq_gemm_i8xi8
    assert f(None, FAKE, 4, 64, 64, None, None, FAKE, None) == bq.BQ_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 4, 64, 100, None, None, FAKE, None) == bq.BQ_ERR_UNSUPPORTED
    g = lib.bq_gemm_f16xi4
    assert g(FAKE, FAKE, 1, 4, 64, 64, None, FAKE, None) == bq.BQ_ERR_INVALID_ARG   # scale required
    assert g(FAKE, FAKE, 1, 4, 64, 64, FAKE, FAKE_ODD, None) == bq.BQ_ERR_ALIGNMENT
    assert g(FAKE, FAKE, 0, 0, 64, 64, None, None, None) == bq.BQ_OK


@pytest.mark.parametrize("name", ["bq_gemm_i8xi4_act", "bq_gemm_i8xi2_act"])
def test_packed_gemm_act_validation(lib, name):
    f = getattr(lib, name)
    ok = dict(A=FAKE, B=FAKE, L=1, M=32, N=64, K=64, rs=None, cs=FAKE, act=bq.ACT_GELU, C=FAKE)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["A"], a["B"], a["L"], a["M"], a["N"], a["K"], a["rs"], a["cs"], a["act"], a["C"], None)

    assert call(act=3) == bq.BQ_ERR_INVALID_ARG
    assert call(act=-1) == bq.BQ_ERR_INVALID_ARG
    assert call(cs=None) == bq.BQ_ERR_INVALID_ARG               # an activation needs the fp16 output
    assert call(cs=None, act=bq.ACT_RELU, M=0) == bq.BQ_ERR_INVALID_ARG
    assert call(cs=None, act=bq.ACT_NONE, M=0) == bq.BQ_OK      # int32 output without activation
    assert call(L=5) == bq.BQ_ERR_INVALID_ARG
    assert call(K=96) == bq.BQ_ERR_UNSUPPORTED
    assert call(A=FAKE_ODD) == bq.BQ_ERR_ALIGNMENT
    assert call(M=0) == bq.BQ_OK


def test_i8xi8_and_f16xi4_act_validation(lib):
    f = lib.bq_gemm_i8xi8_act
    assert f(FAKE, FAKE, 4, 64, 64, None, FAKE, 9, FAKE, None) == bq.BQ_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 4, 64, 64, None, None, bq.ACT_RELU, FAKE, None) == bq.BQ_ERR_INVALID_ARG
    assert f(FAKE, FAKE, 0, 64, 64, None, FAKE, bq.ACT_GELU, FAKE, None) == bq.BQ_OK
    g = lib.bq_gemm_f16xi4_act
    assert g(FAKE, FAKE, 1, 4, 64, 64, FAKE, 7, FAKE, None) == bq.BQ_ERR_INVALID_ARG
    assert g(FAKE, FAKE, 1, 4, 64, 64, None, bq.ACT_GELU, FAKE, None) == bq.BQ_ERR_INVALID_ARG
    assert g(FAKE, FAKE, 1, 4, 64, 64, FAKE, bq.ACT_RELU, FAKE_ODD, None) == bq.BQ_ERR_ALIGNMENT
    assert g(FAKE, FAKE, 1, 0, 64, 64, FAKE, bq.ACT_GELU, FAKE, None) == bq.BQ_OK


def test_batched_validation(lib):
    f = lib.bq_gemm_i8xi4_batched
    # A, sa, Bp, sb, layout, batch, M, N, K, rs, srs, cs, scs, act, C, sc, stream
    ok = dict(A=FAKE, sa=0, B=FAKE, sb=64 * 32, L=1, batch=3, M=32, N=64, K=64, rs=None, srs=0, cs=FAKE, scs=64,
              act=0, C=FAKE, sc=32 * 64)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["A"], a["sa"], a["B"], a["sb"], a["L"], a["batch"], a["M"], a["N"], a["K"], a["rs"], a["srs"],
                 a["cs"], a["scs"], a["act"], a["C"], a["sc"], None)

    assert call(batch=-1) == bq.BQ_ERR_INVALID_ARG
    assert call(sb=-64) == bq.BQ_ERR_INVALID_ARG
    assert call(sc=32 * 64 - 8) == bq.BQ_ERR_INVALID_ARG          # outputs would overlap
    assert call(sc=0) == bq.BQ_ERR_INVALID_ARG
    assert call(sa=40) == bq.BQ_ERR_ALIGNMENT                     # 40-byte item offsets
    assert call(scs=12) == bq.BQ_ERR_ALIGNMENT                    # 24-byte scale offsets
    assert call(sb=1 << 62) == bq.BQ_ERR_UNSUPPORTED               # saturated, no overflow
    assert call(batch=(1 << 16) + 1) == bq.BQ_ERR_UNSUPPORTED
    assert call(act=5) == bq.BQ_ERR_INVALID_ARG
    assert call(K=96) == bq.BQ_ERR_UNSUPPORTED
    assert call(batch=0, C=None, A=None) == bq.BQ_OK              # empty batch
    assert call(M=0) == bq.BQ_OK
    g = lib.bq_gemm_f16xi4_batched
    assert g(FAKE, 0, FAKE, 2048, 1, 2, 4, 64, 64, None, 0, 0, FAKE, 256, None) == bq.BQ_ERR_INVALID_ARG  # scale required
    assert g(FAKE, 0, FAKE, 2048, 1, 2, 0, 64, 64, FAKE, 64, 0, FAKE, 0, None) == bq.BQ_OK


def test_quantized_linear_validation(lib):
    f = lib.bq_quantized_linear
    # (X, M, K, W, bits, layout, N, w_scale, activation, x_scale, Y, stream)
    ok = dict(X=FAKE, M=4, K=128, W=FAKE, bits=4, layout=1, N=64, ws=FAKE, act=0, xs=FAKE, Y=FAKE)

    def call(**kw):
        a = {**ok, **kw}
        return f(a["X"], a["M"], a["K"], a["W"], a["bits"], a["layout"], a["N"], a["ws"], a["act"], a["xs"],
                 a["Y"], None)

    assert call(M=-1) == bq.BQ_ERR_INVALID_ARG
    assert call(bits=3) == bq.BQ_ERR_INVALID_ARG
    assert call(layout=2) == bq.BQ_ERR_INVALID_ARG
    assert call(act=3) == bq.BQ_ERR_INVALID_ARG
    assert call(X=None) == bq.BQ_ERR_INVALID_ARG
    assert call(xs=None) == bq.BQ_ERR_INVALID_ARG
    assert call(W=None) == bq.BQ_ERR_INVALID_ARG
    assert call(ws=None) == bq.BQ_ERR_INVALID_ARG
    assert call(Y=None) == bq.BQ_ERR_INVALID_ARG
    assert call(K=96) == bq.BQ_ERR_UNSUPPORTED
    assert call(N=96) == bq.BQ_ERR_UNSUPPORTED
    assert call(bits=8, K=8256) == bq.BQ_ERR_UNSUPPORTED       # int8 weights: K <= 8192
    assert call(bits=4, K=16448) == bq.BQ_ERR_UNSUPPORTED      # 4-bit: K <= 16384
    # int8 weights, K = 8192 on 32 tiles of 128 x 256: neither K split into ranges of <= 16 k-blocks
    # nor a grid of CTA pairs that fills the GPU keeps every fp32 chain exact
    assert call(bits=8, K=8192, M=512, N=2048) == bq.BQ_ERR_UNSUPPORTED
    assert call(X=FAKE_ODD) == bq.BQ_ERR_ALIGNMENT
    assert call(xs=FAKE_ODD) == bq.BQ_ERR_ALIGNMENT
    assert call(Y=FAKE_ODD) == bq.BQ_ERR_ALIGNMENT
    assert call(M=0, X=None, xs=None) == bq.BQ_OK              # empty
    assert call(N=0, W=None, ws=None, Y=None, xs=None) == bq.BQ_ERR_INVALID_ARG   # x_scale is still written


def test_zero_point_gemm_validation(lib):
    f = lib.bq_gemm_f16xu4_zp
    # (X, Wp, layout, M, N, K, col_scale, zero_point, activation, row_sum, Y, stream)
    assert f(FAKE, FAKE, 2, 4, 64, 128, FAKE, FAKE, 0, FAKE, FAKE, None) == bq.BQ_ERR_INVALID_ARG   # layout
    assert f(FAKE, FAKE, 1, 4, 64, 128, FAKE, FAKE, 5, FAKE, FAKE, None) == bq.BQ_ERR_INVALID_ARG   # activation
    assert f(FAKE, FAKE, 1, 4, 64, 128, FAKE, None, 0, FAKE, FAKE, None) == bq.BQ_ERR_INVALID_ARG   # zero point
    assert f(FAKE, FAKE, 1, 4, 64, 128, None, FAKE, 0, FAKE, FAKE, None) == bq.BQ_ERR_INVALID_ARG   # scale
    assert f(FAKE, FAKE, 1, 4, 64, 128, FAKE, FAKE, 0, None, FAKE, None) == bq.BQ_ERR_INVALID_ARG   # row sums
    assert f(FAKE, FAKE, 1, 4, 64, 96, FAKE, FAKE, 0, FAKE, FAKE, None) == bq.BQ_ERR_UNSUPPORTED    # K % 64
    assert f(FAKE, FAKE, 1, 4, 64, 128, FAKE, FAKE, 0, FAKE_ODD, FAKE, None) == bq.BQ_ERR_ALIGNMENT
    assert f(FAKE, FAKE, 1, 4, 64, 128, FAKE, FAKE_ODD, 0, FAKE, FAKE, None) == bq.BQ_ERR_ALIGNMENT
    assert f(None, None, 1, 0, 64, 128, None, None, 0, None, None, None) == bq.BQ_OK                # empty


def test_device_status_null(lib):
    assert lib.bq_device_status(None, 0) == bq.BQ_ERR_INVALID_ARG


def test_wait_timeout_setter(lib):
    old = bq.bq_set_wait_timeout_ns(12345)
    assert bq.bq_set_wait_timeout_ns(old) == 12345
