"""GPU parity of the fused quantised linear (bq_quantized_linear) against the
oracle's quantize -> integer GEMM -> two-scale dequant chain.

Chain: "BMINF的後訓練量化實現", section 實現代碼分析2 (quantize, igemm,
elementwise_copy_scale).  The activation scales must match bit for bit; so
must every output without GELU (the integer sum is exact and the dequant is
the same sequence of fp32 roundings); GELU outputs are held to the fp16
tolerance of the other GEMM tests plus one fp16 step.  The fused call must
also agree bit for bit with the two-call path (bq_quantize_sym, then the
integer GEMM with both scales).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import quantized_mixed_precision_gb300 as bq  # noqa: E402
from oracle import bq_oracle as O  # noqa: E402
from quantized_mixed_precision_gb300 import workloads as W  # noqa: E402
from tests.test_gpu_parity import assert_f16_close, dev, host  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bq.lib()
    yield
    torch.cuda.synchronize()
    assert bq.bq_device_status(reset=True) == bq.BQ_OK


def make_case(seed, M, N, K, bits):
    """fp16 activations ~ N(0, 1) with special rows, weight codes of the width,
    per-column scales in [1e-3, 1e-2)."""
    rng = np.random.default_rng(seed)
    x = W.normal_f16(rng, (M, K), 1.0)
    if M > 4:
        x[1] = 0                                              # zero row: scale 0, codes 0
        x[2] = (x[2].astype(np.float32) * 2.0 ** -20).astype(np.float16)   # fp16-subnormal scale
        # exact half-integer quotients: x / s = j + 1/2 with s = 2**-6 (ties to even)
        j = rng.integers(-127, 127, size=K)
        x[3] = ((j + 0.5) * 2.0 ** -6).astype(np.float16)
        x[3, 0] = np.float16(127 * 2.0 ** -6)
    if bits == 8:
        wq = W.int8_uniform(rng, (N, K))
    elif bits == 4:
        wq = W.int4_uniform(rng, (N, K))
    else:
        wq = W.int2_uniform(rng, (N, K))
    sw = W.uniform_f16(rng, (N,), 1e-3, 1e-2)
    return x, wq, sw


def weights_on_device(wq, bits, layout):
    if bits == 8:
        return dev(wq)
    return dev(O.pack(wq, bits, layout))


# (M, N, K, bits, layout): CTA pairs (with and without chunked int8
# accumulation, all three weight widths and both layouts), the single-CTA
# kernel with K split over a cluster (8 ranges of 16 k-blocks at K = 8192,
# 4-bit and 2-bit weights) and with four TMEM slices, ragged M everywhere.
SHAPES = [
    (600, 8192, 256, 8, "plain"),
    (600, 8192, 2048, 8, "plain"),
    (700, 4096, 4096, 8, "plain"),
    (600, 8192, 512, 4, "plain"),
    (600, 8192, 512, 4, "interleaved"),
    (600, 8192, 512, 2, "plain"),
    (600, 8192, 512, 2, "interleaved"),
    (40, 4160, 320, 8, "plain"),
    (130, 2048, 1024, 8, "plain"),
    (17, 4096, 8192, 8, "plain"),
    (640, 2048, 4096, 8, "plain"),
    (200, 1024, 1024, 4, "interleaved"),
    (64, 512, 2048, 2, "interleaved"),
    (1, 256, 512, 4, "plain"),
]


@pytest.mark.parametrize("M,N,K,bits,layout", SHAPES)
def test_quantized_linear_parity(M, N, K, bits, layout):
    x, wq, sw = make_case(M + N + K + bits, M, N, K, bits)
    y_ref, sx_ref = O.quantized_linear(x, wq, sw)
    wd = weights_on_device(wq, bits, layout)
    y, sx = bq.bq_quantized_linear(dev(x), wd, bits, dev(sw), layout=layout)
    torch.cuda.synchronize()
    assert bq.bq_device_status(reset=True) == bq.BQ_OK
    assert (host(sx).view(np.uint16) == sx_ref.view(np.uint16)).all()
    yh = host(y)
    bad = yh.view(np.uint16) != y_ref.view(np.uint16)
    assert not bad.any(), f"{bad.sum()} of {bad.size} outputs differ, first at {np.argwhere(bad)[:3].tolist()}"


@pytest.mark.parametrize("M,N,K,bits,layout", [(600, 8192, 2048, 8, "plain"), (600, 8192, 512, 4, "interleaved"),
                                                (130, 2048, 1024, 2, "plain")])
def test_quantized_linear_matches_two_call_path(M, N, K, bits, layout):
    x, wq, sw = make_case(7 * M + K, M, N, K, bits)
    xd, wd, swd = dev(x), weights_on_device(wq, bits, layout), dev(sw)
    y, sx = bq.bq_quantized_linear(xd, wd, bits, swd, layout=layout)
    q, s = bq.bq_quantize_sym(xd, 8, bq.ROUND_F32DIV)
    if bits == 8:
        y2 = bq.bq_gemm_i8xi8(q, wd, row_scale=s, col_scale=swd)
    elif bits == 4:
        y2 = bq.bq_gemm_i8xi4(q, wd, layout, row_scale=s, col_scale=swd)
    else:
        y2 = bq.bq_gemm_i8xi2(q, wd, layout, row_scale=s, col_scale=swd)
    torch.cuda.synchronize()
    assert torch.equal(sx.view(torch.int16), s.view(torch.int16))
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


@pytest.mark.parametrize("act", ["relu", "gelu"])
@pytest.mark.parametrize("M,N,K,bits", [(600, 8192, 2048, 8), (600, 8192, 512, 4), (130, 2048, 1024, 8)])
def test_quantized_linear_activation(act, M, N, K, bits):
    x, wq, sw = make_case(3 * M + K + bits, M, N, K, bits)
    y_ref, sx_ref = O.quantized_linear(x, wq, sw, act)
    y, sx = bq.bq_quantized_linear(dev(x), weights_on_device(wq, bits, "interleaved"), bits, dev(sw),
                                   layout="interleaved", activation=act)
    torch.cuda.synchronize()
    assert (host(sx).view(np.uint16) == sx_ref.view(np.uint16)).all()
    if act == "relu":
        assert (host(y).view(np.uint16) == y_ref.view(np.uint16)).all()
    else:
        scale_ij = sx_ref.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :]
        assert_f16_close(host(y), y_ref, scale_ij, "gelu", f16_ulps=1)


def test_quantized_linear_workload_sampled_rows():
    """The 1024 x 4096 x 4096 workload (fp16 X ~ N(0, 1), weights quantised
    per row from N(0, 0.02)), checked on sampled rows: rows are independent
    (per-row scale, per-row codes), so the oracle runs on the sample only."""
    d = W.cfg1()
    wq, sw = O.quantize_sym(d["W"], 8)
    y, sx = bq.bq_quantized_linear(dev(d["X"]), dev(wq), 8, dev(sw))
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, 1024, 37), [0, 255, 256, 511, 512, 1023]]))
    y_ref, sx_ref = O.quantized_linear(d["X"][rows], wq, sw)
    assert (host(sx)[rows].view(np.uint16) == sx_ref.view(np.uint16)).all()
    assert (host(y)[rows].view(np.uint16) == y_ref.view(np.uint16)).all()


def test_quantized_linear_degenerate_sizes():
    rng = np.random.default_rng(5)
    x = W.normal_f16(rng, (5, 128), 1.0)
    sw = dev(W.uniform_f16(rng, (64,), 1e-3, 1e-2))
    # N == 0: the scales are still written
    _, sx = bq.bq_quantized_linear(dev(x), torch.empty((0, 64), dtype=torch.uint8, device="cuda"), 4,
                                   torch.empty((0,), dtype=torch.float16, device="cuda"))
    torch.cuda.synchronize()
    assert (host(sx).view(np.uint16) == O.quantize_scale(x, 8).view(np.uint16)).all()
    # K == 0: scales 0 and outputs 0
    y, sx = bq.bq_quantized_linear(torch.empty((5, 0), dtype=torch.float16, device="cuda"),
                                   torch.empty((64, 0), dtype=torch.uint8, device="cuda"), 4, sw)
    torch.cuda.synchronize()
    assert not host(sx).any() and not host(y).astype(np.float32).any()
    # M == 0
    y, sx = bq.bq_quantized_linear(torch.empty((0, 128), dtype=torch.float16, device="cuda"),
                                   dev(O.pack(W.int4_uniform(rng, (64, 128)), 4, "interleaved")), 4, sw)
    assert y.shape == (0, 64) and sx.shape == (0,)
