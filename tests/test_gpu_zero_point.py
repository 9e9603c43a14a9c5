"""GPU parity of fp16 x 4-bit weights with a per-column zero point
(bq_gemm_f16xu4_zp) against the oracle's float64 sum of X * s * (u - z).

Form: "BitBLAS自定义操作开发指南", section 实际应用案例 案例2 (fp16 activations,
(N, K // 2) packed weights, per-column fp16 scale and zero point, fp32
accumulation).  Outputs are held to the tolerance of the other fp16 GEMM tests
(1e-3 relative, or 1e-3 of the column scale near zero); the row sums the
epilogue uses are checked against their float64 values; and with zero point 8
and codes u = v + 8 the call must equal the symmetric fp16 x int4 GEMM bit for
bit (the same tensor-core sums, and a zero correction term).
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


def make_case(seed, M, N, K, fractional=True):
    rng = np.random.default_rng(seed)
    x = W.normal_f16(rng, (M, K), 1.0)
    u = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    s = W.uniform_f16(rng, (N,), 1e-3, 1e-2)
    z = rng.integers(0, 16, size=N).astype(np.float16)
    if fractional:
        z[::3] = (z[::3].astype(np.float32) + rng.uniform(-0.5, 0.5, size=z[::3].shape)).astype(np.float16)
    return x, u, s, z


def pack_u(u, layout):
    return dev(O.pack(u.astype(np.int16).astype(np.int8), 4, layout))


def check_row_sum(rs, x):
    exact = x.astype(np.float64).sum(axis=1)
    bound = x.shape[1] * 2.0 ** -23 * np.abs(x.astype(np.float64)).sum(axis=1) + 1e-30
    assert (np.abs(host(rs).astype(np.float64) - exact) <= bound).all()


# M spans every bucket: the skinny kernel (M <= 16), the kernel with the weights as the MMA's A operand
# (16 < M <= 128), the split-K single-CTA kernel and CTA pairs; ragged M and both layouts; K = 576 and
# 448 end the skinny kernel's K steps (128) half way, where the lanes past K feed zeros to the row sums
SHAPES = [(1, 4096, 4096, "interleaved"), (5, 1024, 512, "plain"), (3, 1024, 576, "plain"),
          (16, 2048, 448, "interleaved"), (17, 2048, 1024, "interleaved"),
          (64, 11008, 4096, "interleaved"), (130, 4096, 2048, "plain"), (600, 8192, 512, "interleaved"),
          (1000, 4096, 1024, "plain")]


@pytest.mark.parametrize("M,N,K,layout", SHAPES)
def test_zero_point_parity(M, N, K, layout):
    x, u, s, z = make_case(M + N + K, M, N, K)
    y, rs = bq.bq_gemm_f16xu4_zp(dev(x), pack_u(u, layout), dev(s), dev(z), layout=layout)
    torch.cuda.synchronize()
    assert bq.bq_device_status(reset=True) == bq.BQ_OK
    rows = np.arange(M) if M <= 256 else np.unique(np.concatenate([np.arange(0, M, 7), [M - 1]]))
    y_ref = O.gemm_f16xu4_zp(x[rows], u, s, z)
    assert_f16_close(host(y)[rows], y_ref, s[None, :].astype(np.float64), f"zp {M}x{N}x{K}")
    check_row_sum(rs, x)


@pytest.mark.parametrize("M,N,K", [(3, 1024, 512), (40, 4096, 1024), (200, 4096, 1024), (600, 8192, 512)])
def test_zero_point_eight_equals_symmetric_path(M, N, K):
    rng = np.random.default_rng(M)
    x = W.normal_f16(rng, (M, K), 1.0)
    v = W.int4_uniform(rng, (N, K))
    s = W.uniform_f16(rng, (N,), 1e-3, 1e-2)
    xd, sd = dev(x), dev(s)
    y_sym = bq.bq_gemm_f16xi4(xd, dev(O.pack(v, 4, "interleaved")), sd)
    y_zp, _ = bq.bq_gemm_f16xu4_zp(xd, pack_u((v + 8).astype(np.uint8), "interleaved"), sd,
                                   dev(np.full(N, 8, np.float16)))
    torch.cuda.synchronize()
    # the same kernel family at every M: identical sums, and a zero correction term
    assert torch.equal(y_zp.view(torch.int16), y_sym.view(torch.int16))
    y_ref = O.gemm_f16xq(x, v, s)
    assert_f16_close(host(y_zp), y_ref, s[None, :].astype(np.float64), "zp8")


@pytest.mark.parametrize("act", ["relu", "gelu"])
@pytest.mark.parametrize("M", [9, 600])
def test_zero_point_activation(act, M):
    x, u, s, z = make_case(11 * M, M, 4096, 1024)
    y, _ = bq.bq_gemm_f16xu4_zp(dev(x), pack_u(u, "interleaved"), dev(s), dev(z), activation=act)
    torch.cuda.synchronize()
    y_ref = O.gemm_f16xu4_zp(x, u, s, z, act)
    assert_f16_close(host(y), y_ref, s[None, :].astype(np.float64), act, f16_ulps=1 if act == "gelu" else 0)


def test_zero_point_degenerate_sizes():
    rng = np.random.default_rng(4)
    x = W.normal_f16(rng, (5, 128), 1.0)
    s = dev(W.uniform_f16(rng, (64,), 1e-3, 1e-2))
    z = dev(np.full(64, 3, np.float16))
    # K == 0: row sums 0, outputs 0
    y, rs = bq.bq_gemm_f16xu4_zp(torch.empty((5, 0), dtype=torch.float16, device="cuda"),
                                 torch.empty((64, 0), dtype=torch.uint8, device="cuda"), s, z)
    torch.cuda.synchronize()
    assert not host(rs).any() and not host(y).astype(np.float32).any()
    # N == 0: the row sums are still written
    _, rs = bq.bq_gemm_f16xu4_zp(dev(x), torch.empty((0, 64), dtype=torch.uint8, device="cuda"),
                                 torch.empty((0,), dtype=torch.float16, device="cuda"),
                                 torch.empty((0,), dtype=torch.float16, device="cuda"))
    torch.cuda.synchronize()
    check_row_sum(rs, x)
