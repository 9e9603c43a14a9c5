"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Integer results (codes, packed bytes, int32 accumulators) must match bit for
bit.  fp16 results must satisfy |y - y_ref| <= max(1e-3 |y_ref|, 1e-3 * s_ij)
where s_ij is the dequantisation scale of the element (per-column scale, or
row scale times column scale), and infinities must match exactly.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

import quantized_mixed_precision_gb300 as bq  # noqa: E402
from oracle import bq_oracle as O  # noqa: E402
from quantized_mixed_precision_gb300 import workloads as W  # noqa: E402

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    bq.lib()
    yield
    torch.cuda.synchronize()
    assert bq.bq_device_status(reset=True) == bq.BQ_OK


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def host(t):
    return t.cpu().numpy()


def assert_f16_close(y, y_ref, scale_ij, what="", f16_ulps=0):
    """f16_ulps > 0 also admits that many units in the last place of the
    fp16 reference: for outputs whose last step is evaluated in different
    precisions on the two sides (an fp32 activation against the oracle's
    float64 one), the single rounding to fp16 may land one step apart, and
    in the fp16 subnormal range one step exceeds the relative tolerance."""
    ulp = np.spacing(np.abs(y_ref.astype(np.float16))).astype(np.float64)
    y = y.astype(np.float64)
    y_ref = y_ref.astype(np.float64)
    inf_ref = ~np.isfinite(y_ref)
    assert (np.isfinite(y) == ~inf_ref).all(), f"{what}: inf pattern differs"
    assert (y[inf_ref] == y_ref[inf_ref]).all(), f"{what}: inf sign differs"
    fin = ~inf_ref
    tol = np.maximum(1e-3 * np.abs(y_ref), 1e-3 * np.broadcast_to(scale_ij, y_ref.shape).astype(np.float64))
    if f16_ulps:
        tol = np.maximum(tol, f16_ulps * ulp)
    err = np.abs(y - y_ref)
    bad = fin & (err > tol)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; "
                           f"worst err/tol {np.max(err[fin] / tol[fin]):.3g}")


# ---------------------------------------------------------------------------
# quantiser
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("rows,cols", [(1, 8), (7, 40), (33, 256), (100, 1000), (5, 4096), (3, 5000), (2, 3)])
@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("mode", [bq.ROUND_F32DIV, bq.ROUND_BMINF_HALF])
def test_quantize_parity(rows, cols, bits, mode):
    rng = np.random.default_rng(rows * 7 + cols)
    x = W.normal_f16(rng, (rows, cols), 0.5)
    if rows > 2:
        x[1] = 0                                               # zero row
        x[2, : min(cols, 3)] = np.float16(178 * 2.0 ** -24)    # subnormal scale, saturation
        x[2, min(cols, 3):] = 0
    if rows > 3:
        # exact ties x / s = j + 1/2 with s = 2**-6 (ties to even)
        d = {8: 127, 4: 7, 2: 1}[bits]
        x[3] = ((rng.integers(-d, d, size=cols) + 0.5) * 2.0 ** -6).astype(np.float16)
        x[3, 0] = np.float16(d * 2.0 ** -6)
    q_ref, s_ref = O.quantize_sym(x, bits, "f32div" if mode == bq.ROUND_F32DIV else "bminf_half")
    q, s = bq.bq_quantize_sym(dev(x), bits, mode)
    assert (host(s).view(np.uint16) == s_ref.view(np.uint16)).all()
    assert (host(q) == q_ref).all()


def test_quantize_parity_f32_and_strided():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((9, 300)) * 2).astype(np.float32)
    q_ref, s_ref = O.quantize_sym(x, 8)
    q, s = bq.bq_quantize_sym(dev(x), 8)
    assert (host(s).view(np.uint16) == s_ref.view(np.uint16)).all() and (host(q) == q_ref).all()
    big = W.normal_f16(rng, (6, 512), 1.0)
    xt = dev(big)[:, :256]                                     # leading dimension 512
    q_ref, s_ref = O.quantize_sym(big[:, :256], 4)
    q, s = bq.bq_quantize_sym(xt, 4)
    assert (host(s).view(np.uint16) == s_ref.view(np.uint16)).all() and (host(q) == q_ref).all()


def test_quantize_workload_full_size():
    d = W.cfg1()
    for name in ("W", "X"):
        q_ref, s_ref = O.quantize_sym(d[name], 8)
        q, s = bq.bq_quantize_sym(dev(d[name]), 8)
        assert (host(s).view(np.uint16) == s_ref.view(np.uint16)).all()
        assert (host(q) == q_ref).all()


# ---------------------------------------------------------------------------
# packer
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("layout", ["plain", "interleaved"])
@pytest.mark.parametrize("n,k", [(1, 64), (13, 256), (256, 4096)])
def test_pack_parity(bits, layout, n, k):
    rng = np.random.default_rng(n + k + bits)
    lo = -(1 << (bits - 1))
    q = rng.integers(lo, -lo, size=(n, k), dtype=np.int8)
    p = bq.bq_pack_weights(dev(q), bits, layout)
    assert (host(p) == O.pack(q, bits, layout)).all()


def test_pack_plain_odd_width():
    q = np.array([[1, -1, 3, -8, 7, 0]], np.int8)
    p = bq.bq_pack_weights(dev(q), 4, "plain")
    assert host(p)[0].tolist() == O.pack_plain(q, 4)[0].tolist()


# ---------------------------------------------------------------------------
# integer GEMMs (skinny and tensor-core paths, ragged M, all epilogues)
# ---------------------------------------------------------------------------
def _codes(rng, bits, shape):
    return {8: W.int8_uniform, 4: W.int4_uniform, 2: W.int2_uniform}[bits](rng, shape)


def _run_int_gemm(bits, A, Bq, layout, rs, cs):
    if bits == 8:
        return bq.bq_gemm_i8xi8(dev(A), dev(Bq), row_scale=rs, col_scale=cs)
    Bp = dev(O.pack(Bq, bits, layout))
    fn = bq.bq_gemm_i8xi4 if bits == 4 else bq.bq_gemm_i8xi2
    return fn(dev(A), Bp, layout, row_scale=rs, col_scale=cs)


SHAPES = [(1, 64, 64), (3, 128, 192), (16, 192, 256), (17, 256, 128), (130, 320, 512), (300, 512, 1024),
          (256, 256, 256)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("epi", ["i32", "col", "rowcol"])
def test_int_gemm_parity(M, N, K, bits, epi):
    rng = np.random.default_rng(M * 31 + N * 7 + K + bits)
    A = W.int8_uniform(rng, (M, K))
    Bq = _codes(rng, bits, (N, K))
    sw = W.uniform_f16(rng, (N,), 1e-3, 1e-2)
    sx = W.uniform_f16(rng, (M,), 1e-3, 1e-1)
    c_ref = O.gemm_int(A, Bq)
    for layout in (["interleaved", "plain"] if bits != 8 else ["plain"]):
        if epi == "i32":
            c = host(_run_int_gemm(bits, A, Bq, layout, None, None))
            assert (c == c_ref).all(), f"layout {layout}"
        elif epi == "col":
            y = host(_run_int_gemm(bits, A, Bq, layout, None, dev(sw)))
            assert_f16_close(y, O.dequant(c_ref, sw), sw[None, :].astype(np.float64), f"col {layout}")
        else:
            y = host(_run_int_gemm(bits, A, Bq, layout, dev(sx), dev(sw)))
            s_ij = sx[:, None].astype(np.float64) * sw[None, :].astype(np.float64)
            assert_f16_close(y, O.dequant(c_ref, sw, sx), s_ij, f"rowcol {layout}")


@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("M,N,K", [(2100, 4160, 512), (2048, 4096, 576)])
def test_int_gemm_many_tiles(M, N, K, bits):
    """Grids of more output tiles than the GPU holds at once (several waves of
    CTA pairs), ragged in M and N, with K a whole number of raw stages (512)
    and not (576)."""
    rng = np.random.default_rng(M + N + K + bits)
    A = W.int8_uniform(rng, (M, K))
    Bq = _codes(rng, bits, (N, K))
    sw = W.uniform_f16(rng, (N,), 1e-3, 1e-2)
    sx = W.uniform_f16(rng, (M,), 1e-3, 1e-1)
    c_ref = O.gemm_int(A, Bq)
    for layout in (["interleaved", "plain"] if bits != 8 else ["plain"]):
        c = host(_run_int_gemm(bits, A, Bq, layout, None, None))
        assert (c == c_ref).all(), f"int32 {layout}"
        y = host(_run_int_gemm(bits, A, Bq, layout, dev(sx), dev(sw)))
        s_ij = sx[:, None].astype(np.float64) * sw[None, :].astype(np.float64)
        assert_f16_close(y, O.dequant(c_ref, sw, sx), s_ij, f"rowcol {layout}")
    assert bq.bq_device_status(reset=True) == bq.BQ_OK


@pytest.mark.parametrize("M", [1, 40, 200])
def test_int_gemm_extreme_values_exact(M):
    # Largest magnitudes: -128 * -8 (4-bit, K = 16384) and -128 * -128 (int8,
    # K = 4096 -> 2**26, beyond fp32's exact integers unless sliced).
    K4 = 16384
    A = np.full((M, K4), -128, np.int8)
    B4 = np.full((64, K4), -8, np.int8)
    c = host(bq.bq_gemm_i8xi4(dev(A), dev(O.pack(B4, 4, "interleaved")), "interleaved"))
    assert (c == 1024 * K4).all()
    K8 = 4096
    A8 = np.full((M, K8), -128, np.int8)
    A8[:, ::3] = 127
    B8 = np.full((128, K8), -128, np.int8)
    c8 = host(bq.bq_gemm_i8xi8(dev(A8), dev(B8)))
    assert (c8 == O.gemm_int(A8, B8)).all()


def test_i8xi8_int32_large_k_path():
    rng = np.random.default_rng(21)
    A = W.int8_uniform(rng, (70, 8192))
    B = W.int8_uniform(rng, (128, 8192))
    assert (host(bq.bq_gemm_i8xi8(dev(A), dev(B))) == O.gemm_int(A, B)).all()


def test_gemm_k_zero_and_empty():
    A = torch.empty((5, 0), dtype=torch.int8, device=DEV)
    B = torch.empty((64, 0), dtype=torch.int8, device=DEV)
    c = bq.bq_gemm_i8xi8(A, B)
    assert (host(c) == 0).all()
    A0 = torch.empty((0, 64), dtype=torch.int8, device=DEV)
    B0 = torch.zeros((64, 64), dtype=torch.int8, device=DEV)
    assert bq.bq_gemm_i8xi8(A0, B0).shape == (0, 64)


# ---------------------------------------------------------------------------
# fp16 x 4-bit
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("M,N,K", [(1, 64, 64), (4, 128, 320), (16, 192, 256), (17, 64, 128), (64, 256, 512),
                                   (200, 320, 1024)])
@pytest.mark.parametrize("layout", ["interleaved", "plain"])
def test_f16xi4_parity(M, N, K, layout):
    rng = np.random.default_rng(M + N + K)
    X = W.normal_f16(rng, (M, K), 1.0)
    q = W.int4_uniform(rng, (N, K))
    s = W.uniform_f16(rng, (N,), 0.008, 0.016)
    y = host(bq.bq_gemm_f16xi4(dev(X), dev(O.pack(q, 4, layout)), dev(s), layout))
    assert_f16_close(y, O.gemm_f16xq(X, q, s), s[None, :].astype(np.float64), "f16xi4")


# ---------------------------------------------------------------------------
# fused activation epilogue (ReLU, GELU) on every path: skinny kernels, the
# single-CTA tensor-core kernel (K split over a cluster), CTA pairs, the
# small-M fp16 kernel
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("act", ["relu", "gelu"])
@pytest.mark.parametrize("bits,M,N,K", [(8, 1, 64, 256), (8, 40, 192, 256), (8, 600, 8192, 256),
                                        (4, 1, 128, 512), (4, 40, 320, 512), (4, 600, 8192, 256),
                                        (2, 3, 128, 512), (2, 200, 256, 512), (2, 600, 8192, 256)])
def test_int_gemm_activation(act, bits, M, N, K):
    rng = np.random.default_rng(bits * 7 + M + N + K)
    A = W.int8_uniform(rng, (M, K))
    Bq = _codes(rng, bits, (N, K))
    sw = W.uniform_f16(rng, (N,), 1e-3, 1e-2)
    sx = W.uniform_f16(rng, (M,), 1e-3, 1e-1)
    y_ref = O.dequant(O.gemm_int(A, Bq), sw, sx, act=act)
    rs, cs = dev(sx), dev(sw)
    if bits == 8:
        y = bq.bq_gemm_i8xi8_act(dev(A), dev(Bq), act, row_scale=rs, col_scale=cs)
    else:
        fn = bq.bq_gemm_i8xi4_act if bits == 4 else bq.bq_gemm_i8xi2_act
        y = fn(dev(A), dev(O.pack(Bq, bits, "interleaved")), act, "interleaved", row_scale=rs, col_scale=cs)
    assert_f16_close(host(y), y_ref, (sx[:, None].astype(np.float64) * sw[None, :]), f"{act} bits {bits}",
                     f16_ulps=1 if act == "gelu" else 0)


@pytest.mark.parametrize("act", ["relu", "gelu"])
@pytest.mark.parametrize("M,N,K", [(1, 320, 512), (5, 128, 832), (40, 4160, 320), (512, 8192, 256)])
def test_f16xi4_activation(act, M, N, K):
    rng = np.random.default_rng(M + N + K + (0 if act == "relu" else 1))
    X = W.normal_f16(rng, (M, K), 1.0)
    q = W.int4_uniform(rng, (N, K))
    s = W.uniform_f16(rng, (N,), 0.008, 0.016)
    y = host(bq.bq_gemm_f16xi4_act(dev(X), dev(O.pack(q, 4, "interleaved")), dev(s), act))
    assert_f16_close(y, O.gemm_f16xq(X, q, s, act=act), s[None, :].astype(np.float64), f"f16xi4 {act}",
                     f16_ulps=1 if act == "gelu" else 0)


# ---------------------------------------------------------------------------
# batched GEMMs with broadcast operands (the fused QKV projection: one block
# of activations, three stacked weight matrices)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("bits", [8, 4, 2])
@pytest.mark.parametrize("M", [1, 40, 300])
def test_batched_shared_activations(bits, M):
    rng = np.random.default_rng(100 + bits + M)
    N, K, nb = 192, 256, 3
    A = W.int8_uniform(rng, (1, M, K))
    Bq = [_codes(rng, bits, (N, K)) for _ in range(nb)]
    sw = W.uniform_f16(rng, (nb, N), 1e-3, 1e-2)
    sx = W.uniform_f16(rng, (M,), 1e-3, 1e-1)
    if bits == 8:
        Bw = dev(np.stack(Bq))
        y = host(bq.bq_gemm_i8xi8_batched(dev(A), Bw, row_scale=dev(sx), col_scale=dev(sw), activation="relu"))
        c = host(bq.bq_gemm_i8xi8_batched(dev(A), Bw))
    else:
        Bw = dev(np.stack([O.pack(b, bits, "interleaved") for b in Bq]))
        fn = bq.bq_gemm_i8xi4_batched if bits == 4 else bq.bq_gemm_i8xi2_batched
        y = host(fn(dev(A), Bw, "interleaved", row_scale=dev(sx), col_scale=dev(sw), activation="relu"))
        c = host(fn(dev(A), Bw, "interleaved"))
    for b in range(nb):
        c_ref = O.gemm_int(A[0], Bq[b])
        assert (c[b] == c_ref).all(), f"item {b}"
        assert_f16_close(y[b], O.dequant(c_ref, sw[b], sx, act="relu"), sx[:, None].astype(np.float64) * sw[b][None, :],
                         f"item {b}")


def test_batched_shared_weights_f16xi4():
    rng = np.random.default_rng(7)
    nb, M, N, K = 4, 20, 320, 512
    X = W.normal_f16(rng, (nb, M, K), 1.0)
    q = W.int4_uniform(rng, (N, K))
    s = W.uniform_f16(rng, (N,), 0.008, 0.016)
    Wp = dev(O.pack(q, 4, "interleaved")[None])
    y = host(bq.bq_gemm_f16xi4_batched(dev(X), Wp, dev(s), activation="gelu"))
    for b in range(nb):
        assert_f16_close(y[b], O.gemm_f16xq(X[b], q, s, act="gelu"), s[None, :].astype(np.float64), f"item {b}",
                         f16_ulps=1)


# shapes the CTA-pair kernel serves (short K, or grids that fill the GPU)
@pytest.mark.parametrize("bits,M,N,K", [(8, 320, 448, 256), (8, 600, 3840, 2048), (4, 600, 3840, 1024),
                                        (2, 328, 448, 256)])
def test_batched_one_grid_every_operand_strided(bits, M, N, K):
    """Items on the CTA-pair kernel run as one grid (batch = grid z): A, B, both
    scales and C all per item; int8 x int8 at K = 2048 also exercises the
    chunked accumulation, whose running high parts live in each item's output."""
    rng = np.random.default_rng(200 + bits + K)
    nb = 3
    A = W.int8_uniform(rng, (nb, M, K))
    Bq = [_codes(rng, bits, (N, K)) for _ in range(nb)]
    sw = W.uniform_f16(rng, (nb, N), 1e-3, 1e-2)
    sx = W.uniform_f16(rng, (nb, M), 1e-3, 1e-1)
    if bits == 8:
        Bw = dev(np.stack(Bq))
        y = host(bq.bq_gemm_i8xi8_batched(dev(A), Bw, row_scale=dev(sx), col_scale=dev(sw)))
        c = host(bq.bq_gemm_i8xi8_batched(dev(A), Bw))
    else:
        Bw = dev(np.stack([O.pack(b, bits, "interleaved") for b in Bq]))
        fn = bq.bq_gemm_i8xi4_batched if bits == 4 else bq.bq_gemm_i8xi2_batched
        y = host(fn(dev(A), Bw, "interleaved", row_scale=dev(sx), col_scale=dev(sw)))
        c = host(fn(dev(A), Bw, "interleaved"))
    torch.cuda.synchronize()
    assert bq.bq_device_status(reset=True) == bq.BQ_OK
    for b in range(nb):
        c_ref = O.gemm_int(A[b], Bq[b])
        assert (c[b] == c_ref).all(), f"item {b}"
        assert (y[b].view(np.uint16) == O.dequant(c_ref, sw[b], sx[b]).view(np.uint16)).all(), f"item {b}"


def test_batched_one_grid_f16xi4_per_item():
    rng = np.random.default_rng(9)
    nb, M, N, K = 3, 260, 512, 256
    X = W.normal_f16(rng, (nb, M, K), 1.0)
    q = [W.int4_uniform(rng, (N, K)) for _ in range(nb)]
    s = W.uniform_f16(rng, (nb, N), 0.008, 0.016)
    Wp = dev(np.stack([O.pack(qq, 4, "plain") for qq in q]))
    y = host(bq.bq_gemm_f16xi4_batched(dev(X), Wp, dev(s), layout="plain"))
    for b in range(nb):
        assert_f16_close(y[b], O.gemm_f16xq(X[b], q[b], s[b]), s[b][None, :].astype(np.float64), f"item {b}")


def test_activation_none_matches_plain_call():
    rng = np.random.default_rng(11)
    A = W.int8_uniform(rng, (64, 256))
    Bp = dev(O.pack(W.int4_uniform(rng, (192, 256)), 4, "interleaved"))
    sw = dev(W.uniform_f16(rng, (192,), 1e-3, 1e-2))
    a = host(bq.bq_gemm_i8xi4(dev(A), Bp, "interleaved", col_scale=sw))
    b = host(bq.bq_gemm_i8xi4_act(dev(A), Bp, "none", "interleaved", col_scale=sw))
    assert (a.view(np.uint16) == b.view(np.uint16)).all()


@pytest.mark.parametrize("M,N,K", [(2, 320, 2048), (8, 192, 512), (3, 64, 1344), (5, 128, 832)])
@pytest.mark.parametrize("layout", ["interleaved", "plain"])
def test_f16xi4_skinny_staged_activations(M, N, K, layout):
    """Skinny kernel with the activations staged in shared memory (M * K * 2
    bytes up to 8 KB: the first three shapes, 1344 with a ragged last step)
    and just above that limit (read from global memory)."""
    rng = np.random.default_rng(7 * M + N + K)
    X = W.normal_f16(rng, (M, K), 1.0)
    q = W.int4_uniform(rng, (N, K))
    s = W.uniform_f16(rng, (N,), 0.008, 0.016)
    y = host(bq.bq_gemm_f16xi4(dev(X), dev(O.pack(q, 4, layout)), dev(s), layout))
    assert_f16_close(y, O.gemm_f16xq(X, q, s), s[None, :].astype(np.float64), "f16xi4 staged")


@pytest.mark.parametrize("bits,M,N,K", [(4, 7, 128, 1088), (2, 6, 192, 1344), (2, 1, 64, 8192), (4, 8, 64, 1024)])
def test_int_skinny_staged_activations(bits, M, N, K):
    """int8 activations staged in shared memory (M * K bytes up to 8 KB),
    ragged last steps included: exact int32 results."""
    rng = np.random.default_rng(bits * 1000 + M * 31 + K)
    A = W.int8_uniform(rng, (M, K))
    Bq = _codes(rng, bits, (N, K))
    c_ref = O.gemm_int(A, Bq)
    for layout in ("interleaved", "plain"):
        c = host(_run_int_gemm(bits, A, Bq, layout, None, None))
        assert (c == c_ref).all(), f"layout {layout}"


@pytest.mark.parametrize("M,N,K", [(17, 192, 64), (33, 4160, 320), (100, 320, 1088), (128, 448, 4096)])
@pytest.mark.parametrize("layout", ["interleaved", "plain"])
def test_f16xi4_small_m_parity(M, N, K, layout):
    """16 < M <= 128 (weights as the MMA's A operand): a single k-block, K
    with a ragged last raw stage, N not a multiple of the 128 weight rows of
    a block, and M not a multiple of 16."""
    rng = np.random.default_rng(7 * M + N + K)
    X = W.normal_f16(rng, (M, K), 1.0)
    q = W.int4_uniform(rng, (N, K))
    s = W.uniform_f16(rng, (N,), 0.008, 0.016)
    y = host(bq.bq_gemm_f16xi4(dev(X), dev(O.pack(q, 4, layout)), dev(s), layout))
    assert_f16_close(y, O.gemm_f16xq(X, q, s), s[None, :].astype(np.float64), "f16xi4 small M")
    assert bq.bq_device_status(reset=True) == bq.BQ_OK


# ---------------------------------------------------------------------------
# the five workloads at full size (sampled outputs where the oracle would be slow)
# ---------------------------------------------------------------------------
def test_workload_int8xint4_256_int32():
    d = W.cfg0()
    c = bq.bq_gemm_i8xi4(dev(d["A"]), dev(O.pack(d["B"], 4, "plain")), "plain")
    assert (host(c) == O.gemm_int(d["A"], d["B"])).all()


def test_workload_quantize_int8xint8_1024x4096x4096():
    d = W.cfg1()
    xq, sx = bq.bq_quantize_sym(dev(d["X"]), 8)
    wq, sw = bq.bq_quantize_sym(dev(d["W"]), 8)
    y = host(bq.bq_gemm_i8xi8(xq, wq, row_scale=sx, col_scale=sw))
    y_ref, (xq_r, sx_r, wq_r, sw_r, c_r) = O.quantized_linear_i8(d["X"], d["W"])
    s_ij = sx_r[:, None].astype(np.float64) * sw_r[None, :].astype(np.float64)
    assert_f16_close(y, y_ref, s_ij, "quantized linear")


def test_workload_int8xint4_dequant_4096_sampled():
    d = W.cfg2()
    y = host(bq.bq_gemm_i8xi4(dev(d["A"]), dev(O.pack(d["B"], 4, "interleaved")), "interleaved",
                              col_scale=dev(d["scale"])))
    rows = np.r_[np.arange(0, 4096, 61), 4095]
    y_ref = O.dequant(O.gemm_int(d["A"][rows], d["B"]), d["scale"])
    assert_f16_close(y[rows], y_ref, d["scale"][None, :].astype(np.float64), "4096^3")


@pytest.mark.parametrize("M", [1, 4, 16, 64, 256, 1024])
def test_workload_f16xint4_dynamic_m(M):
    d = W.cfg3(M=M)
    s = O.quantize_scale(d["S"], 4)
    Wp = dev(O.pack(d["W"], 4, "interleaved"))
    y = host(bq.bq_gemm_f16xi4(dev(d["X"]), Wp, dev(s), "interleaved"))
    assert_f16_close(y, O.gemm_f16xq(d["X"], d["W"], s), s[None, :].astype(np.float64), f"M={M}")


@pytest.mark.parametrize("M", [1, 128, 1024])
def test_workload_int8xternary(M):
    d = W.cfg4(M=M)
    Bp = dev(O.pack(d["B"], 2, "interleaved"))
    y = host(bq.bq_gemm_i8xi2(dev(d["A"]), Bp, "interleaved", col_scale=dev(d["scale"])))
    rows = np.arange(M) if M <= 128 else np.r_[np.arange(0, M, 17), M - 1]
    y_ref = O.dequant(O.gemm_int(d["A"][rows], d["B"]), d["scale"])
    assert_f16_close(y[rows], y_ref, d["scale"][None, :].astype(np.float64), f"ternary M={M}")
