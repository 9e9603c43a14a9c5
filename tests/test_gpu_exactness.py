"""GPU exactness and error-path tests, through the C ABI.

* Integer sums whose partial sums pass 2**24 while the total cancels: the
  int8 x int8 products reach 2**14, so a fp32 chain of more than 1024 k would
  round odd partial sums, and a result near zero would then miss the fp16
  tolerance 1e-3 * sx * sw by orders of magnitude.  Every dispatch path
  (split-K clusters, TMEM slices, CTA pairs with chunked accumulation) must
  give the exact int32 sum, and the fp16 epilogue must start from it.
* The fp32 accumulation margin of the fp16 x INT4 workload over several seeds.
* Bounded waits: a zero time limit makes every kernel family report
  BQ_ERR_TIMEOUT (no fault, no hang), and the next call is correct.
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


def err_over_tol(y, y_ref, scale_ij):
    """Largest |y - y_ref| / max(1e-3 |y_ref|, 1e-3 s_ij) over finite entries
    (infinities must match exactly)."""
    y = y.astype(np.float64)
    y_ref = y_ref.astype(np.float64)
    fin = np.isfinite(y_ref)
    assert (np.isfinite(y) == fin).all(), "inf pattern differs"
    assert (y[~fin] == y_ref[~fin]).all(), "inf sign differs"
    tol = np.maximum(1e-3 * np.abs(y_ref), 1e-3 * np.broadcast_to(scale_ij, y_ref.shape).astype(np.float64))
    return float(np.max(np.abs(y - y_ref)[fin] / tol[fin])) if fin.any() else 0.0


def cancelling_inputs(seed, M, N, K):
    """int8 operands whose sums climb far past 2**24 and then cancel.

    Row i of A is a block of large codes of one sign per row followed by its
    negation; row j of B repeats its first half in the second half with a
    perturbation in {-1, 0, 1} (none for every third row).  So
    C[i, j] = -sum_k A[i, k] * delta[j, k] is small (zero for the unperturbed
    rows) while every prefix of the first half is about 2048 * 113 * 113."""
    rng = np.random.default_rng(seed)
    h = K // 2
    sign = np.where(rng.integers(0, 2, size=(M, 1)) == 0, -1, 1)
    a_half = (rng.integers(100, 128, size=(M, h)) * sign).astype(np.int64)
    A = np.concatenate([a_half, -a_half], axis=1).astype(np.int8)
    b_half = rng.integers(100, 127, size=(N, h)).astype(np.int64)
    delta = rng.integers(-1, 2, size=(N, h))
    delta[::3] = 0
    B = np.concatenate([b_half, b_half + delta], axis=1).astype(np.int8)
    sw = W.uniform_f16(rng, (N,), 1e-3, 1e-2)
    sx = W.uniform_f16(rng, (M,), 1e-3, 1e-1)
    return A, B, sw, sx


def describe_mismatch(c, c_ref, rows):
    """Where and by how much an integer result differs (for the failure message)."""
    bad = np.argwhere(c != c_ref)
    d = c.astype(np.int64) - c_ref.astype(np.int64)
    vals = d[c != c_ref]
    return (f"{len(bad)} of {c.size} differ; rows {sorted(set(rows[bad[:, 0]].tolist()))[:12]}; "
            f"cols mod 256 {sorted(set((bad[:, 1] % 256).tolist()))[:24]}; "
            f"diffs {vals[:8].tolist()}; diff mod 8192 {sorted(set((vals % 8192).tolist()))[:8]}")


def sample_rows(M, n=48):
    return np.unique(np.r_[np.linspace(0, M - 1, n).astype(int), M - 1])


# (M, N, K): split-K clusters (chains of <= 16 k-blocks per CTA), four TMEM
# slices of 1024 k, CTA pairs with chunked accumulation (one, two and eight
# chunk boundaries, and the 1024 x 4096 x 4096 quantised-linear shape)
CANCEL_SHAPES = [(40, 192, 4096), (900, 2048, 4096), (600, 8192, 1088), (600, 8192, 1984), (600, 8192, 4096),
                 (1024, 4096, 4096), (600, 4096, 8192)]


@pytest.mark.parametrize("M,N,K", CANCEL_SHAPES)
def test_i8xi8_cancellation_exact(M, N, K):
    A, B, sw, sx = cancelling_inputs(M + N + K, M, N, K)
    rows = sample_rows(M)
    c_ref = O.gemm_int(A[rows], B)
    Ad, Bd = dev(A), dev(B)
    c = host(bq.bq_gemm_i8xi8(Ad, Bd))
    assert (c[rows] == c_ref).all(), "int32 sums: " + describe_mismatch(c[rows], c_ref, rows)
    assert bq.bq_device_status(reset=True) == bq.BQ_OK
    y = host(bq.bq_gemm_i8xi8(Ad, Bd, row_scale=dev(sx), col_scale=dev(sw)))
    s_ij = sx[rows, None].astype(np.float64) * sw[None, :].astype(np.float64)
    r = err_over_tol(y[rows], O.dequant(c_ref, sw, sx[rows]), s_ij)
    assert r <= 1.0, f"fp16 epilogue err/tol {r:.3g}"
    yc = host(bq.bq_gemm_i8xi8(Ad, Bd, col_scale=dev(sw)))
    r = err_over_tol(yc[rows], O.dequant(c_ref, sw), sw[None, :].astype(np.float64))
    assert r <= 1.0, f"fp16 column-scale epilogue err/tol {r:.3g}"
    assert bq.bq_device_status(reset=True) == bq.BQ_OK


def test_i8xi8_cancellation_activation():
    """Chunked accumulation followed by the fused ReLU (CTA pairs)."""
    M, N, K = 600, 8192, 2048
    A, B, sw, sx = cancelling_inputs(5, M, N, K)
    rows = sample_rows(M)
    y = host(bq.bq_gemm_i8xi8_act(dev(A), dev(B), "relu", row_scale=dev(sx), col_scale=dev(sw)))
    y_ref = O.dequant(O.gemm_int(A[rows], B), sw, sx[rows], act="relu")
    s_ij = sx[rows, None].astype(np.float64) * sw[None, :].astype(np.float64)
    assert err_over_tol(y[rows], y_ref, s_ij) <= 1.0


def test_i8xi8_chunk_extremes_exact():
    """Chunked accumulation at the edges of its range (CTA pairs, K = 4416:
    chunks of 16, 16, 16, 16 and 5 k-blocks).  Even rows x even columns are
    all (-128)(-128), so every full chunk sums to exactly 2**24.  Odd rows x
    odd columns: the first two chunks sum to 1, which leaves the lowest
    remainder L = -8191, and every later chunk adds 1024 products -128 * 127
    on top of it (-16654335 at its end)."""
    M, N, K = 600, 8192, 4416
    A = np.zeros((M, K), np.int8)
    B = np.zeros((N, K), np.int8)
    A[0::2] = -128
    B[0::2] = -128
    A[1::2, 0] = 1
    A[1::2, 1024] = 1
    A[1::2, 2048:] = -128
    B[1::2, 0] = 1
    B[1::2, 1024] = 1
    B[1::2, 2048:] = 127
    rows = np.r_[0, 1, 2, 3, M - 2, M - 1]
    c_ref = O.gemm_int(A[rows], B)
    assert c_ref[0, 0] == K * 16384 and c_ref[1, 1] == 2 - (K - 2048) * 16256
    Ad, Bd = dev(A), dev(B)
    c = host(bq.bq_gemm_i8xi8(Ad, Bd))
    assert (c[rows] == c_ref).all(), describe_mismatch(c[rows], c_ref, rows)
    sw = W.uniform_f16(np.random.default_rng(7), (N,), 1e-3, 1e-2)
    y = host(bq.bq_gemm_i8xi8(Ad, Bd, col_scale=dev(sw)))
    r = err_over_tol(y[rows], O.dequant(c_ref, sw), sw[None, :].astype(np.float64))
    assert r <= 1.0, f"fp16 epilogue err/tol {r:.3g}"
    assert bq.bq_device_status(reset=True) == bq.BQ_OK


def test_i8xi8_int32_long_k_exact():
    """int32 output with K = 16384 (CTA pairs, 17 chunk boundaries): every
    product is (-128)(-128) or 127(-128), so |C| reaches 2**28."""
    M, N, K = 640, 4096, 16384
    A = np.full((M, K), -128, np.int8)
    A[1::2, ::5] = 127
    B = np.full((N, K), -128, np.int8)
    B[::3, 1::2] = 127
    rows = np.r_[0, 1, 2, 3, M - 2, M - 1]
    cols = np.r_[0, 1, 2, 3, N - 3, N - 2, N - 1]
    c = host(bq.bq_gemm_i8xi8(dev(A), dev(B)))
    c_ref = O.gemm_int(A[rows], B[cols])
    assert (c[np.ix_(rows, cols)] == c_ref).all(), describe_mismatch(c[np.ix_(rows, cols)], c_ref, rows)


# ---------------------------------------------------------------------------
# accumulation margin of the fp16 x INT4 workload (11008 x 4096 layer)
# ---------------------------------------------------------------------------
MARGIN_SEEDS = [0, 1, 2, 3, 4]


def margin_stats(y, y_ref, s):
    """(worst error in fp16 ulps of the reference where the relative
    tolerance rules, worst err/tol overall, worst err/tol where the absolute
    tolerance 1e-3 * s_j is the larger one).

    Wherever the relative tolerance rules, one ulp of fp16 is at most
    2**-10 < 1e-3 of the value, so a result one rounding step away from the
    correctly rounded one is always inside it (err/tol <= 0.977).  Near
    zero, where 1e-3 * s_j rules, err/tol measures the accumulation error."""
    y = y.astype(np.float64)
    yr = y_ref.astype(np.float64)
    err = np.abs(y - yr)
    ulp = np.spacing(np.abs(y_ref.astype(np.float16))).astype(np.float64)
    s_ij = np.broadcast_to(s[None, :].astype(np.float64), yr.shape)
    tol = np.maximum(1e-3 * np.abs(yr), 1e-3 * s_ij)
    near0 = 1e-3 * s_ij > 1e-3 * np.abs(yr)
    return float(np.max((err / ulp)[~near0])), float(np.max(err / tol)), float(np.max((err / tol)[near0]))


@pytest.mark.parametrize("M", [1, 64, 1024])
def test_f16xint4_margin_over_seeds(M):
    """Away from zero every output is within one fp16 step of the correctly
    rounded value; near zero the accumulation error is at most 0.9 of the
    absolute tolerance; everything inside the tolerance.  Five seeds of the
    full layer."""
    rows = []
    for seed in MARGIN_SEEDS:
        d = W.cfg3(seed=seed, M=M)
        s = O.quantize_scale(d["S"], 4)
        y = host(bq.bq_gemm_f16xi4(dev(d["X"]), dev(O.pack(d["W"], 4, "interleaved")), dev(s), "interleaved"))
        rows.append(margin_stats(y, O.gemm_f16xq(d["X"], d["W"], s), s))
    print(f"M={M}: (ulps, err/tol, near-zero err/tol) per seed {[tuple(round(v, 3) for v in r) for r in rows]}")
    assert max(r[0] for r in rows) <= 1.0, "more than one fp16 step from the correctly rounded value"
    assert max(r[1] for r in rows) <= 1.0
    assert max(r[2] for r in rows) <= 0.9, "accumulation error near zero uses more than 0.9 of the tolerance"


# ---------------------------------------------------------------------------
# bounded waits: every kernel family gives up at a zero limit, reports it and
# leaves the context usable
# ---------------------------------------------------------------------------
def _i8xi4_call(M, N, K):
    rng = np.random.default_rng(M + N + K)
    A = W.int8_uniform(rng, (M, K))
    B = W.int4_uniform(rng, (N, K))
    Ad, Bp = dev(A), dev(O.pack(B, 4, "interleaved"))
    ref = O.gemm_int(A, B)
    return (lambda: bq.bq_gemm_i8xi4(Ad, Bp, "interleaved")), ref, None


def _i8xi8_call(M, N, K):
    rng = np.random.default_rng(M + N + K)
    A = W.int8_uniform(rng, (M, K))
    B = W.int8_uniform(rng, (N, K))
    Ad, Bd = dev(A), dev(B)
    return (lambda: bq.bq_gemm_i8xi8(Ad, Bd)), O.gemm_int(A, B), None


def _f16xi4_call(M, N, K):
    rng = np.random.default_rng(M + N + K)
    X = W.normal_f16(rng, (M, K), 1.0)
    q = W.int4_uniform(rng, (N, K))
    s = W.uniform_f16(rng, (N,), 0.008, 0.016)
    Xd, Wp, sd = dev(X), dev(O.pack(q, 4, "interleaved")), dev(s)
    return (lambda: bq.bq_gemm_f16xi4(Xd, Wp, sd, "interleaved")), O.gemm_f16xq(X, q, s), s


WAIT_CASES = {
    "split_k_clusters": (_i8xi4_call, (256, 256, 1024)),
    "cta_pairs": (_i8xi4_call, (600, 8192, 256)),
    "cta_pairs_chunked": (_i8xi8_call, (600, 8192, 2048)),
    "skinny": (_f16xi4_call, (1, 320, 512)),
    "small_m": (_f16xi4_call, (40, 4160, 320)),
}


@pytest.mark.parametrize("case", list(WAIT_CASES))
def test_wait_timeout_fires_and_recovers(case):
    make, shape = WAIT_CASES[case]
    call, ref, s = make(*shape)
    torch.cuda.synchronize()
    assert bq.bq_device_status(reset=True) == bq.BQ_OK
    old = bq.bq_set_wait_timeout_ns(0)          # give up at the first unsuccessful poll
    seen = []
    try:
        for _ in range(5):
            call()
            torch.cuda.synchronize()
            seen.append(bq.bq_device_status(reset=True))
            if seen[-1] == bq.BQ_ERR_TIMEOUT:
                break
    finally:
        bq.bq_set_wait_timeout_ns(old)
    assert bq.BQ_ERR_TIMEOUT in seen, f"{case}: no wait gave up in {len(seen)} calls ({seen})"
    assert set(seen) <= {bq.BQ_OK, bq.BQ_ERR_TIMEOUT}
    out = host(call())
    if s is None:
        assert (out == ref).all()
    else:
        assert err_over_tol(out, ref, s[None, :].astype(np.float64)) <= 1.0
    assert bq.bq_device_status(reset=True) == bq.BQ_OK
