"""CPU checks of the arithmetic of the chunked int8 x int8 accumulation.

The CTA-pair kernel sums K in chunks of 16 k-blocks of 64 in fp32 tensor
memory.  After a chunk it splits each accumulator value D (an integer) as
D = 8192 h + L with u = RU(D * 2**-13 + 1.5 * 2**23) (one fma rounded toward
+infinity): h = u - 1.5 * 2**23 = ceil(D / 8192), and L = D - 8192 h, which
lies in (-8192, 0], is written back.  The epilogue splits the two final
accumulators the same way with round-to-nearest, adds the high parts as
integers, and rounds 8192 H + (L0 + L1) once to fp32 with one fma.  These
tests replay those fp32 steps with exact float64 intermediates (every
intermediate here is exact in float64) and one rounding to fp32 in the stated
mode, and check them against their definitions.  Neither the library nor the
oracle is involved.
"""

import numpy as np

MAGIC = 12582912.0          # 1.5 * 2**23
MAGIC_BITS = 0x4B400000     # its fp32 bit pattern
PROD_MIN, PROD_MAX = -128 * 127, 128 * 128
CHUNK = 16 * 64             # products per chunk


def rn(x):
    """Round float64 values (exact intermediates) to fp32, to nearest even."""
    return np.asarray(x, np.float64).astype(np.float32)


def ru(x):
    """Round float64 values to fp32 toward +infinity."""
    x = np.asarray(x, np.float64)
    f = x.astype(np.float32)
    low = f.astype(np.float64) < x
    f[low] = np.nextafter(f[low], np.float32(np.inf))
    return f


def bits(f):
    return f.view(np.uint32).astype(np.int64)


def split(d, up):
    """(u, h, L) of the kernel's split of integer-valued fp32 values d."""
    d64 = d.astype(np.float64)
    u = (ru if up else rn)(d64 * 2.0 ** -13 + MAGIC)
    h = u.astype(np.float64) - MAGIC
    low = rn(-8192.0 * h + d64)                     # fma(-8192, u - magic, d), u - magic exact
    return u, h.astype(np.int64), low.astype(np.float64)


def sample_accumulators(rng, n):
    """Integers the accumulators can hold: the chunk range and its edges."""
    lo, hi = -8191 + CHUNK * PROD_MIN, CHUNK * PROD_MAX
    edges = np.array([lo, hi, 0, 1, -1, 4096, -4096, 8192, -8192, 8193, -8193, 12288, -12288, 2 ** 24 - 1], np.int64)
    return np.concatenate([edges, rng.integers(lo, hi + 1, n), rng.integers(-20000, 20000, n)])


def test_chunk_on_the_remainder_stays_exact_in_fp32():
    """A chunk of 16 k-blocks started on L in (-8192, 0] keeps every partial
    sum within +-2**24, where fp32 holds every integer."""
    assert CHUNK * PROD_MAX <= 2 ** 24                       # a fresh chunk, all (-128)(-128)
    assert -8191 + CHUNK * PROD_MIN >= -(2 ** 24)              # the lowest remainder, all -128 * 127
    assert 0 + CHUNK * PROD_MAX <= 2 ** 24                     # the highest remainder is 0
    # a round-to-nearest split (|L| <= 4096) would not allow 16 k-blocks
    assert 4096 + CHUNK * PROD_MAX > 2 ** 24


def test_round_up_split_is_ceil_and_exact():
    rng = np.random.default_rng(0)
    d = sample_accumulators(rng, 400000)
    df = d.astype(np.float32)
    assert (df.astype(np.int64) == d).all()
    u, h, low = split(df, up=True)
    assert (h == -((-d) // 8192)).all(), "h = ceil(D / 8192)"
    assert (8192 * h + low.astype(np.int64) == d).all() and (low == np.round(low)).all()
    assert ((low > -8192) & (low <= 0)).all()
    assert (bits(u) == MAGIC_BITS + h).all(), "u's pattern is that of 1.5 * 2**23 plus h"
    assert (((bits(u) & 0xFFFF) - h) % 65536 == 0).all(), "its low 16 bits are h modulo 2**16"


def test_nearest_split_is_rint_and_exact():
    rng = np.random.default_rng(1)
    d = sample_accumulators(rng, 400000)
    u, h, low = split(d.astype(np.float32), up=False)
    assert (h == np.round(d / 8192.0).astype(np.int64)).all(), "h = rint(D / 8192), ties to even"
    assert (8192 * h + low.astype(np.int64) == d).all() and (np.abs(low) <= 4096).all()


def test_epilogue_sum_rounds_once():
    """8192 H + L, with H = h0 + h1 + the drained high parts and L = L0 + L1,
    rounded once by an fma equals the int32 sum rounded to fp32 (what an
    int-to-float conversion of the exact sum gives); the int32 form equals the
    sum itself."""
    rng = np.random.default_rng(2)
    n = 300000
    d0 = sample_accumulators(rng, n)[: 2 * n]
    d1 = rng.permutation(sample_accumulators(rng, n))[: d0.size]
    hd = rng.integers(-12288, 12289, d0.size)                  # drained high parts (int16 range at K <= 8192)
    # sums half way between two fp32 values (2**24 + 1 and 2**25 + 8190, where fp32 steps by 2 and 4) and
    # the lowest accumulators with the lowest drained parts
    top = 2 ** 24
    d0[:6] = [top - 1, top - 1, top - 1, top, -16654335, -16654335]
    d1[:6] = [2, top - 1, top - 1, top, -16654335, 1]
    hd[:6] = [0, 0, 1, 0, -12288, 0]
    exact = d0 + d1 + 8192 * hd
    u0, h0, l0 = split(d0.astype(np.float32), up=False)
    u1, h1, l1 = split(d1.astype(np.float32), up=False)
    big_h = h0 + h1 + hd
    assert ((bits(u0) + bits(u1) - MAGIC_BITS + hd) == MAGIC_BITS + big_h).all()
    assert (np.abs(big_h) < 2 ** 22).all()
    low = rn(l0 + l1).astype(np.float64)
    assert (low == l0 + l1).all() and (np.abs(low) <= 8192).all()  # the low sum is exact
    hf = rn((big_h + MAGIC_BITS).astype(np.uint32).view(np.float32).astype(np.float64) - MAGIC)
    assert (hf.astype(np.int64) == big_h).all()
    y = rn(8192.0 * hf.astype(np.float64) + low)                 # one fma
    assert exact[0] == top + 1 and exact[2] % 4 == 2                 # two ties (fp32 steps of 2 and 4 there)
    assert (y == exact.astype(np.float32)).all(), "one rounding of the exact sum"
    # the int32 branch: 8192 H + int(L), with int(L) from the pattern of L + 1.5 * 2**23
    li = bits(rn(low + MAGIC)) - MAGIC_BITS
    assert (big_h * 8192 + li == exact).all()
