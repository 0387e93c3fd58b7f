"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Every check here compares the oracle with one of: a value a page prints for a
worked example (``tests/golden``), a closed form worked by hand, an exact
computation in wider precision or rational arithmetic, a numpy library
routine, or brute force on tiny inputs.  Each check is chosen so that a
plausible slip in the oracle (a dropped term, a swapped leading dimension, an
off-by-one in a mask, the wrong fill) makes it fail.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from conftest import read_golden
from masking_tm_affine_gb300 import synth

F32 = np.float32


def f32_bits(x):
    return np.asarray(x, dtype=np.float32).view(np.uint32)


# --------------------------------------------------------------------------
# Tile walk ("Slicing, bounds and masking", "Loops over a dynamic extent")
# --------------------------------------------------------------------------
def test_tile_walk_matches_printed_example(oracle):
    (row,) = read_golden("tile_walk.txt")
    K, T, whole, masked, rem = map(int, row)
    w = oracle.tile_walk(K, T)
    assert (w["whole"], w["masked"], w["rem"]) == (whole, masked, rem)
    assert w["iters"] == whole + masked


@pytest.mark.parametrize("K", list(range(0, 130)) + [1000, 4096, 4100, 8192])
@pytest.mark.parametrize("T", [1, 3, 4, 7, 16, 32, 64, 128])
def test_tile_walk_closed_form(oracle, K, T):
    # floor / remainder / ceiling: whole = K // T; one masked iteration iff K % T
    w = oracle.tile_walk(K, T)
    assert w["whole"] == K // T
    assert w["masked"] == (1 if K % T else 0)
    assert w["rem"] == K % T
    assert w["iters"] == -(-K // T)


def test_tile_walk_rowmax_config(oracle):
    # N = 1000 columns in BC = 64 tiles: 15 whole tiles and one of 40 columns
    w = oracle.tile_walk(1000, 64)
    assert (w["whole"], w["masked"], w["rem"]) == (15, 1, 40)


def test_tile_walk_rejects_nonpositive_tile(oracle):
    with pytest.raises(ValueError):
        oracle.tile_walk(10, 0)
    with pytest.raises(ValueError):
        oracle.tile_walk(10, -4)


# --------------------------------------------------------------------------
# Per-tile mask ("Slicing, bounds and masking", "Masking" figure)
# --------------------------------------------------------------------------
def _brute_valid(M, N, TM, TN, pm, pn):
    mask = np.zeros(((pm + 1) * TM + 8, (pn + 1) * TN + 8), dtype=bool)
    mask[:M, :N] = True
    return int(mask[pm * TM:(pm + 1) * TM, pn * TN:(pn + 1) * TN].sum())


def test_tile_mask_matches_printed_example(oracle):
    (row,) = read_golden("tile_mask.txt")
    TM, TN, ba, bb, valid, total, masked, mult = map(int, row)
    assert valid + masked == total == TM * TN
    # Search every extent pair that is a multiple of 4 (the page's assumption)
    # for those where block (ba, bb) holds exactly `valid` in-bounds elements.
    # Both readings of the block index order are checked (rows first, or
    # columns first); each must have the 4 x 4 corner as its unique solution.
    for pm, pn in [(ba, bb), (bb, ba)]:
        hits = []
        for M in range(mult, 65, mult):
            for N in range(mult, 65, mult):
                v = oracle.tile_valid(M, N, TM, TN, pm, pn)
                assert v == _brute_valid(M, N, TM, TN, pm, pn)
                if v == valid:
                    hits.append((M, N))
        assert hits == [(pm * TM + 4, pn * TN + 4)]


@pytest.mark.parametrize("M,N,TM,TN", [(4100, 1000, 64, 64), (20, 28, 8, 8), (8192, 8192, 32, 128),
                                       (1, 1, 32, 128), (37, 5, 16, 16)])
def test_tile_valid_partition(oracle, M, N, TM, TN):
    # the tiles partition the tensor: the valid counts add up to M*N, and a
    # tile is whole exactly when it lies inside both extents
    mt, nt = -(-M // TM), -(-N // TN)
    if M * N > 200000:
        # spot-check the classes the ragged workload has: interior, right edge,
        # bottom edge, corner (closed form min(TM, M - pm*TM) * min(TN, N - pn*TN))
        picks = {(0, 0), (0, nt - 1), (mt - 1, 0), (mt - 1, nt - 1)}
        total = 0
        for pm, pn in picks:
            v = oracle.tile_valid(M, N, TM, TN, pm, pn)
            assert v == min(TM, M - pm * TM) * min(TN, N - pn * TN)
        whole_m, whole_n = M // TM, N // TN
        rm, rn = M % TM, N % TN
        total = whole_m * whole_n * TM * TN + whole_m * TM * rn + rm * whole_n * TN + rm * rn
        assert total == M * N
    else:
        total = sum(oracle.tile_valid(M, N, TM, TN, pm, pn) for pm in range(mt) for pn in range(nt))
        assert total == M * N


def test_ragged_copy_tile_census(oracle):
    # [4100, 1000] in 64 x 64 tiles: 65 x 16 = 1040 tiles; 960 whole; 64 on the
    # right edge with 40 columns; 15 on the bottom edge with 4 rows; 1 corner 4 x 40
    M, N, T = 4100, 1000, 64
    counts = {}
    for pm in (0, 64):
        for pn in (0, 15):
            counts[(pm, pn)] = oracle.tile_valid(M, N, T, T, pm, pn)
    assert counts[(0, 0)] == 4096
    assert counts[(0, 15)] == 64 * 40
    assert counts[(64, 0)] == 4 * 64
    assert counts[(64, 15)] == 4 * 40
    assert 960 * 4096 + 64 * 64 * 40 + 15 * 4 * 64 + 4 * 40 == M * N


def test_promise(oracle):
    assert oracle.promise_kept(8192, 8192, 32, 128)
    assert not oracle.promise_kept(4100, 1000, 64, 64)
    assert not oracle.promise_kept(8192, 8100, 32, 128)
    assert not oracle.promise_kept(8190, 8192, 32, 128)
    assert oracle.promise_kept(0, 0, 64, 64)
    with pytest.raises(ValueError):
        oracle.promise_kept(64, 64, 0, 64)


# --------------------------------------------------------------------------
# Affine map out = a*2 + 1 ("Aligned Load & Store", "The exercise")
# --------------------------------------------------------------------------
FLT_MAX = float(np.finfo(np.float32).max)
# (a, expected) worked by hand from out = 2a + 1 with one rounding to float32
AFFINE_HAND = [
    (-0.5, 0.0), (-1.0, -1.0), (0.5, 2.0), (0.0, 1.0), (3.0, 7.0), (-3.0, -5.0),
    (0.25, 1.5), (1e-30, 1.0), (-1e-30, 1.0), (1e-45, 1.0),
    (4194304.5, 8388610.0),        # 2^22 + 0.5 -> 2^23 + 2, exact
    (8388607.5, 16777216.0),       # 2^23 - 0.5 -> 2^24, exact
    (8388608.0, 16777216.0),       # 2^24 + 1 is a tie -> even neighbour 2^24
    (8388609.0, 16777220.0),       # 2^24 + 3 is a tie -> even neighbour 2^24 + 4
    (FLT_MAX, math.inf), (-FLT_MAX, -math.inf), (math.inf, math.inf), (-math.inf, -math.inf),
]


def test_affine_hand_values(oracle):
    a = np.array([p[0] for p in AFFINE_HAND], dtype=np.float32)
    want = np.array([p[1] for p in AFFINE_HAND], dtype=np.float32)
    got = oracle.affine(a)
    assert np.array_equal(f32_bits(got), f32_bits(want)), list(zip(a, got, want))


def test_affine_negative_zero_and_nan(oracle):
    got = oracle.affine(np.array([-0.0, np.nan], dtype=np.float32))
    assert f32_bits(got[0]) == f32_bits(F32(1.0))   # -0*2 + 1 = +1
    assert np.isnan(got[1])


def _round_exact_to_f32(q: Fraction) -> np.float32:
    """Round an exact rational to the nearest float32 (ties to even), by
    bracketing it between adjacent float32 values."""
    lo = np.float32(float(q))  # a nearby float32 (float() of a Fraction is correctly rounded)
    # walk to the float32 pair that brackets q
    while Fraction(float(lo)) > q:
        lo = np.nextafter(lo, np.float32(-np.inf))
    hi = np.nextafter(lo, np.float32(np.inf))
    while Fraction(float(hi)) < q:
        lo, hi = hi, np.nextafter(hi, np.float32(np.inf))
    dlo, dhi = q - Fraction(float(lo)), Fraction(float(hi)) - q
    if dlo < dhi:
        return lo
    if dhi < dlo:
        return hi
    return lo if (int(f32_bits(lo)) & 1) == 0 else hi


def test_affine_single_rounding_exact_rationals(oracle):
    # the exact value 2a + 1 in rational arithmetic, rounded once to float32
    g = synth.rng(1234)
    bits = g.integers(0, 2**32, size=600, dtype=np.uint64).astype(np.uint32)
    a = bits.view(np.float32)
    a = a[np.isfinite(a) & (np.abs(a) < 1e30)]
    a = np.concatenate([a, synth.uniform((200,), -1.0, 1.0, 7)])
    got = oracle.affine(a)
    for ai, gi in zip(a, got):
        want = _round_exact_to_f32(2 * Fraction(float(ai)) + 1)
        assert f32_bits(gi) == f32_bits(want), (ai, gi, want)


def test_affine_config_invariant(oracle):
    # on the 1M-element workload: 2a + 1 is exact in float64 for every |a| < 1,
    # so one rounding of it is the answer; and for a in [-1, -0.5] the float32
    # result needs no rounding at all (Sterbenz), so out - 1 == 2a exactly
    a = synth.workload_input("affine_1m")
    out = oracle.affine(a)
    exact = 2.0 * a.astype(np.float64) + 1.0
    assert np.array_equal(out, exact.astype(np.float32))
    neg = (a >= -1.0) & (a <= -0.5)
    assert neg.sum() > 100000
    assert np.array_equal(out[neg].astype(np.float64) - 1.0, 2.0 * a[neg].astype(np.float64))


# --------------------------------------------------------------------------
# Scale Y = alpha*X ("@aligned", "A minimal kernel") and masking
# --------------------------------------------------------------------------
def _canary_buf(M, ld, extra=64):
    return np.full(M * ld + extra, synth.CANARY_U32, dtype=np.uint32).view(np.float32)


@pytest.mark.parametrize("M,N,ldx,ldy", [(5, 7, 7, 7), (6, 33, 37, 41), (1, 1, 1, 3), (0, 5, 5, 5),
                                         (5, 0, 4, 4), (20, 28, 32, 36)])
def test_scale2d_exact_and_masked(oracle, M, N, ldx, ldy):
    alpha = np.float32(1.5)
    x = synth.normal((max(M, 1), max(N, 1)), 11)[:M, :N]
    X = synth.pad_rows(x, ldx) if M and N else np.full(max(M * ldx, 1), synth.POISON_F32, np.float32)
    Y = _canary_buf(M, ldy)
    oracle.scale2d(X, ldx, Y, ldy, M, N, alpha)
    Yv = Y[: M * ldy].reshape(M, ldy) if M else Y[:0].reshape(0, ldy)
    # in bounds: the exact product (exact in float64: 24 + 24 bits) rounded once
    want = (x.astype(np.float64) * np.float64(alpha)).astype(np.float32)
    assert np.array_equal(f32_bits(Yv[:, :N]), f32_bits(want))
    # every other word (ld gap and past the end) keeps its canary
    assert np.all(f32_bits(Yv[:, N:]) == synth.CANARY_U32)
    assert np.all(f32_bits(Y[M * ldy:]) == synth.CANARY_U32)


def test_scale2d_hand_values(oracle):
    X = np.array([2.0, -4.0, 0.0, -0.0, 1e-45, np.inf], dtype=np.float32)
    Y = np.zeros(6, dtype=np.float32)
    oracle.scale2d(X, 6, Y, 6, 1, 6, 1.5)
    # 1.5 * 2^-149 lies halfway between 2^-149 and 2^-148; ties-to-even picks 2^-148
    want = np.array([3.0, -6.0, 0.0, -0.0, 2.0**-148, np.inf], dtype=np.float32)
    assert np.array_equal(f32_bits(Y), f32_bits(want))


# --------------------------------------------------------------------------
# Copy B = A ("Slicing, bounds and masking", "Promising whole tiles with @aligned")
# --------------------------------------------------------------------------
def test_copy2d_bitwise_with_payloads_and_gaps(oracle):
    M, N, lda, ldb = 9, 13, 16, 20
    g = synth.rng(5)
    A = g.integers(0, 2**32, size=M * lda, dtype=np.uint64).astype(np.uint32)
    A[:4] = [0x7FA00001, 0xFFC12345, 0x80000000, 0x00000001]   # sNaN, qNaN payload, -0, denormal
    B = np.full(M * ldb + 32, synth.CANARY_U32, dtype=np.uint32)
    oracle.copy2d(A, lda, B, ldb, M, N)
    Bv = B[: M * ldb].reshape(M, ldb)
    assert np.array_equal(Bv[:, :N], A.reshape(M, lda)[:, :N])   # numpy slicing as the reference
    assert np.all(Bv[:, N:] == synth.CANARY_U32)
    assert np.all(B[M * ldb:] == synth.CANARY_U32)


@pytest.mark.parametrize("M", range(0, 10))
def test_copy2d_brute_force_tiny(oracle, M):
    for N in range(0, 10):
        ld = N + 3
        A = np.arange(max(M * ld, 1), dtype=np.uint32) + 1
        B = np.zeros(M * ld + 8, dtype=np.uint32)
        oracle.copy2d(A, ld, B, ld, M, N)
        want = np.zeros_like(B)
        for i in range(M):
            for j in range(N):
                want[i * ld + j] = A[i * ld + j]
        assert np.array_equal(B, want)


# --------------------------------------------------------------------------
# Row and column sums ("Memory Coalescing and Tensor Layout", "What it actually costs")
# --------------------------------------------------------------------------
@pytest.mark.parametrize("M,N,ld", [(7, 11, 13), (64, 33, 33), (1, 1000, 1003), (300, 2, 8)])
def test_sums_closed_form(oracle, M, N, ld):
    # X[i, j] = i + 2j; ld-gap words hold 3e38 poison, so a gap read shows
    i = np.arange(M, dtype=np.float64)[:, None]
    j = np.arange(N, dtype=np.float64)[None, :]
    x = (i + 2 * j).astype(np.float32)
    X = synth.pad_rows(x, ld)
    r = oracle.rowsum(X, ld, M, N)
    c = oracle.colsum(X, ld, M, N)
    ii = np.arange(M, dtype=np.float64)
    jj = np.arange(N, dtype=np.float64)
    assert np.array_equal(r, N * ii + N * (N - 1))                 # sum_j (i + 2j)
    assert np.array_equal(c, M * (M - 1) / 2 + 2 * jj * M)         # sum_i (i + 2j)


def test_sums_accumulate_in_fp64(oracle):
    x = np.array([[1e8, 1.0, -1e8, 1.0]], dtype=np.float32)        # fp32 left-to-right gives 1
    assert oracle.rowsum(x, 4, 1, 4)[0] == 2.0
    assert np.array_equal(oracle.colsum(x.T.copy(), 1, 4, 1), [2.0])


def test_sums_match_exact_fsum(oracle):
    x = synth.uniform((40, 4096), 0.0, 1.0, 3)
    r = oracle.rowsum(x, 4096, 40, 4096)
    c = oracle.colsum(x.T.copy(), 40, 4096, 40)
    for k in range(40):
        exact = math.fsum(x[k].astype(np.float64))
        bound = 4096 * 2.0**-53 * math.fsum(np.abs(x[k].astype(np.float64)))
        assert abs(r[k] - exact) <= bound
        assert abs(c[k] - exact) <= bound


def test_sums_transpose_invariant(oracle):
    x = synth.normal((37, 53), 9)
    assert np.array_equal(oracle.colsum(x, 53, 37, 53), oracle.rowsum(x.T.copy(), 37, 53, 37))


def test_sums_empty(oracle):
    assert oracle.rowsum(np.zeros(1, np.float32), 0, 0, 0).shape == (0,)
    assert np.array_equal(oracle.rowsum(np.zeros(4, np.float32), 1, 4, 0), np.zeros(4))
    assert np.array_equal(oracle.colsum(np.zeros(4, np.float32), 4, 0, 4), np.zeros(4))


# --------------------------------------------------------------------------
# Ragged row-max ("Slicing, bounds and masking", "Reductions over a ragged tile")
# --------------------------------------------------------------------------
@pytest.mark.parametrize("N", [0, 1, 4, 39, 40, 63, 64, 65, 128, 1000])
@pytest.mark.parametrize("BC", [16, 64])
def test_rowmax_neg_inf_fill_is_plain_max(oracle, N, BC):
    M, ld = 9, N + 5
    s = synth.normal((M, max(N, 1)), 21)[:, :N] * np.float32(10.0)
    s[0] = -np.abs(s[0]) - np.float32(1.0)                        # an all-negative row
    S = synth.pad_rows(s, ld)
    m = oracle.rowmax_masked(S, ld, M, N, BC, oracle.FILL_NEG_INF)
    if N == 0:
        assert np.all(m == -np.inf)
    else:
        assert np.array_equal(m, s.max(axis=1))                   # numpy's max as the reference
        assert m[0] < 0


@pytest.mark.parametrize("N,BC", [(1000, 64), (40, 64), (128, 64), (1000, 8), (5, 16)])
def test_rowmax_zero_fill_pitfall(oracle, N, BC):
    # the page's pitfall: negative scores padded with zeros have a max of 0
    M = 6
    s = synth.uniform((M, N), -30.0, -1.0, 4)
    m0 = oracle.rowmax_masked(s, N, M, N, BC, oracle.FILL_ZERO)
    mi = oracle.rowmax_masked(s, N, M, N, BC, oracle.FILL_NEG_INF)
    assert np.array_equal(mi, s.max(axis=1))
    assert np.all(mi < 0)
    if N % BC:
        assert np.all(f32_bits(m0) == f32_bits(F32(0.0)))         # exactly +0, never the true max
    else:
        assert np.array_equal(m0, mi)                              # no padding, no pitfall


def test_rowmax_fill_below_page_literal(oracle):
    # scores below -1e30 in a ragged row: a -1e30 fill would win; -inf never does
    s = np.full((1, 40), -3.0e38, dtype=np.float32)
    s[0, 7] = -2.0e38
    m = oracle.rowmax_masked(s, 40, 1, 40, 64, oracle.FILL_NEG_INF)
    assert m[0] == np.float32(-2.0e38)


def test_rowmax_nan_ignored(oracle):
    s = np.array([[np.nan, -5.0, -3.0, np.nan, -4.0]], dtype=np.float32)
    m = oracle.rowmax_masked(s, 5, 1, 5, 4, oracle.FILL_NEG_INF)
    assert m[0] == np.nanmax(s)


def test_rowmax_config_workload(oracle):
    # [8192, 1000] at BC = 64 (15 whole tiles + one of 40): sampled rows
    s = synth.workload_input("rowmax_8192")
    assert s.max() < 0
    rows = s[:256]
    m = oracle.rowmax_masked(rows, 1000, 256, 1000, 64, oracle.FILL_NEG_INF)
    assert np.array_equal(m, rows.max(axis=1))
    assert np.all(m != 0)
    for k in range(0, 256, 17):                                   # the max is an element of its row
        assert m[k] in rows[k]


# --------------------------------------------------------------------------
# Unit convention of the measurements ("What it actually costs", table)
# --------------------------------------------------------------------------
def test_bandwidth_units_match_page_table():
    from bench import gbps
    for access, rows, cols, nbytes, t_us, bw in read_golden("coalescing_table.txt"):
        assert int(nbytes) == int(rows) * int(cols) * 4 == 2**26
        assert abs(gbps(int(nbytes), float(t_us) * 1e-6) - float(bw)) / float(bw) < 1e-3


# --------------------------------------------------------------------------
# Softmax row statistics (the softmax of "Reductions over a ragged tile")
# --------------------------------------------------------------------------
def test_softmax_stats_constant_rows(oracle):
    # s = c everywhere: m = c and every term is exp(0) = 1, so l = N exactly
    for N, BC in [(1, 64), (40, 64), (64, 64), (1000, 64), (7, 16)]:
        s = np.full((3, N), -7.25, dtype=np.float32)
        m, l = oracle.softmax_rowstats(s, N, 3, N, BC)
        assert np.all(m == np.float32(-7.25)) and np.all(l == float(N))


def test_softmax_stats_match_scipy_logsumexp(oracle):
    from scipy.special import logsumexp
    s = synth.uniform((20, 1000), -30.0, -1.0, 4)
    m, l = oracle.softmax_rowstats(s, 1000, 20, 1000, 64)
    assert np.array_equal(m, s.max(axis=1))
    lse = logsumexp(s.astype(np.float64), axis=1)
    assert np.allclose(m.astype(np.float64) + np.log(l), lse, rtol=0, atol=1e-12)


def test_softmax_stats_two_values_by_hand(oracle):
    # scores {2, 2 - ln 3}: m = 2 and l = 1 + e^(-ln 3) = 4/3, up to the float32
    # rounding of the second score (exactly 1 + exp(s1 - 2) with math.exp)
    s = np.array([[2.0, 2.0 - np.log(3.0)]], dtype=np.float32)
    m, l = oracle.softmax_rowstats(s, 2, 1, 2, 64)
    assert m[0] == np.float32(2.0)
    assert abs(l[0] - (1.0 + math.exp(float(s[0, 1]) - 2.0))) < 1e-15
    assert abs(l[0] - 4.0 / 3.0) < 1e-7


def test_softmax_stats_zero_fill_pitfall(oracle):
    # negative scores, ragged last tile, no where step: padding zeros win the max
    # and each padded column adds exp(0 - 0) = 1 to l
    N, BC = 1000, 64
    s = synth.uniform((5, N), -30.0, -1.0, 8)
    m0, l0 = oracle.softmax_rowstats(s, N, 5, N, BC, oracle.FILL_ZERO)
    pad = BC - N % BC
    assert np.all(m0 == 0.0)
    want = np.exp(s.astype(np.float64)).sum(axis=1) + pad
    assert np.allclose(l0, want, rtol=1e-13, atol=0)
    mi, li = oracle.softmax_rowstats(s, N, 5, N, BC, oracle.FILL_NEG_INF)
    assert np.all(mi < 0) and np.all(li >= 1.0) and np.all(li < N)


def test_softmax_stats_empty_and_infinite(oracle):
    m, l = oracle.softmax_rowstats(np.zeros(4, np.float32), 1, 4, 0, 64)
    assert np.all(m == -np.inf) and np.all(l == 0.0)
    s = np.full((1, 10), -np.inf, dtype=np.float32)
    m, l = oracle.softmax_rowstats(s, 10, 1, 10, 16)
    assert m[0] == -np.inf and l[0] == 0.0
    s[0, 3] = -5.0
    m, l = oracle.softmax_rowstats(s, 10, 1, 10, 16)
    assert m[0] == np.float32(-5.0) and l[0] == 1.0


# --------------------------------------------------------------------------
# Per-channel scale and bias ("Memory Coalescing and Tensor Layout", "NCHW versus NHWC")
# --------------------------------------------------------------------------
def _fma_exact(x, s, b):
    """fl(x*s + b) with one rounding: the exact rational, rounded to float32."""
    return _round_exact_to_f32(Fraction(float(x)) * Fraction(float(s)) + Fraction(float(b)))


def test_channel_affine_single_rounding(oracle):
    g = synth.rng(31)
    R, C = 40, 12
    x = synth.normal((R, C), 32)
    sc = synth.uniform((C,), 0.25, 4.0, 33)
    bi = synth.normal((C,), 34)
    Y = np.zeros(R * C, np.float32)
    oracle.channel_affine(x, C, R, C, sc, bi, C, oracle.CHANNELS_LAST, Y, C)
    Yv = Y.reshape(R, C)
    for i in range(0, R, 3):
        for j in range(C):
            assert f32_bits(Yv[i, j]) == f32_bits(_fma_exact(x[i, j], sc[j], bi[j]))


def test_channel_affine_layouts_agree_with_4d_broadcast(oracle):
    # the same [B, C, H, W] tensor through both views equals numpy's fp64
    # broadcast rounded to fp32 (that double rounding could differ from one
    # rounding at rare ties -- none occurs for these seeded values; the exact
    # rational test above pins the single rounding itself)
    B, C, H, W = 3, 5, 4, 6
    t = synth.normal((B, C, H, W), 35)
    sc = synth.uniform((C,), 0.5, 2.0, 36)
    bi = synth.uniform((C,), -1.0, 1.0, 37)
    want = (t.astype(np.float64) * sc[None, :, None, None] + bi[None, :, None, None]).astype(np.float32)
    # channels first: rows b*C + c of length H*W
    Y1 = np.zeros(t.size, np.float32)
    oracle.channel_affine(t.reshape(-1), H * W, B * C, H * W, sc, bi, C, oracle.CHANNELS_FIRST, Y1, H * W)
    assert np.array_equal(Y1.reshape(B, C, H, W), want)
    # channels last: the NHWC copy as [B*H*W, C]
    nhwc = np.ascontiguousarray(t.transpose(0, 2, 3, 1))
    Y2 = np.zeros(t.size, np.float32)
    oracle.channel_affine(nhwc.reshape(-1), C, B * H * W, C, sc, bi, C, oracle.CHANNELS_LAST, Y2, C)
    assert np.array_equal(Y2.reshape(B, H, W, C).transpose(0, 3, 1, 2), want)


def test_channel_affine_bias_only_scale_only_and_gaps(oracle):
    R, K, ld = 7, 9, 13
    x = synth.normal((R, K), 38)
    X = synth.pad_rows(x, ld)
    bi = synth.normal((K,), 39)
    sc = synth.normal((K,), 40)
    Y = np.full(R * ld, synth.CANARY_U32, np.uint32).view(np.float32)
    oracle.channel_affine(X, ld, R, K, None, bi, K, oracle.CHANNELS_LAST, Y, ld)
    Yv = Y.reshape(R, ld)
    assert np.array_equal(Yv[:, :K], x + bi[None, :])            # one rounding of x + b
    assert np.all(f32_bits(Yv[:, K:]) == synth.CANARY_U32)
    oracle.channel_affine(X, ld, R, K, sc, None, K, oracle.CHANNELS_LAST, Y, ld)
    assert np.array_equal(Yv[:, :K], x * sc[None, :])            # one rounding of x * s
    with pytest.raises(ValueError):
        oracle.channel_affine(X, ld, R, K, sc, bi, K - 1, oracle.CHANNELS_LAST, Y, ld)


# --------------------------------------------------------------------------
# Keeping the promise by padding ("@aligned", "Interactions";
# "Memory Coalescing and Tensor Layout", "The alignment constraint")
# --------------------------------------------------------------------------
@pytest.mark.parametrize("extent", [0, 1, 31, 32, 33, 255, 256, 1000, 4100, 8192, 8193])
@pytest.mark.parametrize("tiles", [[32], [64], [32, 256], [4, 16], [64, 128, 256], [3, 5]])
def test_padded_extent_is_lcm_multiple(oracle, extent, tiles):
    L = math.lcm(*tiles)
    got = oracle.padded_extent(extent, tiles)
    assert got == -(-extent // L) * L                      # round up to the lcm (math.lcm as reference)
    assert all(oracle.promise_kept(got, got, t, t) for t in tiles)


def test_padded_extent_autotune_pairing(oracle):
    # the gemm's tuner picks TILE_M from {32, 256}: the host must pad M to a
    # multiple of 256 so that whichever it picks, the promise holds
    assert oracle.padded_extent(1000, [32, 256]) == 1024
    assert oracle.padded_extent(4100, [32, 256]) == 4352
    assert oracle.padded_extent(4100, [64]) == 4160
    with pytest.raises(ValueError):
        oracle.padded_extent(10, [0])


def test_row_stride_16_byte_rows(oracle):
    # 16-byte rows are four fp32 elements: N rounds up to a multiple of 4
    for N in range(0, 40):
        assert oracle.row_stride(N, 16) == -(-N // 4) * 4
        assert oracle.row_stride(N, 32) == -(-N // 8) * 8
    assert oracle.row_stride(1000, 16) == 1000 and oracle.row_stride(1001, 16) == 1004
    with pytest.raises(ValueError):
        oracle.row_stride(10, 6)


@pytest.mark.parametrize("M,N,Mp,Np,lda,ldb", [(5, 7, 8, 8, 7, 8), (0, 3, 4, 4, 3, 4), (3, 0, 4, 4, 1, 6),
                                               (20, 28, 32, 32, 28, 36), (4100, 1000, 4160, 1024, 1000, 1024)])
def test_pad2d_definition_and_sum_invariance(oracle, M, N, Mp, Np, lda, ldb):
    x = synth.normal((max(M, 1), max(N, 1)), 60)[:M, :N]
    A = synth.pad_rows(x, lda) if M and N else np.zeros(max(M * lda, 1), np.float32)
    B = np.full(Mp * ldb + 16, synth.CANARY_U32, np.uint32)
    oracle.pad2d(A, lda, M, N, B, ldb, Mp, Np)
    Bv = B[:Mp * ldb].reshape(Mp, ldb)
    want = np.zeros((Mp, Np), np.float32)
    want[:M, :N] = x                                        # numpy slicing as the reference
    assert np.array_equal(Bv[:, :Np].view(np.float32), want)
    assert np.all(Bv[:, Np:] == synth.CANARY_U32) and np.all(B[Mp * ldb:] == synth.CANARY_U32)
    if M and N:
        # zero padding is the masked-load value: sums over the padded tensor are
        # the sums over the original, exactly
        Bf = Bv.view(np.float32).reshape(-1)
        assert np.array_equal(oracle.rowsum(Bf, ldb, Mp, Np)[:M], oracle.rowsum(A, lda, M, N))
        assert np.array_equal(oracle.colsum(Bf, ldb, Mp, Np)[:N], oracle.colsum(A, lda, M, N))


# --------------------------------------------------------------------------
# The gemm ("@aligned" gemm example; "Loops over a dynamic extent")
# --------------------------------------------------------------------------
def test_gemm_rows_matches_numpy_float64(oracle):
    M, N, K = 37, 29, 1000                               # K = 1000: the page's ragged K
    A = synth.normal((M, K), 70)
    B = synth.normal((K, N), 71)
    C = synth.normal((M, N), 72)
    rows = np.arange(M)
    got = oracle.gemm_rows(A, K, B, N, C, N, rows, N, K, 1.25, -0.5)
    want = (1.25 * (A.astype(np.float64) @ B.astype(np.float64)) - 0.5 * C.astype(np.float64)).astype(np.float32)
    # fp64 sums in different orders: equal after rounding to fp32 except at rare ties
    assert np.mean(got == want) > 0.999
    assert np.allclose(got, want, rtol=1e-6, atol=1e-6)


def test_gemm_rows_closed_forms(oracle):
    # identity B: A @ I = A exactly; all-ones: every entry is the row sum of A
    M, K = 5, 12
    A = synth.uniform((M, K), -4.0, 4.0, 73)
    I = np.eye(K, dtype=np.float32)
    assert np.array_equal(oracle.gemm_rows(A, K, I, K, None, 0, np.arange(M), K, K), A)
    ones = np.ones((K, 3), np.float32)
    got = oracle.gemm_rows(A, K, ones, 3, None, 0, np.arange(M), 3, K)
    rs = A.astype(np.float64).sum(axis=1).astype(np.float32)
    assert np.array_equal(got, np.repeat(rs[:, None], 3, axis=1))
    # beta only (K = 0): C_out = beta * C_in, one rounding
    C = synth.normal((M, 4), 74)
    got = oracle.gemm_rows(A, K, ones, 3, C, 4, np.arange(M), 4, 0, 2.0, 0.75)
    assert np.array_equal(got, (0.75 * C.astype(np.float64)).astype(np.float32))


def test_gemm_rows_row_subset_and_lds(oracle):
    M, N, K, lda, ldb = 50, 20, 33, 40, 24
    A = synth.pad_rows(synth.normal((M, K), 75), lda)
    B = synth.pad_rows(synth.normal((K, N), 76), ldb)          # gaps hold 3e38 poison
    rows = np.array([0, 7, 49])
    got = oracle.gemm_rows(A, lda, B, ldb, None, 0, rows, N, K)
    Af = A.reshape(M, lda)[:, :K].astype(np.float64)
    Bf = B.reshape(K, ldb)[:, :N].astype(np.float64)
    assert np.allclose(got, (Af @ Bf)[rows].astype(np.float32), rtol=1e-6, atol=1e-6)


def test_gemm_rows_exact_rationals_brute_force(oracle):
    # small dyadic entries: every fp64 product and partial sum is exact, so the
    # oracle must equal the exact rational result rounded once to fp32
    from fractions import Fraction
    rng = np.random.Generator(np.random.PCG64(77))
    for M, N, K in [(1, 1, 1), (2, 3, 4), (3, 5, 7), (4, 2, 9)]:
        A = (rng.integers(-64, 65, (M, K)) / 16.0).astype(np.float32)
        B = (rng.integers(-64, 65, (K, N)) / 8.0).astype(np.float32)
        C = (rng.integers(-64, 65, (M, N)) / 4.0).astype(np.float32)
        alpha, beta = -0.75, 1.5
        got = oracle.gemm_rows(A, K, B, N, C, N, np.arange(M), N, K, alpha, beta)
        for i in range(M):
            for j in range(N):
                exact = Fraction(alpha) * sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K)) \
                    + Fraction(beta) * Fraction(float(C[i, j]))
                assert got[i, j] == np.float32(float(exact)), (M, N, K, i, j)


def test_gemm_rows_rounds_once(oracle):
    # 1 + 2^-24 + 2^-24: an fp32 running sum rounds each step back to 1 (ties to
    # even); the definition's exact sum 1 + 2^-23 is an fp32 number
    A = np.array([[1.0, 2.0 ** -24, 2.0 ** -24]], np.float32)
    B = np.ones((3, 1), np.float32)
    got = oracle.gemm_rows(A, 3, B, 1, None, 0, np.arange(1), 1, 3)
    assert got[0, 0] == np.float32(1.0 + 2.0 ** -23)
    f32 = np.float32(0.0)
    for x in A[0]:
        f32 = np.float32(f32 + x)
    assert f32 == np.float32(1.0)       # the mistake this pin catches


def test_gemm_rows_beta_zero_ignores_c(oracle):
    # beta == 0 takes no term from C (BLAS convention): NaN in C stays out
    A = synth.uniform((3, 4), -1.0, 1.0, 78)
    B = synth.uniform((4, 2), -1.0, 1.0, 79)
    C = np.full((3, 2), np.nan, np.float32)
    got = oracle.gemm_rows(A, 4, B, 2, C, 2, np.arange(3), 2, 4, 2.0, 0.0)
    want = oracle.gemm_rows(A, 4, B, 2, None, 0, np.arange(3), 2, 4, 2.0, 0.0)
    assert np.all(np.isfinite(got)) and np.array_equal(got, want)
    # alpha == 0, beta == 1: C passes through unchanged
    C2 = synth.normal((3, 2), 80)
    assert np.array_equal(oracle.gemm_rows(A, 4, B, 2, C2, 2, np.arange(3), 2, 4, 0.0, 1.0), C2)
