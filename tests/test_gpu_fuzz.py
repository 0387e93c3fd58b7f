"""Seeded random cases of every entry point against the oracle.

Each case draws its own extents (1 .. ~600), leading dimensions (ld >= N,
sometimes not a multiple of 4), start offsets (0 .. 3 floats, so 16-byte
alignment comes and goes), tile from the instantiated set, flags (the aligned
promise only where it holds) and, for the reductions and the column sum,
variant and fill -- the combinations the hand-picked tests do not reach.
Maps and maxima must match the oracle bit for bit, sums within 1e-5 of
sum |x| ("Slicing, bounds and masking", "Masking"; "Memory Coalescing and
Tensor Layout", "What it actually costs").  Every buffer carries canaries.
"""
import numpy as np
import pytest

from gpu_util import CANARY, DevBuf, same_f32
from masking_tm_affine_gb300 import synth, tm

pytestmark = pytest.mark.gpu

MAP_TILES = [(8, 8), (16, 16), (32, 32), (64, 64), (32, 128), (128, 128)]
CASES = 60


def draw_matrix(rng, M, N, ld):
    x = synth.uniform((M, N), -8.0, 8.0, int(rng.integers(1 << 30)))
    return synth.pad_rows(x, ld), x


def extents(rng):
    M = int(rng.integers(1, 600))
    N = int(rng.integers(1, 600))
    if rng.random() < 0.5:
        N = (N + 3) // 4 * 4  # vector-friendly half the time
    ld = N + int(rng.choice([0, 0, 1, 3, 4, 8]))
    return M, N, ld


@pytest.mark.parametrize("case", range(CASES))
def test_maps_random(cuda, oracle, case):
    rng = np.random.default_rng(1000 + case)
    M, N, ldx = extents(rng)
    ldy = N + int(rng.choice([0, 2, 4]))
    TM, TN = MAP_TILES[int(rng.integers(len(MAP_TILES)))]
    lead_x, lead_y = int(rng.integers(4)), int(rng.integers(4))
    X, _ = draw_matrix(rng, M, N, ldx)
    aligned = (M % TM == 0 and N % TN == 0 and ldx % 4 == 0 and ldy % 4 == 0 and lead_x == 0 and lead_y == 0)
    flags = tm.TM_ALIGNED if aligned and rng.random() < 0.7 else 0
    if rng.random() < 0.2:
        flags |= tm.TM_PATH_SCALAR
    op = ["scale", "copy"][case % 2]
    XD = DevBuf(X, lead_x)
    YD = DevBuf(np.full(M * ldy, CANARY, dtype=np.uint32), lead_y)
    if op == "scale":
        tm.tm_scale2d(XD.ptr, ldx, YD.ptr, ldy, M, N, 1.5, TM, TN, flags)
    else:
        tm.tm_copy2d(XD.ptr, ldx, YD.ptr, ldy, M, N, TM, TN, flags)
    tm.tm_check()
    assert XD.guards_intact() and YD.guards_intact()
    want = np.full(M * ldy, CANARY, dtype=np.uint32)
    if op == "scale":
        oracle.scale2d(X, ldx, want.view(np.float32), ldy, M, N, 1.5)
        assert same_f32(YD.payload_f32(), want.view(np.float32)), (M, N, ldx, ldy, TM, TN, flags, lead_x, lead_y)
    else:
        oracle.copy2d(X, ldx, want, ldy, M, N)
        assert np.array_equal(YD.payload_u32(), want), (M, N, ldx, ldy, TM, TN, flags, lead_x, lead_y)


@pytest.mark.parametrize("case", range(CASES))
def test_row_reductions_random(cuda, oracle, case):
    rng = np.random.default_rng(2000 + case)
    M, N, ld = extents(rng)
    lead = int(rng.integers(4))
    X, x = draw_matrix(rng, M, N, ld)
    TM = int(rng.choice([1, 2, 4, 8, 16, 32]))
    TN = int(rng.choice([16, 32, 64, 128, 256, 512, 1024]))
    flags = tm.TM_PATH_SCALAR if rng.random() < 0.2 else 0
    XD = DevBuf(X, lead)
    R, Mx = DevBuf.empty(M), DevBuf.empty(M)
    tm.tm_rowsum(XD.ptr, ld, M, N, R.ptr, TM, TN, flags)
    fill = tm.TM_FILL_ZERO if rng.random() < 0.3 else tm.TM_FILL_NEG_INF
    BC = int(rng.choice([16, 32, 64, 128, 256, 512]))
    tm.tm_rowmax_masked(XD.ptr, ld, M, N, Mx.ptr, TM, BC, fill, flags)
    tm.tm_check()
    assert XD.guards_intact() and R.guards_intact() and Mx.guards_intact()
    absx = np.abs(x.astype(np.float64)).sum(axis=1)
    r_want = oracle.rowsum(X, ld, M, N)
    assert np.all(np.abs(R.payload_f32().astype(np.float64) - r_want) <= 1e-5 * absx + 1e-30), (M, N, ld, TM, TN)
    m_want = oracle.rowmax_masked(X, ld, M, N, BC, fill)
    assert same_f32(Mx.payload_f32(), m_want), (M, N, ld, TM, BC, fill)


@pytest.mark.parametrize("case", range(CASES))
def test_column_sums_random(cuda, oracle, case):
    rng = np.random.default_rng(3000 + case)
    M, N, ld = extents(rng)
    lead = int(rng.integers(4))
    X, x = draw_matrix(rng, M, N, ld)
    variant = [tm.TM_VAR_AUTO, tm.TM_VAR_NAIVE, tm.TM_VAR_STAGED, tm.TM_VAR_REGDIRECT, tm.TM_VAR_CLUSTER][case % 5]
    TM = int(rng.choice([8, 16, 32, 64]))
    TN = int(rng.choice([64, 128, 256]))
    if variant == tm.TM_VAR_STAGED:
        # the TMA tile needs 16-byte rows and a staged shape; fall back to REGDIRECT otherwise
        if not (lead == 0 and ld % 4 == 0 and TM * TN <= 8192 and TM >= 1024 // TN):
            variant = tm.TM_VAR_REGDIRECT
    ws = tm.tm_colsum_workspace_bytes(M, N, TM, TN, variant if variant == tm.TM_VAR_NAIVE else tm.TM_VAR_AUTO)
    XD = DevBuf(X, lead)
    C = DevBuf.empty(N)
    W = DevBuf.empty(max(ws // 4, 4))
    tm.tm_colsum(XD.ptr, ld, M, N, C.ptr, W.ptr, max(ws, 16), TM, TN, variant, 0)
    tm.tm_check()
    assert XD.guards_intact() and C.guards_intact() and W.guards_intact()
    absx = np.abs(x.astype(np.float64)).sum(axis=0)
    want = oracle.colsum(X, ld, M, N)
    got = C.payload_f32().astype(np.float64)
    assert np.all(np.abs(got - want) <= 1e-5 * absx + 1e-30), (M, N, ld, TM, TN, variant, lead)


@pytest.mark.parametrize("case", range(CASES // 2))
def test_softmax_and_affine_random(cuda, oracle, case):
    rng = np.random.default_rng(4000 + case)
    M, N, ld = extents(rng)
    lead = int(rng.integers(4))
    X, x = draw_matrix(rng, M, N, ld)
    BR = int(rng.choice([1, 4, 8, 16]))
    BC = int(rng.choice([16, 64, 256]))
    XD = DevBuf(X, lead)
    Mx, L = DevBuf.empty(M), DevBuf.empty(M)
    tm.tm_softmax_rowstats(XD.ptr, ld, M, N, Mx.ptr, L.ptr, BR, BC, tm.TM_FILL_NEG_INF, 0)
    n = int(rng.integers(1, 5000))
    a = synth.uniform(n, -1.0, 1.0, int(rng.integers(1 << 30)))
    AD, OD = DevBuf(a, int(rng.integers(8))), DevBuf.empty(n, int(rng.integers(8)))
    variant = [tm.TM_VAR_AUTO, tm.TM_VAR_SCALAR, tm.TM_VAR_VEC_UNALIGNED][case % 3]
    tm.tm_affine(AD.ptr, OD.ptr, n, variant)
    tm.tm_check()
    assert XD.guards_intact() and Mx.guards_intact() and L.guards_intact() and OD.guards_intact()
    m_want, l_want = oracle.softmax_rowstats(X, ld, M, N, BC)
    assert same_f32(Mx.payload_f32(), m_want)
    assert np.all(np.abs(L.payload_f32().astype(np.float64) - l_want) <= 1e-5 * np.abs(l_want))
    assert same_f32(OD.payload_f32(), oracle.affine(a))


@pytest.mark.parametrize("case", range(40))
def test_gemm_random_integers_exact(cuda, oracle, case):
    """Integer-valued operands (every product and partial sum exact): random
    extents, strides, offsets, tiles, modes and alpha, beta, bit for bit."""
    rng = np.random.default_rng(5000 + case)
    M, N, K = (int(rng.integers(1, 400)) for _ in range(3))
    lda, ldb, ldc = K + int(rng.integers(4)), N + int(rng.integers(4)), N + int(rng.integers(5))
    TM = int(rng.choice([128, 256]))
    TN = int(rng.choice([128, 256]))
    TK = int(rng.choice([16, 32]))
    flags = tm.TM_GEMM_TF32 if rng.random() < 0.3 else 0
    alpha, beta = float(rng.choice([1.0, -2.0, 0.5])), float(rng.choice([0.0, 1.0, 0.25]))
    ints = lambda shape: np.round(synth.uniform(shape, -8.5, 8.5, int(rng.integers(1 << 30)))).astype(np.float32)
    a, b, c = ints((M, K)), ints((K, N)), ints((M, N))
    Ah, Bh, Ch = synth.pad_rows(a, lda), synth.pad_rows(b, ldb), synth.pad_rows(c, ldc)
    AD, BD, CD = DevBuf(Ah, int(rng.integers(4))), DevBuf(Bh, int(rng.integers(4))), DevBuf(Ch, int(rng.integers(4)))
    import torch
    wsb = tm.tm_gemm_workspace_bytes(M, N, K, TN)
    raw = torch.empty(wsb + 1024, dtype=torch.uint8, device="cuda")
    ws = (raw.data_ptr() + 1023) // 1024 * 1024
    tm.tm_gemm(AD.ptr, lda, BD.ptr, ldb, CD.ptr, ldc, M, N, K, alpha, beta, ws, wsb, TM, TN, TK, flags)
    tm.tm_check()
    assert AD.guards_intact() and BD.guards_intact() and CD.guards_intact()
    want = oracle.gemm_rows(Ah, lda, Bh, ldb, Ch, ldc, np.arange(M), N, K, alpha, beta)
    got = CD.payload_f32().reshape(M, ldc)
    assert np.array_equal(got[:, :N].view(np.uint32), want.view(np.uint32)), (M, N, K, TM, TN, TK, flags)
    # the ld gap of C is never written
    assert np.array_equal(CD.payload_u32().reshape(M, ldc)[:, N:], Ch.view(np.uint32).reshape(M, ldc)[:, N:])


@pytest.mark.parametrize("case", range(30))
def test_channel_affine_and_pad_random(cuda, oracle, case):
    rng = np.random.default_rng(6000 + case)
    # channel affine: either layout, either parameter vector absent, random tile and strides
    layout = [tm.TM_CHANNELS_LAST, tm.TM_CHANNELS_FIRST][case % 2]
    C = int(rng.integers(1, 300))
    R, K = (int(rng.integers(1, 500)), C) if layout == tm.TM_CHANNELS_LAST else \
        (C * int(rng.integers(1, 6)), int(rng.integers(1, 500)))
    if layout == tm.TM_CHANNELS_LAST and rng.random() < 0.3:
        K = int(rng.integers(1, C + 1))  # fewer columns than channels
    ldx, ldy = K + int(rng.integers(5)), K + int(rng.integers(5))
    TM, TN = MAP_TILES[int(rng.integers(len(MAP_TILES)))]
    sc = synth.uniform((C,), 0.5, 2.0, int(rng.integers(1 << 30))) if rng.random() < 0.8 else None
    bi = synth.normal((C,), int(rng.integers(1 << 30))) if (sc is None or rng.random() < 0.8) else None
    x = synth.normal((R, K), int(rng.integers(1 << 30)))
    X = synth.pad_rows(x, ldx)
    XD, YD = DevBuf(X, int(rng.integers(4))), DevBuf(np.full(R * ldy, CANARY, dtype=np.uint32), int(rng.integers(4)))
    lead_p = int(rng.integers(4))
    SD = None if sc is None else DevBuf(sc, lead_p)
    BD = None if bi is None else DevBuf(bi, lead_p)
    tm.tm_channel_affine(XD.ptr, ldx, R, K, None if SD is None else SD.ptr, None if BD is None else BD.ptr, C, layout,
                         YD.ptr, ldy, TM, TN, 0)
    # pad2d: random source and padded extents and strides
    M, N = int(rng.integers(0, 300)), int(rng.integers(0, 300))
    Mp, Np = M + int(rng.integers(0, 40)), N + int(rng.integers(0, 40))
    lda, ldb = max(N, 1) + int(rng.integers(4)), max(Np, 1) + int(rng.integers(4))
    a = synth.normal((max(M, 1), max(N, 1)), int(rng.integers(1 << 30)))[:M, :N]
    A = synth.pad_rows(a, lda) if M and N else np.zeros(max(M * lda, 1), np.float32)
    AD = DevBuf(A, int(rng.integers(4)))
    PD = DevBuf(np.full(max(Mp * ldb, 1), CANARY, dtype=np.uint32), int(rng.integers(4)))
    tm.tm_pad2d(AD.ptr, lda, M, N, PD.ptr, ldb, Mp, Np)
    tm.tm_check()
    assert XD.guards_intact() and YD.guards_intact() and AD.guards_intact() and PD.guards_intact()
    want = np.full(R * ldy, CANARY, dtype=np.uint32).view(np.float32)
    oracle.channel_affine(X, ldx, R, K, sc, bi, C, layout, want, ldy)
    assert same_f32(YD.payload_f32(), want), (layout, C, R, K, ldx, ldy, TM, TN, sc is None, bi is None)
    want_p = np.full(max(Mp * ldb, 1), CANARY, dtype=np.uint32)
    if Mp and Np:
        oracle.pad2d(A, lda, M, N, want_p, ldb, Mp, Np)
    assert np.array_equal(PD.payload_u32(), want_p), (M, N, lda, Mp, Np, ldb)
