"""Maximum sizes: tensors past 2^31 elements (8.6 - 9.6 GB each), where any
32-bit element offset would wrap.  Inputs are a seeded integer pattern built
on the device; sampled rows (including the last ones) are checked against the
oracle, which computes them one by one."""
import numpy as np
import pytest
import torch

from masking_tm_affine_gb300 import tm

pytestmark = pytest.mark.gpu


def pattern(rows, cols, seed):
    """fp32 values k/64 for small integers k from a seeded hash of the
    position: exact in fp32 and cheap to rebuild on the host."""
    i = torch.arange(rows, device="cuda", dtype=torch.int64)[:, None]
    j = torch.arange(cols, device="cuda", dtype=torch.int64)[None, :]
    h = (i * 1000003 + j * 7919 + seed * 104729) % 2039
    return ((h - 1019).to(torch.float32) / 64.0)


def pattern_host(rows_idx, cols, seed):
    i = np.asarray(rows_idx, dtype=np.int64)[:, None]
    j = np.arange(cols, dtype=np.int64)[None, :]
    h = (i * 1000003 + j * 7919 + seed * 104729) % 2039
    return ((h - 1019).astype(np.float32) / np.float32(64.0))


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.empty_cache()


def test_affine_past_2_31_elements(cuda, oracle):
    n = (1 << 31) + 5
    a = pattern(1, n, 1).reshape(-1)
    out = torch.empty_like(a)
    tm.tm_affine(a, out, n)
    tm.tm_check()
    for start in (0, (1 << 31) - 64, n - 64):
        seg = a[start:start + 64].cpu().numpy()
        assert np.array_equal(out[start:start + 64].cpu().numpy().view(np.uint32), oracle.affine(seg).view(np.uint32))
    del a, out


def test_scale2d_and_copy2d_past_2_31_elements(cuda, oracle):
    M, N = 40001, 60000                           # 2.4e9 elements, ragged for 32 x 128 tiles
    X = pattern(M, N, 2)
    Y = torch.empty_like(X)
    rows = [0, 17, M // 2, M - 2, M - 1]
    tm.tm_scale2d(X, N, Y, N, M, N, 1.5, 32, 128)
    tm.tm_check()
    xs = pattern_host(rows, N, 2)
    want = np.zeros_like(xs)
    oracle.scale2d(xs, N, want, N, len(rows), N, 1.5)
    assert np.array_equal(Y[rows].cpu().numpy(), want)
    tm.tm_copy2d(X, N, Y, N, M, N, 64, 64)
    tm.tm_check()
    assert np.array_equal(Y[rows].cpu().numpy(), xs)
    del X, Y


def test_reductions_past_2_31_elements(cuda, oracle):
    M, N = 70001, 32768                           # 2.3e9 elements
    X = pattern(M, N, 3)
    rows = [0, 1, M // 3, M - 1]
    xs = pattern_host(rows, N, 3)
    r = torch.empty(M, device="cuda")
    tm.tm_rowsum(X, N, M, N, r, 1, 1024)
    m = torch.empty(M, device="cuda")
    tm.tm_rowmax_masked(X, N, M, N, m, 1, 64)
    c = torch.empty(N, device="cuda")
    ws = tm.tm_colsum_workspace_bytes(M, N, 32, 128)
    W = torch.empty(ws // 4, device="cuda")
    tm.tm_colsum(X, N, M, N, c, W, ws, 32, 128)
    tm.tm_check()
    # values are k/64 with |k| <= 1019: every partial sum is exact in fp32 while
    # below 2^24/64, so row sums (|sum| < 2^14) must match exactly
    assert np.array_equal(r[rows].cpu().numpy(), oracle.rowsum(xs, N, len(rows), N).astype(np.float32))
    assert np.array_equal(m[rows].cpu().numpy(), oracle.rowmax_masked(xs, N, len(rows), N, 64))
    # column sums: checked against an exact integer column sum of the pattern
    cols = np.array([0, 1, N // 2, N - 1])
    i = np.arange(M, dtype=np.int64)[:, None]
    h = (i * 1000003 + cols[None, :] * 7919 + 3 * 104729) % 2039
    exact = (h - 1019).sum(axis=0) / 64.0
    got = c.cpu().numpy()[cols].astype(np.float64)
    assert np.all(np.abs(got - exact) <= 1e-5 * (np.abs(h - 1019).sum(axis=0) / 64.0))
    del X, W


def small_pattern(rows, cols, seed, row0=0):
    """fp32 values k/64 with |k| <= 16 from the same kind of seeded hash: with
    K <= 1040 every product and partial sum of two of them is exact in fp32."""
    i = torch.arange(row0, row0 + rows, device="cuda", dtype=torch.int64)[:, None]
    j = torch.arange(cols, device="cuda", dtype=torch.int64)[None, :]
    h = (i * 1000003 + j * 7919 + seed * 104729) % 33
    return ((h - 16).to(torch.float32) / 64.0)


def small_pattern_host(rows_idx, cols, seed):
    i = np.asarray(rows_idx, dtype=np.int64)[:, None]
    j = np.arange(cols, dtype=np.int64)[None, :]
    h = (i * 1000003 + j * 7919 + seed * 104729) % 33
    return ((h - 16).astype(np.float32) / np.float32(64.0))


def test_gemm_past_2_31_elements(cuda, oracle):
    # A [2^21 + 5, 1040]: 2.18e9 elements (8.7 GB), its split operands 17.7 GB;
    # ragged in M (5 rows past a 128-row tile), N (72 of a 128-wide tile) and K
    M, N, K = (1 << 21) + 5, 72, 1040
    A = torch.empty((M, K), dtype=torch.float32, device="cuda")
    step = 1 << 18
    for r0 in range(0, M, step):  # built in slices to bound the index temporaries
        A[r0:r0 + step] = small_pattern(min(step, M - r0), K, 5, r0)
    B = small_pattern(K, N, 6)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    wsb = tm.tm_gemm_workspace_bytes(M, N, K, 128)
    raw = torch.empty(wsb + 1024, dtype=torch.uint8, device="cuda")
    ws = (raw.data_ptr() + 1023) // 1024 * 1024
    tm.tm_gemm(A, K, B, N, C, N, M, N, K, 1.0, 0.0, ws, wsb, 128, 128, 16)
    tm.tm_check()
    rows = [0, 1, 127, 128, M // 2, M - 6, M - 5, M - 1]
    a = small_pattern_host(rows, K, 5)
    b = small_pattern_host(np.arange(K), N, 6)
    want = oracle.gemm_rows(a, K, b, N, None, 0, np.arange(len(rows)), N, K, 1.0, 0.0)
    assert np.array_equal(C[rows].cpu().numpy(), want)
    del A, B, C, raw


def test_one_pass_colsums_with_64_bit_offsets(cuda):
    # (M + 128) * ld > 2^32: the one-pass forms take 64-bit element offsets
    # (and STAGED's tensor map row coordinates pass 2^17); 18.4 GB on the device
    M, N = 140001, 32768
    assert (M + 128) * N > (1 << 32)
    X = torch.empty((M, N), device="cuda")
    for r0 in range(0, M, 8192):  # the pattern in row chunks: bounded temporaries
        r1 = min(M, r0 + 8192)
        i = torch.arange(r0, r1, device="cuda", dtype=torch.int64)[:, None]
        j = torch.arange(N, device="cuda", dtype=torch.int64)[None, :]
        X[r0:r1] = (((i * 1000003 + j * 7919 + 5 * 104729) % 2039) - 1019).to(torch.float32) / 64.0
        del i, j
    got = {}
    for var in (tm.TM_VAR_CLUSTER, tm.TM_VAR_STAGED, tm.TM_VAR_REGDIRECT):
        ws = tm.tm_colsum_workspace_bytes(M, N, 32, 128, var)
        W = torch.empty(max(ws // 4, 4), device="cuda")
        c = torch.full((N,), float("nan"), device="cuda")
        tm.tm_colsum(X, N, M, N, c, W, ws, 32, 128, var)
        tm.tm_check()
        got[var] = c.cpu().numpy()
        del W
    # the two one-pass forms add the same rows in the same order
    assert np.array_equal(got[tm.TM_VAR_CLUSTER].view(np.uint32), got[tm.TM_VAR_STAGED].view(np.uint32))
    cols = np.array([0, 1, 127, 128, N // 2 + 3, N - 1])
    i = np.arange(M, dtype=np.int64)[:, None]
    h = (i * 1000003 + cols[None, :] * 7919 + 5 * 104729) % 2039 - 1019
    exact = h.sum(axis=0) / 64.0
    tol = 1e-5 * (np.abs(h).sum(axis=0) / 64.0)
    for var, c in got.items():
        assert np.all(np.abs(c[cols].astype(np.float64) - exact) <= tol), var
    del X
