"""GPU parity of tm_rowsum / tm_colsum against the fp64 CPU oracle.

"Memory Coalescing and Tensor Layout", "What it actually costs": the same
bytes walked by rows and by columns.  fp32 sums must lie within 1e-5 of the
fp64 oracle relative to sum |x| (the data of the coalescing workload is
non-negative, so that is 1e-5 of the sum itself); integer-valued inputs small
enough to be exact in fp32 must match exactly.
"""
import numpy as np
import pytest

from gpu_util import DevBuf
from masking_tm_affine_gb300 import synth, tm

pytestmark = pytest.mark.gpu

REL = 1e-5
COL_VARIANTS = [tm.TM_VAR_AUTO, tm.TM_VAR_NAIVE, tm.TM_VAR_STAGED, tm.TM_VAR_REGDIRECT, tm.TM_VAR_CLUSTER]


def within(got, want, absref):
    got = np.asarray(got, dtype=np.float64)
    return np.all(np.abs(got - want) <= REL * absref + 1e-30)


def rowsum(X, ld, M, N, TM=8, TN=512, flags=0, lead=0):
    XD = DevBuf(X, lead)
    R = DevBuf.empty(M)
    tm.tm_rowsum(XD.ptr, ld, M, N, R.ptr, TM, TN, flags)
    tm.tm_check()
    assert R.guards_intact() and XD.guards_intact()
    return R.payload_f32()


def colsum(X, ld, M, N, TM=32, TN=128, variant=tm.TM_VAR_AUTO, flags=0, lead=0):
    XD = DevBuf(X, lead)
    C = DevBuf.empty(N)
    ws = tm.tm_colsum_workspace_bytes(M, N, TM, TN, variant if variant == tm.TM_VAR_NAIVE else tm.TM_VAR_AUTO)
    W = DevBuf.empty(max(ws // 4, 1))
    tm.tm_colsum(XD.ptr, ld, M, N, C.ptr, W.ptr, ws, TM, TN, variant, flags)
    tm.tm_check()
    assert C.guards_intact() and W.guards_intact() and XD.guards_intact()
    return C.payload_f32()


@pytest.fixture(scope="module")
def coalesce():
    return synth.workload_input("coalesce_4096")   # [4096, 4096] U[0,1) seed 3, 64 MiB


def test_rowsum_4096_workload(cuda, oracle, coalesce):
    x = coalesce
    want = oracle.rowsum(x, 4096, 4096, 4096)
    for TM, TN, flags in [(8, 512, 0), (8, 512, tm.TM_ALIGNED), (4, 1024, 0), (32, 128, 0),
                          (8, 256, tm.TM_PATH_SCALAR)]:
        got = rowsum(x, 4096, 4096, 4096, TM, TN, flags)
        assert within(got, want, want), (TM, TN, flags)


@pytest.mark.parametrize("variant", COL_VARIANTS)
def test_colsum_4096_workload(cuda, oracle, coalesce, variant):
    x = coalesce
    want = oracle.colsum(x, 4096, 4096, 4096)
    got = colsum(x, 4096, 4096, 4096, 32, 128, variant)
    assert within(got, want, want)
    if variant != tm.TM_VAR_NAIVE:
        got_a = colsum(x, 4096, 4096, 4096, 32, 128, variant, tm.TM_ALIGNED)
        assert within(got_a, want, want)


@pytest.mark.parametrize("M,N", [(1000, 1000), (4096, 1000), (777, 1000), (8192, 1000), (4096, 4096), (8192, 4096)])
def test_colsum_staged_equals_cluster_bitwise(cuda, coalesce, M, N):
    # Both one-pass forms take the same cluster size (16 CTAs per strip for
    # few strips, else 8), split a strip's row tiles the same way and add the
    # same rows to the same lanes in the same order (TMA's zero fill past M
    # adds +0): identical bits
    x = coalesce[:M, :N] if M <= 4096 else np.concatenate([coalesce, coalesce])[:, :N]
    for TM, TN in [(32, 128), (16, 64), (8, 256), (64, 64), (128, 64), (32, 256)]:
        a = colsum(x, N, M, N, TM, TN, tm.TM_VAR_STAGED)
        b = colsum(x, N, M, N, TM, TN, tm.TM_VAR_CLUSTER)
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), (M, N, TM, TN)


@pytest.mark.parametrize("variant", [tm.TM_VAR_STAGED, tm.TM_VAR_CLUSTER, tm.TM_VAR_AUTO])
def test_colsum_one_pass_many_strips(cuda, oracle, variant):
    # many strips: 128 64-column strips of [512, 8192] (8-CTA clusters, all
    # resident), and 512 256-wide strips of a 2^17-wide matrix (8-CTA
    # clusters in several waves; AUTO takes the two-pass form there)
    for M, N, TM, TN in [(512, 8192, 16, 64), (64, 1 << 17, 8, 256), (2048, 8192, 32, 64)]:
        x = synth.uniform((M, N), 0.0, 1.0, M + N)
        got = colsum(x, N, M, N, TM, TN, variant)
        want = oracle.colsum(x, N, M, N)
        assert within(got, want, want), (variant, M, N, TM, TN)


def test_colsum_deterministic(cuda, coalesce):
    a = colsum(coalesce, 4096, 4096, 4096)
    b = colsum(coalesce, 4096, 4096, 4096)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


@pytest.mark.parametrize("M,N,ld", [(1, 1, 1), (1, 4, 4), (3, 7, 9), (37, 129, 131), (100, 1000, 1000),
                                    (257, 260, 264), (1000, 64, 64), (4100, 1000, 1024), (5, 3000, 3001)])
def test_sums_ragged_shapes(cuda, oracle, M, N, ld):
    x = synth.normal((M, N), M + N)
    X = synth.pad_rows(x, ld)                 # 3e38 poison in the gaps: a gap read shows
    absx = np.abs(x.astype(np.float64))
    rw, cw = oracle.rowsum(X, ld, M, N), oracle.colsum(X, ld, M, N)
    for TM, TN in [(8, 128), (1, 256), (32, 1024)]:
        assert within(rowsum(X, ld, M, N, TM, TN), rw, absx.sum(axis=1)), (TM, TN)
    for variant in COL_VARIANTS:
        for TM, TN in [(32, 128), (8, 64), (16, 256), (256, 64)]:
            if variant == tm.TM_VAR_STAGED and (TM * TN > 8192 or TM < 1024 // TN or ld % 4):
                continue
            got = colsum(X, ld, M, N, TM, TN, variant)
            assert within(got, cw, absx.sum(axis=0)), (variant, TM, TN)


def test_sums_integer_inputs_exact(cuda):
    # small integers: every partial sum is exact in fp32, whatever the order
    for M, N in [(513, 772), (513, 770)]:
        x = (synth.rng(2).integers(-8, 9, size=(M, N))).astype(np.float32)
        rw = x.astype(np.int64).sum(axis=1).astype(np.float32)
        cw = x.astype(np.int64).sum(axis=0).astype(np.float32)
        assert np.array_equal(rowsum(x, N, M, N, 8, 256), rw)
        for v in COL_VARIANTS:
            if v == tm.TM_VAR_STAGED and N % 4:
                continue              # TMA needs rows that are whole multiples of 16 bytes
            assert np.array_equal(colsum(x, N, M, N, 32, 128, v), cw), (v, N)


@pytest.mark.parametrize("path", [tm.TM_PATH_SCALAR, tm.TM_PATH_VEC])
def test_sums_forced_paths(cuda, oracle, path):
    M, N = 300, 520
    x = synth.uniform((M, N), 0.0, 1.0, 11)
    rw, cw = oracle.rowsum(x, N, M, N), oracle.colsum(x, N, M, N)
    assert within(rowsum(x, N, M, N, 8, 256, path), rw, rw)
    assert within(colsum(x, N, M, N, 32, 128, tm.TM_VAR_REGDIRECT, path), cw, cw)


def test_sums_misaligned_base(cuda, oracle):
    M, N = 90, 301
    x = synth.uniform((M, N), 0.0, 1.0, 12)
    rw, cw = oracle.rowsum(x, N, M, N), oracle.colsum(x, N, M, N)
    assert within(rowsum(x, N, M, N, 8, 128, lead=1), rw, rw)
    assert within(colsum(x, N, M, N, 32, 128, tm.TM_VAR_AUTO, lead=3), cw, cw)
    assert within(colsum(x, N, M, N, 32, 128, tm.TM_VAR_NAIVE, lead=3), cw, cw)


def test_sums_empty_extents(cuda):
    X = np.zeros(16, np.float32)
    assert np.array_equal(rowsum(X, 4, 4, 0), np.zeros(4, np.float32))        # empty rows sum to 0
    C = DevBuf.empty(7)
    XD = DevBuf(X)
    tm.tm_colsum(XD.ptr, 7, 0, 7, C.ptr, None, 0, 32, 128)                    # no rows: zeros, no scratch
    tm.tm_check()
    assert np.array_equal(C.payload_f32(), np.zeros(7, np.float32)) and C.guards_intact()
    R = DevBuf.empty(3)
    tm.tm_rowsum(XD.ptr, 4, 0, 4, R.ptr, 8, 128)                               # no rows: nothing written
    tm.tm_check()
    assert np.all(R.words() == 0xDEADBEEF)


def test_colsum_workspace_errors(cuda, oracle):
    M, N = 1000, 128                      # 16 row chunks: the one-pass variants need scratch
    x = np.ones((M, N), np.float32)
    XD = DevBuf(x)
    C = DevBuf.empty(N)
    ws = tm.tm_colsum_workspace_bytes(M, N, 32, 128)
    assert ws > 0
    W = DevBuf.empty(ws // 4, lead=1)     # misaligned scratch
    for ptr, nbytes in [(W.ptr, ws), (W.ptr - 4, ws - 4), (None, 0)]:
        for variant in (tm.TM_VAR_AUTO, tm.TM_VAR_REGDIRECT):
            with pytest.raises(tm.TmError) as e:
                tm.tm_colsum(XD.ptr, N, M, N, C.ptr, ptr, nbytes, 32, 128, variant)
            assert e.value.status == tm.TM_ERR_WORKSPACE
    assert np.all(C.words() == 0xDEADBEEF)
    # one chunk per strip: no scratch at all, c written directly
    assert tm.tm_colsum_workspace_bytes(64, N, 32, 128) == 0
    for variant in (tm.TM_VAR_AUTO, tm.TM_VAR_REGDIRECT, tm.TM_VAR_STAGED):
        C = DevBuf.empty(N)
        tm.tm_colsum(XD.ptr, N, 64, N, C.ptr, None, 0, 32, 128, variant)
        tm.tm_check()
        assert C.guards_intact() and np.all(C.payload_f32() == 64.0), variant


def test_colsum_cluster_needs_no_workspace(cuda, oracle):
    # the one-pass variant keeps its partials on chip: NULL workspace, 0 bytes
    M, N = 777, 1000
    x = synth.uniform((M, N), 0.0, 1.0, 13)
    assert tm.tm_colsum_workspace_bytes(M, N, 32, 128, tm.TM_VAR_CLUSTER) == 0
    XD, C = DevBuf(x), DevBuf.empty(N)
    tm.tm_colsum(XD.ptr, N, M, N, C.ptr, None, 0, 32, 128, tm.TM_VAR_CLUSTER)
    tm.tm_check()
    assert C.guards_intact()
    cw = oracle.colsum(x, N, M, N)
    assert within(C.payload_f32(), cw, cw)
    # M == 0: zeros, still without a workspace
    tm.tm_colsum(XD.ptr, N, 0, N, C.ptr, None, 0, 32, 128, tm.TM_VAR_CLUSTER)
    tm.tm_check()
    assert np.all(C.payload_f32() == 0)
