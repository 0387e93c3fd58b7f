"""GPU parity of tm_pad2d against the oracle, and the workflow it exists for:
pad a ragged tensor so every candidate tile divides its extents, then run the
unmasked aligned path on it ("@aligned", "Interactions"; "Memory Coalescing
and Tensor Layout", "The alignment constraint")."""
import numpy as np
import pytest

from gpu_util import CANARY, DevBuf, same_f32
from masking_tm_affine_gb300 import synth, tm

pytestmark = pytest.mark.gpu


def pad(x, M, N, lda, Mp, Np, ldb, lead_a=0, lead_b=0):
    A = synth.pad_rows(x, lda) if M and N else np.zeros(max(M * lda, 1), np.float32)
    AD = DevBuf(A, lead_a)
    BD = DevBuf(np.full(Mp * ldb, CANARY, dtype=np.uint32), lead_b)
    tm.tm_pad2d(AD.ptr, lda, M, N, BD.ptr, ldb, Mp, Np)
    tm.tm_check()
    assert BD.guards_intact() and AD.guards_intact()
    return A, BD


@pytest.mark.parametrize("M,N,lda,Mp,Np,ldb", [(1, 1, 1, 1, 1, 1), (5, 7, 7, 8, 8, 8), (20, 28, 28, 32, 32, 36),
                                               (33, 100, 100, 64, 128, 132), (130, 4, 4, 256, 64, 64),
                                               (4100, 1000, 1000, 4160, 1024, 1024), (0, 5, 5, 4, 8, 8),
                                               (6, 0, 1, 8, 4, 4), (37, 33, 35, 40, 41, 43)])
def test_pad2d_matches_oracle(cuda, oracle, M, N, lda, Mp, Np, ldb):
    x = synth.normal((max(M, 1), max(N, 1)), M + N)[:M, :N]
    for lead in (0, 1):
        A, BD = pad(x, M, N, lda, Mp, Np, ldb, lead_a=lead, lead_b=lead)
        want = np.full(Mp * ldb, CANARY, dtype=np.uint32)
        oracle.pad2d(A, lda, M, N, want, ldb, Mp, Np)
        assert np.array_equal(BD.payload_u32(), want)


def test_pad_then_aligned_path(cuda, oracle):
    # the ragged [4100, 1000] tensor, padded for 64 x 64 tiles, runs the
    # unmasked aligned scale; its [4100, 1000] corner equals the oracle's scale
    # of the original, and the padding stays 0
    x = synth.workload_input("ragged_4100")
    M, N = x.shape
    Mp, Np = tm.tm_padded_extent(M, [64]), tm.tm_padded_extent(N, [64])
    ldb = tm.tm_row_stride(Np, 16)
    assert (Mp, Np, ldb) == (4160, 1024, 1024)
    A, BD = pad(x, M, N, N, Mp, Np, ldb)
    YD = DevBuf.empty(Mp * ldb)
    tm.tm_scale2d(BD.ptr, ldb, YD.ptr, ldb, Mp, Np, 1.5, 64, 64, tm.TM_ALIGNED)
    tm.tm_check()
    y = YD.payload_f32().reshape(Mp, ldb)
    want = np.zeros(M * N, np.float32)
    oracle.scale2d(x, N, want, N, M, N, 1.5)
    assert same_f32(y[:M, :N], want.reshape(M, N))
    assert np.all(y[M:, :Np] == 0) and np.all(y[:, N:Np] == 0)
    # sums over the padded tensor equal the sums over the original, row by row
    R = DevBuf.empty(Mp)
    tm.tm_rowsum(BD.ptr, ldb, Mp, Np, R.ptr, 1, 1024, tm.TM_ALIGNED)
    tm.tm_check()
    rw = oracle.rowsum(x, N, M, N)
    assert np.all(np.abs(R.payload_f32()[:M] - rw) <= 1e-5 * oracle.rowsum(np.abs(x), N, M, N))
    assert np.all(R.payload_f32()[M:] == 0)


def test_pad2d_errors(cuda):
    AD = DevBuf(np.zeros(64, np.float32))
    BD = DevBuf.empty(64)
    for args in [(8, 8, 8, 4, 8, 8), (8, 8, 8, 8, 4, 8), (8, 8, 8, 8, 8, 7)]:   # Mp < M, Np < N, ldb < Np
        M, N, lda, Mp, Np, ldb = args
        with pytest.raises(tm.TmError) as e:
            tm.tm_pad2d(AD.ptr, lda, M, N, BD.ptr, ldb, Mp, Np)
        assert e.value.status == tm.TM_ERR_INVALID_ARG
    with pytest.raises(tm.TmError) as e:
        tm.tm_pad2d(AD.ptr, 8, 4, 4, AD.ptr + 64, 8, 4, 8)                   # overlap
    assert e.value.status == tm.TM_ERR_INVALID_ARG
    assert np.all(BD.words() == CANARY)
