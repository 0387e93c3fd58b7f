"""GPU parity of tm_softmax_rowstats against the CPU oracle.

"Slicing, bounds and masking", "Reductions over a ragged tile": with the
-inf fill the statistics of a ragged row are those of its real scores; with
the zero fill (the pitfall) padding enters both.  m must equal the oracle bit
for bit (max is exact); l, an fp32 sum of CUDA expf values rescaled online,
must lie within 1e-5 relative of the fp64 oracle (every term is positive and
the largest is exp(0) = 1, so l >= 1 whenever N > 0).
"""
import numpy as np
import pytest

from gpu_util import DevBuf, same_f32
from masking_tm_affine_gb300 import synth, tm

pytestmark = pytest.mark.gpu
REL = 1e-5


def stats(S, ld, M, N, BR=4, BC=64, fill=tm.TM_FILL_NEG_INF, flags=0, lead=0):
    SD = DevBuf(S, lead)
    MD, LD = DevBuf.empty(M), DevBuf.empty(M)
    tm.tm_softmax_rowstats(SD.ptr, ld, M, N, MD.ptr, LD.ptr, BR, BC, fill, flags)
    tm.tm_check()
    assert MD.guards_intact() and LD.guards_intact() and SD.guards_intact()
    return MD.payload_f32(), LD.payload_f32()


def close(l_gpu, l_ref):
    l_gpu = l_gpu.astype(np.float64)
    fin = np.isfinite(l_ref)
    return (np.array_equal(np.isnan(l_gpu), np.isnan(l_ref)) and
            np.all(np.abs(l_gpu[fin] - l_ref[fin]) <= REL * np.abs(l_ref[fin])))


def test_softmax_stats_8192x1000_workload(cuda, oracle):
    s = synth.workload_input("rowmax_8192")        # U[-30,-1) seed 4, BC = 64: 15 whole tiles + 1 of 40
    mw, lw = oracle.softmax_rowstats(s, 1000, 8192, 1000, 64)
    for BR in (1, 4, 8):
        m, l = stats(s, 1000, 8192, 1000, BR)
        assert np.array_equal(m, mw), BR
        assert close(l, lw), BR
    m0, l0 = stats(s, 1000, 8192, 1000, 4, fill=tm.TM_FILL_ZERO)
    mw0, lw0 = oracle.softmax_rowstats(s, 1000, 8192, 1000, 64, oracle.FILL_ZERO)
    assert np.all(m0.view(np.uint32) == 0) and np.array_equal(m0, mw0)
    assert close(l0, lw0)


@pytest.mark.parametrize("BC", [16, 64, 256])
@pytest.mark.parametrize("N", [0, 1, 4, 15, 40, 63, 64, 65, 100, 999, 1000, 1024])
def test_softmax_stats_tiles_and_extents(cuda, oracle, BC, N):
    M, ld = 37, N + 5
    s = synth.normal((M, max(N, 1)), N + BC)[:, :N] * np.float32(4.0)
    S = synth.pad_rows(s, ld)                      # +3e38 in the gaps: a gap read would become the max
    for fill in (oracle.FILL_NEG_INF, oracle.FILL_ZERO):
        mw, lw = oracle.softmax_rowstats(S, ld, M, N, BC, fill)
        for BR in (1, 8, 32):
            m, l = stats(S, ld, M, N, BR, BC, fill)
            assert same_f32(m, mw), (BR, fill)
            assert close(l, lw), (BR, fill)


@pytest.mark.parametrize("path", [0, tm.TM_PATH_SCALAR, tm.TM_PATH_VEC])
def test_softmax_stats_paths(cuda, oracle, path):
    M, N = 130, 1000
    s = synth.uniform((M, N), -30.0, -1.0, 19)
    mw, lw = oracle.softmax_rowstats(s, N, M, N, 64)
    m, l = stats(s, N, M, N, 4, 64, flags=path)
    assert np.array_equal(m, mw) and close(l, lw)


def test_softmax_stats_aligned_and_misaligned(cuda, oracle):
    M, N = 256, 1024
    s = synth.normal((M, N), 23)
    mw, lw = oracle.softmax_rowstats(s, N, M, N, 64)
    m, l = stats(s, N, M, N, 8, 64, flags=tm.TM_ALIGNED)
    assert np.array_equal(m, mw) and close(l, lw)
    m, l = stats(s, N, M, N, 8, 64, lead=1)        # 4-byte aligned base: scalar path
    assert np.array_equal(m, mw) and close(l, lw)
    with pytest.raises(tm.TmError) as e:
        stats(s[:, :1000].copy(), 1000, M, 1000, 8, 64, flags=tm.TM_ALIGNED)
    assert e.value.status == tm.TM_ERR_BROKEN_PROMISE


def test_softmax_stats_special_rows(cuda, oracle):
    s = synth.uniform((6, 70), -5.0, -1.0, 14)
    s[0, :] = -np.inf                   # nothing but -inf: m = -inf, l = 0
    s[1, :] = -np.inf
    s[1, 17] = -2.0                     # one finite score: l = 1 exactly
    s[2, :] = -7.5                      # constant row: l = N exactly
    mw, lw = oracle.softmax_rowstats(s, 70, 6, 70, 64)
    m, l = stats(s, 70, 6, 70, 2, 64)
    assert same_f32(m, mw) and close(l, lw)
    assert m[0] == -np.inf and l[0] == 0.0 and l[1] == 1.0 and l[2] == 70.0


def test_softmax_stats_empty_rows(cuda):
    m, l = stats(np.zeros(12, np.float32), 4, 3, 0)
    assert np.all(m == -np.inf) and np.all(l == 0.0)
