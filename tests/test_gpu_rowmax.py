"""GPU parity of tm_rowmax_masked against the CPU oracle (bit-exact).

"Slicing, bounds and masking", "Reductions over a ragged tile": with the
where/iota fill the ragged row-max of all-negative scores is never 0; without
it (the zero-fill foil) the padding wins and the result is exactly 0.
"""
import numpy as np
import pytest

from gpu_util import DevBuf, same_f32
from masking_tm_affine_gb300 import synth, tm

pytestmark = pytest.mark.gpu


def rowmax(S, ld, M, N, BR=8, BC=64, fill=tm.TM_FILL_NEG_INF, flags=0, lead=0):
    SD = DevBuf(S, lead)
    MD = DevBuf.empty(M)
    tm.tm_rowmax_masked(SD.ptr, ld, M, N, MD.ptr, BR, BC, fill, flags)
    tm.tm_check()
    assert MD.guards_intact() and SD.guards_intact()
    return MD.payload_f32()


def test_rowmax_8192x1000_workload(cuda, oracle):
    s = synth.workload_input("rowmax_8192")     # U[-30,-1) seed 4; BC = 64: 15 whole tiles + 1 of 40
    assert s.max() < 0
    want = oracle.rowmax_masked(s, 1000, 8192, 1000, 64, oracle.FILL_NEG_INF)
    got = rowmax(s, 1000, 8192, 1000)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert np.all(got < 0) and not np.any(got == 0)
    foil = rowmax(s, 1000, 8192, 1000, fill=tm.TM_FILL_ZERO)
    assert np.all(foil.view(np.uint32) == 0)   # exactly +0.0: the pitfall
    assert np.array_equal(foil, oracle.rowmax_masked(s, 1000, 8192, 1000, 64, oracle.FILL_ZERO))


@pytest.mark.parametrize("BC", [16, 32, 64, 128, 256, 512])
@pytest.mark.parametrize("N", [0, 1, 4, 15, 40, 63, 64, 65, 100, 128, 999, 1000, 1024])
def test_rowmax_tiles_and_extents(cuda, oracle, BC, N):
    M = 67
    ld = N + 5
    s = (synth.normal((M, max(N, 1)), N + BC)[:, :N] * np.float32(10.0)) - np.float32(3.0)
    S = synth.pad_rows(s, ld)                  # +3e38 poison in the gaps: a gap read would win the max
    for fill in (oracle.FILL_NEG_INF, oracle.FILL_ZERO):
        want = oracle.rowmax_masked(S, ld, M, N, BC, fill)
        for BR in (1, 8, 32):
            got = rowmax(S, ld, M, N, BR, BC, fill)
            assert same_f32(got, want), (BR, fill)


@pytest.mark.parametrize("path", [0, tm.TM_PATH_SCALAR, tm.TM_PATH_VEC])
def test_rowmax_paths(cuda, oracle, path):
    M, N = 130, 1000
    s = synth.uniform((M, N), -30.0, -1.0, 9)
    want = oracle.rowmax_masked(s, N, M, N, 64)
    assert np.array_equal(rowmax(s, N, M, N, 4, 64, flags=path), want)


def test_rowmax_scalar_for_odd_extents(cuda, oracle):
    M, N, ld = 50, 1001, 1003
    s = synth.uniform((M, N), -30.0, -1.0, 10)
    S = synth.pad_rows(s, ld)
    want = oracle.rowmax_masked(S, ld, M, N, 64)
    assert np.array_equal(rowmax(S, ld, M, N, 8, 64), want)
    assert np.array_equal(rowmax(S, ld, M, N, 8, 64, lead=1), want)


def test_rowmax_aligned_promise(cuda, oracle):
    M, N = 256, 1024
    s = synth.uniform((M, N), -30.0, -1.0, 13)
    want = oracle.rowmax_masked(s, N, M, N, 64)
    assert np.array_equal(rowmax(s, N, M, N, 8, 64, flags=tm.TM_ALIGNED), want)
    with pytest.raises(tm.TmError) as e:
        rowmax(s[:, :1000].copy(), 1000, M, 1000, 8, 64, flags=tm.TM_ALIGNED)
    assert e.value.status == tm.TM_ERR_BROKEN_PROMISE


def test_rowmax_values_below_page_fill(cuda, oracle):
    s = np.full((3, 40), -3.0e38, dtype=np.float32)
    s[:, 7] = -2.0e38
    got = rowmax(s, 40, 3, 40, 1, 64)
    assert np.all(got == np.float32(-2.0e38))


def test_rowmax_nan_and_inf(cuda, oracle):
    s = synth.uniform((8, 70), -5.0, -1.0, 14)
    s[0, 3] = np.nan
    s[1, :] = np.nan
    s[2, 69] = np.inf
    s[3, :] = -np.inf
    want = oracle.rowmax_masked(s, 70, 8, 70, 64)
    got = rowmax(s, 70, 8, 70, 8, 64)
    assert same_f32(got, want)


def test_rowmax_empty_rows_give_neg_inf(cuda):
    got = rowmax(np.zeros(12, np.float32), 4, 3, 0)
    assert np.all(got == -np.inf)
