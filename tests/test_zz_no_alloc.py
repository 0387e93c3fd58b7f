"""tm_colsum_noalloc: the column sum for callers that cannot allocate device
memory -- code hosted inside a framework whose allocator owns every device
byte, loops under a fixed memory budget that must not fail halfway, and paths
where cudaMalloc's device-wide synchronization is not allowed.  Its scratch
(the partial sums of its first pass) lives in the library's own static device
array.

Each call goes through the C ABI and is checked against the fp64 oracle and
against tm_colsum with a caller workspace, within the 1e-5 relative tolerance
of the other column-sum tests.  Calls come in pairs in a row on one stream:
the first, on the [8192, 8192] matrix, fills half of the array with its
partials, so a second call that read a partial it had not written first
would come out wrong.
This file is collected last so that a failure here never hides another
test's result; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

from gpu_util import DevBuf
from masking_tm_affine_gb300 import synth, tm

REL = 1e-5  # the tolerance of tests/test_gpu_sums.py

VARIANTS = [tm.TM_VAR_AUTO, tm.TM_VAR_REGDIRECT, tm.TM_VAR_STAGED, tm.TM_VAR_CLUSTER, tm.TM_VAR_NAIVE]

# (M, N, ld, TM, TN): the first fills half the scratch with partials (AUTO runs
# REGDIRECT there: 64 strips are too many for the cluster form), the second is
# ragged with 3e38 poison in its ld gap
BIG = (8192, 8192, 8192, 32, 128)
SMALL = (1500, 1001, 1004, 16, 64)


@pytest.fixture(scope="module")
def inputs():
    big = synth.normal((BIG[0], BIG[1]), 31)
    small = synth.normal((SMALL[0], SMALL[1]), 32)
    return [(big, synth.pad_rows(big, BIG[2])), (small, synth.pad_rows(small, SMALL[2]))]


def within(got, x, want):
    scale = np.abs(x.astype(np.float64)).sum(axis=0)
    return bool(np.all(np.abs(got.astype(np.float64) - want) <= REL * scale))


def with_workspace(XD, ld, M, N, TM, TN, variant):
    C = DevBuf.empty(N)
    ws = tm.tm_colsum_workspace_bytes(M, N, TM, TN, variant)
    W = DevBuf.empty(max(ws // 4, 4))
    rc = tm.load().tm_colsum(XD.ptr, ld, M, N, C.ptr, W.ptr, max(ws, 16), TM, TN, variant, 0, None)
    assert rc == tm.TM_OK, tm.status_string(rc)
    assert tm.load().tm_check(None) == tm.TM_OK
    return C.payload_f32()


@pytest.mark.gpu
@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("second_flags", [0, tm.TM_PDL])
def test_noalloc_two_calls_in_a_row(cuda, oracle, inputs, variant, second_flags):
    XDs = [DevBuf(X) for _, X in inputs]
    Cs = [DevBuf.empty(BIG[1]), DevBuf.empty(SMALL[1])]
    for k, ((M, N, ld, TM, TN), flags) in enumerate(zip((BIG, SMALL), (0, second_flags))):
        assert tm.tm_colsum_workspace_bytes(M, N, TM, TN, variant) <= tm.TM_NOALLOC_SCRATCH_BYTES
        # no synchronization between the two: stream order alone keeps them apart
        rc = tm.load().tm_colsum_noalloc(XDs[k].ptr, ld, M, N, Cs[k].ptr, TM, TN, variant, flags, None)
        assert rc == tm.TM_OK, tm.status_string(rc)
    assert tm.load().tm_check(None) == tm.TM_OK
    for k, ((x, X), (M, N, ld, TM, TN)) in enumerate(zip(inputs, (BIG, SMALL))):
        got = Cs[k].payload_f32()
        assert Cs[k].guards_intact() and XDs[k].guards_intact(), (variant, k)
        assert within(got, x, oracle.colsum(X, ld, M, N)), (variant, k)
        assert within(got, x, with_workspace(XDs[k], ld, M, N, TM, TN, variant).astype(np.float64)), (variant, k)


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_its_scratch(cuda, oracle):
    # [192, 768000] at 8 x 256 tiles: 3000 strips of 3 chunks, a 1 KB partial
    # each, 9000 KB -- beyond the array, so rejected before anything runs,
    # output untouched ...
    M, N, TM, TN = 192, 768000, 8, 256
    x = synth.uniform((M, N), 0.0, 1.0, 33)
    XD = DevBuf(x)
    for variant in (tm.TM_VAR_AUTO, tm.TM_VAR_REGDIRECT):
        assert tm.tm_colsum_workspace_bytes(M, N, TM, TN, variant) > tm.TM_NOALLOC_SCRATCH_BYTES
        C = DevBuf.empty(N)
        rc = tm.load().tm_colsum_noalloc(XD.ptr, N, M, N, C.ptr, TM, TN, variant, 0, None)
        assert rc == tm.TM_ERR_WORKSPACE, variant
        assert tm.load().tm_check(None) == tm.TM_OK
        assert np.all(C.words() == 0xDEADBEEF)
    # ... except by CLUSTER and STAGED, which add their partials on chip and
    # need none
    for variant in (tm.TM_VAR_CLUSTER, tm.TM_VAR_STAGED):
        assert tm.tm_colsum_workspace_bytes(M, N, TM, TN, variant) == 0
        C = DevBuf.empty(N)
        rc = tm.load().tm_colsum_noalloc(XD.ptr, N, M, N, C.ptr, TM, TN, variant, 0, None)
        assert rc == tm.TM_OK, tm.status_string(rc)
        assert tm.load().tm_check(None) == tm.TM_OK
        assert C.guards_intact()
        assert within(C.payload_f32(), x, oracle.colsum(x, N, M, N)), variant
