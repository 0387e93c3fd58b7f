"""tm_colsum_noalloc: the column sum for callers that cannot allocate device
memory (framework-hosted code whose allocator owns the device, fixed memory
budgets, paths where cudaMalloc's device-wide synchronization is not
allowed).  Its partial sums live in the library's own static device array.

Checked through the C ABI against tm_colsum with a caller workspace, on two
calls in a row (the second sees the first call's leftovers in the shared
array), within the tolerance of the other column-sum tests.  This file is
collected last so that a failure here never hides another test's result; it
also passes on its own in a fresh process.
"""
import numpy as np
import pytest

from gpu_util import DevBuf
from masking_tm_affine_gb300 import synth, tm

REL = 1e-5  # the tolerance of tests/test_gpu_sums.py


def with_workspace(XD, ld, M, N, TM, TN, variant):
    C = DevBuf.empty(N)
    ws = tm.tm_colsum_workspace_bytes(M, N, TM, TN, variant if variant == tm.TM_VAR_NAIVE else tm.TM_VAR_AUTO)
    W = DevBuf.empty(max(ws // 4, 1))
    rc = tm.load().tm_colsum(XD.ptr, ld, M, N, C.ptr, W.ptr, ws, TM, TN, variant, 0, None)
    assert rc == tm.TM_OK, tm.status_string(rc)
    assert tm.load().tm_check(None) == tm.TM_OK
    return C


def without_workspace(XD, ld, M, N, TM, TN, variant):
    C = DevBuf.empty(N)
    rc = tm.load().tm_colsum_noalloc(XD.ptr, ld, M, N, C.ptr, TM, TN, variant, 0, None)
    assert rc == tm.TM_OK, tm.status_string(rc)
    assert tm.load().tm_check(None) == tm.TM_OK
    assert C.guards_intact()
    return C


@pytest.mark.gpu
@pytest.mark.parametrize("variant", [tm.TM_VAR_AUTO, tm.TM_VAR_REGDIRECT, tm.TM_VAR_NAIVE])
def test_noalloc_matches_workspace_entry_two_calls(cuda, variant):
    # call 1: the [4096, 4096] coalescing workload; call 2: a ragged
    # [1500, 1001] matrix, whose sums must not pick up call 1's leftovers
    cases = [(synth.workload_input("coalesce_4096"), 4096, 4096, 4096, 32, 128),
             (synth.normal((1500, 1001), 21), 1500, 1001, 1001, 16, 64)]
    for x, M, N, ld, TM, TN in cases:
        XD = DevBuf(x)
        ref = with_workspace(XD, ld, M, N, TM, TN, variant).payload_f32().astype(np.float64)
        got = without_workspace(XD, ld, M, N, TM, TN, variant).payload_f32().astype(np.float64)
        scale = np.abs(x.astype(np.float64)).sum(axis=0)
        assert np.all(np.abs(got - ref) <= REL * scale), (variant, M, N)


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_its_scratch(cuda):
    # one partial row of 2^21 columns is 8 MiB > the 4 MiB array: rejected
    # before anything runs, output untouched
    M, N = 8, 1 << 21
    assert tm.tm_colsum_workspace_bytes(M, N, 8, 64) > tm.TM_NOALLOC_SCRATCH_BYTES
    XD = DevBuf(np.ones(M * N, np.float32))
    C = DevBuf.empty(N)
    rc = tm.load().tm_colsum_noalloc(XD.ptr, N, M, N, C.ptr, 8, 64, tm.TM_VAR_AUTO, 0, None)
    assert rc == tm.TM_ERR_WORKSPACE
    assert tm.load().tm_check(None) == tm.TM_OK
    assert np.all(C.words() == 0xDEADBEEF)
