"""GPU parity of tm_scale2d / tm_copy2d against the CPU oracle.

"@aligned" ("A minimal kernel") and "Slicing, bounds and masking"
("Masking", "Promising whole tiles with @aligned"): in-bounds results
bit-exact; every word outside [M, N] (ld gaps, past the last row, the 4 KB
canary past each tensor) untouched; a broken promise stores nothing.
"""
import numpy as np
import pytest

from gpu_util import CANARY, DevBuf, same_f32
from masking_tm_affine_gb300 import synth, tm

pytestmark = pytest.mark.gpu

TILES = [(8, 8), (16, 16), (32, 32), (64, 64), (32, 128), (128, 128)]
OPS = ["scale", "copy"]


def run(op, x, M, N, ldx, ldy, TM, TN, flags=0, alpha=1.5, lead_x=0, lead_y=0, out_fill=CANARY):
    X = synth.pad_rows(x, ldx) if M and N else np.full(max(M * ldx, 0), synth.POISON_F32, np.float32)
    XD = DevBuf(X, lead_x)
    YD = DevBuf(np.full(M * ldy, out_fill, dtype=np.uint32), lead_y)
    if op == "scale":
        tm.tm_scale2d(XD.ptr, ldx, YD.ptr, ldy, M, N, alpha, TM, TN, flags)
    else:
        tm.tm_copy2d(XD.ptr, ldx, YD.ptr, ldy, M, N, TM, TN, flags)
    tm.tm_check()
    assert XD.guards_intact() and np.array_equal(XD.payload_u32(), X.view(np.uint32))
    assert YD.guards_intact(), "canary past the output changed"
    return X, YD.payload_u32()


def expect(oracle, op, X, M, N, ldx, ldy, alpha=1.5, out_fill=CANARY):
    want = np.full(M * ldy, out_fill, dtype=np.uint32)
    if op == "scale":
        w = want.view(np.float32)
        oracle.scale2d(X, ldx, w, ldy, M, N, alpha)
    else:
        oracle.copy2d(X, ldx, want, ldy, M, N)
    return want


def check(oracle, op, x, M, N, ldx, ldy, TM, TN, flags=0, **kw):
    X, got = run(op, x, M, N, ldx, ldy, TM, TN, flags, **kw)
    want = expect(oracle, op, X, M, N, ldx, ldy)
    if op == "copy":
        assert np.array_equal(got, want)
    else:
        assert same_f32(got.view(np.float32), want.view(np.float32))


def test_scale_8192_aligned_workload(cuda, oracle):
    # [8192, 8192], N(0,1) seed 1, alpha 1.5, TM = 32, TN = 128, promise kept: the fast path
    x = synth.workload_input("scale_8192")
    X, got = run("scale", x, 8192, 8192, 8192, 8192, 32, 128, tm.TM_ALIGNED)
    want = expect(oracle, "scale", X, 8192, 8192, 8192, 8192)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("op", OPS)
def test_ragged_4100x1000_workload(cuda, oracle, op):
    # [4100, 1000], U[-8,8) seed 2, 64 x 64 tiles, no promise: 960 whole tiles,
    # 64 + 15 edge tiles and a 4 x 40 corner; canaries past both tensors
    x = synth.workload_input("ragged_4100")
    check(oracle, op, x, 4100, 1000, 1000, 1000, 64, 64)


@pytest.mark.parametrize("op", OPS)
def test_ragged_4100x1000_with_gaps(cuda, oracle, op):
    # ld = 1024: 3e38 poison in the input gaps, canaries in the output gaps
    x = synth.workload_input("ragged_4100")
    check(oracle, op, x, 4100, 1000, 1024, 1024, 64, 64)


@pytest.mark.parametrize("TM,TN", TILES)
@pytest.mark.parametrize("op", OPS)
@pytest.mark.parametrize("M,N,ldx,ldy", [(1, 1, 1, 1), (7, 5, 9, 6), (20, 28, 28, 32), (33, 65, 68, 72),
                                         (130, 260, 260, 264), (257, 129, 131, 133), (64, 256, 256, 256)])
def test_tiles_shapes_ragged(cuda, oracle, TM, TN, op, M, N, ldx, ldy):
    x = synth.uniform((M, N), -8.0, 8.0, M * 1000 + N)
    check(oracle, op, x, M, N, ldx, ldy, TM, TN)


@pytest.mark.parametrize("path", [tm.TM_PATH_SCALAR, tm.TM_PATH_VEC])
@pytest.mark.parametrize("TM,TN", TILES)
def test_forced_paths(cuda, oracle, path, TM, TN):
    M, N = 150, 300
    x = synth.normal((M, N), 8)
    check(oracle, "scale", x, M, N, 304, 300, TM, TN, path)
    check(oracle, "copy", x, M, N, 300, 308, TM, TN, path)


@pytest.mark.parametrize("TM,TN", TILES)
@pytest.mark.parametrize("op", OPS)
def test_aligned_promise_kept(cuda, oracle, TM, TN, op):
    M, N = TM * 5, TN * 3
    x = synth.normal((M, N), 4)
    check(oracle, op, x, M, N, N, N + 4, TM, TN, tm.TM_ALIGNED)                 # 16-byte rows
    check(oracle, op, x, M, N, N + 8, N + 8, TM, TN, tm.TM_ALIGNED)             # 32-byte rows
    check(oracle, op, x, M, N, N, N, TM, TN, tm.TM_ALIGNED, lead_x=4, lead_y=4)  # 16- but not 32-byte bases
    check(oracle, op, x, M, N, N, N, TM, TN, tm.TM_ALIGNED | tm.TM_PATH_SCALAR)


def test_misaligned_inputs_take_scalar_path(cuda, oracle):
    M, N = 70, 90
    x = synth.normal((M, N), 6)
    check(oracle, "scale", x, M, N, 91, 93, 32, 32, lead_x=1, lead_y=3)
    check(oracle, "copy", x, M, N, 90, 90, 64, 64, lead_x=2, lead_y=1)


def test_masking_census_figure_case(cuda):
    # "Slicing, bounds and masking", "Masking": with 8 x 8 tiles over [20, 28],
    # block (2, 3) has 16 of 64 elements in bounds; count the stores it makes
    M, N, ld = 20, 28, 32
    x = np.ones((M, N), np.float32)
    _, got = run("copy", x, M, N, N, ld, 8, 8)
    g = got.reshape(M, ld)
    block = np.zeros((8, 8), dtype=bool)
    sub = g[16:24, 24:32]
    block[:sub.shape[0], :sub.shape[1]] = sub != CANARY
    assert block.sum() == 16
    assert np.count_nonzero(g != CANARY) == M * N


def test_copy_preserves_nan_payloads(cuda):
    M, N = 33, 40
    g = synth.rng(3)
    raw = g.integers(0, 2**32, size=M * N, dtype=np.uint64).astype(np.uint32)
    raw[:6] = [0x7FA00001, 0xFFC12345, 0x7F800001, 0x80000000, 0x00000001, 0xFF800000]
    for flags in (0, tm.TM_PATH_SCALAR):
        _, got = run("copy", raw.view(np.float32).reshape(M, N), M, N, N, N, 32, 32, flags)
        assert np.array_equal(got, raw)


def test_scale_in_place(cuda, oracle):
    M, N, ld = 100, 200, 204
    x = synth.normal((M, N), 12)
    X = synth.pad_rows(x, ld)
    D = DevBuf(X)
    tm.tm_scale2d(D.ptr, ld, D.ptr, ld, M, N, 1.5, 32, 128)
    tm.tm_check()
    want = X.copy()
    oracle.scale2d(X, ld, want, ld, M, N, 1.5)
    assert D.guards_intact() and same_f32(D.payload_f32(), want)


def test_broken_promise_host_check_stores_nothing(cuda):
    x = synth.normal((64, 100), 1)
    XD = DevBuf(synth.pad_rows(x, 100))
    YD = DevBuf.empty(64 * 100)
    with pytest.raises(tm.TmError) as e:
        tm.tm_scale2d(XD.ptr, 100, YD.ptr, 100, 64, 100, 1.5, 32, 128, tm.TM_ALIGNED)
    assert e.value.status == tm.TM_ERR_BROKEN_PROMISE
    tm.tm_check()
    assert np.all(YD.words() == CANARY)


@pytest.mark.parametrize("M,N", [(64, 100), (60, 128), (33, 129)])
def test_broken_promise_device_entry_check(cuda, M, N):
    # the kernel itself refuses: no block stores anything, tm_check reports it
    x = synth.normal((M, N), 2)
    XD = DevBuf(synth.pad_rows(x, N + (-N) % 4))
    YD = DevBuf.empty(M * (N + (-N) % 4))
    tm.tm_scale2d_unchecked(XD.ptr, N + (-N) % 4, YD.ptr, N + (-N) % 4, M, N, 1.5, 32, 128)
    with pytest.raises(tm.TmError) as e:
        tm.tm_check()
    assert e.value.status == tm.TM_ERR_BROKEN_PROMISE
    assert np.all(YD.words() == CANARY)
    tm.tm_check()  # the status word was cleared


def test_misaligned_device_entry_check(cuda):
    M, N = 64, 128
    XD = DevBuf(synth.normal((M * N,), 5), lead=1)   # 4-byte aligned base
    YD = DevBuf.empty(M * N)
    tm.tm_scale2d_unchecked(XD.ptr, N, YD.ptr, N, M, N, 1.5, 32, 128)
    with pytest.raises(tm.TmError) as e:
        tm.tm_check()
    assert e.value.status == tm.TM_ERR_MISALIGNED
    assert np.all(YD.words() == CANARY)


def test_unchecked_with_kept_promise_runs(cuda, oracle):
    M, N = 96, 256
    x = synth.normal((M, N), 7)
    XD = DevBuf(x)
    YD = DevBuf.empty(M * N)
    tm.tm_scale2d_unchecked(XD.ptr, N, YD.ptr, N, M, N, 1.5, 32, 128)
    tm.tm_check()
    want = np.zeros(M * N, np.float32)
    oracle.scale2d(x, N, want, N, M, N, 1.5)
    assert same_f32(YD.payload_f32(), want)


def test_empty_shapes_do_nothing(cuda):
    YD = DevBuf.empty(64)
    XD = DevBuf(np.zeros(64, np.float32))
    tm.tm_scale2d(XD.ptr, 8, YD.ptr, 8, 0, 8, 1.5, 8, 8)
    tm.tm_copy2d(XD.ptr, 8, YD.ptr, 8, 8, 0, 8, 8)
    tm.tm_check()
    assert np.all(YD.words() == CANARY)
