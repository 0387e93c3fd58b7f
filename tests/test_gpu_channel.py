"""GPU parity of tm_channel_affine (per-channel scale and bias) against the CPU
oracle, bit for bit ("Memory Coalescing and Tensor Layout", "NCHW versus NHWC":
the [B, C, H, W] tensor read as [B*H*W, C] with channels last, or as
[B*C, H*W] with channels first)."""
import numpy as np
import pytest

from gpu_util import CANARY, DevBuf, same_f32
from masking_tm_affine_gb300 import synth, tm

pytestmark = pytest.mark.gpu
TILES = [(8, 8), (16, 16), (32, 32), (64, 64), (32, 128), (128, 128)]


def run(x, R, K, ldx, ldy, sc, bi, C, layout, TM=32, TN=128, flags=0, lead_p=0, in_place=False):
    X = synth.pad_rows(x, ldx)
    XD = DevBuf(X)
    YD = XD if in_place else DevBuf(np.full(R * ldy, CANARY, dtype=np.uint32))
    SD = None if sc is None else DevBuf(sc, lead_p)
    BD = None if bi is None else DevBuf(bi, lead_p)
    tm.tm_channel_affine(XD.ptr, ldx, R, K, None if SD is None else SD.ptr, None if BD is None else BD.ptr,
                         C, layout, YD.ptr, ldy, TM, TN, flags)
    tm.tm_check()
    assert YD.guards_intact()
    want = X.copy() if in_place else np.full(R * ldy, CANARY, dtype=np.uint32).view(np.float32)
    return YD.payload_f32(), want, X


def check(oracle, x, R, K, ldx, ldy, sc, bi, C, layout, **kw):
    got, want, X = run(x, R, K, ldx, ldy, sc, bi, C, layout, **kw)
    oracle.channel_affine(X, ldx, R, K, sc, bi, C, layout, want, ldy)
    assert same_f32(got, want)


@pytest.mark.parametrize("layout", [tm.TM_CHANNELS_LAST, tm.TM_CHANNELS_FIRST])
def test_activation_shaped_tensor(cuda, oracle, layout):
    B, C, H, W = 4, 64, 28, 28
    sc = synth.uniform((C,), 0.5, 2.0, 41)
    bi = synth.normal((C,), 42)
    if layout == tm.TM_CHANNELS_LAST:
        R, K = B * H * W, C
    else:
        R, K = B * C, H * W
    x = synth.normal((R, K), 43)
    check(oracle, x, R, K, K, K, sc, bi, C, layout)
    if R % 32 == 0 and K % 128 == 0:
        check(oracle, x, R, K, K, K, sc, bi, C, layout, flags=tm.TM_ALIGNED)


@pytest.mark.parametrize("TM,TN", TILES)
@pytest.mark.parametrize("layout", [tm.TM_CHANNELS_LAST, tm.TM_CHANNELS_FIRST])
@pytest.mark.parametrize("R,K,ldx,ldy", [(1, 4, 4, 4), (37, 20, 24, 28), (130, 68, 68, 72), (33, 129, 131, 133)])
def test_tiles_shapes_layouts(cuda, oracle, TM, TN, layout, R, K, ldx, ldy):
    C = K if layout == tm.TM_CHANNELS_LAST else 7
    sc = synth.uniform((C,), -2.0, 2.0, R + K)
    bi = synth.normal((C,), R * K)
    x = synth.normal((R, K), R + 3 * K)
    check(oracle, x, R, K, ldx, ldy, sc, bi, C, layout, TM=TM, TN=TN)


@pytest.mark.parametrize("which", ["bias", "scale", "neither"])
def test_missing_vectors(cuda, oracle, which):
    R, K = 96, 256
    sc = None if which in ("bias", "neither") else synth.uniform((K,), 0.5, 2.0, 44)
    bi = None if which in ("scale", "neither") else synth.normal((K,), 45)
    x = synth.normal((R, K), 46)
    check(oracle, x, R, K, K, K, sc, bi, K, tm.TM_CHANNELS_LAST)
    check(oracle, x, R, K, K, K, sc, bi, K, tm.TM_CHANNELS_LAST, flags=tm.TM_ALIGNED)


def test_unaligned_parameters_and_paths(cuda, oracle):
    R, K = 128, 256
    sc = synth.uniform((K,), 0.5, 2.0, 47)
    bi = synth.normal((K,), 48)
    x = synth.normal((R, K), 49)
    check(oracle, x, R, K, K, K, sc, bi, K, tm.TM_CHANNELS_LAST, lead_p=1)     # 4-byte aligned vectors
    for flags in (tm.TM_PATH_SCALAR, tm.TM_PATH_VEC, tm.TM_ALIGNED | tm.TM_PATH_SCALAR):
        check(oracle, x, R, K, K, K, sc, bi, K, tm.TM_CHANNELS_LAST, flags=flags)
    with pytest.raises(tm.TmError) as e:
        run(x, R, K, K, K, sc, bi, K, tm.TM_CHANNELS_LAST, flags=tm.TM_PATH_VEC, lead_p=1)
    assert e.value.status == tm.TM_ERR_MISALIGNED


def test_in_place(cuda, oracle):
    R, K = 64, 384
    sc = synth.uniform((K,), 0.5, 2.0, 50)
    bi = synth.normal((K,), 51)
    x = synth.normal((R, K), 52)
    check(oracle, x, R, K, K, K, sc, bi, K, tm.TM_CHANNELS_LAST, in_place=True)


def test_errors(cuda):
    x = np.zeros(64, np.float32)
    XD, YD, P = DevBuf(x), DevBuf(x), DevBuf(np.ones(8, np.float32))
    for args, code in [((8, 8, P.ptr, P.ptr, 4, tm.TM_CHANNELS_LAST), tm.TM_ERR_INVALID_ARG),    # K > C
                       ((8, 8, P.ptr, P.ptr, 0, tm.TM_CHANNELS_FIRST), tm.TM_ERR_INVALID_ARG),   # C = 0
                       ((8, 8, P.ptr, P.ptr, 8, 5), tm.TM_ERR_INVALID_ARG),                      # layout
                       ((8, 8, P.ptr, YD.ptr, 8, tm.TM_CHANNELS_LAST), tm.TM_ERR_INVALID_ARG)]:  # bias overlaps Y
        R, K, s, b, C, layout = args
        with pytest.raises(tm.TmError) as e:
            tm.tm_channel_affine(XD.ptr, K, R, K, s, b, C, layout, YD.ptr, K, 8, 8)
        assert e.value.status == code
    assert np.all(YD.payload_u32() == 0)


@pytest.mark.parametrize("name", ["channel_nhwc", "channel_nchw"])
def test_full_size_workloads(cuda, oracle, name):
    # [32, 256, 56, 56] fp32 in each view, the case bench.py times (32 x 128 tiles)
    w = synth.WORKLOADS[name]
    x = synth.workload_input(name)
    sc, bi = synth.channel_params(w["C"])
    check(oracle, x, w["M"], w["N"], w["N"], w["N"], sc, bi, w["C"], w["layout"], TM=w["TM"], TN=w["TN"])
