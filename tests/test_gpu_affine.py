"""GPU parity of tm_affine (out = a*2 + 1) against the CPU oracle.

"Aligned Load & Store": the three kernels compute the same map and all print
"passed"; here every variant must equal the oracle bit for bit, write every
element (including the n % 4 tail), and leave the 4 KB canary past `out` intact.
"""
import numpy as np
import pytest

from gpu_util import DevBuf, same_f32
from masking_tm_affine_gb300 import synth, tm

pytestmark = pytest.mark.gpu

VARIANTS = [tm.TM_VAR_AUTO, tm.TM_VAR_SCALAR, tm.TM_VAR_VEC_UNALIGNED, tm.TM_VAR_VEC4, tm.TM_VAR_VEC8]


def run(a, variant, lead_a=0, lead_o=0):
    A = DevBuf(a, lead_a)
    O = DevBuf.empty(a.size, lead_o)
    tm.tm_affine(A.ptr, O.ptr, a.size, variant)
    tm.tm_check()
    assert A.guards_intact() and O.guards_intact()
    assert np.array_equal(A.payload_u32(), a.view(np.uint32)), "input modified"
    return O.payload_f32()


@pytest.mark.parametrize("variant", VARIANTS)
def test_affine_1m_workload_bit_exact(cuda, oracle, variant):
    a = synth.workload_input("affine_1m")           # n = 2^20, U[-1, 1), seed 0
    got = run(a, variant)
    assert same_f32(got, oracle.affine(a))


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 9, 31, 33, 255, 257, 1023, 1024, 1025, 4095, 4097,
                               2047 * 8 + 5, 65536 + 3, 300007])
@pytest.mark.parametrize("variant", VARIANTS)
def test_affine_ragged_lengths(cuda, oracle, n, variant):
    a = synth.uniform((n,), -4.0, 4.0, n)
    assert same_f32(run(a, variant), oracle.affine(a))


@pytest.mark.parametrize("lead_a,lead_o", [(1, 1), (2, 2), (3, 3), (5, 5), (1, 2), (0, 3), (4, 4), (6, 6)])
def test_affine_auto_misaligned_pointers(cuda, oracle, lead_a, lead_o):
    # AUTO peels a scalar prologue when both pointers share their misalignment,
    # else runs the scalar kernel; either way the result is the oracle's
    a = synth.uniform((50021,), -1.0, 1.0, 17)
    assert same_f32(run(a, tm.TM_VAR_AUTO, lead_a, lead_o), oracle.affine(a))


@pytest.mark.parametrize("variant", [tm.TM_VAR_SCALAR, tm.TM_VAR_VEC_UNALIGNED])
def test_affine_scalar_variants_any_alignment(cuda, oracle, variant):
    a = synth.uniform((1001,), -1.0, 1.0, 5)
    assert same_f32(run(a, variant, 3, 1), oracle.affine(a))


def test_affine_special_values(cuda, oracle):
    fmax = np.finfo(np.float32).max
    a = np.array([0.0, -0.0, 1e-45, -1e-45, 1e-38, fmax, -fmax, fmax / 2, np.inf, -np.inf, np.nan,
                  8388608.0, 8388609.0, -0.5, 0.5, 3.0] * 5, dtype=np.float32)
    want = oracle.affine(a)
    for v in VARIANTS:
        assert same_f32(run(a, v), want), v


def test_affine_in_place(cuda, oracle):
    a = synth.uniform((100003,), -1.0, 1.0, 9)
    A = DevBuf(a)
    tm.tm_affine(A.ptr, A.ptr, a.size, tm.TM_VAR_AUTO)
    tm.tm_check()
    assert A.guards_intact()
    assert same_f32(A.payload_f32(), oracle.affine(a))


def test_affine_variants_agree(cuda):
    a = synth.normal((123457,), 3)
    outs = [run(a, v) for v in VARIANTS]
    for o in outs[1:]:
        assert np.array_equal(o.view(np.uint32), outs[0].view(np.uint32))


def test_affine_errors(cuda):
    A = DevBuf(np.zeros(64, np.float32), 1)   # 4-byte aligned only
    O = DevBuf.empty(64)
    with pytest.raises(tm.TmError) as e:
        tm.tm_affine(A.ptr, O.ptr, 63, tm.TM_VAR_VEC4)
    assert e.value.status == tm.TM_ERR_MISALIGNED
    with pytest.raises(tm.TmError) as e:
        tm.tm_affine(O.ptr, O.ptr + 8, 16, tm.TM_VAR_AUTO)
    assert e.value.status == tm.TM_ERR_INVALID_ARG
    assert O.guards_intact() and np.all(O.payload_u32() == 0xDEADBEEF)
    tm.tm_affine(A.ptr, O.ptr, 0)                 # empty is fine
    tm.tm_check()
