"""The device-side tile-walk planner every kernel uses, read back through
tm_tile_walk_probe, against the page's worked example and the closed form
("Slicing, bounds and masking", "Loops over a dynamic extent"); and the
streaming-read probe the reductions' floor is measured with, against the
oracle's sums of the same blocks."""
import numpy as np
import pytest
import torch

from conftest import read_golden
from gpu_util import DevBuf
from masking_tm_affine_gb300 import synth, tm

pytestmark = pytest.mark.gpu


def probe(K, T):
    out = torch.zeros(4, dtype=torch.int64, device="cuda")
    tm.tm_tile_walk_probe(K, T, out)
    tm.tm_check()
    return [int(v) for v in out.cpu()]


def test_probe_printed_example(cuda):
    (row,) = read_golden("tile_walk.txt")
    K, T, whole, masked, rem = map(int, row)
    assert probe(K, T) == [whole, masked, rem, whole + masked]


def test_probe_closed_form_sweep(cuda):
    for K in list(range(0, 70)) + [1000, 4096, 4100, 2**31 + 5, 2**40 + 3]:
        for T in [1, 3, 16, 40, 64, 128, 512]:
            w = probe(K, T)
            assert w == [K // T, 1 if K % T else 0, K % T, -(-K // T)], (K, T)


def test_check_clean(cuda):
    tm.tm_check()
    assert np.isfinite(1.0)


def test_bounded_wait_times_out_and_context_survives(cuda):
    # a wait on a barrier nothing arrives at gives up after ~1 s and reports
    # TM_ERR_TIMEOUT through tm_check; the context keeps working afterwards
    tm.tm_check()
    tm.tm_wait_timeout_probe()
    with pytest.raises(tm.TmError) as e:
        tm.tm_check()
    assert e.value.status == tm.TM_ERR_TIMEOUT
    tm.tm_check()                                   # the status word was cleared
    a = torch.arange(1000, dtype=torch.float32, device="cuda")
    out = torch.empty_like(a)
    tm.tm_affine(a, out, 1000)
    tm.tm_check()
    assert torch.equal(out, a * 2 + 1)


@pytest.mark.gpu
@pytest.mark.parametrize("per_thread", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("n", [4096 * 4096, 1 << 20, 1024 * 16 * 3 + 4 * 37])
def test_read_probe_block_sums(cuda, oracle, per_thread, n):
    # block b sums elements [b*1024*U, (b+1)*1024*U); the last block may be ragged
    x = synth.uniform((n,), 0.0, 1.0, 40)
    blocks = tm.tm_read_probe_blocks(n, per_thread)
    span = 1024 * per_thread
    assert blocks == -(-n // span)
    padded = np.zeros(blocks * span, np.float32)
    padded[:n] = x
    want = oracle.rowsum(padded, span, blocks, span)
    out = DevBuf.empty(blocks)
    tm.tm_read_probe(DevBuf(x).ptr, n, out.ptr, per_thread)
    tm.tm_check()
    assert out.guards_intact()
    assert np.all(np.abs(out.payload_f32() - want) <= 1e-5 * want)


@pytest.mark.parametrize("n,blocks", [(1 << 24, 512), (1 << 24, 608), (4_100_000, 300), (8192, 5), (4, 1)])
def test_read_probe_fixed_block_sums(cuda, oracle, n, blocks):
    # block b sums elements [b*share, min((b+1)*share, n)); blocks past n write 0
    x = synth.uniform((n,), 0.0, 1.0, 41)
    share = tm.tm_read_probe_fixed_share(n, blocks)
    assert share % 8192 == 0 and share * blocks >= n and share * (blocks - 1) < n + 8192 * blocks
    padded = np.zeros(blocks * share, np.float32)
    padded[:n] = x
    want = oracle.rowsum(padded, share, blocks, share)
    out = DevBuf.empty(blocks)
    tm.tm_read_probe_fixed(DevBuf(x).ptr, n, out.ptr, blocks)
    tm.tm_check()
    assert out.guards_intact()
    got = out.payload_f32()
    assert np.all(np.abs(got - want) <= 1e-5 * want)
    assert np.all(got[want == 0] == 0)
