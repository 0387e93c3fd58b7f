"""The bench line's per-config block checks every output against the oracle
before it times anything.  Here each of its entries (the workloads' kernels
and the two floors C3 and C4 are read against) runs once on its full-size
input through the same call the bench times, and must pass that check; the
same check must reject the output once one element of the host copy is moved
(so a check that accepts anything would fail here)."""
import numpy as np
import pytest
import torch

import bench
from masking_tm_affine_gb300 import synth

pytestmark = pytest.mark.gpu

_inputs = {}


def _input(wl):
    if wl not in _inputs:
        _inputs.clear()  # one workload resident at a time
        _inputs[wl] = synth.workload_input(wl)
    return _inputs[wl]


@pytest.mark.parametrize("entry", bench.CONFIG_ENTRIES, ids=[e[0] for e in bench.CONFIG_ENTRIES])
def test_config_entry_passes_its_oracle_check(cuda, oracle, entry):
    key, cfg, wl, kern, path, target = entry
    x = _input(wl)
    dev = torch.device("cuda", 0)
    desc, on, call, nbytes, wn, check = bench.config_kernel(cuda, kern, path, synth.WORKLOADS[wl], x, dev)
    assert nbytes >= 4 * x.size  # every entry reads its whole input at least once
    X = torch.from_numpy(x.reshape(-1)).to(dev)
    O = torch.full((on,), float("nan"), dtype=torch.float32, device=dev)
    W = torch.empty(max(wn, 4), dtype=torch.float32, device=dev)
    s = torch.cuda.current_stream(dev).cuda_stream
    call(X, O, W, s, False)
    cuda.tm_check(s)
    o = O.cpu().numpy()
    assert check(o), (key, desc)
    # the overlapped form of the call gives the same result
    O2 = torch.full((on,), float("nan"), dtype=torch.float32, device=dev)
    call(X, O2, W, s, True)
    cuda.tm_check(s)
    assert check(O2.cpu().numpy()), (key, "TM_PDL")
    # one element moved by at least 1: beyond every tolerance these checks use
    bad = o.copy()
    k = on // 3
    bad[k] = bad[k] + max(1.0, abs(float(bad[k])))
    assert not check(bad), key
