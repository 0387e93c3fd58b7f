"""The hot path at full size, in the launch configuration bench.py times.

One step of the benchmark -- the fp32 [8192, 8192] batch (X ~ N(0,1), seed 1)
through affine, scale2d (32 x 128, aligned), copy2d (64 x 64, aligned),
rowsum, colsum and rowmax_masked with exactly the calls and tiles bench.py
makes, overlapped (TM_PDL, as timed) and plain -- checked against the oracle
on every row of every output.
"""
import pytest
import torch

import bench
from masking_tm_affine_gb300 import synth, tm

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("overlap", [True, False], ids=["overlapped", "plain"])
def test_bench_step_full_size_every_row(cuda, oracle, overlap):
    dev = torch.device("cuda", 0)
    x = synth.workload_input(bench.WORKLOAD)
    bufs, ws_bytes = bench.make_buffers(tm, x, dev)
    stream = torch.cuda.Stream(device=dev)
    step = bench.make_step(tm, bufs, ws_bytes, stream, overlap=overlap)
    with torch.cuda.stream(stream):
        for _ in range(2):          # twice: the second pass must not depend on the first's leftovers
            for _, launch in step:
                launch()
    tm.tm_check(stream.cuda_stream)
    torch.cuda.synchronize(dev)
    bench.verify_step(bufs, x, oracle, rows="all")
