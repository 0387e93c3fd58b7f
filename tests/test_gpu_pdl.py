"""Overlapped launches (TM_PDL): results and stream order.

A call that passes TM_PDL may start while the previous kernel in its stream
drains: its loads of the inputs may run ahead of that kernel, its stores and
its completion may not.  These tests check that (1) every entry point gives
the oracle's result when every call of a chain is overlapped, and (2) the
ordering the flag keeps: a store never overtakes an earlier kernel's read of
the same buffer (write after read), one or two calls back, nor its write
(write after write), and back-to-back column sums may share one workspace.
Each ordering case is repeated on tensors of 64-128 MiB, where a store that
ran early would land inside the earlier kernel's walk.
"""
import numpy as np
import pytest
import torch

from gpu_util import same_f32
from masking_tm_affine_gb300 import synth, tm

pytestmark = pytest.mark.gpu

REL = 1e-5
P = tm.TM_PDL


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.cpu().numpy()


def sums_close(got, want, absref):
    got = np.asarray(got, dtype=np.float64)
    return bool(np.all(np.abs(got - want) <= REL * absref + 1e-30))


def test_overlapped_chain_matches_oracle(cuda, oracle):
    """Every entry point in one stream, each call overlapped on the one before."""
    x = synth.workload_input("ragged_4100")                       # [4100, 1000] U[-8, 8) seed 2
    M, N = x.shape
    xa = synth.uniform((4096, 1024), -8.0, 8.0, seed=21)          # whole 32 x 128 and 64 x 64 tiles
    scale, bias = synth.channel_params(N, seed=6)
    s = synth.uniform((8192, 1000), -30.0, -1.0, seed=4)          # the row-max scores
    a = synth.workload_input("affine_1m")                         # 1M U[-1, 1) seed 0

    X, XA, S, A = dev(x), dev(xa), dev(s), dev(a)
    SC, BI = dev(scale), dev(bias)
    out = {k: torch.empty(n, dtype=torch.float32, device="cuda") for k, n in [
        ("aff_auto", a.size), ("aff_scalar", a.size), ("aff_unal", a.size), ("aff_v4", a.size), ("aff_v8", a.size),
        ("scale", x.size), ("scale_al", xa.size), ("copy_sc", x.size), ("chan", x.size),
        ("rs", M), ("cs_auto", N), ("cs_naive", N), ("cs_staged", N), ("cs_reg", N), ("cs_cl", N), ("cs_na", N),
        ("rm", s.shape[0]), ("sm_m", s.shape[0]), ("sm_l", s.shape[0])]}
    ws = max(tm.tm_colsum_workspace_bytes(M, N, 32, 128, v) for v in (tm.TM_VAR_AUTO, tm.TM_VAR_NAIVE))
    W = torch.empty(ws // 4 + 4, dtype=torch.float32, device="cuda")

    st = torch.cuda.Stream()
    q = st.cuda_stream
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        for name, v in [("aff_auto", tm.TM_VAR_AUTO), ("aff_scalar", tm.TM_VAR_SCALAR),
                        ("aff_unal", tm.TM_VAR_VEC_UNALIGNED), ("aff_v4", tm.TM_VAR_VEC4),
                        ("aff_v8", tm.TM_VAR_VEC8)]:
            tm.tm_affine(A, out[name], a.size, v | P, q)
        tm.tm_scale2d(X, N, out["scale"], N, M, N, 1.5, 64, 64, P, q)                       # ragged vectors
        tm.tm_scale2d(XA, 1024, out["scale_al"], 1024, 4096, 1024, 1.5, 32, 128, tm.TM_ALIGNED | P, q)
        tm.tm_copy2d(X, N, out["copy_sc"], N, M, N, 64, 64, tm.TM_PATH_SCALAR | P, q)       # masked scalars
        tm.tm_channel_affine(X, N, M, N, SC, BI, N, tm.TM_CHANNELS_LAST, out["chan"], N, 32, 128, P, q)
        tm.tm_rowsum(X, N, M, N, out["rs"], 8, 512, P, q)
        for name, v in [("cs_auto", tm.TM_VAR_AUTO), ("cs_naive", tm.TM_VAR_NAIVE),
                        ("cs_staged", tm.TM_VAR_STAGED), ("cs_reg", tm.TM_VAR_REGDIRECT),
                        ("cs_cl", tm.TM_VAR_CLUSTER)]:
            tm.tm_colsum(X, N, M, N, out[name], W, W.numel() * 4, 32, 128, v, P, q)
        tm.tm_colsum_noalloc(X, N, M, N, out["cs_na"], 32, 128, tm.TM_VAR_AUTO, P, q)
        tm.tm_rowmax_masked(S, 1000, 8192, 1000, out["rm"], 8, 64, tm.TM_FILL_NEG_INF, P, q)
        tm.tm_softmax_rowstats(S, 1000, 8192, 1000, out["sm_m"], out["sm_l"], 16, 64, tm.TM_FILL_NEG_INF, P, q)
    tm.tm_check(q)
    torch.cuda.synchronize()

    want_aff = oracle.affine(a)
    for name in ("aff_auto", "aff_scalar", "aff_unal", "aff_v4", "aff_v8"):
        assert same_f32(host(out[name]), want_aff), name
    want = np.empty_like(x)
    oracle.scale2d(x, N, want, N, M, N, 1.5)
    assert same_f32(host(out["scale"]).reshape(M, N), want)
    want_al = np.empty_like(xa)
    oracle.scale2d(xa, 1024, want_al, 1024, 4096, 1024, 1.5)
    assert same_f32(host(out["scale_al"]).reshape(4096, 1024), want_al)
    assert np.array_equal(host(out["copy_sc"]).view(np.uint32), x.reshape(-1).view(np.uint32))
    want_ch = np.empty_like(x)
    oracle.channel_affine(x, N, M, N, scale, bias, N, 0, want_ch, N)
    assert same_f32(host(out["chan"]).reshape(M, N), want_ch)

    absx = np.abs(x.astype(np.float64))
    assert sums_close(host(out["rs"]), oracle.rowsum(x, N, M, N), absx.sum(axis=1))
    want_c = oracle.colsum(x, N, M, N)
    for name in ("cs_auto", "cs_naive", "cs_staged", "cs_reg", "cs_cl", "cs_na"):
        assert sums_close(host(out[name]), want_c, absx.sum(axis=0)), name

    assert same_f32(host(out["rm"]), oracle.rowmax_masked(s, 1000, 8192, 1000, 64))
    m_ref, l_ref = oracle.softmax_rowstats(s, 1000, 8192, 1000, 64)
    assert same_f32(host(out["sm_m"]), m_ref)
    l_gpu = host(out["sm_l"]).astype(np.float64)
    assert np.all(np.abs(l_gpu - l_ref) <= REL * np.abs(l_ref))


@pytest.fixture(scope="module")
def big():
    """X [4096, 8192] ~ N(0,1) and an older Y ~ U[-1, 1): 128 MiB each."""
    x = synth.normal((4096, 8192), seed=31)
    y0 = synth.uniform((4096, 8192), -1.0, 1.0, seed=32)
    return x, y0


def test_store_waits_for_earlier_read(cuda, oracle, big):
    """rowsum reads Y, then an overlapped scale2d overwrites Y: the sums are Y's old ones."""
    x, y0 = big
    M, N = x.shape
    want = oracle.rowsum(y0, N, M, N)
    absref = np.abs(y0.astype(np.float64)).sum(axis=1)
    X, Y0 = dev(x), dev(y0)
    Y = torch.empty_like(Y0)
    r = torch.empty(M, dtype=torch.float32, device="cuda")
    st = torch.cuda.Stream()
    for trial in range(8):
        Y.copy_(Y0)
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            tm.tm_rowsum(Y, N, M, N, r, 1, 1024, tm.TM_ALIGNED, st.cuda_stream)
            tm.tm_scale2d(X, N, Y, N, M, N, 1.5, 32, 128, tm.TM_ALIGNED | P, st.cuda_stream)
        tm.tm_check(st.cuda_stream)
        torch.cuda.synchronize()
        assert sums_close(host(r), want, absref), trial


def test_store_waits_two_calls_back(cuda, oracle, big):
    """rowmax reads Y; an overlapped copy2d of X; an overlapped affine map into Y.
    The third call's stores wait for the second, which completes only after the first."""
    x, y0 = big
    M, N = x.shape
    want = oracle.rowmax_masked(y0, N, M, N, 64)
    X, Y0 = dev(x), dev(y0)
    Y, B = torch.empty_like(Y0), torch.empty_like(X)
    m = torch.empty(M, dtype=torch.float32, device="cuda")
    st = torch.cuda.Stream()
    for trial in range(8):
        Y.copy_(Y0)
        torch.cuda.synchronize()
        with torch.cuda.stream(st):
            tm.tm_rowmax_masked(Y, N, M, N, m, 1, 64, tm.TM_FILL_NEG_INF, tm.TM_ALIGNED, st.cuda_stream)
            tm.tm_copy2d(X, N, B, N, M, N, 64, 64, tm.TM_ALIGNED | P, st.cuda_stream)
            tm.tm_affine(X, Y, M * N, tm.TM_VAR_AUTO | P, st.cuda_stream)
        tm.tm_check(st.cuda_stream)
        torch.cuda.synchronize()
        assert same_f32(host(m), want), trial
    assert np.array_equal(host(B).reshape(-1).view(np.uint32), x.reshape(-1).view(np.uint32))
    assert same_f32(host(Y).reshape(-1), oracle.affine(x).reshape(-1))


def test_store_waits_for_earlier_write(cuda, big):
    """scale2d writes Y, then an overlapped copy2d writes Y again: the copy wins everywhere."""
    x, y0 = big
    M, N = x.shape
    X, Z = dev(x), dev(y0)
    Y = torch.empty_like(X)
    st = torch.cuda.Stream()
    for trial in range(8):
        flags = P if trial % 2 else 0     # the first call overlapped too, on odd trials
        with torch.cuda.stream(st):
            tm.tm_scale2d(X, N, Y, N, M, N, 1.5, 32, 128, tm.TM_ALIGNED | flags, st.cuda_stream)
            tm.tm_copy2d(Z, N, Y, N, M, N, 64, 64, tm.TM_ALIGNED | P, st.cuda_stream)
        tm.tm_check(st.cuda_stream)
        torch.cuda.synchronize()
        assert np.array_equal(host(Y).reshape(-1).view(np.uint32), y0.reshape(-1).view(np.uint32)), trial


@pytest.mark.parametrize("variant", [tm.TM_VAR_AUTO, tm.TM_VAR_NAIVE, tm.TM_VAR_STAGED])
def test_back_to_back_column_sums_share_a_workspace(cuda, oracle, variant):
    """Three overlapped column sums of different tensors through one workspace,
    and three through the library's built-in scratch."""
    M, N = 4096, 4096
    xs = [synth.uniform((M, N), 0.0, 1.0, seed=40 + k) for k in range(3)]
    wants = [oracle.colsum(x, N, M, N) for x in xs]
    Xs = [dev(x) for x in xs]
    ws = tm.tm_colsum_workspace_bytes(M, N, 32, 128, variant)
    W = torch.empty(ws // 4 + 4, dtype=torch.float32, device="cuda")
    cs = [torch.empty(N, dtype=torch.float32, device="cuda") for _ in range(6)]
    st = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(st):
        for rep in range(4):
            for k in range(3):
                tm.tm_colsum(Xs[k], N, M, N, cs[k], W, W.numel() * 4, 32, 128, variant, P, st.cuda_stream)
            for k in range(3):
                tm.tm_colsum_noalloc(Xs[k], N, M, N, cs[3 + k], 32, 128, variant, P, st.cuda_stream)
    tm.tm_check(st.cuda_stream)
    torch.cuda.synchronize()
    for k in range(3):
        for c in (cs[k], cs[3 + k]):
            assert sums_close(host(c), wants[k], wants[k]), (variant, k)


def test_overlapped_launch_on_the_default_stream(cuda, oracle):
    """TM_PDL on the legacy default stream (a NULL stream handle), after another kernel there."""
    x = synth.workload_input("ragged_4100")
    M, N = x.shape
    X = dev(x)
    Y, B = torch.empty_like(X), torch.empty_like(X)
    torch.cuda.synchronize()
    tm.tm_copy2d(X, N, B, N, M, N, 64, 64, 0, 0)
    tm.tm_scale2d(X, N, Y, N, M, N, 1.5, 64, 64, P, 0)
    tm.tm_check(0)
    torch.cuda.synchronize()
    want = np.empty_like(x)
    oracle.scale2d(x, N, want, N, M, N, 1.5)
    assert same_f32(host(Y), want)
    assert np.array_equal(host(B).view(np.uint32), x.view(np.uint32))


def test_overlapped_step_replays_from_a_cuda_graph(cuda, oracle):
    """The bench step (six overlapped calls) captured once into a CUDA graph,
    whose dependent launches become programmatic edges, and replayed: once on
    the batch, once after a new batch was copied into the same X."""
    import bench
    dev_ = torch.device("cuda", 0)
    x = synth.workload_input(bench.WORKLOAD)
    bufs, ws_bytes = bench.make_buffers(tm, x, dev_)
    stream = torch.cuda.Stream(device=dev_)
    step = bench.make_step(tm, bufs, ws_bytes, stream)
    with torch.cuda.stream(stream):
        for _, launch in step:          # once outside the graph (first-use set-up happens here)
            launch()
    tm.tm_check(stream.cuda_stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _, launch in step:
            launch()
    for k in ("A1", "Y", "B", "r", "c", "m"):
        bufs[k].fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    tm.tm_check()
    bench.verify_step(bufs, x, oracle)
    x2 = synth.normal((bench.M, bench.N), seed=33)
    bufs["X"].copy_(torch.from_numpy(x2.reshape(-1)))
    g.replay()
    torch.cuda.synchronize()
    tm.tm_check()
    bench.verify_step(bufs, x2, oracle)
