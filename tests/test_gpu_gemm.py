"""GPU parity of tm_gemm against the oracle ("@aligned", the gemm example;
"Slicing, bounds and masking", "Loops over a dynamic extent").

Three kinds of check:
* integer-valued operands (|a|, |b|, |c| <= 8): every product and partial sum
  is exact in tf32 and fp32, so the tensor-core result must equal the oracle's
  bit for bit -- this pins the data movement (split, transpose, zero padding of
  the K remainder, tile offsets, masked edges) independently of rounding;
* one nonzero per column of B: each output is a single product, so the only
  error is the operand split's -- a dropped hi*lo or lo*hi term (2^-11
  relative) fails the 3xTF32 bound (about 2^-20) by orders of magnitude;
* real-valued operands: every element within the bound include/tm.h states.
"""
import numpy as np
import pytest
import torch

from gpu_util import CANARY, DevBuf
from masking_tm_affine_gb300 import synth, tm

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def ints(shape, seed):
    return np.round(synth.uniform(shape, -8.5, 8.5, seed)).astype(np.float32)


def workspace(M, N, K, TN):
    ws = tm.tm_gemm_workspace_bytes(M, N, K, TN)
    raw = torch.empty(ws + 1024, dtype=torch.uint8, device="cuda")
    base = raw.data_ptr()
    return raw, (base + 1023) // 1024 * 1024, ws


def run(a, b, c, alpha, beta, TN=256, flags=0, lda=None, ldb=None, ldc=None, TK=32, TM=128):
    """C <- alpha a b + beta c on the GPU; returns (the [M, ldc] result, the
    padded host inputs, and a guard check)."""
    M, K = a.shape
    N = b.shape[1]
    lda, ldb, ldc = lda or K or 1, ldb or N, ldc or N
    Ah = synth.pad_rows(a, lda) if M and K else np.zeros(max(M * lda, 1), np.float32)
    Bh = synth.pad_rows(b, ldb) if K and N else np.zeros(max(K * ldb, 1), np.float32)
    Ch = synth.pad_rows(c, ldc) if M and N else np.zeros(max(M * ldc, 1), np.float32)
    AD, BD, CD = DevBuf(Ah), DevBuf(Bh), DevBuf(Ch)
    raw, ws, wsb = workspace(max(M, 1), max(N, 1), K, TN)
    tm.tm_gemm(AD.ptr, lda, BD.ptr, ldb, CD.ptr, ldc, M, N, K, alpha, beta, ws, wsb, TM, TN, TK, flags)
    tm.tm_check()
    assert AD.guards_intact() and BD.guards_intact() and CD.guards_intact()
    out = CD.payload_f32()
    if M and N:
        gaps = CD.payload_u32().reshape(M, ldc)[:, N:]
        assert np.array_equal(gaps, Ch.view(np.uint32).reshape(M, ldc)[:, N:]), "C's ld gap was written"
    return out, Ah, Bh, Ch, lda, ldb, ldc


def bound(a, b, c, alpha, beta, want, three=True):
    """Per-element error bound (include/tm.h, tm_gemm, Accuracy) in fp64."""
    K = a.shape[1]
    S = abs(alpha) * (np.abs(a.astype(np.float64)) @ np.abs(b.astype(np.float64)))
    split = 3 * 2.0 ** -22 if three else 2 * 2.0 ** -11 + 2.0 ** -22
    passes = 3 if three else 1
    return (split + passes * K * 2.0 ** -23) * S + 2.0 ** -22 * (np.abs(beta * c.astype(np.float64))
                                                                  + np.abs(want.astype(np.float64)) + S)


SHAPES = [(1, 1, 1), (1, 5, 3), (7, 9, 13), (128, 256, 32), (128, 128, 64), (130, 200, 1000), (257, 300, 33),
          (300, 513, 95), (64, 1000, 1000), (1000, 36, 8), (4, 4, 4), (129, 132, 40)]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("TN", [128, 256])
@pytest.mark.parametrize("TK", [16, 32])
@pytest.mark.parametrize("flags", [0, tm.TM_GEMM_TF32])
@pytest.mark.parametrize("c_rows", ["tma", "direct"])
@pytest.mark.parametrize("TM", [128, 256])
def test_gemm_integers_exact(cuda, oracle, M, N, K, TN, TK, flags, c_rows, TM):
    # TM 256: CTA pairs (cta_group::2), each CTA holding half of every B tile
    # c_rows: ldc a multiple of 4 (C moves through TMA chunks when N % 4 == 0,
    # the edges clipped by the copy engine; direct stores otherwise, with the
    # ld gap right after a row end that is not 16-byte aligned) or ldc not a
    # multiple of 4 (direct stores)
    ldc = (N + 3) // 4 * 4 + 4 if c_rows == "tma" else N + 2
    if c_rows == "direct" and ldc % 4 == 0:
        ldc += 1
    a, b, c = ints((M, K), 11 + M), ints((K, N), 12 + N), ints((M, N), 13 + K)
    out, Ah, Bh, Ch, lda, ldb, ldc = run(a, b, c, 1.5, 0.5, TN, flags, lda=K + 3, ldb=N + 1, ldc=ldc, TK=TK, TM=TM)
    want = oracle.gemm_rows(Ah, lda, Bh, ldb, Ch, ldc, np.arange(M), N, K, 1.5, 0.5)
    got = out.reshape(M, ldc)[:, :N]
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("M,N,K", [(128, 256, 32), (256, 512, 1024), (384, 128, 96), (2048, 1024, 48)])
@pytest.mark.parametrize("TN", [128, 256])
@pytest.mark.parametrize("TK", [16, 32])
@pytest.mark.parametrize("TM", [128, 256])
def test_gemm_aligned_promise_exact(cuda, oracle, M, N, K, TN, TK, TM):
    if N % TN or K % TK or M % TM:
        pytest.skip("extents not whole tiles")
    a, b, c = ints((M, K), 21), ints((K, N), 22), ints((M, N), 23)
    out, Ah, Bh, Ch, lda, ldb, ldc = run(a, b, c, -1.0, 2.0, TN, tm.TM_ALIGNED, TK=TK, TM=TM)
    want = oracle.gemm_rows(Ah, lda, Bh, ldb, Ch, ldc, np.arange(M), N, K, -1.0, 2.0)
    assert np.array_equal(out.reshape(M, N).view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("flags", [0, tm.TM_GEMM_TF32])
@pytest.mark.parametrize("TM", [128, 256])
def test_gemm_single_product_split_accuracy(cuda, oracle, flags, TM):
    # B holds one nonzero per column: C[i, j] = alpha * A[i, k_j] * B[k_j, j]
    M, N, K = 200, 300, 77
    a = synth.uniform((M, K), -1.0, 1.0, 31)
    vals = synth.uniform((N,), 0.5, 2.0, 32)
    kj = (np.arange(N) * 37) % K
    b = np.zeros((K, N), np.float32)
    b[kj, np.arange(N)] = vals
    c = np.zeros((M, N), np.float32)
    out, Ah, Bh, Ch, lda, ldb, ldc = run(a, b, c, 1.0, 0.0, 256, flags, TM=TM)
    want = oracle.gemm_rows(Ah, lda, Bh, ldb, Ch, ldc, np.arange(M), N, K, 1.0, 0.0)
    got = out.reshape(M, N).astype(np.float64)
    rel = np.abs(got - want) / np.maximum(np.abs(want.astype(np.float64)), 1e-30)
    if flags == 0:
        # three passes: the dropped lo*lo term and the lo roundings, 3 * 2^-22, plus two
        # accumulations (truncating at worst) and the oracle's one rounding
        assert rel.max() <= 3 * 2.0 ** -22 + 2 * 2.0 ** -23 + U
    else:
        # one pass: both operands rounded to tf32 (2^-11 each)
        assert rel.max() <= 2 * 2.0 ** -11 + 2.0 ** -22 + 2.0 ** -23 + U
        assert rel.max() > 2.0 ** -16, "tf32-only result unexpectedly accurate"


@pytest.mark.parametrize("M,N,K", [(130, 200, 1000), (257, 300, 33), (1, 1000, 4099), (500, 37, 1),
                                   (2100, 700, 260)])
@pytest.mark.parametrize("flags", [0, tm.TM_GEMM_TF32])
@pytest.mark.parametrize("TM,TN,TK", [(128, 256, 32), (128, 128, 16), (256, 256, 16), (256, 128, 32)])
def test_gemm_real_within_bound(cuda, oracle, M, N, K, flags, TM, TN, TK):
    a = synth.uniform((M, K), -1.0, 1.0, 41)
    b = synth.normal((K, N), 42)
    c = synth.uniform((M, N), -4.0, 4.0, 43)
    out, Ah, Bh, Ch, lda, ldb, ldc = run(a, b, c, 1.5, -0.5, TN, flags, TK=TK, TM=TM)
    want = oracle.gemm_rows(Ah, lda, Bh, ldb, Ch, ldc, np.arange(M), N, K, 1.5, -0.5)
    got = out.reshape(M, N)
    err = np.abs(got.astype(np.float64) - want)
    assert np.all(err <= bound(a, b, c, 1.5, -0.5, want, three=(flags == 0)))


def test_gemm_degenerate(cuda, oracle):
    # K == 0: C = beta * C
    c = ints((70, 90), 51)
    out, *_ = run(np.zeros((70, 0), np.float32), np.zeros((0, 90), np.float32), c, 1.5, 0.5, lda=1, ldb=90)
    assert np.array_equal(out.reshape(70, 90), 0.5 * c)
    # beta == 0 never reads C: NaN in C does not reach the result (direct and TMA epilogues)
    a, b = ints((40, 20), 52), ints((20, 30), 53)
    cn = np.full((40, 30), np.nan, np.float32)
    for ldc in (30, 36):
        out, Ah, Bh, Ch, lda, ldb, ldc = run(a, b, cn, 1.0, 0.0, ldc=ldc)
        want = oracle.gemm_rows(Ah, lda, Bh, ldb, None, 0, np.arange(40), 30, 20, 1.0, 0.0)
        assert np.array_equal(out.reshape(40, ldc)[:, :30], want)
    # empty M or N: nothing launched, nothing written
    CD = DevBuf.empty(16)
    raw, ws, wsb = workspace(1, 1, 4, 256)
    tm.tm_gemm(CD.ptr, 4, CD.ptr, 4, CD.ptr, 4, 0, 4, 4, 1.0, 0.0, ws, wsb)
    tm.tm_gemm(CD.ptr, 4, CD.ptr, 4, CD.ptr, 4, 4, 0, 4, 1.0, 0.0, ws, wsb)
    tm.tm_check()
    assert np.all(CD.words() == CANARY)


def test_gemm_errors(cuda):
    AD, BD, CD = DevBuf.empty(256), DevBuf.empty(256), DevBuf.empty(256)
    raw, ws, wsb = workspace(16, 16, 16, 256)

    def status(*args, **kw):
        with pytest.raises(tm.TmError) as e:
            tm.tm_gemm(*args, **kw)
        return e.value.status

    base = (AD.ptr, 16, BD.ptr, 16, CD.ptr, 16, 16, 16, 16, 1.0, 0.0)
    assert status(*base, ws, wsb, TM=64) == tm.TM_ERR_UNSUPPORTED_TILE
    assert status(*base, ws, wsb, TN=64) == tm.TM_ERR_UNSUPPORTED_TILE
    assert status(*base, ws, wsb, TK=8) == tm.TM_ERR_UNSUPPORTED_TILE
    assert status(*base, ws, wsb, flags=tm.TM_ALIGNED) == tm.TM_ERR_BROKEN_PROMISE
    assert status(*base, ws, wsb, flags=0x2) == tm.TM_ERR_INVALID_ARG
    assert status(*base, ws, wsb - 4) == tm.TM_ERR_WORKSPACE
    assert status(*base, ws + 16, wsb) == tm.TM_ERR_WORKSPACE                  # not 1024-byte aligned
    assert status(*base, None, wsb) == tm.TM_ERR_WORKSPACE
    assert status(AD.ptr, 16, BD.ptr, 16, AD.ptr, 16, 16, 16, 16, 1.0, 0.0, ws, wsb) == tm.TM_ERR_INVALID_ARG
    assert status(AD.ptr + 2, 16, BD.ptr, 16, CD.ptr, 16, 16, 16, 16, 1.0, 0.0, ws, wsb) == tm.TM_ERR_MISALIGNED
    tm.tm_check()
    assert np.all(CD.words() == CANARY)


@pytest.mark.parametrize("name", ["gemm_4100", "gemm_8192"])
@pytest.mark.parametrize("TM", [128, 256])
def test_gemm_full_size_sampled_rows(cuda, oracle, name, TM):
    # the bench workloads, in the launch configuration the bench times; rows at
    # tile edges and a seeded sample, each checked element by element
    w = synth.WORKLOADS[name]
    M, N, K = w["M"], w["N"], w["K"]
    a, b, c = synth.gemm_inputs(name)
    A, B, C = (torch.from_numpy(t).cuda() for t in (a, b, c))
    raw, ws, wsb = workspace(M, N, K, w["TN"])
    aligned = M % TM == 0 and N % w["TN"] == 0 and K % w["TK"] == 0
    tm.tm_gemm(A, K, B, N, C, N, M, N, K, w["alpha"], w["beta"], ws, wsb, TM, w["TN"], w["TK"],
               tm.TM_ALIGNED if aligned else 0)
    tm.tm_check()
    rng = np.random.Generator(np.random.PCG64(M + K))
    rows = np.unique(np.concatenate([[0, 1, 127, 128, M // 2, M - 2, M - 1], rng.integers(0, M, 25)]))
    got = C[torch.from_numpy(rows).cuda()].cpu().numpy()
    want = oracle.gemm_rows(a, K, b, N, c, N, rows, N, K, w["alpha"], w["beta"])
    err = np.abs(got.astype(np.float64) - want)
    assert np.all(err <= bound(a[rows], b, c[rows], w["alpha"], w["beta"], want))


@pytest.mark.parametrize("TM", [128, 256])
@pytest.mark.parametrize("lead", [1, 2, 3])
def test_gemm_unaligned_bases(cuda, oracle, TM, lead):
    # A, B and C start `lead` words past a 16-byte boundary: the split reads
    # with 4-byte loads and C takes the direct epilogue (no TMA on C); the ld
    # gaps hold poison that must never be read, the lead words and canaries
    # must come back untouched
    M, N, K = 150, 132, 70
    a, b, c = ints((M, K), 61), ints((K, N), 62), ints((M, N), 63)
    lda, ldb, ldc = K + 2, N + 4, N + 4
    Ah, Bh, Ch = synth.pad_rows(a, lda), synth.pad_rows(b, ldb), synth.pad_rows(c, ldc)
    AD, BD, CD = DevBuf(Ah, lead), DevBuf(Bh, lead), DevBuf(Ch, lead)
    raw, ws, wsb = workspace(M, N, K, 256)
    tm.tm_gemm(AD.ptr, lda, BD.ptr, ldb, CD.ptr, ldc, M, N, K, 1.5, 0.5, ws, wsb, TM, 256, 32)
    tm.tm_check()
    assert AD.guards_intact() and BD.guards_intact() and CD.guards_intact()
    got = CD.payload_u32().reshape(M, ldc)
    want = oracle.gemm_rows(Ah, lda, Bh, ldb, Ch, ldc, np.arange(M), N, K, 1.5, 0.5)
    assert np.array_equal(got[:, :N], want.view(np.uint32))
    assert np.array_equal(got[:, N:], Ch.view(np.uint32).reshape(M, ldc)[:, N:])


# Tile counts that leave at most half of the last round of units (152 CTAs, or 76 CTA pairs, on GB300)
# busy, with enough K stages for split-K (it must take >= 48 stages off the critical path): each of that
# round's tiles is cut along K into units // tiles parts -- 3 here for 2560 x 2560, 2 for 2500 x 2600 --
# run side by side, and finished by the unit that ran the first part.
# With TN = 128 and N = 1152 the last round holds 14 of 76 pair tiles (28 of 152 CTA tiles): 5 parts each.
SK_CASES = [(2560, 2560, 4096, 32, 256), (2560, 2560, 4096, 16, 256), (2500, 2600, 3200, 32, 256),
            (2560, 1152, 4096, 32, 128)]


@pytest.mark.parametrize("M,N,K,TK,TN", SK_CASES)
@pytest.mark.parametrize("flags", [0, tm.TM_GEMM_TF32])
@pytest.mark.parametrize("TM", [128, 256])
def test_gemm_split_k_integers_exact(cuda, oracle, M, N, K, TK, TN, flags, TM):
    a, b, c = ints((M, K), 31), ints((K, N), 32), ints((M, N), 33)
    out, Ah, Bh, Ch, lda, ldb, ldc = run(a, b, c, 1.5, 0.5, TN, flags, ldc=N + 4, TK=TK, TM=TM)
    rows = np.unique(np.r_[np.arange(0, M, 29), np.arange(M - 70, M)])
    want = oracle.gemm_rows(Ah, lda, Bh, ldb, Ch, ldc, rows, N, K, 1.5, 0.5)
    got = out.reshape(M, ldc)[rows, :N]
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


@pytest.mark.parametrize("TM", [128, 256])
def test_gemm_split_k_deterministic(cuda, TM):
    """Real-valued operands: two calls give the same bits (a split tile's
    parts are added in K order, whichever unit finishes first)."""
    M, N, K = 2500, 2600, 3200
    a = synth.uniform((M, K), -1.0, 1.0, 41)
    b = synth.uniform((K, N), -1.0, 1.0, 42)
    c = synth.uniform((M, N), -1.0, 1.0, 43)
    first = run(a, b, c, 1.5, 0.5, 256, TM=TM)[0]
    second = run(a, b, c, 1.5, 0.5, 256, TM=TM)[0]
    assert np.array_equal(first.view(np.uint32), second.view(np.uint32))
