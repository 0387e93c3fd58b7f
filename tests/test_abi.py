"""The C-ABI library loads, exports every symbol include/tm.h declares, and
rejects bad arguments on the host before touching CUDA (no GPU needed)."""
import os
import re

import pytest

from conftest import ROOT
from masking_tm_affine_gb300 import tm

HEADER = os.path.join(ROOT, "include", "tm.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tm_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from masking_tm_affine_gb300 import build
    build.build()
    return tm.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ["tm_affine", "tm_scale2d", "tm_copy2d", "tm_rowsum", "tm_colsum", "tm_colsum_workspace_bytes",
              "tm_rowmax_masked", "tm_check", "tm_status_string"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert set(names) == set(tm.SIGNATURES), "binding and header disagree"
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    for code in range(0, 8):
        s = tm.status_string(code)
        assert s.startswith("TM_")
    assert tm.status_string(99) == "TM_ERR_UNKNOWN"
    assert tm.tm_version() >= 10000


# Fake but well-aligned device addresses: every case below must be rejected on
# the host, before any CUDA call, so nothing ever dereferences them.
P0, P1 = 0x7F0000000000, 0x7F0100000000


def st(fn, *args):
    # fake addresses: only ever passed where no device exists, so a case that
    # slipped past the host checks fails with TM_ERR_CUDA instead of launching
    import torch
    if torch.cuda.is_available():
        pytest.skip("fake-address host checks run only on a machine without a GPU")
    return getattr(tm.load(), fn)(*args)


def test_affine_host_validation(lib):
    assert st("tm_affine", P0, P1, -1, 0, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_affine", None, P1, 5, 0, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_affine", P0, P1, 5, 99, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_affine", P0 + 4, P1, 5, tm.TM_VAR_VEC4, None) == tm.TM_ERR_MISALIGNED
    assert st("tm_affine", P0 + 16, P1, 5, tm.TM_VAR_VEC8, None) == tm.TM_ERR_MISALIGNED
    assert st("tm_affine", P0 + 2, P1, 5, 0, None) == tm.TM_ERR_MISALIGNED
    assert st("tm_affine", P0, P0 + 8, 5, 0, None) == tm.TM_ERR_INVALID_ARG  # partial overlap
    assert st("tm_affine", P0, P1, 0, 0, None) == tm.TM_OK                   # empty: no launch


@pytest.mark.parametrize("fn", ["tm_scale2d", "tm_copy2d"])
def test_map2d_host_validation(lib, fn):
    def call(X, ldx, Y, ldy, M, N, TM, TN, flags):
        if fn == "tm_scale2d":
            return st(fn, X, ldx, Y, ldy, M, N, 1.5, TM, TN, flags, None)
        return st(fn, X, ldx, Y, ldy, M, N, TM, TN, flags, None)
    A = tm.TM_ALIGNED
    assert call(P0, 8, P1, 8, -1, 8, 32, 128, 0) == tm.TM_ERR_INVALID_ARG
    assert call(P0, 7, P1, 8, 4, 8, 32, 128, 0) == tm.TM_ERR_INVALID_ARG        # ld < N
    assert call(None, 8, P1, 8, 4, 8, 32, 128, 0) == tm.TM_ERR_INVALID_ARG
    assert call(P0, 8, P1, 8, 4, 8, 32, 128, 0x8) == tm.TM_ERR_INVALID_ARG      # unknown flag
    assert call(P0, 8, P1, 8, 4, 8, 32, 128, tm.TM_PATH_SCALAR | tm.TM_PATH_VEC) == tm.TM_ERR_INVALID_ARG
    assert call(P0, 8, P1, 8, 4, 8, 0, 128, 0) == tm.TM_ERR_UNSUPPORTED_TILE    # divisor must be positive
    assert call(P0, 8, P1, 8, 4, 8, 32, 64, 0) == tm.TM_ERR_UNSUPPORTED_TILE    # not instantiated
    assert call(P0, 8192, P1, 8192, 8192, 8100, 32, 128, A) == tm.TM_ERR_BROKEN_PROMISE
    assert call(P0, 8192, P1, 8192, 8190, 8192, 32, 128, A) == tm.TM_ERR_BROKEN_PROMISE
    assert call(P0 + 4, 8192, P1, 8192, 8192, 8192, 32, 128, A) == tm.TM_ERR_MISALIGNED
    assert call(P0, 8190, P1, 8192, 64, 128, 32, 128, A) == tm.TM_ERR_MISALIGNED  # ld % 4 != 0
    assert call(P0, 8, P0 + 8, 8, 4, 8, 8, 8, 0) == tm.TM_ERR_INVALID_ARG         # partial overlap
    assert call(P0, 8, P0, 12, 4, 8, 8, 8, 0) == tm.TM_ERR_INVALID_ARG            # same base, other ld
    assert call(P0, 8, P1, 8, 0, 8, 8, 8, 0) == tm.TM_OK                          # empty
    assert call(P0, 8, P1, 8, 4, 0, 8, 8, 0) == tm.TM_OK


def test_reduction_host_validation(lib):
    A = tm.TM_ALIGNED
    assert st("tm_rowsum", P0, 8, 4, 8, P1, 3, 128, 0, None) == tm.TM_ERR_UNSUPPORTED_TILE
    assert st("tm_rowsum", P0, 8, 4, 8, P1, 8, 100, 0, None) == tm.TM_ERR_UNSUPPORTED_TILE
    assert st("tm_rowsum", P0, 8, 4, 8, None, 8, 128, 0, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_rowsum", P0, 4096, 4096, 4000, P1, 8, 512, A, None) == tm.TM_ERR_BROKEN_PROMISE
    assert st("tm_rowmax_masked", P0, 1000, 8192, 1000, P1, 8, 64, 0, A, None) == tm.TM_ERR_BROKEN_PROMISE
    assert st("tm_rowmax_masked", P0, 1000, 8192, 1000, P1, 8, 64, 7, 0, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_rowmax_masked", P0, 1000, 8192, 1000, P1, 8, 48, 0, 0, None) == tm.TM_ERR_UNSUPPORTED_TILE
    ws = tm.tm_colsum_workspace_bytes(4096, 4096, 32, 128)
    assert ws > 0 and ws % 16 == 0
    assert st("tm_colsum", P0, 4096, 4096, 4096, P1, None, ws, 32, 128, 0, 0, None) == tm.TM_ERR_WORKSPACE
    assert st("tm_colsum", P0, 4096, 4096, 4096, P1, P1 + (1 << 30), ws - 4, 32, 128, 0, 0, None) \
        == tm.TM_ERR_WORKSPACE
    assert st("tm_colsum", P0, 4096, 4096, 4096, P1, P1 + (1 << 30), ws, 32, 96, 0, 0, None) \
        == tm.TM_ERR_UNSUPPORTED_TILE
    assert st("tm_colsum", P0, 4096, 4096, 4000, P1, P1 + (1 << 30), ws, 32, 128, 0, A, None) \
        == tm.TM_ERR_BROKEN_PROMISE
    assert st("tm_tile_walk_probe", 10, 0, P0, None) == tm.TM_ERR_INVALID_ARG
    # the streaming-read probe: n % 4, per_thread, alignment, overlap
    assert tm.tm_read_probe_blocks(1 << 24, 4) == 4096 and tm.tm_read_probe_blocks(4100, 1) == 5
    assert tm.tm_read_probe_blocks(6, 4) == -1 and tm.tm_read_probe_blocks(8, 3) == -1
    assert st("tm_read_probe", P0, 6, P1, 4, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_read_probe", P0, 8, P1, 5, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_read_probe", None, 8, P1, 4, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_read_probe", P0 + 4, 8, P1, 4, None) == tm.TM_ERR_MISALIGNED
    assert st("tm_read_probe", P0, 1 << 20, P0 + 64, 4, None) == tm.TM_ERR_INVALID_ARG  # out inside x
    assert st("tm_read_probe", P0, 0, None, 4, None) == tm.TM_OK                      # nothing to read
    # the fixed-share read: whole 8192-float steps per block, blocks in 1 .. 65535
    assert tm.tm_read_probe_fixed_share(1 << 26, 512) == (1 << 26) // 512
    assert tm.tm_read_probe_fixed_share(1 << 26, 608) == 8192 * -(-(1 << 26) // (8192 * 608))
    assert tm.tm_read_probe_fixed_share(4, 1) == 8192 and tm.tm_read_probe_fixed_share(0, 7) == 0
    assert tm.tm_read_probe_fixed_share(6, 4) == -1 and tm.tm_read_probe_fixed_share(8, 0) == -1
    assert tm.tm_read_probe_fixed_share(8, 65536) == -1
    assert st("tm_read_probe_fixed", P0, 6, P1, 4, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_read_probe_fixed", P0, 8, P1, 0, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_read_probe_fixed", P0, 8, None, 4, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_read_probe_fixed", P0 + 4, 8, P1, 4, None) == tm.TM_ERR_MISALIGNED
    assert st("tm_read_probe_fixed", P0, 1 << 20, P0 + 64, 4, None) == tm.TM_ERR_INVALID_ARG  # out inside x
    assert st("tm_read_probe_fixed", P0, 0, None, 4, None) == tm.TM_OK


def test_overlap_flag_host_validation(lib):
    """TM_PDL is accepted wherever flags are (and OR-ed into tm_affine's variant):
    the other checks still run and decide the status; tm_gemm does not take it."""
    A, D = tm.TM_ALIGNED, tm.TM_PDL
    assert st("tm_affine", P0 + 4, P1, 5, tm.TM_VAR_VEC4 | D, None) == tm.TM_ERR_MISALIGNED
    assert st("tm_affine", P0, P1, 5, 99 | D, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_affine", P0, P1, 5, 0x400, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_affine", P0, P1, 0, tm.TM_VAR_AUTO | D, None) == tm.TM_OK
    assert st("tm_scale2d", P0, 8192, P1, 8192, 8192, 8100, 1.5, 32, 128, A | D, None) == tm.TM_ERR_BROKEN_PROMISE
    assert st("tm_copy2d", P0, 8192, P1, 8192, 8190, 8192, 32, 128, A | D, None) == tm.TM_ERR_BROKEN_PROMISE
    assert st("tm_copy2d", P0, 8, P1, 8, 0, 8, 8, 8, D, None) == tm.TM_OK
    assert st("tm_channel_affine", P0, 256, 8192, 256, None, None, 256, tm.TM_CHANNELS_LAST, P1, 256, 32, 128,
              D | 0x8, None) == tm.TM_ERR_INVALID_ARG
    assert st("tm_channel_affine", P0, 256, 8190, 256, None, None, 256, tm.TM_CHANNELS_LAST, P1, 256, 32, 128,
              A | D, None) == tm.TM_ERR_BROKEN_PROMISE
    assert st("tm_rowsum", P0, 4096, 4096, 4000, P1, 8, 512, A | D, None) == tm.TM_ERR_BROKEN_PROMISE
    assert st("tm_rowmax_masked", P0, 1000, 8192, 1000, P1, 8, 64, 0, A | D, None) == tm.TM_ERR_BROKEN_PROMISE
    assert st("tm_softmax_rowstats", P0, 1000, 8192, 1000, P1, P1 + (1 << 20), 8, 64, 0, A | D, None) \
        == tm.TM_ERR_BROKEN_PROMISE
    ws = tm.tm_colsum_workspace_bytes(4096, 4096, 32, 128)
    assert st("tm_colsum", P0, 4096, 4096, 4096, P1, None, ws, 32, 128, 0, D, None) == tm.TM_ERR_WORKSPACE
    assert st("tm_colsum", P0, 4096, 4096, 4000, P1, P1 + (1 << 30), ws, 32, 128, 0, A | D, None) \
        == tm.TM_ERR_BROKEN_PROMISE
    W = 0x7F0200000000
    gws = tm.tm_gemm_workspace_bytes(4100, 4100, 1000, 256)
    assert st("tm_gemm", P0, 1000, P1, 4100, W + (1 << 34), 4100, 4100, 4100, 1000, 1.5, 0.5, 256, 256, 32, D,
              W, gws, None) == tm.TM_ERR_INVALID_ARG


def colsum_plan(M, N, TM, TN, target_units=8192, min_rows=64):
    """The one-pass column sum's chunk plan: S strips of TN columns, P row
    chunks of CT row tiles each (about target_units units, at least min_rows
    rows per chunk)."""
    S, RT = -(-N // TN), -(-M // TM)
    P = min(max(-(-target_units // S), 1), RT)
    CT = max(-(-RT // P), -(-min_rows // TM))
    return S, -(-RT // CT)


def test_colsum_workspace_plan(lib):
    # NAIVE: one partial row (N rounded up to 4) per 256-row program block
    assert tm.tm_colsum_workspace_bytes(4096, 4096, 32, 128, tm.TM_VAR_NAIVE) == 16 * 4096 * 4
    assert tm.tm_colsum_workspace_bytes(4100, 1001, 32, 128, tm.TM_VAR_NAIVE) == 17 * 1004 * 4
    assert tm.tm_colsum_workspace_bytes(0, 4096, 32, 128) == 0
    assert tm.tm_colsum_workspace_bytes(100, 0, 32, 128) == 0
    assert tm.tm_colsum_workspace_bytes(100, 10, 33, 128) == 0
    assert tm.tm_colsum_workspace_bytes(4096, 4096, 32, 128, tm.TM_VAR_CLUSTER) == 0
    assert tm.tm_colsum_workspace_bytes(4096, 4096, 32, 128, tm.TM_VAR_STAGED) == 0  # partials meet on chip
    # REGDIRECT (and AUTO, which sizes for it): a TN-wide partial per (strip,
    # chunk); none when every strip is one chunk
    for M, N, TM, TN in [(4100, 1001, 32, 128), (4096, 4096, 32, 128), (8192, 8192, 32, 128), (8192, 1000, 8, 64),
                         (3, 1 << 20, 8, 256), (1 << 20, 3, 256, 64), (192, 768000, 8, 256)]:
        S, P = colsum_plan(M, N, TM, TN)
        want = 0 if P == 1 else S * P * TN * 4
        for v in (tm.TM_VAR_AUTO, tm.TM_VAR_REGDIRECT):
            assert tm.tm_colsum_workspace_bytes(M, N, TM, TN, v) == want, (M, N, TM, TN, v)
        assert tm.tm_colsum_workspace_bytes(M, N, TM, TN, tm.TM_VAR_STAGED) == 0
    assert colsum_plan(4100, 1001, 32, 128) == (8, 65)
    assert tm.tm_colsum_workspace_bytes(4100, 1001, 32, 128) == 8 * 65 * 128 * 4
    assert tm.tm_colsum_workspace_bytes(64, 4096, 32, 128) == 0  # one 64-row chunk per strip
    assert tm.tm_colsum_workspace_bytes(8192, 8192, 32, 128) == 4 << 20
    assert colsum_plan(192, 768000, 8, 256) == (3000, 3)
    assert tm.tm_colsum_workspace_bytes(192, 768000, 8, 256) == 9000 * 1024 > tm.TM_NOALLOC_SCRATCH_BYTES


def test_padding_helpers_match_oracle(lib, oracle):
    # host-only entry points (no CUDA call): against the oracle's search definitions
    for tiles in ([32], [64], [32, 256], [4, 16], [64, 128, 256], [3, 5], [1]):
        for extent in list(range(0, 70)) + [1000, 4100, 8192, 8193, 10**9 + 7]:
            if extent > 10**6 and max(tiles) < 32:
                continue  # the oracle's search is linear in the gap
            assert tm.tm_padded_extent(extent, tiles) == oracle.padded_extent(extent, tiles), (extent, tiles)
    for N in list(range(0, 100)) + [1000, 1001, 4099, 10**9 + 3]:
        for align in (4, 16, 32, 128):
            assert tm.tm_row_stride(N, align) == oracle.row_stride(N, align), (N, align)
    assert tm.tm_padded_extent(10, [0]) == -1
    assert tm.tm_padded_extent(-1, [4]) == -1
    assert tm.tm_padded_extent(10, []) == -1
    assert tm.tm_row_stride(10, 6) == -1 and tm.tm_row_stride(10, 12) == -1
    assert tm.tm_padded_extent(2**63 - 1, [2]) == -1       # the next multiple of 2 overflows int64
    assert tm.tm_padded_extent(2**62, [3, 5, 7]) == -(-2**62 // 105) * 105


def test_gemm_host_validation(lib):
    W = 0x7F0200000000  # 1024-byte aligned fake workspace
    ws = tm.tm_gemm_workspace_bytes(4100, 4100, 1000, 256)
    # operands zero-padded to whole tiles (rows of A to 256, either TM): [4352, 1024] hi + lo twice;
    # then split-K partials for at most 256 accumulators of 128 x TN rows (there are 34 x 17 such
    # tiles here) and 256 flags
    assert ws == 2 * 4352 * 1024 * 4 + 2 * 4352 * 1024 * 4 + 256 * 128 * 256 * 4 + 1024
    # short K: no split-K, no partials
    assert tm.tm_gemm_workspace_bytes(4100, 4100, 0, 256) == 4 * 4352 * 32 * 4 + 1024
    # few tiles: partials only for as many 128-row accumulators as C has (2 x 1 here)
    assert tm.tm_gemm_workspace_bytes(200, 200, 1000, 256) == 4 * 256 * 1024 * 4 + 2 * 128 * 256 * 4 + 1024
    # K of at most 48 * 16: no split-K, no partials
    assert tm.tm_gemm_workspace_bytes(200, 200, 768, 256) == 4 * 256 * 768 * 4 + 1024
    assert tm.tm_gemm_workspace_bytes(0, 4, 4, 256) == 0 and tm.tm_gemm_workspace_bytes(4, 4, 4, 64) == 0

    def g(A=P0, lda=1000, B=P1, ldb=4100, C=W + (1 << 34), ldc=4100, M=4100, N=4100, K=1000, TM=128, TN=256,
          TK=32, flags=0, ws_ptr=W, ws_bytes=ws):
        return st("tm_gemm", A, lda, B, ldb, C, ldc, M, N, K, 1.5, 0.5, TM, TN, TK, flags, ws_ptr, ws_bytes, None)

    assert g(TM=64) == tm.TM_ERR_UNSUPPORTED_TILE
    assert g(TM=512) == tm.TM_ERR_UNSUPPORTED_TILE
    assert g(M=4224, N=4096, K=1024, lda=1024, ldb=4096, ldc=4096, TM=256,
             flags=tm.TM_ALIGNED) == tm.TM_ERR_BROKEN_PROMISE       # 4224 % 256 != 0
    assert g(TK=8) == tm.TM_ERR_UNSUPPORTED_TILE
    assert g(TK=64) == tm.TM_ERR_UNSUPPORTED_TILE
    assert g(TN=512) == tm.TM_ERR_UNSUPPORTED_TILE
    assert g(M=-1) == tm.TM_ERR_INVALID_ARG
    assert g(lda=999) == tm.TM_ERR_INVALID_ARG
    assert g(flags=0x4) == tm.TM_ERR_INVALID_ARG
    assert g(A=None) == tm.TM_ERR_INVALID_ARG
    assert g(A=P0 + 2) == tm.TM_ERR_MISALIGNED
    assert g(flags=tm.TM_ALIGNED) == tm.TM_ERR_BROKEN_PROMISE
    assert g(M=4096, N=4096, K=1000, ldc=4096, flags=tm.TM_ALIGNED, ws_bytes=ws) == tm.TM_ERR_BROKEN_PROMISE
    assert g(ws_bytes=ws - 1) == tm.TM_ERR_WORKSPACE
    assert g(ws_ptr=W + 512) == tm.TM_ERR_WORKSPACE
    assert g(ws_ptr=None) == tm.TM_ERR_WORKSPACE
    assert g(C=P0 + 4096) == tm.TM_ERR_INVALID_ARG                     # C overlaps A
    assert g(ws_ptr=P1) == tm.TM_ERR_INVALID_ARG                       # workspace overlaps B
    assert g(M=2**31, ws_bytes=1 << 62) == tm.TM_ERR_INVALID_ARG        # padded M beyond 2^31 - 1
    assert g(M=0) == tm.TM_OK and g(N=0) == tm.TM_OK                   # empty: nothing launched


C_PROGRAM = r"""
#include "tm.h"
#include <stdio.h>
#include <string.h>

int main(void)
{
    /* host-side checks only: nothing here reaches the GPU */
    int bad = 0;
    bad |= tm_version() < 10000;
    bad |= strcmp(tm_status_string(TM_OK), "TM_OK") != 0;
    bad |= tm_affine(NULL, NULL, -1, TM_VAR_AUTO, NULL) != TM_ERR_INVALID_ARG;
    bad |= tm_scale2d(NULL, 8, NULL, 8, 4, 8, 1.5f, 32, 128, TM_ALIGNED | TM_PDL, NULL) != TM_ERR_INVALID_ARG;
    bad |= tm_rowsum(NULL, 8, 0, 8, NULL, 8, 128, 0, NULL) != TM_OK;            /* empty: no launch */
    bad |= tm_padded_extent(1000, (const int32_t[]){16, 64}, 2) != 1024;
    bad |= tm_row_stride(1001, 16) != 1004;
    bad |= tm_gemm_workspace_bytes(0, 4, 4, 256) != 0;
    printf("%s\n", bad ? "FAIL" : "ok");
    return bad;
}
"""


def test_header_is_plain_c_and_links(lib):
    """include/tm.h compiles as strict C99 and a C program links against
    libtm.so and calls it (host-side checks only)."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from masking_tm_affine_gb300 import build
    work = os.path.join(build.BUILD, "abi_check")  # the package's (ignored) build folder
    os.makedirs(work, exist_ok=True)
    src = os.path.join(work, "abi_check.c")
    with open(src, "w") as f:
        f.write(C_PROGRAM)
    exe = os.path.join(work, "abi_check")
    libdir = os.path.dirname(build.LIB)
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-L", libdir, "-ltm", "-Wl,-rpath," + libdir, "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0 and run.stdout.strip() == "ok", run.stdout + run.stderr


def _prototypes():
    """Each declared function's C parameter types, from include/tm.h."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    protos = {}
    for m in re.finditer(r"\b[\w ]+?\*?\s*\b(tm_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = " ".join(m.group(2).split())
        protos[m.group(1)] = [] if params in ("", "void") else [p.strip() for p in params.split(",")]
    return protos


def _ctype_of(param):
    """The ctypes type a C parameter maps to under this binding's conventions."""
    import ctypes
    decl = param.rsplit(" ", 1)[0] if not param.endswith("*") else param
    if "*" in param or "tm_stream_t" in param:
        return ctypes.c_void_p
    for key, ct in (("int64_t", ctypes.c_int64), ("int32_t", ctypes.c_int32), ("uint32_t", ctypes.c_uint32),
                    ("size_t", ctypes.c_size_t), ("float", ctypes.c_float), ("tm_variant", ctypes.c_int),
                    ("tm_fill", ctypes.c_int), ("tm_status", ctypes.c_int)):
        if decl.split()[0] == key:
            return ct
    raise AssertionError("unmapped parameter type: %r" % param)


def test_binding_signatures_match_the_header():
    """Every binding signature has the header's parameter count and types, so a
    change to include/tm.h cannot silently misalign the ctypes calls."""
    protos = _prototypes()
    assert set(protos) == set(tm.SIGNATURES)
    for name, params in protos.items():
        _, argtypes = tm.SIGNATURES[name]
        assert len(params) == len(argtypes), (name, params, argtypes)
        for p, at in zip(params, argtypes):
            assert _ctype_of(p) == at, (name, p, at)
