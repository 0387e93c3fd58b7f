"""Thin ctypes binding of ``libtm.so`` (declared in ``include/tm.h``).

Argument marshalling only: every entry point keeps its C name and argument
order; pointers may be given as integers or as objects with ``data_ptr()``
(torch tensors); ``stream=None`` means torch's current CUDA stream when torch
is loaded, else the legacy default stream.  A non-OK status raises
``TmError`` (its ``.status`` holds the code).  There is no fallback: if the
library was not built this module raises on first use.
"""
from __future__ import annotations

import ctypes
import os
import sys
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libtm.so")

# status codes (tm_status)
TM_OK = 0
TM_ERR_INVALID_ARG = 1
TM_ERR_UNSUPPORTED_TILE = 2
TM_ERR_MISALIGNED = 3
TM_ERR_BROKEN_PROMISE = 4
TM_ERR_CUDA = 5
TM_ERR_WORKSPACE = 6
TM_ERR_TIMEOUT = 7

# flags
TM_ALIGNED = 0x1
TM_PATH_SCALAR = 0x10
TM_PATH_VEC = 0x20
TM_PATH_TMA = 0x40
TM_PDL = 0x200  # overlapped launch; tm_affine takes it OR-ed into the variant

# tm_variant
TM_VAR_AUTO = 0
TM_VAR_SCALAR = 1
TM_VAR_VEC_UNALIGNED = 2
TM_VAR_VEC4 = 3
TM_VAR_VEC8 = 4
TM_VAR_NAIVE = 5
TM_VAR_STAGED = 6
TM_VAR_REGDIRECT = 7
TM_VAR_CLUSTER = 8

# tm_fill
TM_FILL_NEG_INF = 0
TM_FILL_ZERO = 1

# Every function include/tm.h declares, with its ctypes signature.
_i64, _i32, _u32, _f32, _vp, _sz = (ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_float,
                                    ctypes.c_void_p, ctypes.c_size_t)
_st = ctypes.c_int
SIGNATURES = {
    "tm_status_string": (ctypes.c_char_p, [_st]),
    "tm_version": (ctypes.c_int, []),
    "tm_affine": (_st, [_vp, _vp, _i64, _st, _vp]),
    "tm_scale2d": (_st, [_vp, _i64, _vp, _i64, _i64, _i64, _f32, _i32, _i32, _u32, _vp]),
    "tm_copy2d": (_st, [_vp, _i64, _vp, _i64, _i64, _i64, _i32, _i32, _u32, _vp]),
    "tm_channel_affine": (_st, [_vp, _i64, _i64, _i64, _vp, _vp, _i64, _i32, _vp, _i64, _i32, _i32, _u32, _vp]),
    "tm_padded_extent": (_i64, [_i64, _vp, _i32]),
    "tm_row_stride": (_i64, [_i64, _i32]),
    "tm_pad2d": (_st, [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _i64, _vp]),
    "tm_rowsum": (_st, [_vp, _i64, _i64, _i64, _vp, _i32, _i32, _u32, _vp]),
    "tm_colsum_workspace_bytes": (_sz, [_i64, _i64, _i32, _i32, _st]),
    "tm_colsum": (_st, [_vp, _i64, _i64, _i64, _vp, _vp, _sz, _i32, _i32, _st, _u32, _vp]),
    "tm_rowmax_masked": (_st, [_vp, _i64, _i64, _i64, _vp, _i32, _i32, _st, _u32, _vp]),
    "tm_softmax_rowstats": (_st, [_vp, _i64, _i64, _i64, _vp, _vp, _i32, _i32, _st, _u32, _vp]),
    "tm_colsum_noalloc": (_st, [_vp, _i64, _i64, _i64, _vp, _i32, _i32, _st, _u32, _vp]),
    "tm_gemm_workspace_bytes": (_sz, [_i64, _i64, _i64, _i32]),
    "tm_gemm": (_st, [_vp, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _i64, _f32, _f32, _i32, _i32, _i32, _u32,
                      _vp, _sz, _vp]),
    "tm_check": (_st, [_vp]),
    "tm_tile_walk_probe": (_st, [_i64, _i32, _vp, _vp]),
    "tm_scale2d_unchecked": (_st, [_vp, _i64, _vp, _i64, _i64, _i64, _f32, _i32, _i32, _vp]),
    "tm_wait_timeout_probe": (_st, [_vp]),
    "tm_read_probe_blocks": (_i64, [_i64, _i32]),
    "tm_read_probe": (_st, [_vp, _i64, _vp, _i32, _vp]),
    "tm_read_probe_fixed_share": (_i64, [_i64, _i32]),
    "tm_read_probe_fixed": (_st, [_vp, _i64, _vp, _i32, _vp]),
}

_lib = None
_lock = threading.Lock()


class TmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s" % (where, status_string(status)))


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libtm.so (once) and attach the signatures; raise if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError("libtm.so is not built (%s); run "
                                   "`python -m masking_tm_affine_gb300.build`" % path)
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(s) -> int | None:
    if s is None:
        torch = sys.modules.get("torch")
        if torch is not None and torch.cuda.is_available() and torch.cuda.is_initialized():
            return torch.cuda.current_stream().cuda_stream
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _ok(st: int, where: str) -> None:
    if st != TM_OK:
        raise TmError(st, where)


def status_string(st: int) -> str:
    return load().tm_status_string(st).decode()


def tm_version() -> int:
    return load().tm_version()


def tm_affine(a, out, n: int, variant: int = TM_VAR_AUTO, stream=None) -> None:
    _ok(load().tm_affine(_ptr(a), _ptr(out), n, variant, _stream(stream)), "tm_affine")


def tm_scale2d(X, ldx: int, Y, ldy: int, M: int, N: int, alpha: float, TM: int, TN: int,
               flags: int = 0, stream=None) -> None:
    _ok(load().tm_scale2d(_ptr(X), ldx, _ptr(Y), ldy, M, N, alpha, TM, TN, flags, _stream(stream)),
        "tm_scale2d")


def tm_copy2d(A, lda: int, B, ldb: int, M: int, N: int, TM: int, TN: int, flags: int = 0,
              stream=None) -> None:
    _ok(load().tm_copy2d(_ptr(A), lda, _ptr(B), ldb, M, N, TM, TN, flags, _stream(stream)), "tm_copy2d")


TM_CHANNELS_LAST = 0
TM_CHANNELS_FIRST = 1


def tm_channel_affine(X, ldx: int, R: int, K: int, scale, bias, C: int, layout: int, Y, ldy: int,
                      TM: int = 32, TN: int = 128, flags: int = 0, stream=None) -> None:
    _ok(load().tm_channel_affine(_ptr(X), ldx, R, K, _ptr(scale), _ptr(bias), C, layout, _ptr(Y), ldy, TM, TN,
                                 flags, _stream(stream)), "tm_channel_affine")


def tm_padded_extent(extent: int, tiles) -> int:
    arr = (ctypes.c_int32 * len(tiles))(*tiles)
    return int(load().tm_padded_extent(extent, ctypes.cast(arr, ctypes.c_void_p), len(tiles)))


def tm_row_stride(N: int, align_bytes: int = 16) -> int:
    return int(load().tm_row_stride(N, align_bytes))


def tm_pad2d(A, lda: int, M: int, N: int, B, ldb: int, Mp: int, Np: int, stream=None) -> None:
    _ok(load().tm_pad2d(_ptr(A), lda, M, N, _ptr(B), ldb, Mp, Np, _stream(stream)), "tm_pad2d")


def tm_rowsum(X, ldx: int, M: int, N: int, r, TM: int = 8, TN: int = 512, flags: int = 0,
              stream=None) -> None:
    _ok(load().tm_rowsum(_ptr(X), ldx, M, N, _ptr(r), TM, TN, flags, _stream(stream)), "tm_rowsum")


def tm_colsum_workspace_bytes(M: int, N: int, TM: int = 32, TN: int = 128,
                              variant: int = TM_VAR_AUTO) -> int:
    return int(load().tm_colsum_workspace_bytes(M, N, TM, TN, variant))


def tm_colsum(X, ldx: int, M: int, N: int, c, workspace, ws_bytes: int, TM: int = 32, TN: int = 128,
              variant: int = TM_VAR_AUTO, flags: int = 0, stream=None) -> None:
    _ok(load().tm_colsum(_ptr(X), ldx, M, N, _ptr(c), _ptr(workspace), ws_bytes, TM, TN, variant, flags,
                         _stream(stream)), "tm_colsum")


TM_NOALLOC_SCRATCH_BYTES = 8 << 20  # include/tm.h


def tm_colsum_noalloc(X, ldx: int, M: int, N: int, c, TM: int = 32, TN: int = 128,
                      variant: int = TM_VAR_AUTO, flags: int = 0, stream=None) -> None:
    """tm_colsum without a workspace, for callers that cannot allocate device
    memory; see include/tm.h for the scratch limit and the concurrency rule."""
    _ok(load().tm_colsum_noalloc(_ptr(X), ldx, M, N, _ptr(c), TM, TN, variant, flags, _stream(stream)),
        "tm_colsum_noalloc")


def tm_rowmax_masked(S, lds: int, M: int, N: int, m, BR: int = 8, BC: int = 64,
                     fill: int = TM_FILL_NEG_INF, flags: int = 0, stream=None) -> None:
    _ok(load().tm_rowmax_masked(_ptr(S), lds, M, N, _ptr(m), BR, BC, fill, flags, _stream(stream)),
        "tm_rowmax_masked")


def tm_softmax_rowstats(S, lds: int, M: int, N: int, m, l, BR: int = 8, BC: int = 64,
                        fill: int = TM_FILL_NEG_INF, flags: int = 0, stream=None) -> None:
    _ok(load().tm_softmax_rowstats(_ptr(S), lds, M, N, _ptr(m), _ptr(l), BR, BC, fill, flags, _stream(stream)),
        "tm_softmax_rowstats")


TM_GEMM_TF32 = 0x100  # include/tm.h


def tm_gemm_workspace_bytes(M: int, N: int, K: int, TN: int = 256) -> int:
    return load().tm_gemm_workspace_bytes(M, N, K, TN)


def tm_gemm(A, lda: int, B, ldb: int, C, ldc: int, M: int, N: int, K: int, alpha: float, beta: float,
            workspace, ws_bytes: int, TM: int = 256, TN: int = 256, TK: int = 32, flags: int = 0,
            stream=None) -> None:
    """C = alpha * (A B) + beta * C on the tensor cores (3xTF32 unless TM_GEMM_TF32).
    TM = 256 runs CTA pairs (the default, fastest); TM = 128 single CTAs."""
    _ok(load().tm_gemm(_ptr(A), lda, _ptr(B), ldb, _ptr(C), ldc, M, N, K, alpha, beta, TM, TN, TK, flags,
                       _ptr(workspace), ws_bytes, _stream(stream)), "tm_gemm")


def tm_check(stream=None) -> None:
    _ok(load().tm_check(_stream(stream)), "tm_check")


def tm_tile_walk_probe(K: int, T: int, out4, stream=None) -> None:
    _ok(load().tm_tile_walk_probe(K, T, _ptr(out4), _stream(stream)), "tm_tile_walk_probe")


def tm_read_probe_blocks(n: int, per_thread: int = 4) -> int:
    return int(load().tm_read_probe_blocks(n, per_thread))


def tm_read_probe(x, n: int, out, per_thread: int = 4, stream=None) -> None:
    """The plain streaming read of n floats (one fp32 sum per 1024*per_thread elements)."""
    _ok(load().tm_read_probe(_ptr(x), n, _ptr(out), per_thread, _stream(stream)), "tm_read_probe")


def tm_read_probe_fixed_share(n: int, blocks: int) -> int:
    return int(load().tm_read_probe_fixed_share(n, blocks))


def tm_read_probe_fixed(x, n: int, out, blocks: int, stream=None) -> None:
    """The same read with exactly `blocks` blocks, each summing its own fixed contiguous share."""
    _ok(load().tm_read_probe_fixed(_ptr(x), n, _ptr(out), blocks, _stream(stream)), "tm_read_probe_fixed")


def tm_wait_timeout_probe(stream=None) -> None:
    """A bounded wait that runs out (~1 s): the next tm_check raises TM_ERR_TIMEOUT."""
    _ok(load().tm_wait_timeout_probe(_stream(stream)), "tm_wait_timeout_probe")


def tm_scale2d_unchecked(X, ldx: int, Y, ldy: int, M: int, N: int, alpha: float, TM: int, TN: int,
                         stream=None) -> None:
    _ok(load().tm_scale2d_unchecked(_ptr(X), ldx, _ptr(Y), ldy, M, N, alpha, TM, TN, _stream(stream)),
        "tm_scale2d_unchecked")
