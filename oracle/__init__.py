"""CPU oracle for the tiled fp32 maps -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it; the two meet only on the seeded inputs that
``masking_tm_affine_gb300.synth`` generates.

The arithmetic lives in ``tm_oracle.c`` (plain single-threaded C, compiled with
``-O2 -fno-fast-math -ffp-contract=off``); this module compiles it on demand
with gcc and marshals numpy arrays through ctypes.  Each wrapper names the page
passage its C function follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None

FILL_NEG_INF = 0  # where(iota < N - kt, s, -inf): the ragged row-max mask
FILL_ZERO = 1     # no where step: masked loads read 0 (the pitfall)


def build(force: bool = False) -> str:
    """Compile ``tm_oracle.c`` into ``liboracle.so`` (if missing or stale)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, f32, vp, i32 = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
        lib.oracle_tile_walk.argtypes = [i64, i64, vp]
        lib.oracle_tile_walk.restype = i32
        lib.oracle_tile_valid.argtypes = [i64, i64, i64, i64, i64, i64]
        lib.oracle_tile_valid.restype = i64
        lib.oracle_promise_kept.argtypes = [i64, i64, i64, i64]
        lib.oracle_promise_kept.restype = i32
        lib.oracle_affine.argtypes = [vp, vp, i64]
        lib.oracle_affine.restype = None
        lib.oracle_scale2d.argtypes = [vp, i64, vp, i64, i64, i64, f32]
        lib.oracle_scale2d.restype = None
        lib.oracle_copy2d.argtypes = [vp, i64, vp, i64, i64, i64]
        lib.oracle_copy2d.restype = None
        lib.oracle_rowsum.argtypes = [vp, i64, i64, i64, vp]
        lib.oracle_rowsum.restype = None
        lib.oracle_colsum.argtypes = [vp, i64, i64, i64, vp]
        lib.oracle_colsum.restype = None
        lib.oracle_rowmax_masked.argtypes = [vp, i64, i64, i64, i64, i32, vp]
        lib.oracle_rowmax_masked.restype = i32
        lib.oracle_softmax_rowstats.argtypes = [vp, i64, i64, i64, i64, i32, vp, vp]
        lib.oracle_softmax_rowstats.restype = i32
        lib.oracle_channel_affine.argtypes = [vp, i64, i64, i64, vp, vp, i64, i32, vp, i64]
        lib.oracle_channel_affine.restype = i32
        lib.oracle_padded_extent.argtypes = [i64, vp, i32]
        lib.oracle_padded_extent.restype = i64
        lib.oracle_row_stride.argtypes = [i64, i32]
        lib.oracle_row_stride.restype = i64
        lib.oracle_pad2d.argtypes = [vp, i64, i64, i64, vp, i64, i64, i64]
        lib.oracle_pad2d.restype = None
        lib.oracle_gemm_rows.argtypes = [vp, i64, vp, i64, vp, i64, vp, i64, i64, i64, f32, f32, vp]
        lib.oracle_gemm_rows.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _as_f32_flat(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    if x.dtype != np.float32:
        raise TypeError("oracle expects float32 input, got %s" % x.dtype)
    return x.reshape(-1)


def _check_2d(buf: np.ndarray, ld: int, M: int, N: int, what: str) -> None:
    if M < 0 or N < 0 or ld < N:
        raise ValueError("%s: need M, N >= 0 and ld >= N (M=%d N=%d ld=%d)" % (what, M, N, ld))
    if M > 0 and N > 0 and buf.size < (M - 1) * ld + N:
        raise ValueError("%s: buffer of %d words is too small for [%d, %d] with ld=%d"
                         % (what, buf.size, M, N, ld))


def tile_walk(K: int, T: int) -> dict:
    """Whole/masked split of ``for kt in range(0, K, T)`` ("Slicing, bounds and
    masking", "Loops over a dynamic extent")."""
    out = np.zeros(4, dtype=np.int64)
    if _load().oracle_tile_walk(K, T, _ptr(out)) != 0:
        raise ValueError("tile walk needs K >= 0 and T > 0")
    return {"whole": int(out[0]), "masked": int(out[1]), "rem": int(out[2]), "iters": int(out[3])}


def tile_valid(M: int, N: int, TM: int, TN: int, pm: int, pn: int) -> int:
    """In-bounds element count of tile (pm, pn) ("Slicing, bounds and masking", "Masking")."""
    return int(_load().oracle_tile_valid(M, N, TM, TN, pm, pn))


def promise_kept(M: int, N: int, TM: int, TN: int) -> bool:
    """Whether ``@aligned(M = TM, N = TN)`` holds ("@aligned", "When the promise is broken")."""
    r = _load().oracle_promise_kept(M, N, TM, TN)
    if r < 0:
        raise ValueError("tile divisors must be positive")
    return bool(r)


def affine(a) -> np.ndarray:
    """out = a*2 + 1 over every element ("Aligned Load & Store", "The exercise")."""
    a = _as_f32_flat(a)
    out = np.empty_like(a)
    _load().oracle_affine(_ptr(a), _ptr(out), a.size)
    return out


def scale2d(X: np.ndarray, ldx: int, Y: np.ndarray, ldy: int, M: int, N: int, alpha: float) -> None:
    """In place on ``Y``: Y[i, j] = alpha*X[i, j] for i < M, j < N; other words
    untouched ("@aligned", "A minimal kernel"; "Masking")."""
    X = _as_f32_flat(X)
    if Y.dtype != np.float32 or not Y.flags.c_contiguous:
        raise TypeError("Y must be a contiguous float32 array")
    _check_2d(X, ldx, M, N, "X")
    _check_2d(Y.reshape(-1), ldy, M, N, "Y")
    _load().oracle_scale2d(_ptr(X), ldx, _ptr(Y), ldy, M, N, float(alpha))


def copy2d(A: np.ndarray, lda: int, B: np.ndarray, ldb: int, M: int, N: int) -> None:
    """In place on ``B``: bitwise B[i, j] = A[i, j] for i < M, j < N
    ("Slicing, bounds and masking", "Promising whole tiles with @aligned")."""
    A = np.ascontiguousarray(A).reshape(-1).view(np.uint32)
    if B.dtype.itemsize != 4 or not B.flags.c_contiguous:
        raise TypeError("B must be a contiguous 4-byte array")
    _check_2d(A, lda, M, N, "A")
    _check_2d(B.reshape(-1), ldb, M, N, "B")
    _load().oracle_copy2d(_ptr(A), lda, _ptr(B), ldb, M, N)


def rowsum(X, ldx: int, M: int, N: int) -> np.ndarray:
    """fp64 per-row sums ("Memory Coalescing and Tensor Layout", "What it actually costs")."""
    X = _as_f32_flat(X)
    _check_2d(X, ldx, M, N, "X")
    r = np.zeros(M, dtype=np.float64)
    _load().oracle_rowsum(_ptr(X), ldx, M, N, _ptr(r))
    return r


def colsum(X, ldx: int, M: int, N: int) -> np.ndarray:
    """fp64 per-column sums ("Memory Coalescing and Tensor Layout", "What it actually costs")."""
    X = _as_f32_flat(X)
    _check_2d(X, ldx, M, N, "X")
    c = np.zeros(N, dtype=np.float64)
    _load().oracle_colsum(_ptr(X), ldx, M, N, _ptr(c))
    return c


def rowmax_masked(S, lds: int, M: int, N: int, BC: int, fill: int = FILL_NEG_INF) -> np.ndarray:
    """Ragged row-max over BC-wide column tiles with the where/iota mask
    ("Slicing, bounds and masking", "Reductions over a ragged tile")."""
    S = _as_f32_flat(S)
    _check_2d(S, lds, M, N, "S")
    m = np.empty(M, dtype=np.float32)
    if _load().oracle_rowmax_masked(_ptr(S), lds, M, N, BC, fill, _ptr(m)) != 0:
        raise ValueError("rowmax needs BC > 0 and a known fill")
    return m


def softmax_rowstats(S, lds: int, M: int, N: int, BC: int, fill: int = FILL_NEG_INF):
    """Row maximum m (float32) and normaliser l = sum exp(s - m) (float64) over
    BC-wide ragged column tiles ("Slicing, bounds and masking", "Reductions over
    a ragged tile": the softmax needs the same -inf fill as the maximum)."""
    S = _as_f32_flat(S)
    _check_2d(S, lds, M, N, "S")
    m = np.empty(M, dtype=np.float32)
    l = np.empty(M, dtype=np.float64)
    if _load().oracle_softmax_rowstats(_ptr(S), lds, M, N, BC, fill, _ptr(m), _ptr(l)) != 0:
        raise ValueError("softmax row statistics need BC > 0 and a known fill")
    return m, l


CHANNELS_LAST = 0   # [N, C] view of [B, C, H, W]: channel = column
CHANNELS_FIRST = 1  # [B*C, H*W] view: channel = row mod C


def channel_affine(X, ldx: int, R: int, K: int, scale, bias, C: int, layout: int, Y: np.ndarray, ldy: int) -> None:
    """In place on ``Y``: Y = X*scale[ch] + bias[ch] per channel, one rounding
    ("Memory Coalescing and Tensor Layout", "NCHW versus NHWC")."""
    X = _as_f32_flat(X)
    if Y.dtype != np.float32 or not Y.flags.c_contiguous:
        raise TypeError("Y must be a contiguous float32 array")
    _check_2d(X, ldx, R, K, "X")
    _check_2d(Y.reshape(-1), ldy, R, K, "Y")
    sp = None if scale is None else _as_f32_flat(scale)
    bp = None if bias is None else _as_f32_flat(bias)
    for v in (sp, bp):
        if v is not None and v.size < C:
            raise ValueError("parameter vector shorter than C")
    if _load().oracle_channel_affine(_ptr(X), ldx, R, K, None if sp is None else _ptr(sp),
                                     None if bp is None else _ptr(bp), C, layout, _ptr(Y), ldy) != 0:
        raise ValueError("channel affine needs C > 0, a known layout, and K <= C for channels last")


def padded_extent(extent: int, tiles) -> int:
    """Smallest extent >= the given one that every candidate tile divides
    ("@aligned", "Interactions")."""
    t = np.ascontiguousarray(tiles, dtype=np.int32)
    r = _load().oracle_padded_extent(extent, _ptr(t), t.size)
    if r < 0:
        raise ValueError("bad extent or tiles")
    return int(r)


def row_stride(N: int, align_bytes: int = 16) -> int:
    """Smallest row stride >= N whose rows are whole multiples of align_bytes
    ("Memory Coalescing and Tensor Layout", "The alignment constraint")."""
    r = _load().oracle_row_stride(N, align_bytes)
    if r < 0:
        raise ValueError("bad N or alignment")
    return int(r)


def pad2d(A, lda: int, M: int, N: int, B: np.ndarray, ldb: int, Mp: int, Np: int) -> None:
    """In place on ``B``: A inside [M, N], zeros in the rest of [Mp, Np]."""
    A = np.ascontiguousarray(A).reshape(-1).view(np.uint32)
    if B.dtype.itemsize != 4 or not B.flags.c_contiguous:
        raise TypeError("B must be a contiguous 4-byte array")
    if Mp < M or Np < N:
        raise ValueError("padded extents must cover the source")
    _check_2d(A, lda, M, N, "A")
    _check_2d(B.reshape(-1), ldb, Mp, Np, "B")
    _load().oracle_pad2d(_ptr(A), lda, M, N, _ptr(B), ldb, Mp, Np)


def gemm_rows(A, lda: int, B, ldb: int, Cin, ldc: int, rows, N: int, K: int, alpha: float = 1.0,
              beta: float = 0.0) -> np.ndarray:
    """Rows ``rows`` of alpha*(A B) + beta*Cin, fp64 then rounded once to fp32
    ("@aligned", the gemm example; "Slicing, bounds and masking", "Loops over a
    dynamic extent").  A [*, lda] rows hold K used columns, B [K, ldb] rows N."""
    A = _as_f32_flat(A)
    B = _as_f32_flat(B)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if K > 0 and (lda < K or ldb < N):
        raise ValueError("leading dimensions too small")
    if B.size < max(0, (K - 1) * ldb + N) and K > 0 and N > 0:
        raise ValueError("B too small")
    if rows.size and A.size < (int(rows.max()) * lda + K):
        raise ValueError("A too small for the requested rows")
    if beta != 0.0:
        Cin = _as_f32_flat(Cin)
        if rows.size and Cin.size < int(rows.max()) * ldc + N:
            raise ValueError("C too small for the requested rows")
        cptr = _ptr(Cin)
    else:
        cptr = None
    out = np.empty((rows.size, N), dtype=np.float32)
    _load().oracle_gemm_rows(_ptr(A), lda, _ptr(B), ldb, cptr, ldc, _ptr(rows), rows.size, N, K,
                             float(alpha), float(beta), _ptr(out))
    return out
