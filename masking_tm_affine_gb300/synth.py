"""Seeded synthetic inputs shaped like the pages' workloads.

This module holds no arithmetic of the maps themselves: it only draws the
random tensors that both the CUDA path and the CPU oracle consume, so that the
two see identical bits.  Draws use numpy's PCG64 generator in float64 and are
rounded to float32 once; uniform draws are then clamped into [lo, hi) so the
half-open bound holds exactly after rounding.

Workloads (sizes from the pages; distributions and seeds fixed here):

* ``affine_1m``    -- 1-D, n = 1,048,576, U[-1, 1), seed 0
  ("Aligned Load & Store", "The exercise": a 1M-element float32 buffer).
* ``scale_8192``   -- [8192, 8192], N(0, 1), seed 1, tiles 32 x 128
  ("@aligned", "A minimal kernel": TM = 32, TN = 128).
* ``ragged_4100``  -- [4100, 1000], U[-8, 8), seed 2, tiles 64 x 64
  ("Slicing, bounds and masking", "Promising whole tiles with @aligned":
  extents multiples of 4 but not of the tile).
* ``coalesce_4096`` -- [4096, 4096], U[0, 1), seed 3
  ("Memory Coalescing and Tensor Layout", "What it actually costs": 64 MB).
* ``aligned_4096`` -- [4096, 1000], U[-8, 8), seed 2, tiles 8 x 8: the ragged
  workload's bytes on whole tiles (a measurement companion, not a page workload).
* ``rowmax_8192``  -- [8192, 1000], U[-30, -1), seed 4, BC = 64
  ("Slicing, bounds and masking", "Reductions over a ragged tile": negative
  scores, last column tile ragged).
* ``gemm_4100`` / ``gemm_8192`` -- the gemm of "@aligned" on U[-1, 1)
  operands: [4100, 1000] x [1000, 4100] (K = 1000 from "Loops over a dynamic
  extent") and [8192, 8192] x [8192, 8192] on whole tiles.
"""
from __future__ import annotations

import numpy as np

POISON_F32 = np.float32(3.0e38)     # written into input ld-gaps: must never be read
CANARY_U32 = np.uint32(0xDEADBEEF)  # written past every output: must never change


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def uniform(shape, lo: float, hi: float, seed: int) -> np.ndarray:
    """float32 draws with lo <= x < hi exactly."""
    g = rng(seed)
    x = (lo + (hi - lo) * g.random(shape, dtype=np.float64)).astype(np.float32)
    top = np.nextafter(np.float32(hi), np.float32(lo))
    np.minimum(x, top, out=x)
    np.maximum(x, np.float32(lo), out=x)
    return x


def normal(shape, seed: int) -> np.ndarray:
    """float32 standard-normal draws."""
    return rng(seed).standard_normal(shape, dtype=np.float64).astype(np.float32)


def pad_rows(x: np.ndarray, ld: int, fill=POISON_F32) -> np.ndarray:
    """Lay an [M, N] array out with leading dimension ld >= N; the gap words
    hold ``fill``.  Returns the flat ``M*ld`` buffer."""
    M, N = x.shape
    if ld < N:
        raise ValueError("ld must be >= N")
    out = np.full((M, ld), fill, dtype=x.dtype)
    out[:, :N] = x
    return out.reshape(-1)


WORKLOADS = {
    "affine_1m": dict(kind="affine", n=1 << 20, dist=("uniform", -1.0, 1.0), seed=0),
    "scale_8192": dict(kind="scale2d", M=8192, N=8192, dist=("normal",), seed=1,
                       TM=32, TN=128, alpha=1.5),
    "ragged_4100": dict(kind="copy_scale", M=4100, N=1000, dist=("uniform", -8.0, 8.0), seed=2,
                        TM=64, TN=64, alpha=1.5),
    "coalesce_4096": dict(kind="sums", M=4096, N=4096, dist=("uniform", 0.0, 1.0), seed=3),
    # the ragged workload's aligned companion: nearly the same bytes on whole
    # 8 x 8 tiles, so that a ragged-minus-aligned gap is the cost of masking
    "aligned_4096": dict(kind="copy_scale", M=4096, N=1000, dist=("uniform", -8.0, 8.0), seed=2,
                         TM=8, TN=8, alpha=1.5),
    "rowmax_8192": dict(kind="rowmax", M=8192, N=1000, dist=("uniform", -30.0, -1.0), seed=4,
                        BC=64),
    # per-channel scale and bias ("Memory Coalescing and Tensor Layout", "NCHW versus
    # NHWC"): an activation-shaped [B, C, H, W] = [32, 256, 56, 56] fp32 tensor
    # (25.7M elements, 103 MB) read as [B*H*W, C] (channels last) or [B*C, H*W]
    "channel_nhwc": dict(kind="channel", M=32 * 56 * 56, N=256, C=256, layout=0,
                         dist=("normal",), seed=5, TM=32, TN=128),
    "channel_nchw": dict(kind="channel", M=32 * 256, N=56 * 56, C=256, layout=1,
                         dist=("normal",), seed=5, TM=32, TN=128),
    # the gemm of "@aligned" (A [M, K] B [K, N], alpha, beta): K = 1000 as in "Slicing,
    # bounds and masking", "Loops over a dynamic extent" (ragged against TILE_K = 32),
    # M = N = 4100 like the ragged 2-D workload; and a square whole-tile case
    "gemm_4100": dict(kind="gemm", M=4100, N=4100, K=1000, seeds=(7, 8, 9), alpha=1.5, beta=0.5,
                      TM=256, TN=256, TK=32),
    "gemm_8192": dict(kind="gemm", M=8192, N=8192, K=8192, seeds=(10, 11, 12), alpha=1.5, beta=0.5,
                      TM=256, TN=256, TK=32),
}


def gemm_inputs(name: str):
    """A [M, K], B [K, N] ~ U[-1, 1) and C [M, N] ~ U[-1, 1) of a gemm workload."""
    w = WORKLOADS[name]
    sa, sb, sc = w["seeds"]
    return (uniform((w["M"], w["K"]), -1.0, 1.0, sa), uniform((w["K"], w["N"]), -1.0, 1.0, sb),
            uniform((w["M"], w["N"]), -1.0, 1.0, sc))


def channel_params(C: int, seed: int = 6):
    """Per-channel scale in [0.5, 2) and bias ~ N(0, 1)."""
    return uniform((C,), 0.5, 2.0, seed), normal((C,), seed + 1)


def draw(dist, shape, seed: int) -> np.ndarray:
    if dist[0] == "uniform":
        return uniform(shape, dist[1], dist[2], seed)
    if dist[0] == "normal":
        return normal(shape, seed)
    raise ValueError("unknown distribution %r" % (dist,))


def workload_input(name: str) -> np.ndarray:
    """The seeded input tensor of a named workload (1-D for affine, else [M, N])."""
    w = WORKLOADS[name]
    shape = (w["n"],) if w["kind"] == "affine" else (w["M"], w["N"])
    return draw(w["dist"], shape, w["seed"])
