"""Benchmark of the tiled fp32 maps on one GB300 (filled in with the kernels)."""


def gbps(nbytes: int, seconds: float) -> float:
    """Bandwidth in GB/s with GB = 1e9 bytes (the pages' convention: their
    "64 MB" read in 111.6 us is quoted as 601 GB/s, i.e. 2^26 bytes / 1e9)."""
    return nbytes / seconds / 1e9
