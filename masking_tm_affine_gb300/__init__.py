"""GB300-native masked/aligned tiled fp32 maps.

The compute path is ``libtm.so`` (hand-written sm_103a CUDA behind a C ABI,
declared in ``include/tm.h``); ``masking_tm_affine_gb300.tm`` is its thin
ctypes binding.  Importing this package does not load the library; the first
call into ``tm`` does, and raises if the library was not built.
"""
__all__ = ["tm", "synth"]
