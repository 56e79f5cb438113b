"""libfattn: FlashAttention-style forward pass (tiled online softmax) for GB300.

The compute path is the CUDA library ``libfattn.so`` built from ``csrc/`` for
sm_103a; this package only marshals arguments to its C ABI (``fattn.py``).
Importing the package does not load the library: the first call does, and it
raises if the library has not been built (there is no CPU fallback).
"""
__all__ = ["attn_fwd", "attn_fwd_fp16", "attn_bwd", "attn_fwd_host", "attn_fwd_simt", "attn_fwd_split", "split_count",
           "split_workspace_size", "softmax_rows", "row_sum", "FattnError", "device_status",
           "library_path", "version"]


def __getattr__(name):
    if name in __all__:
        from . import fattn
        return getattr(fattn, name)
    raise AttributeError(name)
