"""libfattn: FlashAttention-style forward pass (tiled online softmax) for GB300.

The compute path is the CUDA library ``libfattn.so`` built from ``csrc/`` for
sm_103a; this package only marshals arguments to its C ABI.  Importing the
package does not load the library: the first call does, and it raises if the
library has not been built.
"""
__all__ = ["attn_fwd", "attn_fwd_host", "FattnError", "inputs"]


def __getattr__(name):
    if name in ("attn_fwd", "attn_fwd_host", "FattnError", "device_status", "library_path"):
        from . import fattn
        return getattr(fattn, name)
    raise AttributeError(name)
