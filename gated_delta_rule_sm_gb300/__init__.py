"""GB300 (sm_103a) Kimi Delta Attention: chunkwise gated delta rule, forward and backward.

The computation lives in the CUDA library ``libkda_gb300.so`` behind the C
ABI in ``include/kda.h``; this package only marshals torch tensors to it
(``forward`` / ``backward``, the layer's short-convolution prologue
``short_conv`` / ``short_conv_backward`` and its gated output norm ``gated_norm`` /
``gated_norm_backward``) and draws seeded synthetic inputs
(``inputs``).  Importing the package does not load the library; the first
call does, and raises if it has not been built.
"""
from ._lib import (KdaError, backward, device_status, forward, gated_norm, gated_norm_backward, load,  # noqa: F401
                   saved_size, short_conv, short_conv_backward)

__all__ = ["forward", "backward", "saved_size", "short_conv", "short_conv_backward", "gated_norm",
           "gated_norm_backward", "load", "device_status", "KdaError"]
