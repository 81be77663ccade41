"""Fused exact attention (FlashAttention-style forward and backward) for GB300.

The computation lives in the CUDA library libattn_gb300.so (C interface in
include/attn.h); this package is its thin Python binding.  There is no CPU or
PyTorch fallback: calls fail if the library is not built.
"""

from ._abi import AttnError  # noqa: F401
from .api import (  # noqa: F401
    attention_bwd,
    attention_decode,
    attention_fwd,
    check,
    make_params,
    workspace,
    workspace_size,
)
