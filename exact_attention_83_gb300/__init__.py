"""Exact scaled-dot-product attention (FlashAttention-2 form) for GB300.

The compute path is libfa (hand-written CUDA for sm_103a behind the C ABI in
include/fa.h); `fa` is its thin Python binding.
"""

from .fa import (FAError, attention, attention_bwd, attention_fwd, bwd, bwd_preprocess,
                 device_status, fwd, load_library, set_path, set_wait_timeout_ns)

__all__ = ["FAError", "attention", "attention_bwd", "attention_fwd", "bwd", "bwd_preprocess",
           "device_status", "fwd", "load_library", "set_path", "set_wait_timeout_ns"]
