"""GB300 (sm_103a) exact attention: forward (plain and with an additive mask),
backward, and an FP8 forward.

The compute runs in ``libattn_gb300.so`` (hand-written CUDA behind the C ABI
of ``include/attn.h``); this package only marshals torch tensors into that
call.  Importing the package does not load the library; the first call does,
and raises if the library has not been built.
"""
from .binding import (AttnError, attn_bwd, attn_fp8_quantize, attn_fwd, attn_fwd_fp8,  # noqa: F401
                      attn_fwd_host, attn_fwd_plan, attn_fwd_status, attn_set_debug, attn_shutdown,
                      attn_strerror, attn_version, library_path, load_library)

__all__ = ["AttnError", "attn_bwd", "attn_fp8_quantize", "attn_fwd", "attn_fwd_fp8", "attn_fwd_host",
           "attn_fwd_plan", "attn_fwd_status", "attn_set_debug", "attn_shutdown", "attn_strerror",
           "attn_version", "library_path", "load_library"]
