"""Exact, IO-aware attention (forward and backward) for NVIDIA GB300.

The computation lives in libflashattn.so (hand-written sm_103a CUDA behind the
C ABI of include/flash_attn.h, plus the standard materialising attention of
include/standard_attn.h that serves as the IO baseline); this package holds
its ctypes binding, the in-place build script, the seeded synthetic inputs
and FLOP accounting.
Importing the package does not load the library; the first call does, and
raises if it is missing.
"""
from ._lib import (FlashAttnError, attention_bwd, attention_fwd, device_error, fa_options,
                   flash_attn_bwd, flash_attn_bwd_ex, flash_attn_bwd_noalloc, flash_attn_fwd_ex, flash_attn_bwd_workspace_size, flash_attn_fwd,
                   flash_attn_get_device_error, flash_attn_set_profile_events,
                   flash_attn_status_string, flash_attn_tile_map, flash_attn_version, load,
                   profile_next_call, standard_attention_bwd, standard_attention_fwd, standard_attn_bwd,
                   standard_attn_fwd, standard_attn_workspace_size, tile_map)

__all__ = [
    "FlashAttnError", "attention_bwd", "attention_fwd", "device_error", "fa_options", "flash_attn_bwd",
    "flash_attn_bwd_ex", "flash_attn_bwd_noalloc", "flash_attn_fwd_ex",
    "flash_attn_bwd_workspace_size", "flash_attn_fwd", "flash_attn_get_device_error",
    "flash_attn_set_profile_events", "flash_attn_status_string", "flash_attn_tile_map",
    "flash_attn_version", "load", "profile_next_call", "standard_attention_bwd", "standard_attention_fwd",
    "standard_attn_bwd", "standard_attn_fwd", "standard_attn_workspace_size", "tile_map",
]
