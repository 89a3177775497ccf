"""CPU float64 oracle for exact attention (test infrastructure only).

Only the tests, the package smoke check and the bench's CPU-baseline leg import
this package. The library never does.
"""
from .attention import (allowed_mask, head_forward, head_backward, head_rows, attention_fwd,
                        attention_fwd_bwd, tile_states, SKIP, FULL, PARTIAL, TILE)
from .loops import loop_attention_fwd_bwd
from .dropout import (attention_fwd_bwd_dropout, keep_mask, philox4x32_10, philox4x32_10_scalar,
                      random_bytes, threshold)
