"""fp64 CPU oracle (test infrastructure; see ``encoder_fp64``).

Only tests, the smoke check and the benchmark's CPU-baseline leg use this
package.  It shares no code with the CUDA library and imports nothing from it.
"""
from .encoder_fp64 import (  # noqa: F401
    LN_EPS, allowed_keys, encoder_forward, encoder_layer,
    first_row_closed_form, gelu_erf, layer_norm,
    masked_attention, merge_heads, qkv_projection, split_heads,
)
