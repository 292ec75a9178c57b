"""CPU oracle for the FLUX.3 Image Klein transformer block -- TEST INFRASTRUCTURE.

Only the tests, the smoke check and the benchmark's CPU-baseline leg import this
package.  The product path (the CUDA library and its Python binding) never imports it
and shares no code with it.
"""
from .flux3_block import (  # noqa: F401
    round_bf16, layer_norm, segment_ids, modulate, ada_ln, rope_angles, rope_rotate,
    rms_norm, attention, attention_rows, swiglu, Weights, BlockOut, block_forward, final_layer,
    dit_forward, euler_step, block_forward_rows, block_keys_values,
)
