"""CPU float64 oracle for exact attention.  TEST INFRASTRUCTURE ONLY.

Imported by ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU
baseline / reference arm, and by nothing else.  Parity: pinned (see
``tests/test_oracle_pins.py``); every function here has at least one pin that
does not re-use its own formula.
"""
from .attention import (  # noqa: F401
    LN2,
    backward,
    backward_gqa,
    backward_window,
    decode,
    flops_backward,
    flops_forward,
    forward,
    forward_fp8_reference,
    forward_gqa,
    forward_window,
    hadamard_matrix,
    dequantize_e4m3,
    dequantize_e4m3_blocks,
    quantize_e4m3_blocks_reference,
    quantize_e4m3_reference,
    rotate_rows,
    head_backward,
    head_forward,
    head_forward_online,
    online_softmax_vector,
    row_dot,
    scores,
    softmax_stats,
)
