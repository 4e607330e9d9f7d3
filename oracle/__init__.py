"""CPU float64 oracle for Jagged Flash Attention.

Test infrastructure: imported only by the tests, the package smoke check and the
benchmark's CPU-baseline leg.  The library never routes through it.
"""
from .jfa_oracle import (  # noqa: F401
    causal_visible,
    jagged_bias_grad,
    jagged_general_bias_grad,
    jagged_backward,
    jagged_forward,
    jagged_bias_block,
    padded_dense_forward,
    relpos_bias,
    sequence_backward,
    sequence_bias_grad,
    sequence_score_grad,
    sequence_forward,
    sequence_reference,
    softmax_rows,
    tiled_subtraction_forward,
    to_f64,
)
