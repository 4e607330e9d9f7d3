"""Jagged Flash Attention for GB300 (sm_103a): exact softmax attention, forward and
backward, on jagged (values + int64 offsets) sequences, through a C-ABI library of
hand-written tcgen05/TMA kernels.  See include/jfa.h for the ABI."""
from .jfa import (  # noqa: F401
    EXPORTED_SYMBOLS,
    JaggedAttention,
    JfaError,
    jagged_attention,
    jfa_backward,
    jfa_check_status,
    jfa_forward,
    jfa_last_launch_count,
    jfa_nsp_max_tiles,
    jfa_set_nsp_max_tiles,
    jfa_timing_enable,
    jfa_timing_read,
    jfa_trace_configure,
    decode_trace,
    KERNEL_KINDS,
    library_path,
    load_library,
    status_string,
    workspace_size,
)
