"""Failure detection and tracing on the GPU.  The failure is made safely: a bounded
wait on a barrier nothing signals must run out, be reported as JFA_ERR_TIMEOUT, and
leave the context usable (no trap, no fault, no hang)."""
import ctypes

import numpy as np
import pytest
import torch

from jagged_attention_recsys_jfa_gb300 import decode_trace, jfa_check_status, jfa_trace_configure, load_library
from jagged_attention_recsys_jfa_gb300.inputs import CONFIGS, make_batch
from parity_utils import compare_out_lse, gpu_run, oracle_full

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    lib = load_library()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.jfa_selftest_wait_timeout(ws.data_ptr(), 20_000_000, stream) == 0   # 20 ms limit
    assert jfa_check_status(ws) == 6          # JFA_ERR_TIMEOUT
    assert jfa_check_status(ws) == 0          # read-and-clear
    # out-of-range limits are rejected on the host
    assert lib.jfa_selftest_wait_timeout(ws.data_ptr(), 0, stream) == 1
    # the context is still healthy: a full forward/backward still matches the oracle
    batch = make_batch(CONFIGS["tiny"], device="cuda")
    res = gpu_run(batch)
    ref = oracle_full(batch)
    compare_out_lse(res["out"], res["lse"], ref["out"], ref["lse"], "after timeout")


@pytest.mark.parametrize("kind", ["forward", "bwd_dkdv", "bwd_dq", "bwd_fused", "bwd_nsp"])
def test_trace_records_ordered_events(kind):
    # sequences of more than 8 query tiles (split backward passes), of 3 (non-sequence-
    # parallel pass) and of one (fused).  The first CTA records; CTAs claim items as they free
    # up and each claims its first two at once, so every list holds more than two items per
    # SM to be sure the first CTA works
    lq = [1100, 300, 40] * 160
    batch = make_batch(CONFIGS["tiny"], device="cuda", q_lengths=lq, kv_lengths=[1100, 300, 260] * 160)
    buf = torch.zeros(5 * 1024, dtype=torch.int64, device="cuda")
    from jagged_attention_recsys_jfa_gb300 import jfa_set_nsp_max_tiles
    prev = jfa_set_nsp_max_tiles(8 if kind == "bwd_nsp" else 0)  # the 3-tile sequences take that pass
    jfa_trace_configure(buf, kind)
    try:
        gpu_run(batch)
    finally:
        jfa_trace_configure(None)
        jfa_set_nsp_max_tiles(prev)
    roles = decode_trace(buf)
    assert len(roles[1]) > 0, "MMA issuer recorded nothing"
    for r, events in enumerate(roles):
        clocks = [c for c, _ in events]
        assert clocks == sorted(clocks), f"role {r} events out of order"
