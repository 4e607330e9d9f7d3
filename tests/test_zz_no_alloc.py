"""jfa_forward_noalloc, the forward for callers that cannot allocate device memory
(inference-runtime plugins, services on a fixed memory arena): called through the C
ABI, it must give the workspace forward's results, on two calls in a row that reuse
its fixed scratch array.  Kept in a file of its own that pytest collects last."""
import ctypes

import pytest
import torch

from jagged_attention_recsys_jfa_gb300 import jfa_check_status, jfa_forward, load_library
from jagged_attention_recsys_jfa_gb300.inputs import CONFIGS, make_batch
from jagged_attention_recsys_jfa_gb300.jfa import _Bias

pytestmark = pytest.mark.gpu


def _noalloc(lib, batch, out, lse):
    cfg = batch.cfg
    bias = _Bias(1, batch.bias.data_ptr(), batch.bias.shape[1], cfg.bias_center) if batch.bias is not None else None
    return lib.jfa_forward_noalloc(batch.q.data_ptr(), batch.k.data_ptr(), batch.v.data_ptr(),
                                   batch.q_offsets.data_ptr(), batch.kv_offsets.data_ptr(),
                                   batch.q_offsets.numel() - 1, cfg.heads, cfg.head_dim, batch.q.shape[0],
                                   batch.k.shape[0], ctypes.byref(bias) if bias is not None else None, cfg.scale,
                                   1 if cfg.causal else 0, out.data_ptr(), lse.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)


def test_noalloc_forward_matches_workspace_forward_twice():
    lib = load_library()
    import dataclasses
    cases = [dataclasses.replace(CONFIGS["gem_self"], batch=24),
             dataclasses.replace(CONFIGS["biased_causal"], batch=16)]
    for call, cfg in enumerate(cases):
        batch = make_batch(cfg, device="cuda", seed=call)
        center = cfg.bias_center if batch.bias is not None else 0
        ref_out, ref_lse, ws = jfa_forward(batch.q, batch.k, batch.v, batch.q_offsets, batch.kv_offsets,
                                           batch.bias, center, cfg.scale, cfg.causal)
        assert jfa_check_status(ws) == 0
        out = torch.full_like(batch.q, float("nan"))
        lse = torch.full((cfg.heads, batch.q.shape[0]), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(lib, batch, out, lse) == 0, f"call {call}"
        torch.cuda.synchronize()
        # the same kernels on the same inputs: the results must be bit-identical (a stale
        # scratch would show here even if it stayed inside the oracle's tolerances)
        assert torch.equal(out, ref_out), f"call {call}: out differs from the workspace forward"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs from the workspace forward"


def test_noalloc_rejects_sizes_beyond_its_scratch():
    lib = load_library()
    batch = make_batch(CONFIGS["tiny"], device="cuda")
    out = torch.empty_like(batch.q)
    lse = torch.empty((2, batch.q.shape[0]), dtype=torch.float32, device="cuda")
    # a batch count whose per-sequence tensor maps alone need more than 8 MiB
    st = lib.jfa_forward_noalloc(batch.q.data_ptr(), batch.k.data_ptr(), batch.v.data_ptr(),
                                 batch.q_offsets.data_ptr(), batch.kv_offsets.data_ptr(), 1 << 20, 2, 64,
                                 batch.q.shape[0], batch.k.shape[0], None, 0.125, 0, out.data_ptr(),
                                 lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 3   # JFA_ERR_WORKSPACE, nothing enqueued
