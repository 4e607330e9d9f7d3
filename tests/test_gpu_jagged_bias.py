"""GPU parity of the general jagged bias (kind 2: one Lq x Lk bf16 block per sequence and
head, rows padded to a multiple of 8 elements): forward and backward against the float64
oracle on the same seeded inputs, with the tolerances of the other parity tests."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle.jfa_oracle as orc
from jagged_attention_recsys_jfa_gb300 import jfa_check_status, jfa_forward
from jagged_attention_recsys_jfa_gb300.inputs import CONFIGS, JaggedConfig, make_batch
from parity_utils import GRAD_RTOL, compare_grads, compare_out_lse, gpu_run, oracle_full, rel_frob

pytestmark = pytest.mark.gpu

CASES = {
    # (heads, d, q lengths, kv lengths or None, causal)
    "self_d128": (2, 128, [300, 5, 129, 1, 260], None, False),
    "causal_d64": (3, 64, [1100, 300, 129, 7], None, True),
    # fused short-query pass only (Lq <= 128), keys up to several tiles
    "cross_fused_d128": (2, 128, [33, 1, 100, 128, 64], [500, 2, 129, 900, 1], False),
    # both passes, empty sequences, unequal lengths, causal
    "mixed_causal_d128": (2, 128, [0, 5, 140, 7, 400, 90], [3, 0, 140, 9, 260, 300], True),
    # last tiles reaching past the tensors' ends (tail maps)
    "tails_causal_d64": (3, 64, [129, 3, 0], [131, 0, 2], True),
    # both sides of the fused pass's half-width limit (64 queries), causal, d = 64
    "half_width_causal_d64": (3, 64, [64, 65, 20, 1], [64, 200, 300, 70], True),
}


def _cfg(name, H, d, n, causal):
    return JaggedConfig(name, n, H, d, ("uniform", 1, 1), causal=causal, general_bias=True)


@pytest.mark.parametrize("name", list(CASES))
def test_jagged_bias_parity(name):
    H, d, lq, lk, causal = CASES[name]
    batch = make_batch(_cfg(name, H, d, len(lq), causal), device="cuda", q_lengths=lq, kv_lengths=lk)
    res = gpu_run(batch)
    ref = oracle_full(batch)
    # hand-made edge shapes (1-key rows, empty sequences): the bf16 rounding allowance
    # applies to their |oracle| >= 2 elements only, and is reported when used
    compare_out_lse(res["out"], res["lse"], ref["out"], ref["lse"], name, with_rounding=True)
    compare_grads(res, ref, name)


def test_jagged_bias_bad_block_offsets_reported():
    batch = make_batch(_cfg("bad", 2, 64, 3, False), device="cuda", q_lengths=[40, 7, 130])
    bad = batch.jbias_offsets.clone()
    bad[1] += 8   # the first block claims one row more than Lq x round_up(Lk, 8)
    _, _, ws = jfa_forward(batch.q, batch.k, batch.v, batch.q_offsets, batch.kv_offsets, None, 0,
                           batch.cfg.scale, False, jagged_bias=(batch.jbias, bad))
    assert jfa_check_status(ws) == 5   # JFA_ERR_BAD_OFFSETS
    res = gpu_run(batch, backward=False)   # still usable, and right with the true offsets
    ref = oracle_full(batch, backward=False)
    compare_out_lse(res["out"], res["lse"], ref["out"], ref["lse"], "after bad offsets", with_rounding=True)


def test_jagged_bias_autograd():
    from jagged_attention_recsys_jfa_gb300 import jagged_attention
    batch = make_batch(_cfg("ag", 2, 64, 4, True), device="cuda", q_lengths=[200, 3, 129, 60])
    q = batch.q.clone().requires_grad_(True)
    k = batch.k.clone().requires_grad_(True)
    v = batch.v.clone().requires_grad_(True)
    out = jagged_attention(q, k, v, batch.q_offsets, batch.kv_offsets, None, 0, batch.cfg.scale, True,
                           jagged_bias=(batch.jbias, batch.jbias_offsets))
    out.backward(batch.dout)
    ref = oracle_full(batch)
    compare_out_lse(out, ref["lse"], ref["out"], ref["lse"], "autograd", with_rounding=True)
    compare_grads({"dq": q.grad, "dk": k.grad, "dv": v.grad}, ref, "autograd")


def test_jagged_bias_full_size_sampled():
    """The full jagged_bias_causal workload in the launch configuration the benchmark
    times; the oracle recomputes sampled (sequence, head) pairs one by one."""
    batch = make_batch(CONFIGS["jagged_bias_causal"], device="cuda")
    res = gpu_run(batch)
    cfg = batch.cfg
    rng = np.random.default_rng(0)
    qo = batch.q_offsets.cpu().numpy()
    lq = batch.q_lengths.numpy()
    picks = {int(np.argmax(lq)), int(np.argmin(lq))} | {int(x) for x in rng.integers(lq.size, size=4)}
    for b in sorted(picks):
        h = int(rng.integers(cfg.heads))
        o, lse, dq, dk, dv = orc.sequence_reference(
            b, h, batch.q, batch.k, batch.v, batch.q_offsets, batch.kv_offsets, cfg.scale, cfg.causal,
            dout=batch.dout, jagged_bias=(batch.jbias, batch.jbias_offsets))
        sl = slice(qo[b], qo[b + 1])
        compare_out_lse(res["out"][sl, h], res["lse"][h, sl], o, lse, f"b={b} h={h}")
        for gname, g, r in (("dq", res["dq"][sl, h], dq), ("dk", res["dk"][sl, h], dk), ("dv", res["dv"][sl, h], dv)):
            e = rel_frob(g, r)
            assert e <= GRAD_RTOL, f"b={b} h={h} {gname} rel err {e:.3g}"


@pytest.mark.parametrize("name", ["causal_d64", "cross_fused_d128", "mixed_causal_d128"])
def test_jagged_bias_gradient(name):
    """The general bias's gradient (dS of every block element, 0 where the causal mask hides
    the pair and on the row padding) against the oracle, over the whole [H, plane] array."""
    from jagged_attention_recsys_jfa_gb300 import jfa_backward
    H, d, lq, lk, causal = CASES[name]
    batch = make_batch(_cfg(name, H, d, len(lq), causal), device="cuda", q_lengths=lq, kv_lengths=lk)
    cfg = batch.cfg
    jb = (batch.jbias, batch.jbias_offsets)
    out, lse, ws = jfa_forward(batch.q, batch.k, batch.v, batch.q_offsets, batch.kv_offsets, None, 0, cfg.scale,
                               cfg.causal, jagged_bias=jb)
    g = torch.full_like(batch.jbias, float("nan"))   # every element must be written
    dq, dk, dv, ws2 = jfa_backward(batch.dout, batch.q, batch.k, batch.v, out, lse, batch.q_offsets,
                                   batch.kv_offsets, None, 0, cfg.scale, cfg.causal, jagged_bias=jb,
                                   jagged_bias_grad=g)
    assert jfa_check_status(ws) == 0 and jfa_check_status(ws2) == 0
    torch.cuda.synchronize()
    assert torch.isfinite(g.float()).all(), "unwritten or non-finite gradient elements"
    ref = orc.jagged_general_bias_grad(batch.dout, batch.q, batch.k, batch.v, batch.q_offsets, batch.kv_offsets,
                                       cfg.scale, cfg.causal, jb)
    e = rel_frob(g, ref)
    assert e <= GRAD_RTOL, f"{name}: general bias gradient relative error {e:.3g}"
    # the other gradients are unchanged by asking for it
    compare_grads({"dq": dq, "dk": dk, "dv": dv}, oracle_full(batch), name)


def test_jagged_bias_gradient_autograd():
    from jagged_attention_recsys_jfa_gb300 import jagged_attention
    batch = make_batch(_cfg("ag2", 2, 128, 3, False), device="cuda", q_lengths=[200, 7, 129], kv_lengths=[150, 300, 9])
    values = batch.jbias.clone().requires_grad_(True)
    out = jagged_attention(batch.q, batch.k, batch.v, batch.q_offsets, batch.kv_offsets, None, 0, batch.cfg.scale,
                           False, jagged_bias=(values, batch.jbias_offsets))
    out.backward(batch.dout)
    ref = orc.jagged_general_bias_grad(batch.dout, batch.q, batch.k, batch.v, batch.q_offsets, batch.kv_offsets,
                                       batch.cfg.scale, False, (batch.jbias, batch.jbias_offsets))
    e = rel_frob(values.grad, ref)
    assert e <= GRAD_RTOL, f"autograd general bias gradient relative error {e:.3g}"
