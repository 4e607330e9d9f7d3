"""GPU parity of the non-sequence-parallel backward pass ("Jagged Flash Attention (JFA)",
"Four generations" item 2, the reading in which one CTA owns a sequence and head): with
every sequence of 2 .. 16 query tiles routed to it, dq, dk and dv (and both bias gradients)
against the float64 oracle on the workload shapes and edge sets, bit-reproducible across
calls, and the same as the split passes' results to the rounding of the dQ sums."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle.jfa_oracle as orc
from jagged_attention_recsys_jfa_gb300 import jfa_backward, jfa_check_status, jfa_forward, jfa_set_nsp_max_tiles
from jagged_attention_recsys_jfa_gb300.inputs import CONFIGS, JaggedConfig, make_batch
from parity_utils import GRAD_RTOL, compare_grads, compare_out_lse, gpu_run, oracle_full, rel_frob

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def nsp_on():
    prev = jfa_set_nsp_max_tiles(16)
    yield
    jfa_set_nsp_max_tiles(prev)


def small(name, batch, **kw):
    return dataclasses.replace(CONFIGS[name], batch=batch, **kw)


CASES = {
    "gem_self_b12": small("gem_self", 12),
    "biased_causal_b8": small("biased_causal", 8),
    "longtail_causal_b8": small("longtail_causal", 8, lengths=("lognormal", 300.0, 1.2, 16, 1500)),
    "jagged_bias_causal_b6": small("jagged_bias_causal", 6),
}


@pytest.mark.parametrize("name", list(CASES))
def test_nsp_parity_elementwise(name):
    batch = make_batch(CASES[name], device="cuda")
    res = gpu_run(batch)
    ref = oracle_full(batch)
    compare_out_lse(res["out"], res["lse"], ref["out"], ref["lse"], name)
    compare_grads(res, ref, name)


EDGE = {
    # (heads, d, q lengths, kv lengths or None, causal, relative-position bias)
    "tile_boundaries_d128": (2, 128, [129, 255, 256, 257, 1, 128], None, False, False),
    "causal_lq_gt_lk_d64": (2, 64, [300, 640, 129], [40, 1, 128], True, False),
    "causal_lq_lt_lk_d128": (2, 128, [140, 300, 129], [300, 1000, 129], True, True),
    "no_keys_d64": (2, 64, [300, 129, 5], [0, 0, 7], False, False),
    "sixteen_tiles_d64": (1, 64, [2048, 1500], None, True, True),
    "tails_d128": (3, 128, [131, 257], [129, 300], False, False),
}


@pytest.mark.parametrize("name", list(EDGE))
def test_nsp_parity_edges(name):
    H, d, lq, lk, causal, bias = EDGE[name]
    cfg = JaggedConfig(name, len(lq), H, d, ("uniform", 1, 1), causal=causal,
                       bias_buckets=4096 if bias else 0, bias_center=2048 if bias else 0)
    batch = make_batch(cfg, device="cuda", q_lengths=lq, kv_lengths=lk)
    res = gpu_run(batch)
    ref = oracle_full(batch)
    compare_out_lse(res["out"], res["lse"], ref["out"], ref["lse"], name, with_rounding=True)
    compare_grads(res, ref, name)


def test_nsp_bias_gradients():
    """The relative-position table's gradient (fp32 reductions) and the general bias's
    gradient (dS, written by the pass) against the oracle."""
    cfg = JaggedConfig("tb", 4, 2, 64, ("uniform", 1, 1), causal=True, bias_buckets=4096, bias_center=2048)
    batch = make_batch(cfg, device="cuda", q_lengths=[700, 300, 129, 40])
    out, lse, ws = jfa_forward(batch.q, batch.k, batch.v, batch.q_offsets, batch.kv_offsets, batch.bias, 2048,
                               cfg.scale, True)
    g = torch.full_like(batch.bias, float("nan"))
    jfa_backward(batch.dout, batch.q, batch.k, batch.v, out, lse, batch.q_offsets, batch.kv_offsets, batch.bias, 2048,
                 cfg.scale, True, bias_grad=g)
    torch.cuda.synchronize()
    ref = orc.jagged_bias_grad(batch.dout, batch.q, batch.k, batch.v, batch.q_offsets, batch.kv_offsets, cfg.scale,
                               True, batch.bias, 2048)
    assert rel_frob(g, ref) <= GRAD_RTOL
    cfg2 = JaggedConfig("jb", 3, 2, 128, ("uniform", 1, 1), causal=False, general_bias=True)
    b2 = make_batch(cfg2, device="cuda", q_lengths=[300, 129, 9], kv_lengths=[200, 400, 129])
    jb = (b2.jbias, b2.jbias_offsets)
    out, lse, _ = jfa_forward(b2.q, b2.k, b2.v, b2.q_offsets, b2.kv_offsets, None, 0, cfg2.scale, False, jagged_bias=jb)
    gj = torch.full_like(b2.jbias, float("nan"))
    jfa_backward(b2.dout, b2.q, b2.k, b2.v, out, lse, b2.q_offsets, b2.kv_offsets, None, 0, cfg2.scale, False,
                 jagged_bias=jb, jagged_bias_grad=gj)
    torch.cuda.synchronize()
    assert torch.isfinite(gj.float()).all()
    refj = orc.jagged_general_bias_grad(b2.dout, b2.q, b2.k, b2.v, b2.q_offsets, b2.kv_offsets, cfg2.scale, False, jb)
    assert rel_frob(gj, refj) <= GRAD_RTOL


def test_nsp_deterministic_and_matches_split_path():
    """Each dQ row has one writer adding the key tiles in order: bit-identical across calls.
    The split passes sum dQ in TMEM instead, so the two paths agree to rounding."""
    batch = make_batch(small("biased_causal", 6), device="cuda")
    a = gpu_run(batch)
    b = gpu_run(batch)
    for key in a:
        assert torch.equal(a[key], b[key]), key
    jfa_set_nsp_max_tiles(0)
    c = gpu_run(batch)
    assert torch.equal(a["out"], c["out"]) and torch.equal(a["lse"], c["lse"])
    for key in ("dq", "dk", "dv"):
        e = rel_frob(a[key], c[key].double().cpu().numpy())
        assert e <= 1e-2, f"{key}: paths differ by {e:.3g}"


def test_nsp_full_size_gem_self_sampled():
    """The full GEM-like workload (every sequence of 2 .. 8 query tiles in this pass) in the
    benchmark's launch configuration; the oracle recomputes sampled (sequence, head) pairs."""
    batch = make_batch(CONFIGS["gem_self"], device="cuda")
    res = gpu_run(batch)
    cfg = batch.cfg
    rng = np.random.default_rng(0)
    qo = batch.q_offsets.cpu().numpy()
    lq = batch.q_lengths.numpy()
    picks = {int(np.argmax(lq))} | {int(x) for x in rng.choice(np.nonzero(lq > 128)[0], 4, replace=False)}
    for b in sorted(picks):
        h = int(rng.integers(cfg.heads))
        o, lse, dq, dk, dv = orc.sequence_reference(b, h, batch.q, batch.k, batch.v, batch.q_offsets,
                                                    batch.kv_offsets, cfg.scale, cfg.causal, dout=batch.dout)
        sl = slice(qo[b], qo[b + 1])
        for gname, g, r in (("dq", res["dq"][sl, h], dq), ("dk", res["dk"][sl, h], dk), ("dv", res["dv"][sl, h], dv)):
            e = rel_frob(g, r)
            assert e <= GRAD_RTOL, f"b={b} h={h} {gname} rel err {e:.3g}"
    for gname in ("dq", "dk", "dv"):
        assert torch.isfinite(res[gname].float()).all(), gname
