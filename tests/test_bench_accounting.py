"""The benchmark's work accounting (host logic, CPU): visited pairs against brute force,
and the flops / bytes split across the kernels that share the work."""
import importlib.util
import os
import sys

import numpy as np
import pytest
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    b = importlib.util.module_from_spec(spec)
    argv, sys.argv = sys.argv, ["bench.py"]
    try:
        spec.loader.exec_module(b)
    finally:
        sys.argv = argv
    return b


def _brute_pairs(lq, lk, causal):
    n = 0
    for a, c in zip(lq, lk):
        for i in range(a):
            for j in range(c):
                n += 1 if (not causal or j <= i + (c - a)) else 0
    return n


@pytest.mark.parametrize("causal", [False, True])
def test_valid_pairs_brute_force(causal):
    b = _bench()
    rng = np.random.default_rng(3)
    for _ in range(50):
        B = int(rng.integers(1, 6))
        lq = rng.integers(0, 40, B).tolist()
        lk = rng.integers(0, 40, B).tolist()
        assert b.valid_pairs(lq, lk, causal) == _brute_pairs(lq, lk, causal), (lq, lk)


def test_flops_split_adds_up():
    b = _bench()
    from jagged_attention_recsys_jfa_gb300.inputs import CONFIGS, make_batch
    for name in ("tiny", "biased_causal"):
        batch = make_batch(CONFIGS[name], device="cpu")
        f = b.workload_flops(batch, nsp_rows=1024)
        dH = batch.cfg.head_dim * batch.cfg.heads
        assert f["fwd"] == 4.0 * dH * f["pairs"]
        assert f["bwd"] == 10.0 * dH * f["pairs"]
        # the split passes, the fused pass and the non-sequence-parallel pass cover every
        # visited pair once
        assert f["dkdv"] / 8 + f["fused"] / 10 + f["nsp"] / 10 == pytest.approx(f["pairs"] * dH)
        assert f["dq"] * 4 == pytest.approx(f["dkdv"])
        lq = np.asarray(batch.q_lengths)
        assert (f["nsp"] > 0) == bool(((lq > 128) & (lq <= 1024)).any())
        assert (f["dkdv"] > 0) == bool((lq > 1024).any())


def test_general_bias_bytes_counted_once_per_pass():
    b = _bench()
    import dataclasses
    from jagged_attention_recsys_jfa_gb300.inputs import CONFIGS, make_batch
    plain = make_batch(dataclasses.replace(CONFIGS["jagged_bias_causal"], batch=6, general_bias=False), device="cpu")
    jb = make_batch(dataclasses.replace(CONFIGS["jagged_bias_causal"], batch=6), device="cpu")
    w0, w1 = b.workload_bytes(plain, nsp_rows=1024), b.workload_bytes(jb, nsp_rows=1024)
    H = jb.cfg.heads
    lq, lk = jb.q_lengths.numpy(), jb.kv_lengths.numpy()
    # the visited pairs' elements only (causal: the lower triangle; never the row padding)
    blocks = np.array([2.0 * H * _brute_pairs([a], [c], True) for a, c in zip(lq, lk)])
    assert blocks.sum() < 2.0 * H * (lq * ((lk + 7) // 8 * 8)).sum() * 0.6
    long_ = lq > 1024
    nsp = (lq > 128) & ~long_
    assert w1["forward"] - w0["forward"] == pytest.approx(blocks.sum())
    assert w1["bwd_dkdv"] - w0["bwd_dkdv"] == pytest.approx(blocks[long_].sum())
    assert w1["bwd_dq"] - w0["bwd_dq"] == pytest.approx(blocks[long_].sum())
    assert w1["bwd_nsp"] - w0["bwd_nsp"] == pytest.approx(blocks[nsp].sum())
    assert w1["bwd_fused"] - w0["bwd_fused"] == pytest.approx(blocks[lq <= 128].sum())
    assert jb.jbias.numel() == (lq * ((lk + 7) // 8 * 8)).sum() * H


def test_clock_report_uses_samples_inside_the_timed_region():
    """The clocks object summarises the nvidia-smi samples whose timestamps fall inside the
    timed region, keeps throttle reasons seen there, and says when none fell inside."""
    import datetime

    b = _bench()
    t = 1_800_000_000.0

    def line(dt, mhz, power_cap="Not Active", uuid="GPU-aa11"):
        ts = datetime.datetime.fromtimestamp(t + dt).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        return (f"{ts}, 0, {uuid}, {mhz} MHz, 2070 MHz, 900.00 W, 0x0, Not Active, Not Active, "
                f"Not Active, {power_cap}")

    lines = [line(-0.30, 900), line(0.011, 2070), line(0.022, 2040, "Active"), line(0.033, 2055),
             line(0.25, 1200), line(0.02, 1000, uuid="GPU-other")]
    rep = b.ClockSampler.parse(lines, "GPU-aa11", t, t + 0.036)
    assert rep["samples"] == 3 and rep["samples_total"] == 5
    assert rep["sm_mhz"] == 2055.0 and rep["sm_max_mhz"] == 2070.0
    assert rep["reasons"] == ["sw_power_cap"] and "note" not in rep
    none = b.ClockSampler.parse(lines, "GPU-aa11", t + 10, t + 11)
    assert none["samples"] == 0 and "note" in none
    assert b.ClockSampler.parse([], "GPU-aa11", t, t + 1)["reasons"] == ["no samples"]
