#!/usr/bin/env python
"""Jagged Flash Attention benchmark on GB300.

One step = the whole hot path on one synthetic jagged batch: planner + forward, then
planner + preprocess + the backward passes (jfa_forward + jfa_backward): sequences of one
query tile in the fused pass, of 2 .. 8 in the non-sequence-parallel pass, longer ones in
the split dK/dV and dQ passes.
Metric: valid-token TFLOPS (bf16), forward+backward, counting only the (query, key)
pairs the attention visits: fwd 4*d*H*P, bwd 10*d*H*P flops, P = sum_b Lq_b*Lk_b
(causal: the visible pairs).  Inputs are resident in HBM for `value`; `e2e` times
the same step through the public call with pinned host buffers copied in and the
results copied out every step (consecutive steps overlapped: the next step's inputs
stream in while this one computes and its results stream out).  Workloads with a
bias (relative-position table or general jagged bias) also report `bias_grad`: the
backward that writes the bias's gradient as well, timed against the plain backward (the
step itself holds the bias constant).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl jfa|reference]
                  [--no-configs] [--shard]

The JSON line is the headline workload (--config, gem_self by default); at N=1 its
`configs` key then holds every other workload (tiny, cross, biased_causal,
longtail_causal, jagged_bias_causal), each timed the same way on the same GPU with its
forward / backward split, per-kernel roofline and the padded dense SDPA comparison.

Multi-GPU (torchrun, one process per GPU): every rank runs its own batch of the same
workload (independent problems, no collective on the data path): weak scaling.  With
--shard the ranks split ONE batch by sequence instead (longest-processing-time over
visited pairs, sharding.py): strong scaling, still no collective on the data path.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from jagged_attention_recsys_jfa_gb300.inputs import CONFIGS, make_batch  # noqa: E402

METRIC = "jagged attn fwd/bwd valid-token TFLOPS bf16 on 1 GB300; % of tensor peak"
DEFAULT_CONFIG = "gem_self"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------------------- accounting
def valid_pairs(lq, lk, causal):
    """Visited (query, key) pairs: Lq*Lk, or with bottom-right causal alignment the
    pairs j <= i + (Lk - Lq)."""
    lq = np.asarray(lq, dtype=np.int64)
    lk = np.asarray(lk, dtype=np.int64)
    if not causal:
        return int((lq * lk).sum())
    tot = 0
    for a, b in zip(lq.tolist(), lk.tolist()):
        first = max(0, a - b)            # rows before this see no key
        n = a - first
        if n <= 0 or b <= 0:
            continue
        s0 = first + (b - a) + 1         # keys seen by row `first`
        tot += n * s0 + n * (n - 1) // 2
    return tot


SHORT_Q = 128  # sequences with at most one query tile: backward in the fused pass


def nsp_max_rows():
    """Query rows up to which a sequence's backward takes the non-sequence-parallel pass
    (the library's process-wide setting; 0 when the library is not loaded)."""
    try:
        from jagged_attention_recsys_jfa_gb300 import jfa
        return 128 * jfa.jfa_nsp_max_tiles() if jfa._LIB is not None else 0
    except Exception:
        return 0


def _split(batch, nsp_rows=None):
    """Which backward pass covers each sequence: (fused, non-sequence-parallel, split)."""
    lq = np.asarray(batch.q_lengths)
    nsp_rows = nsp_max_rows() if nsp_rows is None else nsp_rows
    short = lq <= SHORT_Q
    nsp = (lq > SHORT_Q) & (lq <= nsp_rows)
    return short, nsp, ~(short | nsp)


def workload_flops(batch, nsp_rows=None):
    """Algorithmic flops: forward 4*d*H per visited pair; backward 10*d*H, of which the
    split passes take 8 (dK/dV) and 2 (dQ), and the fused pass (one query tile) and the
    non-sequence-parallel pass (if enabled for the sequence's length) all 10."""
    lq, lk, causal = np.asarray(batch.q_lengths), np.asarray(batch.kv_lengths), batch.cfg.causal
    short, nsp, long_ = _split(batch, nsp_rows)
    P = valid_pairs(lq, lk, causal)
    Pl = valid_pairs(lq[long_], lk[long_], causal)
    Ps = valid_pairs(lq[short], lk[short], causal)
    Pn = valid_pairs(lq[nsp], lk[nsp], causal)
    dH = batch.cfg.head_dim * batch.cfg.heads
    return {"pairs": P, "fwd": 4.0 * dH * P, "bwd": 10.0 * dH * P, "dkdv": 8.0 * dH * Pl, "dq": 2.0 * dH * Pl,
            "fused": 10.0 * dH * Ps, "nsp": 10.0 * dH * Pn}


def workload_bytes(batch, nsp_rows=None):
    """Algorithmic DRAM bytes per launch of each kernel: every input read once, every
    output written once (the per-query lse / D vectors on 128-row-padded rows).  A general
    jagged bias counts 2 bytes per visited (query, key) pair and head for each pass that
    covers its sequence: the elements the method reads (causally hidden pairs and the row
    padding are never needed)."""
    H, d = batch.cfg.heads, batch.cfg.head_dim
    row = 2.0 * H * d
    lq, lk = np.asarray(batch.q_lengths), np.asarray(batch.kv_lengths)
    Tq = float(lq.sum())
    if batch.cfg.general_bias:
        jb = np.array([2.0 * H * valid_pairs([a], [b], batch.cfg.causal) for a, b in zip(lq, lk)])
    else:
        jb = 0.0 * lq

    def part(sel):  # query rows, key rows, padded lse / D vector bytes, bias bytes of a subset
        return (float(lq[sel].sum()), float(lk[sel].sum()), 8.0 * H * float(((lq[sel] + 127) // 128 * 128).sum()),
                float(np.sum(jb[sel])))
    short, nsp, long_ = _split(batch, nsp_rows)
    Tql, Tkl, vecl, jbl = part(long_)
    Tqs, Tks, vecs, jbs = part(short)
    Tqn, Tkn, vecn, jbn = part(nsp)
    vec = vecl + vecs + vecn
    Tk = float(lk.sum())
    # the single-pass backwards read q, dO, k, v once and write dq, dk, dv once
    one_pass = lambda Tq_, Tk_, vec_, jb_: (2 * Tq_ + 2 * Tk_) * row + vec_ + (Tq_ + 2 * Tk_) * row + jb_
    return {"forward": (Tq + 2 * Tk) * row + Tq * row + 4.0 * H * Tq + float(np.sum(jb)),
            "bwd_preprocess": 2 * Tq * row + 4.0 * H * Tq + vec,
            "bwd_dkdv": (2 * Tql + 2 * Tkl) * row + vecl + 2 * Tkl * row + jbl,
            "bwd_dq": (2 * Tql + 2 * Tkl) * row + vecl + Tql * row + jbl,
            "bwd_fused": one_pass(Tqs, Tks, vecs, jbs),
            "bwd_nsp": one_pass(Tqn, Tkn, vecn, jbn)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return FALLBACK_PEAKS, "fallback"


def config_dict(cfg, name):
    d = {"workload": name, "batch": cfg.batch, "heads": cfg.heads, "head_dim": cfg.head_dim,
         "lengths": list(cfg.lengths), "causal": cfg.causal,
         "kv_lengths": list(cfg.kv_lengths) if cfg.kv_lengths else "same as query",
         "bias": f"relpos table [H,{cfg.bias_buckets}] fp32, bucket j-i+{cfg.bias_center}" if cfg.bias_buckets
         else ("general jagged bias, bf16 Lq x Lk block per sequence and head" if cfg.general_bias else None),
         "seed": cfg.seed, "l2": "inputs larger than L2, no flush"}
    return d


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampled every ~10 ms with timestamps; `window(t0, t1)` marks the timed
    region (host wall-clock seconds), and the report is taken from the samples inside it
    (all samples when none fell inside, which it then says)."""
    QUERY = ("timestamp,index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.path = tempfile.mktemp(prefix="jfa_clocks_", suffix=".csv")
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.uuid = str(getattr(torch.cuda.get_device_properties(device_index), "uuid", ""))
        except Exception:
            self.uuid = ""

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader",
                                          "-lms", "10"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def window(self, t0, t1):
        self.t0, self.t1 = t0, t1

    @staticmethod
    def parse(lines, uuid="", t0=None, t1=None):
        """Summarise nvidia-smi CSV lines (the QUERY fields, no header)."""
        import datetime
        rows = []
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 11:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            rows.append((ts, parts[1:]))
        if uuid:
            mine = [r for r in rows if uuid.replace("GPU-", "") in r[1][1]]
            rows = mine or rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        idx0 = rows[0][1][0]
        rows = [r for r in rows if r[1][0] == idx0]
        inside = [r for r in rows if t0 is not None and t0 <= r[0] <= t1]
        use = [r[1] for r in (inside or rows)]

        def num(x):
            try:
                return float(x.split()[0])
            except Exception:
                return None
        sm = [num(r[2]) for r in use if num(r[2]) is not None]
        mx = [num(r[3]) for r in use if num(r[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in use for n, v in zip(names, r[6:10]) if v.lower() == "active"})
        loaded = sm if inside else ([x for x in sm if mx and x >= 0.5 * max(mx)] or sm)
        out = {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
               "reasons": reasons, "samples": len(inside), "samples_total": len(rows)}
        if not inside:
            out["note"] = "no sample fell inside the timed region: figures from all samples of the run"
        return out

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        with open(self.path) as f:
            lines = f.readlines()
        os.unlink(self.path)
        return self.parse(lines, self.uuid, self.t0, self.t1)


# ----------------------------------------------------------------------------- CPU oracle leg
def oracle_sample(batch, budget_s, rng_seed=0):
    """Run the float64 oracle forward+backward on (sequence, head) pairs of the batch,
    drawn in a seeded order, until `budget_s` of wall time is spent.  Returns
    (valid fwd+bwd flops processed, seconds, pairs done)."""
    import oracle.jfa_oracle as orc

    cfg = batch.cfg
    rng = np.random.default_rng(rng_seed)
    B = batch.q_lengths.numel()
    order = rng.permutation(B)
    lq, lk = batch.q_lengths.numpy(), batch.kv_lengths.numpy()
    center = cfg.bias_center if batch.bias is not None else 0
    done_flops, pairs, t0 = 0.0, 0, time.perf_counter()
    dH = cfg.head_dim
    for b in order:
        h = int(rng.integers(cfg.heads))
        orc.sequence_reference(int(b), h, batch.q, batch.k, batch.v, batch.q_offsets, batch.kv_offsets,
                               cfg.scale, cfg.causal, batch.bias, center, dout=batch.dout,
                               jagged_bias=(batch.jbias, batch.jbias_offsets) if batch.jbias is not None else None)
        P = valid_pairs([lq[b]], [lk[b]], cfg.causal)
        done_flops += 14.0 * dH * P
        pairs += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return done_flops, time.perf_counter() - t0, pairs


def cpu_cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count() or 1


# ----------------------------------------------------------------------------- padded SDPA
def padded_sdpa(batch, steps):
    """Dense SDPA on the batch padded to its longest sequence (the padding-waste
    comparison): time per fwd+bwd step after three warm-up steps (a process's first call
    of a backend ran several times slower) and peak memory."""
    from torch.nn.attention import SDPBackend, sdpa_kernel

    cfg = batch.cfg
    dev = batch.q.device
    B, H, d = batch.q_lengths.numel(), cfg.heads, cfg.head_dim
    Lq, Lk = int(batch.q_lengths.max()), int(batch.kv_lengths.max())
    qo, ko = batch.q_offsets.cpu().tolist(), batch.kv_offsets.cpu().tolist()

    def pad(x, off, L):
        out = torch.zeros((B, L, H, d), dtype=x.dtype, device=dev)
        for b in range(B):
            out[b, : off[b + 1] - off[b]] = x[off[b]:off[b + 1]]
        return out.transpose(1, 2).contiguous()

    q, k, v = pad(batch.q, qo, Lq), pad(batch.k, ko, Lk), pad(batch.v, ko, Lk)
    do = pad(batch.dout, qo, Lq)
    mask = None
    if not cfg.causal:
        mask = (torch.arange(Lk, device=dev)[None, :] < batch.kv_lengths.to(dev)[:, None])[:, None, None, :]
    if cfg.bias_buckets:
        i = torch.arange(Lq, device=dev)[:, None]
        j = torch.arange(Lk, device=dev)[None, :]
        idx = (j - i + cfg.bias_center).clamp(0, cfg.bias_buckets - 1)
        bias = batch.bias[:, idx][None]  # [1, H, Lq, Lk]
        if cfg.causal:
            bias = bias.masked_fill(j > i, float("-inf"))
        mask = bias.to(torch.bfloat16)
    if cfg.general_bias:
        # the blocks copied into the padded score shape; padding and hidden pairs -inf
        jbo = batch.jbias_offsets.cpu().tolist()
        mask = torch.full((B, H, Lq, Lk), float("-inf"), dtype=torch.bfloat16, device=dev)
        for b in range(B):
            lqb, lkb = qo[b + 1] - qo[b], ko[b + 1] - ko[b]
            pitch = (lkb + 7) // 8 * 8
            blk = batch.jbias[:, jbo[b]:jbo[b] + lqb * pitch].reshape(H, lqb, pitch)[:, :, :lkb]
            if cfg.causal:
                vis = torch.ones(lqb, lkb, dtype=torch.bool, device=dev).tril(diagonal=lkb - lqb)
                blk = blk.masked_fill(~vis, float("-inf"))
            mask[b, :, :lqb, :lkb] = blk
    backends = [SDPBackend.FLASH_ATTENTION, SDPBackend.EFFICIENT_ATTENTION, SDPBackend.MATH] if mask is None \
        else [SDPBackend.EFFICIENT_ATTENTION, SDPBackend.CUDNN_ATTENTION, SDPBackend.MATH]
    for be in backends:
        try:
            qq, kk, vv = (t.clone().requires_grad_(True) for t in (q, k, v))

            def step():
                with sdpa_kernel([be]):
                    o = torch.nn.functional.scaled_dot_product_attention(
                        qq, kk, vv, attn_mask=mask, is_causal=cfg.causal and mask is None, scale=cfg.scale)
                o.backward(do)
            for _ in range(3):  # a process's first calls load and set up the backend's kernels
                step()
            torch.cuda.synchronize()
            torch.cuda.reset_peak_memory_stats()
            base = torch.cuda.memory_allocated()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                step()
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / steps
            peak = torch.cuda.max_memory_allocated() - base
            return {"backend": str(be).split(".")[-1], "ms_per_step": round(ms, 3),
                    "padded_shape": [B, H, Lq, Lk], "peak_extra_gb": round(peak / 1e9, 3)}
        except Exception as e:  # backend not applicable: try the next
            last = repr(e)[:200]
            torch.cuda.synchronize()
            continue
    return {"unavailable": last}


# ----------------------------------------------------------------------------- main arms
OTHER_CONFIGS = ("tiny", "cross", "biased_causal", "longtail_causal", "jagged_bias_causal")


def shard_batch(batch, index):
    """The sequences `index` of a batch as a batch of their own (values packed, offsets
    rebuilt, a general bias's blocks moved with their sequences; a table is shared)."""
    import dataclasses

    from jagged_attention_recsys_jfa_gb300.sharding import select_bias_blocks, select_sequences

    q, qo = select_sequences(batch.q, batch.q_offsets, index)
    k, ko = select_sequences(batch.k, batch.kv_offsets, index)
    v, _ = select_sequences(batch.v, batch.kv_offsets, index)
    do, _ = select_sequences(batch.dout, batch.q_offsets, index)
    jb = jbo = None
    if batch.jbias is not None:
        jb, jbo = select_bias_blocks(batch.jbias, batch.jbias_offsets, index)
    idx = torch.as_tensor(list(index), dtype=torch.int64)
    return dataclasses.replace(batch, q_lengths=batch.q_lengths[idx], kv_lengths=batch.kv_lengths[idx],
                               q_offsets=qo, kv_offsets=ko, q=q.contiguous(), k=k.contiguous(), v=v.contiguous(),
                               dout=do.contiguous(), jbias=jb, jbias_offsets=jbo)


class Step:
    """One step of the hot path on one resident batch: jfa_forward then jfa_backward through
    the public binding, outputs and workspaces allocated once."""

    def __init__(self, batch, device):
        from jagged_attention_recsys_jfa_gb300 import jfa

        self.jfa, self.batch, cfg = jfa, batch, batch.cfg
        self.center = cfg.bias_center if batch.bias is not None else 0
        self.out = torch.empty_like(batch.q)
        self.lse = torch.empty((cfg.heads, batch.q.shape[0]), dtype=torch.float32, device=device)
        self.dq, self.dk, self.dv = torch.empty_like(batch.q), torch.empty_like(batch.k), torch.empty_like(batch.v)
        B, H, d = batch.q_lengths.numel(), cfg.heads, cfg.head_dim
        Tq, Tk = batch.q.shape[0], batch.k.shape[0]
        self.ws_f = jfa.new_workspace(B, H, d, Tq, Tk, False, device)
        self.ws_b = jfa.new_workspace(B, H, d, Tq, Tk, True, device)
        self.jb = (batch.jbias, batch.jbias_offsets) if batch.jbias is not None else None

    def fwd(self):
        b, c = self.batch, self.batch.cfg
        self.jfa.jfa_forward(b.q, b.k, b.v, b.q_offsets, b.kv_offsets, b.bias, self.center, c.scale, c.causal,
                             out=self.out, lse=self.lse, workspace=self.ws_f, jagged_bias=self.jb)

    def bwd(self, bias_grad=None, jagged_bias_grad=None):
        b, c = self.batch, self.batch.cfg
        self.jfa.jfa_backward(b.dout, b.q, b.k, b.v, self.out, self.lse, b.q_offsets, b.kv_offsets, b.bias,
                              self.center, c.scale, c.causal, dq=self.dq, dk=self.dk, dv=self.dv,
                              workspace=self.ws_b, jagged_bias=self.jb, bias_grad=bias_grad,
                              jagged_bias_grad=jagged_bias_grad)

    def __call__(self):
        self.fwd()
        self.bwd()

    def check(self, where):
        st = (self.jfa.jfa_check_status(self.ws_f), self.jfa.jfa_check_status(self.ws_b))
        if st != (0, 0):
            raise RuntimeError(f"device status {st} {where}")


def kernel_pass(step, steps, stream):
    """The K steps again with events around the forward / backward halves and around every
    kernel launch (jfa_timing_enable): (median forward ms, median backward ms, per kernel
    {kind: (total ms, launches)})."""
    jfa = step.jfa
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3)) for _ in range(steps)]
    jfa.jfa_timing_read()  # drop anything recorded before
    jfa.jfa_timing_enable(True)
    for i in range(steps):
        ev[i][0].record(stream)
        step.fwd()
        ev[i][1].record(stream)
        step.bwd()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    jfa.jfa_timing_enable(False)
    per_kernel = jfa.jfa_timing_read()
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    bwd_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    return fwd_ms, bwd_ms, per_kernel


def roofline_of(batch, name, per_kernel, peaks, peak_src):
    """Per-kernel algorithmic rates and the roofline of the kernel with the largest time
    share: tensor-bound when its algorithmic flops per byte reach the ridge of the measured
    peaks, else HBM-bound."""
    fl = workload_flops(batch)
    kinds = {k: v for k, v in per_kernel.items() if v[1] > 0}
    dom = max(kinds, key=lambda k: kinds[k][0])
    algo = {"forward": fl["fwd"], "bwd_dkdv": fl["dkdv"], "bwd_dq": fl["dq"], "bwd_fused": fl["fused"],
            "bwd_nsp": fl["nsp"]}
    algo_bytes = workload_bytes(batch)
    ms_dom, n_dom = kinds[dom]
    t_dom = ms_dom / n_dom / 1e3
    traffic = load_traffic(dom, name)
    ridge = float(peaks["bf16_tflops"]) * 1e12 / (float(peaks["hbm_gbs"]) * 1e9)
    if dom in algo and algo_bytes.get(dom, 0) > 0 and algo[dom] / algo_bytes[dom] >= ridge:
        achieved = algo[dom] / t_dom / 1e12
        peak = float(peaks["bf16_tflops"])
        roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                    "unit": "TFLOP/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                    "peak_source": f"{peak_src} bf16 dense (burst)",
                    "frac_of_sustained": round(achieved / float(peaks["bf16_tflops_sustained"]), 4),
                    "flop_per_byte": round(algo[dom] / algo_bytes[dom], 1), "ridge": round(ridge, 1)}
    elif algo_bytes.get(dom, 0) > 0:
        achieved = algo_bytes[dom] / t_dom / 1e9
        peak = float(peaks["hbm_gbs"])
        roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                    "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                    "peak_source": f"{peak_src} HBM copy",
                    "algorithmic_bytes": algo_bytes[dom],
                    "flop_per_byte": round(algo[dom] / algo_bytes[dom], 1) if dom in algo else None,
                    "ridge": round(ridge, 1)}
    else:
        roofline = {"bound": "hbm", "kernel": dom, "achieved": None, "peak": float(peaks["hbm_gbs"]),
                    "unit": "GB/s", "frac": None, "traffic": traffic}
    kernels = {k: {"ms_per_launch": round(v[0] / v[1], 4), "launches": v[1],
                   "share": round(v[0] / sum(x[0] for x in kinds.values()), 4)} for k, v in kinds.items()}
    for k, f in algo.items():
        if k in kernels:
            kernels[k]["algorithmic_tflops"] = round(f / (kernels[k]["ms_per_launch"] / 1e3) / 1e12, 1)
    for k, nb in algo_bytes.items():
        if k in kernels:
            kernels[k]["algorithmic_gbs"] = round(nb / (kernels[k]["ms_per_launch"] / 1e3) / 1e9, 1)
    return roofline, kernels


def split_rates(fl, fwd_ms, bwd_ms, peak_tf):
    return ({"ms": round(fwd_ms, 4), "tflops": round(fl["fwd"] / (fwd_ms / 1e3) / 1e12, 1),
             "pct_of_peak": round(100 * fl["fwd"] / (fwd_ms / 1e3) / 1e12 / peak_tf, 2)},
            {"ms": round(bwd_ms, 4), "tflops": round(fl["bwd"] / (bwd_ms / 1e3) / 1e12, 1),
             "pct_of_peak": round(100 * fl["bwd"] / (bwd_ms / 1e3) / 1e12 / peak_tf, 2)})


def measure_config(name, args, device, peaks, peak_src):
    """One more workload on this GPU, timed like the headline (warm-up, then `steps` whole
    steps between two events on the launching stream; inputs larger than L2 or launch-bound),
    with its forward / backward split, per-kernel roofline and the padded dense SDPA
    comparison."""
    cfg = CONFIGS[name]
    batch = make_batch(cfg, device=device)
    fl = workload_flops(batch)
    step = Step(batch, device)
    for _ in range(args.warmup):
        step()
    step.check("after warm-up")
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / args.steps
    fwd_ms, bwd_ms, per_kernel = kernel_pass(step, args.steps, stream)
    step.check("in the timed region")
    peak_tf = float(peaks["bf16_tflops"])
    fwd, bwd = split_rates(fl, fwd_ms, bwd_ms, peak_tf)
    roofline, kernels = roofline_of(batch, name, per_kernel, peaks, peak_src)
    value = (fl["fwd"] + fl["bwd"]) / (ms / 1e3) / 1e12
    res = {"config": config_dict(cfg, name), "value": round(value, 2), "unit": "TFLOPS", "ms_per_step": round(ms, 4),
           "pct_of_tensor_peak": round(100 * value / peak_tf, 2), "fwd": fwd, "bwd": bwd,
           "valid_pairs": fl["pairs"], "roofline": roofline, "kernels": kernels,
           "gpu_launches": sum(c for _, c in per_kernel.values())}
    if not args.no_extras and int(np.asarray(batch.q_lengths).max()) > SHORT_Q:
        res["non_sequence_parallel"] = nsp_leg(step, batch, args.steps, stream, device)
    if not args.no_sdpa:
        del step
        torch.cuda.synchronize()
        sd = padded_sdpa(batch, 2)
        if "ms_per_step" in sd:
            sd["valid_tflops"] = round((fl["fwd"] + fl["bwd"]) / (sd["ms_per_step"] / 1e3) / 1e12, 2)
            sd["jfa_ms_per_step"] = round(ms, 4)
        res["padded_sdpa"] = sd
    del batch
    torch.cuda.empty_cache()
    return res


def run_jfa(args, rank, world, device):
    from jagged_attention_recsys_jfa_gb300.sharding import shard_sequences

    name = args.config
    cfg = CONFIGS[name]
    if args.batch:
        import dataclasses
        cfg = dataclasses.replace(cfg, batch=args.batch)
    if args.shard:
        # strong scaling: one batch, the same on every rank, split by sequence; each rank
        # runs only its shard (no collective on the data path)
        full = make_batch(cfg, device=device, seed=cfg.seed)
        mine = shard_sequences(full.q_lengths.tolist(), full.kv_lengths.tolist(), world, cfg.causal)[rank]
        batch = shard_batch(full, mine) if world > 1 else full
        del full
    else:
        batch = make_batch(cfg, device=device, seed=cfg.seed + rank)
    fl = workload_flops(batch)
    step = Step(batch, device)

    for _ in range(args.warmup):
        step()
    step.check("after warm-up")
    torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # ---- timed region: inputs resident in HBM
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(device.index or 0)
    torch.cuda.reset_peak_memory_stats()
    mem_base = torch.cuda.memory_allocated()
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    # the timed region: K whole steps, nothing recorded between the kernels
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    host_t0 = time.time()  # the stream is idle: the GPU starts the region now
    t_start.record(stream)
    for i in range(args.steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    host_t1 = time.time()
    clocks.window(host_t0, host_t1)
    time.sleep(0.05)  # let the sampler flush the region's last samples
    barrier()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    fwd_ms, bwd_ms, per_kernel = kernel_pass(step, args.steps, stream)
    peak_mem = torch.cuda.max_memory_allocated() - mem_base
    step.check("in the timed region (first error since warm-up)")

    # max over ranks of the timed region, sum of work over ranks
    t_local = torch.tensor([total_ms], dtype=torch.float64, device=device)
    w_local = torch.tensor([fl["fwd"] + fl["bwd"]], dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t_local, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.all_reduce(w_local, op=torch.distributed.ReduceOp.SUM)
    t_max_s = float(t_local.item()) / 1e3
    total_flops = float(w_local.item()) * args.steps
    value = total_flops / t_max_s / 1e12
    launches = sum(c for _, c in per_kernel.values())

    graph_ms = None
    if not args.no_extras:
        graph_ms = graph_replay(step, args.steps, stream, device)
    bias_grad = None
    if not args.no_extras and (batch.bias is not None or batch.jbias is not None):
        bias_grad = bias_grad_leg(step, batch, args.steps, stream)
    e2e = None
    if not args.no_extras:
        e2e_s = e2e_leg(step, batch, args, device, barrier)
        t_e2e = torch.tensor([e2e_s["seconds"]], dtype=torch.float64, device=device)
        if world > 1:
            torch.distributed.all_reduce(t_e2e, op=torch.distributed.ReduceOp.MAX)
        e2e = {"value": round(total_flops / float(t_e2e.item()) / 1e12, 2), "unit": "TFLOPS",
               "h2d_bytes_per_step": e2e_s["h2d"], "d2h_bytes_per_step": e2e_s["d2h"],
               # both directions' bytes per second: what the host link carried
               "host_link_gbs": round((e2e_s["h2d"] + e2e_s["d2h"]) * args.steps / float(t_e2e.item()) / 1e9, 1)}
    nsp_cmp = None
    if not args.no_extras and world == 1 and int(np.asarray(batch.q_lengths).max()) > SHORT_Q:
        nsp_cmp = nsp_leg(step, batch, args.steps, stream, device)

    if rank != 0:
        return None
    return finish(args, name, cfg, batch, step, fl, world, value, t_max_s, total_ms, fwd_ms, bwd_ms, per_kernel,
                  peak_mem, launches, clk, graph_ms, bias_grad, e2e, device, nsp_cmp)


def graph_replay(step, steps, stream, device):
    """The same step captured once in a CUDA graph and replayed: the planner reads the
    offsets on the device, so one capture serves every batch of the same shape; replays
    drop the per-call host work and launch gaps (what launch-bound small batches gain).
    Returns ms per replayed step."""
    side = torch.cuda.Stream(device=device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(3):
        graph.replay()
    g_start, g_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    g_start.record(stream)
    for _ in range(steps):
        graph.replay()
    g_end.record(stream)
    torch.cuda.synchronize()
    step.check("in the graph replays")
    del graph
    return g_start.elapsed_time(g_end) / steps


def bias_grad_leg(step, batch, steps, stream):
    """Workloads with a bias: the same backward also writing the bias's gradient, timed
    against the plain backward on the same inputs (the step holds the bias constant)."""
    jfa = step.jfa
    dbias = torch.empty_like(batch.bias) if batch.bias is not None else None
    djb = torch.empty_like(batch.jbias) if batch.jbias is not None else None

    def timed(fn):
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / steps

    bwd_g = lambda: step.bwd(bias_grad=dbias, jagged_bias_grad=djb)
    t_plain, t_grad = timed(step.bwd), timed(bwd_g)
    jfa.jfa_timing_read()
    jfa.jfa_timing_enable(True)
    timed(bwd_g)
    jfa.jfa_timing_enable(False)
    pk = jfa.jfa_timing_read()
    step.check("after the bias-gradient backward")
    return {"kind": "relative-position table" if batch.bias is not None else "general jagged bias",
            "bwd_ms": round(t_grad, 4), "bwd_ms_without": round(t_plain, 4),
            "overhead": round(t_grad / t_plain - 1, 4),
            "kernels_ms": {k: round(v[0] / v[1], 4) for k, v in pk.items() if v[1]}}


def nsp_leg(step, batch, steps, stream, device):
    """Row N2 against the split passes on the same inputs: the backward timed with the
    library's routing as it stands (by default every sequence of more than one query tile
    takes the dK/dV + dQ passes) and again with sequences of 2 .. 16 query tiles sent to the
    non-sequence-parallel pass, each with its per-kernel times and the share of query rows
    that took each path.  The setting is restored afterwards."""
    jfa = step.jfa
    prev = jfa.jfa_nsp_max_tiles()
    lq = np.asarray(batch.q_lengths)
    rows = max(int(lq.sum()), 1)

    def one(tiles):
        jfa.jfa_set_nsp_max_tiles(tiles)
        ws_keep = step.ws_b
        b, c = batch, batch.cfg
        step.ws_b = jfa.new_workspace(b.q_lengths.numel(), c.heads, c.head_dim, b.q.shape[0], b.k.shape[0], True,
                                      device)
        try:
            for _ in range(3):
                step.bwd()
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(steps):
                step.bwd()
            e.record(stream)
            torch.cuda.synchronize()
            jfa.jfa_timing_read()
            jfa.jfa_timing_enable(True)
            step.bwd()
            torch.cuda.synchronize()
            jfa.jfa_timing_enable(False)
            pk = jfa.jfa_timing_read()
            step.check(f"in the backward with non-sequence-parallel tiles <= {tiles}")
        finally:
            step.ws_b = ws_keep
        short, nsp, split = _split(batch, 128 * tiles if tiles > 1 else 0)
        return {"nsp_max_tiles": tiles, "bwd_ms": round(a.elapsed_time(e) / steps, 4),
                "kernels_ms": {k: round(v[0] / v[1], 4) for k, v in pk.items() if v[1]},
                "query_rows": {"fused": round(float(lq[short].sum()) / rows, 4),
                               "non_sequence_parallel": round(float(lq[nsp].sum()) / rows, 4),
                               "split": round(float(lq[split].sum()) / rows, 4)}}

    try:
        return {"default": one(prev), "all_multi_tile_nsp": one(16)}
    finally:
        jfa.jfa_set_nsp_max_tiles(prev)
        step.bwd()  # the step's gradients as the default routing computes them again
        torch.cuda.synchronize()


def e2e_leg(step, batch, args, device, barrier):
    """End to end through the public call with host buffers.  Every step copies its inputs
    in from pinned host memory and its results (out, lse, dq, dk, dv) back out.  Consecutive
    steps overlap the way a training loop would run them: the next step's inputs stream in
    on one copy stream while this step computes, and its results stream out on another;
    device inputs and outputs are double-buffered so no copy touches a buffer a kernel
    still uses.  Returns the wall seconds of `steps` steps and the bytes copied per step."""
    jfa, cfg, center = step.jfa, batch.cfg, step.center
    pin = lambda t: t.cpu().pin_memory()
    in_names = ("q", "k", "v", "dout", "q_offsets", "kv_offsets") + (
        ("jbias", "jbias_offsets") if batch.jbias is not None else ())  # a general bias is per-batch input
    h_in = {n: pin(getattr(batch, n)) for n in in_names}
    out_names = ("out", "lse", "dq", "dk", "dv")
    res = {"out": step.out, "lse": step.lse, "dq": step.dq, "dk": step.dk, "dv": step.dv}
    h_out = [{n: torch.empty(res[n].shape, dtype=res[n].dtype, pin_memory=True) for n in out_names}
             for _ in range(2)]
    d_in = [{n: torch.empty_like(getattr(batch, n)) for n in h_in} for _ in range(2)]
    d_out = [{n: torch.empty_like(res[n]) for n in out_names} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in h_in.values())
    d2h = sum(t.numel() * t.element_size() for t in h_out[0].values())
    s_comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def e2e_step(i):
        b = i & 1
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(ev_done[b])  # the step that last used these inputs has computed
            for n in h_in:
                d_in[b][n].copy_(h_in[n], non_blocking=True)
            ev_in[b].record(s_in)
        s_comp.wait_event(ev_in[b])
        if used[b]:
            s_comp.wait_event(ev_free[b])  # its results have been copied out
        x, o = d_in[b], d_out[b]
        xjb = (x["jbias"], x["jbias_offsets"]) if "jbias" in x else None
        jfa.jfa_forward(x["q"], x["k"], x["v"], x["q_offsets"], x["kv_offsets"], batch.bias, center, cfg.scale,
                        cfg.causal, out=o["out"], lse=o["lse"], workspace=step.ws_f, jagged_bias=xjb)
        jfa.jfa_backward(x["dout"], x["q"], x["k"], x["v"], o["out"], o["lse"], x["q_offsets"], x["kv_offsets"],
                         batch.bias, center, cfg.scale, cfg.causal, dq=o["dq"], dk=o["dk"], dv=o["dv"],
                         workspace=step.ws_b, jagged_bias=xjb)
        ev_done[b].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_done[b])
            for n in out_names:
                h_out[b][n].copy_(o[n], non_blocking=True)
            ev_free[b].record(s_out)
        used[b] = True

    for i in range(max(2, args.warmup)):
        e2e_step(i)
    torch.cuda.synchronize()
    # the copied-out results are the resident run's (the kernels are deterministic)
    if not (torch.equal(h_out[0]["out"], step.out.cpu()) and torch.equal(h_out[0]["dq"], step.dq.cpu())):
        raise RuntimeError("end-to-end results differ from the resident run")
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i)
    torch.cuda.synchronize()
    secs = time.perf_counter() - t0
    return {"seconds": secs, "h2d": h2d, "d2h": d2h}


def finish(args, name, cfg, batch, step, fl, world, value, t_max_s, total_ms, fwd_ms, bwd_ms, per_kernel, peak_mem,
           launches, clk, graph_ms, bias_grad, e2e, device, nsp_cmp=None):
    """Rank 0: the roofline, the CPU baseline, the padded SDPA comparison and every other
    workload, then the JSON line."""
    peaks, peak_src = load_peaks()
    roofline, kernels = roofline_of(batch, name, per_kernel, peaks, peak_src)
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu_batch = make_batch(cfg, device="cpu")
        f_done, secs, npairs = oracle_sample(cpu_batch, args.cpu_seconds)
        cpu = {"value": round(f_done / secs / 1e12, 6), "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
               "sample": f"{npairs} (sequence, head) pairs of the {name} workload (CPU-seeded batch), float64 "
                         f"forward+backward, {secs:.1f} s"}
    sdpa = None
    if not args.no_sdpa and world == 1:
        s = padded_sdpa(batch, max(2, min(args.steps, 5)))
        if "ms_per_step" in s:
            s["valid_tflops"] = round((fl["fwd"] + fl["bwd"]) / (s["ms_per_step"] / 1e3) / 1e12, 1)
            s["jfa_ms_per_step"] = round(total_ms / args.steps, 3)
            s["jfa_peak_extra_gb"] = round(peak_mem / 1e9, 3)
        sdpa = s

    # ---- every other workload on the same GPU, after the headline's timed region
    others = None
    if world == 1 and not args.no_configs and not args.shard:
        del step
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        others = {}
        for other in OTHER_CONFIGS:
            if other != name:
                others[other] = measure_config(other, args, device, peaks, peak_src)

    step_ms = t_max_s * 1e3 / args.steps
    peak_tf = float(peaks["bf16_tflops"])
    fwd, bwd = split_rates(fl, fwd_ms, bwd_ms, peak_tf)
    cfgd = config_dict(cfg, name)
    if args.shard:
        cfgd["sharded"] = f"one batch split by sequence over {world} rank(s) (longest-processing-time)"
    return {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 4), "higher_is_better": True,
        "scaling": "strong" if args.shard else "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded jagged batch, values N(0,1) in bf16)",
        "config": cfgd,
        "pct_of_tensor_peak": round(100 * value / world / peak_tf, 2),
        "fwd": fwd, "bwd": bwd,
        "valid_pairs": fl["pairs"], "kernels": kernels, "roofline": roofline, "cpu_baseline": cpu,
        "graph_replay": None if graph_ms is None else {
            "ms_per_step": round(graph_ms, 4),
            "value": round((fl["fwd"] + fl["bwd"]) / (graph_ms * 1e-3) / 1e12, 2), "unit": "TFLOPS"},
        "e2e": e2e, "gpu_launches": launches, "clocks": clk, "padded_sdpa": sdpa, "bias_grad": bias_grad,
        "non_sequence_parallel": nsp_cmp,
        "peak_mem_extra_gb": round(peak_mem / 1e9, 3),
        "configs": others,
    }


KERNEL_SOURCE = {"forward": "jfa_fwd.cu", "bwd_preprocess": "jfa_bwd.cu", "bwd_dkdv": "jfa_bwd.cu",
                 "bwd_dq": "jfa_bwd.cu", "bwd_fused": "jfa_bwd.cu", "bwd_nsp": "jfa_bwd.cu", "plan": "jfa_plan.cu"}


def kernel_source_hash(kernel):
    """Hash of the sources a kernel's DRAM traffic depends on: its translation unit, the
    planner (which orders the work and so decides what is re-read from L2) and every shared
    header; DRAM counters taken from other sources are stale."""
    import glob
    import hashlib
    csrc = os.path.join(ROOT, "jagged_attention_recsys_jfa_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in sorted({KERNEL_SOURCE[kernel], "jfa_plan.cu"})]
    files += sorted(glob.glob(os.path.join(csrc, "*.cuh")) + glob.glob(os.path.join(csrc, "*.h")))
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_traffic(kernel, workload):
    """DRAM bytes (read + write) per launch from the committed ncu summary, if one matches
    this workload and was taken on the kernel's sources as they are now (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        if t.get("source_sha", {}).get(kernel) != kernel_source_hash(kernel):
            return None
        return t.get(workload, {}).get(kernel)
    except Exception:
        return None


def run_reference(args):
    """The oracle as the reference arm: float64 on the host cores, a bounded sample of
    the workload per step."""
    name = args.config
    cfg = CONFIGS[name]
    batch = make_batch(cfg, device="cpu")
    per_step = max(2.0, min(20.0, 150.0 / max(1, args.steps + args.warmup)))
    for w in range(args.warmup):
        oracle_sample(batch, per_step / 4, rng_seed=100 + w)
    f_tot, s_tot, n_tot = 0.0, 0.0, 0
    for i in range(args.steps):
        f, s, n = oracle_sample(batch, per_step, rng_seed=i)
        f_tot, s_tot, n_tot = f_tot + f, s_tot + s, n_tot + n
    value = f_tot / s_tot / 1e12
    sample = (f"{n_tot} (sequence, head) pairs of the {name} workload over {args.steps} steps "
              f"(about {per_step:.0f} s each), float64 forward+backward")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOPS", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * s_tot / args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded jagged batch, values N(0,1) in bf16)", "config": config_dict(cfg, name),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=sorted(CONFIGS))
    ap.add_argument("--impl", default="jfa", choices=["jfa", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sdpa", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="time only --config (by default every other workload follows, at N=1)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's sequence count (smaller cases for profiling)")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the CUDA-graph, bias-gradient and end-to-end legs")
    ap.add_argument("--shard", action="store_true",
                    help="split one batch of --config over the ranks by sequence (strong scaling) instead of "
                         "one batch per rank (weak scaling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group("nccl", device_id=device)
    try:
        res = run_jfa(args, rank, world, device)
        if rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
