"""Seeded synthetic jagged-attention inputs.

This module only draws random numbers and lays them out as jagged tensors; it
holds none of the attention arithmetic.  Both the CPU oracle and the CUDA path
consume what it returns, so it is the single source of inputs for parity.

Workloads (sequence-length mixes, head counts, head dims) follow the jagged
recommendation workloads that "Jagged Flash Attention (JFA)" describes (Definition:
user sequences from a few hundred up to tens of thousands of tokens, query and
key/value lengths that differ, an additive bias; Results: jaggedness around one
half).  Production length distributions are not public; the uniform and log-normal
mixes below stand in for them.

Draw order (one generator per call): lengths -> q -> k -> v -> bias -> dout -> general
bias (the last only for workloads that have one, so the others are unchanged by it).
Values are float32 normal samples rounded to bfloat16 (round to nearest even);
the oracle promotes exactly these bf16 values to float64.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class JaggedConfig:
    """One synthetic workload.

    lengths: ("uniform", lo, hi) inclusive, or ("lognormal", median, sigma, lo, hi).
    kv_lengths: None for self-attention (key lengths equal query lengths), else a
    second length spec drawn independently per sample (cross-attention).
    """

    name: str
    batch: int
    heads: int
    head_dim: int
    lengths: tuple
    kv_lengths: Optional[tuple] = None
    causal: bool = False
    bias_buckets: int = 0          # 0 = no bias; else per-head relative-position table size
    bias_center: int = 0           # bucket = clamp(j - i + center, 0, buckets - 1)
    bias_std: float = 0.5
    general_bias: bool = False     # a general jagged bias: one Lq x Lk bf16 matrix per sequence and head
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


# The five workloads, smallest first.  "tiny" is the correctness case the CPU
# oracle finishes in milliseconds; the rest are production-shaped.
CONFIGS = {
    "tiny": JaggedConfig("tiny", 4, 2, 64, ("uniform", 1, 64)),
    "gem_self": JaggedConfig("gem_self", 256, 8, 128, ("uniform", 1, 1024)),
    "cross": JaggedConfig("cross", 512, 4, 128, ("uniform", 1, 64),
                          kv_lengths=("uniform", 256, 8192)),
    "biased_causal": JaggedConfig("biased_causal", 128, 4, 64, ("uniform", 1, 2048),
                                  causal=True, bias_buckets=4096, bias_center=2048),
    "longtail_causal": JaggedConfig("longtail_causal", 64, 8, 128,
                                    ("lognormal", 512.0, 1.2, 16, 16384), causal=True),
    # the biased_causal shape with a general jagged bias (one Lq x Lk block per sequence
    # and head) in place of the relative-position table
    "jagged_bias_causal": JaggedConfig("jagged_bias_causal", 128, 4, 64, ("uniform", 1, 2048),
                                       causal=True, general_bias=True),
}


def _draw_lengths(spec: tuple, n: int, g: torch.Generator) -> torch.Tensor:
    kind = spec[0]
    if kind == "uniform":
        lo, hi = int(spec[1]), int(spec[2])
        return torch.randint(lo, hi + 1, (n,), generator=g, dtype=torch.int64)
    if kind == "lognormal":
        median, sigma, lo, hi = float(spec[1]), float(spec[2]), int(spec[3]), int(spec[4])
        z = torch.randn(n, generator=g, dtype=torch.float64)
        lens = torch.round(torch.exp(math.log(median) + sigma * z)).to(torch.int64)
        return lens.clamp_(lo, hi)
    if kind == "fixed":
        return torch.tensor(list(spec[1]), dtype=torch.int64)
    raise ValueError(f"unknown length spec {spec!r}")


def jagged_bias_offsets(q_lengths: torch.Tensor, kv_lengths: torch.Tensor) -> torch.Tensor:
    """Block offsets of a general jagged bias: sequence b's Lq_b x Lk_b block takes
    Lq_b * round_up(Lk_b, 8) elements (rows padded to a multiple of 8), blocks packed."""
    sizes = q_lengths.to(torch.int64) * ((kv_lengths.to(torch.int64) + 7) // 8 * 8)
    return offsets_from_lengths(sizes)


def offsets_from_lengths(lengths: torch.Tensor) -> torch.Tensor:
    """int64 [B+1] exclusive prefix sum: off[0] = 0, off[b+1] = off[b] + len[b]."""
    off = torch.zeros(lengths.numel() + 1, dtype=torch.int64)
    off[1:] = torch.cumsum(lengths.to(torch.int64), 0)
    return off


@dataclasses.dataclass
class JaggedBatch:
    cfg: JaggedConfig
    q_lengths: torch.Tensor      # int64 [B], CPU
    kv_lengths: torch.Tensor     # int64 [B], CPU
    q_offsets: torch.Tensor      # int64 [B+1], on `device`
    kv_offsets: torch.Tensor     # int64 [B+1], on `device`
    q: torch.Tensor              # bf16 [Tq, H, d]
    k: torch.Tensor              # bf16 [Tk, H, d]
    v: torch.Tensor              # bf16 [Tk, H, d]
    bias: Optional[torch.Tensor]  # fp32 [H, buckets] or None
    dout: torch.Tensor           # bf16 [Tq, H, d]
    jbias: Optional[torch.Tensor] = None          # bf16 [H, plane]: general jagged bias, or None
    jbias_offsets: Optional[torch.Tensor] = None  # int64 [B+1] block offsets, on `device`

    @property
    def total_q(self) -> int:
        return int(self.q_lengths.sum())

    @property
    def total_kv(self) -> int:
        return int(self.kv_lengths.sum())


def make_batch(cfg: JaggedConfig, device="cpu", seed: Optional[int] = None,
               q_lengths=None, kv_lengths=None) -> JaggedBatch:
    """Draw one batch.  Lengths come from a CPU generator (identical on every
    device); values come from a generator on `device`, seeded the same way, so a
    batch is reproducible per device type.  Explicit lengths override the spec."""
    seed = cfg.seed if seed is None else seed
    device = torch.device(device)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    B = cfg.batch
    if q_lengths is None:
        lq = _draw_lengths(cfg.lengths, B, g)
    else:
        lq = torch.as_tensor(q_lengths, dtype=torch.int64).clone()
        B = lq.numel()
    if kv_lengths is not None:
        lk = torch.as_tensor(kv_lengths, dtype=torch.int64).clone()
    elif cfg.kv_lengths is None:
        lk = lq.clone()
    else:
        lk = _draw_lengths(cfg.kv_lengths, B, g)
    if lk.numel() != lq.numel():
        raise ValueError("query and key/value length lists differ in batch size")

    gv = torch.Generator(device=device)
    gv.manual_seed(seed + 1)
    H, d = cfg.heads, cfg.head_dim
    Tq, Tk = int(lq.sum()), int(lk.sum())

    def normal_bf16(n_rows):
        x = torch.randn((n_rows, H, d), generator=gv, device=device, dtype=torch.float32)
        return x.to(torch.bfloat16)

    q = normal_bf16(Tq)
    k = normal_bf16(Tk)
    v = normal_bf16(Tk)
    bias = None
    if cfg.bias_buckets:
        bias = torch.randn((H, cfg.bias_buckets), generator=gv, device=device,
                           dtype=torch.float32) * cfg.bias_std
    dout = normal_bf16(Tq)
    jbias = jboff = None
    if cfg.general_bias:
        jboff = jagged_bias_offsets(lq, lk)
        plane = int(jboff[-1])
        jbias = (torch.randn((H, plane), generator=gv, device=device, dtype=torch.float32)
                 * cfg.bias_std).to(torch.bfloat16)
        jboff = jboff.to(device)
    return JaggedBatch(cfg, lq, lk, offsets_from_lengths(lq).to(device),
                       offsets_from_lengths(lk).to(device), q, k, v, bias, dout, jbias, jboff)
