"""CPU float64 oracle for Jagged Flash Attention (test infrastructure only).

This module is the correctness reference that the CUDA path is checked against.
Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
may import it; the library itself never calls it and has no CPU fallback.

What it computes (plain definitions, no tiling, no fusion):

* Exact softmax attention per jagged sequence -- exact in the sense of the
  FlashAttention lineage that "TLX-Optimized Jagged Flash Attention" builds on
  (section "Why Jagged Flash Attention Deserves Attention": tiling plus online
  softmax never changes the result) -- applied directly to variable-length
  sequences packed as values plus int64 offsets ("Jagged Flash Attention (JFA)",
  Definition), with asymmetric query/key lengths and an additive per-head bias.
* The backward of the same function (the Definition lists a backward pass among
  JFA's features; the gradient formulas are the standard ones of FlashAttention-2),
  and the gradient of the relative-position bias table (the Definition's custom
  biases as a trained parameter: the chain rule through s_ij = ... + table[bucket]).
* Two independent formulations used to pin the first one: brute-force padded
  dense attention with a -inf mask (the masking that "Four generations" item 1
  replaces), and a step-by-step float64 emulation of the tiled online softmax
  with zero-padded tails and the subtraction correction ("Four generations"
  item 1: padded rows enter as zeros and their exponentials are taken back out of
  the row sum).

Readings where the pages are silent (each also listed in the design notes):

* layout: jagged values are token-major [T, H, d]; lse is [H, T];
* scores: s_ij = scale * q_i . k_j + beta_h(i, j); bias is added after scaling;
* bias: per-head relative-position table, beta_h(i, j) = table[h, clamp(j - i +
  center, 0, buckets - 1)] with i, j local 0-based positions; or a general jagged
  bias, one Lq x Lk matrix per sequence and head, stored row-major with rows padded
  to a multiple of 8 elements from a per-sequence block offset;
* causal with unequal lengths: bottom-right alignment, key j visible to query i
  iff j <= i + (Lk - Lq);
* a query row that sees no key (empty key sequence, or causal with Lq > Lk):
  output 0, lse = -inf, zero gradient;
* lse is the natural logarithm of sum_j exp(s_ij).

All arithmetic is float64 on the exact bf16 input values.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def to_f64(x):
    """Promote a torch tensor (any dtype, any device) or array to a float64 ndarray."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch  # local import: the oracle itself is numpy

        return x.detach().to("cpu", torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def to_i64(x):
    if hasattr(x, "detach"):
        return x.detach().to("cpu").numpy().astype(np.int64)
    return np.asarray(x, dtype=np.int64)


# ---------------------------------------------------------------------------
# per-sequence building blocks
# ---------------------------------------------------------------------------

def relpos_bias(table_row, Lq, Lk, center):
    """beta(i, j) = table_row[clamp(j - i + center, 0, n - 1)] as an [Lq, Lk] matrix."""
    n = table_row.shape[0]
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    idx = np.clip(j - i + center, 0, n - 1)
    return table_row[idx]


def jagged_bias_block(values_h, off_b, Lq, Lk):
    """One sequence's block of a general jagged bias (one head's plane `values_h`): the
    Lq x Lk matrix stored row-major from element `off_b` with its rows padded to a
    multiple of 8 elements."""
    pitch = (Lk + 7) // 8 * 8
    return values_h[off_b:off_b + Lq * pitch].reshape(Lq, pitch)[:, :Lk]


def causal_visible(Lq, Lk):
    """Bottom-right aligned causal visibility: j <= i + (Lk - Lq)."""
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    return j <= i + (Lk - Lq)


def sequence_scores(q, k, scale, bias=None, visible=None):
    """S = scale * Q K^T (+ bias), masked entries -inf.  q: [Lq, d], k: [Lk, d]."""
    s = scale * (q @ k.T)
    if bias is not None:
        s = s + bias
    if visible is not None:
        s = np.where(visible, s, NEG_INF)
    return s


def softmax_rows(s):
    """Row softmax of a score matrix.  Returns (P, lse); rows with no finite score
    get P = 0 and lse = -inf."""
    Lq = s.shape[0]
    if s.shape[1] == 0:
        return np.zeros_like(s), np.full(Lq, NEG_INF)
    m = s.max(axis=1)
    live = np.isfinite(m)
    m_safe = np.where(live, m, 0.0)
    e = np.exp(s - m_safe[:, None])          # exp(-inf) = 0 for masked entries
    l = e.sum(axis=1)
    lse = np.where(live, m_safe + np.log(np.where(live, l, 1.0)), NEG_INF)
    p = np.where(live[:, None], e / np.where(live, l, 1.0)[:, None], 0.0)
    return p, lse


def sequence_forward(q, k, v, scale, bias=None, visible=None):
    """O = softmax(S) V, lse = log sum exp S, per row."""
    s = sequence_scores(q, k, scale, bias, visible)
    p, lse = softmax_rows(s)
    return p @ v, lse


def sequence_score_grad(do, q, k, v, scale, bias=None, visible=None):
    """Gradient of sum(dO * O) w.r.t. the scores s_ij, and P.

    dP = dO V^T;  D_i = sum_j P_ij dP_ij (= rowsum(dO * O));  dS = P * (dP - D).
    Hidden pairs have P = 0 and so dS = 0.
    """
    s = sequence_scores(q, k, scale, bias, visible)
    p, _ = softmax_rows(s)
    o = p @ v
    dp = do @ v.T
    D = (do * o).sum(axis=1)
    return p * (dp - D[:, None]), p


def sequence_backward(do, q, k, v, scale, bias=None, visible=None):
    """Gradients of sum(dO * O) w.r.t. q, k, v (bias held constant).

    dV = P^T dO;  dS as in `sequence_score_grad`;  dQ = scale * dS K;  dK = scale * dS^T Q.
    """
    ds, p = sequence_score_grad(do, q, k, v, scale, bias, visible)
    dv = p.T @ do
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


def sequence_bias_grad(ds, num_buckets, center):
    """Gradient of the loss w.r.t. one head's relative-position table from this
    sequence's dS: s_ij depends on table[clamp(j - i + center, 0, n - 1)] with slope 1,
    so each table entry collects the dS of every (i, j) whose bucket it is."""
    Lq, Lk = ds.shape
    i = np.arange(Lq)[:, None]
    j = np.arange(Lk)[None, :]
    idx = np.clip(j - i + center, 0, num_buckets - 1)
    return np.bincount(idx.ravel(), weights=ds.ravel(), minlength=num_buckets).astype(np.float64)


# ---------------------------------------------------------------------------
# jagged front ends
# ---------------------------------------------------------------------------

def _seq_inputs(b, h, q, k, v, qo, ko, scale, causal, bias_table, bias_center, jagged_bias=None):
    q0, q1 = int(qo[b]), int(qo[b + 1])
    k0, k1 = int(ko[b]), int(ko[b + 1])
    qb, kb, vb = q[q0:q1, h, :], k[k0:k1, h, :], v[k0:k1, h, :]
    Lq, Lk = q1 - q0, k1 - k0
    bias = None
    if bias_table is not None:
        bias = relpos_bias(bias_table[h], Lq, Lk, bias_center)
    elif jagged_bias is not None:
        values, boff = jagged_bias
        bias = jagged_bias_block(values[h], int(boff[b]), Lq, Lk)
    vis = causal_visible(Lq, Lk) if causal else None
    return (q0, q1, k0, k1), qb, kb, vb, bias, vis


def _jagged_bias_f64(jagged_bias):
    if jagged_bias is None:
        return None
    values, boff = jagged_bias
    return to_f64(values), to_i64(boff)


def check_offsets(off, total):
    off = to_i64(off)
    if off.ndim != 1 or off.size < 1 or off[0] != 0 or off[-1] != total or np.any(np.diff(off) < 0):
        raise ValueError("offsets must start at 0, be non-decreasing and end at the row count")
    return off


def jagged_forward(q, k, v, q_offsets, kv_offsets, scale, causal=False,
                   bias_table=None, bias_center=0, heads=None, jagged_bias=None):
    """Jagged attention forward.

    q: [Tq, H, d]; k, v: [Tk, H, d]; offsets int64 [B+1].
    Returns out float64 [Tq, H, d] and lse float64 [H, Tq].
    `heads` optionally restricts the computation to a subset of heads (the other
    heads' entries are left as NaN) -- used to sample large workloads.
    `jagged_bias` = (values [H, plane], block offsets [B+1]): a general additive bias,
    one block per sequence (see `jagged_bias_block`), instead of the relative-position
    table.
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    Tq, H, d = q.shape
    qo = check_offsets(q_offsets, Tq)
    ko = check_offsets(kv_offsets, k.shape[0])
    bt = to_f64(bias_table)
    jb = _jagged_bias_f64(jagged_bias)
    out = np.full((Tq, H, d), np.nan)
    lse = np.full((H, Tq), np.nan)
    for b in range(qo.size - 1):
        for h in (range(H) if heads is None else heads):
            (q0, q1, _, _), qb, kb, vb, bias, vis = _seq_inputs(
                b, h, q, k, v, qo, ko, scale, causal, bt, bias_center, jb)
            o, l = sequence_forward(qb, kb, vb, scale, bias, vis)
            out[q0:q1, h, :] = o
            lse[h, q0:q1] = l
    return out, lse


def jagged_backward(dout, q, k, v, q_offsets, kv_offsets, scale, causal=False,
                    bias_table=None, bias_center=0, jagged_bias=None):
    """Jagged attention backward: (dq, dk, dv), float64, shapes of q, k, v."""
    do, q, k, v = to_f64(dout), to_f64(q), to_f64(k), to_f64(v)
    Tq, H, d = q.shape
    qo = check_offsets(q_offsets, Tq)
    ko = check_offsets(kv_offsets, k.shape[0])
    bt = to_f64(bias_table)
    jb = _jagged_bias_f64(jagged_bias)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(qo.size - 1):
        for h in range(H):
            (q0, q1, k0, k1), qb, kb, vb, bias, vis = _seq_inputs(
                b, h, q, k, v, qo, ko, scale, causal, bt, bias_center, jb)
            g = sequence_backward(do[q0:q1, h, :], qb, kb, vb, scale, bias, vis)
            dq[q0:q1, h, :] = g[0]
            dk[k0:k1, h, :] = g[1]
            dv[k0:k1, h, :] = g[2]
    return dq, dk, dv


def jagged_bias_grad(dout, q, k, v, q_offsets, kv_offsets, scale, causal, bias_table, bias_center,
                     heads=None):
    """Gradient of sum(dout * out) w.r.t. the relative-position bias table: float64
    [H, num_buckets], summed over every sequence (the table is shared by the batch).
    `heads` optionally restricts it to a subset of heads (other rows NaN)."""
    do, q, k, v = to_f64(dout), to_f64(q), to_f64(k), to_f64(v)
    Tq, H, d = q.shape
    qo = check_offsets(q_offsets, Tq)
    ko = check_offsets(kv_offsets, k.shape[0])
    bt = to_f64(bias_table)
    n = bt.shape[1]
    g = np.full((H, n), np.nan)
    for h in (range(H) if heads is None else heads):
        g[h] = 0.0
        for b in range(qo.size - 1):
            (q0, q1, _, _), qb, kb, vb, bias, vis = _seq_inputs(
                b, h, q, k, v, qo, ko, scale, causal, bt, bias_center)
            ds, _ = sequence_score_grad(do[q0:q1, h, :], qb, kb, vb, scale, bias, vis)
            g[h] += sequence_bias_grad(ds, n, bias_center)
    return g


def jagged_general_bias_grad(dout, q, k, v, q_offsets, kv_offsets, scale, causal, jagged_bias):
    """Gradient of sum(dout * out) w.r.t. a general jagged bias: s_ij depends on its own
    bias element with slope 1, so the gradient of element (h, b, i, j) is dS_ij of that
    sequence and head.  Returned in the bias's own layout [H, plane] (row padding 0)."""
    do, q, k, v = to_f64(dout), to_f64(q), to_f64(k), to_f64(v)
    Tq, H, d = q.shape
    qo = check_offsets(q_offsets, Tq)
    ko = check_offsets(kv_offsets, k.shape[0])
    jb = _jagged_bias_f64(jagged_bias)
    g = np.zeros_like(jb[0])
    for b in range(qo.size - 1):
        Lq, Lk = int(qo[b + 1] - qo[b]), int(ko[b + 1] - ko[b])
        pitch = (Lk + 7) // 8 * 8
        off = int(jb[1][b])
        for h in range(H):
            (q0, q1, _, _), qb, kb, vb, bias, vis = _seq_inputs(
                b, h, q, k, v, qo, ko, scale, causal, None, 0, jb)
            ds, _ = sequence_score_grad(do[q0:q1, h, :], qb, kb, vb, scale, bias, vis)
            blk = g[h, off:off + Lq * pitch].reshape(Lq, pitch)
            blk[:, :Lk] = ds
    return g


def sequence_reference(b, h, q, k, v, q_offsets, kv_offsets, scale, causal=False,
                       bias_table=None, bias_center=0, dout=None, jagged_bias=None):
    """Oracle results for one (sequence, head): (o, lse) and, if dout is given,
    also (dq, dk, dv).  Inputs may be full jagged tensors on any device; only the
    rows of sequence b are copied to the host."""
    qo, ko = to_i64(q_offsets), to_i64(kv_offsets)
    q0, q1, k0, k1 = int(qo[b]), int(qo[b + 1]), int(ko[b]), int(ko[b + 1])
    qb = to_f64(q[q0:q1, h])
    kb = to_f64(k[k0:k1, h])
    vb = to_f64(v[k0:k1, h])
    bias = None
    if bias_table is not None:
        bias = relpos_bias(to_f64(bias_table[h]), q1 - q0, k1 - k0, bias_center)
    elif jagged_bias is not None:
        values, boff = jagged_bias
        off_b = int(to_i64(boff[b:b + 1])[0])
        pitch = (k1 - k0 + 7) // 8 * 8
        bias = jagged_bias_block(to_f64(values[h, off_b:off_b + (q1 - q0) * pitch]), 0, q1 - q0, k1 - k0)
    vis = causal_visible(q1 - q0, k1 - k0) if causal else None
    o, lse = sequence_forward(qb, kb, vb, scale, bias, vis)
    if dout is None:
        return o, lse
    g = sequence_backward(to_f64(dout[q0:q1, h]), qb, kb, vb, scale, bias, vis)
    return (o, lse) + tuple(g)


# ---------------------------------------------------------------------------
# independent formulation 1: brute-force padded dense attention, -inf mask
# ---------------------------------------------------------------------------

def padded_dense_forward(q, k, v, q_offsets, kv_offsets, scale, causal=False,
                         bias_table=None, bias_center=0, jagged_bias=None):
    """Pad every sequence to the batch maximum, build the full [B, H, Lq, Lk]
    score tensor, put -inf on every padded or causally hidden entry, softmax, and
    unpad.  Shares only numpy with the per-sequence path above."""
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    Tq, H, d = q.shape
    qo, ko = to_i64(q_offsets), to_i64(kv_offsets)
    B = qo.size - 1
    Lq = np.diff(qo)
    Lk = np.diff(ko)
    Mq = int(Lq.max()) if B else 0
    Mk = int(Lk.max()) if B else 0
    Qp = np.zeros((B, H, Mq, d))
    Kp = np.zeros((B, H, Mk, d))
    Vp = np.zeros((B, H, Mk, d))
    for b in range(B):
        Qp[b, :, :Lq[b]] = q[qo[b]:qo[b + 1]].transpose(1, 0, 2)
        Kp[b, :, :Lk[b]] = k[ko[b]:ko[b + 1]].transpose(1, 0, 2)
        Vp[b, :, :Lk[b]] = v[ko[b]:ko[b + 1]].transpose(1, 0, 2)
    S = scale * np.einsum("bhid,bhjd->bhij", Qp, Kp)
    ii = np.arange(Mq)[None, :, None]
    jj = np.arange(Mk)[None, None, :]
    if bias_table is not None:
        bt = to_f64(bias_table)
        idx = np.clip(jj[0] - ii[0] + bias_center, 0, bt.shape[1] - 1)   # [Mq, Mk]
        S = S + bt[:, idx][None]
    if jagged_bias is not None:
        # general bias: sequence b's block starts at element boff[b] of each head's plane,
        # rows of round_up(Lk_b, 8) elements; read element by element
        vals, boff = to_f64(jagged_bias[0]), to_i64(jagged_bias[1])
        for b in range(B):
            pitch = -(-int(Lk[b]) // 8) * 8
            for i in range(int(Lq[b])):
                for j in range(int(Lk[b])):
                    S[b, :, i, j] += vals[:, int(boff[b]) + i * pitch + j]
    mask = (ii < Lq[:, None, None]) & (jj < Lk[:, None, None])          # [B, Mq, Mk]
    if causal:
        mask &= jj <= ii + (Lk - Lq)[:, None, None]
    S = np.where(mask[:, None], S, NEG_INF)
    m = S.max(axis=-1, keepdims=True) if Mk else np.full(S.shape[:-1] + (1,), NEG_INF)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    E = np.exp(S - m_safe)
    L = E.sum(axis=-1, keepdims=True)
    P = np.where(L > 0, E / np.where(L > 0, L, 1.0), 0.0)
    O = np.einsum("bhij,bhjd->bhid", P, Vp)
    lse_p = np.where(L[..., 0] > 0, m_safe[..., 0] + np.log(np.where(L[..., 0] > 0, L[..., 0], 1.0)), NEG_INF)
    out = np.zeros((Tq, H, d))
    lse = np.zeros((H, Tq))
    for b in range(B):
        out[qo[b]:qo[b + 1]] = O[b, :, :Lq[b]].transpose(1, 0, 2)
        lse[:, qo[b]:qo[b + 1]] = lse_p[b, :, :Lq[b]]
    return out, lse


# ---------------------------------------------------------------------------
# independent formulation 2: tiled online softmax with the subtraction scheme
# ---------------------------------------------------------------------------

def tiled_subtraction_forward(q, k, v, q_offsets, kv_offsets, scale, causal=False,
                              bias_table=None, bias_center=0, block_n=128):
    """Float64 emulation of the jagged kernel's forward algorithm.

    Per (sequence, head, query row): key/value rows are taken in tiles of
    `block_n`; rows past the sequence end are zeros (what a bounds-clipped tile
    load delivers), so their scores are exactly 0 and bias is not added there.
    The running max m may include those zeros.  The running sum is kept in the
    usual online form, l <- l * exp(m_old - m_new) + sum_j exp(s_j - m_new), and
    on the last tile the n_pad padded columns' contribution n_pad * exp(0 - m)
    is subtracted ("Four generations" item 1: zero-mask, then subtract the extra
    exponents).  Causally hidden entries are -inf (a real mask: causality is not
    a jagged boundary).  Finally O = acc / l and lse = m + log(l).
    """
    q, k, v = to_f64(q), to_f64(k), to_f64(v)
    Tq, H, d = q.shape
    qo, ko = to_i64(q_offsets), to_i64(kv_offsets)
    bt = to_f64(bias_table)
    out = np.zeros((Tq, H, d))
    lse = np.zeros((H, Tq))
    for b in range(qo.size - 1):
        Lq, Lk = int(qo[b + 1] - qo[b]), int(ko[b + 1] - ko[b])
        n_tiles = -(-Lk // block_n)
        Kp = np.zeros((n_tiles * block_n, H, d))
        Vp = np.zeros((n_tiles * block_n, H, d))
        Kp[:Lk] = k[ko[b]:ko[b + 1]]
        Vp[:Lk] = v[ko[b]:ko[b + 1]]
        for h in range(H):
            for i in range(Lq):
                qi = q[qo[b] + i, h]
                m, l, acc = NEG_INF, 0.0, np.zeros(d)
                last_visible = Lk - 1 if not causal else min(Lk - 1, i + Lk - Lq)
                if last_visible < 0:
                    out[qo[b] + i, h] = 0.0
                    lse[h, qo[b] + i] = NEG_INF
                    continue
                t_end = last_visible // block_n + 1
                for t in range(t_end):
                    j = np.arange(t * block_n, (t + 1) * block_n)
                    s = scale * (Kp[j, h] @ qi)
                    real = j < Lk
                    if bt is not None:
                        bidx = np.clip(j - i + bias_center, 0, bt.shape[1] - 1)
                        s = np.where(real, s + bt[h, bidx], s)
                    if causal:
                        s = np.where(j <= i + Lk - Lq, s, NEG_INF)
                    m_new = max(m, s.max())
                    alpha = np.exp(m - m_new) if np.isfinite(m) else 0.0
                    p = np.exp(s - m_new)
                    l = l * alpha + p.sum()
                    acc = acc * alpha + p @ Vp[j, h]
                    m = m_new
                    if t == n_tiles - 1 and not causal:
                        n_pad = int((~real).sum())
                        l -= n_pad * np.exp(0.0 - m)
                out[qo[b] + i, h] = acc / l
                lse[h, qo[b] + i] = m + np.log(l)
    return out, lse
