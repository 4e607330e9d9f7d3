"""Pins for the CPU oracle: each check ties it to something other than itself.

* hand-derived worked examples (tests/golden), closed forms;
* brute-force padded dense attention with a -inf mask;
* torch's own float64 scaled_dot_product_attention (forward and autograd);
* central finite differences of the backward;
* invariants of softmax attention;
* the tiled online softmax with the subtraction correction ("Jagged Flash
  Attention (JFA)", "Four generations" item 1) reproduces exact attention;
* planted mistakes in the oracle are caught by these pins.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle.jfa_oracle as orc

HERE = os.path.dirname(os.path.abspath(__file__))


def rand_batch(rng, lq, lk, H=2, d=8, bias_buckets=0, scale_vals=1.0):
    lq, lk = np.asarray(lq), np.asarray(lk)
    qo = np.concatenate([[0], np.cumsum(lq)]).astype(np.int64)
    ko = np.concatenate([[0], np.cumsum(lk)]).astype(np.int64)
    q = rng.standard_normal((qo[-1], H, d)) * scale_vals
    k = rng.standard_normal((ko[-1], H, d)) * scale_vals
    v = rng.standard_normal((ko[-1], H, d))
    do = rng.standard_normal((qo[-1], H, d))
    bt = rng.standard_normal((H, bias_buckets)) * 0.5 if bias_buckets else None
    return q, k, v, do, qo, ko, bt


CASES = [
    # (lq, lk, causal, bias)
    ([3, 1, 5], [3, 1, 5], False, False),
    ([3, 1, 5], [3, 1, 5], True, False),
    ([4, 2, 6], [7, 1, 3], False, True),
    ([4, 2, 6], [7, 1, 3], True, True),
    ([0, 5, 2], [4, 0, 2], False, False),
    ([0, 5, 2, 3], [4, 0, 2, 3], True, True),
]


# --------------------------------------------------------------------------- golden
def _ev(x):
    return eval(x, {"__builtins__": {}}, {"log": math.log}) if isinstance(x, str) else x


def _arr(x):
    if x is None:
        return None
    return np.vectorize(_ev, otypes=[np.float64])(np.array(x, dtype=object))


@pytest.mark.parametrize("case", json.load(open(os.path.join(HERE, "golden", "worked_examples.json")))["cases"],
                         ids=lambda c: c["name"])
def test_worked_examples(case):
    q, k, v, do = (_arr(case[n]) for n in ("q", "k", "v", "dout"))
    bt = _arr(case["bias_table"])
    args = dict(scale=_ev(case["scale"]), causal=case["causal"], bias_table=bt,
                bias_center=case["bias_center"])
    out, lse = orc.jagged_forward(q, k, v, case["q_offsets"], case["kv_offsets"], **args)
    np.testing.assert_allclose(out, _arr(case["out"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, _arr(case["lse"]), rtol=0, atol=1e-13)
    dq, dk, dv = orc.jagged_backward(do, q, k, v, case["q_offsets"], case["kv_offsets"], **args)
    np.testing.assert_allclose(dq, _arr(case["dq"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, _arr(case["dk"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, _arr(case["dv"]), rtol=0, atol=1e-13)


# --------------------------------------------------------------------------- brute force
@pytest.mark.parametrize("lq,lk,causal,bias", CASES)
def test_matches_padded_dense(lq, lk, causal, bias):
    rng = np.random.default_rng(1)
    q, k, v, _, qo, ko, bt = rand_batch(rng, lq, lk, bias_buckets=16 if bias else 0)
    kw = dict(scale=0.37, causal=causal, bias_table=bt, bias_center=8)
    o1, l1 = orc.jagged_forward(q, k, v, qo, ko, **kw)
    o2, l2 = orc.padded_dense_forward(q, k, v, qo, ko, **kw)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    fin = np.isfinite(l2)
    assert np.array_equal(fin, np.isfinite(l1))
    np.testing.assert_allclose(l1[fin], l2[fin], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- library
def _sdpa_seq(qb, kb, vb, scale, mask):
    """torch float64 SDPA for one sequence, one head; mask bool [Lq, Lk] (True = visible)
    or a float additive matrix, or None."""
    t = lambda a: torch.tensor(a, dtype=torch.float64, requires_grad=True)
    Q, K, V = t(qb[None, None]), t(kb[None, None]), t(vb[None, None])
    attn_mask = None if mask is None else torch.tensor(mask)[None, None]
    o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=attn_mask, scale=scale)
    return Q, K, V, o


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Lq,Lk", [(5, 5), (3, 7), (6, 6), (1, 4)])
def test_matches_torch_sdpa_fwd_bwd(causal, Lq, Lk):
    rng = np.random.default_rng(2)
    d, scale = 6, 0.41
    qb, kb, vb, dob = (rng.standard_normal((n, d)) for n in (Lq, Lk, Lk, Lq))
    mask = torch.ones(Lq, Lk, dtype=torch.bool).tril(diagonal=Lk - Lq).numpy() if causal else None
    Q, K, V, o = _sdpa_seq(qb, kb, vb, scale, mask)
    o.backward(torch.tensor(dob)[None, None])
    vis = orc.causal_visible(Lq, Lk) if causal else None
    o_ref, _ = orc.sequence_forward(qb, kb, vb, scale, None, vis)
    np.testing.assert_allclose(o_ref, o.detach()[0, 0].numpy(), rtol=0, atol=1e-12)
    dq, dk, dv = orc.sequence_backward(dob, qb, kb, vb, scale, None, vis)
    np.testing.assert_allclose(dq, Q.grad[0, 0].numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, K.grad[0, 0].numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, V.grad[0, 0].numpy(), rtol=0, atol=1e-12)


def test_additive_bias_matches_torch_float_mask():
    rng = np.random.default_rng(3)
    Lq, Lk, d, scale = 4, 6, 5, 0.3
    qb, kb, vb, dob = (rng.standard_normal((n, d)) for n in (Lq, Lk, Lk, Lq))
    bias = rng.standard_normal((Lq, Lk))
    Q, K, V, o = _sdpa_seq(qb, kb, vb, scale, bias)
    o.backward(torch.tensor(dob)[None, None])
    o_ref, lse = orc.sequence_forward(qb, kb, vb, scale, bias, None)
    np.testing.assert_allclose(o_ref, o.detach()[0, 0].numpy(), rtol=0, atol=1e-12)
    dq, dk, dv = orc.sequence_backward(dob, qb, kb, vb, scale, bias, None)
    np.testing.assert_allclose(dq, Q.grad[0, 0].numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, K.grad[0, 0].numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, V.grad[0, 0].numpy(), rtol=0, atol=1e-12)
    # lse is the natural log-sum-exp of the scaled, biased scores
    ref = torch.logsumexp(torch.tensor(scale * qb @ kb.T + bias), dim=1).numpy()
    np.testing.assert_allclose(lse, ref, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- finite differences
def _objective(q, k, v, do, qo, ko, kw):
    out, _ = orc.jagged_forward(q, k, v, qo, ko, **kw)
    return float(np.sum(do * out))


@pytest.mark.parametrize("lq,lk,causal,bias", [
    ([2, 5], [3, 4], False, True),
    ([4, 3], [2, 3], True, True),
    ([3, 1], [3, 1], True, False),
])
def test_backward_finite_differences(lq, lk, causal, bias):
    rng = np.random.default_rng(4)
    q, k, v, do, qo, ko, bt = rand_batch(rng, lq, lk, H=2, d=4, bias_buckets=12 if bias else 0)
    kw = dict(scale=0.7, causal=causal, bias_table=bt, bias_center=6)
    grads = orc.jagged_backward(do, q, k, v, qo, ko, **kw)
    eps = 1e-6
    for which, g in zip(range(3), grads):
        num = np.zeros_like(g)
        base = [q, k, v]
        it = np.nditer(base[which], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [a.copy() for a in base]
            minus = [a.copy() for a in base]
            plus[which][idx] += eps
            minus[which][idx] -= eps
            num[idx] = (_objective(*plus, do, qo, ko, kw) - _objective(*minus, do, qo, ko, kw)) / (2 * eps)
        rel = np.linalg.norm(num - g) / max(np.linalg.norm(g), 1e-30)
        assert rel <= 1e-7, (which, rel)


@pytest.mark.parametrize("lq,lk,causal,nb,center", [
    ([2, 5], [3, 4], False, 12, 6),   # every relative position has its own bucket
    ([4, 3], [2, 3], True, 12, 6),
    ([2, 5], [3, 4], False, 5, 2),    # |j - i| > 2 clamps onto the edge buckets
    ([4, 3, 0], [6, 3, 2], True, 4, 1),
])
def test_bias_grad_finite_differences(lq, lk, causal, nb, center):
    """The table gradient against central differences of sum(dout * out) in float64."""
    rng = np.random.default_rng(8)
    q, k, v, do, qo, ko, bt = rand_batch(rng, lq, lk, H=2, d=4, bias_buckets=nb)
    kw = dict(scale=0.7, causal=causal, bias_table=bt, bias_center=center)
    g = orc.jagged_bias_grad(do, q, k, v, qo, ko, 0.7, causal, bt, center)
    eps = 1e-6
    num = np.zeros_like(g)
    for idx in np.ndindex(*bt.shape):
        plus, minus = bt.copy(), bt.copy()
        plus[idx] += eps
        minus[idx] -= eps
        num[idx] = (_objective(q, k, v, do, qo, ko, dict(kw, bias_table=plus))
                    - _objective(q, k, v, do, qo, ko, dict(kw, bias_table=minus))) / (2 * eps)
    rel = np.linalg.norm(num - g) / max(np.linalg.norm(g), 1e-30)
    assert rel <= 1e-7, rel


def test_bias_grad_two_keys_closed_form():
    """One query, two keys: softmax over two scores has dP_0 - dP_1 as its only
    direction, so the two buckets get +-P_0 P_1 (dO.v_0 - dO.v_1)."""
    rng = np.random.default_rng(9)
    q, k, v, do, qo, ko, bt = rand_batch(rng, [1], [2], H=1, d=5, bias_buckets=7)
    scale, center = 0.9, 3
    g = orc.jagged_bias_grad(do, q, k, v, qo, ko, scale, False, bt, center)
    s0 = scale * q[0, 0] @ k[0, 0] + bt[0, center]
    s1 = scale * q[0, 0] @ k[1, 0] + bt[0, center + 1]
    p0 = 1.0 / (1.0 + math.exp(s1 - s0))
    want = p0 * (1.0 - p0) * (do[0, 0] @ v[0, 0] - do[0, 0] @ v[1, 0])
    expect = np.zeros(7)
    expect[center], expect[center + 1] = want, -want
    np.testing.assert_allclose(g[0], expect, rtol=1e-12, atol=1e-15)


def test_bias_grad_sums_to_zero_per_head():
    """Adding one constant to a whole table row leaves every output unchanged (softmax
    shift invariance), so each head's gradient entries sum to zero."""
    rng = np.random.default_rng(10)
    q, k, v, do, qo, ko, bt = rand_batch(rng, [9, 1, 0, 17], [12, 4, 3, 17], H=3, d=6, bias_buckets=20)
    for causal in (False, True):
        g = orc.jagged_bias_grad(do, q, k, v, qo, ko, 0.5, causal, bt, 10)
        for h in range(3):
            assert abs(g[h].sum()) <= 1e-12 * max(np.abs(g[h]).sum(), 1.0), (causal, h, g[h].sum())
            assert np.abs(g[h]).sum() > 1e-3


def _pack_jagged_bias(blocks, lq, lk, H):
    """Lay per-sequence [H, Lq, Lk] bias blocks out in the packed format (rows padded to a
    multiple of 8, blocks back to back), element by element."""
    pitch = [(int(b) + 7) // 8 * 8 for b in lk]
    off = np.concatenate([[0], np.cumsum([int(a) * p for a, p in zip(lq, pitch)])]).astype(np.int64)
    vals = np.full((H, int(off[-1])), np.nan)   # padding columns must never be read
    for b, blk in enumerate(blocks):
        for h in range(H):
            for i in range(int(lq[b])):
                for j in range(int(lk[b])):
                    vals[h, off[b] + i * pitch[b] + j] = blk[h, i, j]
    return vals, off


@pytest.mark.parametrize("lq,lk,causal", [
    ([3, 1, 5], [3, 1, 5], False),
    ([4, 2, 6], [7, 1, 3], True),
    ([0, 5, 2, 9], [4, 0, 2, 11], False),
    ([0, 5, 2, 9], [4, 0, 2, 11], True),
])
def test_jagged_bias_matches_padded_dense(lq, lk, causal):
    """The general bias read through the oracle's block layout against the padded dense
    formulation, which reads the packed values element by element."""
    rng = np.random.default_rng(11)
    q, k, v, _, qo, ko, _ = rand_batch(rng, lq, lk)
    H = q.shape[1]
    vals, off = _pack_jagged_bias([rng.standard_normal((H, a, b)) for a, b in zip(lq, lk)], lq, lk, H)
    jb = (np.nan_to_num(vals, nan=1e300), off)   # a padding read would show up as a huge score
    kw = dict(scale=0.37, causal=causal, jagged_bias=jb)
    o1, l1 = orc.jagged_forward(q, k, v, qo, ko, **kw)
    o2, l2 = orc.padded_dense_forward(q, k, v, qo, ko, **kw)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)
    fin = np.isfinite(l2)
    assert np.array_equal(fin, np.isfinite(l1))
    np.testing.assert_allclose(l1[fin], l2[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_jagged_bias_equal_to_relpos_table(causal):
    """A general bias whose blocks hold the relative-position lookup gives the relative-
    position results exactly (forward and backward)."""
    rng = np.random.default_rng(12)
    lq, lk = [6, 2, 9], [5, 4, 9]
    q, k, v, do, qo, ko, bt = rand_batch(rng, lq, lk, bias_buckets=9)
    center = 4
    H = q.shape[1]
    blocks = []
    for a, b in zip(lq, lk):
        blk = np.zeros((H, a, b))
        for i in range(a):
            for j in range(b):
                blk[:, i, j] = bt[:, min(max(j - i + center, 0), 8)]
        blocks.append(blk)
    jb = _pack_jagged_bias(blocks, lq, lk, H)
    jb = (np.nan_to_num(jb[0], nan=1e300), jb[1])
    r1 = orc.jagged_forward(q, k, v, qo, ko, 0.5, causal, bias_table=bt, bias_center=center)
    r2 = orc.jagged_forward(q, k, v, qo, ko, 0.5, causal, jagged_bias=jb)
    for a, b in zip(r1, r2):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)
    g1 = orc.jagged_backward(do, q, k, v, qo, ko, 0.5, causal, bias_table=bt, bias_center=center)
    g2 = orc.jagged_backward(do, q, k, v, qo, ko, 0.5, causal, jagged_bias=jb)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_general_bias_grad_finite_differences(causal):
    """The general bias's gradient against central differences of sum(dout * out) with
    respect to every stored element (padding elements have gradient 0)."""
    rng = np.random.default_rng(13)
    lq, lk = [3, 0, 4], [5, 2, 4]
    q, k, v, do, qo, ko, _ = rand_batch(rng, lq, lk, H=2, d=4)
    H = q.shape[1]
    vals, off = _pack_jagged_bias([rng.standard_normal((H, a, b)) for a, b in zip(lq, lk)], lq, lk, H)
    vals = np.nan_to_num(vals, nan=0.0)
    g = orc.jagged_general_bias_grad(do, q, k, v, qo, ko, 0.6, causal, (vals, off))
    eps = 1e-6
    num = np.zeros_like(vals)
    kw = lambda vv: dict(scale=0.6, causal=causal, jagged_bias=(vv, off))
    for idx in np.ndindex(*vals.shape):
        plus, minus = vals.copy(), vals.copy()
        plus[idx] += eps
        minus[idx] -= eps
        num[idx] = (_objective(q, k, v, do, qo, ko, kw(plus)) - _objective(q, k, v, do, qo, ko, kw(minus))) / (2 * eps)
    rel = np.linalg.norm(num - g) / max(np.linalg.norm(g), 1e-30)
    assert rel <= 1e-7, rel
    if causal:   # hidden pairs do not move the output: sequence 0 (3 x 5), row 0 sees keys 0..2
        assert np.abs(g[:, int(off[0]) + 3:int(off[0]) + 5]).max() == 0.0


# --------------------------------------------------------------------------- one-pair entry point
@pytest.mark.parametrize("bias_kind", ["none", "table", "general"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("as_torch", [False, True])
def test_sequence_reference_matches_jagged_front_ends(bias_kind, causal, as_torch):
    """`sequence_reference` (the per-(sequence, head) entry point that checks the full-size
    GPU runs and times the CPU baseline) slices q, k, v, dout and the bias on its own.  Its
    results must be exactly the matching slices of `jagged_forward` / `jagged_backward`, for
    every sequence and head: empty query and key sequences, one-key rows, Lq != Lk (causal
    rows that see no key), a table small enough that the bucket clamp fires, and a general
    bias whose row padding holds huge values that a mis-sliced block would pick up.  Inputs
    are passed both as numpy arrays and as the bf16 torch tensors the GPU tests hand it."""
    rng = np.random.default_rng(21)
    lq, lk = [0, 5, 1, 9, 4, 3], [3, 0, 1, 11, 2, 3]
    q, k, v, do, qo, ko, bt = rand_batch(rng, lq, lk, H=3, d=8, bias_buckets=7 if bias_kind == "table" else 0)
    H = q.shape[1]
    jb = None
    if bias_kind == "general":
        vals, off = _pack_jagged_bias([rng.standard_normal((H, a, b)) for a, b in zip(lq, lk)], lq, lk, H)
        jb = (np.nan_to_num(vals, nan=1e300), off)
    if as_torch:
        bf = lambda x: torch.from_numpy(x).to(torch.bfloat16)
        q, k, v, do = bf(q), bf(k), bf(v), bf(do)
        bt = torch.from_numpy(bt).float() if bt is not None else None
        qo, ko = torch.from_numpy(qo), torch.from_numpy(ko)
        if jb is not None:   # bf16 rounds 1e300 to inf: padding reads would give NaN / inf
            jb = (bf(jb[0]), torch.from_numpy(jb[1]))
    kw = dict(scale=0.41, causal=causal, bias_table=bt, bias_center=3, jagged_bias=jb)
    out, lse = orc.jagged_forward(q, k, v, qo, ko, **kw)
    dq, dk, dv = orc.jagged_backward(do, q, k, v, qo, ko, **kw)
    qo_, ko_ = orc.to_i64(qo), orc.to_i64(ko)
    for b in range(len(lq)):
        sq, sk = slice(qo_[b], qo_[b + 1]), slice(ko_[b], ko_[b + 1])
        for h in range(H):
            o1, l1, dq1, dk1, dv1 = orc.sequence_reference(b, h, q, k, v, qo, ko, 0.41, causal, bt, 3, dout=do,
                                                           jagged_bias=jb)
            assert o1.shape == (lq[b], q.shape[2]) and dk1.shape == (lk[b], q.shape[2])
            np.testing.assert_allclose(o1, out[sq, h], rtol=0, atol=1e-13)
            fin = np.isfinite(lse[h, sq])
            assert np.array_equal(fin, np.isfinite(l1))
            np.testing.assert_allclose(l1[fin], lse[h, sq][fin], rtol=0, atol=1e-13)
            np.testing.assert_allclose(dq1, dq[sq, h], rtol=0, atol=1e-13)
            np.testing.assert_allclose(dk1, dk[sk, h], rtol=0, atol=1e-13)
            np.testing.assert_allclose(dv1, dv[sk, h], rtol=0, atol=1e-13)
            o2, l2 = orc.sequence_reference(b, h, q, k, v, qo, ko, 0.41, causal, bt, 3, jagged_bias=jb)
            assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    # the pin bites: a sequence_reference that reads its general-bias block one row off
    # (or a table with the wrong center) no longer matches
    if bias_kind != "none":
        b, h = 3, 1
        shifted = dict(bias_table=bt, bias_center=4) if bias_kind == "table" else dict(
            jagged_bias=(jb[0], (orc.to_i64(jb[1]) + 16)))
        o_bad, _ = orc.sequence_reference(b, h, q, k, v, qo, ko, 0.41, causal, dout=None,
                                          **{"bias_table": None, "bias_center": 3, **shifted})
        assert not np.allclose(o_bad, out[qo_[b]:qo_[b + 1], h], rtol=0, atol=1e-6)


# --------------------------------------------------------------------------- invariants
def test_rows_sum_to_one_and_D_identity():
    rng = np.random.default_rng(5)
    Lq, Lk, d = 5, 9, 4
    qb, kb, vb, dob = (rng.standard_normal((n, d)) for n in (Lq, Lk, Lk, Lq))
    vis = orc.causal_visible(Lq, Lk)
    s = orc.sequence_scores(qb, kb, 0.5, None, vis)
    p, _ = orc.softmax_rows(s)
    np.testing.assert_allclose(p.sum(1), 1.0, atol=1e-14)
    assert np.all(p[~vis] == 0)
    o = p @ vb
    dp = dob @ vb.T
    np.testing.assert_allclose((dob * o).sum(1), (p * dp).sum(1), atol=1e-13)


def test_constant_v_gives_constant_output():
    rng = np.random.default_rng(6)
    q, k, v, _, qo, ko, bt = rand_batch(rng, [3, 7], [5, 2], bias_buckets=16)
    c = rng.standard_normal(v.shape[1:])
    v[:] = c
    out, _ = orc.jagged_forward(q, k, v, qo, ko, 0.8, causal=False, bias_table=bt, bias_center=8)
    np.testing.assert_allclose(out, np.broadcast_to(c, out.shape), atol=1e-13)


def test_single_key_closed_form():
    rng = np.random.default_rng(7)
    Lq, d, scale = 4, 5, 0.3
    qb, dob = rng.standard_normal((Lq, d)), rng.standard_normal((Lq, d))
    kb, vb = rng.standard_normal((1, d)), rng.standard_normal((1, d))
    o, lse = orc.sequence_forward(qb, kb, vb, scale)
    np.testing.assert_allclose(o, np.repeat(vb, Lq, 0), atol=1e-14)
    np.testing.assert_allclose(lse, scale * (qb @ kb[0]), atol=1e-14)
    dq, dk, dv = orc.sequence_backward(dob, qb, kb, vb, scale)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    np.testing.assert_allclose(dv[0], dob.sum(0), atol=1e-13)


def test_key_permutation_invariance():
    rng = np.random.default_rng(8)
    Lq, Lk, d = 4, 9, 6
    qb, kb, vb = (rng.standard_normal((n, d)) for n in (Lq, Lk, Lk))
    bias = rng.standard_normal((Lq, Lk))
    perm = rng.permutation(Lk)
    o1, l1 = orc.sequence_forward(qb, kb, vb, 0.5, bias)
    o2, l2 = orc.sequence_forward(qb, kb[perm], vb[perm], 0.5, bias[:, perm])
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_sequence_permutation_and_duplication():
    rng = np.random.default_rng(9)
    lq, lk = [3, 5, 2], [4, 1, 6]
    q, k, v, _, qo, ko, bt = rand_batch(rng, lq, lk, bias_buckets=16)
    kw = dict(scale=0.6, causal=True, bias_table=bt, bias_center=8)
    o, l = orc.jagged_forward(q, k, v, qo, ko, **kw)
    order = [2, 0, 2, 1]
    cat = lambda x, off: np.concatenate([x[off[b]:off[b + 1]] for b in order])
    lq2 = [lq[b] for b in order]
    lk2 = [lk[b] for b in order]
    qo2 = np.concatenate([[0], np.cumsum(lq2)])
    ko2 = np.concatenate([[0], np.cumsum(lk2)])
    o2, l2 = orc.jagged_forward(cat(q, qo), cat(k, ko), cat(v, ko), qo2, ko2, **kw)
    np.testing.assert_allclose(o2, cat(o, qo), atol=1e-14)
    np.testing.assert_allclose(l2, np.concatenate([l[:, qo[b]:qo[b + 1]] for b in order], 1), atol=1e-14)


def test_zero_scale_gives_mean_of_visible_values():
    rng = np.random.default_rng(10)
    Lq, Lk, d = 3, 5, 4
    qb, kb, vb = (rng.standard_normal((n, d)) for n in (Lq, Lk, Lk))
    o, lse = orc.sequence_forward(qb, kb, vb, 0.0)
    np.testing.assert_allclose(o, np.repeat(vb.mean(0, keepdims=True), Lq, 0), atol=1e-14)
    np.testing.assert_allclose(lse, math.log(Lk), atol=1e-14)
    vis = orc.causal_visible(Lq, Lk)    # row i sees the first i + 3 keys
    o, lse = orc.sequence_forward(qb, kb, vb, 0.0, None, vis)
    for i in range(Lq):
        np.testing.assert_allclose(o[i], vb[:i + 3].mean(0), atol=1e-14)
        assert abs(lse[i] - math.log(i + 3)) < 1e-14


def test_constant_bias_shifts_only_lse():
    rng = np.random.default_rng(11)
    q, k, v, _, qo, ko, _ = rand_batch(rng, [4, 3], [6, 2])
    bt = np.full((2, 16), 1.75)
    o1, l1 = orc.jagged_forward(q, k, v, qo, ko, 0.5)
    o2, l2 = orc.jagged_forward(q, k, v, qo, ko, 0.5, bias_table=bt, bias_center=8)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l2 - l1, 1.75, atol=1e-13)


@pytest.mark.parametrize("delta", [-2, 0, 1, 3])
def test_one_hot_bias_selects_relative_position(delta):
    """A dominant bias at bucket center+delta makes query i attend to key i+delta
    (bucket = j - i + center): pins the sign, the index and the center."""
    rng = np.random.default_rng(12)
    L, d, center = 7, 3, 10
    q, k, v, _, qo, ko, _ = rand_batch(rng, [L], [L], H=1, d=d)
    bt = np.zeros((1, 21))
    bt[0, center + delta] = 200.0
    out, lse = orc.jagged_forward(q, k, v, qo, ko, 0.1, bias_table=bt, bias_center=center)
    for i in range(L):
        j = i + delta
        if 0 <= j < L:
            np.testing.assert_allclose(out[i, 0], v[j, 0], atol=1e-12)


def test_bias_bucket_clamps_at_table_edges():
    rng = np.random.default_rng(13)
    L, center = 9, 2
    q, k, v, _, qo, ko, _ = rand_batch(rng, [L], [L], H=1, d=2)
    bt = np.zeros((1, 5))
    bt[0, 4] = 300.0     # last bucket: every j - i + 2 >= 4, i.e. j >= i + 2
    out, _ = orc.jagged_forward(q, k, v, qo, ko, 0.0, bias_table=bt, bias_center=center)
    for i in range(L):
        js = [j for j in range(L) if j - i + center >= 4]
        if js:
            np.testing.assert_allclose(out[i, 0], v[js, 0].mean(0), atol=1e-12)


def test_causal_bottom_right_closed_forms():
    rng = np.random.default_rng(14)
    d, scale = 3, 0.9
    # Lq > Lk: the first Lq - Lk rows see nothing.
    qb, kb, vb, dob = rng.standard_normal((3, d)), rng.standard_normal((1, d)), \
        rng.standard_normal((1, d)), rng.standard_normal((3, d))
    vis = orc.causal_visible(3, 1)
    o, lse = orc.sequence_forward(qb, kb, vb, scale, None, vis)
    assert np.all(o[:2] == 0) and np.all(np.isneginf(lse[:2]))
    np.testing.assert_allclose(o[2], vb[0], atol=1e-14)
    np.testing.assert_allclose(lse[2], scale * qb[2] @ kb[0], atol=1e-14)
    dq, dk, dv = orc.sequence_backward(dob, qb, kb, vb, scale, None, vis)
    assert np.all(dq[:2] == 0)
    np.testing.assert_allclose(dv[0], dob[2], atol=1e-14)
    # Lq < Lk: the last query row sees every key, exactly like non-causal.
    qb, kb, vb = rng.standard_normal((2, d)), rng.standard_normal((5, d)), rng.standard_normal((5, d))
    o_c, _ = orc.sequence_forward(qb, kb, vb, scale, None, orc.causal_visible(2, 5))
    o_n, _ = orc.sequence_forward(qb, kb, vb, scale)
    np.testing.assert_allclose(o_c[1], o_n[1], atol=1e-14)
    o_first, _ = orc.sequence_forward(qb[:1], kb[:4], vb[:4], scale)
    np.testing.assert_allclose(o_c[0], o_first[0], atol=1e-14)


def test_empty_sequences():
    rng = np.random.default_rng(15)
    q, k, v, do, qo, ko, _ = rand_batch(rng, [0, 3, 2], [2, 0, 3])
    out, lse = orc.jagged_forward(q, k, v, qo, ko, 0.5)
    assert np.all(out[0:3] == 0) and np.all(np.isneginf(lse[:, 0:3]))
    dq, dk, dv = orc.jagged_backward(do, q, k, v, qo, ko, 0.5)
    assert np.all(dq[0:3] == 0)
    assert np.all(dk[0:2] == 0) and np.all(dv[0:2] == 0)   # keys of seq 0 have no queries


def test_offsets_validation():
    q = np.zeros((3, 1, 2))
    with pytest.raises(ValueError):
        orc.jagged_forward(q, q, q, [0, 2, 1], [0, 1, 3], 1.0)
    with pytest.raises(ValueError):
        orc.jagged_forward(q, q, q, [1, 3], [0, 3], 1.0)


# --------------------------------------------------------------------------- subtraction scheme
@pytest.mark.parametrize("lq,lk,causal,bias", [
    ([1, 127, 128, 129], [1, 127, 128, 129], False, False),
    ([129, 3], [257, 255], False, True),
    ([130, 5], [130, 5], True, True),
    ([40, 200], [300, 7], True, False),
    ([0, 2, 3], [5, 0, 256], False, False),
])
def test_subtraction_scheme_is_exact(lq, lk, causal, bias):
    rng = np.random.default_rng(16)
    q, k, v, _, qo, ko, bt = rand_batch(rng, lq, lk, H=1, d=8, bias_buckets=1024 if bias else 0)
    kw = dict(scale=0.35, causal=causal, bias_table=bt, bias_center=512)
    o1, l1 = orc.jagged_forward(q, k, v, qo, ko, **kw)
    o2, l2 = orc.tiled_subtraction_forward(q, k, v, qo, ko, **kw)
    np.testing.assert_allclose(o2, o1, rtol=0, atol=1e-12)
    fin = np.isfinite(l1)
    assert np.array_equal(fin, np.isfinite(l2))
    np.testing.assert_allclose(l2[fin], l1[fin], rtol=0, atol=1e-12)


# --------------------------------------------------------------------------- planted mistakes
def _pins_pass(fn):
    try:
        fn()
        return True
    except AssertionError:
        return False


def test_planted_mistakes_are_caught(monkeypatch):
    golden = json.load(open(os.path.join(HERE, "golden", "worked_examples.json")))["cases"]

    def all_pins():
        for c in golden:
            test_worked_examples(c)
        for delta in (-2, 1):
            test_one_hot_bias_selects_relative_position(delta)
        test_backward_finite_differences([2, 5], [3, 4], False, True)
        test_bias_grad_finite_differences([2, 5], [3, 4], False, 5, 2)
        test_causal_bottom_right_closed_forms()
        test_matches_torch_sdpa_fwd_bwd(True, 3, 7)

    assert _pins_pass(all_pins)

    orig_bias = orc.relpos_bias
    orig_vis = orc.causal_visible
    orig_bwd = orc.sequence_backward
    orig_scores = orc.sequence_scores
    orig_bgrad = orc.sequence_bias_grad

    mutants = {
        "bias index i - j": lambda: monkeypatch.setattr(
            orc, "relpos_bias", lambda t, Lq, Lk, c: orig_bias(t, Lk, Lq, c).T if Lq and Lk else orig_bias(t, Lq, Lk, c)),
        "top-left causal": lambda: monkeypatch.setattr(
            orc, "causal_visible", lambda Lq, Lk: np.arange(Lk)[None, :] <= np.arange(Lq)[:, None]),
        "dK without scale": lambda: monkeypatch.setattr(
            orc, "sequence_backward",
            lambda do, q, k, v, s, b=None, vis=None: (lambda g: (g[0], g[1] / s if s else g[1], g[2]))(
                orig_bwd(do, q, k, v, s, b, vis))),
        "bias scaled too": lambda: monkeypatch.setattr(
            orc, "sequence_scores",
            lambda q, k, s, b=None, vis=None: orig_scores(q, k, s, None if b is None else s * b, vis)),
        "bias grad bucket i - j": lambda: monkeypatch.setattr(
            orc, "sequence_bias_grad",
            lambda ds, n, c: orig_bgrad(ds.T, n, c) if ds.size else orig_bgrad(ds, n, c)),
        "bias grad without clamp merge": lambda: monkeypatch.setattr(
            orc, "sequence_bias_grad", lambda ds, n, c: _bias_grad_drop_clamped(ds, n, c)),
        "dropped D term": lambda: monkeypatch.setattr(
            orc, "sequence_backward",
            lambda do, q, k, v, s, b=None, vis=None: _bwd_without_D(orig_scores, do, q, k, v, s, b, vis)),
    }
    for name, plant in mutants.items():
        monkeypatch.undo()
        plant()
        assert not _pins_pass(all_pins), f"planted mistake not caught: {name}"
    monkeypatch.undo()
    assert _pins_pass(all_pins)


def _bwd_without_D(scores, do, q, k, v, s, b, vis):
    p, _ = orc.softmax_rows(scores(q, k, s, b, vis))
    ds = p * (do @ v.T)
    return s * ds @ k, s * ds.T @ q, p.T @ do


def _bias_grad_drop_clamped(ds, n, c):
    """Planted mistake: pairs whose relative position falls outside the table are dropped
    instead of landing on the edge buckets."""
    Lq, Lk = ds.shape
    rel = np.arange(Lk)[None, :] - np.arange(Lq)[:, None] + c
    keep = (rel >= 0) & (rel < n)
    g = np.zeros(n)
    np.add.at(g, rel[keep], ds[keep])
    return g
