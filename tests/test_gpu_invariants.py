"""Properties of the CUDA path that hold at any size (applied at the full workload sizes
the benchmark times): every (sequence, head) is computed the same way wherever it sits in
the batch, so permuting the sequences permutes every output bit for bit, and a duplicated
sequence gets bit-identical results (the oracle's invariants, applied to the GPU)."""
import numpy as np
import pytest
import torch

from jagged_attention_recsys_jfa_gb300.inputs import CONFIGS, JaggedBatch, make_batch, offsets_from_lengths
from parity_utils import gpu_run

pytestmark = pytest.mark.gpu


def _reorder(batch, order):
    """The same sequences in the batch order `order` (a list of original indices, repeats
    allowed)."""
    qo = batch.q_offsets.cpu().tolist()
    ko = batch.kv_offsets.cpu().tolist()
    qi = torch.cat([torch.arange(qo[b], qo[b + 1]) for b in order]).to(batch.q.device)
    ki = torch.cat([torch.arange(ko[b], ko[b + 1]) for b in order]).to(batch.k.device)
    lq = batch.q_lengths[order]
    lk = batch.kv_lengths[order]
    dev = batch.q.device
    return JaggedBatch(batch.cfg, lq, lk, offsets_from_lengths(lq).to(dev), offsets_from_lengths(lk).to(dev),
                       batch.q[qi].contiguous(), batch.k[ki].contiguous(), batch.v[ki].contiguous(), batch.bias,
                       batch.dout[qi].contiguous()), qi, ki


@pytest.mark.parametrize("name", ["gem_self", "biased_causal", "longtail_causal"])
def test_permuting_sequences_permutes_results(name):
    batch = make_batch(CONFIGS[name], device="cuda")
    B = batch.q_lengths.numel()
    order = np.random.default_rng(5).permutation(B).tolist()
    pb, qi, ki = _reorder(batch, order)
    a = gpu_run(batch)
    b = gpu_run(pb)
    assert torch.equal(b["out"], a["out"][qi]), "out"
    assert torch.equal(b["lse"], a["lse"][:, qi]), "lse"
    assert torch.equal(b["dq"], a["dq"][qi]), "dq"
    assert torch.equal(b["dk"], a["dk"][ki]), "dk"
    assert torch.equal(b["dv"], a["dv"][ki]), "dv"


def test_duplicated_sequences_get_identical_results():
    batch = make_batch(CONFIGS["cross"], device="cuda", q_lengths=[40, 64, 1, 130, 300],
                       kv_lengths=[900, 257, 3000, 130, 128])
    order = [0, 1, 2, 3, 4, 3, 0, 4, 2]
    db, _, _ = _reorder(batch, order)
    r = gpu_run(db)
    qo = db.q_offsets.cpu().tolist()
    ko = db.kv_offsets.cpu().tolist()
    for first, again in ((3, 5), (0, 6), (4, 7), (2, 8)):
        sq = lambda b: slice(qo[b], qo[b + 1])
        sk = lambda b: slice(ko[b], ko[b + 1])
        for key, sl in (("out", sq), ("dq", sq), ("dk", sk), ("dv", sk)):
            assert torch.equal(r[key][sl(first)], r[key][sl(again)]), (key, first, again)
        assert torch.equal(r["lse"][:, sq(first)], r["lse"][:, sq(again)]), ("lse", first, again)
