"""The forward + backward step captured in a CUDA graph: replays reproduce the eager
results bit for bit, and because the planner reads the offsets on the device, one graph
serves any batch with the same sequence count and token totals (new lengths written into
the captured offset buffers, replayed, checked against an eager run on those lengths)."""
import pytest
import torch

from jagged_attention_recsys_jfa_gb300.inputs import CONFIGS, make_batch
from jagged_attention_recsys_jfa_gb300.jfa import jfa_backward, jfa_check_status, jfa_forward, new_workspace

pytestmark = pytest.mark.gpu


def _eager(batch, q_off, kv_off, causal):
    cfg = batch.cfg
    out, lse, ws = jfa_forward(batch.q, batch.k, batch.v, q_off, kv_off, None, 0, cfg.scale, causal)
    dq, dk, dv, ws2 = jfa_backward(batch.dout, batch.q, batch.k, batch.v, out, lse, q_off, kv_off, None, 0,
                                   cfg.scale, causal)
    assert jfa_check_status(ws) == 0 and jfa_check_status(ws2) == 0
    return out, lse, dq, dk, dv


@pytest.mark.parametrize("causal", [False, True])
def test_graph_replay_matches_eager_and_follows_new_lengths(causal):
    cfg = CONFIGS["tiny"]
    lq, lk = [300, 40, 7, 129], [300, 260, 9, 140]
    batch = make_batch(cfg, device="cuda", q_lengths=lq, kv_lengths=lk)
    B, (Tq, H, d), Tk = len(lq), batch.q.shape, batch.k.shape[0]
    q_off = batch.q_offsets.clone()
    kv_off = batch.kv_offsets.clone()
    ref = _eager(batch, q_off, kv_off, causal)

    out, lse = torch.empty_like(batch.q), torch.empty((H, Tq), dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(batch.q), torch.empty_like(batch.k), torch.empty_like(batch.v)
    ws_f = new_workspace(B, H, d, Tq, Tk, False, "cuda")
    ws_b = new_workspace(B, H, d, Tq, Tk, True, "cuda")

    def step():
        jfa_forward(batch.q, batch.k, batch.v, q_off, kv_off, None, 0, cfg.scale, causal, out=out, lse=lse,
                    workspace=ws_f)
        jfa_backward(batch.dout, batch.q, batch.k, batch.v, out, lse, q_off, kv_off, None, 0, cfg.scale, causal,
                     dq=dq, dk=dk, dv=dv, workspace=ws_b)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # one eager pass on the capture stream before capturing
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert jfa_check_status(ws_f) == 0 and jfa_check_status(ws_b) == 0
    for got, want in zip((out, lse, dq, dk, dv), ref):
        assert torch.equal(got, want)

    # same totals, different split: the captured graph plans the new batch on the device
    lq2, lk2 = [7, 129, 300, 40], [140, 9, 300, 260]
    assert sum(lq2) == Tq and sum(lk2) == Tk
    q_off.copy_(torch.tensor([0] + list(torch.tensor(lq2).cumsum(0)), dtype=torch.int64))
    kv_off.copy_(torch.tensor([0] + list(torch.tensor(lk2).cumsum(0)), dtype=torch.int64))
    graph.replay()
    torch.cuda.synchronize()
    assert jfa_check_status(ws_f) == 0 and jfa_check_status(ws_b) == 0
    ref2 = _eager(batch, q_off, kv_off, causal)
    for got, want in zip((out, lse, dq, dk, dv), ref2):
        assert torch.equal(got, want)
    # and the new results differ from the first batch's (the lengths really changed)
    assert not torch.equal(out, ref[0])
