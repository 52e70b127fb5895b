"""Every entry point captured in a CUDA graph (needs a GPU).

The library promises that its calls are asynchronous on the caller's stream
and may be captured.  Each case runs the calls eagerly, captures the same
calls into a graph on static buffers, replays it and requires the replay to
give the eager bits; then it writes new inputs into the captured buffers,
replays again and requires the bits of an eager run on the new inputs (so
nothing the host computed at capture time is baked into the graph).
"""
import pytest
import torch

from logprob_drift_scoring_gb300 import binding as B
from logprob_drift_scoring_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _capture(step):
    """Warm up on a side stream (one-time set-up happens outside capture),
    then capture step() into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    return g


def _check_replays(inputs, fresh_inputs, outputs, step):
    """inputs / fresh_inputs: lists of tensors (the captured buffers and new
    contents for them); outputs: the captured output buffers."""
    step()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outputs]
    g = _capture(step)
    for o in outputs:
        o.fill_(0)  # only the replay can restore them
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(outputs, eager):
        assert torch.equal(a, b)
    for buf, new in zip(inputs, fresh_inputs):
        buf.copy_(new)
    step()
    torch.cuda.synchronize()
    eager2 = [o.clone() for o in outputs]
    assert not all(torch.equal(a, b) for a, b in zip(eager, eager2))
    for o in outputs:
        o.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(outputs, eager2):
        assert torch.equal(a, b)


def test_score_entropy_and_backward_in_a_graph():
    w = W.synthetic(300, 20000, seed=71, device=DEV, active_prob=0.8)
    w2 = W.synthetic(300, 20000, seed=72, device=DEV, active_prob=0.8)
    n = w.n_rows
    outs = [torch.empty(n, dtype=torch.float32, device=DEV) for _ in range(5)]
    met = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=DEV)
    met2 = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=DEV)
    ws = torch.empty(B.lpd_workspace_size(B.LPD_KIND_SCORE, n), dtype=torch.uint8, device=DEV)
    ws2 = torch.empty_like(ws)
    grad = torch.randn(n, device=DEV)
    dlog = torch.empty((n, 20000), dtype=torch.bfloat16, device=DEV)
    ops = [(B.LPD_OP_SOFTCAP, 30.0), (B.LPD_OP_SCALE, 1 / 0.7)]

    def step():
        B.lpd_score(w.train, w.rollout, w.token_ids, w.action_mask, 0.8, 1.2, *outs[:3], met, ws)
        B.lpd_score_entropy(w.train, w.rollout, w.token_ids, w.action_mask, 0.8, 1.2, outs[0], outs[1], outs[2],
                            outs[3], outs[4], met2, ws2)
        B.lpd_logprob_backward(w.train, w.token_ids, w.action_mask, outs[0], grad, dlog)
        B.lpd_score_transformed(w.train, w.rollout, ops, ops, w.token_ids, w.action_mask, 0.8, 1.2, *outs[:3], met,
                                ws)

    _check_replays([w.train, w.rollout, w.token_ids, w.action_mask],
                   [w2.train, w2.rollout, w2.token_ids, w2.action_mask], outs + [met, met2, dlog], step)


def test_attention_merge_and_drift_in_a_graph():
    a = W.attn_partials(300, 8, 128, 8, seed=73, device=DEV)
    a2 = W.attn_partials(300, 8, 128, 8, seed=74, device=DEV)
    n = a.n_rows
    out = torch.empty((n, 128), device=DEV)
    lse = torch.empty(n, device=DEV)
    out_b = torch.empty_like(out)
    lse_b = torch.empty_like(lse)
    rdo, rdl = torch.empty(n, device=DEV), torch.empty(n, device=DEV)
    drift = torch.empty(B.MERGE_DRIFT_BYTES, dtype=torch.uint8, device=DEV)

    def step():
        B.lpd_attn_merge(a.out_parts, a.lse_parts, [3, 1, 0, 2, 7, 6, 5, 4], out, lse)
        B.lpd_attn_merge_order_drift(a.out_parts, a.lse_parts, None, [7, 6, 5, 4, 3, 2, 1, 0], out_b, lse_b, rdo, rdl,
                                     drift)

    _check_replays([a.out_parts, a.lse_parts], [a2.out_parts, a2.lse_parts], [out, lse, out_b, lse_b, rdo, rdl, drift],
                   step)


def test_sharded_topologies_and_union_metrics_in_a_graph():
    base = W.synthetic(200, 12000, seed=75, device=DEV)
    base2 = W.synthetic(200, 12000, seed=76, device=DEV)
    bounds = [(0, 3000), (3000, 7001), (7001, 12000)]
    ts = [base.train[:, lo:hi].contiguous() for lo, hi in bounds]
    rs = [base.rollout[:, lo:hi].contiguous() for lo, hi in bounds]
    ts2 = [base2.train[:, lo:hi].contiguous() for lo, hi in bounds]
    rs2 = [base2.rollout[:, lo:hi].contiguous() for lo, hi in bounds]
    n = base.n_rows
    outs = [[torch.empty(n, device=DEV) for _ in range(3)] for _ in range(3)]
    mets = [torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=DEV) for _ in range(4)]
    wss = [torch.empty(B.lpd_topology_workspace_size(t, n, 12000, 3, B.LPD_BF16, B.LPD_BF16), dtype=torch.uint8,
                       device=DEV) for t in range(3)]
    ws_u = torch.empty(B.lpd_workspace_size(B.LPD_KIND_SCORE, n), dtype=torch.uint8, device=DEV)
    summ = torch.empty(B.LOGP_DRIFT_BYTES, dtype=torch.uint8, device=DEV)

    def step():
        for t in range(3):
            B.lpd_score_sharded_topology(ts, rs, bounds, base.token_ids, base.action_mask, 0.8, 1.2, t, [2, 0, 1],
                                         *outs[t], mets[t], wss[t])
        B.lpd_drift_metrics_from_dlogp(outs[0][2], base.action_mask, 0.8, 1.2, mets[3], ws_u)
        # two arms' per-token results summarised against each other
        B.lpd_logp_drift_summary(outs[0][0], outs[0][1], outs[1][0], outs[1][1], base.action_mask, summ)

    flat = [o for arm in outs for o in arm]
    _check_replays(ts + rs + [base.token_ids], ts2 + rs2 + [base2.token_ids], flat + mets + [summ], step)


def test_fused_head_in_a_graph():
    h = W.head(300, 512, 8192, seed=77, device=DEV)
    h2 = W.head(300, 512, 8192, seed=78, device=DEV)
    n = h.n_rows
    outs = [torch.empty(n, device=DEV) for _ in range(6)]
    met = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=DEV)
    met2 = torch.empty_like(met)
    ws = torch.empty(B.lpd_fused_workspace_size(n, 512, 8192), dtype=torch.uint8, device=DEV)
    ops = [(B.LPD_OP_SCALE, 10.0), (B.LPD_OP_SOFTCAP, 5.0)]

    def step():
        B.lpd_score_fused(h.hidden_train, h.hidden_rollout, h.weight, h.token_ids, h.action_mask, 0.8, 1.2,
                          *outs[:3], met, ws)
        B.lpd_score_fused_transformed(h.hidden_train, h.hidden_rollout, h.weight, ops, ops[::-1], h.token_ids,
                                      h.action_mask, 0.8, 1.2, *outs[3:], met2, ws)

    _check_replays([h.hidden_train, h.hidden_rollout, h.weight, h.token_ids],
                   [h2.hidden_train, h2.hidden_rollout, h2.weight, h2.token_ids], outs + [met, met2], step)
