"""The seeded synthetic inputs (the input recipes of the scoring, LM-head and
attention workloads), checked on small CPU instances: the same seed gives the
same tensors, and each generator produces the structure its recipe states."""
import math

import torch

from logprob_drift_scoring_gb300 import workloads as W


def _same(a, b):
    return torch.equal(a, b)


def test_synthetic_is_seeded_and_shaped():
    a = W.synthetic(300, 777, seed=4, device="cpu", row_pad=5, spike_frac=0.1)
    b = W.synthetic(300, 777, seed=4, device="cpu", row_pad=5, spike_frac=0.1)
    c = W.synthetic(300, 777, seed=5, device="cpu", row_pad=5, spike_frac=0.1)
    for x, y in ((a.train, b.train), (a.rollout, b.rollout), (a.token_ids, b.token_ids), (a.action_mask, b.action_mask)):
        assert _same(x, y)
    assert not _same(a.train, c.train)
    assert a.train.shape == (300, 777) and a.train.stride(0) == 782  # padded rows
    assert a.train.dtype == torch.bfloat16 and a.token_ids.dtype == torch.int32
    assert int(a.token_ids.min()) >= 0 and int(a.token_ids.max()) < 777
    # N(0, 3^2) logits, rollout = train + N(0, (2e-3)^2) rounded to bf16
    x = a.train.float()
    assert 2.8 < float(x[x.abs() < 12].std()) < 3.2
    d = (a.rollout.float() - a.train.float()).abs()
    assert float(d.max()) < 0.1 and float(d.mean()) > 0
    # Bernoulli(0.9) mask
    assert 0.85 < float(a.action_mask.float().mean()) < 0.95
    # 10 % of rows (30) carry a +15 spike on one column: their maximum stands
    # out (a spiked value passes 14 with probability ~0.63), unlike unspiked rows
    plain = W.synthetic(300, 777, seed=4, device="cpu", row_pad=5).train.float()
    assert int((x.max(dim=1).values > 14).sum()) >= 12
    assert int((plain.max(dim=1).values > 14).sum()) <= 2


def test_tiny_recipe():
    w = W.tiny(device="cpu")
    assert w.train.shape == (128, 1024)
    m = w.action_mask.view(2, 64)
    assert int(m[:, :16].sum()) == 0 and int(m[:, 56:].sum()) == 0   # prompt and right padding off
    assert 60 <= int(m.sum()) <= 80                                   # response positions at ~0.9
    assert _same(w.train, W.tiny(device="cpu").train)


def test_head_recipe():
    h = W.head(40, 128, 300, seed=7, device="cpu", active_prob=0.5)
    assert h.hidden_train.shape == (40, 128) and h.weight.shape == (300, 128)
    assert abs(float(h.weight.float().std()) - 0.02) < 0.003
    assert float((h.hidden_rollout.float() - h.hidden_train.float()).abs().max()) < 0.05
    assert _same(h.weight, W.head(40, 128, 300, seed=7, device="cpu", active_prob=0.5).weight)


def test_attention_partials_are_causal_blocks():
    T, H, d, K = 64, 2, 16, 4
    a = W.attn_partials(T, H, d, K, seed=3, device="cpu", masked_fill=float("nan"))
    assert a.out_parts.shape == (K, T * H, d) and a.lse_parts.shape == (K, T * H)
    tok = torch.arange(T).repeat_interleave(H)
    for k in range(K):
        start = k * T // K
        dead = tok < start                      # queries before the block saw none of its keys
        assert bool(torch.all(torch.isinf(a.lse_parts[k][dead]) & (a.lse_parts[k][dead] < 0)))
        assert bool(torch.all(torch.isfinite(a.lse_parts[k][~dead])))
        assert bool(torch.all(torch.isnan(a.out_parts[k][dead])))          # never to be read
        assert bool(torch.all(torch.isfinite(a.out_parts[k][~dead])))
    # about (K - 1) / 2K of the (row, part) pairs have no keys
    frac = float(torch.isinf(a.lse_parts).float().mean())
    assert abs(frac - (K - 1) / (2 * K)) < 0.05
    # base-2 lse is the natural one divided by ln 2, on the same draws
    b = W.attn_partials(T, H, d, K, seed=3, device="cpu", lse_base2=True)
    live = torch.isfinite(a.lse_parts)
    assert torch.allclose(b.lse_parts[live] * math.log(2.0), a.lse_parts[live], rtol=1e-5, atol=1e-5)
