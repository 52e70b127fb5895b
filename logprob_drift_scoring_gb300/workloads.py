"""Seeded synthetic inputs for the scorer, shaped like the workloads the drift
contract is run on.  This module draws random numbers and lays out tensors;
it contains none of the scoring arithmetic, and serves the tests, the
benchmark and the CPU oracle alike.

The pages measure on a real Qwen3-8B rollout ("WS2 Cross-Config Logprob Drift
Contract", section "Revised Modular PR Roadmap", M1; "Attention Debug
Matrix"); no checkpoint or dataset is used here.  Random logits of the same
shapes, dtypes, vocab sizes, padding layouts and masks stand in for it:

  tiny     B=2 x T=64, V=1024, bf16 N(0, 2^2); prompt 16, right pad 8; the
           response positions are active with probability 0.9; rollout =
           bf16(train + N(0, 1e-3^2)); ids uniform.
  qwen     B=8 x T=4096, V=151936, bf16 N(0, 3^2); 1% of rows get +15 on one
           uniform column (before rounding); prompt U{256..1024}, right pad
           U{0..512}; every response token active; rollout = bf16(train +
           N(0, 2e-3^2)); ids uniform.
  llama    B=64 x T=1024, V=128256; train bf16 N(0, 3^2); rollout fp32 =
           train + N(0, 1e-3^2) (not rounded); left pad U{0..512}, then prompt
           U{64..256}, then response (active); ids sampled from the train
           row's softmax by the Gumbel-max trick (teacher-forced sampling).
  sharded  B=1 x T=32768, V=151936 as 4 contiguous vocab shards of 37984
           columns per side, bf16 N(0, 3^2); rollout = bf16(train + N(0,
           2e-3^2)); all rows active; ids uniform.
  fused    LM head: hidden [16384, 4096] bf16 N(0, 1), W [151936, 4096] bf16
           N(0, 0.02^2), rollout hidden = bf16(hidden + N(0, 1e-3^2)); all
           rows active; ids uniform.
  attn     attention partials of a context-parallel causal prefill: T=32768
           tokens x 32 query heads (Qwen3-8B), head_dim 128, keys split into
           K=8 contiguous blocks of T/K.  Row = (token t, head h), token-major.
           Part k saw n_k = |block k intersect [0, t]| keys: lse_k = log(n_k)
           + N(2, 1^2) when n_k > 0, else -inf (and its out is 0, as many
           kernels leave it); out_k N(0, 0.5^2) f32.  About (K-1)/2K of the
           (row, part) pairs have no keys.

Noise scales are standard deviations.  Generation runs on the target device
with a seeded torch.Generator; large tensors are generated in row chunks.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

CLIP = (0.8, 1.2)


@dataclass
class Workload:
    name: str
    train: object              # Tensor [R, V] (or list of shard tensors)
    rollout: object
    token_ids: torch.Tensor    # int32 [R]
    action_mask: torch.Tensor  # uint8 [R]
    vocab: int
    clip: tuple = CLIP
    v_ranges: list | None = None
    meta: dict = field(default_factory=dict)

    @property
    def n_rows(self) -> int:
        return int(self.token_ids.shape[0])

    def logits_bytes(self) -> int:
        ts = self.train if isinstance(self.train, list) else [self.train]
        rs = self.rollout if isinstance(self.rollout, list) else [self.rollout]
        return sum(t.numel() * t.element_size() for t in ts + rs)


def _gen(device, seed: int) -> torch.Generator:
    return torch.Generator(device=torch.device(device)).manual_seed(seed)


def _chunk_rows(vocab: int, budget_elems: int = 1 << 28) -> int:
    return max(1, budget_elems // max(vocab, 1))


def _fill_noisy(train_f32: torch.Tensor, sigma_noise: float, g, out_dtype) -> torch.Tensor:
    noise = torch.randn(train_f32.shape, generator=g, device=train_f32.device, dtype=torch.float32)
    return (train_f32 + sigma_noise * noise).to(out_dtype)


def synthetic(n_rows: int, vocab: int, *, seed: int = 0, device="cpu", dtype_train=torch.bfloat16,
              dtype_rollout=torch.bfloat16, sigma: float = 3.0, rollout_noise: float = 2e-3,
              active_prob: float = 0.9, row_pad: int = 0, spike_frac: float = 0.0,
              spike: float = 15.0) -> Workload:
    """Generic seeded case: rows of N(0, sigma^2) logits, rollout = train plus
    N(0, rollout_noise^2) in the rollout dtype, Bernoulli(active_prob) mask,
    uniform ids.  row_pad > 0 stores each row with that many extra columns
    (row stride vocab + row_pad) holding garbage that must never be read."""
    g = _gen(device, seed)
    stride = vocab + row_pad
    train = torch.empty((n_rows, stride), dtype=dtype_train, device=device)
    rollout = torch.empty((n_rows, stride), dtype=dtype_rollout, device=device)
    n_spike = int(round(spike_frac * n_rows))
    spike_rows = torch.randperm(n_rows, generator=g, device=device)[:n_spike]
    spike_cols = torch.randint(0, vocab, (n_spike,), generator=g, device=device)
    step = _chunk_rows(stride)
    for c in range(0, n_rows, step):
        n = min(step, n_rows - c)
        x = sigma * torch.randn((n, stride), generator=g, device=device, dtype=torch.float32)
        sel = (spike_rows >= c) & (spike_rows < c + n)
        if bool(sel.any()):
            x[spike_rows[sel] - c, spike_cols[sel]] += spike
        tc = x.to(dtype_train)
        train[c:c + n] = tc
        rollout[c:c + n] = _fill_noisy(tc.float(), rollout_noise, g, dtype_rollout)
    if row_pad:
        # the padding columns hold values that would dominate any sum that read them
        train[:, vocab:] = 1e4
        rollout[:, vocab:] = -1e4
    mask = (torch.rand(n_rows, generator=g, device=device) < active_prob).to(torch.uint8)
    ids = torch.randint(0, vocab, (n_rows,), generator=g, device=device, dtype=torch.int32)
    return Workload("synthetic", train[:, :vocab], rollout[:, :vocab], ids, mask, vocab,
                    meta={"seed": seed, "sigma": sigma, "rollout_noise": rollout_noise})


def tiny(seed: int = 0, device="cpu") -> Workload:
    B, T, V = 2, 64, 1024
    g = _gen(device, seed)
    R = B * T
    train = (2.0 * torch.randn((R, V), generator=g, device=device)).to(torch.bfloat16)
    rollout = _fill_noisy(train.float(), 1e-3, g, torch.bfloat16)
    pos = torch.arange(T, device=device).repeat(B)
    response = (pos >= 16) & (pos < T - 8)
    mask = (response & (torch.rand(R, generator=g, device=device) < 0.9)).to(torch.uint8)
    ids = torch.randint(0, V, (R,), generator=g, device=device, dtype=torch.int32)
    return Workload("tiny", train, rollout, ids, mask, V, meta={"B": B, "T": T, "seed": seed})


def qwen(seed: int = 1, device="cuda", batch: int = 8, seq: int = 4096) -> Workload:
    V = 151936
    R = batch * seq
    w = synthetic(R, V, seed=seed, device=device, sigma=3.0, rollout_noise=2e-3, active_prob=1.0,
                  spike_frac=0.01, spike=15.0)
    g = _gen(device, seed + 1000)
    prompt = torch.randint(256, 1025, (batch,), generator=g, device=device)
    pad = torch.randint(0, 513, (batch,), generator=g, device=device)
    t = torch.arange(seq, device=device)[None, :]
    mask = ((t >= prompt[:, None]) & (t < seq - pad[:, None])).reshape(-1).to(torch.uint8)
    return Workload("qwen3-8b-vocab", w.train, w.rollout, w.token_ids, mask, V,
                    meta={"B": batch, "T": seq, "seed": seed, "padding": "right"})


def llama(seed: int = 2, device="cuda", batch: int = 64, seq: int = 1024) -> Workload:
    V = 128256
    R = batch * seq
    g = _gen(device, seed)
    train = torch.empty((R, V), dtype=torch.bfloat16, device=device)
    rollout = torch.empty((R, V), dtype=torch.float32, device=device)
    ids = torch.empty(R, dtype=torch.int32, device=device)
    step = _chunk_rows(V)
    for c in range(0, R, step):
        n = min(step, R - c)
        tc = (3.0 * torch.randn((n, V), generator=g, device=device)).to(torch.bfloat16)
        train[c:c + n] = tc
        rollout[c:c + n] = tc.float() + 1e-3 * torch.randn((n, V), generator=g, device=device)
        # teacher-forced ids: a sample from softmax(train row) via Gumbel-max
        u = torch.rand((n, V), generator=g, device=device).clamp_(min=1e-30)
        ids[c:c + n] = torch.argmax(tc.float() - torch.log(-torch.log(u)), dim=1).to(torch.int32)
    g2 = _gen(device, seed + 1000)
    pad = torch.randint(0, 513, (batch,), generator=g2, device=device)
    prompt = torch.randint(64, 257, (batch,), generator=g2, device=device)
    t = torch.arange(seq, device=device)[None, :]
    mask = (t >= (pad + prompt)[:, None]).reshape(-1).to(torch.uint8)
    return Workload("llama-vocab-mixed", train, rollout, ids, mask, V,
                    meta={"B": batch, "T": seq, "seed": seed, "padding": "left"})


def sharded(seed: int = 3, device="cuda", seq: int = 32768, n_shards: int = 4, vocab: int = 151936) -> Workload:
    assert vocab % n_shards == 0
    width = vocab // n_shards
    g = _gen(device, seed)
    ts, rs = [], []
    for _ in range(n_shards):
        t = torch.empty((seq, width), dtype=torch.bfloat16, device=device)
        r = torch.empty((seq, width), dtype=torch.bfloat16, device=device)
        step = _chunk_rows(width)
        for c in range(0, seq, step):
            n = min(step, seq - c)
            tc = (3.0 * torch.randn((n, width), generator=g, device=device)).to(torch.bfloat16)
            t[c:c + n] = tc
            r[c:c + n] = _fill_noisy(tc.float(), 2e-3, g, torch.bfloat16)
        ts.append(t)
        rs.append(r)
    ids = torch.randint(0, vocab, (seq,), generator=g, device=device, dtype=torch.int32)
    mask = torch.ones(seq, dtype=torch.uint8, device=device)
    v_ranges = [(k * width, (k + 1) * width) for k in range(n_shards)]
    return Workload("vocab-sharded-tp4", ts, rs, ids, mask, vocab, v_ranges=v_ranges,
                    meta={"B": 1, "T": seq, "seed": seed, "n_shards": n_shards})


@dataclass
class HeadWorkload:
    name: str
    hidden_train: torch.Tensor   # [R, H] bf16
    hidden_rollout: torch.Tensor
    weight: torch.Tensor         # [V, H] bf16
    token_ids: torch.Tensor
    action_mask: torch.Tensor
    clip: tuple = CLIP
    meta: dict = field(default_factory=dict)

    @property
    def n_rows(self) -> int:
        return int(self.token_ids.shape[0])

    @property
    def vocab(self) -> int:
        return int(self.weight.shape[0])

    @property
    def hidden(self) -> int:
        return int(self.weight.shape[1])


def head(n_rows: int, hidden: int, vocab: int, *, seed: int = 4, device="cuda", w_sigma: float = 0.02,
         rollout_noise: float = 1e-3, active_prob: float = 1.0) -> HeadWorkload:
    """LM-head case: hidden N(0, 1), W N(0, w_sigma^2), rollout hidden = bf16(hidden + noise)."""
    g = _gen(device, seed)
    ht = torch.randn((n_rows, hidden), generator=g, device=device).to(torch.bfloat16)
    hr = _fill_noisy(ht.float(), rollout_noise, g, torch.bfloat16)
    W = torch.empty((vocab, hidden), dtype=torch.bfloat16, device=device)
    step = _chunk_rows(hidden)
    for c in range(0, vocab, step):
        n = min(step, vocab - c)
        W[c:c + n] = (w_sigma * torch.randn((n, hidden), generator=g, device=device)).to(torch.bfloat16)
    ids = torch.randint(0, vocab, (n_rows,), generator=g, device=device, dtype=torch.int32)
    mask = (torch.rand(n_rows, generator=g, device=device) < active_prob).to(torch.uint8)
    return HeadWorkload("head", ht, hr, W, ids, mask, meta={"seed": seed})


def fused(seed: int = 4, device="cuda", rows: int = 16384) -> HeadWorkload:
    w = head(rows, 4096, 151936, seed=seed, device=device)
    w.name = "fused-lm-head"
    return w


@dataclass
class AttnWorkload:
    name: str
    out_parts: torch.Tensor   # [K, n_rows, head_dim] f32 or bf16
    lse_parts: torch.Tensor   # [K, n_rows] f32
    n_tokens: int
    n_heads: int
    lse_base2: bool = False
    meta: dict = field(default_factory=dict)

    @property
    def n_parts(self) -> int:
        return int(self.out_parts.shape[0])

    @property
    def n_rows(self) -> int:
        return int(self.out_parts.shape[1])

    @property
    def head_dim(self) -> int:
        return int(self.out_parts.shape[2])

    def keyed_pairs(self) -> int:
        """(row, part) pairs whose part saw at least one key."""
        return int(torch.isfinite(self.lse_parts).sum().item())


def attn_partials(n_tokens: int, n_heads: int, head_dim: int, n_parts: int, *, seed: int = 5, device="cuda",
                  dtype=torch.float32, causal: bool = True, lse_base2: bool = False,
                  masked_fill: float = 0.0, out_sigma: float = 0.5) -> AttnWorkload:
    """Per-block attention partials of T tokens x H heads over K contiguous key
    blocks (the attn recipe).  masked_fill is written into the out rows of
    parts that saw no keys (0, or NaN to prove they are never read)."""
    g = _gen(device, seed)
    T, H, K = n_tokens, n_heads, n_parts
    t = torch.arange(T, device=device)
    lse = torch.empty((K, T * H), dtype=torch.float32, device=device)
    out = torch.empty((K, T * H, head_dim), dtype=dtype, device=device)
    step = _chunk_rows(head_dim)
    for k in range(K):
        start, end = k * T // K, (k + 1) * T // K
        n_k = (torch.clamp(torch.minimum(t + 1, torch.tensor(end, device=device)) - start, min=0) if causal
               else torch.full((T,), end - start, device=device))
        base = torch.log(n_k.to(torch.float32)).repeat_interleave(H)          # -inf where n_k == 0
        lk = base + 2.0 + torch.randn((T * H,), generator=g, device=device)
        if lse_base2:
            lk = lk / torch.log(torch.tensor(2.0, device=device))
        lse[k] = lk
        for c in range(0, T * H, step):
            n = min(step, T * H - c)
            out[k, c:c + n] = (out_sigma * torch.randn((n, head_dim), generator=g, device=device)).to(dtype)
        dead = ~torch.isfinite(lse[k])
        out[k][dead] = torch.tensor(masked_fill, dtype=dtype, device=device)
    return AttnWorkload("attn", out, lse, T, H, lse_base2,
                        meta={"seed": seed, "causal": causal, "masked_fill": masked_fill})


def attn(seed: int = 5, device="cuda", n_tokens: int = 32768, dtype=torch.float32) -> AttnWorkload:
    w = attn_partials(n_tokens, 32, 128, 8, seed=seed, device=device, dtype=dtype)
    w.name = "cp8-attention-partials"
    return w
