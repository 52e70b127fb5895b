"""lpd_score_noalloc: lpd_score for callers that cannot allocate device memory.

Callers running inside another engine whose allocator owns the device, or
plugins that receive only a stream and tensors, cannot pass lpd_score a
workspace.  lpd_score_noalloc uses an array of device memory built into the
library instead.  It launches the same kernels in the same order as lpd_score,
so its results must be bitwise those of lpd_score (given a workspace allocated
here): the per-token outputs compared with torch.equal, every metrics field
with ==.

The cases run back to back on the one shared array, each twice, so every call
after the first runs on scratch that still holds an earlier call's contents:
  * exactly LPD_NOALLOC_MAX_ROWS rows (the array's sizing; 8 blocks of the
    multi-block active-row compaction, whose per-block counts live in the
    array's header),
  * 9000 rows (3 compaction blocks, fewer than the previous call left behind),
  * 700 rows of mixed dtypes (the single-CTA compaction), then the limit again.

This file is collected last on purpose; it also passes when run alone in a
fresh process (the first call on the device does the one-time set-up).
"""
import ctypes

import pytest

from logprob_drift_scoring_gb300 import binding as B


def test_noalloc_rejects_more_rows_than_its_scratch_holds():
    # checked on the host before the GPU is touched
    t = B.LpdLogits(0x7F0000000000, B.LPD_BF16, 0, 16)
    rc = B.lib().lpd_score_noalloc(ctypes.byref(t), ctypes.byref(t), B.LPD_NOALLOC_MAX_ROWS + 1, 16,
                                   0x7F0000000000, 0x7F0000000000, 0.8, 1.2, None, None, None,
                                   0x7F0000000000, None)
    assert rc == B.LPD_ERR_UNSUPPORTED


@pytest.mark.gpu
def test_noalloc_equals_lpd_score_bitwise_on_calls_in_a_row():
    import torch

    from logprob_drift_scoring_gb300 import workloads as W

    dev = "cuda"
    limit = B.LPD_NOALLOC_MAX_ROWS
    big = W.synthetic(limit, 4096, seed=41, device=dev)                                   # bf16 / bf16
    mid = W.synthetic(9000, 20000, seed=43, device=dev, active_prob=0.7)                 # 3 compaction blocks
    small = W.synthetic(700, 9000, seed=42, device=dev, dtype_rollout=torch.float32,    # mixed dtypes,
                        rollout_noise=0.3)                                              # clipping active
    assert big.n_rows == limit
    for w in (big, big, mid, mid, small, small, big):
        n = w.n_rows
        want = B.score(w.train, w.rollout, w.token_ids, w.action_mask, w.clip)
        outs = [torch.full((n,), float("nan"), dtype=torch.float32, device=dev) for _ in range(3)]
        met = torch.zeros(B.METRICS_BYTES, dtype=torch.uint8, device=dev)
        B.lpd_score_noalloc(w.train, w.rollout, w.token_ids, w.action_mask, w.clip[0], w.clip[1], *outs, met)
        torch.cuda.synchronize()
        for got, exp in zip(outs, (want.logp_train, want.logp_rollout, want.dlogp)):
            assert torch.equal(got, exp)
        got_m = B.read_metrics(met)
        assert got_m["status"] == 0 and got_m["n_active"] == int(w.action_mask.sum().item())
        assert got_m == want.metrics
