"""Per-rank drift reports for data-parallel runs.

"WS2 Cross-Config Logprob Drift Contract", section "Diagnostics": when the run
is distributed, the same metrics are reported per rank, with enough metadata
to identify the rank and its local active-token count.  Each rank scores its
own rows with the CUDA library; this module only exchanges the small
per-rank metric records (torch.distributed, any backend) and combines them:

* gather_rank_metrics: every rank's metrics record, in rank order;
* merge_rank_metrics: the global values that can be combined exactly from the
  records (the library's lpd_merge_rank_metrics, a host call): the
  active-token count, the token-weighted means (ratio0_mean, clipfrac0,
  approx_kl0, mean_abs_dlogp) and the worst token (largest max_abs_dlogp,
  lowest global row on ties).  Percentiles of the union are not a function of
  per-rank percentiles;
* gather_rank_rows / global_drift_metrics: every rank's per-token dlogp and
  mask (5 bytes a row) gathered in rank order, and the full metrics record of
  the union computed from them on the GPU (lpd_drift_metrics_from_dlogp),
  percentiles included.

The merge visits ranks in rank order, so its result does not depend on the
collective's algorithm or arrival order ("[WS2] Framework for ablation
experiment", LogProb knobs table, row 5: merge order as a drift source).
"""
from __future__ import annotations


def gather_rank_metrics(metrics: dict, *, rank_meta: dict | None = None, group=None) -> list[dict]:
    """All ranks' metric records (plus optional metadata such as the rank's
    row offset, dtype or padding side), ordered by rank."""
    import torch.distributed as dist

    record = dict(metrics)
    record["rank"] = dist.get_rank(group)
    if rank_meta:
        record.update(rank_meta)
    out = [None] * dist.get_world_size(group)
    dist.all_gather_object(out, record, group=group)
    return sorted(out, key=lambda r: r["rank"])


def merge_rank_metrics(per_rank: list[dict], row_offsets: list[int] | None = None) -> dict:
    """Global metrics from per-rank records taken in rank order
    (lpd_merge_rank_metrics: the arithmetic is the library's).  row_offsets[k]
    maps rank k's local row indices to global ones (default 0).  p95/p99 come
    back NaN with LPD_FLAG_NO_PERCENTILES set."""
    from logprob_drift_scoring_gb300 import binding as B

    return B.merge_rank_metrics(per_rank, row_offsets)


def gather_rank_rows(local_dlogp, local_mask, group=None):
    """Every rank's per-row dlogp (float32) and mask (uint8), concatenated in
    rank order.  Ranks may hold different numbers of rows.  The tensors travel
    on their own device (NCCL for CUDA tensors, gloo for CPU ones)."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    sizes = [None] * world
    dist.all_gather_object(sizes, int(local_dlogp.shape[0]), group=group)
    width = max(max(sizes), 1)
    d = torch.zeros(width, dtype=torch.float32, device=local_dlogp.device)
    m = torch.zeros(width, dtype=torch.uint8, device=local_mask.device)
    d[:local_dlogp.shape[0]] = local_dlogp
    m[:local_mask.shape[0]] = local_mask
    ds = [torch.empty_like(d) for _ in range(world)]
    ms = [torch.empty_like(m) for _ in range(world)]
    dist.all_gather(ds, d, group=group)
    dist.all_gather(ms, m, group=group)
    return (torch.cat([x[:n] for x, n in zip(ds, sizes)]), torch.cat([x[:n] for x, n in zip(ms, sizes)]))


def global_drift_metrics(local_dlogp, local_mask, clip=(0.8, 1.2), group=None) -> dict:
    """The metrics record of all ranks' rows together, identical on every rank
    (CUDA tensors: the union is scored by the library on this rank's GPU)."""
    from logprob_drift_scoring_gb300 import binding as B

    d, m = gather_rank_rows(local_dlogp, local_mask, group)
    return B.drift_metrics_from_dlogp(d, m, clip)
