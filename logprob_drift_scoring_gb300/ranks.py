"""Per-rank drift reports for data-parallel runs.

"WS2 Cross-Config Logprob Drift Contract", section "Diagnostics": when the run
is distributed, the same metrics are reported per rank, with enough metadata
to identify the rank and its local active-token count.  Each rank scores its
own rows with the CUDA library; this module only exchanges the small
per-rank metric records (torch.distributed, any backend) and combines them:

* gather_rank_metrics: every rank's metrics record, in rank order;
* merge_rank_metrics: the global values that can be combined exactly from the
  records: the active-token count, the token-weighted means (ratio0_mean,
  clipfrac0, approx_kl0, mean_abs_dlogp) and the worst token (largest
  max_abs_dlogp, lowest global row on ties).  Percentiles of the union are not
  a function of per-rank percentiles and are left to a pass over the gathered
  dlogp values.

The merge visits ranks in rank order, so its result does not depend on the
collective's algorithm or arrival order ("[WS2] Framework for ablation
experiment", LogProb knobs table, row 5: merge order as a drift source).
"""
from __future__ import annotations

MEAN_KEYS = ("ratio0_mean", "clipfrac0", "approx_kl0", "mean_abs_dlogp")


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
    """Global metrics from per-rank records taken in rank order.  row_offsets[k]
    maps rank k's local row indices to global ones (default 0)."""
    offsets = row_offsets or [0] * len(per_rank)
    total = sum(int(r["n_active"]) for r in per_rank)
    out = {"n_active": total, "status": 0, "flags": 0 if total else 1, "argmax_row": -1,
           "max_abs_dlogp": 0.0}
    for k in MEAN_KEYS:
        out[k] = 0.0
    best = -1.0
    for r, off in zip(per_rank, offsets):
        out["status"] |= int(r["status"])
        a = int(r["n_active"])
        if a == 0:
            continue
        for k in MEAN_KEYS:
            out[k] += r[k] * a
        if r["max_abs_dlogp"] > best:  # strict: earlier ranks hold lower global rows
            best = r["max_abs_dlogp"]
            out["max_abs_dlogp"] = best
            out["argmax_row"] = int(r["argmax_row"]) + int(off)
    if total:
        for k in MEAN_KEYS:
            out[k] /= total
    return out
