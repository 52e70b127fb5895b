#!/usr/bin/env python3
"""Benchmark of the selected-token logprob drift scorer on GB300.

One step = the whole scoring path over one batch: stage 1 (active-row
selection), stage 2 (the streaming row pass over both logits tensors plus the
per-row finalise) and stage 3 (the drift metrics and the percentile select),
exactly the kernels lpd_score launches, on one stream.  The default workload
is the Qwen3-8B-vocab shape: B=8 x T=4096 rows, V=151936, bf16 logits on both
sides (19.9 GB, far larger than the 129 MB L2, so no L2 flush is needed
between steps).

Printed (one JSON line, rank 0):
  value      active tokens scored per second, device-timed (CUDA events)
  roofline   stage 2's algorithmic bytes / its average duration vs the
             measured HBM copy bandwidth
  e2e        the same metric through the C ABI (lpd_score_host) with the
             inputs in pinned host memory: every step copies the active rows
             of both sides plus ids and mask to the device, scores them and
             reads the metrics record back
  cpu_baseline  the float64 CPU oracle on a bounded sample of the workload

--impl reference times the oracle alone: the reference arm (the method is
published as text without code, so the float64 oracle stands in for it).
Multi-GPU (torchrun, N>1): every rank scores its own batch (replicas, weak
scaling, no collective on the data path); the step time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import threading
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

CONFIGS = {
    "qwen": dict(workload="qwen3-8b-vocab B=8 T=4096 V=151936 bf16/bf16", vocab=151936),
    "llama": dict(workload="llama-vocab B=64 T=1024 V=128256 bf16/fp32", vocab=128256),
    "sharded": dict(workload="vocab-sharded B=1 T=32768 V=151936 (4 shards) bf16/bf16", vocab=151936),
    "tiny": dict(workload="tiny B=2 T=64 V=1024 bf16/bf16", vocab=1024),
    "fused": dict(workload="fused LM head: 16384 tokens x H=4096, W [151936, 4096] bf16", vocab=151936),
    "attn": dict(workload="CP-8 causal attention partials: T=32768 x 32 heads, head_dim 128, f32", vocab=0),
}
ATTN_METRIC = "attention rows merged/sec (token x head, split-KV (out, lse) merge); achieved HBM GB/s"
ATTN_UNIT = "rows/s"
METRIC = "active tokens/sec scored; achieved HBM GB/s vs GB300 peak (logp+drift pass)"
UNIT = "active_tokens/s"
KERNEL_SOURCES = ["logprob_drift_scoring_gb300/csrc/lpd_rows.cu"]


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def measured_peaks() -> dict:
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        return {"hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def kernel_source_hash() -> str:
    h = hashlib.sha1()
    for rel in KERNEL_SOURCES + ["logprob_drift_scoring_gb300/csrc/lpd_internal.cuh",
                                 "logprob_drift_scoring_gb300/csrc/lpd_acc.cuh",
                                 "logprob_drift_scoring_gb300/csrc/lpd_xform.cuh"]:
        h.update((ROOT / rel).read_bytes())
    return h.hexdigest()[:12]


def profiled_row_kernel(config: str) -> dict | None:
    """The row pass's committed ncu summary for this config, if it was captured
    on the current kernel source: DRAM bytes per launch scaled to the full
    workload, and the DRAM throughput (% of peak) of the captured case."""
    p = ROOT / "profiles" / f"row_kernel_{config}.md"
    if not p.exists():
        return None
    text = p.read_text()
    m_src = re.search(r"kernel_source_sha1:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"traffic_bytes_per_launch_full_size:\s*([0-9.eE+]+)", text)
    m_pct = re.search(r"gpu__dram_throughput\.avg\.pct_of_peak_sustained_elapsed \| ([0-9.]+) %", text)
    if not m_src or not m_tr or m_src.group(1) != kernel_source_hash():
        return None
    return {"traffic": float(m_tr.group(1)), "dram_pct": float(m_pct.group(1)) if m_pct else None}


def profiled_traffic(config: str):
    prof = profiled_row_kernel(config)
    return prof["traffic"] if prof else None


def host_cpu() -> dict:
    """Core count and CPU model of the host the oracle runs on."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        m = re.search(r"Model name:\s*(.+)", out)
        model = m.group(1).strip() if m else None
    except (OSError, subprocess.SubprocessError):
        pass
    return {"nproc": os.cpu_count(), "model": model}


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd += ["-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            # start the timed region only once sampling is running (the first
            # sample is taken just before it, the next ones every 200 ms inside)
            t0 = time.time()
            while not self.lines and time.time() - t0 < 3.0 and self.proc.poll() is None:
                time.sleep(0.01)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_uuid():
    import torch

    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return None


# ---------------------------------------------------------------- workloads

def make_workload(config: str, device, seed_offset: int = 0, batch=None, seq=None):
    """The named workload; batch/seq shrink it (used only for small ncu captures)."""
    from logprob_drift_scoring_gb300 import workloads as W

    if config == "qwen":
        return W.qwen(seed=1 + seed_offset, device=device, batch=batch or 8, seq=seq or 4096)
    if config == "llama":
        return W.llama(seed=2 + seed_offset, device=device, batch=batch or 64, seq=seq or 1024)
    if config == "sharded":
        return W.sharded(seed=3 + seed_offset, device=device, seq=seq or 32768)
    if config == "tiny":
        return W.tiny(seed=0 + seed_offset, device=device)
    if config == "fused":
        return W.fused(seed=4 + seed_offset, device=device, rows=seq or 16384)
    if config == "attn":
        return W.attn(seed=5 + seed_offset, device=device, n_tokens=seq or 32768)
    raise SystemExit(f"unknown config {config}")


def bytes_per_active_token(w) -> int:
    """Algorithmic bytes of the row pass per active token: both logits rows
    once, the token id, and the three fp32 per-token outputs."""
    ts = w.train if isinstance(w.train, list) else [w.train]
    rs = w.rollout if isinstance(w.rollout, list) else [w.rollout]
    row = sum(t.shape[1] * t.element_size() for t in ts) + sum(r.shape[1] * r.element_size() for r in rs)
    return row + 4 + 12


# ---------------------------------------------------------------- our arm

class Runner:
    """Buffers and the stage sequence of one workload on one device."""

    def __init__(self, w):
        import torch
        from logprob_drift_scoring_gb300 import binding as B

        self.B, self.w, self.torch = B, w, torch
        dev = w.token_ids.device
        n = w.n_rows
        self.sharded = isinstance(w.train, list)
        self.outs = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(3)]
        self.met = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=dev)
        if self.sharded:
            ws = B.lpd_workspace_size(B.LPD_KIND_SHARDED, n, w.vocab, len(w.v_ranges))
        else:
            ws = B.lpd_workspace_size(B.LPD_KIND_SCORE, n)
        self.ws = torch.empty(ws, dtype=torch.uint8, device=dev)
        self.launches_per_step = select_launches(n) + 4 if n > 0 else 2
        self.chain = None
        self.entropy = None      # [ent_train, ent_rollout] when timing lpd_score_entropy
        self.backward = None     # (grad, out_dlogits) when timing lpd_logprob_backward
        self.topology = None     # reduction-topology arm when timing lpd_score_sharded_topology

    def use_topology(self, topo: int):
        B, w, torch = self.B, self.w, self.torch
        self.topology = topo
        need = B.lpd_topology_workspace_size(topo, w.n_rows, w.vocab, len(w.v_ranges),
                                             B._dtype_code(w.train[0]), B._dtype_code(w.rollout[0]))
        self.ws = torch.empty(need, dtype=torch.uint8, device=w.token_ids.device)

    def step(self, ev=None):
        """One pass of the path; with ev = (e0, e1, e2, e3) records events
        around stage 1, stage 2 and stage 3 on the current stream."""
        B, w = self.B, self.w
        lt, lr, d = self.outs
        if self.backward is not None:
            grad, out = self.backward
            if ev:
                ev[0].record()
            B.lpd_logprob_backward(w.train, w.token_ids, w.action_mask, lt, grad, out)
            if ev:
                ev[3].record()
            return
        if self.entropy is not None:
            if ev:
                ev[0].record()
            B.lpd_score_entropy(w.train, w.rollout, w.token_ids, w.action_mask, *w.clip, lt, lr, d, *self.entropy,
                                self.met, self.ws)
            if ev:
                ev[3].record()
            return
        if self.chain is not None:
            if ev:
                ev[0].record()
            B.lpd_score_transformed(w.train, w.rollout, self.chain, self.chain, w.token_ids, w.action_mask,
                                    *w.clip, lt, lr, d, self.met, self.ws)
            if ev:
                ev[3].record()
            return
        if self.sharded and self.topology is not None:
            if ev:
                ev[0].record()
            B.lpd_score_sharded_topology(w.train, w.rollout, w.v_ranges, w.token_ids, w.action_mask, *w.clip,
                                         self.topology, None, lt, lr, d, self.met, self.ws)
            if ev:
                ev[3].record()
            return
        if self.sharded:
            if ev:
                ev[0].record()
            B.lpd_score_sharded(w.train, w.rollout, w.v_ranges, w.token_ids, w.action_mask, *w.clip, None,
                                lt, lr, d, None, None, self.met, self.ws)
            if ev:
                ev[3].record()
            return
        if ev:
            ev[0].record()
        B.lpd_select_active(w.token_ids, w.action_mask, lt, lr, d, self.met, self.ws)
        if ev:
            ev[1].record()
        B.lpd_token_logp(w.train, w.rollout, lt, lr, d, self.met, self.ws)
        if ev:
            ev[2].record()
        B.lpd_drift_metrics(w.n_rows, w.clip[0], w.clip[1], self.met, self.ws)
        if ev:
            ev[3].record()


def barrier_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def _single_core_oracle(config: str, rows: int = 1024, seed: int = 1234) -> dict:
    """The float64 oracle as it stands, on one core: a seeded slice of `rows`
    active rows drawn with the workload's recipe, scored serially."""
    import numpy as np
    import torch

    import oracle
    from logprob_drift_scoring_gb300 import workloads as W

    vocab = CONFIGS[config]["vocab"]
    dt_r = torch.float32 if config == "llama" else torch.bfloat16
    sigma = 2.0 if config == "tiny" else 3.0
    noise = {"tiny": 1e-3, "llama": 1e-3}.get(config, 2e-3)
    lib = oracle.load()
    w = W.synthetic(rows, vocab, seed=seed, device="cpu", dtype_rollout=dt_r, sigma=sigma, rollout_noise=noise,
                    active_prob=1.0)
    tn, rn = oracle_host(w.train), oracle_host(w.rollout)
    t0 = time.perf_counter()
    oracle.score_rows(tn, rn, w.token_ids.numpy(), np.arange(rows), lib=lib)
    elapsed = time.perf_counter() - t0
    return {"value": round(rows / elapsed, 2), "unit": UNIT, "cores": 1, "seconds": round(elapsed, 2),
            "sample": f"{rows} active rows of the {config} recipe, both sides, float64 serial C"}


def oracle_host(t):
    """Host numpy view of a CPU tensor for the oracle (bf16 as uint16 bits)."""
    import numpy as np
    import torch

    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    return t.contiguous().numpy()


def time_cpu_oracle(config: str, w, single_rows: int = 1024) -> dict:
    """The float64 oracle as it stands, timed on the host cores two ways:
    all cores, over every active row of this very workload (copied off the
    device chunk by chunk while one host thread per core scores earlier
    chunks: oracle/stream.py, which only schedules the serial C); and one
    core, on a seeded slice of the same recipe (its time for the whole
    workload is that rate extrapolated linearly)."""
    import numpy as np

    from oracle import stream

    threads = stream.host_threads()
    mask = w.action_mask.cpu().numpy()
    rows = np.flatnonzero(mask)
    t0 = time.perf_counter()
    if isinstance(w.train, list):
        stream.score_sharded_rows_device(w.train, w.rollout, w.v_ranges, w.token_ids, rows, threads=threads)
    else:
        stream.score_rows_device(w.train, w.rollout, w.token_ids, rows, threads=threads)
    elapsed = time.perf_counter() - t0
    one = _single_core_oracle(config, rows=min(single_rows, max(16, rows.size)))
    one["extrapolated_full_run_s"] = round(rows.size / one["value"], 1)
    return {"value": round(rows.size / elapsed, 2), "unit": UNIT, "cores": threads, "kind": "oracle",
            "host": host_cpu(), "seconds": round(elapsed, 2),
            "sample": f"all {rows.size} active rows of this workload, one host thread per core running the "
                      f"serial float64 C on 64-row chunks copied off the device (copies overlapped)",
            "single_core": one}


def measured_tflops(timed_s: float) -> dict:
    """The measured bf16 GEMM peak that fits a timed region of timed_s
    seconds: the power-capped sustained figure for regions of 2 s or more,
    else the burst figure."""
    sustained = timed_s >= 2.0
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        d = json.loads(p.read_text())
        if sustained:
            return {"tflops": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "source": "measured sustained"}
        return {"tflops": d["bf16_tflops"], "source": "measured burst"}
    return {"tflops": 1700.0, "source": "fallback sustained"} if sustained else \
        {"tflops": 1900.0, "source": "fallback burst"}


def select_launches(n_rows: int) -> int:
    """Kernels of stage 1 (active-row compaction): a count and a compaction
    kernel for 2 to 31 blocks of 4096 rows, else one single-CTA kernel."""
    blocks = -(-n_rows // 4096)
    return 2 if 2 <= blocks <= 31 else 1


def time_cpu_oracle_head(w, rows: int = 64) -> dict:
    """The float64 oracle's LM-head scorer (logits materialised in double) as
    it stands, on every host core, over `rows` rows of this workload spread
    over its row tiles (oracle/stream.py schedules; each row is serial C)."""
    import numpy as np

    from oracle import stream

    threads = stream.host_threads()
    n = w.n_rows
    sel = np.linspace(0, n - 1, num=min(rows, n)).astype(np.int64)
    ht, hr, W = oracle_host(w.hidden_train.cpu()), oracle_host(w.hidden_rollout.cpu()), oracle_host(w.weight.cpu())
    t0 = time.perf_counter()
    stream.score_head_rows_parallel(ht, hr, W, w.token_ids.cpu().numpy(), sel, chunk=2, threads=threads)
    elapsed = time.perf_counter() - t0
    return {"value": round(sel.size / elapsed, 3), "unit": UNIT, "cores": threads, "kind": "oracle",
            "host": host_cpu(), "seconds": round(elapsed, 2),
            "sample": f"{sel.size} rows of this workload (both sides, H={w.hidden}, V={w.vocab}), one host thread "
                      f"per core running the serial float64 head and scorer"}


def run_fused(args, w, world, rank):
    """The fused LM-head path: one lpd_score_fused call per step (with
    --transform, lpd_score_fused_transformed with that chain on both sides)."""
    import torch
    from logprob_drift_scoring_gb300 import binding as B

    dev = w.token_ids.device
    n = w.n_rows
    outs = [torch.empty(n, dtype=torch.float32, device=dev) for _ in range(3)]
    met = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=dev)
    ws = torch.empty(B.lpd_fused_workspace_size(n, w.hidden, w.vocab), dtype=torch.uint8, device=dev)
    chain = parse_chain(args.transform) if args.transform else None

    def step():
        if chain is None:
            B.lpd_score_fused(w.hidden_train, w.hidden_rollout, w.weight, w.token_ids, w.action_mask, *w.clip,
                              *outs, met, ws)
        else:
            B.lpd_score_fused_transformed(w.hidden_train, w.hidden_rollout, w.weight, chain, chain, w.token_ids,
                                          w.action_mask, *w.clip, *outs, met, ws)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_uuid()) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        start.record()
        for _ in range(args.steps):
            step()
        stop.record()
        torch.cuda.synchronize()
        barrier(world)
    ms = barrier_max(start.elapsed_time(stop) / args.steps, world)
    n_active = int(w.action_mask.sum().item())
    flops = 2.0 * 2.0 * n_active * w.hidden * w.vocab  # both sides
    peak = measured_tflops(ms * args.steps / 1e3)
    achieved = flops / (ms / 1e3) / 1e12

    e2e = None
    if not args.no_e2e:
        # per step: both sides' hidden states, ids and mask from pinned host
        # memory to the device (the head W stays resident, like model weights),
        # the call, and the metrics record back
        pinned = True
        try:
            host = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
                    for t in (w.hidden_train, w.hidden_rollout, w.token_ids, w.action_mask)]
            met_host = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, pin_memory=True)
        except RuntimeError:
            host = [torch.empty(t.shape, dtype=t.dtype)
                    for t in (w.hidden_train, w.hidden_rollout, w.token_ids, w.action_mask)]
            met_host = torch.empty(B.METRICS_BYTES, dtype=torch.uint8)
            pinned = False
        for h, t in zip(host, (w.hidden_train, w.hidden_rollout, w.token_ids, w.action_mask)):
            h.copy_(t)
        dbuf = [torch.empty_like(t) for t in (w.hidden_train, w.hidden_rollout, w.token_ids, w.action_mask)]

        def one():
            for d, h in zip(dbuf, host):
                d.copy_(h, non_blocking=True)
            if chain is None:
                B.lpd_score_fused(dbuf[0], dbuf[1], w.weight, dbuf[2], dbuf[3], *w.clip, *outs, met, ws)
            else:
                B.lpd_score_fused_transformed(dbuf[0], dbuf[1], w.weight, chain, chain, dbuf[2], dbuf[3], *w.clip,
                                              *outs, met, ws)
            met_host.copy_(met, non_blocking=True)

        for _ in range(2):
            one()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.e2e_steps):
            one()
        e1.record()
        torch.cuda.synchronize()
        ems = barrier_max(e0.elapsed_time(e1) / args.e2e_steps, world)
        e2e = {"value": round(world * n_active / (ems / 1e3), 1), "unit": UNIT,
               "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in host),
               "d2h_bytes_per_step": B.METRICS_BYTES, "ms_per_step": round(ems, 3), "pinned": pinned,
               "steps": args.e2e_steps, "copies": "hidden states of both sides, ids, mask (W resident)"}
        del dbuf, host
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = time_cpu_oracle_head(w)
    if rank != 0:
        return None
    out = {
        "metric": METRIC, "value": round(world * n_active / (ms / 1e3), 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": CONFIGS["fused"]["workload"]
                   + (f" + transform {args.transform}" if args.transform else ""), "rows": n,
                   "active_tokens": n_active,
                   "hidden": w.hidden, "vocab": w.vocab, "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak["tflops"], "unit": "TFLOP/s",
                     "frac": round(achieved / peak["tflops"], 4), "traffic": None,
                     "peak_source": f"{peak['source']} bf16 GEMM", "timed_region_s": round(ms * args.steps / 1e3, 3),
                     "span": "whole lpd_score_fused call" if chain is None
                     else "whole lpd_score_fused_transformed call",
                     "algorithmic_flops_per_launch": flops},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": (select_launches(n) + 5) * args.steps,
        "clocks": clocks.summary(),
        "impl": "lpd",
    }
    print(json.dumps(out), flush=True)
    return out


def attn_bytes(w, drift: bool) -> int:
    """Algorithmic HBM bytes of one merge: the out chunks of every (row, part)
    pair that saw keys, every part's lse, the merged out and lse; with the
    order-drift diagnostic also its two per-row columns."""
    es = w.out_parts.element_size()
    n, d, K = w.n_rows, w.head_dim, w.n_parts
    b = w.keyed_pairs() * d * es + K * n * 4 + n * d * 4 + n * 4
    return b + (8 * n if drift else 0)


def time_cpu_oracle_attn(target_s: float = 12.0, seed: int = 1234):
    """The float64 oracle merge as it stands, on every host core (rows split
    into chunks over one thread per core), on a shorter sequence of the same
    recipe (rows per second scale with rows)."""
    from oracle import stream
    from logprob_drift_scoring_gb300 import workloads as W

    threads = stream.host_threads()
    probe = W.attn_partials(64, 32, 128, 8, seed=seed, device="cpu")
    t0 = time.perf_counter()
    stream.attn_merge_parallel(probe.out_parts.numpy(), probe.lse_parts.numpy(), threads=threads)
    per_row = (time.perf_counter() - t0) / probe.n_rows
    tokens = int(max(64, min(8192, target_s / max(per_row, 1e-12) / 32)))
    tokens -= tokens % 8
    w = W.attn_partials(tokens, 32, 128, 8, seed=seed + 1, device="cpu")
    parts, lse = w.out_parts.numpy(), w.lse_parts.numpy()
    t0 = time.perf_counter()
    stream.attn_merge_parallel(parts, lse, threads=threads)
    elapsed = time.perf_counter() - t0
    return {"value": w.n_rows / elapsed, "unit": ATTN_UNIT, "cores": threads, "kind": "oracle", "host": host_cpu(),
            "sample": f"{w.n_rows} rows (T={tokens} x 32 heads, K=8 causal, head_dim 128) of the attn recipe, "
                      f"float64 C on {threads} host threads, {elapsed:.1f} s"}


def run_attn(args, w, world, rank):
    """The split-KV attention merge: one lpd_attn_merge call per step (with
    --drift, one lpd_attn_merge_order_drift call comparing ascending and
    descending part order)."""
    import torch
    from logprob_drift_scoring_gb300 import binding as B

    dev = w.out_parts.device
    n, d, K = w.n_rows, w.head_dim, w.n_parts
    out = torch.empty((n, d), dtype=torch.float32, device=dev)
    lse = torch.empty((n,), dtype=torch.float32, device=dev)
    rdo = torch.empty((n,), dtype=torch.float32, device=dev)
    rdl = torch.empty((n,), dtype=torch.float32, device=dev)
    drift = torch.empty(B.MERGE_DRIFT_BYTES, dtype=torch.uint8, device=dev)
    rev = list(range(K))[::-1]
    stream = torch.cuda.current_stream()

    def step(parts=w.out_parts, lses=w.lse_parts):
        if args.drift:
            B.lpd_attn_merge_order_drift(parts, lses, None, rev, out, lse, rdo, rdl, drift, stream=stream)
        else:
            B.lpd_attn_merge(parts, lses, None, out, lse, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_uuid()) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        start.record(stream)
        for _ in range(args.steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    ms = barrier_max(start.elapsed_time(stop) / args.steps, world)
    nbytes = attn_bytes(w, args.drift)
    peaks = measured_peaks()
    achieved = nbytes / (ms / 1e3) / 1e9

    e2e = None
    if not args.no_e2e:
        # host partials -> device, merge, merged (out, lse) back to the host
        pinned = True
        try:
            hp = torch.empty(w.out_parts.shape, dtype=w.out_parts.dtype, pin_memory=True)
            hl = torch.empty(w.lse_parts.shape, dtype=torch.float32, pin_memory=True)
            ho = torch.empty((n, d), dtype=torch.float32, pin_memory=True)
            hs = torch.empty((n,), dtype=torch.float32, pin_memory=True)
        except RuntimeError:
            hp, hl = torch.empty(w.out_parts.shape, dtype=w.out_parts.dtype), torch.empty(w.lse_parts.shape)
            ho, hs = torch.empty((n, d)), torch.empty((n,))
            pinned = False
        hp.copy_(w.out_parts)
        hl.copy_(w.lse_parts)
        dp, dl = torch.empty_like(w.out_parts), torch.empty_like(w.lse_parts)

        def one():
            dp.copy_(hp, non_blocking=True)
            dl.copy_(hl, non_blocking=True)
            step(dp, dl)
            ho.copy_(out, non_blocking=True)
            hs.copy_(lse, non_blocking=True)

        for _ in range(2):  # warm-up: the first pass over fresh pinned buffers is slow
            one()
        torch.cuda.synchronize()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(args.e2e_steps):
            one()
        s1.record(stream)
        torch.cuda.synchronize()
        ems = barrier_max(s0.elapsed_time(s1) / args.e2e_steps, world)
        e2e = {"value": round(world * n / (ems / 1e3), 1), "unit": ATTN_UNIT,
               "h2d_bytes_per_step": hp.numel() * hp.element_size() + hl.numel() * 4,
               "d2h_bytes_per_step": ho.numel() * 4 + hs.numel() * 4, "ms_per_step": round(ems, 3),
               "pinned": pinned, "steps": args.e2e_steps}
        del hp, hl, dp, dl
        torch.cuda.empty_cache()
    if rank != 0:
        return None
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = time_cpu_oracle_attn(target_s=args.cpu_seconds)
    wl = CONFIGS["attn"]["workload"] if args.seq is None else f"attn reduced T={args.seq}"
    res = {
        "metric": ATTN_METRIC, "value": round(world * n / (ms / 1e3), 1), "unit": ATTN_UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl + (" + order drift (ascending vs descending)" if args.drift else ""),
                   "rows": n, "parts": K, "head_dim": d, "keyed_pairs": w.keyed_pairs(),
                   "parts_bytes": w.out_parts.numel() * w.out_parts.element_size(),
                   "l2": "inputs exceed L2 (no flush)", "parallelism": f"replicas x{world}"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None,
                     "peak_source": f"{peaks['source']} copy bandwidth (burst)",
                     "span": "whole call", "algorithmic_bytes_per_launch": nbytes},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": (3 if args.drift else 1) * args.steps,
        "clocks": clocks.summary(), "impl": "lpd",
    }
    print(json.dumps(res), flush=True)
    return res


def parse_chain(text: str):
    """'softcap:30,scale:1.4286' -> [(LPD_OP_SOFTCAP, 30.0), (LPD_OP_SCALE, 1.4286)]."""
    from logprob_drift_scoring_gb300 import binding as B

    kinds = {"scale": B.LPD_OP_SCALE, "softcap": B.LPD_OP_SOFTCAP}
    out = []
    for item in text.split(","):
        name, val = item.split(":")
        out.append((kinds[name.strip()], float(val)))
    return out


def run_ours(args):
    import torch

    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    from logprob_drift_scoring_gb300 import binding as B

    B.lib()  # fail loudly here if the CUDA library is missing
    w = make_workload(args.config, dev, seed_offset=rank, batch=args.batch, seq=args.seq)
    if args.config in ("fused", "attn"):
        out = (run_fused if args.config == "fused" else run_attn)(args, w, world, rank)
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
        return out
    runner = Runner(w)
    n_active = int(w.action_mask.sum().item())
    bpt = bytes_per_active_token(w)
    extra_bytes = 0
    if args.transform:
        runner.chain = parse_chain(args.transform)
    if args.topology:
        if not runner.sharded:
            raise SystemExit("--topology needs --config sharded")
        runner.use_topology(B.TOPOLOGIES[args.topology])
        if args.topology == "allgather_logits":
            runner.launches_per_step += 1  # the gather kernel
        if args.topology == "allgather_logits":
            # the all-gather reads every row of every shard and writes the full
            # rows once before the scoring pass reads the active ones
            extra_bytes = 2 * w.logits_bytes()
    if args.entropy:
        runner.entropy = [torch.empty(w.n_rows, dtype=torch.float32, device=dev) for _ in range(2)]
        bpt += 8
    if args.backward:
        runner.step()  # the forward's logp feeds the backward
        torch.cuda.synchronize()
        g = torch.Generator(device=dev).manual_seed(11)
        grad = torch.randn(w.n_rows, generator=g, device=dev)
        out = torch.empty((w.n_rows, w.vocab), dtype=torch.bfloat16, device=dev)
        runner.backward = (grad, out)
        # one read of the train row and one bf16 write per active row; inactive rows are zero-filled
        elt = w.train.element_size()
        bpt = w.vocab * (elt + 2) + 12
        extra_bytes = (w.n_rows - n_active) * w.vocab * 2

    for _ in range(args.warmup):
        runner.step()
    torch.cuda.synchronize()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_uuid()) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        start.record()
        for k in range(K):
            runner.step(evs[k])
        stop.record()
        torch.cuda.synchronize()
        barrier(world)
    total_ms = start.elapsed_time(stop)
    total_ms = barrier_max(total_ms, world)
    ms_step = total_ms / K
    value = world * n_active / (ms_step / 1e3)

    whole = (runner.sharded or runner.chain is not None or runner.entropy is not None or runner.backward is not None)
    if whole:
        stage2 = sum(e[0].elapsed_time(e[3]) for e in evs) / K
        stage_ms = {"whole_call": stage2}
    else:
        s1 = sum(e[0].elapsed_time(e[1]) for e in evs) / K
        stage2 = sum(e[1].elapsed_time(e[2]) for e in evs) / K
        s3 = sum(e[2].elapsed_time(e[3]) for e in evs) / K
        stage_ms = {"select_active": round(s1, 4), "token_logp": round(stage2, 4), "drift_metrics": round(s3, 4)}

    peaks = measured_peaks()
    achieved = (n_active * bpt + extra_bytes) / (stage2 / 1e3) / 1e9
    prof = profiled_row_kernel(args.config) if not whole else None
    traffic = prof["traffic"] if prof else None
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": traffic,
                "ncu_dram_pct_small_case": prof["dram_pct"] if prof else None,
                "peak_source": f"{peaks['source']} copy bandwidth (burst)",
                "span": "whole call" if whole else "stage 2: row kernel + per-row finalise",
                "algorithmic_bytes_per_launch": n_active * bpt + extra_bytes}

    e2e = None
    if not args.no_e2e and not whole:
        e2e = run_e2e(w, args, world)
    out = None
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cpu = time_cpu_oracle(args.config, w)
        out = {
            "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": round(ms_step, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": (CONFIGS[args.config]["workload"] if not (args.batch or args.seq)
                                    else f"{args.config} reduced B={args.batch} T={args.seq}")
                       + (f" + transform {args.transform}" if args.transform else "")
                       + (" + entropy" if args.entropy else "") + (" [logprob backward, bf16 out]" if args.backward else "")
                       + (f" [reduce: {args.topology}]" if args.topology else ""),
                       "rows": w.n_rows, "active_tokens": n_active,
                       "vocab": w.vocab, "logits_bytes": w.logits_bytes(), "l2": "inputs exceed L2 (no flush)",
                       "parallelism": f"replicas x{world}", "input_dtypes": _dtypes(w)},
            "stage_ms": stage_ms,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": (1 if runner.backward is not None else runner.launches_per_step) * K,

            "clocks": clocks.summary(),
            "impl": "lpd",
        }
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return out


def _dtypes(w):
    t = w.train[0] if isinstance(w.train, list) else w.train
    r = w.rollout[0] if isinstance(w.rollout, list) else w.rollout
    return f"{str(t.dtype).replace('torch.', '')}/{str(r.dtype).replace('torch.', '')}"


def run_e2e(w, args, world: int = 1):
    """Through lpd_score_host with host inputs: per step, the active rows of
    both sides' logits plus ids and mask go from pinned host memory to the
    device, the rows are scored, and the metrics record is read back."""
    import torch
    from logprob_drift_scoring_gb300 import binding as B

    dev = w.token_ids.device
    host = []
    pinned = True
    for t in (w.train, w.rollout, w.token_ids, w.action_mask):
        try:
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        except RuntimeError:
            h = torch.empty(t.shape, dtype=t.dtype)
            pinned = False
        h.copy_(t)
        host.append(h)
    dbuf = [torch.empty_like(t) for t in (w.train, w.rollout, w.token_ids, w.action_mask)]
    outs = [torch.empty(w.n_rows, dtype=torch.float32, device=dev) for _ in range(3)]
    met = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, device=dev)
    met_host = torch.empty(B.METRICS_BYTES, dtype=torch.uint8, pin_memory=pinned)
    ws = torch.empty(B.lpd_workspace_size(B.LPD_KIND_SCORE, w.n_rows), dtype=torch.uint8, device=dev)
    n_active = int(w.action_mask.sum().item())
    copied = []

    def one():
        copied.append(B.lpd_score_host(host[0], host[1], host[2], host[3], w.clip[0], w.clip[1], *dbuf, *outs, met,
                                       ws))
        met_host.copy_(met, non_blocking=True)

    for _ in range(2):  # warm-up: the first pass over fresh pinned buffers is slow
        one()
    torch.cuda.synchronize()
    steps = args.e2e_steps
    # one event between steps as well, so single slow steps (a stalled host
    # copy) show up next to the mean
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record()
    for k in range(steps):
        one()
        ev[k + 1].record()
    torch.cuda.synchronize()
    per_step = sorted(ev[k].elapsed_time(ev[k + 1]) for k in range(steps))
    ms = barrier_max(ev[0].elapsed_time(ev[steps]) / steps, world)
    del dbuf, host
    torch.cuda.empty_cache()
    assert len(set(copied)) == 1  # the same rows every step
    return {"value": round(world * n_active / (ms / 1e3), 1), "unit": UNIT, "h2d_bytes_per_step": copied[0],
            "d2h_bytes_per_step": B.METRICS_BYTES, "ms_per_step": round(ms, 3),
            "ms_per_step_median": round(per_step[len(per_step) // 2], 3), "ms_per_step_max": round(per_step[-1], 3),
            "pinned": pinned,
            "steps": steps, "copies": "active rows of both sides (one 2-D copy per run of active rows), ids, mask",
            "host_memory": "torch pinned (cudaHostAlloc)" if pinned else "pageable"}


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    """The reference arm: the float64 oracle as it stands on the host cores.
    One seeded sample of the workload's recipe (``--ref-rows`` active rows per
    host thread) is drawn once; every step scores all of it with one host
    thread per core running the serial C on its own chunk of rows."""
    rank, _, world = dist_env()
    if rank != 0:
        return None
    import numpy as np
    import torch

    import oracle
    from oracle import stream
    from logprob_drift_scoring_gb300 import workloads as W

    if args.config == "attn":
        return run_reference_attn(args, world)
    vocab = CONFIGS[args.config]["vocab"]
    dt_r = torch.float32 if args.config == "llama" else torch.bfloat16
    threads = stream.host_threads()
    rows_per_step = args.ref_rows * threads
    oracle.load()
    w = W.synthetic(rows_per_step, vocab, seed=5000, device="cpu", dtype_rollout=dt_r, active_prob=1.0)
    tn, rn, ids = oracle_host(w.train), oracle_host(w.rollout), w.token_ids.numpy()
    rows = np.arange(rows_per_step)
    times = []
    for k in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        stream.score_rows_parallel(tn, rn, ids, rows, chunk=args.ref_rows, threads=threads)
        if k >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = rows_per_step / (ms / 1e3)
    sample = (f"{rows_per_step} active rows of the {args.config} recipe (V={vocab}) per step, "
              f"{threads} host threads running the serial float64 C on {args.ref_rows}-row chunks")
    out = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": CONFIGS[args.config]["workload"], "sample_rows_per_step": rows_per_step},
           "impl": "reference",
           "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": threads, "kind": "oracle",
                            "sample": sample, "host": host_cpu()},
           "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return out


def run_reference_attn(args, world):
    import oracle
    from logprob_drift_scoring_gb300 import workloads as W

    lib = oracle.load()
    tokens = 1024  # 32768 rows of the recipe per step
    times = []
    for k in range(args.warmup + args.steps):
        w = W.attn_partials(tokens, 32, 128, 8, seed=6000 + k, device="cpu")
        parts, lse = w.out_parts.numpy(), w.lse_parts.numpy()
        t0 = time.perf_counter()
        oracle.attn_merge(parts, lse, lib=lib)
        if k >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    rows = tokens * 32
    value = rows / (ms / 1e3)
    sample = f"{rows} rows per step (T={tokens} x 32 heads, K=8 causal, head_dim 128), float64 serial C"
    out = {"metric": ATTN_METRIC, "value": round(value, 2), "unit": ATTN_UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": CONFIGS["attn"]["workload"], "sample_rows_per_step": rows},
           "impl": "reference",
           "cpu_baseline": {"value": round(value, 2), "unit": ATTN_UNIT, "cores": 1, "kind": "oracle",
                            "host": host_cpu(),
                            "sample": sample},
           "e2e": {"value": round(value, 2), "unit": ATTN_UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return out


def run_link_probe(args):
    """Host-link bandwidth that bounds the e2e legs: pinned (cudaHostAlloc)
    host->device and device->host copies of --link-gib GiB, one cudaMemcpyAsync
    each, timed with CUDA events on the copying stream (best and median of
    --steps copies after --warmup)."""
    import torch

    n = int(args.link_gib * (1 << 30))
    h = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    h.fill_(1)
    d = torch.empty(n, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    out = {"metric": "pinned host<->device copy bandwidth", "unit": "GB/s", "bytes_per_copy": n, "impl": "lpd",
           "steps": args.steps, "warmup": args.warmup}
    for name, dst, src in (("h2d", d, h), ("d2h", h, d)):
        times = []
        for k in range(args.warmup + args.steps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            dst.copy_(src, non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize()
            if k >= args.warmup:
                times.append(e0.elapsed_time(e1))
        times.sort()
        out[name] = {"best_gbs": round(n / (times[0] / 1e3) / 1e9, 1),
                     "median_gbs": round(n / (times[len(times) // 2] / 1e3) / 1e9, 1),
                     "slowest_gbs": round(n / (times[-1] / 1e3) / 1e9, 1)}
    print(json.dumps(out), flush=True)
    return out


def free_port() -> int:
    import socket

    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def launch_command(n_gpus: int, argv: list[str], port: int) -> list[str]:
    """torchrun command that runs this script as n_gpus ranks on this node
    (one process per GPU, rendezvous on 127.0.0.1)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n_gpus}",
            "--master-addr", "127.0.0.1", f"--master-port={port}", str(ROOT / "bench.py"), *argv]


def plan_launch(n_gpus: int, env: dict, visible_gpus: int) -> str:
    """'run' when this process is the job (one GPU, or a rank that torchrun
    started with a matching world size); 'relaunch' when --gpus N > 1 was
    given outside torchrun.  Refuses N above the visible GPU count and a
    world size that disagrees with --gpus."""
    if n_gpus < 1:
        raise SystemExit("--gpus must be at least 1")
    world = env.get("WORLD_SIZE")
    if world is not None:
        if int(world) != n_gpus:
            raise SystemExit(f"--gpus {n_gpus} under a launcher with WORLD_SIZE={world}")
        return "run"
    if n_gpus == 1:
        return "run"
    if n_gpus > visible_gpus:
        raise SystemExit(f"--gpus {n_gpus}: only {visible_gpus} GPU(s) visible")
    return "relaunch"


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["lpd", "reference"], default="lpd")
    ap.add_argument("--config", choices=sorted(CONFIGS), default="qwen")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=16, help="reference arm: rows per host thread per step")
    ap.add_argument("--transform", default=None,
                    help="logit transform chain on both sides, e.g. softcap:30,scale:1.4286")
    ap.add_argument("--entropy", action="store_true", help="time lpd_score_entropy instead of lpd_score")
    ap.add_argument("--backward", action="store_true", help="time lpd_logprob_backward of the train side")
    ap.add_argument("--topology", choices=["allgather_partials_fixed_merge", "allreduce_partials",
                                           "allgather_logits"], default=None,
                    help="sharded config: time lpd_score_sharded_topology with this reduction arm")
    ap.add_argument("--drift", action="store_true",
                    help="attn config: time lpd_attn_merge_order_drift instead of lpd_attn_merge")
    ap.add_argument("--link-probe", action="store_true",
                    help="measure pinned host<->device copy bandwidth (the e2e legs' bound) instead")
    ap.add_argument("--link-gib", type=float, default=4.0, help="link probe: GiB per copy")
    ap.add_argument("--batch", type=int, default=None, help="override B (small profiling cases only)")
    ap.add_argument("--seq", type=int, default=None, help="override T (small profiling cases only)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        import torch

        if plan_launch(args.gpus, dict(os.environ), torch.cuda.device_count()) == "relaunch":
            # N replicas, one process per GPU; each scores its own batch
            cmd = launch_command(args.gpus, list(sys.argv[1:] if argv is None else argv), free_port())
            raise SystemExit(subprocess.run(cmd).returncode)
    plan_launch(args.gpus, dict(os.environ), 0)
    if args.impl == "reference":
        return run_reference(args)
    if args.link_probe:
        return run_link_probe(args)
    return run_ours(args)


if __name__ == "__main__":
    main()
