"""Host-side helpers of bench.py (no GPU): the command line, the chain
parser, the stage-1 launch count and the profile lookup."""
import subprocess
import sys
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]
sys.path.insert(0, str(ROOT))
import bench  # noqa: E402


def test_help_runs():
    out = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--help"], capture_output=True, text=True,
                         timeout=120)
    assert out.returncode == 0 and "--config" in out.stdout


def test_parse_chain():
    from logprob_drift_scoring_gb300 import binding as B

    assert bench.parse_chain("softcap:30,scale:1.5") == [(B.LPD_OP_SOFTCAP, 30.0), (B.LPD_OP_SCALE, 1.5)]
    with pytest.raises(KeyError):
        bench.parse_chain("cube:2")


@pytest.mark.parametrize("n,expect", [(0, 1), (4096, 1), (4097, 2), (32768, 2), (126976, 2), (126977, 1)])
def test_stage1_launch_count(n, expect):
    # two kernels (count, compact) for 2 to 31 blocks of 4096 rows, else one
    assert bench.select_launches(n) == expect


def test_profile_lookup_follows_the_kernel_source():
    prof = bench.profiled_row_kernel("qwen")
    h = bench.kernel_source_hash()
    text = (ROOT / "profiles" / "row_kernel_qwen.md").read_text()
    if f"kernel_source_sha1: {h}" in text:
        assert prof is not None and prof["traffic"] > 1.5e10
    else:
        assert prof is None  # a stale capture is never reported as traffic
    assert bench.profiled_row_kernel("no_such_config") is None


def test_launch_plan():
    # one GPU, or a rank torchrun started with the matching world size: run here
    assert bench.plan_launch(1, {}, 0) == "run"
    assert bench.plan_launch(4, {"WORLD_SIZE": "4"}, 0) == "run"
    # N > 1 outside torchrun: relaunch as N ranks, if N GPUs are visible
    assert bench.plan_launch(2, {}, 8) == "relaunch"
    with pytest.raises(SystemExit):
        bench.plan_launch(9, {}, 8)
    with pytest.raises(SystemExit):
        bench.plan_launch(2, {"WORLD_SIZE": "4"}, 8)
    with pytest.raises(SystemExit):
        bench.plan_launch(0, {}, 8)


def test_launch_command():
    cmd = bench.launch_command(4, ["--gpus", "4", "--steps", "7"], 29512)
    assert cmd[:3] == [sys.executable, "-m", "torch.distributed.run"]
    assert "--nproc-per-node=4" in cmd and "--nnodes=1" in cmd and "--master-port=29512" in cmd
    assert cmd[cmd.index("--master-addr") + 1] == "127.0.0.1"
    assert cmd[-5:] == [str(ROOT / "bench.py"), "--gpus", "4", "--steps", "7"]


def test_reference_arm_under_two_ranks_prints_one_line():
    # the reference arm launched under torchrun for N = 2 (CPU only): rank 0
    # alone scores and prints; n_gpus is the world size
    import json

    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2", "--master-addr",
           "127.0.0.1", f"--master-port={bench.free_port()}", str(ROOT / "bench.py"), "--impl", "reference",
           "--gpus", "2", "--config", "tiny", "--steps", "1", "--warmup", "3", "--ref-rows", "2"]
    out = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["cpu_baseline"]["cores"] >= 1
