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
