"""bench.py pieces that need no GPU: the reference arm's JSON line (the oracle timed
on the host cores) and the SSD leg's algorithmic byte and flop counts."""
import json
import os
import subprocess
import sys
from types import SimpleNamespace

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def run_bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("args", [("--workload", "tiny_f32"), ("--ssd", "--workload", "ssd_tiny")])
def test_reference_arm_line(args):
    """The reference arm prints one JSON line with the contract's keys, its own
    cpu_baseline and an e2e object that moves no bytes."""
    d = run_bench("--impl", "reference", "--steps", "1", "--warmup", "1", *args)
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["value"] > 0 and d["unit"] == "tokens*channels/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"] == args[-1]


def test_ssd_algorithmic_counts():
    """Bytes and flops of the 2.7B-shaped SSD layer, counted by hand: x, z, out
    (4 x 4096 x 80 x 64 bf16 each), dt (4 x 4096 x 80 bf16), B and C (4 x 4096 x 128
    bf16 each), A, D, dt_bias (80 fp32 each), the final state (4 x 80 x 64 x 128 fp32);
    per 128-step chunk (32 per sequence) and head 2 (128*129/2 (128 + 64) + 2 * 128 * 64 * 128)
    flops."""
    import bench
    w = SimpleNamespace(batch=4, seqlen=4096, nheads=80, headdim=64, ngroups=1, dstate=128, z=True)
    byt, flops = bench.ssd_algorithmic(w)
    assert byt == 3 * 167772160 + 2621440 + 2 * 4194304 + 960 + 10485760
    assert flops == 4 * 80 * 32 * 2 * (8256 * 192 + 2 * 128 * 64 * 128)
