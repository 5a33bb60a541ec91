"""The reference arm of bench.py (`--impl reference`: the fp64 oracle timed on
the host cores) runs without a GPU: its JSON line must carry the contract's
keys for every workload name the bench accepts, on a tiny sample."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
        "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "impl",
        "cpu_baseline", "e2e"}


@pytest.mark.parametrize("workload", ["gdn", "gdn_small", "kda", "rwkv6", "fork", "prefill_kda", "checkpoint",
                                      "readstate"])
def test_reference_arm_line(workload):
    env = dict(os.environ, DL_REF_SLOT_HEADS="16", DL_REF_TOKENS="4")
    env.pop("WORLD_SIZE", None)
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", workload, "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "tokens·heads/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


@pytest.mark.parametrize("workload", ["gdn", "gdn_small", "kda", "rwkv6"])
def test_reference_arm_config_is_ours(workload):
    """Both arms describe a decode workload with the same `config` object."""
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    args = argparse.Namespace(staging="fused", no_graph=False, eager=False, M=0)
    w = bench.WORKLOADS[workload]
    ours = bench.decode_config(w, w["M"], args, 1)
    env = dict(os.environ, DL_REF_SLOT_HEADS="16", DL_REF_TOKENS="4")
    env.pop("WORLD_SIZE", None)
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", workload, "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    d = json.loads([l for l in p.stdout.splitlines() if l.startswith("{")][0])
    assert d["config"] == ours
