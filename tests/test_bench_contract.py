"""The benchmark's reference arm on the host cores (CPU only): one JSON line per run
with the contract's keys, for every workload, and under a two-rank launch only rank 0
prints it."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KEYS = {"impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
        "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"}


def _lines(cmd, **kw):
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=240, **kw)
    assert r.returncode == 0, r.stderr[-2000:]
    return [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]


@pytest.mark.parametrize("workload", ["qwen3-0.6b", "qwen3-1.7b-k4v4", "llama-3.2-1b-k8v4", "d256-mixed",
                                      "blocks-export", "prefill-qwen3-0.6b"])
def test_reference_arm_prints_one_contract_line(workload):
    out = _lines([sys.executable, "bench.py", "--impl", "reference", "--workload", workload,
                  "--steps", "3", "--warmup", "3"])
    assert len(out) == 1
    d = out[0]
    assert KEYS <= d.keys(), KEYS - d.keys()
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 3 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["vs_baseline"] is None and "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def test_reference_arm_under_two_ranks_prints_once():
    out = _lines([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                  "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
                  "--gpus", "2", "--steps", "3", "--warmup", "3"])
    assert len(out) == 1 and out[0]["impl"] == "reference"
