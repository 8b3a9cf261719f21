"""The benchmark's output contract, checked on the host with the reference
arm (the oracle on the host cores; no GPU): one JSON line with the keys the
driver reads, and under torchrun with two ranks still exactly one line
(rank 0 runs and prints, the other rank exits 0 without work).  Also the
per-step launch count behind the line's gpu_launches, on every workload and
path, and (on a GPU) our arm's line."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ARGS = ["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"]


def _lines(stdout):
    return [l for l in stdout.splitlines() if l.startswith("{")]


def _check_line(d, n_gpus):
    for k in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference"
    assert d["n_gpus"] == n_gpus and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert "workload" in d["config"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, "bench.py"] + ARGS, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _lines(r.stdout)
    assert len(lines) == 1, r.stdout
    _check_line(json.loads(lines[0]), 1)


def test_reference_arm_under_torchrun_two_ranks():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--gpus", "2"] + ARGS
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _lines(r.stdout)
    assert len(lines) == 1, r.stdout
    _check_line(json.loads(lines[0]), 2)


@pytest.mark.gpu
def test_our_arm_prints_the_contract_keys():
    r = subprocess.run([sys.executable, "bench.py", "--workload", "tiny", "--steps", "5", "--warmup", "3",
                        "--e2e-steps", "3", "--cpu-seconds", "0.5"], cwd=ROOT, capture_output=True, text=True,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = _lines(r.stdout)
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 5 and d["value"] > 0
    roof = d["roofline"]
    for k in ("bound", "achieved", "peak", "unit", "frac", "traffic"):
        assert k in roof, k
    assert roof["bound"] == "hbm" and roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"])
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 5 * 2                      # layout + dispatch in one kernel, combine
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1


@pytest.mark.parametrize("cfg,path,per_step", [
    ("tiny", "rank", 2),        # few tokens: layout and dispatch in one kernel, then the combine
    ("decode", "rank", 2),
    ("dsv3", "rank", 3),        # one-cluster layout, dispatch, combine
    ("skewed", "rank", 3),
    ("large", "rank", 5),       # T * R > 2^19: the tiled layout's three kernels
    ("dsv3", "expanded", 3),
    ("dsv3", "hierarchical", 5),
    ("large", "hierarchical", 7),
])
def test_launches_per_step(cfg, path, per_step):
    """The bench's gpu_launches claim per step, for the library's launch
    plans (the one-kernel limits of ep_layout_and_dispatch, the tiled
    layout beyond 2^19 token-rank pairs, two kernels per stage on the
    two-stage path)."""
    import bench
    from combine_ep_get_gb300.inputs import CONFIGS
    c = CONFIGS[cfg]
    fused = path == "rank"
    got = bench.kernels_per_step(c.T, c.R, path == "expanded", path == "hierarchical", fused, c.K, c.E)
    assert got == per_step
