"""bench.py --impl reference (the oracle, as it stands, timed on the host cores): the JSON line it prints,
checked on CPU.  The line carries the same metric, unit and direction as the CUDA arm's, an `impl` key,
a `cpu_baseline` describing the run and an end-to-end entry with no host-device bytes."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _reference_line(*args) -> dict:
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *args],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]  # one JSON line
    return json.loads(lines[0])


def test_reference_arm_json_line():
    d = _reference_line("--workload", "dec16k", "--steps", "2", "--warmup", "3")
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert (d["n_gpus"], d["steps"], d["warmup"]) == (1, 2, 3)
    assert d["higher_is_better"] is False and d["unit"] == "us/layer-step"
    assert d["value"] > 0 and abs(d["ms_per_step"] * 1e3 - d["value"]) <= 1e-6 * d["value"]
    assert d["data"] == "synthetic" and d["vs_baseline"] is None
    assert d["config"]["workload"].startswith("single-sequence decode")
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == d["value"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_reference_arm_two_ranks_one_line():
    """Launched like the CUDA arm at N = 2 (torchrun): rank 0 alone runs and prints; the other rank exits 0."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "dec16k"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["cores"] >= 1
