"""The benchmark's reference arm (the float64 oracle timed on the host cores):
it runs without a GPU and prints the contract's JSON line."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _reference_line(*extra):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny-fp32-t512-c128", "--steps", "1", "--warmup", "0", *extra],
                         cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [x for x in out.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


@pytest.mark.parametrize("threads", [None, 1])
def test_reference_arm_line(threads):
    line = _reference_line(*(["--oracle-threads", str(threads)] if threads else []))
    assert line["impl"] == "reference"
    assert line["value"] > 0 and line["unit"] == "TFLOP/s"
    assert line["dtype"] == "f64" and line["higher_is_better"] is True
    base = line["cpu_baseline"]
    assert base["kind"] == "oracle" and base["value"] == line["value"]
    if threads:
        assert base["cores"] == threads        # the BLAS pool was capped before NumPy loaded
    else:
        assert base["cores"] >= 1
    e2e = line["e2e"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] == "tiny-fp32-t512-c128"


def test_reference_arm_under_torchrun_two_ranks():
    """Launched as the multi-GPU bench is (torchrun, two ranks, gloo on the
    CPU here): rank 0 alone times the oracle and prints the one line; the
    other rank exits 0 without work."""
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    out = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                          "--master-addr", "127.0.0.1", "--master-port", str(port),
                          os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--workload", "tiny-fp32-t512-c128", "--steps", "1", "--warmup", "0"],
                         cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [x for x in out.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, out.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0
