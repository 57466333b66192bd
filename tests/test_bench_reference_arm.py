"""bench.py's reference arm (the CPU oracle timed on the host cores) keeps the
one-JSON-line contract without a GPU: at N=1, and under torchrun with two
ranks, where rank 0 alone runs and prints and the other rank exits 0."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _json_lines(stdout):
    return [json.loads(line) for line in stdout.splitlines() if line.startswith("{")]


def _check_line(line, n_gpus, steps, warmup):
    assert line["impl"] == "reference"
    assert line["unit"] == "rows/s" and line["value"] > 0
    assert (line["n_gpus"], line["steps"], line["warmup"]) == (n_gpus, steps, warmup)
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["vs_baseline"] is None
    assert line["ms_per_step"] > 0 and line["dtype"] == "f64" and "synthetic" in line["data"]
    import bench
    # the CUDA arm's config for the same batch: the two lines describe one workload
    assert line["config"] == bench.training_config(line["config"]["rows_per_gpu"], n_gpus)
    assert 0 < line["rows_per_step"] <= line["config"]["rows_per_gpu"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["sample"] and cb["value"] == line["value"]
    e2e = line["e2e"]
    assert e2e == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_single_process_prints_one_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0",
                          "--rows", "2048"],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = _json_lines(out.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 1, 1, 0)


def test_two_ranks_print_one_line_from_rank_0():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--rows", "2048"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = _json_lines(out.stdout)
    assert len(lines) == 1
    _check_line(lines[0], 2, 1, 0)
