"""Host-side logic of bench.py, on the CPU: the reference arm's JSON line, the
GPU arm refusing to run without a GPU (no CPU fallback), the labelling of
recorded ncu traffic, and the N>1 path over gloo at world size 2 (barrier and
max-over-ranks timing; under torchrun rank 0 alone prints the reference
line, the other rank exits 0 without work)."""
import hashlib
import json
import multiprocessing as mp
import os
import socket
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# with a GPU visible bench picks NCCL, one device per rank
needs_two_ranks = pytest.mark.skipif(torch.cuda.is_available() and torch.cuda.device_count() < 2,
                                     reason="two ranks need two GPUs when CUDA is present")

LINE_KEYS = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
             "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
             "cpu_baseline", "e2e")


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def run(cmd, timeout=600):
    env = dict(os.environ, KVR_REF_STEP_SECONDS="0.2")
    return subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=timeout)


def json_lines(out):
    return [json.loads(line) for line in out.splitlines() if line.startswith("{")]


def test_reference_line_contract():
    r = run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    for k in LINE_KEYS:
        assert k in d, k
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["steps"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["config"]["workload"] == "llama3_8b_128k"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_gpu_arm_refuses_to_run_without_a_gpu():
    r = run([sys.executable, "bench.py", "--steps", "3", "--warmup", "3", "--no-cpu-baseline"])
    assert r.returncode != 0
    assert json_lines(r.stdout) == []


def test_recorded_traffic_is_attached_only_to_its_capture(tmp_path, monkeypatch):
    import bench
    csrc = tmp_path / "sparse_decode_attention_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "a.cu").write_text("kernel a\n")
    (csrc / "b.h").write_text("header\n")
    digest = hashlib.sha256(b"kernel a\nheader\n").hexdigest()
    (tmp_path / "profiles").mkdir()
    rec = {"k": {"dram_bytes_per_launch": 1234, "sources": ["a.cu", "b.h"],
                 "workload": "w128", "sources_sha256": digest},
           "k/w1m": {"dram_bytes_per_launch": 5678, "sources": ["a.cu", "b.h"],
                     "workload": "w1m", "sources_sha256": digest}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_traffic("k", "w128") == 1234
    assert bench.measured_traffic("k", "w1m") == 5678       # its own capture
    assert bench.measured_traffic("k", "w32k") is None      # another workload
    assert bench.measured_traffic("k_mag", "w128") is None  # another kernel variant
    (csrc / "a.cu").write_text("kernel a, changed\n")
    assert bench.measured_traffic("k", "w128") is None      # sources changed since
    assert bench.measured_traffic("k", "w1m") is None


def _gloo_rank(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      LOCAL_RANK=str(rank), WORLD_SIZE="2")
    import torch.distributed as dist
    import bench
    r, local, world = bench.dist_setup(None)
    bench.barrier(world)
    m = bench.max_over_ranks(1.5 * (rank + 1), world)
    bench.barrier(world)
    q.put((r, local, world, m))
    dist.destroy_process_group()


@needs_two_ranks
def test_dist_helpers_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_gloo_rank, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert got == [(0, 0, 2, 3.0), (1, 1, 2, 3.0)]
    assert all(p.exitcode == 0 for p in procs)


@needs_two_ranks
def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = free_port()
    r = run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
             "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
             "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = json_lines(r.stdout)
    assert len(lines) == 1
    assert lines[0]["impl"] == "reference" and lines[0]["n_gpus"] == 2


def test_algorithmic_bytes_follow_the_documented_per_unit_counts():
    """Per unit and step at pool P = N - W, C' = min(C, P), k' = min(k, C'),
    row = 2d bytes: select P d/8 + C' row + G d 2 (records: C' 6d/8 in place
    of the rows), attend (k' + W) 2 row + G d 2, encode row + d/8 (records:
    + 6d/8); times the B Hkv units. At 128K: 33.55 MB and 8.92 MB."""
    import bench
    import workloads as wl
    w = wl.LLAMA_128K
    P = w.N - w.W
    Cp, row, G, U = min(w.C, P), 2 * w.d, w.Hq // w.Hkv, w.B * w.Hkv
    kp = min(w.k, Cp)
    ab = bench.algorithmic_bytes(w)
    assert ab["units"] == U
    assert ab["select"] == U * (P * w.d // 8 + Cp * row + G * w.d * 2) == 33546240
    assert ab["attend"] == U * ((kp + w.W) * 2 * row + G * w.d * 2) == 8921088
    assert ab["encode"] == U * (row + w.d // 8)
    rs = bench.algorithmic_bytes(w, "rsq")
    assert rs["select"] == U * (P * w.d // 8 + Cp * 6 * w.d // 8 + G * w.d * 2)
    assert rs["encode"] == U * (row + w.d // 8 + 6 * w.d // 8)
