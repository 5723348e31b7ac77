"""Host-side logic of bench.py on the CPU: rank sharding, the max-over-ranks timing
reduction across two gloo ranks, and the CPU reference arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_shard_sequences_weak_and_strong():
    for world in (1, 2, 3, 8):
        for rank in range(world):
            assert np.array_equal(bench.shard_sequences(64, world, rank, "weak"), np.arange(64))
        parts = [bench.shard_sequences(67, world, r, "strong") for r in range(world)]
        assert np.array_equal(np.concatenate(parts), np.arange(67))
        assert max(len(p) for p in parts) - min(len(p) for p in parts) <= (67 + world - 1) // world


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank), CSA2_BENCH_BACKEND="gloo")
    w, r, _ = bench.dist_setup()
    import torch.distributed as dist
    try:
        bench.barrier(w)
        got = bench.reduce_max(1.5 + 2.0 * r, w, "cpu")
        q.put((r, w, got))
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 3.5), (1, 2, 3.5)]


def test_reference_arm_line_on_tiny_workload():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "1", "--warmup", "0",
                          "--cpu-sample", "1"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["unit"] == bench.UNIT


def test_reference_arm_line_on_decode_append():
    """The write path's reference arm on the decode-time append workload (2 of its 64 new
    tokens through all 12800 projection columns)."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "decode_append", "--steps", "1", "--warmup", "0",
                          "--cpu-sample", "2"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "tokens/s"
    assert line["config"]["workload"].startswith("decode_append") and line["config"]["tokens"] == 64


def test_reference_arm_line_on_draft_chunk():
    """The multi-query workload's reference arm: the oracle on one of its 256 draft queries,
    with the line's metric, unit and workload those of the GPU arm."""
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "draft_chunk", "--steps", "1", "--warmup", "0",
                          "--cpu-sample", "1"], capture_output=True, text=True, timeout=600,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "queries/s"
    assert line["metric"] == bench.CHUNK_METRIC
    assert line["config"]["workload"] == "draft_chunk_64x4x16384"
    assert line["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("world", [2])
def test_reference_arm_under_torchrun_prints_once(world):
    env = dict(os.environ, CSA2_BENCH_BACKEND="gloo")
    out = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                          f"--nproc-per-node={world}", "--master-addr", "127.0.0.1",
                          "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
                          "--impl", "reference", "--workload", "tiny", "--steps", "1",
                          "--warmup", "0", "--cpu-sample", "1", "--gpus", str(world)],
                         capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    assert json.loads(lines[0])["n_gpus"] == world


def test_traffic_hash_ignores_comments_only():
    """The traffic counters stay tied to the index kernels' code: comments and blank space
    do not change the hash, code does."""
    a = "int f(int x) {  // doubled\n  return 2 * x; /* note */ }\n"
    b = "// header\nint f(int x) {\n\n  return 2 * x;\n}\n"
    c = "int f(int x) { return 3 * x; }"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)
    assert len(bench.kernel_hash()) == 16
