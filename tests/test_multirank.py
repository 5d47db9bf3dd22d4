"""Host logic of the multi-rank benchmark path on CPU ranks (gloo, world size 2).

The mixer core shards by request with no exchange, so the only cross-rank steps
are the barrier around the timed region and the max-over-ranks of its duration;
each rank draws its own independent batch.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier()
        t = bench.reduce_max(10.0 * (rank + 1))
        seed = bench.rank_seed(rank)
        gathered = [None] * world
        dist.all_gather_object(gathered, seed)
        out.put((rank, t, gathered))
    finally:
        dist.destroy_process_group()


def test_two_ranks_reduce_max_and_distinct_seeds():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, seeds in results:
        assert t == 20.0  # every rank sees the slowest rank's time
        assert len(set(seeds)) == world  # independent batches per rank


def test_single_process_reduce_is_identity():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    bench.barrier()  # no process group: a no-op


def test_algorithmic_byte_counts():
    import bench
    from gated_deltanet_linear_conv1d_gb300 import synth
    g = synth.FULL_HEADS
    # state read + write, history read + write, QKV0, z, alpha, beta, slot index, Ogate
    assert bench.decode_bytes_per_token(g) == 6291456 + 122880 + 20480 + 12288 + 384 + 4 + 12288
    assert bench.decode_bytes_per_launch(g, 256) == 256 * 6459780 + 163840 + 512
    assert bench.decode_bytes_per_token(synth.RANK_HEADS) == (
        2 * 12 * 128 * 128 * 4 + 2 * 2560 * 3 * 2 + 2560 * 2 + 12 * 128 * 2 + 12 * 8 + 4 + 12 * 128 * 2)
    bf16, tf32 = bench.prefill_flops(g, [64, 1, 65])
    chunks = 1 + 1 + 2
    assert tf32 == chunks * 48 * (2 * 2 * 128 * 64 * 64 + 2 * 128 * 128 * 64)
    assert bf16 == chunks * (48 * 4 * 128 * 64 * 128 + 16 * 2 * 128 * 64 * 128)


def test_reference_arm_prints_one_line(tmp_path):
    """bench.py --impl reference times the oracle on host cores and prints one JSON line with the
    keys the driver reads; under torchrun only rank 0 prints (a rank-1 run prints nothing)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "2", "--warmup", "3"]
    out = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600, check=True)
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["value"] > 0
    for key in ("metric", "unit", "higher_is_better", "config", "cpu_baseline", "e2e", "dtype"):
        assert key in line
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    env = dict(os.environ, RANK="1", WORLD_SIZE="2")
    out1 = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600, check=True, env=env)
    assert out1.stdout.strip() == ""
