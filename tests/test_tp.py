"""Tensor-parallel split of the mixer and Wo (host logic, CPU): the head and channel split of the
page's TP4 table, and on two gloo ranks the sharded oracle step + Wo partials + all-reduce against
the unsharded oracle."""
import os
import socket

import numpy as np
import pytest

from gated_deltanet_linear_conv1d_gb300 import synth, tp

torch = pytest.importorskip("torch")


def test_tp4_heads_follow_the_page_table():
    """Section 06: rank r holds GDN QK heads 4r..4r+3 and V heads 12r..12r+11; every channel lands on
    exactly one rank, 2560 per rank."""
    dims = synth.FULL_HEADS
    seen = []
    for r in range(4):
        s = tp.head_shard(dims, r, 4)
        assert (s.k0, s.hk, s.v0, s.hv) == (4 * r, 4, 12 * r, 12)
        ch = s.channels()
        assert len(ch) == 2560 == s.geometry(4).channels
        seen.append(ch)
    allc = np.concatenate(seen)
    assert np.array_equal(np.sort(allc), np.arange(dims.channels))
    with pytest.raises(ValueError):
        tp.head_shard(dims, 0, 3)  # 16 key heads do not split over 3 ranks


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer(seed=60, N=6):
    dims = synth.Dims(4, 12, 128, 128, 4)
    w = synth.decode_workload(dims, N, 2 * N, seed=seed)
    rng = np.random.default_rng(seed + 1)
    wo = synth.bf16_bits((rng.normal(size=(256, dims.num_v_heads * dims.head_v_dim)) / 40.0).astype(np.float32))
    hidden = synth.bf16_bits(rng.normal(size=(N, 256)).astype(np.float32))
    return dims, w, wo, hidden


def _oracle_step(dims, w, part):
    from oracle import oracle
    N = len(w["slot_idx"])
    qsl = np.arange(N + 1, dtype=np.int32)
    return oracle.forward(dims, part["qkv0"], part["conv_w"], part["conv_hist"], part["state"], qsl, w["slot_idx"],
                          part["alpha"], part["beta"], part["z"], w["gamma"], w["eps"])


def _rank(rank, world, port, q):
    import torch.distributed as dist
    from oracle import oracle
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dims, w, wo, hidden = _layer()
        s = tp.head_shard(dims, rank, world)
        part = tp.shard_step_inputs(s, w["qkv0"], w["conv_w"], w["conv_hist"], w["state"], w["alpha"], w["beta"],
                                    w["z"])
        r = _oracle_step(s.geometry(dims.conv_kernel), w, part)
        og_bits = synth.bf16_bits(r["ogate"].astype(np.float32))
        partial = oracle.out_proj(og_bits, tp.shard_out_proj_weight(s, wo), hidden if rank == 0 else None)
        t = torch.from_numpy(partial)
        dist.all_reduce(t)  # the row-parallel boundary: sum of the ranks' partials
        q.put((rank, t.numpy(), r["state"], og_bits))
    finally:
        dist.destroy_process_group()


def test_two_ranks_sum_to_the_unsharded_layer():
    import torch.multiprocessing as mp
    from oracle import oracle
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict()
    for _ in range(world):
        rank, out, state, og = q.get(timeout=300)
        got[rank] = (out, state, og)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    dims, w, wo, hidden = _layer()
    full = _oracle_step(dims, w, {k: w[k] for k in ("qkv0", "conv_w", "conv_hist", "state", "alpha", "beta", "z")})
    og_full = synth.bf16_bits(full["ogate"].astype(np.float32))
    ref = oracle.out_proj(og_full, wo, hidden)
    for rank in range(world):
        s = tp.head_shard(dims, rank, world)
        out, state, og = got[rank]
        np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)   # every rank holds the reduced result
        np.testing.assert_array_equal(og, og_full[:, s.value_columns()])  # head-local mixer outputs
        np.testing.assert_array_equal(state, full["state"][:, s.value_heads()])
