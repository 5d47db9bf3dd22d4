"""Tensor-parallel split of one GDN layer's mixer and output projection.

Page "Qwen3.8-27B: from model structure to vLLM inference data flow", section
06 (TP4): the weights and heads are cut along the tensor-parallel dimension;
rank r of W holds key heads [r Hk/W, (r+1) Hk/W) and their value heads
[r Hv/W, (r+1) Hv/W), i.e. its own q, k and v channels of QKV0 and the conv,
its rows of the state and conv-history pools, its columns of Z, alpha and
beta, and the matching input columns of Wo (a row-parallel linear layer). Each
rank runs the mixer core on its heads alone; the only exchange is the sum of
the ranks' Wo partial outputs at the row-parallel boundary (the all-reduce).

This module holds the index arithmetic of that split and the per-rank step
(decode + Wo partial + all-reduce through torch.distributed). It works on numpy
arrays and torch tensors alike (the slicing is plain indexing).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class RankGeometry:
    """The head geometry one rank sees (the attribute names of a layer geometry)."""
    num_k_heads: int
    num_v_heads: int
    head_k_dim: int
    head_v_dim: int
    conv_kernel: int

    @property
    def channels(self) -> int:
        return 2 * self.num_k_heads * self.head_k_dim + self.num_v_heads * self.head_v_dim


@dataclass(frozen=True)
class HeadShard:
    """The heads of rank `rank` out of `world`: key heads k0 .. k0+hk-1, value heads v0 .. v0+hv-1."""
    rank: int
    world: int
    k0: int
    hk: int
    v0: int
    hv: int
    dk: int
    dv: int
    Hk: int
    Hv: int

    def channels(self) -> np.ndarray:
        """This rank's QKV0 / conv channels, in the layout [q heads | k heads | v heads] of its heads."""
        q = np.arange(self.k0 * self.dk, (self.k0 + self.hk) * self.dk)
        k = self.Hk * self.dk + q
        v = 2 * self.Hk * self.dk + np.arange(self.v0 * self.dv, (self.v0 + self.hv) * self.dv)
        return np.concatenate([q, k, v])

    def value_columns(self) -> slice:
        """Columns of a [*, Hv*dv] row (Ogate, Z flattened, the input side of Wo)."""
        return slice(self.v0 * self.dv, (self.v0 + self.hv) * self.dv)

    def value_heads(self) -> slice:
        """Value-head index range (alpha, beta, Z and the state pool's head axis)."""
        return slice(self.v0, self.v0 + self.hv)

    def geometry(self, conv_kernel: int) -> RankGeometry:
        return RankGeometry(self.hk, self.hv, self.dk, self.dv, conv_kernel)


def head_shard(dims, rank: int, world: int) -> HeadShard:
    """Rank `rank`'s heads; the key heads must split evenly (value head h reads key head h / (Hv/Hk),
    so whole key-head groups move together)."""
    Hk, Hv = dims.num_k_heads, dims.num_v_heads
    if world <= 0 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} out of a world of {world}")
    if Hk % world != 0 or Hv % Hk != 0:
        raise ValueError(f"{Hk} key heads / {Hv} value heads do not split over {world} ranks")
    hk = Hk // world
    G = Hv // Hk
    return HeadShard(rank, world, rank * hk, hk, rank * hk * G, hk * G, dims.head_k_dim, dims.head_v_dim, Hk, Hv)


def shard_step_inputs(shard: HeadShard, qkv0, conv_w, conv_hist, state, alpha, beta, z) -> dict:
    """The rank's slices of one step's inputs and slot pools (copies, contiguous):
    qkv0 [T, CH] -> [T, CH_r], conv_w [CH, K] -> [CH_r, K], conv_hist [Rs, CH, K-1] -> [Rs, CH_r, K-1],
    state [Rs, Hv, dv, dk] -> [Rs, hv, dv, dk], alpha/beta [T, Hv] -> [T, hv], z [T, Hv, dv] -> [T, hv, dv]."""
    ch = shard.channels()
    vh = shard.value_heads()

    def take(a, idx, axis):
        if isinstance(a, np.ndarray):
            return np.ascontiguousarray(np.take(a, idx, axis=axis))
        import torch
        return a.index_select(axis, torch.as_tensor(idx, device=a.device)).contiguous()

    def cut(a, sl, axis):
        index = [slice(None)] * a.ndim
        index[axis] = sl
        out = a[tuple(index)]
        return np.ascontiguousarray(out) if isinstance(out, np.ndarray) else out.contiguous()

    return {"qkv0": take(qkv0, ch, 1), "conv_w": take(conv_w, ch, 0), "conv_hist": take(conv_hist, ch, 1),
            "state": cut(state, vh, 1), "alpha": cut(alpha, vh, 1), "beta": cut(beta, vh, 1), "z": cut(z, vh, 1)}


def shard_out_proj_weight(shard: HeadShard, wo):
    """Wo [N_out, Hv*dv] (nn.Linear layout) -> the rank's input columns [N_out, hv*dv] (row-parallel)."""
    out = wo[:, shard.value_columns()]
    return np.ascontiguousarray(out) if isinstance(out, np.ndarray) else out.contiguous()


def decode_out_proj_step(b, shard: HeadShard, dims_rank, num_slots: int, inputs: dict, slot_idx, gamma, eps,
                         wo_rank, hidden, group=None, stream=None):
    """One decode step of the rank's heads, then its Wo partial, then the sum over ranks.

    inputs: the rank's slices (shard_step_inputs) as device tensors; the rank's state and history
    pools are updated in place. hidden [N, N_out] bf16 is the residual stream: rank 0 adds it into
    its partial, so the all-reduce yields hidden + Ogate Wo^T. Returns that [N, N_out] bf16 tensor
    (on every rank). With one rank, or no initialised process group, the partial is the result."""
    import torch
    import torch.distributed as dist
    N = inputs["qkv0"].shape[0]
    D = b.make_dims(dims_rank, num_slots)
    og = torch.empty((N, shard.hv * shard.dv), dtype=torch.bfloat16, device=inputs["qkv0"].device)
    b.gdn_decode_step(D, inputs["qkv0"], inputs["conv_w"], inputs["conv_hist"], inputs["state"], slot_idx,
                      inputs["alpha"], inputs["beta"], inputs["z"], gamma, eps, ogate=og, stream=stream)
    part = torch.empty((N, wo_rank.shape[0]), dtype=torch.bfloat16, device=og.device)
    b.gdn_out_proj(og, wo_rank, part, residual=hidden if shard.rank == 0 else None, stream=stream)
    if shard.world > 1 and dist.is_available() and dist.is_initialized():
        dist.all_reduce(part, op=dist.ReduceOp.SUM, group=group)
    return part
