"""Seeded synthetic inputs for the GDN mixer core.

This module is shared by the tests, the benchmark and the oracle harness. It
only draws random numbers and lays them out; it holds none of the mixer's
arithmetic. Every array is a plain numpy array on the host:

* bf16 tensors are carried as ``uint16`` bit patterns (round-to-nearest-even
  from an fp32 draw), so the CPU oracle and the GPU receive identical bits;
* fp32 tensors are ``float32``; index tensors are ``int32``.

Shapes and distributions follow the workload descriptions that accompany the
"Qwen3.8-27B: from model structure to vLLM inference data flow" page
(ai-learning.gods8.com), section 01 LAYER-BY-LAYER, L00 data-structure table:
QKV0 ``[T, 10240]``, Z ``[T, 48, 128]``, S ``[R, 48, 128, 128]`` fp32,
conv history ``[R, 10240, 3]``.

Distributions (second parameter of N(.,.) is the standard deviation):
QKV0 ~ N(0,1) bf16; conv weights ~ N(0,0.25) fp32; Z ~ N(0,1) bf16;
alpha = exp(-u), u ~ U(0.001, 0.1); beta ~ U(0,1); gamma = 1; eps = 1e-6;
initial state ~ N(0,0.02) fp32; initial conv history ~ N(0,1) bf16.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Dims", "FULL_HEADS", "RANK_HEADS", "bf16_bits", "bf16_to_f32",
    "layer_params", "token_inputs", "slot_pool", "zero_pool", "slot_permutation",
    "loguniform_lengths", "pack_offsets", "decode_workload", "prefill_workload",
    "spec_workload",
]


@dataclass(frozen=True)
class Dims:
    """Head geometry of one GDN layer (key heads, value heads, head dims, conv taps)."""
    num_k_heads: int = 16
    num_v_heads: int = 48
    head_k_dim: int = 128
    head_v_dim: int = 128
    conv_kernel: int = 4

    @property
    def channels(self) -> int:
        """Packed QKV channel count: [Q heads | K heads | V heads]."""
        return 2 * self.num_k_heads * self.head_k_dim + self.num_v_heads * self.head_v_dim

    @property
    def group(self) -> int:
        return self.num_v_heads // self.num_k_heads


FULL_HEADS = Dims(16, 48, 128, 128, 4)
RANK_HEADS = Dims(4, 12, 128, 128, 4)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (nearest, ties to even) and return the bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_f32(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    out = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def layer_params(rng: np.random.Generator, dims: Dims) -> dict:
    """Per-layer parameters: depthwise conv taps [CH, K] and the RMSNorm gain [dv]."""
    return {
        "conv_w": _normal_f32(rng, (dims.channels, dims.conv_kernel), 0.25),
        "gamma": np.ones(dims.head_v_dim, dtype=np.float32),
        "eps": 1e-6,
    }


def token_inputs(rng: np.random.Generator, dims: Dims, T: int) -> dict:
    """Per-token inputs for T packed tokens."""
    u = rng.uniform(0.001, 0.1, size=(T, dims.num_v_heads))
    return {
        "qkv0": bf16_bits(_normal_f32(rng, (T, dims.channels), 1.0)),
        "z": bf16_bits(_normal_f32(rng, (T, dims.num_v_heads, dims.head_v_dim), 1.0)),
        "alpha": np.exp(-u).astype(np.float32),
        "beta": rng.uniform(0.0, 1.0, size=(T, dims.num_v_heads)).astype(np.float32),
    }


def slot_pool(rng: np.random.Generator, dims: Dims, num_slots: int) -> dict:
    """A cache pool of num_slots random recurrent states and conv histories."""
    return {
        "state": _normal_f32(rng, (num_slots, dims.num_v_heads, dims.head_v_dim, dims.head_k_dim), 0.02),
        "conv_hist": bf16_bits(_normal_f32(rng, (num_slots, dims.channels, dims.conv_kernel - 1), 1.0)),
    }


def zero_pool(dims: Dims, num_slots: int) -> dict:
    return {
        "state": np.zeros((num_slots, dims.num_v_heads, dims.head_v_dim, dims.head_k_dim), np.float32),
        "conv_hist": np.zeros((num_slots, dims.channels, dims.conv_kernel - 1), np.uint16),
    }


def slot_permutation(rng: np.random.Generator, num_requests: int, num_slots: int) -> np.ndarray:
    """Distinct slot indices for num_requests requests: a random permutation of the pool, truncated."""
    return rng.permutation(num_slots)[:num_requests].astype(np.int32)


def loguniform_lengths(rng: np.random.Generator, n: int, lo: int, hi: int) -> np.ndarray:
    """Request lengths drawn log-uniformly in [lo, hi] (integers)."""
    x = np.exp(rng.uniform(np.log(lo), np.log(hi), size=n))
    return np.clip(np.rint(x), lo, hi).astype(np.int32)


def pack_offsets(lengths) -> np.ndarray:
    """query_start_loc for packed requests: [0, l0, l0+l1, ...]."""
    out = np.zeros(len(lengths) + 1, dtype=np.int32)
    out[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return out


def decode_workload(dims: Dims, num_requests: int, num_slots: int | None = None, seed: int = 1) -> dict:
    """One decode step: num_requests tokens, each continuing a random slot of a random pool.

    The pool has num_slots = 2 * num_requests slots unless given; slot indices are a
    random permutation of the pool (256 requests over 512 slots for the headline case).
    """
    rng = np.random.default_rng(seed)
    Rs = 2 * num_requests if num_slots is None else num_slots
    w = {"dims": dims, "num_slots": Rs, "seed": seed}
    w.update(layer_params(rng, dims))
    w["slot_idx"] = slot_permutation(rng, num_requests, Rs)
    w.update(token_inputs(rng, dims, num_requests))
    w.update(slot_pool(rng, dims, Rs))
    return w


def prefill_workload(dims: Dims, lengths, seed: int = 3, zero_first_half: bool = True,
                     num_slots: int | None = None) -> dict:
    """Varlen prefill: requests of the given lengths packed along the token axis.

    With zero_first_half the first half of the requests starts from a zero state
    and zero conv history (has_init = 0); the rest continue from random slots.
    """
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int32)
    N = len(lengths)
    Rs = 2 * N if num_slots is None else num_slots
    w = {"dims": dims, "num_slots": Rs, "seed": seed, "lengths": lengths}
    w.update(layer_params(rng, dims))
    w["slot_idx"] = slot_permutation(rng, N, Rs)
    w["query_start_loc"] = pack_offsets(lengths)
    has_init = np.ones(N, dtype=np.uint8)
    if zero_first_half:
        has_init[: N // 2] = 0
    w["has_init"] = has_init
    w.update(token_inputs(rng, dims, int(lengths.sum())))
    w.update(slot_pool(rng, dims, Rs))
    return w


def spec_workload(dims: Dims, num_requests: int, num_pos: int = 4, seed: int = 4) -> dict:
    """Speculative verify: num_requests requests x num_pos positions (last sampled token + drafts).

    The pool holds one live slot and num_pos checkpoint slots per request
    (Rs = num_requests * (num_pos + 1)); accepted lengths are drawn U{0..num_pos-1}.
    """
    rng = np.random.default_rng(seed)
    Rs = num_requests * (num_pos + 1)
    w = {"dims": dims, "num_slots": Rs, "seed": seed, "num_pos": num_pos}
    w.update(layer_params(rng, dims))
    perm = rng.permutation(Rs).astype(np.int32)
    w["slot_idx"] = perm[:num_requests].copy()
    w["spec_slot_idx"] = perm[num_requests:].reshape(num_requests, num_pos).copy()
    w.update(token_inputs(rng, dims, num_requests * num_pos))
    w.update(slot_pool(rng, dims, Rs))
    w["accepted"] = rng.integers(0, num_pos, size=num_requests).astype(np.int32)
    return w


def fp8_codes(rng: np.random.Generator, shape) -> np.ndarray:
    """Random E4M3 bit patterns (uint8) with magnitudes from 0.25 up to 3.75: sign bit random,
    exponent field 5..8, mantissa field 0..7. These are stored codes, not a quantisation of anything."""
    sign = rng.integers(0, 2, size=shape, dtype=np.uint8) << 7
    e = rng.integers(5, 9, size=shape, dtype=np.uint8) << 3
    m = rng.integers(0, 8, size=shape, dtype=np.uint8)
    return (sign | e | m).astype(np.uint8)
