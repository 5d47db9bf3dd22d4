"""Tensor-parallel decode + Wo on one GPU: the ranks of a 2- and 4-way split run one after another
on their own slices (state and history pools included), their Wo partials are summed (what the
all-reduce does across GPUs), and the result matches the unsharded oracle layer."""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_conv1d_gb300 import synth, tp
from oracle import oracle
from tests import gdnutil as U

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("needs a GPU")
    from gated_deltanet_linear_conv1d_gb300 import build
    build.build()
    from gated_deltanet_linear_conv1d_gb300 import binding
    return binding


@pytest.mark.parametrize("world", [2, 4])
def test_tp_decode_out_proj_matches_unsharded_oracle(b, world):
    dims = synth.FULL_HEADS
    N = 64
    w = synth.decode_workload(dims, N, 2 * N, seed=61)
    rng = np.random.default_rng(62)
    wo = synth.bf16_bits((rng.normal(size=(5120, 6144)) / np.sqrt(6144)).astype(np.float32))
    hidden = synth.bf16_bits(rng.normal(size=(N, 5120)).astype(np.float32))
    d = U.to_device(w)
    wo_d, hid_d = U.dev_bf16(wo), U.dev_bf16(hidden)
    total = torch.zeros((N, 5120), dtype=torch.float32, device="cuda")
    states = []
    for r in range(world):
        s = tp.head_shard(dims, r, world)
        part = tp.shard_step_inputs(s, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["alpha"], d["beta"],
                                    d["z"])
        out = tp.decode_out_proj_step(b, s, s.geometry(dims.conv_kernel), w["num_slots"], part, d["slot_idx"],
                                      d["gamma"], w["eps"], tp.shard_out_proj_weight(s, wo_d), hid_d)
        total += out.float()  # the all-reduce of the ranks' partials
        states.append((s, part["state"]))
    torch.cuda.synchronize()
    qsl = np.arange(N + 1, dtype=np.int32)
    full = oracle.forward(dims, w["qkv0"], w["conv_w"], w["conv_hist"], w["state"], qsl, w["slot_idx"], w["alpha"],
                          w["beta"], w["z"], w["gamma"], w["eps"])
    ref = oracle.out_proj(synth.bf16_bits(full["ogate"].astype(np.float32)), wo, hidden)
    U.check_out(total.cpu().numpy().astype(np.float64), ref, f"hidden after Wo, {world} ranks")
    slots = w["slot_idx"]
    for s, st in states:
        got = st[torch.from_numpy(slots.astype(np.int64)).cuda()].cpu().numpy()
        U.check_state(got, full["state"][slots][:, s.value_heads()], 1e-4, f"state, rank {s.rank}")
