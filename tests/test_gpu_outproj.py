"""gdn_out_proj (the Wo projection plus residual add after the mixer core) against
the fp64 oracle: small ragged shapes element by element, the full layer shape
(6144 -> 5120) at the decode batch, and the in-place residual form."""
import numpy as np
import pytest
import torch

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


def _case(T, K, N, seed):
    rng = np.random.default_rng(seed)
    a = U.synth.bf16_bits(rng.normal(size=(T, K)).astype(np.float32))
    w = U.synth.bf16_bits((rng.normal(size=(N, K)) / np.sqrt(K)).astype(np.float32))
    r = U.synth.bf16_bits(rng.normal(size=(T, N)).astype(np.float32))
    return a, w, r


@pytest.mark.parametrize("T,K,N,res", [(1, 128, 64, False), (70, 256, 128, True), (257, 6144, 512, True)])
def test_out_proj_matches_oracle(b, T, K, N, res):
    a, w, r = _case(T, K, N, 80 + T)
    out = torch.zeros((T, N), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(b.gdn_out_proj_workspace_bytes(), dtype=torch.uint8, device="cuda")
    b.gdn_out_proj(U.dev_bf16(a), U.dev_bf16(w), out, residual=U.dev_bf16(r) if res else None, workspace=ws)
    U.check_out(U.host_f64_from_bf16(out), oracle.out_proj(a, w, r if res else None), "out")


def test_out_proj_full_layer_in_place_residual(b):
    """Ogate [256, 6144] x Wo^T [6144 -> 5120], residual added in place (out is the residual stream)."""
    T, K, N = 256, 6144, 5120
    a, w, r = _case(T, K, N, 90)
    hidden = U.dev_bf16(r)
    ws = torch.empty(b.gdn_out_proj_workspace_bytes(), dtype=torch.uint8, device="cuda")
    b.gdn_out_proj(U.dev_bf16(a), U.dev_bf16(w), hidden, residual=hidden, workspace=ws)
    U.check_out(U.host_f64_from_bf16(hidden), oracle.out_proj(a, w, r), "hidden")


def test_out_proj_without_workspace_and_empty(b):
    a, w, _ = _case(33, 128, 256, 91)
    out = torch.zeros((33, 256), dtype=torch.bfloat16, device="cuda")
    b.gdn_out_proj(U.dev_bf16(a), U.dev_bf16(w), out)
    U.check_out(U.host_f64_from_bf16(out), oracle.out_proj(a, w), "out")
    empty = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    b.gdn_out_proj(torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda"), U.dev_bf16(w), empty)


def _in_proj_case(dims, T, Dh, seed):
    rng = np.random.default_rng(seed)
    u = U.synth.bf16_bits(rng.normal(size=(T, Dh)).astype(np.float32))
    ws = [U.synth.bf16_bits((rng.normal(size=(n, Dh)) / np.sqrt(Dh)).astype(np.float32))
          for n in (dims.channels, dims.num_v_heads * dims.head_v_dim, 2 * dims.num_v_heads)]
    return u, ws


@pytest.mark.parametrize("heads,T,Dh,with_ab", [("small", 1, 64, True), ("small", 67, 200, False),
                                                ("full", 256, 5120, True)])
def test_in_proj_matches_oracle(b, heads, T, Dh, with_ab):
    """QKV0, Z and [a | b] = U W^T for each of the three in_proj weights; the full case is the layer's
    hidden size 5120 at the decode batch (5120 -> 10240 / 6144 / 96)."""
    dims = U.synth.FULL_HEADS if heads == "full" else U.synth.Dims(1, 2, 128, 128, 4)
    u, (w_qkv, w_z, w_ab) = _in_proj_case(dims, T, Dh, 95 + T)
    D = b.make_dims(dims, 1)
    qkv0 = torch.zeros((T, dims.channels), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros((T, dims.num_v_heads * dims.head_v_dim), dtype=torch.bfloat16, device="cuda")
    ab = torch.zeros((T, 2 * dims.num_v_heads), dtype=torch.float32, device="cuda") if with_ab else None
    ws = torch.empty(b.gdn_out_proj_workspace_bytes(), dtype=torch.uint8, device="cuda")
    b.gdn_in_proj(D, U.dev_bf16(u), U.dev_bf16(w_qkv), U.dev_bf16(w_z), qkv0, z,
                  w_ab=U.dev_bf16(w_ab) if with_ab else None, ab=ab, workspace=ws)
    U.check_out(U.host_f64_from_bf16(qkv0), oracle.out_proj(u, w_qkv), "qkv0")
    U.check_out(U.host_f64_from_bf16(z), oracle.out_proj(u, w_z), "z")
    if with_ab:
        got = ab.cpu().numpy().astype(np.float64)
        ref = oracle.out_proj(u, w_ab)
        # fp32 output: only the accumulation order differs from the fp64 sum
        assert np.abs(got - ref).max() <= 1e-4 * max(1.0, np.abs(ref).max()), "ab"
