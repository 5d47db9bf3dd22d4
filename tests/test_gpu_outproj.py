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
    b.gdn_out_proj(U.dev_bf16(a), U.dev_bf16(w), out, residual=U.dev_bf16(r) if res else None)
    U.check_out(U.host_f64_from_bf16(out), oracle.out_proj(a, w, r if res else None), "out")


def test_out_proj_full_layer_in_place_residual(b):
    """Ogate [256, 6144] x Wo^T [6144 -> 5120], residual added in place (out is the residual stream)."""
    T, K, N = 256, 6144, 5120
    a, w, r = _case(T, K, N, 90)
    hidden = U.dev_bf16(r)
    b.gdn_out_proj(U.dev_bf16(a), U.dev_bf16(w), hidden, residual=hidden)
    U.check_out(U.host_f64_from_bf16(hidden), oracle.out_proj(a, w, r), "hidden")


def test_out_proj_small_and_empty(b):
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
    b.gdn_in_proj(D, U.dev_bf16(u), U.dev_bf16(w_qkv), U.dev_bf16(w_z), qkv0, z,
                  w_ab=U.dev_bf16(w_ab) if with_ab else None, ab=ab)
    U.check_out(U.host_f64_from_bf16(qkv0), oracle.out_proj(u, w_qkv), "qkv0")
    U.check_out(U.host_f64_from_bf16(z), oracle.out_proj(u, w_z), "z")
    if with_ab:
        got = ab.cpu().numpy().astype(np.float64)
        ref = oracle.out_proj(u, w_ab)
        # fp32 output: only the accumulation order differs from the fp64 sum
        assert np.abs(got - ref).max() <= 1e-4 * max(1.0, np.abs(ref).max()), "ab"


# ---------------------------------------------------------------- the GEMM's schedules and tile shapes

@pytest.mark.parametrize("T,K,N", [
    (1, 200, 136),      # swapped tiles (<= 256 tokens): one token, a ragged K slice, a partial weight tile
    (17, 6144, 520),    # swapped, 5 weight tiles: K split over clusters of 4 CTAs
    (128, 64, 8),       # swapped, one K slice (no split possible), eight weight rows
    (129, 1000, 1032),  # swapped, the second half of the token columns partly used, K split 4 ways
    (256, 5120, 384),   # swapped, the full token width (N = 256 MMAs), K split 4 ways
    (256, 6144, 5120),  # the decode-batch Wo: 40 weight tiles, K split 3 ways
    (257, 640, 264),    # 128-token tiles (more than 256 tokens), a partial token tile, K split 4 ways
    (1000, 6144, 512),  # 128-token tiles, 16 tiles, K split 4 ways
    (20000, 256, 1032), # 128-token tiles, many waves: whole tiles on persistent CTAs
])
def test_gemm_schedules_match_oracle(b, T, K, N):
    a, w, r = _case(T, K, N, 300 + T)
    out = U.dev_bf16(r)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.gdn_out_proj(U.dev_bf16(a), U.dev_bf16(w), out, residual=out, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    U.check_out(U.host_f64_from_bf16(out), oracle.out_proj(a, w, r), "out")
    # the split K adds its partial tiles in a fixed order: a second call gives the same bits
    out2 = U.dev_bf16(r)
    b.gdn_out_proj(U.dev_bf16(a), U.dev_bf16(w), out2, residual=out2, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    assert torch.equal(out, out2)


@pytest.mark.parametrize("T", [3, 300])
def test_in_proj_three_outputs_one_launch_ragged(b, T):
    """Three outputs of ragged widths (a 4/12-head layer: 2560, 1536 and 24 fp32 columns) from one
    input, swapped (3 tokens) and 128-token (300 tokens) tiles."""
    dims = U.synth.RANK_HEADS
    u, (w_qkv, w_z, w_ab) = _in_proj_case(dims, T, 5120, 500 + T)
    D = b.make_dims(dims, 1)
    qkv0 = torch.zeros((T, dims.channels), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros((T, dims.num_v_heads * dims.head_v_dim), dtype=torch.bfloat16, device="cuda")
    ab = torch.zeros((T, 2 * dims.num_v_heads), dtype=torch.float32, device="cuda")
    b.gdn_in_proj(D, U.dev_bf16(u), U.dev_bf16(w_qkv), U.dev_bf16(w_z), qkv0, z, w_ab=U.dev_bf16(w_ab), ab=ab)
    U.check_out(U.host_f64_from_bf16(qkv0), oracle.out_proj(u, w_qkv), "qkv0")
    U.check_out(U.host_f64_from_bf16(z), oracle.out_proj(u, w_z), "z")
    ref = oracle.out_proj(u, w_ab)
    assert np.abs(ab.cpu().numpy().astype(np.float64) - ref).max() <= 1e-4 * max(1.0, np.abs(ref).max())
