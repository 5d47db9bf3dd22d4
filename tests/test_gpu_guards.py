"""Stray writes and determinism. Every output buffer of every entry point is the middle of a
larger allocation whose 4 KiB guard bands before and after are filled with a byte pattern; after
the call the bands must be unchanged (a write past either end of any output shows). The state and
history pools are checked the same way, and the slots a call does not name must keep their bits.
The chunked prefill and the speculative verify, run twice on the same inputs, give the same bits."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gated_deltanet_linear_conv1d_gb300 import synth  # noqa: E402
from tests import gdnutil as U  # noqa: E402

GUARD = 4096      # bytes on each side (a multiple of 256, so the middle keeps its alignment)
PATTERN = 0xA5


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_linear_conv1d_gb300 import build
    build.build()
    from gated_deltanet_linear_conv1d_gb300 import binding
    return binding


class Guarded:
    """A device tensor of the given shape and dtype placed between two guard bands."""

    def __init__(self, shape, dtype, fill=None):
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((GUARD + n + GUARD,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + n].view(dtype).view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def check(self, what):
        torch.cuda.synchronize()
        lo, hi = self.raw[:GUARD], self.raw[-GUARD:]
        assert bool((lo == PATTERN).all()), f"{what}: write below the buffer"
        assert bool((hi == PATTERN).all()), f"{what}: write past the buffer"


def _pools(d):
    return Guarded(d["state"].shape, torch.float32, d["state"]), Guarded(d["conv_hist"].shape, torch.bfloat16,
                                                                          d["conv_hist"])


def test_decode_writes_nothing_outside_its_outputs(b):
    geom = synth.FULL_HEADS
    w = synth.decode_workload(geom, 24, 64, seed=81)
    d = U.to_device(w)
    D = b.make_dims(geom, w["num_slots"])
    st, hist = _pools(d)
    o = Guarded((24, geom.num_v_heads, geom.head_v_dim), torch.bfloat16)
    og = Guarded((24, geom.num_v_heads * geom.head_v_dim), torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.gdn_decode_step(D, d["qkv0"], d["conv_w"], hist.t, st.t, d["slot_idx"], d["alpha"], d["beta"], d["z"],
                      d["gamma"], w["eps"], o=o.t, ogate=og.t, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    for g, what in ((st, "state"), (hist, "history"), (o, "o"), (og, "ogate")):
        g.check(what)
    untouched = np.setdiff1d(np.arange(w["num_slots"]), w["slot_idx"])
    idx = torch.from_numpy(untouched.astype(np.int64)).cuda()
    assert torch.equal(st.t[idx].cpu(), torch.from_numpy(w["state"][untouched]))
    np.testing.assert_array_equal(U.host_bits(hist.t[idx]), w["conv_hist"][untouched])


def test_prefill_writes_nothing_outside_its_outputs_and_repeats_bit_for_bit(b):
    geom = synth.FULL_HEADS
    lengths = [70, 1, 130, 0, 64, 3]
    w = synth.prefill_workload(geom, lengths, seed=82)
    T = int(sum(lengths))
    runs = []
    for _ in range(2):
        d = U.to_device(w)
        D = b.make_dims(geom, w["num_slots"])
        st, hist = _pools(d)
        o = Guarded((T, geom.num_v_heads, geom.head_v_dim), torch.bfloat16)
        og = Guarded((T, geom.num_v_heads * geom.head_v_dim), torch.bfloat16)
        ws = Guarded((b.gdn_prefill_workspace_bytes(D, len(lengths), T),), torch.uint8)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        b.gdn_chunk_prefill(D, d["qkv0"], d["conv_w"], hist.t, st.t, d["query_start_loc"], d["slot_idx"],
                            d["alpha"], d["beta"], d["z"], d["gamma"], w["eps"], o=o.t, ogate=og.t,
                            has_init=d["has_init"], workspace=ws.t, dev_err=err)
        assert b.gdn_read_device_error(err) == 0
        for g, what in ((st, "state"), (hist, "history"), (o, "o"), (og, "ogate"), (ws, "workspace")):
            g.check(what)
        runs.append((st.t, hist.t, o.t, og.t))
    for x, y in zip(*runs):
        assert torch.equal(x, y), "a second prefill on the same inputs gave other bits"
    # the empty request (length 0) and slots no request names keep their bits
    named = w["slot_idx"][np.array(lengths) > 0]
    untouched = np.setdiff1d(np.arange(w["num_slots"]), named)
    idx = torch.from_numpy(untouched.astype(np.int64)).cuda()
    assert torch.equal(runs[0][0][idx].cpu(), torch.from_numpy(w["state"][untouched]))


def test_spec_verify_writes_nothing_outside_its_outputs_and_repeats_bit_for_bit(b):
    geom = synth.FULL_HEADS
    N = 12
    w = synth.spec_workload(geom, N, num_pos=4, seed=83)
    P = w["num_pos"]
    runs = []
    for _ in range(2):
        d = U.to_device(w)
        D = b.make_dims(geom, w["num_slots"])
        st, hist = _pools(d)
        og = Guarded((N * P, geom.num_v_heads * geom.head_v_dim), torch.bfloat16)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        b.gdn_spec_verify(D, d["qkv0"], d["conv_w"], hist.t, st.t, d["slot_idx"], d["spec_slot_idx"], d["alpha"],
                          d["beta"], d["z"], d["gamma"], w["eps"], ogate=og.t, dev_err=err)
        assert b.gdn_read_device_error(err) == 0
        for g, what in ((st, "state"), (hist, "history"), (og, "ogate")):
            g.check(what)
        runs.append((st.t, hist.t, og.t))
    for x, y in zip(*runs):
        assert torch.equal(x, y), "a second verify on the same inputs gave other bits"


def test_standalone_kernels_write_nothing_outside_their_outputs(b):
    geom = synth.FULL_HEADS
    rng = np.random.default_rng(84)
    # conv update
    lengths = [5, 64, 1, 77]
    w = synth.prefill_workload(geom, lengths, seed=85)
    d = U.to_device(w)
    T = int(sum(lengths))
    D = b.make_dims(geom, w["num_slots"])
    hist = Guarded(d["conv_hist"].shape, torch.bfloat16, d["conv_hist"])
    y = Guarded((T, geom.channels), torch.bfloat16)
    b.gdn_conv_update(D, d["qkv0"], d["conv_w"], hist.t, d["query_start_loc"], d["slot_idx"], y.t,
                      has_init=d["has_init"])
    hist.check("conv history")
    y.check("conv y")
    # gated RMSNorm
    o = U.dev_bf16(synth.bf16_bits(rng.standard_normal((33, 48, 128)).astype(np.float32)))
    z = U.dev_bf16(synth.bf16_bits(rng.standard_normal((33, 48, 128)).astype(np.float32)))
    gamma = torch.ones(128, device="cuda")
    og = Guarded((33, 48 * 128), torch.bfloat16)
    b.gdn_gated_rmsnorm(o, z, gamma, 1e-6, og.t)
    og.check("gated rmsnorm")
    # input RMSNorm with the residual add
    x = U.dev_bf16(synth.bf16_bits(rng.standard_normal((33, 5120)).astype(np.float32)))
    res = Guarded((33, 5120), torch.bfloat16, x * 0.5)
    u = Guarded((33, 5120), torch.bfloat16)
    b.gdn_rmsnorm(x, torch.ones(5120, device="cuda"), 1e-6, u.t, residual=res.t)
    res.check("rmsnorm residual")
    u.check("rmsnorm out")


@pytest.mark.parametrize("T", [3, 256, 1000, 19500])
def test_projections_write_nothing_outside_their_outputs(b, T):
    """Wo (both tile shapes and the cluster split of the decode size), the three in_proj outputs, and
    the FP8 path (quantisers and GEMM: the decode-sized split through the workspace, and at 19,500
    tokens the CTA-pair schedule over an odd number of row tiles)."""
    rng = np.random.default_rng(86 + T)
    K, N = 512, 384
    a = U.dev_bf16(synth.bf16_bits(rng.standard_normal((T, K)).astype(np.float32)))
    wt = U.dev_bf16(synth.bf16_bits((rng.standard_normal((N, K)) / np.sqrt(K)).astype(np.float32)))
    out = Guarded((T, N), torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    b.gdn_out_proj(a, wt, out.t, dev_err=err)
    out.check("out_proj")
    geom = synth.RANK_HEADS
    D = b.make_dims(geom, 4)
    Dh = 512
    hid = U.dev_bf16(synth.bf16_bits(rng.standard_normal((T, Dh)).astype(np.float32)))
    wq = U.dev_bf16(synth.bf16_bits((rng.standard_normal((geom.channels, Dh)) / 23).astype(np.float32)))
    wz = U.dev_bf16(synth.bf16_bits((rng.standard_normal((geom.num_v_heads * 128, Dh)) / 23).astype(np.float32)))
    wab = U.dev_bf16(synth.bf16_bits((rng.standard_normal((2 * geom.num_v_heads, Dh)) / 23).astype(np.float32)))
    qkv0 = Guarded((T, geom.channels), torch.bfloat16)
    zz = Guarded((T, geom.num_v_heads * 128), torch.bfloat16)
    ab = Guarded((T, 2 * geom.num_v_heads), torch.float32)
    b.gdn_in_proj(D, hid, wq, wz, qkv0.t, zz.t, w_ab=wab, ab=ab.t, dev_err=err)
    for g, what in ((qkv0, "qkv0"), (zz, "z"), (ab, "ab")):
        g.check(what)
    x8 = Guarded((T, K), torch.uint8)
    xs = Guarded((T, K // 128), torch.float32)
    b.gdn_fp8_quant_act(a, x8.t, xs.t)
    w8 = Guarded((N, K), torch.uint8)
    wsc = Guarded(((N + 127) // 128, K // 128), torch.float32)
    b.gdn_fp8_quant_weight(wt, w8.t, wsc.t)
    out8 = Guarded((T, N), torch.bfloat16)
    wsp = Guarded((max(256, b.gdn_fp8_linear_workspace_bytes(T, K, N)),), torch.uint8)
    b.gdn_fp8_linear(x8.t, xs.t, w8.t, wsc.t, out8.t, workspace=wsp.t, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    for g, what in ((x8, "x8"), (xs, "x scale"), (w8, "w8"), (wsc, "w scale"), (out8, "fp8 out"),
                    (wsp, "fp8 workspace")):
        g.check(what)
