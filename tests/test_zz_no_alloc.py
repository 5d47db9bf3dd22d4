"""gdn_chunk_prefill_noalloc (fixed device scratch, no workspace argument) against
gdn_chunk_prefill on two calls in a row: identical Ogate bits after each call and
identical final state and conv history. This file is collected last; the test
also passes on its own in a fresh process."""
import numpy as np
import pytest
import torch

from gated_deltanet_linear_conv1d_gb300 import synth
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


def _halves(w, lengths, cut):
    """Split every request at `cut` tokens: two consecutive varlen calls."""
    qsl = w["query_start_loc"]
    first, second = [], []
    for n, L in enumerate(lengths):
        a = int(qsl[n])
        c = min(cut, L)
        first.append(np.arange(a, a + c))
        second.append(np.arange(a + c, a + L))
    return first, second


def _call(b, fn, D, d, rows, w, lengths_part, has_init, use_ws):
    idx = torch.from_numpy(np.concatenate(rows).astype(np.int64)).cuda()
    qsl = torch.from_numpy(synth.pack_offsets(np.array(lengths_part, np.int32))).cuda()
    T = int(sum(lengths_part))
    og = torch.zeros((T, D.num_v_heads * D.head_v_dim), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    args = (D, d["qkv0"][idx].contiguous(), d["conv_w"], d["conv_hist"], d["state"], qsl, d["slot_idx"],
            d["alpha"][idx].contiguous(), d["beta"][idx].contiguous(), d["z"][idx].contiguous(), d["gamma"],
            w["eps"])
    if use_ws:
        ws = torch.empty(b.gdn_prefill_workspace_bytes(D, len(lengths_part), T), dtype=torch.uint8, device="cuda")
        fn(*args, ogate=og, has_init=has_init, workspace=ws, dev_err=err)
    else:
        fn(*args, ogate=og, has_init=has_init, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    return U.host_bits(og)


def test_noalloc_prefill_matches_the_workspace_entry_point(b):
    lengths = [70, 1, 200, 64, 0, 129]
    w = synth.prefill_workload(synth.RANK_HEADS, lengths, seed=61)
    D = b.make_dims(synth.RANK_HEADS, w["num_slots"])
    first, second = _halves(w, lengths, 65)
    l1 = [len(r) for r in first]
    l2 = [len(r) for r in second]
    da, dn = U.to_device(w), U.to_device(w)
    outs = {}
    for name, d, fn, ws in (("ws", da, b.gdn_chunk_prefill, True), ("noalloc", dn, b.gdn_chunk_prefill_noalloc, False)):
        o1 = _call(b, fn, D, d, first, w, l1, d["has_init"], ws)  # half of the requests from zero
        o2 = _call(b, fn, D, d, second, w, l2, None, ws)  # every request continues from its slot
        torch.cuda.synchronize()
        outs[name] = (o1, o2, d["state"].cpu().numpy(), U.host_bits(d["conv_hist"]))
    for x, y in zip(outs["ws"], outs["noalloc"]):
        np.testing.assert_array_equal(x, y)


def test_noalloc_prefill_rejects_too_many_requests(b):
    """Beyond the fixed arrays: more than 65,535 requests, or more than 2^20 (request, key head)
    tickets with an accepted request count (40,000 requests x 32 key heads)."""
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = dummy.data_ptr()
    for geom, n in ((synth.RANK_HEADS, 65536), (synth.RANK_HEADS, 65537), (synth.Dims(32, 32, 128, 128, 4), 40000)):
        D = b.make_dims(geom, 4)
        st = b._lib.gdn_chunk_prefill_noalloc(b.ctypes.byref(D), None, p, p, p, p, p, None, None, None, None, None,
                                              1e-6, None, p, n, 0, None, None)
        assert st == b.GDN_ERR_INVALID_ARG, (geom, n)


def test_noalloc_prefill_at_its_request_limit(b):
    """65,535 one-token requests from zero (one key head and one value head, so the pools stay
    small): the largest count the fixed schedule takes runs, and matches gdn_chunk_prefill."""
    geom = synth.Dims(1, 1, 128, 128, 4)
    N = 65535
    D = b.make_dims(geom, N)
    rng = np.random.default_rng(62)
    T = N
    qkv0 = U.dev_bf16(synth.bf16_bits(rng.standard_normal((T, geom.channels)).astype(np.float32)))
    conv_w = U.dev((rng.standard_normal((geom.channels, 4)) * 0.25).astype(np.float32))
    alpha = U.dev(np.exp(-rng.uniform(0.001, 0.1, (T, 1))).astype(np.float32))
    beta = U.dev(rng.uniform(0, 1, (T, 1)).astype(np.float32))
    z = U.dev_bf16(synth.bf16_bits(rng.standard_normal((T, 1, 128)).astype(np.float32)))
    gamma = torch.ones(128, dtype=torch.float32, device="cuda")
    qsl = torch.arange(N + 1, dtype=torch.int32, device="cuda")
    slots = torch.from_numpy(rng.permutation(N).astype(np.int32)).cuda()
    has_init = torch.zeros(N, dtype=torch.uint8, device="cuda")
    outs = []
    for fn, ws in ((b.gdn_chunk_prefill, True), (b.gdn_chunk_prefill_noalloc, False)):
        state = torch.zeros((N, 1, 128, 128), dtype=torch.float32, device="cuda")
        hist = torch.zeros((N, geom.channels, 3), dtype=torch.bfloat16, device="cuda")
        og = torch.zeros((T, 128), dtype=torch.bfloat16, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        fn(D, qkv0, conv_w, hist, state, qsl, slots, alpha, beta, z, gamma, 1e-6, ogate=og, has_init=has_init,
           dev_err=err)
        assert b.gdn_read_device_error(err) == 0
        outs.append((og, state, hist))
    assert outs[0][0].any()
    for x, y in zip(*outs):
        assert torch.equal(x, y)
