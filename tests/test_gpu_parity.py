"""GPU parity: every libgdn entry point, called through the C ABI, against the fp64 oracle
on the same seeded inputs (small shapes spanning several tiles and ragged tails, the
workload sizes, and the edge cases)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gated_deltanet_linear_conv1d_gb300 import synth  # noqa: E402
from oracle import oracle  # noqa: E402
from tests import gdnutil as U  # noqa: E402


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_linear_conv1d_gb300 import build
    build.build()
    from gated_deltanet_linear_conv1d_gb300 import binding
    return binding


def _dev_err():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ---------------------------------------------------------------- standalone pieces

@pytest.mark.parametrize("lengths", [[64], [1, 2, 3, 70, 0, 129], [1] * 40, [513, 2, 64, 65, 190, 4]])
def test_conv_update_matches_oracle(b, lengths):
    dims = synth.FULL_HEADS
    w = synth.prefill_workload(dims, lengths, seed=31)
    d = U.to_device(w)
    T = int(sum(lengths))
    y = torch.zeros((T, dims.channels), dtype=torch.bfloat16, device="cuda")
    D = b.make_dims(dims, w["num_slots"])
    err = _dev_err()
    b.gdn_conv_update(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["query_start_loc"], d["slot_idx"], y,
                      has_init=d["has_init"], dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    y_ref, hist_ref = oracle.conv_update(dims, w["qkv0"], w["conv_w"], w["conv_hist"], w["query_start_loc"],
                                         w["slot_idx"], w["has_init"])
    U.check_out(U.host_f64_from_bf16(y), y_ref, "y")
    np.testing.assert_array_equal(U.host_bits(d["conv_hist"]), hist_ref)  # bit-exact, untouched slots too


@pytest.mark.parametrize("T,H,D", [(37, 48, 128), (5, 3, 64), (9, 2, 256), (3, 1, 1000), (2, 2, 1024)])
def test_gated_rmsnorm_matches_oracle(b, T, H, D):
    """The head dim of the layer (four rows per warp) and other row sizes (lanes past D idle, or up
    to eight groups per lane); row counts that leave the last warp's rows partly empty."""
    rng = np.random.default_rng(32 + D)
    o = synth.bf16_bits(rng.standard_normal((T, H, D)).astype(np.float32) * 0.3)
    z = synth.bf16_bits(rng.standard_normal((T, H, D)).astype(np.float32))
    gamma = rng.uniform(0.5, 1.5, D).astype(np.float32)
    out = torch.empty((T, H * D), dtype=torch.bfloat16, device="cuda")
    b.gdn_gated_rmsnorm(U.dev_bf16(o), U.dev_bf16(z), U.dev(gamma), 1e-6, out)
    ref = oracle.gated_rmsnorm(o, z, gamma, 1e-6)
    U.check_out(U.host_f64_from_bf16(out), ref, "ogate")


# ---------------------------------------------------------------- decode

def _run_decode(b, w, want_o=True):
    dims = w["dims"]
    N = len(w["slot_idx"])
    d = U.to_device(w)
    D = b.make_dims(dims, w["num_slots"])
    o = torch.zeros((N, dims.num_v_heads, dims.head_v_dim), dtype=torch.bfloat16, device="cuda") if want_o else None
    og = torch.zeros((N, dims.num_v_heads * dims.head_v_dim), dtype=torch.bfloat16, device="cuda")
    err = _dev_err()
    b.gdn_decode_step(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["slot_idx"], d["alpha"], d["beta"],
                      d["z"], d["gamma"], w["eps"], o=o, ogate=og, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    return d, o, og


def _check_decode(w, d, o, og, requests=None, pool_exact=True):
    N = len(w["slot_idx"])
    requests = np.arange(N) if requests is None else np.asarray(requests)
    r, toks = U.oracle_compact(w, requests)
    if o is not None:
        U.check_out(U.host_f64_from_bf16(o)[toks], r["o"], "o")
    U.check_out(U.host_f64_from_bf16(og)[toks], r["ogate"], "ogate")
    slots = w["slot_idx"][requests]
    st = d["state"][torch.from_numpy(slots.astype(np.int64)).cuda()].cpu().numpy()
    U.check_state(st, r["state"], U.STATE_REL_L2_DECODE, "state")
    hist = U.host_bits(d["conv_hist"][torch.from_numpy(slots.astype(np.int64)).cuda()])
    np.testing.assert_array_equal(hist, r["conv_hist"])
    if pool_exact:  # slots no request names are left bit-for-bit as they were
        untouched = np.setdiff1d(np.arange(w["num_slots"]), w["slot_idx"])
        idx = torch.from_numpy(untouched.astype(np.int64)).cuda()
        np.testing.assert_array_equal(d["state"][idx].cpu().numpy(), w["state"][untouched])
        np.testing.assert_array_equal(U.host_bits(d["conv_hist"][idx]), w["conv_hist"][untouched])


@pytest.mark.parametrize("geom", [synth.FULL_HEADS, synth.RANK_HEADS], ids=["16x48", "4x12"])
@pytest.mark.parametrize("R", [1, 8, 64])
def test_decode_small_batches(b, geom, R):
    w = synth.decode_workload(geom, R, seed=40 + R)
    d, o, og = _run_decode(b, w)
    _check_decode(w, d, o, og)


def test_decode_headline_256_of_512(b):
    """The headline decode step: 256 requests over a 512-slot pool, random permutation."""
    w = synth.decode_workload(synth.FULL_HEADS, 256, 512, seed=1)
    d, o, og = _run_decode(b, w)
    _check_decode(w, d, o, og)


@pytest.mark.parametrize("geom", [synth.FULL_HEADS, synth.RANK_HEADS], ids=["16x48", "4x12"])
def test_decode_1024(b, geom):
    w = synth.decode_workload(geom, 1024, seed=44)
    d, o, og = _run_decode(b, w, want_o=False)
    rng = np.random.default_rng(0)
    _check_decode(w, d, None, og, requests=np.sort(rng.choice(1024, 96, replace=False)), pool_exact=False)


def test_decode_padding_and_bad_slot(b):
    dims = synth.RANK_HEADS
    w = synth.decode_workload(dims, 6, 12, seed=45)
    w["slot_idx"][1] = -1  # padding: skipped
    bad = w["slot_idx"].copy()
    d = U.to_device(w)
    D = b.make_dims(dims, w["num_slots"])
    og = torch.zeros((6, dims.num_v_heads * 128), dtype=torch.bfloat16, device="cuda")
    err = _dev_err()
    b.gdn_decode_step(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["slot_idx"], d["alpha"],
                      d["beta"], d["z"], d["gamma"], w["eps"], ogate=og, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    assert not og[1].any()
    live = np.array([0, 2, 3, 4, 5])
    r, _ = U.oracle_compact(w, live)
    U.check_out(U.host_f64_from_bf16(og)[live], r["ogate"], "ogate")
    # an out-of-range slot is flagged on the device and writes nothing
    bad[3] = 12
    d2 = U.to_device(dict(w, slot_idx=bad))
    og2 = torch.zeros_like(og)
    b.gdn_decode_step(D, d2["qkv0"], d2["conv_w"], d2["conv_hist"], d2["state"], d2["slot_idx"], d2["alpha"],
                      d2["beta"], d2["z"], d2["gamma"], w["eps"], ogate=og2, dev_err=err)
    assert b.gdn_read_device_error(err) == b.GDN_DEVERR_SLOT
    assert not og2[3].any()
    torch.cuda.synchronize()


def test_decode_on_two_streams_at_once(b):
    """Two decode steps on different streams run at the same time (separate pools and inputs); each
    stream's launches claim units from their own counter, so both match the oracle."""
    ws_ = [synth.decode_workload(synth.FULL_HEADS, 64, 128, seed=47 + k) for k in range(2)]
    ds = [U.to_device(w) for w in ws_]
    ogs = [torch.zeros((64, 6144), dtype=torch.bfloat16, device="cuda") for _ in ws_]
    err = _dev_err()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    for rep in range(3):  # repeated so the two streams' launches overlap; each repeat redoes the step
        if rep:
            ds = [U.to_device(w) for w in ws_]
            torch.cuda.synchronize()
        for w, d, og, st in zip(ws_, ds, ogs, streams):
            D = b.make_dims(w["dims"], w["num_slots"])
            b.gdn_decode_step(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["slot_idx"], d["alpha"],
                              d["beta"], d["z"], d["gamma"], w["eps"], ogate=og, dev_err=err, stream=st)
        torch.cuda.synchronize()
    assert b.gdn_read_device_error(err) == 0
    for w, d, og in zip(ws_, ds, ogs):
        _check_decode(w, d, None, og)


def test_decode_is_deterministic(b):
    w = synth.decode_workload(synth.FULL_HEADS, 16, seed=46)
    d1, _, og1 = _run_decode(b, w, want_o=False)
    d2, _, og2 = _run_decode(b, w, want_o=False)
    assert torch.equal(og1, og2) and torch.equal(d1["state"], d2["state"])


# ---------------------------------------------------------------- speculative verify + commit

@pytest.mark.parametrize("N", [5, 256])
def test_spec_verify_and_commit(b, N):
    """Speculative verify at the full head layout: 5 requests (all checked) and the mixed
    workload's 256 requests x 4 positions (32 sampled requests checked against the oracle,
    every request's commit checked bit for bit)."""
    dims = synth.FULL_HEADS
    w = synth.spec_workload(dims, N, num_pos=4, seed=47 + N)
    P = w["num_pos"]
    d = U.to_device(w)
    D = b.make_dims(dims, w["num_slots"])
    o = torch.zeros((N * P, dims.num_v_heads, 128), dtype=torch.bfloat16, device="cuda")
    og = torch.zeros((N * P, dims.num_v_heads * 128), dtype=torch.bfloat16, device="cuda")
    err = _dev_err()
    b.gdn_spec_verify(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["slot_idx"], d["spec_slot_idx"],
                      d["alpha"], d["beta"], d["z"], d["gamma"], w["eps"], o=o, ogate=og, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    sample = np.arange(N) if N <= 8 else np.sort(np.random.default_rng(1).choice(N, 32, replace=False))
    ref, toks = U.oracle_spec_compact(w, sample)
    U.check_out(U.host_f64_from_bf16(o)[toks], ref["o"], "o")
    U.check_out(U.host_f64_from_bf16(og)[toks], ref["ogate"], "ogate")
    ck = w["spec_slot_idx"][sample].reshape(-1)
    idx = torch.from_numpy(ck.astype(np.int64)).cuda()
    U.check_state(d["state"][idx].cpu().numpy(), ref["state"], U.STATE_REL_L2_DECODE, "checkpoints")
    np.testing.assert_array_equal(U.host_bits(d["conv_hist"][idx]), ref["conv_hist"])
    live = torch.from_numpy(w["slot_idx"].astype(np.int64)).cuda()
    for n in range(0, N, 64):  # live slots untouched (in slices, to bound host memory)
        sl = live[n:n + 64]
        np.testing.assert_array_equal(d["state"][sl].cpu().numpy(), w["state"][w["slot_idx"][n:n + 64]])

    # commit by copy: the live slot becomes the accepted checkpoint, bit for bit
    src = torch.from_numpy(w["spec_slot_idx"][np.arange(N), w["accepted"]].astype(np.int64)).cuda()
    b.gdn_spec_commit(D, d["accepted"], d["spec_slot_idx"], d["slot_idx"], d["state"], d["conv_hist"],
                      mode=b.GDN_COMMIT_COPY, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    assert torch.equal(d["state"][live], d["state"][src])
    assert torch.equal(d["conv_hist"][live], d["conv_hist"][src])
    # commit by repoint: only the slot index changes
    slots = d["slot_idx"].clone()
    b.gdn_spec_commit(D, d["accepted"], d["spec_slot_idx"], slots, mode=b.GDN_COMMIT_REPOINT, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    assert torch.equal(slots.long(), src)


@pytest.mark.parametrize("two_streams", [False, True], ids=["one_stream", "two_streams"])
def test_mixed_verify_commit_and_prefill_step(b, two_streams):
    """The speculative-verify step with a prefill in the same step: 256 requests x 4 positions
    verified and committed (copy) at the full head layout, and 8 prefill requests of 2048 tokens
    (half from zero) over their own pool, on one stream back to back or with the prefill on a
    second stream. Verify outputs and checkpoints of 32 sampled requests against the oracle;
    every committed slot bit for bit; every prefill output, state and history against the oracle."""
    dims = synth.FULL_HEADS
    N = 256
    wv = synth.spec_workload(dims, N, num_pos=4, seed=70)
    P = wv["num_pos"]
    wp = synth.prefill_workload(dims, [2048] * 8, seed=71)
    dv, dp = U.to_device(wv), U.to_device(wp)
    Dv, Dp = b.make_dims(dims, wv["num_slots"]), b.make_dims(dims, wp["num_slots"])
    Tp = 8 * 2048
    og_v = torch.zeros((N * P, dims.num_v_heads * 128), dtype=torch.bfloat16, device="cuda")
    og_p = torch.zeros((Tp, dims.num_v_heads * 128), dtype=torch.bfloat16, device="cuda")
    err_v, err_p = _dev_err(), _dev_err()
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream() if two_streams else main
    side.wait_stream(main)
    torch.cuda.synchronize()
    b.gdn_spec_verify(Dv, dv["qkv0"], dv["conv_w"], dv["conv_hist"], dv["state"], dv["slot_idx"],
                      dv["spec_slot_idx"], dv["alpha"], dv["beta"], dv["z"], dv["gamma"], wv["eps"], ogate=og_v,
                      dev_err=err_v, stream=main)
    b.gdn_chunk_prefill(Dp, dp["qkv0"], dp["conv_w"], dp["conv_hist"], dp["state"], dp["query_start_loc"],
                        dp["slot_idx"], dp["alpha"], dp["beta"], dp["z"], dp["gamma"], wp["eps"], ogate=og_p,
                        has_init=dp["has_init"], dev_err=err_p, stream=side)
    b.gdn_spec_commit(Dv, dv["accepted"], dv["spec_slot_idx"], dv["slot_idx"], dv["state"], dv["conv_hist"],
                      mode=b.GDN_COMMIT_COPY, dev_err=err_v, stream=main)
    torch.cuda.synchronize()
    assert b.gdn_read_device_error(err_v) == 0 and b.gdn_read_device_error(err_p) == 0
    # verify: sampled requests' outputs and checkpoints
    sample = np.sort(np.random.default_rng(2).choice(N, 32, replace=False))
    ref, toks = U.oracle_spec_compact(wv, sample)
    U.check_out(U.host_f64_from_bf16(og_v)[toks], ref["ogate"], "verify ogate")
    ck = torch.from_numpy(wv["spec_slot_idx"][sample].reshape(-1).astype(np.int64)).cuda()
    U.check_state(dv["state"][ck].cpu().numpy(), ref["state"], U.STATE_REL_L2_DECODE, "verify checkpoints")
    np.testing.assert_array_equal(U.host_bits(dv["conv_hist"][ck]), ref["conv_hist"])
    # commit: every live slot equals its accepted checkpoint, and for the sample the oracle's
    live = torch.from_numpy(wv["slot_idx"].astype(np.int64)).cuda()
    src = torch.from_numpy(wv["spec_slot_idx"][np.arange(N), wv["accepted"]].astype(np.int64)).cuda()
    assert torch.equal(dv["state"][live], dv["state"][src])
    assert torch.equal(dv["conv_hist"][live], dv["conv_hist"][src])
    acc = wv["accepted"][sample]
    sel = np.arange(len(sample)) * P + acc
    live_s = torch.from_numpy(wv["slot_idx"][sample].astype(np.int64)).cuda()
    U.check_state(dv["state"][live_s].cpu().numpy(), ref["state"][sel], U.STATE_REL_L2_DECODE, "committed state")
    np.testing.assert_array_equal(U.host_bits(dv["conv_hist"][live_s]), ref["conv_hist"][sel])
    # prefill: all 8 requests
    _check_prefill(wp, dp, None, og_p, np.arange(8))


def test_spec_commit_rejects_bad_accepted_length(b):
    dims = synth.RANK_HEADS
    w = synth.spec_workload(dims, 4, num_pos=4, seed=49)
    w["accepted"][2] = 4
    d = U.to_device(w)
    D = b.make_dims(dims, w["num_slots"])
    err = _dev_err()
    slots = d["slot_idx"].clone()
    b.gdn_spec_commit(D, d["accepted"], d["spec_slot_idx"], slots, mode=b.GDN_COMMIT_REPOINT, dev_err=err)
    assert b.gdn_read_device_error(err) == b.GDN_DEVERR_ACCEPTED
    assert int(slots[2]) == int(w["slot_idx"][2])


# ---------------------------------------------------------------- prefill

def _run_prefill(b, w, want_o=True):
    dims = w["dims"]
    T = int(w["query_start_loc"][-1])
    d = U.to_device(w)
    D = b.make_dims(dims, w["num_slots"])
    o = torch.zeros((T, dims.num_v_heads, 128), dtype=torch.bfloat16, device="cuda") if want_o else None
    og = torch.zeros((T, dims.num_v_heads * 128), dtype=torch.bfloat16, device="cuda")
    err = _dev_err()
    b.gdn_chunk_prefill(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["query_start_loc"],
                        d["slot_idx"], d["alpha"], d["beta"], d["z"], d["gamma"], w["eps"], o=o, ogate=og,
                        has_init=d["has_init"], dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    return d, o, og


def _check_prefill(w, d, o, og, requests):
    r, toks = U.oracle_compact(w, requests)
    if o is not None:
        U.check_out(U.host_f64_from_bf16(o)[toks], r["o"], "o")
    U.check_out(U.host_f64_from_bf16(og)[toks], r["ogate"], "ogate")
    slots = torch.from_numpy(w["slot_idx"][requests].astype(np.int64)).cuda()
    U.check_state(d["state"][slots].cpu().numpy(), r["state"], U.STATE_REL_L2_PREFILL, "state")
    np.testing.assert_array_equal(U.host_bits(d["conv_hist"][slots]), r["conv_hist"])


def test_prefill_single_request_from_zero(b):
    """One request of 64 tokens from a zero state (the reference prefill case)."""
    w = synth.prefill_workload(synth.FULL_HEADS, [64], seed=0, zero_first_half=False)
    w["has_init"][:] = 0
    d, o, og = _run_prefill(b, w)
    _check_prefill(w, d, o, og, [0])


@pytest.mark.parametrize("geom", [synth.FULL_HEADS, synth.RANK_HEADS], ids=["16x48", "4x12"])
def test_prefill_ragged_batch(b, geom):
    """Lengths across chunk edges (1, 2, 63, 64, 65, 130), an empty request, half from zero."""
    lengths = [1, 65, 0, 130, 2, 63, 64, 17]
    w = synth.prefill_workload(geom, lengths, seed=50)
    d, o, og = _run_prefill(b, w)
    _check_prefill(w, d, o, og, np.arange(len(lengths)))


def test_prefill_many_short_requests(b):
    """400 requests of 1-5 tokens at 4/12 heads (4,800 CTAs, 1,600 key-head groups): every key head's
    new q/k history is written by the last of its group's CTAs to start, whatever order they run in;
    the whole history pool is checked bit for bit, state and outputs on a sample of requests."""
    rng = np.random.default_rng(52)
    lengths = rng.integers(1, 6, size=400).tolist()
    w = synth.prefill_workload(synth.RANK_HEADS, lengths, seed=52)
    d, _, og = _run_prefill(b, w, want_o=False)
    sample = np.sort(rng.choice(len(lengths), 24, replace=False))
    _check_prefill(w, d, None, og, sample)
    r, _ = U.oracle_compact(w, np.arange(len(lengths)))
    slots = torch.from_numpy(w["slot_idx"].astype(np.int64)).cuda()
    np.testing.assert_array_equal(U.host_bits(d["conv_hist"][slots]), r["conv_hist"])


def test_prefill_varlen_64_requests(b):
    """64 requests, log-uniform lengths in [16, 8192] (71,068 tokens at this seed), half from
    zero: every request's outputs, final state and conv history against the oracle (checked in
    groups of requests to bound host memory)."""
    lengths = synth.loguniform_lengths(np.random.default_rng(3), 64, 16, 8192)
    w = synth.prefill_workload(synth.FULL_HEADS, lengths, seed=3)
    d, o, og = _run_prefill(b, w, want_o=False)
    for g in range(0, 64, 16):
        _check_prefill(w, d, None, og, np.arange(g, g + 16))


def test_prefill_then_decode_continues_the_request(b):
    """Prefill of T1 tokens, then decode steps, equals one oracle pass over all tokens."""
    geom = synth.RANK_HEADS
    T1, T2 = 70, 3
    w = synth.prefill_workload(geom, [T1 + T2], seed=51, zero_first_half=False)
    full, _ = U.oracle_compact(w, [0])
    d = U.to_device(w)
    D = b.make_dims(geom, w["num_slots"])
    og = torch.zeros((T1 + T2, geom.num_v_heads * 128), dtype=torch.bfloat16, device="cuda")
    err = _dev_err()
    qsl = torch.tensor([0, T1], dtype=torch.int32, device="cuda")
    b.gdn_chunk_prefill(D, d["qkv0"][:T1].contiguous(), d["conv_w"], d["conv_hist"], d["state"], qsl,
                        d["slot_idx"], d["alpha"][:T1].contiguous(), d["beta"][:T1].contiguous(),
                        d["z"][:T1].contiguous(), d["gamma"], w["eps"], ogate=og[:T1], dev_err=err)
    for t in range(T1, T1 + T2):
        sl = slice(t, t + 1)
        b.gdn_decode_step(D, d["qkv0"][sl].contiguous(), d["conv_w"], d["conv_hist"], d["state"], d["slot_idx"],
                          d["alpha"][sl].contiguous(), d["beta"][sl].contiguous(), d["z"][sl].contiguous(),
                          d["gamma"], w["eps"], ogate=og[sl], dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    U.check_out(U.host_f64_from_bf16(og), full["ogate"], "ogate")
    slot = int(w["slot_idx"][0])
    U.check_state(d["state"][slot].cpu().numpy(), full["state"][0], U.STATE_REL_L2_PREFILL, "state")
    np.testing.assert_array_equal(U.host_bits(d["conv_hist"][slot]), full["conv_hist"][0])


def test_prefill_with_no_tokens_touches_nothing(b):
    """N requests, all empty (T = 0): the call succeeds and every slot is left as it was."""
    dims = synth.RANK_HEADS
    w = synth.prefill_workload(dims, [0, 0, 0], seed=57)
    d = U.to_device(w)
    D = b.make_dims(dims, w["num_slots"])
    err = _dev_err()
    og = torch.zeros((0, dims.num_v_heads * 128), dtype=torch.bfloat16, device="cuda")
    b.gdn_chunk_prefill(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["query_start_loc"], d["slot_idx"],
                        d["alpha"], d["beta"], d["z"], d["gamma"], w["eps"], ogate=og, has_init=d["has_init"],
                        dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    np.testing.assert_array_equal(d["state"].cpu().numpy(), w["state"])
    np.testing.assert_array_equal(U.host_bits(d["conv_hist"]), w["conv_hist"])


def test_prefill_bad_offsets_are_flagged(b):
    geom = synth.RANK_HEADS
    w = synth.prefill_workload(geom, [5, 7], seed=52)
    w["query_start_loc"] = np.array([0, 5, 13], np.int32)  # the last request ends past T = 12
    d = U.to_device(w)
    D = b.make_dims(geom, w["num_slots"])
    og = torch.zeros((12, geom.num_v_heads * 128), dtype=torch.bfloat16, device="cuda")
    err = _dev_err()
    b.gdn_chunk_prefill(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["query_start_loc"],
                        d["slot_idx"], d["alpha"], d["beta"], d["z"], d["gamma"], w["eps"], ogate=og, dev_err=err)
    assert b.gdn_read_device_error(err) & b.GDN_DEVERR_OFFSETS
    assert og[:5].any() and not og[5:].any()  # the valid request ran, the flagged one wrote nothing
    s1 = int(w["slot_idx"][1])
    np.testing.assert_array_equal(d["state"][s1].cpu().numpy(), w["state"][s1])


# ---------------------------------------------------------------- geometry and position variants

GEOMS = [synth.Dims(4, 4, 128, 128, 4), synth.Dims(2, 16, 128, 128, 4)]  # G = 1 and G = 8


@pytest.mark.parametrize("geom", GEOMS, ids=["G1", "G8"])
def test_decode_group_sizes(b, geom):
    w = synth.decode_workload(geom, 9, 20, seed=60)
    d, o, og = _run_decode(b, w)
    _check_decode(w, d, o, og)


@pytest.mark.parametrize("geom", GEOMS, ids=["G1", "G8"])
def test_prefill_group_sizes(b, geom):
    w = synth.prefill_workload(geom, [3, 70, 129], seed=61)
    d, o, og = _run_prefill(b, w)
    _check_prefill(w, d, o, og, np.arange(3))


@pytest.mark.parametrize("P", [1, 2, 8])
def test_spec_verify_positions(b, P):
    dims = synth.RANK_HEADS
    N = 6
    w = synth.spec_workload(dims, N, num_pos=P, seed=62 + P)
    d = U.to_device(w)
    D = b.make_dims(dims, w["num_slots"])
    og = torch.zeros((N * P, dims.num_v_heads * 128), dtype=torch.bfloat16, device="cuda")
    err = _dev_err()
    b.gdn_spec_verify(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["slot_idx"], d["spec_slot_idx"],
                      d["alpha"], d["beta"], d["z"], d["gamma"], w["eps"], ogate=og, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    ref = oracle.spec_verify(dims, w["qkv0"], w["conv_w"], w["conv_hist"], w["state"], w["slot_idx"],
                             w["spec_slot_idx"], w["alpha"], w["beta"], w["z"], w["gamma"], w["eps"])
    U.check_out(U.host_f64_from_bf16(og), ref["ogate"], "ogate")
    ck = w["spec_slot_idx"].reshape(-1)
    idx = torch.from_numpy(ck.astype(np.int64)).cuda()
    U.check_state(d["state"][idx].cpu().numpy(), ref["state"][ck], U.STATE_REL_L2_DECODE, "checkpoints")
    np.testing.assert_array_equal(U.host_bits(d["conv_hist"][idx]), ref["conv_hist"][ck])


# ---------------------------------------------------------------- align-mode snapshots (prefix caching)

def test_prefill_align_snapshots_equal_prefix_runs(b):
    """Snapshots after every absolute multiple of the block (128) equal the oracle run on that prefix;
    chunks start on absolute multiples of 64 (first chunks of 28, 36 and 1 tokens here); skipped and
    unused snapshot slots stay untouched; the live results equal a plain prefill's."""
    dims = synth.RANK_HEADS
    lengths = [300, 70, 129, 64, 5]
    prefix = np.array([0, 64, 100, 256, 127], np.int32)
    B = 128
    w = synth.prefill_workload(dims, lengths, seed=55)
    N = len(lengths)
    free = np.setdiff1d(np.arange(w["num_slots"]), w["slot_idx"]).astype(np.int32)
    snap = np.full((N, 2), -1, np.int32)
    snap[0] = free[0:2]
    snap[1, 0] = free[2]
    snap[4, 0] = free[3]  # request 2 crosses 128 too but its snapshot is skipped (-1)
    d = U.to_device(w)
    D = b.make_dims(dims, w["num_slots"])
    T = int(sum(lengths))
    og = torch.zeros((T, dims.num_v_heads * 128), dtype=torch.bfloat16, device="cuda")
    err = _dev_err()
    b.gdn_chunk_prefill_align(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["query_start_loc"],
                              d["slot_idx"], d["alpha"], d["beta"], d["z"], d["gamma"], w["eps"], B,
                              snap_slot=U.dev(snap), prefix_len=U.dev(prefix), ogate=og, has_init=d["has_init"],
                              dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    _check_prefill(w, d, None, og, np.arange(N))
    qsl = w["query_start_loc"]
    for n in range(N):
        for j in range(2):
            if snap[n, j] < 0:
                continue
            rel = (prefix[n] // B + 1 + j) * B - prefix[n]
            toks = np.arange(qsl[n], qsl[n] + rel)
            s = int(w["slot_idx"][n])
            r = oracle.forward(dims, w["qkv0"][toks], w["conv_w"], np.ascontiguousarray(w["conv_hist"][[s]]),
                               np.ascontiguousarray(w["state"][[s]]), np.array([0, rel], np.int32),
                               np.zeros(1, np.int32), w["alpha"][toks], w["beta"][toks], w["z"][toks], w["gamma"],
                               w["eps"], has_init=w["has_init"][[n]], inplace=True)
            k = int(snap[n, j])
            U.check_state(d["state"][k].cpu().numpy(), r["state"][0], U.STATE_REL_L2_PREFILL, f"snapshot {n}.{j}")
            np.testing.assert_array_equal(U.host_bits(d["conv_hist"][k]), r["conv_hist"][0])
    untouched = np.setdiff1d(free, snap[snap >= 0])
    idx = torch.from_numpy(untouched.astype(np.int64)).cuda()
    np.testing.assert_array_equal(d["state"][idx].cpu().numpy(), w["state"][untouched])
    np.testing.assert_array_equal(U.host_bits(d["conv_hist"][idx]), w["conv_hist"][untouched])
