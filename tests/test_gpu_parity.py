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
    dims = synth.FULL_HEADS if N == 5 else synth.RANK_HEADS
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
    sample = np.arange(N) if N <= 8 else np.sort(np.random.default_rng(1).choice(N, 24, replace=False))
    ref = oracle.spec_verify(dims, w["qkv0"], w["conv_w"], w["conv_hist"], w["state"], w["slot_idx"],
                             w["spec_slot_idx"], w["alpha"], w["beta"], w["z"], w["gamma"], w["eps"])
    toks = (sample[:, None] * P + np.arange(P)[None, :]).reshape(-1)
    U.check_out(U.host_f64_from_bf16(o)[toks], ref["o"][toks], "o")
    U.check_out(U.host_f64_from_bf16(og)[toks], ref["ogate"][toks], "ogate")
    ck = w["spec_slot_idx"][sample].reshape(-1)
    idx = torch.from_numpy(ck.astype(np.int64)).cuda()
    U.check_state(d["state"][idx].cpu().numpy(), ref["state"][ck], U.STATE_REL_L2_DECODE, "checkpoints")
    np.testing.assert_array_equal(U.host_bits(d["conv_hist"][idx]), ref["conv_hist"][ck])
    live = torch.from_numpy(w["slot_idx"].astype(np.int64)).cuda()
    np.testing.assert_array_equal(d["state"][live].cpu().numpy(), w["state"][w["slot_idx"]])  # live untouched

    # commit by copy: the live slot becomes the accepted checkpoint, bit for bit
    state_before = d["state"].clone()
    hist_before = d["conv_hist"].clone()
    b.gdn_spec_commit(D, d["accepted"], d["spec_slot_idx"], d["slot_idx"], d["state"], d["conv_hist"],
                      mode=b.GDN_COMMIT_COPY, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    src = torch.from_numpy(w["spec_slot_idx"][np.arange(N), w["accepted"]].astype(np.int64)).cuda()
    assert torch.equal(d["state"][live], state_before[src])
    assert torch.equal(d["conv_hist"][live], hist_before[src])
    # commit by repoint: only the slot index changes
    slots = d["slot_idx"].clone()
    b.gdn_spec_commit(D, d["accepted"], d["spec_slot_idx"], slots, mode=b.GDN_COMMIT_REPOINT, dev_err=err)
    assert b.gdn_read_device_error(err) == 0
    assert torch.equal(slots.long(), src)


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


def test_prefill_varlen_64_requests_sampled(b):
    """64 requests, log-uniform lengths in [16, 8192], half from zero; sampled requests checked."""
    lengths = synth.loguniform_lengths(np.random.default_rng(3), 64, 16, 8192)
    w = synth.prefill_workload(synth.FULL_HEADS, lengths, seed=3)
    d, o, og = _run_prefill(b, w, want_o=False)
    order = np.argsort(lengths)
    sample = np.unique(np.concatenate([order[:2], order[-1:], order[30:32]]))
    _check_prefill(w, d, None, og, sample)


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
