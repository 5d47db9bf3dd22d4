"""Pins of the fp64 oracle to facts other than itself (CPU only).

Each check is a closed form, an invariant, a special case or a fixture taken
from the "Qwen3.8-27B: from model structure to vLLM inference data flow" page
(section 01 operator table of a GDN layer; section 03 GDN state lab; section 06
TP4 head split; section 08: decay first, then predict from the decayed state),
chosen so that a plausible slip in the oracle (a dropped term, a wrong sign,
a swapped index or operand, the wrong tap or history order, the wrong
key-head grouping) fails at least one of them.
"""
import json
import os

import numpy as np
import pytest

from gated_deltanet_linear_conv1d_gb300 import synth
from oracle import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
# Tiny geometry with dk != dv so that a transposed state fails shape-sensitive checks.
TINY = synth.Dims(num_k_heads=2, num_v_heads=6, head_k_dim=8, head_v_dim=4, conv_kernel=4)


def unit_rows(rng, T, d):
    x = rng.standard_normal((T, d))
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def silu(x):
    return x / (1.0 + np.exp(-x))


# ---------------------------------------------------------------- the recurrence core

def test_beta_zero_is_pure_decay():
    """beta = 0: S_t = (prod alpha) S0 and o_t = (prod_{i<=t} alpha_i) S0 q_t / sqrt(dk)."""
    rng = np.random.default_rng(10)
    T, dk, dv = 7, 8, 5
    q, k = unit_rows(rng, T, dk), unit_rows(rng, T, dk)
    v = rng.standard_normal((T, dv))
    alpha = rng.uniform(0.5, 1.0, T)
    S0 = rng.standard_normal((dv, dk))
    o, S = oracle.delta_rule_seq(q, k, v, alpha, np.zeros(T), S0)
    decay = np.cumprod(alpha)
    np.testing.assert_allclose(S, decay[-1] * S0, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(o, decay[:, None] * (q @ S0.T) / np.sqrt(dk), rtol=1e-12, atol=1e-14)


def test_exact_retrieval_orthonormal_keys():
    """alpha = beta = 1 with orthonormal keys: S k_j = v_j for every written pair, any S0."""
    rng = np.random.default_rng(11)
    dk, dv = 8, 6
    keys = np.linalg.qr(rng.standard_normal((dk, dk)))[0].T  # rows orthonormal
    vals = rng.standard_normal((dk, dv))
    S0 = rng.standard_normal((dv, dk))
    _, S = oracle.delta_rule_seq(keys, keys, vals, np.ones(dk), np.ones(dk), S0)
    np.testing.assert_allclose(keys @ S.T, vals, rtol=1e-12, atol=1e-12)


def test_beta_one_writes_the_target_after_decay():
    """beta = 1, any alpha, unit k: the step writes v exactly, S_t k_t = v_t.

    Reading k_t back with q_t = k_t gives o_t = v_t / sqrt(dk). This holds only
    when the error is predicted from the decayed state (decay first), with the
    sign e = v - Sbar k."""
    rng = np.random.default_rng(12)
    T, dk, dv = 9, 8, 5
    k = unit_rows(rng, T, dk)
    v = rng.standard_normal((T, dv))
    alpha = rng.uniform(0.2, 0.95, T)
    S0 = rng.standard_normal((dv, dk))
    o, _ = oracle.delta_rule_seq(k, k, v, alpha, np.ones(T), S0)
    np.testing.assert_allclose(o * np.sqrt(dk), v, rtol=1e-12, atol=1e-12)


def test_single_token_from_zero_state():
    """T = 1 from S0 = 0: S = beta v k^T (rows over dv) and o = beta v (k . q) / sqrt(dk)."""
    rng = np.random.default_rng(13)
    dk, dv = 8, 3
    q, k = unit_rows(rng, 1, dk), unit_rows(rng, 1, dk)
    v = rng.standard_normal((1, dv))
    alpha, beta = np.array([0.7]), np.array([0.4])
    o, S = oracle.delta_rule_seq(q, k, v, alpha, beta, np.zeros((dv, dk)))
    np.testing.assert_allclose(S, 0.4 * np.outer(v[0], k[0]), rtol=1e-14)
    np.testing.assert_allclose(o[0], 0.4 * v[0] * (k[0] @ q[0]) / np.sqrt(dk), rtol=1e-13)


def test_two_tokens_brute_force():
    """T = 2 expanded by hand from the page's update equations."""
    rng = np.random.default_rng(14)
    dk, dv = 4, 3
    q, k = unit_rows(rng, 2, dk), unit_rows(rng, 2, dk)
    v = rng.standard_normal((2, dv))
    a, b = np.array([0.9, 0.6]), np.array([0.3, 0.8])
    S0 = rng.standard_normal((dv, dk))
    o, S = oracle.delta_rule_seq(q, k, v, a, b, S0)
    S1 = a[0] * S0 + b[0] * np.outer(v[0] - a[0] * S0 @ k[0], k[0])
    S2 = a[1] * S1 + b[1] * np.outer(v[1] - a[1] * S1 @ k[1], k[1])
    np.testing.assert_allclose(S, S2, rtol=1e-13)
    np.testing.assert_allclose(o, np.stack([S1 @ q[0], S2 @ q[1]]) / np.sqrt(dk), rtol=1e-13)


def test_l2_normalization_scale_invariance():
    """normalize(c q) = normalize(q) for c > 0: scaling raw q, k leaves outputs unchanged."""
    rng = np.random.default_rng(15)
    T, dk, dv = 6, 8, 4
    q, k = rng.standard_normal((T, dk)), rng.standard_normal((T, dk))
    v = rng.standard_normal((T, dv))
    a, b = rng.uniform(0.5, 1, T), rng.uniform(0, 1, T)
    S0 = rng.standard_normal((dv, dk))
    o1, S1 = oracle.delta_rule_seq(q, k, v, a, b, S0, normalize=True)
    o2, S2 = oracle.delta_rule_seq(q * rng.uniform(0.1, 10, (T, 1)), k * rng.uniform(0.1, 10, (T, 1)),
                                   v, a, b, S0, normalize=True)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S1, S2, rtol=1e-12, atol=1e-14)
    # and the normalized core equals the un-normalized core fed unit vectors
    qn, kn = q / np.linalg.norm(q, axis=1, keepdims=True), k / np.linalg.norm(k, axis=1, keepdims=True)
    o3, _ = oracle.delta_rule_seq(qn, kn, v, a, b, S0)
    np.testing.assert_allclose(o1, o3, rtol=1e-10, atol=1e-13)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 130])
def test_chunked_form_equals_recurrent(T):
    """The chunked WY/UT form (chunk 64) equals the token-by-token form in fp64."""
    rng = np.random.default_rng(100 + T)
    dk = dv = 128
    q, k = unit_rows(rng, T, dk), unit_rows(rng, T, dk)
    v = rng.standard_normal((T, dv))
    alpha = np.exp(-rng.uniform(0.001, 0.1, T))
    beta = rng.uniform(0, 1, T)
    S0 = rng.standard_normal((dv, dk)) * 0.02
    o_r, S_r = oracle.delta_rule_seq(q, k, v, alpha, beta, S0)
    o_c, S_c = oracle.chunked_delta_rule(q, k, v, alpha, beta, S0, chunk=64)
    assert np.linalg.norm(o_c - o_r) <= 1e-12 * np.linalg.norm(o_r)
    assert np.linalg.norm(S_c - S_r) <= 1e-12 * np.linalg.norm(S_r)


# ---------------------------------------------------------------- conv, layout, gate

def _tiny_inputs(seed, T, Rs=4):
    rng = np.random.default_rng(seed)
    w = synth.layer_params(rng, TINY)
    w.update(synth.token_inputs(rng, TINY, T))
    w.update(synth.slot_pool(rng, TINY, Rs))
    return w


def _fwd(w, qsl, slots, has_init=None, **kw):
    return oracle.forward(TINY, w["qkv0"], w["conv_w"], w["conv_hist"], w["state"], qsl, slots,
                          w["alpha"], w["beta"], w["z"], w["gamma"], w["eps"], has_init=has_init, **kw)


def test_conv_impulse_response_and_history():
    """An impulse on channel c at t = 0 from a zero history gives SiLU(w[c, t]) for t < 4, then 0:
    tap i multiplies the input i steps back. The history after the call is the last 3 raw inputs."""
    dims = TINY
    CH, T = dims.channels, 6
    rng = np.random.default_rng(16)
    w = rng.standard_normal((CH, 4)).astype(np.float32)
    x = np.zeros((T, CH), np.float32)
    c = 37
    x[0, c] = 1.0
    bits = synth.bf16_bits(x)
    hist = np.zeros((2, CH, 3), np.uint16)
    y, h = oracle.conv_update(dims, bits, w, hist, np.array([0, T], np.int32), np.array([1], np.int32))
    expect = np.zeros((T, CH))
    expect[:4, c] = silu(w[c, :4].astype(np.float64))
    np.testing.assert_allclose(y, expect, rtol=1e-15, atol=0)
    np.testing.assert_array_equal(h[1], bits[-3:].T)
    np.testing.assert_array_equal(h[0], 0)


@pytest.mark.parametrize("L", [1, 2, 3, 5])
def test_conv_short_request_uses_history_oldest_first(L):
    """Entry 2 of the history is the newest input: y_0 = SiLU(w0 x0 + w1 h2 + w2 h1 + w3 h0);
    after L tokens the history is the last 3 of [h0, h1, h2, x0 .. x_{L-1}], bit for bit."""
    dims = synth.Dims(1, 1, 1, 1, 4)  # 3 channels
    rng = np.random.default_rng(17 + L)
    w = rng.standard_normal((3, 4)).astype(np.float32)
    x = synth.bf16_bits(rng.standard_normal((L, 3)).astype(np.float32))
    h0 = synth.bf16_bits(rng.standard_normal((1, 3, 3)).astype(np.float32))
    y, h1 = oracle.conv_update(dims, x, w, h0, np.array([0, L], np.int32), np.array([0], np.int32))
    xf = synth.bf16_to_f32(x).astype(np.float64)
    hf = synth.bf16_to_f32(h0[0]).astype(np.float64)  # [3 channels, 3 entries]
    seq = np.concatenate([hf.T, xf], axis=0)  # time-ascending inputs, [3 + L, 3]
    for t in range(L):
        win = seq[t : t + 4][::-1]  # win[i] = input i steps back
        np.testing.assert_allclose(y[t], silu(np.einsum("ic,ci->c", win, w.astype(np.float64))),
                                   rtol=1e-14)
    all_bits = np.concatenate([h0[0].T, x], axis=0)
    np.testing.assert_array_equal(h1[0], all_bits[-3:].T)


def test_gated_rmsnorm_closed_form():
    """RMSNorm of a constant row a: a / sqrt(a^2 + eps) * gamma, gated by SiLU(z)."""
    T, H, D = 2, 3, 8
    rng = np.random.default_rng(18)
    a = np.array([0.5, -2.0, 1.0, 4.0, -0.25, 2.0], np.float32).reshape(T, H, 1)
    o = synth.bf16_bits(np.broadcast_to(a, (T, H, D)).astype(np.float32))
    zf = synth.bf16_to_f32(synth.bf16_bits(rng.standard_normal((T, H, D)).astype(np.float32)))
    z = synth.bf16_bits(zf)
    gamma = rng.uniform(0.5, 1.5, D).astype(np.float32)
    eps = 1e-6
    out = oracle.gated_rmsnorm(o, z, gamma, eps).reshape(T, H, D)
    af = a.astype(np.float64)
    expect = af / np.sqrt(af * af + eps) * gamma.astype(np.float64) * silu(zf.astype(np.float64))
    np.testing.assert_allclose(out, expect, rtol=1e-14)


def test_gate_is_applied_per_head_in_forward():
    """Ogate[t, h] depends on o[t, h] and z[t, h] only: the RMS is taken per head."""
    w = _tiny_inputs(19, T=3)
    qsl, slots = np.array([0, 3], np.int32), np.array([2], np.int32)
    r = _fwd(w, qsl, slots)
    o = r["o"]
    zf = synth.bf16_to_f32(w["z"]).astype(np.float64)
    rms = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + w["eps"])
    np.testing.assert_allclose(r["ogate"].reshape(o.shape), o / rms * silu(zf), rtol=1e-13)


def test_head_grouping_value_head_reads_key_head_h_div_g():
    """Changing the k channels of key head j changes exactly value heads G*j .. G*j+G-1."""
    G = TINY.group
    w = _tiny_inputs(20, T=4)
    qsl, slots = np.array([0, 4], np.int32), np.array([1], np.int32)
    base = _fwd(w, qsl, slots)
    for j in range(TINY.num_k_heads):
        w2 = dict(w)
        x = synth.bf16_to_f32(w["qkv0"]).copy()
        kc = TINY.num_k_heads * TINY.head_k_dim + j * TINY.head_k_dim
        x[:, kc : kc + TINY.head_k_dim] += 0.75
        w2["qkv0"] = synth.bf16_bits(x)
        r = _fwd(w2, qsl, slots)
        changed = [h for h in range(TINY.num_v_heads)
                   if not np.array_equal(r["o"][:, h], base["o"][:, h])]
        assert changed == list(range(G * j, G * j + G)), (j, changed)


def test_channel_layout_q_then_k_then_v():
    """[Q | K | V] layout: q channels reach only the outputs (the state never reads q), k channels
    reach the state of their group, a v channel of head h reaches head h only."""
    w = _tiny_inputs(21, T=3)
    qsl, slots = np.array([0, 3], np.int32), np.array([3], np.int32)
    base = _fwd(w, qsl, slots)
    x = synth.bf16_to_f32(w["qkv0"])
    dk, dv, Hk = TINY.head_k_dim, TINY.head_v_dim, TINY.num_k_heads

    def run_with(offset):
        x2 = x.copy()
        x2[:, offset] += 1.0
        w2 = dict(w, qkv0=synth.bf16_bits(x2))
        return _fwd(w2, qsl, slots)

    rq = run_with(0 * dk + 1)  # a q channel of key head 0
    np.testing.assert_array_equal(rq["state"], base["state"])
    assert not np.array_equal(rq["o"][:, 0], base["o"][:, 0])
    rk = run_with(Hk * dk + 1)  # a k channel of key head 0
    assert not np.array_equal(rk["state"][3, 0], base["state"][3, 0])
    np.testing.assert_array_equal(rk["state"][3, TINY.group:], base["state"][3, TINY.group:])
    h = 4
    rv = run_with(2 * Hk * dk + h * dv + 2)  # a v channel of value head 4
    diff = [g for g in range(TINY.num_v_heads) if not np.array_equal(rv["state"][3, g], base["state"][3, g])]
    assert diff == [h]


def test_split_invariance_prefill_then_decode():
    """One prefill of T tokens = prefill(T1) then prefill(T - T1) from the carried slot = T decode
    steps. The state is carried through its fp32 pool between calls, hence the 1e-6 tolerance."""
    T, T1 = 11, 4
    w = _tiny_inputs(22, T=T)
    slot = np.array([2], np.int32)
    full = _fwd(w, np.array([0, T], np.int32), slot)

    def part(wd, t0, t1):
        sub = dict(wd)
        for key in ("qkv0", "alpha", "beta", "z"):
            sub[key] = np.ascontiguousarray(w[key][t0:t1])
        return _fwd(sub, np.array([0, t1 - t0], np.int32), slot)

    a = part(w, 0, T1)
    b = part(dict(w, state=a["state"], conv_hist=a["conv_hist"]), T1, T)
    np.testing.assert_array_equal(b["conv_hist"], full["conv_hist"])
    np.testing.assert_allclose(b["state"], full["state"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(np.concatenate([a["o"], b["o"]]), full["o"], rtol=1e-5, atol=1e-6)
    cur = dict(w)
    outs = []
    for t in range(T):
        r = part(cur, t, t + 1)
        outs.append(r["o"])
        cur = dict(cur, state=r["state"], conv_hist=r["conv_hist"])
    np.testing.assert_array_equal(cur["conv_hist"], full["conv_hist"])
    np.testing.assert_allclose(cur["state"], full["state"], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(np.concatenate(outs), full["o"], rtol=1e-5, atol=1e-6)


def test_zero_start_equals_zeroed_slot_and_padding_is_skipped():
    """has_init = 0 starts from S = 0 and a zero history; slot -1 is padding and touches nothing."""
    w = _tiny_inputs(23, T=5)
    qsl = np.array([0, 3, 5], np.int32)
    slots = np.array([1, -1], np.int32)
    r0 = _fwd(w, qsl, slots, has_init=np.array([0, 1], np.uint8))
    wz = dict(w, state=w["state"].copy(), conv_hist=w["conv_hist"].copy())
    wz["state"][1] = 0
    wz["conv_hist"][1] = 0
    r1 = _fwd(wz, qsl, slots)
    np.testing.assert_array_equal(r0["o"], r1["o"])
    np.testing.assert_array_equal(r0["state"][1], r1["state"][1])
    assert not r0["o"][3:].any() and not r0["ogate"][3:].any()
    for s in (0, 2, 3):
        np.testing.assert_array_equal(r0["state"][s], w["state"][s])
        np.testing.assert_array_equal(r0["conv_hist"][s], w["conv_hist"][s])


def test_spec_checkpoints_equal_prefix_runs_and_commit():
    """The checkpoint kept after position p equals a plain run over the first p+1 positions;
    commit copies (or repoints to) the checkpoint of the accepted position."""
    N, P, Rs = 3, 4, 3 * 5
    w = _tiny_inputs(24, T=N * P, Rs=Rs)
    slots = np.array([0, 1, 2], np.int32)
    spec = (3 + np.arange(N * P, dtype=np.int32)).reshape(N, P)
    r = oracle.spec_verify(TINY, w["qkv0"], w["conv_w"], w["conv_hist"], w["state"], slots, spec,
                           w["alpha"], w["beta"], w["z"], w["gamma"], w["eps"])
    for n in range(N):
        np.testing.assert_array_equal(r["state"][slots[n]], w["state"][slots[n]])
        for p in range(P):
            sub = {k: np.ascontiguousarray(w[k][n * P : n * P + p + 1]) for k in ("qkv0", "alpha", "beta", "z")}
            ref = _fwd(dict(w, **sub), np.array([0, p + 1], np.int32), slots[n : n + 1])
            np.testing.assert_array_equal(r["state"][spec[n, p]], ref["state"][slots[n]])
            np.testing.assert_array_equal(r["conv_hist"][spec[n, p]], ref["conv_hist"][slots[n]])
            np.testing.assert_array_equal(r["o"][n * P + p], ref["o"][p])
    acc = np.array([2, 0, 3], np.int32)
    st, hist, sl = oracle.spec_commit(r["state"], r["conv_hist"], slots, spec, acc, mode="copy")
    for n in range(N):
        np.testing.assert_array_equal(st[slots[n]], r["state"][spec[n, acc[n]]])
        np.testing.assert_array_equal(hist[slots[n]], r["conv_hist"][spec[n, acc[n]]])
    _, _, sl2 = oracle.spec_commit(r["state"], r["conv_hist"], slots, spec, acc, mode="repoint")
    np.testing.assert_array_equal(sl2, spec[np.arange(N), acc])


# ---------------------------------------------------------------- page facts

def test_state_and_history_sizes_match_the_page():
    g = json.load(open(os.path.join(GOLDEN, "state_sizes.json")))["facts"]
    d = synth.FULL_HEADS
    assert [d.num_v_heads, d.head_v_dim, d.head_k_dim] == g["state_shape_per_slot"]
    assert d.num_v_heads * d.head_v_dim * d.head_k_dim * 4 == g["state_bytes_per_sequence_per_layer"] == 3 * 2**20
    assert [d.channels, d.conv_kernel - 1] == g["conv_hist_shape_per_slot"]
    r = synth.RANK_HEADS
    assert [r.num_v_heads, r.head_v_dim, r.head_k_dim] == g["tp4_state_shape_per_rank"]
    assert [r.channels, r.conv_kernel - 1] == g["tp4_conv_hist_shape_per_rank"]
    pool = synth.zero_pool(d, 1)
    assert pool["state"].nbytes == g["state_bytes_per_sequence_per_layer"]
    assert list(pool["conv_hist"].shape[1:]) == g["conv_hist_shape_per_slot"]


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 2**-7 + 2**-8, 1.0 + 2**-9, -3.0], np.float32)
    got = synth.bf16_to_f32(synth.bf16_bits(x))
    np.testing.assert_array_equal(got, np.array([1.0, 1.0, 1.0 + 2**-6, 1.0, -3.0], np.float32))


def test_forward_write_through_needs_unit_q_and_k():
    """Whole chain with beta = 1 and each q head a copy of its k head (same inputs, taps and
    history): the step writes v exactly and reads it back, o_t = v_t / sqrt(dk). This holds only if
    both q and k are L2-normalized after the conv and the state is decayed before the prediction."""
    T = 5
    w = _tiny_inputs(25, T=T)
    dk, Hk = TINY.head_k_dim, TINY.num_k_heads
    q_ch, k_ch = slice(0, Hk * dk), slice(Hk * dk, 2 * Hk * dk)
    x = w["qkv0"].copy()
    x[:, q_ch] = x[:, k_ch]
    cw = w["conv_w"].copy()
    cw[q_ch] = cw[k_ch]
    hist = w["conv_hist"].copy()
    hist[:, q_ch] = hist[:, k_ch]
    w2 = dict(w, qkv0=x, conv_w=cw, conv_hist=hist, beta=np.ones_like(w["beta"]))
    r = _fwd(w2, np.array([0, T], np.int32), np.array([0], np.int32), want_y=True)
    v = r["y"][:, 2 * Hk * dk :].reshape(T, TINY.num_v_heads, TINY.head_v_dim)
    np.testing.assert_allclose(r["o"] * np.sqrt(dk), v, rtol=1e-11, atol=1e-12)


def test_empty_request_leaves_its_slot_untouched():
    """A request with no tokens reads and writes nothing, with or without an initial state."""
    w = _tiny_inputs(26, T=3)
    qsl = np.array([0, 0, 3], np.int32)
    slots = np.array([1, 2], np.int32)
    for init in (0, 1):
        r = _fwd(w, qsl, slots, has_init=np.array([init, 1], np.uint8))
        np.testing.assert_array_equal(r["state"][1], w["state"][1])
        np.testing.assert_array_equal(r["conv_hist"][1], w["conv_hist"][1])
        _, h = oracle.conv_update(TINY, w["qkv0"], w["conv_w"], w["conv_hist"], qsl, slots,
                                  np.array([init, 1], np.uint8))
        np.testing.assert_array_equal(h[1], w["conv_hist"][1])


# ---------------------------------------------------------------- output projection (Wo row)

def _bits(x):
    return synth.bf16_bits(np.asarray(x, np.float32))


def test_out_proj_hand_example_and_residual():
    """A 2x3 times (2x3)^T product written out by hand, then the residual add."""
    a = np.array([[1.0, 2.0, -1.0], [0.5, 0.0, 4.0]])
    w = np.array([[1.0, 0.0, 2.0], [-1.0, 3.0, 0.25]])  # [N=2][K=3]
    expect = np.array([[1 + 0 - 2, -1 + 6 - 0.25], [0.5 + 0 + 8, -0.5 + 0 + 1]])
    np.testing.assert_array_equal(oracle.out_proj(_bits(a), _bits(w)), expect)
    r = np.array([[10.0, -2.0], [0.0, 1.5]])
    np.testing.assert_array_equal(oracle.out_proj(_bits(a), _bits(w), _bits(r)), expect + r)


def test_out_proj_one_hot_rows_select_input_columns():
    """Row n of W a one-hot at k: output column n is input column k (W is [N][K], not [K][N])."""
    rng = np.random.default_rng(71)
    T, K, N = 5, 16, 8
    a = rng.normal(size=(T, K))
    cols = rng.permutation(K)[:N]
    w = np.zeros((N, K))
    w[np.arange(N), cols] = 1.0
    got = oracle.out_proj(_bits(a), _bits(w))
    np.testing.assert_array_equal(got, synth.bf16_to_f32(_bits(a)).astype(np.float64)[:, cols])


# ---------------------------------------------------------------- input RMSNorm (U row), fused residual add

def test_rmsnorm_hand_values():
    """[3, 4, 0, 0]: mean of squares 25/4, rms 2.5, so U = [1.2, 1.6, 0, 0] * gamma; a constant row
    c = 1 with eps = 3 gives 1 / sqrt(1 + 3) = 0.5 (eps sits inside the root, added to the mean)."""
    u, res = oracle.rmsnorm(_bits([[3.0, 4.0, 0.0, 0.0]]), np.array([1.0, 2.0, 1.0, 1.0]), 0.0)
    np.testing.assert_allclose(u, [[1.2, 3.2, 0.0, 0.0]], rtol=1e-15)
    assert res is None
    u, _ = oracle.rmsnorm(_bits(np.ones((2, 8))), np.ones(8), 3.0)
    np.testing.assert_array_equal(u, np.full((2, 8), 0.5))


def test_rmsnorm_residual_sum_rounds_once_to_nearest_even():
    """Sums worked by hand on the bf16 grid (8 significant bits: spacing 2^-7 above 1, 2^-8 below):
    1 + 2^-8 is a tie and goes to 1 (even); 1 + 3*2^-8 is a tie between 1 + 2^-7 and 1 + 2^-6 and goes
    to 1 + 2^-6 (even); 1 - 2^-9 is a tie between 1 - 2^-8 and 1 and goes to 1; 1 + 2^-7 is exact."""
    x = np.array([[1.0, 1.0, 1.0, 1.0 + 2.0 ** -7]])
    r = np.array([[2.0 ** -8, 3 * 2.0 ** -8, -2.0 ** -9, 0.0]])
    _, res = oracle.rmsnorm(_bits(x), np.ones(4), 1e-6, _bits(r))
    got = synth.bf16_to_f32(res).astype(np.float64)
    np.testing.assert_array_equal(got, [[1.0, 1.0 + 2.0 ** -6, 1.0, 1.0 + 2.0 ** -7]])
    # the norm is taken of the stored (rounded) sum, not of the exact one
    u, _ = oracle.rmsnorm(_bits(x), np.ones(4), 1e-6, _bits(r))
    s = got[0]
    np.testing.assert_allclose(u[0], s / np.sqrt(np.mean(s * s) + 1e-6), rtol=1e-15)


def test_rmsnorm_scale_invariance_and_unit_rms():
    """With eps = 0, U does not change when a row is scaled by a power of two, and U / gamma has mean
    square exactly 1 per row."""
    rng = np.random.default_rng(72)
    x = _bits(rng.normal(size=(6, 40)))
    g = rng.uniform(0.5, 2.0, size=40)
    u, _ = oracle.rmsnorm(x, g, 0.0)
    u4, _ = oracle.rmsnorm(_bits(4.0 * synth.bf16_to_f32(x)), g, 0.0)
    np.testing.assert_allclose(u4, u, rtol=1e-14)
    np.testing.assert_allclose(np.mean((u / g) ** 2, axis=1), 1.0, rtol=1e-13)


# ---------------------------------------------------------------- FP8 E4M3 block-scaled projections

def test_e4m3_codes_decode_to_the_format_values():
    """OCP E4M3: exponent bias 7, 3 mantissa bits, subnormal step 2^-9, largest finite 448,
    S.1111.111 the only NaN, sign-magnitude (0x80 is -0)."""
    got = oracle.e4m3_to_f64([0x00, 0x01, 0x07, 0x08, 0x38, 0x3C, 0x40, 0x7E, 0xB8, 0x80])
    np.testing.assert_array_equal(got, [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.5, 2.0, 448.0, -1.0, 0.0])
    assert np.signbit(got[-1])
    assert np.isnan(oracle.e4m3_to_f64([0x7F, 0xFF])).all()
    # 254 finite codes, all distinct values apart from +-0
    v = oracle.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    fin = v[~np.isnan(v)]
    assert fin.size == 254 and np.unique(fin).size == 253


def test_e4m3_encoding_rounds_to_nearest_even_and_saturates():
    """Every finite code survives decode -> encode; ties worked by hand go to the even mantissa:
    1 + 1/16 -> 1 (0x38), 1 + 3/16 -> 1.25 (0x3A), 2^-10 -> 0, 3 * 2^-10 -> 2^-8 (0x02);
    magnitudes past 448 saturate (0x7E / 0xFE)."""
    codes = np.arange(256, dtype=np.uint8)
    v = oracle.e4m3_to_f64(codes)
    fin = ~np.isnan(v)
    np.testing.assert_array_equal(oracle.e4m3_from_f32(v[fin].astype(np.float32)), codes[fin])
    got = oracle.e4m3_from_f32(np.array([1 + 1 / 16, 1 + 3 / 16, 2.0 ** -10, 3 * 2.0 ** -10, 500.0, -1e6, 447.0],
                                        np.float32))
    np.testing.assert_array_equal(got, np.array([0x38, 0x3A, 0x00, 0x02, 0x7E, 0xFE, 0x7E], np.uint8))


def test_fp8_quantisers_scale_and_error_bound():
    """A group whose largest magnitude is 448 gets scale 1 and the plain codes; an all-zero group gets
    codes 0 and scale fp32(1e-12)/448; every code is within half a step of x / s (3 mantissa bits:
    relative 2^-4, absolute 2^-10 in the subnormal range); the weight blocks follow the same rule."""
    rng = np.random.default_rng(73)
    x = rng.normal(size=(3, 384)).astype(np.float32)
    x[0, :128] = np.clip(x[0, :128] * 100.0, -440.0, 440.0)
    x[0, 5] = -448.0
    x[1, 128:256] = 0.0
    xb = _bits(x)
    codes, s = oracle.fp8_quant_act(xb)
    xv = synth.bf16_to_f32(xb).astype(np.float64)
    assert s[0, 0] == np.float32(1.0)
    np.testing.assert_array_equal(codes[0, :128], oracle.e4m3_from_f32(xv[0, :128].astype(np.float32)))
    assert np.all(codes[1, 128:256] == 0) and s[1, 1] == np.float32(np.float32(1e-12) / np.float32(448.0))
    deq = oracle.e4m3_to_f64(codes) * np.repeat(s.astype(np.float64), 128, axis=1)
    ratio = xv / np.repeat(s.astype(np.float64), 128, axis=1)
    assert np.all(np.abs(ratio) <= 448.0 * (1 + 1e-6))
    assert np.all(np.abs(deq - xv) <= np.repeat(s.astype(np.float64), 128, axis=1) *
                  (2.0 ** -4 * np.abs(ratio) + 2.0 ** -10) + 1e-30)
    w = rng.normal(size=(200, 256)).astype(np.float32)
    wc, ws = oracle.fp8_quant_weight(_bits(w))
    assert ws.shape == (2, 2)
    wv = synth.bf16_to_f32(_bits(w)).astype(np.float64)
    for nb in range(2):
        for kb in range(2):
            blk = wv[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            assert ws[nb, kb] == np.float32(np.float32(np.abs(blk).max()) / np.float32(448.0))


def test_fp8_linear_hand_example():
    """K = 256 (two scale blocks), one token, one output: codes 1.0 and 0.5, block scales chosen by
    hand: out = 128 * (1 * 0.5) * (2 * 3) + 128 * (1 * 0.5) * (4 * 0.25) = 384 + 64 = 448."""
    x8 = np.full((1, 256), 0x38, np.uint8)
    w8 = np.full((16, 256), 0x30, np.uint8)  # 0.5
    xs = np.array([[2.0, 4.0]], np.float32)
    ws = np.array([[3.0, 0.25]], np.float32)
    out = oracle.fp8_linear(x8, xs, w8, ws)
    np.testing.assert_array_equal(out, np.full((1, 16), 448.0))
    r = np.full((1, 16), -48.0)
    np.testing.assert_array_equal(oracle.fp8_linear(x8, xs, w8, ws, _bits(r)), np.full((1, 16), 400.0))
