"""Python face of the GDN mixer-core oracle (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
import this module. The GPU product path never does.

* ``forward``, ``conv_update``, ``gated_rmsnorm``, ``delta_rule_seq`` and
  ``spec_verify`` call the fp64 C oracle in ``gdn_oracle.c`` (token by token, in
  the order of the "Qwen3.8-27B: from model structure to vLLM inference data
  flow" page, section 01 LAYER-BY-LAYER, GDN operator table).
* ``spec_commit`` applies the greedy accept rule of the "Qwen3.8 MTP" page,
  section 5 (accept / reject): a request keeps the state after its accepted
  position.
* ``out_proj`` is the output projection after the mixer and the residual add
  (first page, section 01 GDN operator table, the Wo row): a plain fp64 matrix
  product of the bf16 inputs.
* ``chunked_delta_rule`` is a separate fp64 numpy statement of the chunked
  (WY / UT) form of the same recurrence, used only to check the chunk algebra
  against the token-by-token form. The first page only says that the block
  recurrence uses the associative structure to run in parallel (section 01,
  "prefill can run in parallel"); the derivation is written out in the
  function's docstring.

Inputs are the numpy arrays of ``gated_deltanet_linear_conv1d_gb300.synth``
(bf16 as uint16 bit patterns).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdn_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_fp = ctypes.POINTER(ctypes.c_float)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (fp64, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_delta_rule_seq.argtypes = [ctypes.c_int] * 3 + [_dp] * 5 + [_dp, _dp, ctypes.c_int]
            lib.oracle_gated_rmsnorm.argtypes = [ctypes.c_int] * 3 + [_u16p, _u16p, _fp, ctypes.c_double, _dp]
            lib.oracle_conv_update.argtypes = [ctypes.c_int, ctypes.c_int, _u16p, _fp, _u16p, _i32p, _i32p,
                                               _u8p, ctypes.c_int, _dp]
            lib.oracle_gdn_forward.argtypes = ([ctypes.c_int] * 5 + [_u16p, _fp, _u16p, _fp, ctypes.c_int,
                                               _i32p, _i32p, _u8p, ctypes.c_int, _fp, _fp, _u16p, _fp,
                                               ctypes.c_double, _i32p, _dp, _dp, _dp])
            _lib = lib
    return _lib


def num_threads() -> int:
    """OpenMP threads the oracle runs with (OMP_NUM_THREADS, else all cores)."""
    return int(_load().oracle_num_threads())


def _ptr(a: np.ndarray | None, ctype):
    if a is None:
        return ctypes.cast(None, ctypes.POINTER(ctype))
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def delta_rule_seq(q, k, v, alpha, beta, S0, normalize: bool = False):
    """Gated delta rule of one head over T tokens (fp64). q, k: [T, dk]; v: [T, dv]; S0: [dv, dk].

    Returns (o [T, dv], S [dv, dk]). With normalize=False the keys and queries
    are used as given (the closed-form checks feed unit keys straight to the core).
    """
    q, k, v = _c(q, np.float64), _c(k, np.float64), _c(v, np.float64)
    alpha, beta = _c(alpha, np.float64), _c(beta, np.float64)
    T, dk = q.shape
    dv = v.shape[1]
    S = _c(S0, np.float64).copy()
    o = np.zeros((T, dv), np.float64)
    _load().oracle_delta_rule_seq(dk, dv, T, _ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                                  _ptr(v, ctypes.c_double), _ptr(alpha, ctypes.c_double),
                                  _ptr(beta, ctypes.c_double), _ptr(S, ctypes.c_double),
                                  _ptr(o, ctypes.c_double), int(bool(normalize)))
    return o, S


def gated_rmsnorm(o_bits, z_bits, gamma, eps):
    """RMSNorm(o) * gamma * SiLU(z) per head; o, z: bf16 bits [T, H, D]. Returns fp64 [T, H*D]."""
    o_bits, z_bits = _c(o_bits, np.uint16), _c(z_bits, np.uint16)
    T, H, D = o_bits.shape
    out = np.zeros((T, H * D), np.float64)
    _load().oracle_gated_rmsnorm(T, H, D, _ptr(o_bits, ctypes.c_uint16), _ptr(z_bits, ctypes.c_uint16),
                                 _ptr(_c(gamma, np.float32), ctypes.c_float), float(eps),
                                 _ptr(out, ctypes.c_double))
    return out


def conv_update(dims, qkv0, conv_w, conv_hist, query_start_loc, slot_idx, has_init=None):
    """Varlen causal conv + SiLU. Returns (y fp64 [T, CH], updated copy of conv_hist)."""
    qkv0 = _c(qkv0, np.uint16)
    hist = _c(conv_hist, np.uint16).copy()
    qsl, slots = _c(query_start_loc, np.int32), _c(slot_idx, np.int32)
    hi = None if has_init is None else _c(has_init, np.uint8)
    T, CH = qkv0.shape
    y = np.zeros((T, CH), np.float64)
    _load().oracle_conv_update(CH, dims.conv_kernel, _ptr(qkv0, ctypes.c_uint16),
                               _ptr(_c(conv_w, np.float32), ctypes.c_float), _ptr(hist, ctypes.c_uint16),
                               _ptr(qsl, ctypes.c_int32), _ptr(slots, ctypes.c_int32),
                               _ptr(hi, ctypes.c_uint8), len(slots), _ptr(y, ctypes.c_double))
    return y, hist


def forward(dims, qkv0, conv_w, conv_hist, state, query_start_loc, slot_idx, alpha, beta, z, gamma,
            eps, has_init=None, ckpt_slot=None, want_y: bool = False, inplace: bool = False):
    """The whole mixer core over packed varlen requests (fp64).

    conv_hist [Rs, CH, K-1] bf16 bits and state [Rs, Hv, dv, dk] fp32 are the
    slot pools; they are updated in place when inplace=True, else on copies.
    Returns a dict with o [T, Hv, dv], ogate [T, Hv*dv] (fp64), the pools
    ("state", "conv_hist") and, when want_y, the conv outputs y [T, CH].
    """
    qkv0 = _c(qkv0, np.uint16)
    T, CH = qkv0.shape
    Hk, Hv, dk, dv, K = (dims.num_k_heads, dims.num_v_heads, dims.head_k_dim, dims.head_v_dim,
                         dims.conv_kernel)
    hist = conv_hist if inplace else np.array(conv_hist, dtype=np.uint16, copy=True)
    st = state if inplace else np.array(state, dtype=np.float32, copy=True)
    assert hist.dtype == np.uint16 and hist.flags["C_CONTIGUOUS"]
    assert st.dtype == np.float32 and st.flags["C_CONTIGUOUS"]
    slots = _c(slot_idx, np.int32)
    qsl = _c(query_start_loc, np.int32)
    hi = None if has_init is None else _c(has_init, np.uint8)
    ck = None if ckpt_slot is None else _c(ckpt_slot, np.int32)
    o = np.zeros((T, Hv, dv), np.float64)
    og = np.zeros((T, Hv * dv), np.float64)
    y = np.zeros((T, CH), np.float64) if want_y else None
    _load().oracle_gdn_forward(
        Hk, Hv, dk, dv, K, _ptr(qkv0, ctypes.c_uint16), _ptr(_c(conv_w, np.float32), ctypes.c_float),
        _ptr(hist, ctypes.c_uint16), _ptr(st, ctypes.c_float), st.shape[0], _ptr(qsl, ctypes.c_int32),
        _ptr(slots, ctypes.c_int32), _ptr(hi, ctypes.c_uint8), len(slots),
        _ptr(_c(alpha, np.float32), ctypes.c_float), _ptr(_c(beta, np.float32), ctypes.c_float),
        _ptr(_c(z, np.uint16), ctypes.c_uint16), _ptr(_c(gamma, np.float32), ctypes.c_float), float(eps),
        _ptr(ck, ctypes.c_int32), _ptr(o, ctypes.c_double), _ptr(og, ctypes.c_double),
        _ptr(y, ctypes.c_double) if y is not None else ctypes.cast(None, _dp))
    out = {"o": o, "ogate": og, "state": st, "conv_hist": hist}
    if want_y:
        out["y"] = y
    return out


def spec_verify(dims, qkv0, conv_w, conv_hist, state, slot_idx, spec_slot_idx, alpha, beta, z,
                gamma, eps, inplace: bool = False):
    """Verify num_pos positions per request, keeping the state and conv history
    after every position p in slot spec_slot_idx[n, p]; the live slots stay as
    they are. qkv0, alpha, beta, z hold the positions request-major ([N*P, ...]).
    """
    spec = _c(spec_slot_idx, np.int32)
    N, P = spec.shape
    qsl = (np.arange(N + 1, dtype=np.int32) * P)
    return forward(dims, qkv0, conv_w, conv_hist, state, qsl, slot_idx, alpha, beta, z, gamma, eps,
                   ckpt_slot=spec.reshape(-1), inplace=inplace)


def spec_commit(state, conv_hist, slot_idx, spec_slot_idx, accepted, mode: str = "copy"):
    """Commit each request at its accepted position a ("Qwen3.8 MTP" page, section 5:
    the longest accepted prefix is kept and the state follows it).

    mode "copy": the checkpoint of position a is copied into the live slot.
    mode "repoint": the live slot index becomes the checkpoint's slot.
    Returns (state, conv_hist, slot_idx) as new arrays.
    """
    spec = np.asarray(spec_slot_idx, np.int32)
    acc = np.asarray(accepted, np.int32)
    src = spec[np.arange(len(acc)), acc]
    slots = np.array(slot_idx, np.int32, copy=True)
    st = np.array(state, copy=True)
    hist = np.array(conv_hist, copy=True)
    if mode == "copy":
        for n in range(len(acc)):
            if slots[n] < 0:
                continue
            st[slots[n]] = state[src[n]]
            hist[slots[n]] = conv_hist[src[n]]
    elif mode == "repoint":
        live = slots >= 0
        slots[live] = src[live]
    else:
        raise ValueError(mode)
    return st, hist, slots


def out_proj(ogate_bits, w_bits, residual_bits=None):
    """out = ogate W^T (+ residual) in fp64 from bf16 bits; ogate [T, K], W [N, K]
    (nn.Linear layout), residual [T, N]. The Wo row of the GDN operator table
    maps [T,6144] to [T,5120]; the residual stream adds the layer input back."""
    a = _bf16(ogate_bits)
    w = _bf16(w_bits)
    out = a @ w.T
    if residual_bits is not None:
        out = out + _bf16(residual_bits)
    return out


def rmsnorm(x_bits, gamma, eps, residual_bits=None):
    """The layer's input norm U = X / sqrt(mean(X^2 over the hidden size) + eps) * gamma in fp64 (page
    "Qwen3.8-27B: from model structure to vLLM inference data flow", section 01 operator table, the U
    row). With a residual, the residual stream is first X + residual, stored as bf16 the way a separate
    add would store it, and the norm is taken of that stored sum (page "DeepSeek-V3 inference pipeline
    walk-through" section 4.2: the fused add-and-norm equals the add followed by the norm).
    Returns (U [T, D] fp64, the new residual as bf16 bits or None)."""
    x = _bf16(x_bits)
    new_res = None
    if residual_bits is not None:
        new_res = _round_bf16(x + _bf16(residual_bits))
        x = _bf16(new_res)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + float(eps)) * np.asarray(gamma, dtype=np.float64), new_res


# ---------------------------------------------------------------- FP8 E4M3 block-scaled projections
# Page "Qwen3.8-27B: from model structure to vLLM inference data flow", section 04 (precision and
# cache): the linear weights are FP8 E4M3 with one scale per 128 x 128 block and activations are
# quantised dynamically. E4M3 here is the OCP FP8 format: 1 sign bit, 4 exponent bits with bias 7,
# 3 mantissa bits, subnormals at exponent 0, no infinities, S.1111.111 the only NaN, 448 the largest
# finite value.

def e4m3_to_f64(codes) -> np.ndarray:
    """E4M3 codes (uint8) to their values, straight from the bit fields."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((e == 15) & ((c & 0x7) == 7), np.nan, mag)
    return sign * mag


def e4m3_from_f32(v) -> np.ndarray:
    """fp32 values to E4M3 codes: round to nearest, ties to even mantissa, magnitudes above 448
    saturate to 448 (the value keeps its sign, zero included)."""
    x = np.asarray(v, dtype=np.float32).astype(np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))       # a = f 2^ex, 1/2 <= f < 1: binade 2^(ex-1)
    e = np.clip(ex - 1, -6, 8)                      # below 2^-6 the spacing stays 2^-9 (subnormals)
    q = np.ldexp(1.0, e - 3)                        # spacing of the binade: 3 mantissa bits
    r = np.minimum(np.round(a / q) * q, 448.0)      # a / q is exact; np.round ties to even
    _, rex = np.frexp(np.where(r > 0, r, 1.0))
    normal = r >= 2.0 ** -6
    E = np.where(normal, rex - 1 + 7, 0)
    M = np.where(normal, r / np.ldexp(1.0, rex - 1) - 1.0, r / 2.0 ** -9)
    M = np.where(normal, M * 8.0, M)
    code = (E.astype(np.int64) << 3) | np.round(M).astype(np.int64)
    return (code | np.where(neg, 0x80, 0)).astype(np.uint8)


def _fp8_block_scale(amax) -> np.ndarray:
    """Block scale s = max(amax, 1e-12) / 448 as an IEEE fp32 division."""
    return (np.maximum(np.asarray(amax, np.float32), np.float32(1e-12)) / np.float32(448.0)).astype(np.float32)


def fp8_quant_act(x_bits):
    """Dynamic activation quantisation: one scale per token and 128-wide group of K. x [T, K] bf16
    bits -> (codes [T, K] uint8, scales [T, K/128] fp32); code = E4M3(x / s), the division in fp32."""
    x = _bf16(x_bits).astype(np.float32)
    T, K = x.shape
    g = x.reshape(T, K // 128, 128)
    s = _fp8_block_scale(np.abs(g).max(axis=2))
    codes = e4m3_from_f32((g / s[:, :, None]).astype(np.float32))
    return codes.reshape(T, K), s


def fp8_quant_weight(w_bits):
    """Weight quantisation with one scale per 128 x 128 block (a last partial row block takes the
    largest magnitude of the rows it has). w [N, K] bf16 bits -> (codes [N, K], scales [ceil(N/128), K/128])."""
    w = _bf16(w_bits).astype(np.float32)
    N, K = w.shape
    NB, KB = (N + 127) // 128, K // 128
    codes = np.zeros((N, K), np.uint8)
    s = np.zeros((NB, KB), np.float32)
    for nb in range(NB):
        for kb in range(KB):
            blk = w[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128]
            s[nb, kb] = _fp8_block_scale(np.abs(blk).max())
            codes[nb * 128:(nb + 1) * 128, kb * 128:(kb + 1) * 128] = e4m3_from_f32((blk / s[nb, kb]).astype(np.float32))
    return codes, s


def fp8_linear(x8, x_scale, w8, w_scale, residual_bits=None):
    """out = dequant(X) dequant(W)^T (+ residual) in fp64, dequant(X)[t, k] = E4M3(x8[t, k]) x_scale[t, k/128]
    and dequant(W)[n, k] = E4M3(w8[n, k]) w_scale[n/128, k/128]."""
    x = e4m3_to_f64(x8) * np.repeat(np.asarray(x_scale, np.float64), 128, axis=1)
    ws = np.repeat(np.repeat(np.asarray(w_scale, np.float64), 128, axis=0), 128, axis=1)
    w = e4m3_to_f64(w8) * ws[:w8.shape[0]]
    out = x @ w.T
    if residual_bits is not None:
        out = out + _bf16(residual_bits)
    return out


def _round_bf16(x) -> np.ndarray:
    """fp64 values to bf16 bits, round to nearest, ties to even, straight from fp64 (one rounding):
    x = m 2^e with 1/2 <= |m| < 1, keep 8 significant bits of m (np.round breaks ties to even)."""
    m, e = np.frexp(np.asarray(x, dtype=np.float64))
    r = np.ldexp(np.round(np.ldexp(m, 8)), e - 8)
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _bf16(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) to fp64 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def chunked_delta_rule(q, k, v, alpha, beta, S0, chunk: int = 64):
    """Chunked (WY / UT) form of the gated delta rule for one head, fp64 numpy.

    Unrolling S_r = alpha_r S_{r-1} + beta_r e_r k_r^T, e_r = v_r - alpha_r S_{r-1} k_r
    inside a chunk that starts from S0, with g_r = sum_{i<=r} ln alpha_i and
    Gamma[r, i] = exp(g_r - g_i):

      S_r = exp(g_r) S0 + sum_{i<=r} Gamma[r, i] E_i k_i^T,       E_i = beta_i e_i
      (I + A) E = diag(beta) V - diag(beta exp(g)) K S0^T,
              A[r, i] = beta_r Gamma[r, i] (k_r . k_i) for i < r, else 0
      W = (I + A)^-1 diag(beta exp(g)) K,  U = (I + A)^-1 diag(beta) V,  E = U - W S0^T
      O = [diag(exp(g)) Q S0^T + ((Q K^T) * Gamma * [i <= r]) E] / sqrt(dk)
      S_C = exp(g_C) S0 + E^T diag(Gamma[C, :]) K

    q, k: [T, dk] (used as given); v: [T, dv]; S0: [dv, dk]. Returns (o, S).
    """
    q, k, v = (np.asarray(a, np.float64) for a in (q, k, v))
    alpha, beta = np.asarray(alpha, np.float64), np.asarray(beta, np.float64)
    T, dk = q.shape
    dv = v.shape[1]
    S = np.array(S0, np.float64, copy=True)
    o = np.zeros((T, dv))
    for c0 in range(0, T, chunk):
        c1 = min(T, c0 + chunk)
        Q, K, V, b = q[c0:c1], k[c0:c1], v[c0:c1], beta[c0:c1]
        L = c1 - c0
        g = np.cumsum(np.log(alpha[c0:c1]))
        mask_incl = np.tril(np.ones((L, L)))
        Gam = np.exp(np.where(mask_incl > 0, g[:, None] - g[None, :], -np.inf))
        A = b[:, None] * Gam * (K @ K.T) * np.tril(np.ones((L, L)), -1)
        I_A = np.eye(L) + A
        W = np.linalg.solve(I_A, (b * np.exp(g))[:, None] * K)
        U = np.linalg.solve(I_A, b[:, None] * V)
        E = U - W @ S.T
        o[c0:c1] = (np.exp(g)[:, None] * (Q @ S.T) + ((Q @ K.T) * Gam) @ E) / np.sqrt(dk)
        S = np.exp(g[-1]) * S + E.T @ (Gam[-1][:, None] * K)
    return o, S
