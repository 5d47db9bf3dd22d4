"""Helpers shared by the GPU parity tests: host <-> device transfer of the synthetic
workloads, oracle runs on compacted slot pools, and the tolerance checks.

Tolerances (fixed by the acceptance criteria of the GDN mixer-core build):
conv history and slot gather/scatter bit-exact; o and Ogate (bf16) relative
L2 error <= 5e-3 and max-abs error <= 2e-2 * max|oracle|; final fp32 state
relative L2 error <= 1e-4 after decode / speculative verify and <= 2e-3 after
chunked prefill.
"""
import numpy as np
import torch

from gated_deltanet_linear_conv1d_gb300 import synth
from oracle import oracle

OUT_REL_L2 = 5e-3
OUT_MAX_ABS_FRAC = 2e-2
STATE_REL_L2_DECODE = 1e-4
STATE_REL_L2_PREFILL = 2e-3


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def host_f64_from_bf16(t: torch.Tensor) -> np.ndarray:
    return synth.bf16_to_f32(host_bits(t)).astype(np.float64)


def rel_l2(a, ref) -> float:
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(a - ref) / (den if den > 0 else 1.0))


def check_out(got, ref, what: str):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    e = rel_l2(got, ref)
    m = float(np.max(np.abs(got - ref))) if ref.size else 0.0
    bound = OUT_MAX_ABS_FRAC * float(np.max(np.abs(ref))) if ref.size else 0.0
    print(f"[parity] {what}: rel-L2 {e:.3e}, max-abs {m:.3e} (bound {bound:.3e})")
    assert e <= OUT_REL_L2, f"{what}: rel-L2 {e:.3e} > {OUT_REL_L2}"
    assert m <= bound, f"{what}: max-abs {m:.3e} > {bound:.3e}"
    return e, m


def check_state(got, ref, tol: float, what: str):
    e = rel_l2(got, ref)
    print(f"[parity] {what}: state rel-L2 {e:.3e} (tolerance {tol})")
    assert np.all(np.isfinite(got)), f"{what}: non-finite state"
    assert e <= tol, f"{what}: state rel-L2 {e:.3e} > {tol}"
    return e


def to_device(w: dict) -> dict:
    """Device copies of a synth workload (bf16 arrays as torch.bfloat16)."""
    d = {}
    for k in ("qkv0", "z", "conv_hist"):
        if k in w:
            d[k] = dev_bf16(w[k])
    for k in ("conv_w", "gamma", "alpha", "beta", "state", "slot_idx", "query_start_loc", "spec_slot_idx",
              "accepted", "has_init"):
        if k in w:
            d[k] = dev(w[k])
    return d


def oracle_compact(w: dict, requests, qsl=None, want_y=False):
    """Runs the oracle on the given requests only, with their slots gathered into a compact pool.

    Returns (result dict, token index array). Slot gather/scatter is exercised by
    the oracle on the compact pool; the GPU result is compared on the real pool.
    """
    requests = np.asarray(requests)
    dims = w["dims"]
    slots = w["slot_idx"][requests]
    if qsl is None:
        qsl = w.get("query_start_loc", np.arange(len(w["slot_idx"]) + 1, dtype=np.int32))
    toks = np.concatenate([np.arange(qsl[n], qsl[n + 1]) for n in requests]).astype(np.int64)
    lens = np.array([qsl[n + 1] - qsl[n] for n in requests], np.int32)
    sub_qsl = synth.pack_offsets(lens)
    st = np.ascontiguousarray(w["state"][slots])
    hist = np.ascontiguousarray(w["conv_hist"][slots])
    has_init = None if "has_init" not in w else np.ascontiguousarray(w["has_init"][requests])
    r = oracle.forward(dims, w["qkv0"][toks], w["conv_w"], hist, st, sub_qsl,
                       np.arange(len(requests), dtype=np.int32), w["alpha"][toks], w["beta"][toks],
                       w["z"][toks], w["gamma"], w["eps"], has_init=has_init, want_y=want_y, inplace=True)
    return r, toks


def oracle_spec_compact(w: dict, requests):
    """The oracle's speculative verify on the given requests only: their live slots and
    checkpoint slots are gathered into a compact pool (live slot of request i at i, its
    checkpoints at len(requests) + i * P + p). Returns the oracle's result dict with
    "state" / "conv_hist" holding only the checkpoint slots, [len(requests) * P, ...],
    in request-major order, and the token index array of the requests' positions."""
    requests = np.asarray(requests)
    dims = w["dims"]
    P = int(w["spec_slot_idx"].shape[1])
    R = len(requests)
    live = w["slot_idx"][requests]
    ck = w["spec_slot_idx"][requests].reshape(-1)
    st = np.ascontiguousarray(np.concatenate([w["state"][live], w["state"][ck]]))
    hist = np.ascontiguousarray(np.concatenate([w["conv_hist"][live], w["conv_hist"][ck]]))
    toks = (requests[:, None] * P + np.arange(P)[None, :]).reshape(-1)
    r = oracle.spec_verify(dims, w["qkv0"][toks], w["conv_w"], hist, st, np.arange(R, dtype=np.int32),
                           (R + np.arange(R * P, dtype=np.int32)).reshape(R, P), w["alpha"][toks],
                           w["beta"][toks], w["z"][toks], w["gamma"], w["eps"], inplace=True)
    r["state"] = r["state"][R:]
    r["conv_hist"] = r["conv_hist"][R:]
    return r, toks
