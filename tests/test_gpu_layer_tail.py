"""The mixer's output through the Wo projection (page "Qwen3.8-27B: from model structure to
vLLM inference data flow", section 01 GDN operator table, the gate and Wo rows), on the GPU
against the oracle's out_proj(gated_rmsnorm(o, z)):

  fused:    the mixer entry point writes Ogate (the gate applied in the mixer kernel), then
            gdn_out_proj adds Ogate Wo^T to the residual stream in place;
  separate: the mixer writes o, gdn_gated_rmsnorm forms Ogate, then gdn_out_proj.

The oracle side runs the fp64 mixer, rounds its Ogate to bf16 (the tensor the two kernels
exchange) and multiplies in fp64. Decode (64 requests over a 128-slot pool) and a varlen
prefill that crosses chunk edges, at the layer's full sizes (6144 -> 5120)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

from gated_deltanet_linear_conv1d_gb300 import synth  # noqa: E402
from oracle import oracle  # noqa: E402
from tests import gdnutil as U  # noqa: E402

HIDDEN = 5120


@pytest.fixture(scope="module")
def b():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_linear_conv1d_gb300 import build
    build.build()
    from gated_deltanet_linear_conv1d_gb300 import binding
    return binding


def _weights(T, K, seed):
    rng = np.random.default_rng(seed)
    wo = synth.bf16_bits((rng.normal(size=(HIDDEN, K)) / np.sqrt(K)).astype(np.float32))
    res = synth.bf16_bits(rng.normal(size=(T, HIDDEN)).astype(np.float32))
    return wo, res


def _tail_both_ways(b, w, d, T, mixer):
    """Runs mixer + Wo in the fused and the separate form on copies of the slot pools;
    returns the two hidden outputs (device tensors)."""
    geom = w["dims"]
    K = geom.num_v_heads * geom.head_v_dim
    wo, res = _weights(T, K, 600 + T)
    wo_d = U.dev_bf16(wo)
    outs = []
    for fused in (True, False):
        state, hist = d["state"].clone(), d["conv_hist"].clone()
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        og = torch.empty((T, K), dtype=torch.bfloat16, device="cuda")
        if fused:
            mixer(state, hist, None, og, err)
        else:
            o = torch.empty((T, geom.num_v_heads, geom.head_v_dim), dtype=torch.bfloat16, device="cuda")
            mixer(state, hist, o, None, err)
            b.gdn_gated_rmsnorm(o, d["z"], d["gamma"], w["eps"], og)
        hidden = U.dev_bf16(res)
        b.gdn_out_proj(og, wo_d, hidden, residual=hidden, dev_err=err)
        assert b.gdn_read_device_error(err) == 0
        outs.append(hidden)
    return outs, wo, res


def _reference(w, requests, wo, res):
    r, toks = U.oracle_compact(w, requests)
    og_bits = synth.bf16_bits(r["ogate"].astype(np.float32))
    return oracle.out_proj(og_bits, wo, res[toks] if res is not None else None), toks


def test_decode_gate_then_wo_matches_oracle(b):
    geom = synth.FULL_HEADS
    R = 64
    w = synth.decode_workload(geom, R, 2 * R, seed=61)
    d = U.to_device(w)
    D = b.make_dims(geom, w["num_slots"])

    def mixer(state, hist, o, og, err):
        b.gdn_decode_step(D, d["qkv0"], d["conv_w"], hist, state, d["slot_idx"], d["alpha"], d["beta"], d["z"],
                          d["gamma"], w["eps"], o=o, ogate=og, dev_err=err)

    (fused, separate), wo, res = _tail_both_ways(b, w, d, R, mixer)
    ref, _ = _reference(w, np.arange(R), wo, res)
    U.check_out(U.host_f64_from_bf16(fused), ref, "decode: mixer with the gate, then Wo")
    U.check_out(U.host_f64_from_bf16(separate), ref, "decode: mixer, standalone gate, then Wo")


def test_prefill_gate_then_wo_matches_oracle(b):
    geom = synth.FULL_HEADS
    lengths = [70, 1, 130, 64, 3]
    w = synth.prefill_workload(geom, lengths, seed=62)
    d = U.to_device(w)
    D = b.make_dims(geom, w["num_slots"])
    T = int(sum(lengths))

    def mixer(state, hist, o, og, err):
        b.gdn_chunk_prefill(D, d["qkv0"], d["conv_w"], hist, state, d["query_start_loc"], d["slot_idx"],
                            d["alpha"], d["beta"], d["z"] if og is not None else None, d["gamma"], w["eps"],
                            o=o, ogate=og, has_init=d["has_init"], dev_err=err)

    (fused, separate), wo, res = _tail_both_ways(b, w, d, T, mixer)
    ref, _ = _reference(w, np.arange(len(lengths)), wo, res)
    U.check_out(U.host_f64_from_bf16(fused), ref, "prefill: mixer with the gate, then Wo")
    U.check_out(U.host_f64_from_bf16(separate), ref, "prefill: mixer, standalone gate, then Wo")
