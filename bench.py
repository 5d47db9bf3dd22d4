"""Benchmark of the GDN mixer core on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gdn|reference]

One step = one pass of the mixer core over one batch: the decode step of 256
requests (one token each) whose recurrent states and conv histories sit in a
512-slot pool, picked by a random permutation (16 key / 48 value heads,
dk = dv = 128, fp32 state). All of the path's steps run in that one fused
kernel: slot gather, conv + SiLU with history update, q/k L2 norm, the
gated-delta-rule step, gated RMSNorm, slot scatter.

`value` is device-timed (CUDA events on the launching stream, inputs resident
in HBM); `e2e` repeats the measurement through the same C-ABI call with the
step's inputs copied from pinned host memory and Ogate copied back inside the
timed region. The touched state (768 MiB per step) is far larger than L2, so no
extra L2 flush is needed between steps.

`--impl reference` times the fp64 CPU oracle (the correctness reference) on
the host cores on a bounded sample of the same workload.

Under torchrun (N > 1) every rank runs its own independent batch (the path
shards by request with no exchange): weak scaling, barrier + max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from gated_deltanet_linear_conv1d_gb300 import synth  # noqa: E402

METRIC = "GDN mixer tokens/s (decode, prefill) and % of HBM / tensor-pipe roofline"
UNIT = "tokens/s"
NUM_REQ, NUM_SLOTS = 256, 512
WORKLOAD = ("decode step: 256 requests x 1 token over a 512-slot pool (random permutation), "
            "16 key / 48 value heads, dk=dv=128, conv 4 taps, fp32 state, bf16 activations")
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------- algorithmic bytes

def decode_bytes_per_token(geom, write_o: bool = False) -> int:
    """HBM bytes one decode token must move: state read + write, conv history read + write,
    QKV0, z, alpha, beta, slot index and the bf16 outputs."""
    state = geom.num_v_heads * geom.head_v_dim * geom.head_k_dim * 4
    hist = geom.channels * (geom.conv_kernel - 1) * 2
    outs = geom.num_v_heads * geom.head_v_dim * 2 * (2 if write_o else 1)
    return (2 * state + 2 * hist + geom.channels * 2 + geom.num_v_heads * geom.head_v_dim * 2
            + geom.num_v_heads * 4 * 2 + 4 + outs)


def decode_bytes_per_launch(geom, n: int, write_o: bool = False) -> int:
    """Per-token bytes x tokens, plus the conv taps and the RMSNorm gain read once."""
    return n * decode_bytes_per_token(geom, write_o) + geom.channels * geom.conv_kernel * 4 + geom.head_v_dim * 4


# ---------------------------------------------------------------- host logic shared by ranks

def rank_seed(rank: int) -> int:
    return 1 + 1000 * rank


def reduce_max(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without torch.distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def load_peaks() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def load_bf16_peak() -> tuple[float, float, str]:
    """(burst, sustained) dense bf16 TFLOP/s of the GB300s, and where they came from."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            j = json.load(f)
        return float(j["bf16_tflops"]), float(j.get("bf16_tflops_sustained", j["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, "fallback"


# tf32 tensor rate relative to bf16 (nominal dense figures: 1.1 vs 2.25 PFLOP/s)
TF32_PER_BF16 = 1.1 / 2.25


def prefill_flops(geom, lengths) -> tuple[float, float]:
    """Tensor-core FLOPs (bf16, tf32) of the chunked prefill for these request lengths.

    Per 64-token chunk and value head: S0 K^T and S0 Q^T (bf16, 2 x 2*128*64*128),
    E^T = Y Tb^T (tf32, 2*128*64*64), E^T P^T (tf32, 2*128*64*64), the state update
    (tf32, 2*128*128*64); per key head [K;Q] K^T (bf16, 2*128*64*128). A partial last
    chunk is computed as a full one.
    """
    chunks = sum((int(L) + 63) // 64 for L in lengths)
    hv, hk = geom.num_v_heads, geom.num_k_heads
    bf16 = chunks * (hv * 2 * 2 * 128 * 64 * 128 + hk * 2 * 128 * 64 * 128)
    tf32 = chunks * hv * (2 * 2 * 128 * 64 * 64 + 2 * 128 * 128 * 64)
    return float(bf16), float(tf32)


def prefill_bytes(geom, lengths, has_init) -> float:
    """HBM bytes a prefill must move: per token QKV0, z, alpha, beta and Ogate; per request the
    state and conv history (read only when continuing a slot) and their write-back."""
    state = geom.num_v_heads * geom.head_v_dim * geom.head_k_dim * 4
    hist = geom.channels * (geom.conv_kernel - 1) * 2
    per_tok = geom.channels * 2 + 2 * geom.num_v_heads * geom.head_v_dim * 2 + geom.num_v_heads * 8
    total = sum(int(L) for L in lengths) * per_tok
    for L, init in zip(lengths, has_init):
        if int(L) > 0:
            total += (state + hist) * (2 if init else 1)
    return float(total + geom.channels * geom.conv_kernel * 4 + geom.head_v_dim * 4)


def load_traffic(summary: str, source: str):
    """dram read+write bytes per launch from a committed ncu summary, if the kernel source it was
    taken on (its sha256 prefix is recorded in the summary) is unchanged."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{summary}.md")
    src = os.path.join(ROOT, "gated_deltanet_linear_conv1d_gb300", "csrc", source)
    try:
        text = open(path).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if line.startswith("traffic_bytes_per_launch:") or line.startswith("source_sha256_16:"):
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("source_sha256_16") != digest or "traffic_bytes_per_launch" not in vals:
        return None
    return int(float(vals["traffic_bytes_per_launch"]))


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (SM clock, throttle reasons) taken while the GPU runs the timed steps."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float) -> dict:
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        inside = [r for r in rows if t0 - 0.25 <= r[0] <= t1 + 0.25]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi sample"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for _, p in inside if num(p[1]) is not None]
        smax = [num(p[2]) for _, p in inside if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in inside for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(inside),
                "window": "timed region +-0.25 s, GPU busy with the same steps"}


# ---------------------------------------------------------------- CPU oracle

def oracle_decode_rate(w: dict, requests: int, min_seconds: float, max_seconds: float) -> dict:
    """The fp64 oracle on `requests` decode tokens of the workload, repeated until min_seconds."""
    from oracle import oracle
    geom = w["dims"]
    req = np.arange(requests)
    slots = w["slot_idx"][req]
    state = np.ascontiguousarray(w["state"][slots])
    hist = np.ascontiguousarray(w["conv_hist"][slots])
    qsl = np.arange(requests + 1, dtype=np.int32)
    local = np.arange(requests, dtype=np.int32)
    args = (w["qkv0"][req], w["conv_w"], hist, state, qsl, local, w["alpha"][req], w["beta"][req], w["z"][req],
            w["gamma"], w["eps"])
    done, t0 = 0, time.perf_counter()
    while True:
        oracle.forward(geom, *args, inplace=True)
        done += requests
        el = time.perf_counter() - t0
        if el >= min_seconds or el >= max_seconds:
            break
    return {"value": done / el, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{requests} of the {NUM_REQ} decode requests, repeated {done // requests}x "
                      f"({el:.1f} s, fp64, OpenMP over (request, key head) units)"}


def run_reference(args):
    """--impl reference: the oracle as it stands, timed on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    geom = synth.FULL_HEADS
    w = synth.decode_workload(geom, NUM_REQ, NUM_SLOTS, seed=rank_seed(0))
    per_step = 16
    from oracle import oracle
    req = np.arange(per_step)
    slots = w["slot_idx"][req]
    state = np.ascontiguousarray(w["state"][slots])
    hist = np.ascontiguousarray(w["conv_hist"][slots])
    qsl = np.arange(per_step + 1, dtype=np.int32)
    local = np.arange(per_step, dtype=np.int32)
    call = (w["qkv0"][req], w["conv_w"], hist, state, qsl, local, w["alpha"][req], w["beta"][req], w["z"][req],
            w["gamma"], w["eps"])
    for _ in range(args.warmup):
        oracle.forward(geom, *call, inplace=True)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward(geom, *call, inplace=True)
    el = time.perf_counter() - t0
    value = per_step * args.steps / el
    cores = oracle.num_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample_per_step": f"{per_step} of {NUM_REQ} requests"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{per_step} decode requests per step (fp64 oracle, host cores)"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

def to_device(w: dict, dev) -> dict:
    """Device copies of a synthetic workload; bf16 bit patterns become torch.bfloat16."""
    import torch
    out = {}
    for k, v in w.items():
        if not isinstance(v, np.ndarray):
            continue
        if k in ("qkv0", "z", "conv_hist"):
            out[k] = torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16).to(dev)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v)).to(dev)
    return out


def device_workload(geom, num_slots, tokens, seed, dev) -> dict:
    """Benchmark-only inputs drawn on the device with the distributions of synth (QKV0, z ~ N(0,1)
    bf16; conv taps ~ N(0, 0.25); alpha = exp(-U(0.001, 0.1)); beta ~ U(0, 1); gamma = 1; state
    ~ N(0, 0.02); history ~ N(0, 1) bf16). Never compared with the oracle."""
    import torch
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    H, D, CH = geom.num_v_heads, geom.head_v_dim, geom.channels

    def randn(*shape, std=1.0, dtype=torch.float32):
        return (torch.randn(shape, generator=gen, device=dev) * std).to(dtype)

    u = torch.rand((tokens, H), generator=gen, device=dev) * (0.1 - 0.001) + 0.001
    return {
        "qkv0": randn(tokens, CH, dtype=torch.bfloat16),
        "z": randn(tokens, H, D, dtype=torch.bfloat16),
        "alpha": torch.exp(-u),
        "beta": torch.rand((tokens, H), generator=gen, device=dev),
        "conv_w": randn(CH, geom.conv_kernel, std=0.25),
        "gamma": torch.ones(D, device=dev),
        "state": randn(num_slots, H, D, geom.head_k_dim, std=0.02),
        "conv_hist": randn(num_slots, CH, geom.conv_kernel - 1, dtype=torch.bfloat16),
    }


def timed(fn, steps: int, warmup: int, stream) -> float:
    """Mean milliseconds of fn() over `steps` launches after `warmup`, CUDA events on `stream`."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def graph_ms(launch, count: int, reps: int, stream, dev) -> float:
    """Device milliseconds per launch of launch(i), i = 0 .. count-1, issued on the current stream:
    warmed up, captured once in a CUDA graph and the graph replayed `reps` times (CUDA events on `stream`
    around the replays). At decode sizes a kernel takes a few microseconds, less than the Python call
    that issues it, so a loop of calls from Python would time the host instead."""
    import torch
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(min(count, 4)):
            launch(i)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(count):
            launch(i)
    ms = timed(graph.replay, reps, 2, stream) / count
    del graph
    return ms


SWEEP_REQUESTS = (1, 8, 64, 256, 1024)
SWEEP_POOL_BYTES = 512 << 20  # >= 4x L2: a slot's state is evicted before the step that uses it again


def measure_decode_sweep(b, dev, stream, peak: float, max_reps: int = 200) -> dict:
    """Decode batch sweep: R in {1, 8, 64, 256, 1024} requests x 1 token at 16/48 and at the
    per-rank 4/12 head layout (the TP4 shard run on one GPU). The pool holds 2R slots or enough
    slots for 512 MiB of state, whichever is more, cut into disjoint sets of R slots that the
    steps take in turn, so every step reads states that left L2 long before (a step of R = 1 at
    4/12 heads touches only 1.5 MiB). The steps are captured in a CUDA graph (64 launches, each
    on its own slot set) and the graph is replayed: at small R a launch takes a few
    microseconds, less than the Python call that issues it, so launches from Python would time
    the host. Each point: ms per launch from CUDA events around the replays on the launching
    stream, tokens/s, and the fraction of the measured copy bandwidth that the point's own
    algorithmic bytes reach."""
    import torch
    out = {}
    per_graph = 64
    for name, geom in (("16x48", synth.FULL_HEADS), ("4x12", synth.RANK_HEADS)):
        slot_bytes = geom.num_v_heads * geom.head_v_dim * geom.head_k_dim * 4
        for R in SWEEP_REQUESTS:
            Rs = max(2 * R, -(-SWEEP_POOL_BYTES // slot_bytes))
            sets = Rs // R
            d = device_workload(geom, Rs, R, seed=900 + R, dev=dev)
            gen = torch.Generator(device="cpu")
            gen.manual_seed(R)
            perm = torch.randperm(Rs, generator=gen)[: sets * R].to(torch.int32).view(sets, R).to(dev)
            D = b.make_dims(geom, Rs)
            og = torch.empty((R, geom.num_v_heads * geom.head_v_dim), dtype=torch.bfloat16, device=dev)
            err = torch.zeros(1, dtype=torch.int32, device=dev)

            def launch(i):  # on the current stream (the capture stream while capturing)
                b.gdn_decode_step(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], perm[i % sets],
                                  d["alpha"], d["beta"], d["z"], d["gamma"], 1e-6, ogate=og, dev_err=err)

            side = torch.cuda.Stream(device=dev)
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                for i in range(3):
                    launch(i)
            stream.wait_stream(side)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(per_graph):
                    launch(i)
            probe = timed(graph.replay, 2, 2, stream) / per_graph
            reps = int(min(max_reps, max(3, 80.0 / max(probe * per_graph, 1e-3))))
            ms = timed(graph.replay, reps, 2, stream) / per_graph
            if b.gdn_read_device_error(err) != 0:
                raise RuntimeError(f"device error flagged in the decode sweep ({name}, R={R})")
            nbytes = decode_bytes_per_launch(geom, R)
            out[f"{name}_R{R}"] = {"requests": R, "slots": Rs, "slot_sets": sets, "launches": reps * per_graph,
                                   "ms_per_step": ms, "tokens_per_s": R / (ms / 1e3),
                                   "algorithmic_bytes": nbytes, "hbm_gbs": nbytes / (ms / 1e3) / 1e9,
                                   "hbm_frac": nbytes / (ms / 1e3) / 1e9 / peak}
            del graph, d, perm, og
            torch.cuda.empty_cache()
    return out


def measure_prefill_single(b, dev, stream, launches: int = 64, reps: int = 50) -> dict:
    """The smallest prefill: one request of 64 tokens from a zero state (16/48 heads), the full mixer
    (conv, L2 norms, one 64-token chunk on the tensor cores, gated RMSNorm). Launch-bound, so the
    launches are captured in a CUDA graph (each on its own slot of a pool larger than L2) and the
    graph is replayed; ms per launch from CUDA events around the replays."""
    import torch
    geom = synth.FULL_HEADS
    T = 64
    slot_bytes = geom.num_v_heads * geom.head_v_dim * geom.head_k_dim * 4
    Rs = max(launches, -(-SWEEP_POOL_BYTES // slot_bytes))
    w = device_workload(geom, Rs, T, seed=0, dev=dev)
    qsl = torch.tensor([0, T], dtype=torch.int32, device=dev)
    zero = torch.zeros(1, dtype=torch.uint8, device=dev)
    slots = torch.arange(Rs, dtype=torch.int32, device=dev).view(Rs, 1)
    og = torch.empty((T, geom.num_v_heads * geom.head_v_dim), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    D = b.make_dims(geom, Rs)
    ws = torch.empty(b.gdn_prefill_workspace_bytes(D, 1, T), dtype=torch.uint8, device=dev)

    def launch(i):
        b.gdn_chunk_prefill(D, w["qkv0"], w["conv_w"], w["conv_hist"], w["state"], qsl, slots[i % Rs], w["alpha"],
                            w["beta"], w["z"], w["gamma"], 1e-6, ogate=og, has_init=zero, workspace=ws, dev_err=err)

    side = torch.cuda.Stream(device=dev)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for i in range(3):
            launch(i)
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(launches):
            launch(i)
    ms = timed(graph.replay, reps, 2, stream) / launches
    if b.gdn_read_device_error(err) != 0:
        raise RuntimeError("device error flagged during the single-request prefill measurement")
    return {"workload": "1 request x 64 tokens from a zero state, 16/48 heads (the smallest prefill)",
            "kernels": "prefill_order_kernel + prefill_tc_kernel (48 CTAs, one chunk each)",
            "ms_per_step": ms, "tokens_per_s": T / (ms / 1e3), "launches": launches * reps}


def measure_prefill(b, dev, stream, steps: int = 5, warmup: int = 2) -> dict:
    """Varlen chunked prefill: 64 requests, log-uniform lengths in [16, 8192], half from zero."""
    import torch
    geom = synth.FULL_HEADS
    lengths = synth.loguniform_lengths(np.random.default_rng(3), 64, 16, 8192)
    N, T = len(lengths), int(lengths.sum())
    Rs = 2 * N
    w = device_workload(geom, Rs, T, seed=3, dev=dev)
    slots = torch.from_numpy(synth.slot_permutation(np.random.default_rng(3), N, Rs)).to(dev)
    qsl = torch.from_numpy(synth.pack_offsets(lengths)).to(dev)
    has_init = np.ones(N, np.uint8)
    has_init[: N // 2] = 0
    hi = torch.from_numpy(has_init).to(dev)
    og = torch.empty((T, geom.num_v_heads * geom.head_v_dim), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    D = b.make_dims(geom, Rs)
    ws = torch.empty(b.gdn_prefill_workspace_bytes(D, N, T), dtype=torch.uint8, device=dev)

    def run():
        b.gdn_chunk_prefill(D, w["qkv0"], w["conv_w"], w["conv_hist"], w["state"], qsl, slots, w["alpha"],
                            w["beta"], w["z"], w["gamma"], 1e-6, ogate=og, has_init=hi, workspace=ws, dev_err=err,
                            stream=stream)

    ms = timed(run, steps, warmup, stream)
    if b.gdn_read_device_error(err) != 0:
        raise RuntimeError("device error flagged during the prefill measurement")
    f_bf16, f_tf32 = prefill_flops(geom, lengths)
    # align mode: the same batch with a state + history snapshot after every 512 tokens of each request
    block = 512
    nsnap = lengths // block
    max_snaps = int(nsnap.max())
    del w
    torch.cuda.empty_cache()
    Rs2 = Rs + int(nsnap.sum())
    w2 = device_workload(geom, Rs2, T, seed=3, dev=dev)
    D2 = b.make_dims(geom, Rs2)
    snap = np.full((N, max(max_snaps, 1)), -1, np.int32)
    nxt = Rs
    for n in range(N):
        for k in range(int(nsnap[n])):
            snap[n, k] = nxt
            nxt += 1
    snap_d = torch.from_numpy(snap).to(dev)

    def run_align():
        b.gdn_chunk_prefill_align(D2, w2["qkv0"], w2["conv_w"], w2["conv_hist"], w2["state"], qsl, slots,
                                  w2["alpha"], w2["beta"], w2["z"], w2["gamma"], 1e-6, block, snap_slot=snap_d,
                                  ogate=og, has_init=hi, workspace=ws, dev_err=err, stream=stream)

    ms_align = timed(run_align, steps, warmup, stream)
    if b.gdn_read_device_error(err) != 0:
        raise RuntimeError("device error flagged during the align-mode prefill measurement")
    snap_bytes = int(nsnap.sum()) * geom.num_v_heads * geom.head_v_dim * geom.head_k_dim * 4
    del w2
    torch.cuda.empty_cache()
    p_bf16, _, kind = load_bf16_peak()
    p_tf32 = p_bf16 * TF32_PER_BF16
    t_peak = f_bf16 / (p_bf16 * 1e12) + f_tf32 / (p_tf32 * 1e12)
    hbm_peak, hbm_kind = load_peaks()
    nbytes = prefill_bytes(geom, lengths, has_init)
    return {"workload": f"{N} requests, log-uniform lengths in [16, 8192] (seed 3), {T} tokens packed, "
                        f"half from a zero state; 16/48 heads; chunk 64",
            "value": T / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "steps": steps, "warmup": warmup,
            "kernel": "prefill_tc_kernel (gdn_chunk_prefill)",
            "tensor": {"achieved_tflops": (f_bf16 + f_tf32) / (ms / 1e3) / 1e12, "bf16_flops": f_bf16,
                       "tf32_flops": f_tf32, "peak_bf16_tflops": p_bf16, "peak_tf32_tflops": p_tf32,
                       "frac": t_peak / (ms / 1e3),
                       "peak_kind": f"{kind} bf16 burst; tf32 = bf16 x 1.1/2.25 (nominal ratio)"},
            "hbm": {"achieved_gbs": nbytes / (ms / 1e3) / 1e9, "algorithmic_bytes": nbytes, "peak": hbm_peak,
                    "frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak, "peak_kind": hbm_kind},
            "align_mode": {"block_tokens": block, "snapshots": int(nsnap.sum()), "snapshot_state_bytes": snap_bytes,
                           "ms_per_step": ms_align, "value": T / (ms_align / 1e3),
                           "overhead_vs_plain": ms_align / ms - 1.0}}


def measure_spec_mixed(b, dev, stream, steps: int = 5, warmup: int = 2) -> dict:
    """One mixed step: speculative verify of 256 requests x 4 positions with per-position
    checkpoints, commit (copy) at accepted lengths U{0..3}, and a prefill of 8 x 2048 tokens."""
    import torch
    geom = synth.FULL_HEADS
    N, P = 256, 4
    Rs = N * (P + 1)
    w = device_workload(geom, Rs, N * P, seed=4, dev=dev)
    rng = np.random.default_rng(4)
    perm = rng.permutation(Rs).astype(np.int32)
    slots = torch.from_numpy(perm[:N].copy()).to(dev)
    spec = torch.from_numpy(perm[N:].reshape(N, P).copy()).to(dev)
    acc = torch.from_numpy(rng.integers(0, P, size=N).astype(np.int32)).to(dev)
    og = torch.empty((N * P, geom.num_v_heads * geom.head_v_dim), dtype=torch.bfloat16, device=dev)
    lengths = np.full(8, 2048, np.int32)
    wp = device_workload(geom, 16, int(lengths.sum()), seed=5, dev=dev)
    pslots = torch.arange(8, dtype=torch.int32, device=dev)
    pqsl = torch.from_numpy(synth.pack_offsets(lengths)).to(dev)
    pog = torch.empty((int(lengths.sum()), geom.num_v_heads * geom.head_v_dim), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    D, Dp = b.make_dims(geom, Rs), b.make_dims(geom, 16)
    pws = torch.empty(b.gdn_prefill_workspace_bytes(Dp, 8, int(lengths.sum())), dtype=torch.uint8, device=dev)

    def spec_only():
        b.gdn_spec_verify(D, w["qkv0"], w["conv_w"], w["conv_hist"], w["state"], slots, spec, w["alpha"],
                          w["beta"], w["z"], w["gamma"], 1e-6, ogate=og, dev_err=err, stream=stream)
        b.gdn_spec_commit(D, acc, spec, slots, w["state"], w["conv_hist"], mode=b.GDN_COMMIT_COPY, dev_err=err,
                          stream=stream)

    def mixed():
        spec_only()
        b.gdn_chunk_prefill(Dp, wp["qkv0"], wp["conv_w"], wp["conv_hist"], wp["state"], pqsl, pslots,
                            wp["alpha"], wp["beta"], wp["z"], wp["gamma"], 1e-6, ogate=pog, workspace=pws,
                            dev_err=err, stream=stream)

    side = torch.cuda.Stream(device=dev)
    fork, join = torch.cuda.Event(), torch.cuda.Event()

    def mixed_two_streams():
        # the prefill on a second stream, so its CTAs can take the SMs the verify leaves idle and vice versa
        fork.record(stream)
        side.wait_event(fork)
        spec_only()
        b.gdn_chunk_prefill(Dp, wp["qkv0"], wp["conv_w"], wp["conv_hist"], wp["state"], pqsl, pslots,
                            wp["alpha"], wp["beta"], wp["z"], wp["gamma"], 1e-6, ogate=pog, workspace=pws,
                            dev_err=err, stream=side)
        join.record(side)
        stream.wait_event(join)

    ms_spec = timed(spec_only, steps, warmup, stream)
    ms_mixed = timed(mixed, steps, warmup, stream)
    ms_two = timed(mixed_two_streams, steps, warmup, stream)
    if b.gdn_read_device_error(err) != 0:
        raise RuntimeError("device error flagged during the speculative-verify measurement")
    state = geom.num_v_heads * geom.head_v_dim * geom.head_k_dim * 4
    hist = geom.channels * (geom.conv_kernel - 1) * 2
    act = geom.channels * 2 + 2 * geom.num_v_heads * geom.head_v_dim * 2 + geom.num_v_heads * 8
    spec_bytes = N * ((state + hist) * (1 + P) + P * act + 2 * (state + hist))  # verify + commit copy
    hbm_peak, _ = load_peaks()
    return {"workload": "A: 256 requests x 4 positions (last sampled token + 3 drafts), a state and history "
                        "checkpoint per position, commit by copy at accepted U{0..3}; B: prefill 8 x 2048 tokens",
            "spec_value": N * P / (ms_spec / 1e3), "unit": "verified tokens/s", "spec_ms": ms_spec,
            "spec_hbm_gbs": spec_bytes / (ms_spec / 1e3) / 1e9, "spec_hbm_frac": spec_bytes / (ms_spec / 1e3) / 1e9 / hbm_peak,
            "mixed_ms": ms_mixed, "mixed_tokens_per_s": (N * P + int(lengths.sum())) / (ms_mixed / 1e3),
            "mixed_two_streams_ms": ms_two,
            "mixed_two_streams_tokens_per_s": (N * P + int(lengths.sum())) / (ms_two / 1e3)}


def measure_conv(b, dev, stream, steps: int = 10, warmup: int = 3) -> dict:
    """Standalone varlen conv + SiLU with the history update, on the prefill batch's packing."""
    import torch
    geom = synth.FULL_HEADS
    lengths = synth.loguniform_lengths(np.random.default_rng(3), 64, 16, 8192)
    N, T = len(lengths), int(lengths.sum())
    w = device_workload(geom, 2 * N, T, seed=3, dev=dev)
    slots = torch.from_numpy(synth.slot_permutation(np.random.default_rng(3), N, 2 * N)).to(dev)
    qsl = torch.from_numpy(synth.pack_offsets(lengths)).to(dev)
    y = torch.empty((T, geom.channels), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    D = b.make_dims(geom, 2 * N)

    def run():
        b.gdn_conv_update(D, w["qkv0"], w["conv_w"], w["conv_hist"], qsl, slots, y, dev_err=err, stream=stream)

    ms = timed(run, steps, warmup, stream)
    if b.gdn_read_device_error(err) != 0:
        raise RuntimeError("device error flagged during the conv measurement")
    hist = geom.channels * (geom.conv_kernel - 1) * 2
    nbytes = T * geom.channels * 4 + N * 2 * hist + geom.channels * geom.conv_kernel * 4
    hbm_peak, hbm_kind = load_peaks()
    return {"workload": f"{N} requests, log-uniform lengths in [16, 8192] (seed 3), {T} tokens, 10240 channels",
            "kernel": "conv_kernel (gdn_conv_update)", "value": T / (ms / 1e3), "unit": UNIT, "ms_per_step": ms,
            "hbm": {"achieved_gbs": nbytes / (ms / 1e3) / 1e9, "algorithmic_bytes": nbytes, "peak": hbm_peak,
                    "frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak, "peak_kind": hbm_kind}}


def measure_out_proj(b, dev, stream) -> dict:
    """Wo projection + residual add (6144 -> 5120, bf16, the library's tcgen05 GEMM) at the decode batch (weight-streaming:
    four distinct weight matrices in rotation, 252 MB, so no step finds its weights in L2) and at the
    prefill batch's token count (tensor-bound)."""
    import torch
    K, N = 6144, 5120
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    weights = [(torch.randn((N, K), generator=g, device=dev) / K ** 0.5).to(torch.bfloat16) for _ in range(4)]
    res = {}
    p_bf16, _, kind = load_bf16_peak()
    hbm_peak, hbm_kind = load_peaks()
    for name, T, steps in (("decode", NUM_REQ, 40), ("prefill", 71068, 5)):
        a = torch.randn((T, K), generator=g, device=dev).to(torch.bfloat16)
        hidden = torch.randn((T, N), generator=g, device=dev).to(torch.bfloat16)
        it = [0]

        def run():
            b.gdn_out_proj(a, weights[it[0] % 4], hidden, residual=hidden, stream=stream)
            it[0] += 1

        ms = timed(run, steps, 4, stream)
        extra = {}
        if name == "decode":  # device time per launch (graph replays); `eager_ms` is the loop of Python calls
            extra["eager_ms"] = ms
            ms = graph_ms(lambda i: b.gdn_out_proj(a, weights[i % 4], hidden, residual=hidden), 16, 30, stream, dev)
        flops = 2.0 * T * K * N
        nbytes = N * K * 2 + T * K * 2 + 2 * T * N * 2
        res[name] = {"tokens": T, "ms": ms, "tflops": flops / (ms / 1e3) / 1e12,
                     "tensor_frac": flops / (ms / 1e3) / 1e12 / p_bf16,
                     "hbm_gbs": nbytes / (ms / 1e3) / 1e9, "hbm_frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak, **extra}
        del a, hidden
    return {"workload": "out = Ogate Wo^T + residual, K=6144 -> N=5120, bf16 in/out, fp32 accumulation",
            "kernel": "gemm_bf16_kernel (gdn_out_proj): at the decode batch swapped 128-weight-row x 256-token "
                      "tiles, K split 3 ways over clusters; at the prefill batch 128 x 256 tiles on persistent CTAs",
            "peak_bf16_tflops": p_bf16, "peak_kind": f"{kind} bf16 burst",
            "hbm_peak_gbs": hbm_peak, **res}


def measure_gate_wo(b, dev, stream) -> dict:
    """Where the gated RMSNorm in front of Wo runs. Two forms of the same work (mixer, gate, Wo with the
    residual add), timed back to back on one stream at the decode batch (256 requests of the 512-slot
    pool) and on the varlen prefill batch (71,068 tokens):
      fused:    the mixer kernel applies RMSNorm(o) * gamma * SiLU(z) to o in registers and writes Ogate;
                the Wo GEMM reads Ogate.
      separate: the mixer writes o only; the standalone gated RMSNorm reads o and z and writes Ogate;
                the Wo GEMM reads Ogate.
    Both move the same z bytes; the separate form adds the o round trip (12 KB per token written and read
    back) and a launch. `mixer_*_ms` are the mixer kernel alone in each output mode (the fused gate's
    cost inside the mixer)."""
    import torch
    geom = synth.FULL_HEADS
    H, Dv = geom.num_v_heads, geom.head_v_dim
    K, Nout = H * Dv, 5120
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    wo = (torch.randn((Nout, K), generator=g, device=dev) / K ** 0.5).to(torch.bfloat16)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    res = {}

    def measure(name, T, mixer, z, gamma, steps, warmup):
        og = torch.empty((T, K), dtype=torch.bfloat16, device=dev)
        o = torch.empty((T, H, Dv), dtype=torch.bfloat16, device=dev)
        hidden = torch.randn((T, Nout), generator=g, device=dev).to(torch.bfloat16)

        def fused():
            mixer(None, og)
            b.gdn_out_proj(og, wo, hidden, residual=hidden, dev_err=err, stream=stream)

        def separate():
            mixer(o, None)
            b.gdn_gated_rmsnorm(o, z, gamma, 1e-6, og, stream=stream)
            b.gdn_out_proj(og, wo, hidden, residual=hidden, dev_err=err, stream=stream)

        r = {"tokens": T,
             "fused_ms": timed(fused, steps, warmup, stream),
             "separate_ms": timed(separate, steps, warmup, stream),
             "mixer_ogate_ms": timed(lambda: mixer(None, og), steps, warmup, stream),
             "mixer_o_only_ms": timed(lambda: mixer(o, None), steps, warmup, stream)}
        r["separate_over_fused"] = r["separate_ms"] / r["fused_ms"]
        if b.gdn_read_device_error(err) != 0:
            raise RuntimeError(f"device error flagged during the gate + Wo measurement ({name})")
        res[name] = r
        del og, o, hidden

    # decode: 256 requests over a 512-slot pool (the headline step)
    d = device_workload(geom, NUM_SLOTS, NUM_REQ, seed=12, dev=dev)
    slots = torch.from_numpy(synth.slot_permutation(np.random.default_rng(12), NUM_REQ, NUM_SLOTS)).to(dev)
    D = b.make_dims(geom, NUM_SLOTS)

    def decode_mixer(o, og):
        b.gdn_decode_step(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], slots, d["alpha"], d["beta"],
                          d["z"], d["gamma"], 1e-6, o=o, ogate=og, dev_err=err, stream=stream)
    measure("decode", NUM_REQ, decode_mixer, d["z"], d["gamma"], 40, 5)
    del d
    torch.cuda.empty_cache()

    # prefill: the varlen batch of the prefill measurement
    lengths = synth.loguniform_lengths(np.random.default_rng(3), 64, 16, 8192)
    N, T = len(lengths), int(lengths.sum())
    Rs = 2 * N
    w = device_workload(geom, Rs, T, seed=3, dev=dev)
    pslots = torch.from_numpy(synth.slot_permutation(np.random.default_rng(3), N, Rs)).to(dev)
    qsl = torch.from_numpy(synth.pack_offsets(lengths)).to(dev)
    has_init = np.ones(N, np.uint8)
    has_init[: N // 2] = 0
    hi = torch.from_numpy(has_init).to(dev)
    Dp = b.make_dims(geom, Rs)
    ws = torch.empty(b.gdn_prefill_workspace_bytes(Dp, N, T), dtype=torch.uint8, device=dev)

    def prefill_mixer(o, og):
        b.gdn_chunk_prefill(Dp, w["qkv0"], w["conv_w"], w["conv_hist"], w["state"], qsl, pslots, w["alpha"],
                            w["beta"], w["z"] if og is not None else None, w["gamma"], 1e-6, o=o, ogate=og,
                            has_init=hi, workspace=ws, dev_err=err, stream=stream)
    measure("prefill", T, prefill_mixer, w["z"], w["gamma"], 5, 2)
    del w
    torch.cuda.empty_cache()
    return {"workload": "mixer (decode step of 256 requests / varlen prefill of 71,068 tokens) + gated RMSNorm + "
                        "Wo 6144 -> 5120 with the residual added in place, bf16",
            "forms": "fused = mixer writes Ogate (gate in its epilogue), then Wo; separate = mixer writes o, "
                     "gdn_gated_rmsnorm, then Wo",
            **res}


def measure_in_proj(b, dev, stream, geom, D) -> dict:
    """The in_proj rows (hidden 5120 -> QKV0 10240, Z 6144, a|b 96 fp32; one launch of the tcgen05 GEMM) at the
    decode batch (weight-streaming: two weight sets in rotation, 338 MB, so no step finds its weights in
    L2) and at the prefill batch's token count (tensor-bound)."""
    import torch
    Dh = 5120
    CH, NZ, NAB = geom.channels, geom.num_v_heads * geom.head_v_dim, 2 * geom.num_v_heads
    g = torch.Generator(device=dev)
    g.manual_seed(6)
    sets = [[(torch.randn((n, Dh), generator=g, device=dev) / Dh ** 0.5).to(torch.bfloat16) for n in (CH, NZ, NAB)]
            for _ in range(2)]
    res = {}
    p_bf16, _, kind = load_bf16_peak()
    hbm_peak, _ = load_peaks()
    for name, T, steps in (("decode", NUM_REQ, 40), ("prefill", 71068, 5)):
        u = torch.randn((T, Dh), generator=g, device=dev).to(torch.bfloat16)
        qkv0 = torch.empty((T, CH), dtype=torch.bfloat16, device=dev)
        z = torch.empty((T, NZ), dtype=torch.bfloat16, device=dev)
        ab = torch.empty((T, NAB), dtype=torch.float32, device=dev)
        it = [0]

        def run():
            wq, wz, wab = sets[it[0] % 2]
            b.gdn_in_proj(D, u, wq, wz, qkv0, z, w_ab=wab, ab=ab, stream=stream)
            it[0] += 1

        ms = timed(run, steps, 4, stream)
        extra = {}
        if name == "decode":  # device time per launch (graph replays); `eager_ms` is the loop of Python calls
            extra["eager_ms"] = ms

            def launch(i):
                wq, wz, wab = sets[i % 2]
                b.gdn_in_proj(D, u, wq, wz, qkv0, z, w_ab=wab, ab=ab)
            ms = graph_ms(launch, 16, 30, stream, dev)
        flops = 2.0 * T * Dh * (CH + NZ + NAB)
        # weights once, the hidden rows once, the outputs once
        nbytes = (CH + NZ + NAB) * Dh * 2 + T * Dh * 2 + T * (CH + NZ) * 2 + T * NAB * 4
        res[name] = {"tokens": T, "ms": ms, "tflops": flops / (ms / 1e3) / 1e12,
                     "tensor_frac": flops / (ms / 1e3) / 1e12 / p_bf16,
                     "hbm_gbs": nbytes / (ms / 1e3) / 1e9, "hbm_frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak, **extra}
        del u, qkv0, z, ab
    return {"workload": "QKV0 = U Wqkv^T, Z = U Wz^T, [a|b] = U Wab^T, 5120 -> 10240 / 6144 / 96, bf16 in, "
                        "bf16 / bf16 / fp32 out, fp32 accumulation",
            "kernel": "gemm_bf16_kernel (gdn_in_proj, the three outputs in one launch)", "peak_bf16_tflops": p_bf16, "peak_kind": f"{kind} bf16 burst",
            "hbm_peak_gbs": hbm_peak, **res}


def measure_fp8_proj(b, dev, stream) -> dict:
    """The projections with FP8 E4M3 block-scaled weights (one scale per 128 x 128 block) and activations
    quantised per token and 128-wide group: Wo (6144 -> 5120) and the QKV + Z rows of in_proj
    (5120 -> 10240 + 6144), each as activation quantisation + the tcgen05 GEMM, at the decode batch
    (weight sets in rotation past L2) and at the prefill batch's token count."""
    import torch
    p_bf16, _, kind = load_bf16_peak()
    p_fp8 = 2.0 * p_bf16  # nominal dense fp8 rate is twice bf16 on this part
    hbm_peak, _ = load_peaks()
    g = torch.Generator(device=dev)
    g.manual_seed(8)
    res = {}
    for proj, K, Ns in (("wo", 6144, (5120,)), ("in_proj", 5120, (10240, 6144))):
        wbytes = sum(Ns) * K
        nsets = max(2, -(-(192 << 20) // wbytes))
        sets = []
        for _ in range(nsets):
            one = []
            for N in Ns:
                w = (torch.randn((N, K), generator=g, device=dev) / K ** 0.5).to(torch.bfloat16)
                w8 = torch.empty((N, K), dtype=torch.uint8, device=dev)
                ws = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=dev)
                b.gdn_fp8_quant_weight(w, w8, ws, stream=stream)
                one.append((w8, ws))
                del w
            sets.append(one)
        for name, T, steps in (("decode", NUM_REQ, 40), ("prefill", 71068, 5)):
            x = torch.randn((T, K), generator=g, device=dev).to(torch.bfloat16)
            x8 = torch.empty((T, K), dtype=torch.uint8, device=dev)
            xs = torch.empty((T, K // 128), dtype=torch.float32, device=dev)
            outs = [torch.empty((T, N), dtype=torch.bfloat16, device=dev) for N in Ns]
            wsps = [torch.zeros(max(256, b.gdn_fp8_linear_workspace_bytes(T, K, N)), dtype=torch.uint8, device=dev)
                    for N in Ns]
            it = [0]

            def gemms():
                for (w8, ws), out, wsp in zip(sets[it[0] % nsets], outs, wsps):
                    b.gdn_fp8_linear(x8, xs, w8, ws, out, workspace=wsp, stream=stream)
                it[0] += 1

            def run():
                b.gdn_fp8_quant_act(x, x8, xs, stream=stream)
                gemms()

            ms = timed(run, steps, 4, stream)
            ms_gemm = timed(gemms, steps, 4, stream)
            extra = {}
            if name == "decode":  # device time per step (graph replays); `eager_*` are loops of Python calls
                extra = {"eager_ms": ms, "eager_gemm_ms": ms_gemm}

                def gemms_i(i):
                    for (w8, ws), out, wsp in zip(sets[i % nsets], outs, wsps):
                        b.gdn_fp8_linear(x8, xs, w8, ws, out, workspace=wsp)

                def run_i(i):
                    b.gdn_fp8_quant_act(x, x8, xs)
                    gemms_i(i)
                ms = graph_ms(run_i, 16, 30, stream, dev)
                ms_gemm = graph_ms(gemms_i, 16, 30, stream, dev)
            flops = 2.0 * T * K * sum(Ns)
            nbytes = wbytes + T * K * len(Ns) + T * sum(Ns) * 2
            res[f"{proj}_{name}"] = {"tokens": T, "ms": ms, "gemm_ms": ms_gemm, **extra,
                                     "gemm_tflops": flops / (ms_gemm / 1e3) / 1e12,
                                     "gemm_tensor_frac_of_fp8": flops / (ms_gemm / 1e3) / 1e12 / p_fp8,
                                     "gemm_hbm_frac": nbytes / (ms_gemm / 1e3) / 1e9 / hbm_peak}
            del x, x8, xs, outs, wsps
        del sets
        torch.cuda.empty_cache()
    return {"workload": "E4M3 weights, one fp32 scale per 128x128 block; activations quantised per token and "
                        "128-wide group (gdn_fp8_quant_act) then gdn_fp8_linear; ms = quantise + GEMM(s)",
            "kernel": "fp8_gemm_wide_kernel (128 x 256 tiles per CTA; at prefill token counts persistent CTA "
                      "pairs issuing cta_group::2 MMAs of 256 x 256, at decode token counts each tile's K blocks "
                      "split over a cluster): tcgen05 kind::f8f6f4, per-block promotion in registers",
            "peak_fp8_tflops": p_fp8, "peak_kind": f"2 x {kind} bf16 burst (nominal fp8/bf16 ratio)",
            "hbm_peak_gbs": hbm_peak, **res}


def measure_rmsnorm(b, dev, stream) -> dict:
    """The layer's input RMSNorm fused with the residual add (hidden 5120, bf16) at the decode batch and
    at the prefill batch's token count: reads x and the residual, writes the residual and U."""
    import torch
    Dh = 5120
    g = torch.Generator(device=dev)
    g.manual_seed(7)
    gamma = torch.rand(Dh, generator=g, device=dev) + 0.5
    hbm_peak, _ = load_peaks()
    res = {}
    for name, T, steps in (("decode", NUM_REQ, 40), ("prefill", 71068, 10)):
        # several independent buffer sets in rotation so that the decode batch's 10 MB does not stay in L2
        nset = max(1, (1 << 30) // (T * Dh * 2 * 3))
        sets = [[torch.randn((T, Dh), generator=g, device=dev).to(torch.bfloat16) for _ in range(3)]
                for _ in range(nset)]
        it = [0]

        def run():
            x, r, u = sets[it[0] % nset]
            b.gdn_rmsnorm(x, gamma, 1e-6, u, residual=r, stream=stream)
            it[0] += 1

        ms = timed(run, steps, 4, stream)
        extra = {}
        if name == "decode":  # device time per launch (graph replays); `eager_ms` is the loop of Python calls
            extra["eager_ms"] = ms

            def launch(i):
                x, r, u = sets[i % nset]
                b.gdn_rmsnorm(x, gamma, 1e-6, u, residual=r)
            ms = graph_ms(launch, 64, 30, stream, dev)
        nbytes = 4 * T * Dh * 2 + Dh * 4
        res[name] = {"tokens": T, "ms": ms, "hbm_gbs": nbytes / (ms / 1e3) / 1e9,
                     "hbm_frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak, **extra}
        del sets
    return {"workload": "residual <- x + residual; U = RMSNorm(residual) * gamma, hidden 5120, bf16",
            "kernel": "rmsnorm_kernel (gdn_rmsnorm)", "hbm_peak_gbs": hbm_peak, **res}


def measure_gated_rmsnorm(b, dev, stream) -> dict:
    """The gated RMSNorm on its own (Ogate = RMSNorm(o) * gamma * SiLU(z) per head, 48 heads x 128), for
    callers that take o and z from elsewhere; the mixer kernels fuse it. Decode batch and prefill batch."""
    import torch
    H, Dv = 48, 128
    g = torch.Generator(device=dev)
    g.manual_seed(9)
    gamma = torch.rand(Dv, generator=g, device=dev) + 0.5
    hbm_peak, _ = load_peaks()
    res = {}
    for name, T, steps in (("decode", NUM_REQ, 40), ("prefill", 71068, 10)):
        nset = max(1, (1 << 30) // (T * H * Dv * 2 * 3))
        sets = [[torch.randn((T, H, Dv), generator=g, device=dev).to(torch.bfloat16) for _ in range(2)]
                + [torch.empty((T, H * Dv), dtype=torch.bfloat16, device=dev)] for _ in range(nset)]
        it = [0]

        def run():
            o, z, out = sets[it[0] % nset]
            b.gdn_gated_rmsnorm(o, z, gamma, 1e-6, out, stream=stream)
            it[0] += 1

        ms = timed(run, steps, 4, stream)
        extra = {}
        if name == "decode":  # device time per launch (graph replays); `eager_ms` is the loop of Python calls
            extra["eager_ms"] = ms

            def launch(i):
                o, z, out = sets[i % nset]
                b.gdn_gated_rmsnorm(o, z, gamma, 1e-6, out)
            ms = graph_ms(launch, 64, 30, stream, dev)
        nbytes = 3 * T * H * Dv * 2 + Dv * 4
        res[name] = {"tokens": T, "ms": ms, "hbm_gbs": nbytes / (ms / 1e3) / 1e9,
                     "hbm_frac": nbytes / (ms / 1e3) / 1e9 / hbm_peak, **extra}
        del sets
    return {"workload": "Ogate = o / sqrt(mean(o^2) + eps) * gamma * SiLU(z), 48 heads x 128, bf16",
            "kernel": "gated_rmsnorm_kernel (gdn_gated_rmsnorm)", "hbm_peak_gbs": hbm_peak, **res}


def run_gpu(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from gated_deltanet_linear_conv1d_gb300 import build as gdn_build
    gdn_build.build()
    from gated_deltanet_linear_conv1d_gb300 import binding as b

    geom = synth.FULL_HEADS
    w = synth.decode_workload(geom, NUM_REQ, NUM_SLOTS, seed=rank_seed(rank))
    d = to_device(w, dev)
    D = b.make_dims(geom, NUM_SLOTS)
    N = NUM_REQ
    og = torch.empty((N, geom.num_v_heads * geom.head_v_dim), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream()

    def step(qkv0, alpha, beta, z, slot_idx, out):
        b.gdn_decode_step(D, qkv0, d["conv_w"], d["conv_hist"], d["state"], slot_idx, alpha, beta, z,
                          d["gamma"], w["eps"], ogate=out, dev_err=err, stream=stream)

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler:
        sampler.start()
    for _ in range(args.warmup):
        step(d["qkv0"], d["alpha"], d["beta"], d["z"], d["slot_idx"], og)
    torch.cuda.synchronize()

    # ---- device-timed region: exactly K steps, back to back (no events between them: the region
    # holds K launches of the decode kernel and nothing else, so its time over K is the kernel's
    # average launch duration, gaps between launches included)
    barrier(dev)
    torch.cuda.synchronize()
    w0 = time.time()
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    t_all0.record(stream)
    for _ in range(args.steps):
        step(d["qkv0"], d["alpha"], d["beta"], d["z"], d["slot_idx"], og)
    t_all1.record(stream)
    torch.cuda.synchronize()
    barrier(dev)
    w1 = time.time()
    total_ms = t_all0.elapsed_time(t_all1)
    if b.gdn_read_device_error(err) != 0:
        raise RuntimeError("device error flagged during the timed steps")
    max_ms = reduce_max(total_ms, dev)
    value = world * N * args.steps / (max_ms / 1e3)

    # ---- end-to-end through the C ABI: pinned host inputs in, Ogate out, every step. A serving loop
    # overlaps the transfers with the compute: step i+1's inputs go up on one copy stream and step
    # i-1's Ogate comes down on another while step i runs (two staging sets, two Ogate buffers).
    host = {k: d[k].cpu().pin_memory() for k in ("qkv0", "alpha", "beta", "z", "slot_idx")}
    og_host = torch.empty(og.shape, dtype=og.dtype).pin_memory()
    staged = [{k: torch.empty_like(d[k]) for k in host} for _ in range(2)]
    ogs = [torch.empty_like(og) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = og_host.numel() * og_host.element_size()
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]

    def upload(i):
        bi = i % 2
        up.wait_event(done[bi])  # step i-2 has consumed this staging set
        with torch.cuda.stream(up):
            for k, t in host.items():
                staged[bi][k].copy_(t, non_blocking=True)
        in_ready[bi].record(up)

    def run_steps(count):
        upload(0)
        for i in range(count):
            bi = i % 2
            if i + 1 < count:
                upload(i + 1)
            stream.wait_event(in_ready[bi])
            stream.wait_event(out_read[bi])  # step i-2's Ogate has been read back
            sb = staged[bi]
            step(sb["qkv0"], sb["alpha"], sb["beta"], sb["z"], sb["slot_idx"], ogs[bi])
            done[bi].record(stream)
            down.wait_event(done[bi])
            with torch.cuda.stream(down):
                og_host.copy_(ogs[bi], non_blocking=True)
            out_read[bi].record(down)
        for s_ in (up, down):
            stream.wait_stream(s_)

    run_steps(args.warmup)
    torch.cuda.synchronize()
    barrier(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_stream(stream)
    down.wait_stream(stream)
    run_steps(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(dev)
    e2e_ms = reduce_max(e0.elapsed_time(e1), dev)
    e2e_value = world * N * args.steps / (e2e_ms / 1e3)
    if sampler:
        sampler.stop()

    if rank != 0:
        return
    clocks = sampler.summary(w0, w1)
    peak, peak_kind = load_peaks()
    bytes_launch = decode_bytes_per_launch(geom, N)
    mean_kernel_ms = total_ms / args.steps
    achieved = bytes_launch / (mean_kernel_ms / 1e3) / 1e9
    traffic = load_traffic("stream_kernel_decode_256x48", "decode.cu")
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "kernel": "stream_kernel (gdn_decode_step)",
                "algorithmic_bytes_per_launch": bytes_launch, "mean_launch_ms": mean_kernel_ms,
                "launch_timing": "CUDA events around the K back-to-back launches of the timed region, / K"}
    cpu = oracle_decode_rate(w, NUM_REQ, min_seconds=10.0, max_seconds=30.0)
    del d
    torch.cuda.empty_cache()
    extra = {}
    if not args.decode_only:
        # graph replays per point: up to 200 for a full run, fewer for a short one
        extra["decode_sweep"] = measure_decode_sweep(b, dev, stream, peak, max_reps=max(3, min(200, args.steps // 5)))
        torch.cuda.empty_cache()
        extra["prefill"] = measure_prefill(b, dev, stream)
        torch.cuda.empty_cache()
        extra["prefill_single"] = measure_prefill_single(b, dev, stream)
        torch.cuda.empty_cache()
        extra["spec_mixed"] = measure_spec_mixed(b, dev, stream)
        torch.cuda.empty_cache()
        extra["conv"] = measure_conv(b, dev, stream)
        torch.cuda.empty_cache()
        extra["out_proj"] = measure_out_proj(b, dev, stream)
        extra["in_proj"] = measure_in_proj(b, dev, stream, geom, D)
        torch.cuda.empty_cache()
        extra["rmsnorm"] = measure_rmsnorm(b, dev, stream)
        torch.cuda.empty_cache()
        extra["gated_rmsnorm"] = measure_gated_rmsnorm(b, dev, stream)
        torch.cuda.empty_cache()
        extra["gate_wo"] = measure_gate_wo(b, dev, stream)
        torch.cuda.empty_cache()
        extra["fp8_proj"] = measure_fp8_proj(b, dev, stream)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "requests_per_rank": N, "slots_per_rank": NUM_SLOTS,
                       "l2": "no flush: 768 MiB of state touched per step, inputs larger than L2",
                       "parallelism": f"{world} independent replica(s), requests sharded by rank"},
            "roofline": roofline, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "transfers": "every step: its inputs up from pinned host memory, its Ogate down; step i+1's "
                                 "upload and step i-1's readback on two copy streams overlap step i"},
            "gpu_launches": args.steps, "clocks": clocks}
    line.update(extra)
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    ap.add_argument("--decode-only", action="store_true",
                    help="skip the prefill and speculative-verify lines (decode headline only)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
