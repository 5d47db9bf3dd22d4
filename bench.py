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


def load_traffic(kernel: str):
    """dram read+write bytes per launch from a committed ncu summary, if its source hash still matches."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"{kernel}.md")
    src = os.path.join(ROOT, "gated_deltanet_linear_conv1d_gb300", "csrc", "decode.cu")
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

    # ---- device-timed region: exactly K steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(dev)
    torch.cuda.synchronize()
    w0 = time.time()
    t_all0 = torch.cuda.Event(enable_timing=True)
    t_all1 = torch.cuda.Event(enable_timing=True)
    t_all0.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        step(d["qkv0"], d["alpha"], d["beta"], d["z"], d["slot_idx"], og)
        ends[i].record(stream)
    t_all1.record(stream)
    torch.cuda.synchronize()
    barrier(dev)
    w1 = time.time()
    total_ms = t_all0.elapsed_time(t_all1)
    kernel_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    if b.gdn_read_device_error(err) != 0:
        raise RuntimeError("device error flagged during the timed steps")
    max_ms = reduce_max(total_ms, dev)
    value = world * N * args.steps / (max_ms / 1e3)

    # ---- end-to-end through the C ABI: pinned host inputs in, Ogate out, every step
    host = {k: d[k].cpu().pin_memory() for k in ("qkv0", "alpha", "beta", "z", "slot_idx")}
    og_host = torch.empty(og.shape, dtype=og.dtype).pin_memory()
    staged = {k: torch.empty_like(d[k]) for k in host}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = og_host.numel() * og_host.element_size()

    def e2e_step():
        for k, t in host.items():
            staged[k].copy_(t, non_blocking=True)
        step(staged["qkv0"], staged["alpha"], staged["beta"], staged["z"], staged["slot_idx"], og)
        og_host.copy_(og, non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    barrier(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
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
    mean_kernel_ms = sum(kernel_ms) / len(kernel_ms)
    achieved = bytes_launch / (mean_kernel_ms / 1e3) / 1e9
    traffic = load_traffic("decode_step_256x48")
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": traffic, "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                if peak_kind == "measured" else "fallback 6.8 TB/s",
                "kernel": "decode_kernel (gdn_decode_step)",
                "algorithmic_bytes_per_launch": bytes_launch, "mean_launch_ms": mean_kernel_ms}
    cpu = oracle_decode_rate(w, NUM_REQ, min_seconds=10.0, max_seconds=30.0)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": max_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "requests_per_rank": N, "slots_per_rank": NUM_SLOTS,
                       "l2": "no flush: 768 MiB of state touched per step, inputs larger than L2",
                       "parallelism": f"{world} independent replica(s), requests sharded by rank"},
            "roofline": roofline, "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": args.steps, "clocks": clocks}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gdn", "reference"], default="gdn")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
