"""Runs one libgdn entry point a few times on a synthetic workload, for profilers.

    python -m gated_deltanet_linear_conv1d_gb300.profile_case decode  --requests 64 --slots 128 --launches 3
    python -m gated_deltanet_linear_conv1d_gb300.profile_case prefill --lengths 2048x8 --launches 2
    python -m gated_deltanet_linear_conv1d_gb300.profile_case spec    --requests 64 --launches 2
    python -m gated_deltanet_linear_conv1d_gb300.profile_case commit  --requests 256 --launches 3
    python -m gated_deltanet_linear_conv1d_gb300.profile_case fp8     --requests 4096 --k 6144 --n 5120
    python -m gated_deltanet_linear_conv1d_gb300.profile_case gemm    --requests 256 --k 6144 --n 5120

Each launch is preceded by the same warm-up launches (--warmup) and followed
by a device synchronisation; nothing else runs on the GPU besides the input
upload, so a profiler can select the kernel by name and skip the warm-ups.
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import synth


def _dev(w, dev):
    out = {}
    for k, v in w.items():
        if not isinstance(v, np.ndarray):
            continue
        if k in ("qkv0", "z", "conv_hist"):
            out[k] = torch.from_numpy(np.ascontiguousarray(v).view(np.int16)).view(torch.bfloat16).to(dev)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(v)).to(dev)
    return out


def _lengths(spec: str) -> list[int]:
    out = []
    for part in spec.split(","):
        if "x" in part:
            n, c = part.split("x")
            out += [int(n)] * int(c)
        else:
            out.append(int(part))
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["decode", "prefill", "spec", "commit", "conv", "rmsnorm", "fp8", "gemm"])
    ap.add_argument("--heads", choices=["full", "rank"], default="full")
    ap.add_argument("--requests", type=int, default=64)
    ap.add_argument("--slots", type=int, default=0)
    ap.add_argument("--lengths", default="2048x8", help="prefill lengths, e.g. 2048x8 or 16,300,8192")
    ap.add_argument("--loguniform", type=int, default=0, help="prefill: N log-uniform lengths in [16, 8192]")
    ap.add_argument("--k", type=int, default=6144, help="fp8, gemm: input features")
    ap.add_argument("--n", type=int, default=5120, help="fp8, gemm: output features")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=2)
    args = ap.parse_args(argv)

    from . import binding as b
    geom = synth.FULL_HEADS if args.heads == "full" else synth.RANK_HEADS
    dev = torch.device("cuda", 0)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    if args.case == "decode":
        w = synth.decode_workload(geom, args.requests, args.slots or 2 * args.requests, seed=1)
        d = _dev(w, dev)
        D = b.make_dims(geom, w["num_slots"])
        og = torch.empty((args.requests, geom.num_v_heads * 128), dtype=torch.bfloat16, device=dev)

        def run():
            b.gdn_decode_step(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["slot_idx"], d["alpha"],
                              d["beta"], d["z"], d["gamma"], w["eps"], ogate=og, dev_err=err)
    elif args.case in ("prefill", "conv"):
        lengths = (synth.loguniform_lengths(np.random.default_rng(3), args.loguniform, 16, 8192)
                   if args.loguniform else _lengths(args.lengths))
        w = synth.prefill_workload(geom, lengths, seed=3)
        d = _dev(w, dev)
        D = b.make_dims(geom, w["num_slots"])
        T = int(np.sum(lengths))
        og = torch.empty((T, geom.num_v_heads * 128), dtype=torch.bfloat16, device=dev)
        y = torch.empty((T, geom.channels), dtype=torch.bfloat16, device=dev) if args.case == "conv" else None
        ws = torch.empty(b.gdn_prefill_workspace_bytes(D, len(lengths), T), dtype=torch.uint8, device=dev)

        def run():
            if args.case == "conv":
                b.gdn_conv_update(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["query_start_loc"], d["slot_idx"],
                                  y, has_init=d["has_init"], dev_err=err)
            else:
                b.gdn_chunk_prefill(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["query_start_loc"],
                                    d["slot_idx"], d["alpha"], d["beta"], d["z"], d["gamma"], w["eps"], ogate=og,
                                    has_init=d["has_init"], workspace=ws, dev_err=err)
    elif args.case in ("spec", "commit"):
        w = synth.spec_workload(geom, args.requests, num_pos=4, seed=4)
        d = _dev(w, dev)
        D = b.make_dims(geom, w["num_slots"])
        og = torch.empty((args.requests * 4, geom.num_v_heads * 128), dtype=torch.bfloat16, device=dev)
        acc = torch.from_numpy(w["accepted"]).to(dev)

        def run():
            if args.case == "commit":  # copy the accepted position's checkpoint into the live slot
                b.gdn_spec_commit(D, acc, d["spec_slot_idx"], d["slot_idx"], d["state"], d["conv_hist"],
                                  mode=b.GDN_COMMIT_COPY, dev_err=err)
            else:
                b.gdn_spec_verify(D, d["qkv0"], d["conv_w"], d["conv_hist"], d["state"], d["slot_idx"],
                                  d["spec_slot_idx"], d["alpha"], d["beta"], d["z"], d["gamma"], w["eps"], ogate=og,
                                  dev_err=err)
    elif args.case == "fp8":
        # out [T, N] = dequant(x8) dequant(w8)^T with block scales: random E4M3 codes and scales
        rng = np.random.default_rng(6)
        T, K, N = args.requests, args.k, args.n
        x8 = torch.from_numpy(synth.fp8_codes(rng, (T, K))).to(dev)
        w8 = torch.from_numpy(synth.fp8_codes(rng, (N, K))).to(dev)
        xs = torch.from_numpy(rng.uniform(0.002, 0.02, size=(T, K // 128)).astype(np.float32)).to(dev)
        ws = torch.from_numpy(rng.uniform(1e-4, 1e-3, size=((N + 127) // 128, K // 128)).astype(np.float32)).to(dev)
        out = torch.empty((T, N), dtype=torch.bfloat16, device=dev)
        wsp = torch.zeros(max(256, b.gdn_fp8_linear_workspace_bytes(T, K, N)), dtype=torch.uint8, device=dev)

        def run():
            b.gdn_fp8_linear(x8, xs, w8, ws, out, workspace=wsp, dev_err=err)
    elif args.case == "gemm":
        # out [T, N] = x [T, K] w[N, K]^T + out (gdn_out_proj, the residual in place)
        g = torch.Generator(device=dev)
        g.manual_seed(7)
        T, K, N = args.requests, args.k, args.n
        x = torch.randn((T, K), generator=g, device=dev).to(torch.bfloat16)
        wt = (torch.randn((N, K), generator=g, device=dev) / K ** 0.5).to(torch.bfloat16)
        out = torch.randn((T, N), generator=g, device=dev).to(torch.bfloat16)

        def run():
            b.gdn_out_proj(x, wt, out, residual=out, dev_err=err)
    else:
        rng = np.random.default_rng(5)
        T = args.requests
        o = torch.from_numpy(synth.bf16_bits(rng.standard_normal((T, 48, 128)).astype(np.float32)).view(np.int16))
        z = torch.from_numpy(synth.bf16_bits(rng.standard_normal((T, 48, 128)).astype(np.float32)).view(np.int16))
        o, z = o.view(torch.bfloat16).to(dev), z.view(torch.bfloat16).to(dev)
        gamma = torch.ones(128, dtype=torch.float32, device=dev)
        out = torch.empty((T, 48 * 128), dtype=torch.bfloat16, device=dev)

        def run():
            b.gdn_gated_rmsnorm(o, z, gamma, 1e-6, out)

    times = []
    for it in range(args.warmup + args.launches):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        run()
        e1.record()
        torch.cuda.synchronize()
        if it >= args.warmup:
            times.append(e0.elapsed_time(e1))
    flag = b.gdn_read_device_error(err)
    tokens = {"decode": args.requests, "spec": args.requests * 4, "commit": args.requests,
              "fp8": args.requests, "gemm": args.requests}.get(args.case)
    if args.case in ("prefill", "conv"):
        tokens = T
    ms = sum(times) / max(1, len(times))
    rate = f", {tokens / (ms / 1e3):.4g} tokens/s" if tokens else ""
    print(f"profile_case {args.case}: {args.launches} launches after {args.warmup} warm-up, "
          f"mean {ms:.4f} ms{rate}, device error word {flag}")
    if flag:
        raise SystemExit(1)


if __name__ == "__main__":
    main()
