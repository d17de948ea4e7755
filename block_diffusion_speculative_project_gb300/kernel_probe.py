"""Time each C-ABI step call of one workload with CUDA events (a profiling aid).

  python -m block_diffusion_speculative_project_gb300.kernel_probe \
      [--workload NAME] [--nb NB] [--layers N] [--only lm_head|draft_block|ctx_project|all] \
      [--iters K]

Weights are seeded random (device-side generator, not the parity generator) and the
context cache is filled with random values, so the probe starts in seconds and
keeps the device footprint small enough for an ncu capture (use --layers 1).
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import dflash_inputs as di  # noqa: E402
from block_diffusion_speculative_project_gb300.drafter import Drafter  # noqa: E402


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default=di.QWEN3_8B.name, choices=sorted(di.WORKLOADS))
    ap.add_argument("--nb", type=int, default=0)
    ap.add_argument("--layers", type=int, default=0)
    ap.add_argument("--only", default="all", choices=["all", "lm_head", "draft_block", "ctx_project"])
    ap.add_argument("--iters", type=int, default=20)
    ap.add_argument("--cublas", action="store_true",
                    help="also time torch.nn.functional.linear (cuBLAS) on the step's GEMM shapes")
    args = ap.parse_args()
    w = di.WORKLOADS[args.workload]
    if args.nb:
        w = w.with_(nb=args.nb)
    if args.layers:
        w = w.with_(N=args.layers)
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    weights = {}
    for name, shp in di.weight_shapes(w).items():
        t = torch.randn(shp, device=dev, generator=g) * 0.02
        if name.rsplit(".", 1)[-1].startswith("g_"):
            t += 1.0
        weights[name] = t.to(torch.bfloat16)
    ctx = di.context_lengths(w).astype(np.int32)
    Cmax = int(ctx.max()) + w.B
    dr = Drafter(w, weights, w.nb, Cmax, w.B)
    dr.kcache.normal_(generator=g)
    dr.vcache.normal_(generator=g)
    i32 = lambda x: torch.tensor(np.asarray(x, np.int32), device=dev)
    tp = di.tau_prev(w).astype(np.int32)
    hv = torch.randn(w.nb, w.B, w.L * w.Dt, device=dev, generator=g).to(torch.bfloat16)
    base = i32(ctx - tp)
    ctx_len = base.clone()
    ncommit = i32(tp)
    block = i32(di.block_ids(w, di.anchors(w)))
    hidden = torch.randn(w.nb, w.B, w.D, device=dev, generator=g).to(torch.bfloat16)
    tid = torch.empty(w.nb, w.B - 1, w.k_top, dtype=torch.int32, device=dev)
    tv = torch.empty(w.nb, w.B - 1, w.k_top, dtype=torch.float32, device=dev)
    calls = {
        "ctx_project": lambda: (ctx_len.copy_(base), dr.ctx_project(w.nb, w.B, hv, ncommit, ctx_len)),
        "draft_block": lambda: dr.draft_block(w.nb, block, i32(ctx), hidden, max_ctx_hint=int(ctx.max())),
        "lm_head": lambda: dr.lm_head_topk(w.nb, hidden, w.k_top, tid, tv),
    }
    names = list(calls) if args.only == "all" else [args.only]
    for n in names:
        calls[n]()
    torch.cuda.synchronize()
    if dr.status() != 0:
        raise RuntimeError("device status reports an error")
    for n in names:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for _ in range(args.iters):
            e0.record()
            calls[n]()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        print(f"{w.name} nb={w.nb} N={w.N} {n}: median {np.median(ts):.4f} ms  min {np.min(ts):.4f} ms")
    if args.cublas:
        M = w.nb * w.B
        shapes = {"W_c": (M, w.D, w.L * w.Dt), "qkv": (M, (w.Hq + 2 * w.Hkv) * w.hd, w.D),
                  "o": (M, w.D, w.Hq * w.hd), "gate|up": (M, 2 * w.F, w.D), "down": (M, w.D, w.F),
                  "lm_head": (w.nb * (w.B - 1), w.V, w.D)}
        for name, (m, n, k) in shapes.items():
            a = torch.randn(m, k, device=dev, generator=g).to(torch.bfloat16)
            b = torch.randn(n, k, device=dev, generator=g).to(torch.bfloat16) * 0.02
            for _ in range(3):
                torch.nn.functional.linear(a, b)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ts = []
            for _ in range(args.iters):
                e0.record()
                torch.nn.functional.linear(a, b)
                e1.record()
                e1.synchronize()
                ts.append(e0.elapsed_time(e1))
            t = float(np.median(ts))
            print(f"cublas {name} [{m}x{k}]x[{k}x{n}]: {t * 1e3:.1f} us  {2 * n * k / (t * 1e-3) / 1e9:.0f} GB/s")


if __name__ == "__main__":
    main()
