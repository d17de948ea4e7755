"""Benchmark of the one-pass block-diffusion draft step on GB300.

One step = rewind ctx_len, dflash_ctx_project (append the previous round's committed
verifier rows; relay rows with the relay workload), dflash_draft_block,
dflash_lm_head_topk (+ dflash2_select with the DFlash 2 workload), dflash_accept,
over one batch of seeded synthetic inputs already resident in HBM. The step is
captured in a CUDA graph and replayed; K timed replays are bracketed by a barrier and
a device synchronize, timed with CUDA events on the launching stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]
  python bench.py --profile-case {lm_head,draft_block,ctx_project,sampling} [--layers N] ...

N > 1 (torchrun, one process per GPU) runs N independent replicas (the step shards
by sequence with no exchange); value = sequences of all ranks / the slowest rank's
time. --impl reference times the CPU oracle (the only reference this method has) on
the host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dflash_inputs as di  # noqa: E402

DEFAULT_WORKLOAD = di.QWEN3_8B.name
METRIC = "draft blocks/sec (Qwen3-8B-shaped, B=16)"
PROJ_CHUNK = 2048   # rows per sequence of one ctx_project call when filling the context
PREFILL_ROWS = 2048  # prompt rows per sequence of the measured prefill


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def step_bytes_flops(w: di.Workload, ctx: np.ndarray, tp: np.ndarray):
    """Algorithmic bytes and FLOPs of one step (each weight read once, each context
    K/V row read once per layer, inputs and outputs once)."""
    qkv_n = (w.Hq + 2 * w.Hkv) * w.hd
    per_layer_w = (qkv_n * w.D + w.D * w.Hq * w.hd + 3 * w.F * w.D + 2 * w.Hkv * w.hd * w.D)
    if w.flags & di.FLAG_CONV:
        per_layer_w += 4 * (2 * (w.D // w.conv_group) * w.D + 2 * w.D)
    wbytes = 2 * (w.N * per_layer_w + w.D * w.L * w.Dt + w.V * w.D + 2 * w.D * w.N + 2 * w.D)
    if w.flags & di.FLAG_SELECT:
        wbytes += 2 * 3 * w.sel_dim * w.D
    if w.flags & di.FLAG_FILM:
        wbytes += 2 * 5 * w.D * w.film_width
    kv_bytes = int(ctx.sum()) * w.N * 2 * w.Hkv * w.hd * 2
    M = w.nb * w.B
    rows_proj = w.nb * w.B
    io = rows_proj * w.L * w.Dt * 2 + w.nb * w.B * w.D * 2 + int(tp.sum()) * w.N * 2 * w.Hkv * w.hd * 2
    flops = 2 * rows_proj * w.D * w.L * w.Dt + 2 * rows_proj * w.N * 2 * w.Hkv * w.hd * w.D
    flops += 2 * M * w.N * (qkv_n * w.D + w.D * w.Hq * w.hd + 3 * w.F * w.D)
    flops += 2 * 2 * w.N * (w.Hq * w.B) * w.hd * int((ctx + w.B).sum())
    flops += 2 * w.nb * (w.B - 1) * w.V * w.D
    if w.flags & di.FLAG_FILM:
        flops += 2 * M * 5 * w.D * w.film_width
    if w.temperature > 0:
        # draft logits written by the LM head and read by the draw (not with the DFlash 2
        # walk); target logits read for their normaliser; one target row (and one draft
        # row) per sequence read again by the residual draw
        if not w.flags & di.FLAG_SELECT:
            io += 2 * w.nb * (w.B - 1) * w.V * 4 + w.nb * w.V * 4
        io += w.nb * w.B * w.V * 4 + w.nb * w.V * 4
    return wbytes + kv_bytes + io, flops, wbytes, kv_bytes


def kernels_per_step(w: di.Workload) -> int:
    """Launches of libdflash kernels in one step (see dflash_api.cu)."""
    n = 4                                 # ctx_project: W_c GEMM, RMSNorm, K/V GEMM, relay/len
    if w.flags & di.FLAG_FILM:
        n += 4                            # FiLM: conditioning rows, W1 GEMM, W2 GEMM, apply
    n += 1                                # embedding (+ first RMSNorm)
    per_layer = 6                         # QKV, attention, merge, O, gate|up, down (norms deferred)
    if w.flags & di.FLAG_CONV:
        per_layer += 4 * 2 + 2            # each conv: GEMM + apply; RMSNorm after conv0, conv2
        n += 1                            # bf16 copy of the embedding for layer 0's conv0
    n += w.N * per_layer
    n += 1                                # final RMSNorm
    n += 2                                # LM head GEMM + merge
    if w.flags & di.FLAG_SELECT:
        n += 5                            # gather, A|B GEMM, G GEMM, score table, walk
    if w.temperature > 0 and w.flags & di.FLAG_SELECT:
        n += 4                            # verify of the sampling walk (target lse x2, walk x2)
    elif w.temperature > 0:
        n += 2 + 4                        # draw (partial, merge); verify (target lse x2, walk x2)
    else:
        n += 1                            # accept
    return n


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.index = index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[4:8]))
            except ValueError:
                continue
        if not rows:
            return None
        sm = [r[0] for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[2][k].lower().startswith("active")})
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def traffic_from_profile(kernel_src: str):
    """dram bytes per launch of the LM-head GEMM from the committed ncu summary, or
    None when the kernel source changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "lm_head_topk_traffic.txt")
    if not os.path.exists(p):
        return None
    kv = dict(line.split("=", 1) for line in open(p).read().split() if "=" in line)
    sha = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()[:16]
    if kv.get("gemm_source_sha") != sha:
        return None
    try:
        return float(kv["dram_bytes_per_full_launch"])
    except (KeyError, ValueError):
        return None


def max_over_ranks(values, device=None):
    """Element-wise max of a list of floats over all ranks (identity when not distributed).
    The only cross-rank communication in the benchmark: the draft step itself shards by
    sequence and exchanges nothing."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    dev = device if (device is not None and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu().tolist()]


# ----------------------------------------------------------------------------- GPU arm

def measure_workload(w, weights, dev, world, steps, warmup, full=True):
    """Set up one workload on this GPU (caches, context prefill, step inputs), capture its
    step in a CUDA graph and time `steps` replays; with `full`, also the LM head inside the
    step, the end-to-end leg through host buffers and the prompt prefill. Returns the raw
    measurements (times are maxima over ranks)."""
    import torch
    from block_diffusion_speculative_project_gb300.drafter import Drafter, to_device_bf16

    seed = 0  # every replica runs the same workload
    ctx = di.context_lengths(w, seed).astype(np.int32)
    tp = di.tau_prev(w, seed).astype(np.int32)
    relay = bool(w.flags & di.FLAG_RELAY)
    if relay:
        a = di.accepted_prev(w, seed).astype(np.int32)
        tp = (a + 1).astype(np.int32)
    base = (ctx - tp).astype(np.int32)
    Cmax = int(ctx.max()) + w.B
    if w.paged:
        Cmax = -(-Cmax // di.PAGE_ROWS) * di.PAGE_ROWS
    num_pages = w.nb * (Cmax // di.PAGE_ROWS) if w.paged else 0
    dr = Drafter(w, weights, w.nb, Cmax, max(PROJ_CHUNK, PREFILL_ROWS, w.B), num_pages=num_pages)
    i32 = lambda x: torch.tensor(np.asarray(x, np.int32), device=dev)
    if w.paged:  # every sequence's pages in a seeded shuffled order
        dr.set_block_table(i32(di.block_table(w.nb, Cmax, seed)))

    # prefill C_i - tau_prev_i context rows per sequence (outside every timed region)
    g = torch.Generator(device=dev)
    g.manual_seed(1234)
    ctx_len = i32(np.zeros(w.nb))
    done = np.zeros(w.nb, np.int64)
    while (done < base).any():
        R = PROJ_CHUNK
        ncommit = np.minimum(R, base - done).astype(np.int32)
        hv = torch.randn(w.nb, R, w.L * w.Dt, device=dev, generator=g).to(torch.bfloat16)
        dr.ctx_project(w.nb, R, hv, i32(ncommit), ctx_len)
        done += ncommit
    del hv
    ctx_base = ctx_len.clone()
    assert np.array_equal(ctx_base.cpu().numpy(), base)

    # step inputs, resident in HBM
    hv_step = to_device_bf16(di.verifier_rows(w, w.B, seed, name="hv_step"), dev)
    # every int32 input of the step lives in one device buffer, so that the end-to-end
    # leg's single host-to-device copy is exactly what the step consumes
    parts = {"n_commit": tp, "block": di.block_ids(w, di.anchors(w, seed)),
             "target": np.zeros((w.nb, w.B), np.int32)}
    if relay:
        parts["relay_a"] = a
    if w.flags & di.FLAG_FILM:
        parts["relay_b"], parts["relay_y"] = di.relay_tokens(w, seed)
    host_in_np = np.concatenate([np.asarray(v, np.int32).ravel() for v in parts.values()])
    step_in = i32(host_in_np)
    views, spans, off = {}, {}, 0
    for name, v in parts.items():
        n = int(np.asarray(v).size)
        views[name] = step_in[off:off + n].view(np.asarray(v).shape)
        spans[name] = (off, off + n)
        off += n
    n_commit = views["n_commit"]
    relay_a = views.get("relay_a")
    film = {k: views[k] for k in ("relay_b", "relay_y") if k in views}
    x0 = torch.empty(w.nb, w.B, w.D, dtype=torch.bfloat16, device=dev) if relay else None
    block = views["block"]
    hidden = torch.empty(w.nb, w.B, w.D, dtype=torch.bfloat16, device=dev)
    k = w.k_top
    # the step's results (tau, bonus, the top-k ids) in one device buffer, so the end-to-end
    # leg reads them back with one copy
    nt = w.nb * (w.B - 1) * k
    out_dev = torch.zeros(nt + 2 * w.nb, dtype=torch.int32, device=dev)
    tid = out_dev[:nt].view(w.nb, w.B - 1, k)
    tv = torch.empty(w.nb, w.B - 1, k, dtype=torch.float32, device=dev)
    path = torch.empty(w.nb, w.B - 1, dtype=torch.int32, device=dev)
    target = views["target"]
    tau = out_dev[nt:nt + w.nb]
    bonus = out_dev[nt + w.nb:]
    select = bool(w.flags & di.FLAG_SELECT)
    draft = path if select else tid[..., 0]
    draft_c = torch.empty(w.nb, w.B - 1, dtype=torch.int32, device=dev)
    sampling = w.temperature > 0
    if sampling:  # the target model's verify logits stand resident in HBM (it runs on this GPU)
        # the plain draw needs the draft logits; the DFlash 2 walk's draft distribution lives
        # on the k candidates, so it needs none
        draft_logits = None if select else torch.empty(w.nb, w.B - 1, w.V, dtype=torch.float32, device=dev)
        draft_lse = torch.empty(w.nb, w.B - 1, dtype=torch.float32, device=dev)
        walk_logq = torch.empty(w.nb, w.B - 1, k, dtype=torch.float32, device=dev)
        tgt_logits = torch.from_numpy(di.target_logits(w, seed)).to(dev)
        sample_seed = 0x5EED_0000 + seed
    max_ctx = int(ctx.max())
    stream = torch.cuda.Stream(device=dev)
    try:  # event-record nodes inside the captured step (torch >= 2.7)
        ev_lm = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
        lm_in_graph = True
    except TypeError:
        ev_lm = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        lm_in_graph = False

    def step(s, lm_events=None):
        ctx_len.copy_(ctx_base)
        dr.ctx_project(w.nb, w.B, hv_step, n_commit, ctx_len, relay_a=relay_a, x0_relay=x0, stream=s,
                       **film)
        dr.draft_block(w.nb, block, ctx_len, hidden, x0_relay=x0, max_ctx_hint=max_ctx, stream=s)
        if lm_events:
            lm_events[0].record(s)
        dr.lm_head_topk(w.nb, hidden, k, tid, tv, draft_logits if sampling else None, stream=s)
        if lm_events:
            lm_events[1].record(s)
        if sampling and select:  # DFlash 2 sampling walk, verified against its distribution
            dr.select_sample(w.nb, k, tid, tv, hidden, block, w.temperature, sample_seed, path, walk_logq,
                             stream=s)
            dr.verify_sample_walk(w.nb, k, tid, walk_logq, path, tgt_logits, w.temperature, sample_seed,
                                  tau, bonus, stream=s)
            return
        if sampling:  # draw over the written logits, then the verify
            dr.sample(w.nb * (w.B - 1), draft_logits, w.temperature, sample_seed, draft_c, draft_lse,
                      stream=s)
            dr.verify_sample(w.nb, draft_logits, draft_lse, draft_c, tgt_logits, w.temperature,
                             sample_seed, tau, bonus, stream=s)
            return
        if select:  # the walk's path is the draft
            dr.select(w.nb, k, tid, tv, hidden, block, path, stream=s)
            dr.accept(w.nb, path, target, tau, bonus, stream=s)
        else:  # the first entry of each offset's top-k list is the draft
            dr.accept_topk(w.nb, tid, k, target, tau, bonus, stream=s)

    with torch.cuda.stream(stream):
        step(stream)
    stream.synchronize()
    if dr.status(stream) != 0:
        raise RuntimeError("device status reports an error after the first step")
    if not sampling:
        trow = di.target_row_from_draft(draft.contiguous().cpu().numpy(), w.V, seed)
        target.copy_(i32(trow))
        # the host copy of the step's inputs carries the same target row, so the end-to-end
        # leg runs exactly the step the timed region runs
        t0_, t1_ = spans["target"]
        host_in_np[t0_:t1_] = np.asarray(trow, np.int32).ravel()

    # capture one step in a CUDA graph (warm-up launches above configured every kernel)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        step(stream)  # one more eager step before capture
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            step(stream)
    lm_graph = None
    if lm_in_graph:
        lm_graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(lm_graph, stream=stream):
                step(stream, ev_lm)

    for _ in range(warmup):
        with torch.cuda.stream(stream):
            graph.replay()
    stream.synchronize()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # timed region
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(dev.index)
    time.sleep(0.3)
    torch.cuda.nvtx.range_push("timed")
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            graph.replay()
        e1.record(stream)
    stream.synchronize()
    torch.cuda.nvtx.range_pop()
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    ms_total = e0.elapsed_time(e1)

    # dominant kernel (LM head GEMM + top-k): events on its stream inside the replayed
    # graph, averaged over replays of the same step
    lm_ms = []
    for _ in range(max(5, min(50, steps // 10))):
        with torch.cuda.stream(stream):
            if lm_graph is not None:
                lm_graph.replay()
            else:
                step(stream, ev_lm)
        stream.synchronize()
        lm_ms.append(ev_lm[0].elapsed_time(ev_lm[1]))
    if dr.status(stream) != 0:
        raise RuntimeError("device status reports an error after the timed steps")
    tau_h = tau.cpu().numpy()

    e2e = pre_ms = None
    if full:
        # e2e through the public API with host buffers: H2D of the step's inputs from pinned
        # memory and D2H of its results, every step, inside the timed region. Each step waits
        # for its results on the host before the next begins (the next step's inputs come from
        # the verifier, which needs this step's draft). Events split each step into the copies
        # in, the step, the copy out; the rest is host-side launch and wake-up time.
        host_hv = hv_step.cpu().pin_memory()
        host_in = torch.from_numpy(host_in_np).pin_memory()
        host_out = torch.empty(out_dev.numel(), dtype=torch.int32).pin_memory()
        e2e_steps = 300
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(e2e_steps)]
        barrier()
        torch.cuda.synchronize(dev)
        t_e2e = time.perf_counter()
        with torch.cuda.stream(stream):
            for it in range(e2e_steps):
                ev = evs[it]
                ev[0].record(stream)
                hv_step.copy_(host_hv, non_blocking=True)
                step_in.copy_(host_in, non_blocking=True)
                ev[1].record(stream)
                graph.replay()
                ev[2].record(stream)
                host_out.copy_(out_dev, non_blocking=True)
                ev[3].record(stream)
                stream.synchronize()
        e2e_s = time.perf_counter() - t_e2e
        barrier()
        e2e_parts = np.array([[ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2]), ev[2].elapsed_time(ev[3])]
                              for ev in evs]).mean(axis=0)
        if not np.array_equal(host_out[nt:nt + w.nb].numpy(), tau.cpu().numpy()):
            raise RuntimeError("the end-to-end leg's result differs from the device result")
        h2d = host_hv.numel() * 2 + host_in.numel() * 4
        d2h = host_out.numel() * 4

        # prompt prefill through dflash_ctx_project (the large-context path, compute-bound W_c
        # GEMM over nb * PREFILL_ROWS rows): after the step timing, so rewriting the first
        # context rows of the caches does not matter any more
        hv_pre = torch.randn(w.nb, PREFILL_ROWS, w.L * w.Dt, device=dev, generator=g).to(torch.bfloat16)
        pre_commit = i32(np.full(w.nb, PREFILL_ROWS))
        pre_zero = i32(np.zeros(w.nb))
        pre_len = pre_zero.clone()
        pre_ms = []
        with torch.cuda.stream(stream):
            for rep in range(4):
                pre_len.copy_(pre_zero)
                p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                p0.record(stream)
                dr.ctx_project(w.nb, PREFILL_ROWS, hv_pre, pre_commit, pre_len, stream=stream)
                p1.record(stream)
                stream.synchronize()
                if rep:
                    pre_ms.append(p0.elapsed_time(p1))
        if dr.status(stream) != 0:
            raise RuntimeError("device status reports an error after the prefill")
        del hv_pre
        e2e = dict(steps=e2e_steps, s=e2e_s, parts=e2e_parts, h2d=h2d, d2h=d2h)
    e2e_s = e2e["s"] if e2e else 0.0
    ms_step, e2e_s = max_over_ranks([ms_total / steps, e2e_s], dev)
    if e2e:
        e2e["s"] = e2e_s
    return dict(w=w, ctx=ctx, tp=tp, k=k, ms_step=ms_step, lm_ms=lm_ms, clk=clk, tau=tau_h, e2e=e2e,
                pre_ms=pre_ms)


def step_summary(m, world):
    """Blocks/s and the step's roofline fraction of one measured workload."""
    w = m["w"]
    hbm, tf_burst, tf_sus, _ = load_peaks()
    total_bytes, flops, _, _ = step_bytes_flops(w, m["ctx"], m["tp"])
    step_t_roof = max(total_bytes / (hbm * 1e9), flops / (tf_sus * 1e12 if tf_sus else tf_burst * 1e12))
    value = w.nb * world / (m["ms_step"] * 1e-3)
    return {"value": round(value, 2), "unit": "blocks/s", "ms_per_step": round(m["ms_step"], 4),
            "draft_tokens_per_s": round(value * (w.B - 1), 1),
            "step_roofline": {"bytes": total_bytes, "flops": flops, "t_roofline_ms": round(step_t_roof * 1e3, 4),
                              "frac": round(step_t_roof * 1e3 / m["ms_step"], 4)},
            "config": {"nb_per_gpu": w.nb, "B": w.B, "context": int(m["ctx"].mean()),
                       "context_range": [int(m["ctx"].min()), int(m["ctx"].max())]},
            "clocks": m["clk"], "tau_mean": round(float(m["tau"].mean()), 3)}


# The 64-sequence B = 8 serving configuration (ragged contexts in [1024, 8192]), timed in
# the same process as the default workload so that one benchmark run reports both.
EXTRA_WORKLOADS = (di.SWEEP_NB64.name,)


def run_gpu(args, rank, world):
    import torch
    from block_diffusion_speculative_project_gb300.drafter import to_device_bf16

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = di.WORKLOADS[args.workload]
    t0 = time.time()
    bits = di.make_weights(w, 0)
    weights = {k: to_device_bf16(v, dev) for k, v in bits.items()}
    t_gen = time.time() - t0
    m = measure_workload(w, weights, dev, world, args.steps, args.warmup, full=True)
    extra = {}
    if args.workload == DEFAULT_WORKLOAD and not args.no_extra_workloads:
        for name in EXTRA_WORKLOADS:
            torch.cuda.empty_cache()
            m2 = measure_workload(di.WORKLOADS[name], weights, dev, world, max(args.steps, 100),
                                  args.warmup, full=False)
            extra[name] = step_summary(m2, world)
            extra[name]["steps"] = max(args.steps, 100)
    ctx, tp, k, lm_ms, clk, tau_h, pre_ms = m["ctx"], m["tp"], m["k"], m["lm_ms"], m["clk"], m["tau"], m["pre_ms"]
    ms_step = m["ms_step"]
    e2e_steps, e2e_s, e2e_parts = m["e2e"]["steps"], m["e2e"]["s"], m["e2e"]["parts"]
    h2d, d2h = m["e2e"]["h2d"], m["e2e"]["d2h"]

    if rank != 0:
        return None
    hbm, tf_burst, tf_sus, src = load_peaks()
    total_bytes, flops, _, _ = step_bytes_flops(w, ctx, tp)
    lm_bytes = 2 * w.V * w.D + 2 * w.nb * (w.B - 1) * w.D + 8 * w.nb * (w.B - 1) * k
    if w.temperature > 0 and not w.flags & di.FLAG_SELECT:
        lm_bytes += 4 * w.nb * (w.B - 1) * w.V  # the fp32 logits the draw reads
    lm_avg = float(np.mean(lm_ms))
    achieved = lm_bytes / (lm_avg * 1e-3) / 1e9
    traffic = traffic_from_profile(os.path.join(ROOT, "block_diffusion_speculative_project_gb300",
                                                "csrc", "gemm_tc.cu"))
    blocks = w.nb * world
    value = blocks / (ms_step * 1e-3)
    pre_rows = w.nb * PREFILL_ROWS
    pre_flops = 2 * pre_rows * w.D * (w.L * w.Dt + 2 * w.N * w.Hkv * w.hd)
    pre_t = float(np.mean(pre_ms)) * 1e-3
    step_t_roof = max(total_bytes / (hbm * 1e9), flops / (tf_sus * 1e12 if tf_sus else tf_burst * 1e12))
    line = {
        "metric": METRIC if args.workload == DEFAULT_WORKLOAD else f"draft blocks/sec ({args.workload})",
        "value": round(value, 2),
        "unit": "blocks/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded: weights N(0,0.02), verifier states N(0,1))",
        "config": {"workload": w.name, "nb_per_gpu": w.nb, "B": w.B, "context": int(ctx.mean()),
                   "context_range": [int(ctx.min()), int(ctx.max())], "parallelism": f"replicas{world}",
                   "l2": f"inputs larger than L2 ({total_bytes / 1e9:.2f} GB read per step)",
                   "cuda_graph": True},
        "draft_tokens_per_s": round(value * (w.B - 1), 1),
        "step_roofline": {"bytes": total_bytes, "flops": flops, "t_roofline_ms": round(step_t_roof * 1e3, 4),
                          "frac": round(step_t_roof * 1e3 / ms_step, 4),
                          "hbm_frac_at_8TBps": round(total_bytes / 8e12 * 1e3 / ms_step, 4)},
        "roofline": {"kernel": "gemm_tc_kernel<256,EPI_TOPK> (LM head + fused top-k) + top-k merge",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": traffic, "peak_source": src,
                     "avg_launch_ms": round(lm_avg, 4), "bytes_per_launch": lm_bytes},
        "prefill": {"rows_per_seq": PREFILL_ROWS, "rows": pre_rows, "ms": round(pre_t * 1e3, 4),
                    "prompt_rows_per_s": round(pre_rows / pre_t, 1), "bound": "tensor",
                    "achieved": round(pre_flops / pre_t / 1e12, 1), "peak": tf_burst, "unit": "TFLOP/s",
                    "frac": round(pre_flops / pre_t / 1e12 / tf_burst, 4),
                    "what": "dflash_ctx_project: W_c GEMM, RMSNorm, K/V GEMMs of every layer into the caches"},
        "e2e": {"value": round(blocks * e2e_steps / e2e_s, 2), "unit": "blocks/s",
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps,
                "ms_per_step": round(e2e_s * 1e3 / e2e_steps, 4),
                "breakdown_ms": {"h2d": round(float(e2e_parts[0]), 4), "step": round(float(e2e_parts[1]), 4),
                                 "d2h": round(float(e2e_parts[2]), 4),
                                 "host": round(e2e_s * 1e3 / e2e_steps - float(e2e_parts.sum()), 4)}},
        "gpu_launches": kernels_per_step(w) * args.steps,
        "clocks": clk,
        "tau_mean": round(float(tau_h.mean()), 3),
        "setup_s": {"weights": round(t_gen, 1)},
    }
    if extra:
        line["workloads"] = extra
    if not args.no_cpu_baseline and rank == 0:
        line["cpu_baseline"] = cpu_baseline(w, bits, args.cpu_seconds)
    return line




# ----------------------------------------------------------------------------- oracle (CPU)

def cpu_baseline(w: di.Workload, bits=None, budget_s: float = 15.0):
    """The oracle, as it stands, in float32 on this host's cores over a bounded sample:
    whole draft steps of single sequences of the workload (context filled with seeded
    values, the step's own append, draft, LM head, top-k and accept)."""
    from oracle import dflash_oracle as orc
    cores = len(os.sched_getaffinity(0))
    if bits is None:
        bits = di.make_weights(w)
    W = orc.widen_all(bits, np.float32)
    ctx = di.context_lengths(w).astype(np.int64)
    tp = di.tau_prev(w).astype(np.int64)
    a = None
    if w.flags & di.FLAG_RELAY:
        a = di.accepted_prev(w).astype(np.int64)
        tp = a + 1
    fb = fy = None
    if w.flags & di.FLAG_FILM:
        fb, fy = di.relay_tokens(w)
    ids = di.block_ids(w, di.anchors(w))
    Z = di.target_logits(w).astype(np.float32) if w.temperature > 0 else None
    rng = np.random.default_rng(7)
    done, t_used = 0, 0.0
    while t_used < budget_s and done < w.nb:
        i = done
        Cmax = int(ctx[i]) + w.B
        cache = orc.KVCache(w.N, 1, w.Hkv, Cmax, w.hd, np.float32)
        base = int(ctx[i] - tp[i])
        for n in range(w.N):
            cache.K[n][0][:, :base] = rng.standard_normal((w.Hkv, base, w.hd), dtype=np.float32)
            cache.V[n][0][:, :base] = rng.standard_normal((w.Hkv, base, w.hd), dtype=np.float32)
        hv = orc.widen(di.verifier_rows(w.with_(nb=1), w.B, name=f"hv_cpu{i}"), np.float32)
        t0 = time.perf_counter()
        o = orc.draft_step(w, W, hv, tp[i:i + 1], [base], cache, ids[i:i + 1],
                           np.zeros((1, w.B), np.int32), relay_a=None if a is None else a[i:i + 1],
                           relay_b=None if fb is None else fb[i:i + 1],
                           relay_y=None if fy is None else fy[i:i + 1])
        if w.temperature > 0 and w.flags & di.FLAG_SELECT:
            path, logq, _ = orc.select_walk_sample(w, W, o["ids"], o["vals"], o["hidden"], ids[i:i + 1, 0],
                                                   w.temperature, i)
            orc.verify_sample_walk(o["ids"], logq, path, Z[i:i + 1], w.temperature, i)
        elif w.temperature > 0:
            cand, _, _, _ = orc.sample_candidates(o["logits"], w.temperature, i)
            orc.verify_sample(o["logits"], cand, Z[i:i + 1], w.temperature, i)
        t_used += time.perf_counter() - t0
        done += 1
    per_seq = t_used / done
    return {"value": round(1.0 / per_seq, 4), "unit": "blocks/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} whole-step sequence(s) of {w.name} (fp32 numpy oracle), {t_used:.1f} s",
            "seconds_per_block": round(per_seq, 3)}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = di.WORKLOADS[args.workload]
    t0 = time.time()
    bits = di.make_weights(w)
    gen = time.time() - t0
    budget = max(5.0, min(60.0, args.cpu_seconds))
    per_step = []
    for _ in range(args.warmup + args.steps):
        per_step.append(cpu_baseline(w, bits, budget / max(1, args.steps + args.warmup)))
    timed = per_step[args.warmup:]
    spb = float(np.mean([t["seconds_per_block"] for t in timed]))
    value = 1.0 / spb
    cb = dict(timed[-1])
    cb["value"] = round(value, 4)
    return {"impl": "reference", "metric": METRIC if args.workload == DEFAULT_WORKLOAD else
            f"draft blocks/sec ({args.workload})", "value": round(value, 4), "unit": "blocks/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(spb * w.nb * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "nb_per_gpu": w.nb, "B": w.B},
            "cpu_baseline": cb, "e2e": {"value": round(value, 4), "unit": "blocks/s",
                                        "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "setup_s": {"weights": round(gen, 1)}}


# ----------------------------------------------------------------------------- profiling cases

def run_profile_case(args):
    """Small, self-contained cases of the step's kernels for ncu captures (no JSON line,
    no timing contract): weights and caches come from a device-side generator, so a case
    starts in seconds and holds little device memory.

      lm_head      the LM head + top-k of the workload (the full vocabulary)
      draft_block  dflash_draft_block with --layers layers (default 1) and a 4096-token
                   vocabulary (the QKV, attention, merge, O, gate|up and down launches at the
                   workload's shapes)
      ctx_project  the context append (W_c GEMM, RMSNorm, grouped K/V GEMM) of the step, or
                   of --rows rows per sequence (a prefill)
      sampling     dflash_sample + dflash_verify_sample at V = 151936, 16 sequences of B = 16
                   (draft and target logits both larger than L2), tiny drafter otherwise
    Prints the per-call CUDA-event time of each iteration's median."""
    import torch
    from block_diffusion_speculative_project_gb300.drafter import Drafter

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    case = args.profile_case
    w = di.WORKLOADS[args.workload]
    if args.nb:
        w = w.with_(nb=args.nb)
    if case == "sampling":
        w = di.TINY.with_(V=151936, B=16, nb=16)
    elif case == "draft_block":
        w = w.with_(N=args.layers or 1, V=4096, L=1)
    elif args.layers:
        w = w.with_(N=args.layers)
    weights = {}
    for name, shp in di.weight_shapes(w).items():
        t = torch.randn(shp, device=dev, generator=g) * 0.02
        if name.rsplit(".", 1)[-1].startswith("g_"):
            t += 1.0
        weights[name] = t.to(torch.bfloat16)
    i32 = lambda x: torch.tensor(np.asarray(x, np.int32), device=dev)
    ctx = di.context_lengths(w).astype(np.int32)
    rows = max(w.B, args.rows)
    Cmax = int(ctx.max()) + max(w.B, rows)
    dr = Drafter(w, weights, w.nb, Cmax, rows)
    dr.kcache.normal_(generator=g)
    dr.vcache.normal_(generator=g)
    if case == "sampling":
        nr = w.nb * (w.B - 1)
        U = torch.randn(w.nb, w.B - 1, w.V, device=dev, generator=g) * 2
        Z = torch.randn(w.nb, w.B, w.V, device=dev, generator=g) * 2
        cand = torch.zeros(w.nb, w.B - 1, dtype=torch.int32, device=dev)
        lse = torch.zeros(w.nb, w.B - 1, device=dev)
        tau = torch.zeros(w.nb, dtype=torch.int32, device=dev)
        tok = torch.zeros_like(tau)
        calls = {"sample": lambda: dr.sample(nr, U, 1.0, 99, cand, lse),
                 "verify_sample": lambda: dr.verify_sample(w.nb, U, lse, cand, Z, 1.0, 99, tau, tok)}
    elif case == "ctx_project":
        tp = di.tau_prev(w).astype(np.int32) if rows == w.B else np.full(w.nb, rows, np.int32)
        hv = torch.randn(w.nb, rows, w.L * w.Dt, device=dev, generator=g).to(torch.bfloat16)
        base = i32(np.zeros(w.nb) if rows > w.B else ctx - tp)
        ctx_len = base.clone()
        ncommit = i32(tp)
        calls = {"ctx_project": lambda: (ctx_len.copy_(base), dr.ctx_project(w.nb, rows, hv, ncommit, ctx_len))}
    else:
        block = i32(di.block_ids(w, di.anchors(w)))
        hidden = torch.randn(w.nb, w.B, w.D, device=dev, generator=g).to(torch.bfloat16)
        tid = torch.empty(w.nb, w.B - 1, w.k_top, dtype=torch.int32, device=dev)
        tv = torch.empty(w.nb, w.B - 1, w.k_top, dtype=torch.float32, device=dev)
        ctx_t = i32(ctx)
        if case == "lm_head":
            calls = {"lm_head_topk": lambda: dr.lm_head_topk(w.nb, hidden, w.k_top, tid, tv)}
        else:
            calls = {"draft_block": lambda: dr.draft_block(w.nb, block, ctx_t, hidden,
                                                           max_ctx_hint=int(ctx.max()))}
    for f in calls.values():
        f()
    torch.cuda.synchronize()
    if dr.status() != 0:
        raise RuntimeError("device status reports an error")
    for name, f in calls.items():
        ts = []
        for _ in range(args.iters):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            f()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        print(f"{case}: {w.name} nb={w.nb} N={w.N} {name}: median {np.median(ts) * 1e3:.1f} us, "
              f"min {np.min(ts) * 1e3:.1f} us over {args.iters} calls (host launch time included)")
    if dr.status() != 0:
        raise RuntimeError("device status reports an error")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(di.WORKLOADS))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-workloads", action="store_true",
                    help="time only --workload (by default the default workload's run also times the "
                         "batch-64 ragged workload)")
    ap.add_argument("--profile-case", choices=["lm_head", "draft_block", "ctx_project", "sampling"],
                    help="run one small kernel case for an ncu capture instead of the benchmark")
    ap.add_argument("--layers", type=int, default=0, help="drafter layers of a --profile-case")
    ap.add_argument("--nb", type=int, default=0, help="sequences of a --profile-case (0: the workload's)")
    ap.add_argument("--rows", type=int, default=0, help="rows per sequence of --profile-case ctx_project")
    ap.add_argument("--iters", type=int, default=3, help="timed calls of a --profile-case")
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group(backend)
    line = run_reference(args, rank, world) if args.impl == "reference" else run_gpu(args, rank, world)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
