#!/usr/bin/env python
"""Benchmark of the DFlash2 draft step on GB300: draft steps/s and proposed
tokens/s, with the fraction of the step roofline and of the dominant
kernel's roofline (the lm_head contraction with its fused top-k).

One step = dflash2_draft_step + dflash2_select_path_table +
dflash2_verify_accept (feature projection of B newly committed positions
per sequence, paged K/V append, one non-causal block forward, lm_head +
top-k, selector, verify), captured as one CUDA graph.  The selector's
per-token factor table is built once at setup, like the weights themselves
(it is a function of the frozen embedding and selector weights only).
Inputs are resident in HBM.  Every step streams the whole weight set (0.6 to
2.7 GB) through the 129 MB L2 (inputs larger than L2), so steps run back to
back without an explicit flush; the same steps with a 256 MiB write before
each one (outside the CUDA-event interval) are reported beside them as
`value_l2_flushed`.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME [--batch B] [--context C]] [--sweep] [--profile-steps K]

With no workload flags: the Qwen3-8B-shaped step at batch 1, context 2048
(one JSON line).  --workload picks another workload of dflash2_synth
(qwen3_8b_b32_paged, qwen3_27b_b8, a3b_30b_fp8 with --batch/--context);
--sweep prints one line for each of the 8B batch-1 and batch-32 steps, the
27B step and the eight 30B-A3B fp8 sweep points.  --impl reference times
the CPU oracle (float64 numpy) on the same workload.  Multi-GPU (torchrun):
independent replicas, one per rank, no collective on the data path; the
timing is the max over ranks.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = "qwen3_8b_b1"
METRIC = "DFlash2 draft steps/s & proposed tokens/s at 8B shape; % of HBM/tensor roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20
SWEEP_STEPS = 300

FAMILY = {
    "qwen3_8b_b1": "Qwen3-8B-shaped draft",
    "qwen3_8b_b32_paged": "Qwen3-8B-shaped draft, batch 32 over a randomly paged cache",
    "qwen3_27b_b8": "27B-shaped draft",
    "a3b_30b_fp8": "30B-A3B-shaped draft, fp8-e4m3 weights with per-channel scales",
}


def args_(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=WORKLOAD)
    p.add_argument("--batch", type=int, default=0, help="batch override (30B-A3B sweep points)")
    p.add_argument("--context", type=int, default=0, help="context override (30B-A3B sweep points)")
    p.add_argument("--sweep", action="store_true", help="one line per workload and sweep point")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--attention", choices=["auto", "cluster", "tc"], default="auto",
                   help="attention kernel (a diagnostic switch through the test library): the library's "
                        "choice, the mma.sync cluster kernel, or the tcgen05 kernel wherever it applies")
    p.add_argument("--profile-steps", type=int, default=0,
                   help="for profiler captures: run this many eager steps after two warm-up steps, each inside "
                        "an NVTX range named 'step', and exit (no timing, no JSON line)")
    p.add_argument("--cpu-step-only", action="store_true", help=argparse.SUPPRESS)
    p.add_argument("--cpu-cap", type=int, default=1, help=argparse.SUPPRESS)
    p.add_argument("--cpu-budget", type=float, default=10.0, help=argparse.SUPPRESS)
    return p.parse_args(argv)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def config_for(workload, batch=0, context=0):
    import dflash2_synth as S
    over = {}
    if batch:
        over["batch"] = batch
    if context:
        over["context"] = context
    return S.config_of(workload, **over)


def dtype_name(cfg):
    return {"bf16": "bf16", "f32": "f32", "fp8w": "fp8-e4m3 weights (per-row fp32 scales), bf16 activations"}[
        cfg["dtype"]]


def workload_text(name, cfg):
    ctx = cfg["context"]
    ctx_s = f"{ctx[0]}..{ctx[1]} (uniform)" if isinstance(ctx, tuple) else str(ctx)
    return (f"{name}: {FAMILY.get(name, name)}, hidden {cfg['hidden']}, {cfg['n_q_heads']}q/{cfg['n_kv_heads']}kv x "
            f"{cfg['head_dim']}, MLP {cfg['intermediate']}, vocab {cfg['vocab']}, {cfg['n_layers']} draft layer(s), "
            f"{cfg['n_taps']} taps, block {cfg['block_size']}, top_k {cfg['top_k']}, rank {cfg['selector_rank']}, "
            f"batch {cfg['batch']}, context {ctx_s}")


# ---------------------------------------------------------------- model of the work

def work_model(cfg, ctx_after, n_new):
    """Algorithmic bytes and FLOPs of one step (b sequences), per the method:
    weights once, context K/V once, new taps, gathered embedding rows.
    fp8 weights count one byte per element plus a 4-byte scale per output
    row; activations and the cache are bf16 (fp32 for the fp32 workload).
    Returns (bytes, flops, lm_head bytes, lm_head flops)."""
    H, V, T = cfg["hidden"], cfg["vocab"], cfg["n_taps"]
    nq, nkv, d, I = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["intermediate"]
    L, B, k, r = cfg["n_layers"], cfg["block_size"], cfg["top_k"], cfg["selector_rank"]
    D = B - 1
    G = H // cfg["conv_group_size"]
    ctx_after, n_new = [int(c) for c in ctx_after], [int(n) for n in n_new]
    b = len(ctx_after)
    fp8 = cfg["dtype"] == "fp8w"
    ea = 4 if cfg["dtype"] == "f32" else 2        # activations, cache, embedding
    ew = 1 if fp8 else ea                          # weight matrices
    p_layer = H * (nq + 2 * nkv) * d + nq * d * H + 3 * H * I + 2 * (2 * G * H)
    rows_layer = (nq + 2 * nkv) * d + H + 2 * I + H + 2 * 2 * G
    w_bytes = (L * p_layer + T * H * H + V * H + 2 * r * H) * ew
    if fp8:
        w_bytes += 4 * (L * rows_layer + H + V + 2 * r)
    kv_tok = L * 2 * nkv * d * ea
    sum_ctx = sum(ctx_after)
    sum_new = sum(n_new)
    bytes_ = (w_bytes + (sum_ctx - sum_new) * kv_tok + sum_new * (T * H * ea + kv_tok)
              + b * (B + D * k + 1) * H * ea)
    flops = (2 * b * B * L * p_layer + 2 * sum_new * (T * H * H + L * 2 * H * nkv * d) + 2 * b * D * V * H
             + 2 * b * (D * k + 1) * 2 * r * H + L * sum(4 * B * nq * d * (c + B) for c in ctx_after))
    lm_bytes = V * H * ew + (4 * V if fp8 else 0) + b * D * H * ea
    lm_flops = 2 * b * D * V * H
    return bytes_, flops, lm_bytes, lm_flops


# ---------------------------------------------------------------- clocks

class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            out["reasons"] = ["nvidia-smi unavailable"]
            return out
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.f.name)
        if sm:
            out.update(sm_mhz=statistics.median(sm), sm_max_mhz=max(mx), samples=len(sm))
        out["reasons"] = sorted(reasons)
        return out


# ---------------------------------------------------------------- ranks

def max_over_ranks(x, device):
    """The largest x over the ranks of the default process group (x alone
    without one): the slowest replica sets the whole job's time."""
    import torch
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return x
    if torch.distributed.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(steps, world, max_total_ms):
    """Steps/s of the whole job: every replica ran `steps` steps of its own
    sequences (weak scaling), in at most max_total_ms."""
    return world * steps / (max_total_ms / 1e3)


# ---------------------------------------------------------------- our arm

LM_PROFILE = os.path.join(ROOT, "profiles", "lm_head_topk_qwen3_8b_b1.md")
LM_SOURCES = [os.path.join(ROOT, "block_speculative_decoding_dflash2_gb300", "csrc", f)
              for f in ("gemm_tc.cu", "common.cuh")]


def profiled_traffic(workload):
    """DRAM bytes (read + write) per lm_head launch from the committed ncu
    capture of this workload, or None when there is none or the kernel
    source changed since that capture."""
    import hashlib
    if workload != WORKLOAD:
        return None
    try:
        kv = dict(line.split(" = ", 1) for line in open(LM_PROFILE).read().splitlines() if " = " in line)
        h = hashlib.sha256(b"".join(open(f, "rb").read() for f in LM_SOURCES)).hexdigest()[:16]
        return int(kv["traffic_bytes_per_launch"]) if kv.get("source_digest", "").strip() == h else None
    except (OSError, KeyError, ValueError):
        return None


def step_inputs(cfg):
    """Context lengths (after this step's append), rows appended this step
    (B per sequence: the upper bound) and the lengths before it."""
    import numpy as np

    import dflash2_synth as S
    ctx = S.make_context_lengths(cfg)
    n_new = np.full(cfg["batch"], cfg["block_size"], dtype=np.int32)
    return ctx, n_new, (ctx - n_new).astype(np.int32)


def run_ours(a, cfg, name, rank, world, W=None):
    import numpy as np
    import torch

    import dflash2_synth as S
    from block_speculative_decoding_dflash2_gb300 import binding as Bd
    from block_speculative_decoding_dflash2_gb300.build import build
    from block_speculative_decoding_dflash2_gb300.runner import DraftRunner

    build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    b = cfg["batch"]
    B = cfg["block_size"]
    D = B - 1
    ctx, n_new, ctx_before = step_inputs(cfg)
    W = W if W is not None else S.make_weights(cfg)
    Wd = S.device_weights(W)
    bt, n_pages = S.paged_layout(int(ctx.max()) + B, cfg["page_size"], b, 1000 + cfg["index"])
    r = DraftRunner(cfg, Wd, b, int(ctx.max()) + B, max_new=max(int(ctx_before.max()), int(n_new.sum())),
                    block_table=torch.from_numpy(bt), n_pages=n_pages)
    r.build_selector_table()
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    # prefill (untimed): the committed context before this step, every
    # sequence from the same tap stream (its first ctx_before[s] rows), one
    # sequence per call so the host never holds a whole batch of taps
    pre = S.to_torch(S.make_taps(cfg, int(ctx_before.max()), stream="bench_prefill"))
    for s in range(b):
        off = np.zeros(b + 1, np.int32)
        off[s + 1:] = ctx_before[s]
        r.append(dev(np.zeros(b, np.int32)), pre[:int(ctx_before[s])].contiguous(), dev(off))
    torch.cuda.synchronize()
    del pre
    taps_h = S.make_taps(cfg, int(n_new.sum()), stream="bench_step")
    taps = S.to_torch(taps_h)
    new_off = dev(np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32))
    ctx_d = dev(ctx_before)
    anchor = dev(S.make_tokens(cfg, (b,), stream="bench_anchor"))
    target = dev(S.make_tokens(cfg, (b, B), stream="bench_target"))
    seq = torch.zeros(b, dtype=torch.int32, device="cuda")

    def step():
        r.draft(ctx_d, taps, new_off, anchor)
        r.select(anchor)
        r.verify(target, seq)

    if a.profile_steps:
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        for _ in range(a.profile_steps):
            torch.cuda.nvtx.range_push("step")
            step()
            torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        assert r.device_status() == 0
        return None, W

    # launches per step, from the library's own counter, on one eager step
    c0 = Bd.lib().dflash2_launch_count()
    step()
    torch.cuda.synchronize()
    launches_per_step = int(Bd.lib().dflash2_launch_count() - c0)
    assert r.device_status() == 0

    # Two graphs of the same step: `g` (timed) as a user captures it, and
    # `gs` with the library's stage events recorded inside it.  An event node
    # ends programmatic dependent launch at its boundary, so the stage and
    # lm_head durations come from `gs`, replayed between the timed steps.
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        step()                                       # warm the capture stream
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            step()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    keep = Bd.dflash2_set_stage_events(evs)  # noqa: F841  (keeps the events alive while gs exists)
    gs = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(gs, stream=s):
            step()
    Bd.lib().dflash2_set_stage_events(None)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    for _ in range(max(3, a.warmup)):
        flush.zero_()
        g.replay()
        flush.zero_()
        gs.replay()
    torch.cuda.synchronize()

    clk = Clocks(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clk.start()
    time.sleep(0.2)  # let the sampler start; the timed steps below run for about a second
    step_ms, lm_ms, stage_ms, flushed_ms = [], [], [[] for _ in range(4)], []
    for _ in range(a.steps):
        t0.record()
        g.replay()
        t1.record()
        t1.synchronize()
        step_ms.append(t0.elapsed_time(t1))
        gs.replay()
        evs[4].synchronize()
        lm_ms.append(evs[2].elapsed_time(evs[3]))
        for i in range(4):
            stage_ms[i].append(evs[i].elapsed_time(evs[i + 1]))
    for _ in range(a.steps):
        flush.zero_()
        t0.record()
        g.replay()
        t1.record()
        t1.synchronize()
        flushed_ms.append(t0.elapsed_time(t1))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.stop()
    total_ms = max_over_ranks(sum(step_ms), "cuda")
    flushed_total = max_over_ranks(sum(flushed_ms), "cuda")
    assert r.device_status() == 0

    # end to end through the public API with host buffers (pinned), per step:
    # one H2D copy of the step's packed inputs (taps, context lengths, row
    # offsets, anchors, target tokens), the three calls, one D2H copy of the
    # packed int32 results (path, accept lengths, output tokens, next anchors)
    ins = [taps, ctx_d, new_off, anchor, target]
    offs, total = [], 0
    for t in ins:
        offs.append(total)
        total += -(-t.numel() * t.element_size() // 256) * 256
    h_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_pack = torch.empty(total, dtype=torch.uint8, device="cuda")

    def view(buf, t, o):
        return buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)

    for t, o in zip(ins, offs):
        view(h_pack, t, o).copy_(t.cpu())
    d_taps, d_ctx, d_off, d_anchor, d_target = [view(d_pack, t, o) for t, o in zip(ins, offs)]
    h_res = torch.empty_like(r.results, device="cpu").pin_memory()
    h2d = total
    d2h = h_res.numel() * h_res.element_size()

    def e2e_step():
        d_pack.copy_(h_pack, non_blocking=True)
        r.draft(d_ctx, d_taps, d_off, d_anchor)
        r.select(d_anchor)
        r.verify(d_target, seq)
        h_res.copy_(r.results, non_blocking=True)

    # the caller captures the step, copies included, as one CUDA graph (the
    # calls are graph-capturable) and replays it every step; the eager loop
    # of the same calls is reported beside it
    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    ge = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        e2e_step()
        torch.cuda.synchronize()
        with torch.cuda.graph(ge, stream=s):
            e2e_step()
    for _ in range(3):
        ge.replay()
    torch.cuda.synchronize()
    e2e_ms, eager_ms = [], []
    for _ in range(a.steps):
        t0.record()
        ge.replay()
        t1.record()
        t1.synchronize()
        e2e_ms.append(t0.elapsed_time(t1))
    for _ in range(a.steps):
        t0.record()
        e2e_step()
        t1.record()
        t1.synchronize()
        eager_ms.append(t0.elapsed_time(t1))
    e2e_total = max_over_ranks(sum(e2e_ms), "cuda")
    eager_total = max_over_ranks(sum(eager_ms), "cuda")
    assert r.device_status() == 0

    pk, src = peaks()
    hbm, tc = pk["hbm_gbs"] * 1e9, pk["bf16_tflops"] * 1e12
    bytes_, flops, lm_bytes, lm_flops = work_model(cfg, [int(x) for x in ctx], [int(x) for x in n_new])
    lm_avg_s = statistics.mean(lm_ms) / 1e3
    step_s = total_ms / a.steps / 1e3
    steps_per_s = whole_job_rate(a.steps, world, total_ms)
    t_roof = max(bytes_ / hbm, flops / tc)
    # the lm_head's own bound: its weight bytes at HBM speed, or its FLOPs
    # on the bf16 tensor cores (fp8 weights are contracted as bf16 values)
    lm_hbm = lm_bytes / hbm >= lm_flops / tc
    if lm_hbm:
        roof = {"bound": "hbm", "achieved": lm_bytes / lm_avg_s / 1e9, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "algorithmic_bytes": lm_bytes, "peak_source": f"{src} (burst copy GB/s)"}
    else:
        roof = {"bound": "tensor", "achieved": lm_flops / lm_avg_s / 1e12, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "algorithmic_flops": lm_flops,
                "peak_source": f"{src} (burst cuBLAS bf16 TFLOP/s; the fp8 weights are contracted as bf16)"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = profiled_traffic(name)
    roof["kernel"] = "tc_gemm_kernel (lm_head + streaming top-k)"
    roof["avg_launch_us"] = lm_avg_s * 1e6
    res = {
        "metric": METRIC,
        "value": steps_per_s,
        "value_l2_flushed": whole_job_rate(a.steps, world, flushed_total),
        "unit": "draft steps/s",
        "n_gpus": world,
        "steps": a.steps,
        "warmup": max(3, a.warmup),
        "ms_per_step": total_ms / a.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_name(cfg),
        "data": "synthetic (seeded N(0,0.02) weights, RMS-normalised N(0,1) taps; no trained weights)",
        "config": {"workload": workload_text(name, cfg),
                   "batch": b, "context": int(ctx.max()), "new_rows_per_step": int(n_new.sum()),
                   "page_size": cfg["page_size"],
                   "graph": "one CUDA graph per step (stage and lm_head events from a second graph of the "
                            "same step, replayed between timed steps)",
                   "l2": f"inputs larger than L2: each step streams {bytes_ / 1e9:.2f} GB through the 129 MB L2; "
                         "no flush between steps (value_l2_flushed: a 256 MiB write before each step)",
                   "parallelism": f"replicas x{world}"},
        "proposed_tokens_per_s": steps_per_s * b * D,
        "stage_ms": {n: statistics.mean(v) for n, v in zip(
            ["append", "block_forward", "lm_head_topk", "topk_merge"], stage_ms)},
        "step_roofline": {"bytes": bytes_, "flops": flops,
                          "bound": "hbm" if bytes_ / hbm >= flops / tc else "tensor",
                          "t_roof_us": 1e6 * t_roof, "frac": t_roof / step_s},
        "roofline": roof,
        "clocks": clocks,
        "e2e": {"value": whole_job_rate(a.steps, world, e2e_total), "unit": "draft steps/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "dflash2_draft_step + dflash2_select_path_table + dflash2_verify_accept with the "
                       "H2D/D2H copies, captured once by the caller as a CUDA graph and replayed per step",
                "eager_value": whole_job_rate(a.steps, world, eager_total)},
        "gpu_launches": launches_per_step * a.steps,
        "gpu_launches_per_step": launches_per_step,
    }
    del g, gs, ge, r
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res, W


# ---------------------------------------------------------------- oracle (CPU)

def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def oracle_state(cfg, W, cap, random_context):
    """Inputs of an oracle step on the first `cap` sequences of the
    workload: the weights' values, the store, each sequence's context (from
    the prefill stream through the oracle's own append, or, with
    random_context, N(0,1) K/V arrays of the same shape, which the step's
    arithmetic does not depend on), the new taps, anchors and targets."""
    import numpy as np

    import dflash2_synth as S
    import oracle as O
    _, n_new, ctx_before = step_inputs(cfg)
    ctx_before, n_new = ctx_before[:cap], n_new[:cap]
    Wv = S.values_of(W)
    st = O.Store(cfg["dtype"] != "f32")
    nkv, d, L = cfg["n_kv_heads"], cfg["head_dim"], cfg["n_layers"]
    ctxs = []
    if random_context:
        g = np.random.default_rng(7)
        for P in ctx_before:
            ctxs.append([(g.standard_normal((int(P), nkv, d)), g.standard_normal((int(P), nkv, d)))
                         for _ in range(L)])
    else:
        pre = S.make_taps(cfg, int(ctx_before.max()), stream="bench_prefill")
        z = np.zeros((0, nkv, d))
        for P in ctx_before:
            ctxs.append(O.append_context(cfg, Wv, [(z, z)] * L, pre.values[:int(P)], 0, st))
    taps_step = S.make_taps(cfg, int(S.make_context_lengths(cfg).size) * cfg["block_size"], stream="bench_step")
    new, off = [], 0
    for n in n_new:
        new.append(taps_step.values[off:off + n])
        off += n
    anchor = S.make_tokens(cfg, (cfg["batch"],), stream="bench_anchor")[:cap]
    target = S.make_tokens(cfg, (cfg["batch"], cfg["block_size"]), stream="bench_target")[:cap]
    return Wv, st, ctxs, new, anchor, target


def oracle_step(cfg, Wv, st, ctxs, new, anchor, target):
    import oracle as O
    _, _, ids, vals = O.draft_step(cfg, Wv, ctxs, anchor, new, st)
    for s in range(len(anchor)):
        p, _, _ = O.select_path(cfg, Wv, int(anchor[s]), ids[s], vals[s])
        O.verify_accept(p, target[s])


def time_oracle(cfg, state, budget_s, max_steps=50):
    """Whole oracle steps of the capped batch, at least one, until about
    budget_s of CPU work; returns (steps, seconds)."""
    n, t_all = 0, 0.0
    while (t_all < budget_s or n == 0) and n < max_steps:
        t = time.perf_counter()
        oracle_step(cfg, *state)
        t_all += time.perf_counter() - t
        n += 1
    return n, t_all


def one_core_rate(a, cfg, name, cap):
    """The same oracle timing in a child process whose BLAS and OpenMP pools
    have one thread (the variables must be set before numpy loads)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1")
    cmd = [sys.executable, os.path.abspath(__file__), "--cpu-step-only", "--workload", name,
           "--batch", str(cfg["batch"]), "--cpu-cap", str(cap), "--cpu-budget", str(a.cpu_budget)]
    if not isinstance(cfg["context"], tuple):
        cmd += ["--context", str(cfg["context"])]
    try:
        out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=900)
        return json.loads(out.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError, OSError):
        return None


def cpu_baseline(a, cfg, name, W):
    """The oracle as it stands (float64 numpy, the precision it computes in),
    timed on this host's cores on whole draft+select+verify steps of a capped
    batch of the same workload (the context K/V are drawn instead of
    prefilled, except at batch 1, context 2048), then once more with one
    BLAS thread; steps/s of the full batch = capped steps/s * cap / batch."""
    b = cfg["batch"]
    cap = min(b, a.cpu_cap)
    random_ctx = not (name == WORKLOAD and b == 1)
    state = oracle_state(cfg, W, cap, random_ctx)
    n, t = time_oracle(cfg, state, a.cpu_budget)
    per_seq = t / (n * cap)
    one = one_core_rate(a, cfg, name, cap)
    sample = (f"{n} oracle step(s) of {cap} of the {b} sequences (float64 numpy; context "
              f"{'drawn' if random_ctx else 'prefilled through the oracle'}, untimed), {t:.1f} s; "
              f"steps/s of the whole batch = 1 / (seconds per sequence x {b})")
    out = {"value": 1.0 / (per_seq * b), "unit": "draft steps/s", "cores": cpu_cores(), "kind": "oracle",
           "sample": sample, "batch_cap": cap, "precision": "float64 (the oracle's own; no float32 path)"}
    if one is not None:
        out["one_core"] = {"value": one["value"], "cores": 1, "sample": one["sample"]}
    return out


def run_cpu_step_only(a):
    """Child process of one_core_rate: prints {"value", "sample"}."""
    import dflash2_synth as S
    cfg = config_for(a.workload, a.batch, a.context)
    W = S.make_weights(cfg)
    cap = min(cfg["batch"], a.cpu_cap)
    state = oracle_state(cfg, W, cap, True)
    n, t = time_oracle(cfg, state, a.cpu_budget)
    print(json.dumps({"value": 1.0 / (t / (n * cap) * cfg["batch"]),
                      "sample": f"{n} step(s) of {cap} sequence(s), one BLAS thread, context drawn, {t:.1f} s"}))
    return 0


def run_reference(a):
    import dflash2_synth as S
    cfg = config_for(a.workload, a.batch, a.context)
    W = S.make_weights(cfg)
    b = cfg["batch"]
    cap = min(b, a.cpu_cap)
    random_ctx = not (a.workload == WORKLOAD and b == 1)
    state = oracle_state(cfg, W, cap, random_ctx)
    budget = 150.0
    t = time.perf_counter()
    oracle_step(cfg, *state)                       # one warm-up step
    first = time.perf_counter() - t
    warm = 1
    steps = max(1, min(a.steps, int(budget / max(first, 1e-3))))
    t = time.perf_counter()
    for _ in range(steps):
        oracle_step(cfg, *state)
    total = time.perf_counter() - t
    v = steps * cap / (total * b)
    sample = (f"{steps} whole oracle steps of {cap} of the {b} sequences (of {a.steps} requested; capped to "
              f"~{budget:.0f} s) after {warm} warm-up step, float64 numpy oracle")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "draft steps/s", "n_gpus": 1,
            "steps": steps, "warmup": warm, "ms_per_step": 1e3 / v, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_text(a.workload, cfg), "batch": b},
            "cpu_baseline": {"value": v, "unit": "draft steps/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "draft steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def sweep_points():
    import dflash2_synth as S
    pts = [("qwen3_8b_b1", 0, 0), ("qwen3_8b_b32_paged", 0, 0), ("qwen3_27b_b8", 0, 0)]
    return pts + [("a3b_30b_fp8", bb, cc) for bb, cc in S.A3B_SWEEP]


def main():
    a = args_()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if a.cpu_step_only:
        return run_cpu_step_only(a)
    if a.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(a)))
        return 0
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl")
    if a.attention != "auto":
        from block_speculative_decoding_dflash2_gb300 import binding as B
        B.dflash2_test_force_attention({"cluster": 1, "tc": 2}[a.attention])
    points = sweep_points() if a.sweep else [(a.workload, a.batch, a.context)]
    if a.sweep and "--steps" not in sys.argv:
        a.steps = SWEEP_STEPS
    W, W_name = None, None
    for name, bb, cc in points:
        cfg = config_for(name, bb, cc)
        res, W = run_ours(a, cfg, name, rank, world, W if W_name == name else None)
        W_name = name
        if res is None:  # --profile-steps
            continue
        if rank == 0 and not a.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(a, cfg, name, W)
        if rank == 0:
            print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
