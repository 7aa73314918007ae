#!/usr/bin/env python
"""Benchmark of the DFlash2 draft step on GB300: draft steps/s and proposed
tokens/s at the Qwen3-8B draft shape (batch 1, context 2048, block 8), with
the roofline fraction of the dominant kernel (the lm_head contraction with
its fused top-k).

One step = dflash2_draft_step + dflash2_select_path_table +
dflash2_verify_accept (feature projection of 8 new committed positions, paged
K/V append, one non-causal block forward, lm_head + top-k, selector, verify),
captured as one CUDA graph.  The selector's per-token factor table is built
once at setup, like the weights themselves (it is a function of the frozen
embedding and selector weights only).  Inputs are resident in HBM.  Every
step streams 1.75 GB of weights through the 129 MB L2 (inputs larger than
L2), so steps run back to back without an explicit flush; the same steps
with a 256 MiB write before each one (outside the CUDA-event interval) are
reported beside them as `value_l2_flushed`.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (float64 numpy) on the same workload.
Multi-GPU (torchrun): independent replicas, one per rank, no collective on
the data path; the timing is the max over ranks.
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


def args_():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=WORKLOAD)
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------- model of the work

def work_model(cfg, ctx_after, n_new):
    """Algorithmic bytes and FLOPs of one step (b sequences), per the method:
    weights once, context K/V once, new taps, gathered embedding rows."""
    H, V, T = cfg["hidden"], cfg["vocab"], cfg["n_taps"]
    nq, nkv, d, I = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["intermediate"]
    L, B, k, r = cfg["n_layers"], cfg["block_size"], cfg["top_k"], cfg["selector_rank"]
    D = B - 1
    G = H // cfg["conv_group_size"]
    b = len(ctx_after)
    es = 2 if cfg["dtype"] == "bf16" else 4
    p_layer = H * (nq + 2 * nkv) * d + nq * d * H + 3 * H * I + 2 * (2 * G * H)
    w_elems = L * p_layer + T * H * H + V * H + 2 * r * H
    kv_tok = L * 2 * nkv * d * es
    sum_ctx = sum(ctx_after)
    sum_new = sum(n_new)
    bytes_ = (w_elems * es + (sum_ctx - sum_new) * kv_tok + sum_new * (T * H * es + kv_tok)
              + b * (B + D * k + 1) * H * es)
    flops = (2 * b * B * L * p_layer + 2 * sum_new * (T * H * H + L * 2 * H * nkv * d) + 2 * b * D * V * H
             + 2 * b * (D * k + 1) * 2 * r * H + L * sum(4 * B * nq * d * (c + B) for c in ctx_after))
    lm_bytes = V * H * es + b * D * H * es
    return bytes_, flops, lm_bytes


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

LM_PROFILE = os.path.join(ROOT, "profiles", "lm_head_topk_qwen3_8b_b1.txt")
LM_SOURCES = [os.path.join(ROOT, "block_speculative_decoding_dflash2_gb300", "csrc", f)
              for f in ("gemm_tc.cu", "common.cuh")]


def profiled_traffic():
    """DRAM bytes (read + write) per lm_head launch from the committed ncu
    capture, or None when the kernel source changed since that capture."""
    import hashlib
    try:
        kv = dict(line.split(" = ", 1) for line in open(LM_PROFILE).read().splitlines() if " = " in line)
        h = hashlib.sha256(b"".join(open(f, "rb").read() for f in LM_SOURCES)).hexdigest()[:16]
        return int(kv["traffic_bytes_per_launch"]) if kv.get("source_digest", "").strip() == h else None
    except (OSError, KeyError, ValueError):
        return None


def run_ours(a, rank, world):
    import numpy as np
    import torch

    import dflash2_synth as S
    from block_speculative_decoding_dflash2_gb300 import binding as Bd
    from block_speculative_decoding_dflash2_gb300.build import build
    from block_speculative_decoding_dflash2_gb300.runner import DraftRunner

    build()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    cfg = S.config_of(a.workload)
    b = cfg["batch"]
    ctx = S.make_context_lengths(cfg)
    B = cfg["block_size"]
    D = B - 1
    n_new = np.full(b, B, dtype=np.int32)            # n_b = B committed rows per step (upper bound)
    ctx_before = (ctx - n_new).astype(np.int32)      # context after the append = ctx
    W = S.make_weights(cfg)
    Wd = S.device_weights(W)
    bt, n_pages = S.paged_layout(int(ctx.max()) + B, cfg["page_size"], b, 1000 + cfg["index"])
    r = DraftRunner(cfg, Wd, b, int(ctx.max()) + B, max_new=int(ctx_before.sum()),
                    block_table=torch.from_numpy(bt), n_pages=n_pages)
    r.build_selector_table()
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    # prefill (untimed): the committed context before this step
    pre = S.make_taps(cfg, int(ctx_before.sum()), stream="bench_prefill")
    r.append(dev(np.zeros(b, np.int32)), S.to_torch(pre),
             dev(np.concatenate([[0], np.cumsum(ctx_before)]).astype(np.int32)))
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

    pk, src = peaks()
    bytes_, flops, lm_bytes = work_model(cfg, [int(x) for x in ctx], [int(x) for x in n_new])
    lm_avg_s = statistics.mean(lm_ms) / 1e3
    step_s = total_ms / a.steps / 1e3
    lm_ach = lm_bytes / lm_avg_s / 1e9
    steps_per_s = whole_job_rate(a.steps, world, total_ms)
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
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights, RMS-normalised N(0,1) taps; no trained weights)",
        "config": {"workload": f"{a.workload}: Qwen3-8B-shaped draft, hidden {cfg['hidden']}, "
                               f"{cfg['n_q_heads']}q/{cfg['n_kv_heads']}kv x {cfg['head_dim']}, MLP "
                               f"{cfg['intermediate']}, vocab {cfg['vocab']}, 1 layer, 3 taps, block "
                               f"{B}, top_k {cfg['top_k']}, rank {cfg['selector_rank']}",
                   "batch": b, "context": int(ctx.max()), "new_rows_per_step": int(n_new.sum()),
                   "page_size": cfg["page_size"], "graph": "one CUDA graph per step (stage and lm_head events from a second graph of the same step, replayed between timed steps)",
                   "l2": "inputs larger than L2: each step streams 1.75 GB of weights through the 129 MB L2; "
                         "no flush between steps (value_l2_flushed: a 256 MiB write before each step)",
                   "parallelism": f"replicas x{world}"},
        "proposed_tokens_per_s": steps_per_s * b * D,
        "stage_ms": {n: statistics.mean(v) for n, v in zip(
            ["append", "block_forward", "lm_head_topk", "topk_merge"], stage_ms)},
        "step_roofline": {"bytes": bytes_, "flops": flops, "bound": "hbm",
                          "t_roof_us": 1e6 * max(bytes_ / (pk["hbm_gbs"] * 1e9),
                                                 flops / (pk["bf16_tflops"] * 1e12)),
                          "frac": max(bytes_ / (pk["hbm_gbs"] * 1e9),
                                      flops / (pk["bf16_tflops"] * 1e12)) / step_s},
        "roofline": {"bound": "hbm", "achieved": lm_ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": lm_ach / pk["hbm_gbs"], "traffic": profiled_traffic(),
                     "kernel": "tc_gemm_kernel<16,1> (lm_head + streaming top-k)",
                     "algorithmic_bytes": lm_bytes, "avg_launch_us": lm_avg_s * 1e6,
                     "peak_source": f"{src} (burst copy GB/s)"},
        "clocks": clocks,
        "e2e": {"value": whole_job_rate(a.steps, world, e2e_total), "unit": "draft steps/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "dflash2_draft_step + dflash2_select_path_table + dflash2_verify_accept with the "
                       "H2D/D2H copies, captured once by the caller as a CUDA graph and replayed per step",
                "eager_value": whole_job_rate(a.steps, world, eager_total)},
        "gpu_launches": launches_per_step * a.steps,
        "gpu_launches_per_step": launches_per_step,
    }
    if rank == 0 and not a.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(cfg, W, ctx_before, n_new, taps_h, budget_s=20.0)
    return res


# ---------------------------------------------------------------- oracle (CPU)

def oracle_state(cfg, W, ctx_before, n_new, taps_step):
    import numpy as np

    import dflash2_synth as S
    import oracle as O
    Wv = S.values_of(W)
    st = O.Store(cfg["dtype"] == "bf16")
    pre = S.make_taps(cfg, int(ctx_before.sum()), stream="bench_prefill")
    ctxs, off = [], 0
    z = np.zeros((0, cfg["n_kv_heads"], cfg["head_dim"]))
    for L in ctx_before:
        ctxs.append(O.append_context(cfg, Wv, [(z, z)] * cfg["n_layers"], pre.values[off:off + L], 0, st))
        off += L
    new, off = [], 0
    for n in n_new:
        new.append(taps_step.values[off:off + n])
        off += n
    anchor = S.make_tokens(cfg, (len(ctx_before),), stream="bench_anchor")
    target = S.make_tokens(cfg, (len(ctx_before), cfg["block_size"]), stream="bench_target")
    return Wv, st, ctxs, new, anchor, target


def oracle_step(cfg, Wv, st, ctxs, new, anchor, target):
    import oracle as O
    _, _, ids, vals = O.draft_step(cfg, Wv, ctxs, anchor, new, st)
    for s in range(len(anchor)):
        p, _, _ = O.select_path(cfg, Wv, int(anchor[s]), ids[s], vals[s])
        O.verify_accept(p, target[s])


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_baseline(cfg, W, ctx_before, n_new, taps_step, budget_s=20.0):
    """The oracle as it stands, timed on this host on whole steps of the same
    workload until about budget_s of CPU work."""
    state = oracle_state(cfg, W, ctx_before, n_new, taps_step)
    n, t_all = 0, 0.0
    while t_all < budget_s and n < 50:
        t = time.perf_counter()
        oracle_step(cfg, *state)
        t_all += time.perf_counter() - t
        n += 1
    return {"value": n / t_all, "unit": "draft steps/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{n} whole draft+select+verify steps of the same workload (float64 numpy, "
                      f"context prefilled untimed), {t_all:.1f} s"}


def run_reference(a):
    import numpy as np

    import dflash2_synth as S
    cfg = S.config_of(a.workload)
    ctx = S.make_context_lengths(cfg)
    B = cfg["block_size"]
    n_new = np.full(cfg["batch"], B, dtype=np.int32)
    ctx_before = (ctx - n_new).astype(np.int32)
    W = S.make_weights(cfg)
    taps_h = S.make_taps(cfg, int(n_new.sum()), stream="bench_step")
    state = oracle_state(cfg, W, ctx_before, n_new, taps_h)
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
    v = steps / total
    sample = (f"{steps} whole steps (of {a.steps} requested; capped to ~{budget:.0f} s) after {warm} "
              f"warm-up step, float64 numpy oracle")
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "draft steps/s", "n_gpus": 1,
            "steps": steps, "warmup": warm, "ms_per_step": 1e3 * total / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": a.workload, "batch": cfg["batch"], "context": int(ctx.max())},
            "cpu_baseline": {"value": v, "unit": "draft steps/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": v, "unit": "draft steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    a = args_()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if a.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(a)))
        return 0
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group("nccl")
    res = run_ours(a, rank, world)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
