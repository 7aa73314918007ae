"""Times the widened variants of the draft step at the Qwen3-8B shape
(batch 1, block 8, top-16): each variant's whole step captured once as a
CUDA graph and replayed; inputs are larger than L2, so replays run back to
back without a flush.  Prints the mean and median step time per variant.

  python -m block_speculative_decoding_dflash2_gb300.variant_bench [--replays 300]

Variants:
  dflash2    draft + selector on the factor table + greedy verify (the bench step)
  knobs      the same with draft_n_max = 3 and draft_p_min = 0.3 (the _ex
             selector and verify)
  v1         DFlash (v1): no convolution around the sublayers, the
             per-position top-1 path (dflash2_select_top1)
  ctx8k      context 8192, every key of the prefix
  window512  context 8192, sliding window of 512 context keys
  sampled    draft + selector + lossless sampled verification against
             target distributions over the whole vocabulary
and, alone, the sampled verification kernel (back-to-back launches).

Weights, taps and tokens are the seeded synthetic inputs of dflash2_synth
(run from the repository root); no parity is checked here.
"""

import argparse

import numpy as np
import torch

import dflash2_synth as S

from . import binding as B
from .build import build
from .runner import DraftRunner


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


class Setup:
    """A runner of one config over shared device weights, its context
    prefilled, and the step's inputs on the device."""

    def __init__(self, cfg, Wd):
        self.cfg = cfg
        b, Bk = cfg["batch"], cfg["block_size"]
        ctx = S.make_context_lengths(cfg)
        n_new = np.full(b, Bk, dtype=np.int32)
        ctx_before = (ctx - n_new).astype(np.int32)
        bt, n_pages = S.paged_layout(int(ctx.max()) + Bk, cfg["page_size"], b, 1000 + cfg["index"])
        self.r = DraftRunner(cfg, Wd, b, int(ctx.max()) + Bk, max_new=int(ctx_before.sum()),
                             block_table=torch.from_numpy(bt), n_pages=n_pages)
        self.r.build_selector_table()
        pre = S.make_taps(cfg, int(ctx_before.sum()), stream="bench_prefill")
        self.r.append(_dev(np.zeros(b, np.int32)), S.to_torch(pre),
                      _dev(np.concatenate([[0], np.cumsum(ctx_before)]).astype(np.int32)))
        del pre
        self.taps = S.to_torch(S.make_taps(cfg, int(n_new.sum()), stream="bench_step"))
        self.new_off = _dev(np.concatenate([[0], np.cumsum(n_new)]).astype(np.int32))
        self.ctx = _dev(ctx_before)
        self.anchor = _dev(S.make_tokens(cfg, (b,), stream="bench_anchor"))
        self.target = _dev(S.make_tokens(cfg, (b, Bk), stream="bench_target"))
        self.seq = torch.zeros(b, dtype=torch.int32, device="cuda")
        self.n_draft = torch.zeros(b, dtype=torch.int32, device="cuda")

    def draft(self):
        self.r.draft(self.ctx, self.taps, self.new_off, self.anchor)


def time_graph(step, replays):
    step()
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        step()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(20):
        g.replay()
    ms = []
    for _ in range(replays):
        e0.record()
        g.replay()
        e1.record()
        e1.synchronize()
        ms.append(e0.elapsed_time(e1))
    torch.cuda.synchronize()
    return 1e3 * float(np.mean(ms)), 1e3 * float(np.median(ms))


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--replays", type=int, default=300)
    a = p.parse_args()
    build()
    base = S.config_of("qwen3_8b_b1")
    Wd = S.device_weights(S.make_weights(base))
    out = []

    def report(name, us):
        out.append((name, us))
        print(f"{name:10s} {us[0]:8.1f} us mean  {us[1]:8.1f} us median per step", flush=True)

    st = Setup(base, Wd)
    r = st.r
    b, Bk, V = base["batch"], base["block_size"], base["vocab"]

    def step_dflash2():
        st.draft()
        r.select(st.anchor)
        r.verify(st.target, st.seq)
    report("dflash2", time_graph(step_dflash2, a.replays))

    def step_knobs():
        st.draft()
        B.dflash2_select_path_table_ex(r.cfg, b, st.anchor, r.cand_id, r.cand_logit, r.sel_table, 3, 0.3, r.path,
                                       r.path_score, st.n_draft, r.workspace)
        B.dflash2_verify_accept_ex(b, Bk, r.path, st.n_draft, st.target, r.accept_len, r.out_tok, r.n_out,
                                   r.next_anchor, st.seq, r.counters)
    report("knobs", time_graph(step_knobs, a.replays))

    prob = torch.from_numpy(S.make_target_probs(b * Bk, V, 7)).cuda().view(b, Bk, V)
    g = np.random.default_rng(7)
    u_acc = _dev(g.random((b, Bk - 1)).astype(np.float32))
    u_smp = _dev(g.random(b).astype(np.float32))

    def verify_sampled():
        B.dflash2_verify_sampled(b, Bk, V, r.path, None, prob, u_acc, u_smp, r.accept_len, r.out_tok, r.n_out,
                                 r.next_anchor, st.seq, r.counters)

    def step_sampled():
        st.draft()
        r.select(st.anchor)
        verify_sampled()
    report("sampled", time_graph(step_sampled, a.replays))
    verify_sampled()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(100):
        verify_sampled()
    e1.record()
    e1.synchronize()
    print(f"verify_sampled kernel alone: {e0.elapsed_time(e1) * 10:.1f} us per call (back to back, "
          f"V = {V}, {b} sequence(s))", flush=True)
    del st, r, prob

    v1 = Setup(S.config_of("qwen3_8b_b1", conv_kernel_size=0), Wd)

    def step_v1():
        v1.draft()
        rv = v1.r
        B.dflash2_select_top1(rv.cfg, b, rv.cand_id, rv.cand_logit, 0, 0.0, rv.path, rv.path_score, v1.n_draft,
                              rv.workspace)
        B.dflash2_verify_accept_ex(b, Bk, rv.path, v1.n_draft, v1.target, rv.accept_len, rv.out_tok, rv.n_out,
                                   rv.next_anchor, v1.seq, rv.counters)
    report("v1", time_graph(step_v1, a.replays))
    del v1

    for name, over in (("ctx8k", dict(context=8192)), ("window512", dict(context=8192, sliding_window=512))):
        w = Setup(S.config_of("qwen3_8b_b1", **over), Wd)

        def step_w(w=w):
            w.draft()
            w.r.select(w.anchor)
            w.r.verify(w.target, w.seq)
        report(name, time_graph(step_w, a.replays))
        del w
    return out


if __name__ == "__main__":
    main()
