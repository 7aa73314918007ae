"""Writes bf16_chaos_floor.txt: how far the oracle's own bf16-storage logits
move when its weights are nudged by one part in a million.

The bf16 pipeline rounds its activations to bf16 at every storage point
(the feature rows, the context K/V, each sublayer's normed and convolved
rows, q/k/v, the attention output, the MLP activation, the final-normed
rows).  A relative perturbation of 1e-6 of the weights, the size of the
difference between fp32 and fp64 accumulation, moves a few pre-rounding
values across a bf16 rounding boundary; the flipped roundings propagate
through the layers and the attention.  The largest logit change this causes
is a floor under any end-to-end comparison of two correct implementations
of the same bf16 pipeline that accumulate in different orders or
precisions.

For every full-size end-to-end case of the GPU tests (the same workload,
sequences, context lengths and input streams), this script computes the
oracle's logits of the sampled sequences with the weights as drawn and
with every weight element w replaced by w * (1 + 1e-6 * e), e = +-1 drawn
per element (two independent draws), and records the largest absolute
logit change.  It calls the oracle and the input generators only.

  python tests/golden/make_bf16_chaos_floor.py [case ...]
"""

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import dflash2_synth as S  # noqa: E402
import oracle as O  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "bf16_chaos_floor.txt")
NUDGE = 1e-6
DRAWS = 2


def _case_inputs(cfg, ctx_lens, n_new, seed, seqs):
    """The per-sequence prefill rows, new rows and anchors of the test
    harness's Case (streams prefill{seed}, step{seed}, anchor{seed})."""
    ctx_lens = np.asarray(ctx_lens)
    n_new = np.asarray(n_new)
    pre = S.make_taps(cfg, int(ctx_lens.sum()), stream=f"prefill{seed}").values
    new = S.make_taps(cfg, int(n_new.sum()), stream=f"step{seed}").values
    anchor = S.make_tokens(cfg, (len(ctx_lens),), stream=f"anchor{seed}")
    p0 = np.concatenate([[0], np.cumsum(ctx_lens)])
    n0 = np.concatenate([[0], np.cumsum(n_new)])
    return [(pre[p0[s]:p0[s] + ctx_lens[s]], new[n0[s]:n0[s] + n_new[s]], int(ctx_lens[s]), int(anchor[s]))
            for s in seqs]


def _a3b_inputs(cfg, batch, context, seqs):
    """The 30B-A3B sweep test's sampled sequences: own context streams
    a3b_seq{s}, the step rows of stream a3b_step, anchors a3b_anchor."""
    B = cfg["block_size"]
    L = context - B
    step = S.make_taps(cfg, batch * B, stream="a3b_step").values
    anchor = S.make_tokens(cfg, (batch,), stream="a3b_anchor")
    return [(S.make_taps(cfg, L, stream=f"a3b_seq{s}").values, step[s * B:(s + 1) * B], L, int(anchor[s]))
            for s in seqs]


def _logits(cfg, Wv, inputs):
    st = O.Store(True)
    z0 = [(np.zeros((0, cfg["n_kv_heads"], cfg["head_dim"])),) * 2 for _ in range(cfg["n_layers"])]
    out = []
    for pre, new, L, anchor in inputs:
        ctx = O.append_context(cfg, Wv, z0, pre, 0, st) if L else z0
        ctx = O.append_context(cfg, Wv, ctx, new, L, st)
        out.append(O.draft_block(cfg, Wv, anchor, ctx, st))
    return np.stack(out)


def _nudged(Wv, rng):
    def one(a):
        a = np.asarray(a, dtype=np.float64)
        return a * (1.0 + NUDGE * (2.0 * rng.integers(0, 2, size=a.shape) - 1.0))
    out = {k: one(v) for k, v in Wv.items() if k != "layers"}
    out["layers"] = [{k: one(v) for k, v in L.items()} for L in Wv["layers"]]
    return out


def cases():
    c8 = S.config_of("qwen3_8b_b1")
    c8w = S.config_of("qwen3_8b_b1", sliding_window=512)
    c32 = S.config_of("qwen3_8b_b32_paged")
    c27 = S.config_of("qwen3_27b_b8")
    ca = S.config_of("a3b_30b_fp8")
    ctx32 = S.make_context_lengths(c32) - c32["block_size"]
    ctx27 = S.make_context_lengths(c27) - c27["block_size"]
    return {
        # test_gpu_draft: the 8B shape at batch 1
        "qwen3_8b_b1": (c8, lambda: _case_inputs(c8, [2040], [8], 21, [0])),
        # test_gpu_variants: the same shape with a 512-key window
        "qwen3_8b_b1_window512": (c8w, lambda: _case_inputs(c8w, [2040], [8], 32, [0])),
        # test_gpu_full_configs: sampled sequences of the batch-32 and 27B steps
        "qwen3_8b_b32_paged": (c32, lambda: _case_inputs(c32, ctx32, np.full(32, 8), 31, [0, 13, 31])),
        "qwen3_27b_b8": (c27, lambda: _case_inputs(c27, ctx27, np.full(8, 16), 41, [5])),
        # test_gpu_fp8: the 30B-A3B sweep's sampled sequence 0, both contexts
        "a3b_30b_fp8_ctx1024": (dict(ca, batch=1, context=1024), lambda: _a3b_inputs(ca, 1, 1024, [0])),
        "a3b_30b_fp8_ctx8192": (dict(ca, batch=1, context=8192), lambda: _a3b_inputs(ca, 1, 8192, [0])),
    }


def floor_of(name):
    cfg, make_inputs = cases()[name]
    W = S.values_of(S.make_weights(cfg))
    inputs = make_inputs()
    z = _logits(cfg, W, inputs)
    worst = 0.0
    for d in range(DRAWS):
        zn = _logits(cfg, _nudged(W, np.random.default_rng(1000 + d)), inputs)
        worst = max(worst, float(np.max(np.abs(zn - z))))
    return worst


def main(names):
    rows = {}
    if os.path.exists(OUT):
        for line in open(OUT):
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = [f.strip() for f in line.split("|")]
                rows[k] = v
    for name in names or list(cases()):
        f = floor_of(name)
        rows[name] = f"{f:.6f}"
        print(name, rows[name], flush=True)
    with open(OUT, "w") as fh:
        fh.write("# Largest |logit change| of the oracle's bf16-storage logits under +-1e-6 relative weight\n"
                 "# nudges (two draws), per full-size end-to-end test case.  Written by\n"
                 "# make_bf16_chaos_floor.py (oracle and input generators only); the GPU tests hold each case\n"
                 "# to max(2e-2, 1.6 x this floor).\n"
                 "# case | floor\n")
        for k in cases():
            if k in rows:
                fh.write(f"{k} | {rows[k]}\n")


if __name__ == "__main__":
    main(sys.argv[1:])
