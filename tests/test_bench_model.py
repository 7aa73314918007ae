"""bench.work_model, the algorithmic bytes and FLOPs behind every roofline
fraction the bench reports, against figures stated independently of it.

The step's bytes are the weights read once, the committed context K/V read
once, the new taps and their K/V, and the gathered embedding rows; fp8
weights count one byte per element plus a 4-byte scale per output row.  The
per-workload totals below were worked out by hand from the workload shapes
(Qwen3-8B-, 27B- and 30B-A3B-shaped drafts) and are quoted at the precision
they were worked to.  They take the workload's context length as the
positions committed before the step, the step appending B more rows per
sequence (the bench's own lines count the context after the append; the two
differ by B rows of K/V per sequence).
"""

import pytest

import bench
import dflash2_synth as S

# (workload, overrides, step bytes in GB and its last printed digit)
STEP_BYTES = [
    ("qwen3_8b_b1", {}, 1.746, 1e-3),
    ("qwen3_8b_b32_paged", {}, 2.07, 1e-2),
    ("qwen3_27b_b8", {}, 2.68, 1e-2),
    ("a3b_30b_fp8", dict(batch=1, context=1024), 0.56, 1e-2),
    ("a3b_30b_fp8", dict(batch=64, context=1024), 0.87, 1e-2),
    ("a3b_30b_fp8", dict(batch=256, context=1024), 1.81, 1e-2),
    ("a3b_30b_fp8", dict(batch=256, context=8192), 9.33, 1e-2),
]


def _model(name, **over):
    cfg = S.config_of(name, **over)
    ctx, n_new, _ = bench.step_inputs(cfg)
    return cfg, ctx, n_new, bench.work_model(cfg, ctx, n_new)


@pytest.mark.parametrize("name,over,gb,digit", STEP_BYTES, ids=[f"{w}-{o}" for w, o, _, _ in STEP_BYTES])
def test_step_bytes_match_the_hand_worked_totals(name, over, gb, digit):
    cfg, ctx, n_new, _ = _model(name, **over)
    nbytes = bench.work_model(cfg, ctx + n_new, n_new)[0]
    assert abs(nbytes / 1e9 - gb) <= digit / 2, nbytes


def test_lm_head_bytes_and_flops_exact():
    # the 8B lm_head reads its 151936 x 4096 bf16 weights once and the 7 normed
    # rows of one sequence; 2 FLOPs per weight and row
    _, _, _, (_, flops, lm_bytes, lm_flops) = _model("qwen3_8b_b1")
    assert lm_bytes == 151936 * 4096 * 2 + 7 * 4096 * 2 == 1_244_717_056
    assert lm_flops == 2 * 7 * 151936 * 4096
    assert abs(flops / 1e9 - 13.2) <= 0.05
    # fp8: one byte per weight plus a float32 scale per vocabulary row
    _, _, _, (_, _, lm8, _) = _model("a3b_30b_fp8", batch=1, context=1024)
    assert lm8 == 131072 * 2688 + 4 * 131072 + 6 * 2688 * 2


def test_each_context_key_adds_its_k_and_v_once_per_layer():
    for name, over in [("qwen3_8b_b1", {}), ("a3b_30b_fp8", dict(batch=1, context=1024))]:
        cfg, ctx, n_new, (b0, f0, _, _) = _model(name, **over)
        b1, f1, _, _ = bench.work_model(cfg, [int(ctx[0]) + 1], n_new)
        kv_tok = cfg["n_layers"] * 2 * cfg["n_kv_heads"] * cfg["head_dim"] * 2
        assert b1 - b0 == kv_tok
        # and one more key for every query row of every layer's attention
        assert f1 - f0 == cfg["n_layers"] * 4 * cfg["block_size"] * cfg["n_q_heads"] * cfg["head_dim"]


def test_weights_are_counted_once_per_step_whatever_the_batch():
    cfg, _, _, _ = _model("qwen3_8b_b1")
    one = bench.work_model(cfg, [2048], [8])[0]
    two = bench.work_model(cfg, [2048, 2048], [8, 8])[0]
    # a second identical sequence adds its own context, taps and embedding
    # rows, never the weights again
    per_seq = two - one
    assert 0 < per_seq < 0.02 * one
    assert bench.work_model(cfg, [2048] * 3, [8] * 3)[0] - two == per_seq
