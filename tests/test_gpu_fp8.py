"""The fp8-weight path (DFLASH2_FP8W: e4m3 matrices with per-row scales,
bf16 activations): draft-step parity with the oracle on the dequantised
weights, stage by stage and end to end, the selector and verify on the
GPU's lattice, and the lossless loop; at a small shape and at the
30B-A3B-shaped sweep points."""

import functools

import numpy as np
import pytest

import dflash2_synth as S
import oracle as O
from tests.helpers import TOL, Case, e2e_tol, lib, record_near_ties, topk_compare
from tests.test_gpu_draft import check_case
from tests.test_gpu_full_configs import check_select_and_verify
from tests.test_gpu_stagewise import run_stagewise

pytestmark = pytest.mark.gpu


def small_fp8(**over):
    return S.small_bf16_config(dtype="fp8w", **over)


def test_fp8_small_one_layer_stagewise():
    cfg = small_fp8(n_layers=1, index=21)
    case = Case(cfg, ctx_lens=[60, 0, 150], n_new=[3, 8, 1], seed=21).run_gpu()
    assert case.status == 0
    run_stagewise(case)
    check_case(case)


def test_fp8_small_two_layers_ragged_batch():
    cfg = small_fp8(index=22)
    case = Case(cfg, ctx_lens=[40, 0, 200], n_new=[1, 8, 3], seed=22).run_gpu()
    check_case(case)
    check_select_and_verify(case, [0, 1, 2], None, "fp8 small, two layers")


def test_fp8_small_wide_batch_unfused_paths():
    # 10 sequences: activation tiles wider than the fused epilogues take
    cfg = small_fp8(n_q_heads=8, index=23)
    ctx = [5, 17, 40, 0, 64, 3, 31, 90, 12, 8]
    case = Case(cfg, ctx_lens=ctx, n_new=[1, 2, 8, 3, 0, 5, 1, 4, 2, 6], seed=23).run_gpu()
    check_case(case)


def test_fp8_select_paths_agree():
    """The selector on fp8 W_sel: the per-step contraction and the factor
    table give the oracle's path on the GPU's lattice."""
    cfg = small_fp8(index=24)
    case = Case(cfg, ctx_lens=[30, 77], n_new=[4, 4], seed=24).run_gpu()
    assert case.status == 0
    r = case.runner
    anchor = case.dev(case.anchor)
    r.select(anchor)
    p_gemm = r.path.cpu().numpy().copy()
    r.build_selector_table()
    r.select(anchor)
    p_table = r.path.cpu().numpy()
    cid, cz = r.cand_id.cpu().numpy(), r.cand_logit.cpu().numpy().astype(np.float64)
    for s in range(case.b):
        p, _, _ = O.select_path(cfg, case.Wv, int(case.anchor[s]), cid[s], cz[s])
        assert list(p_gemm[s]) == list(p) and list(p_table[s]) == list(p)


@functools.lru_cache(maxsize=1)
def a3b_weights():
    return S.make_weights(S.config_of("a3b_30b_fp8"))


@pytest.mark.slow
@pytest.mark.parametrize("batch,context", S.A3B_SWEEP)
def test_a3b_30b_fp8_sweep_point(batch, context):
    """Every 30B-A3B sweep point at full size (2 layers, vocab 131072, block
    7, batch x context up to 256 x 8192): end to end against the oracle on
    sampled sequences, the top-k of every sequence from the GPU's own logits
    bit-exact, selector and verify on the GPU's lattice.

    Input recipe: the sampled sequences' contexts are their own tap streams;
    every other sequence's context is one shared stream of the same length
    (its content only has to exist), appended per sequence, so the host never
    holds the whole batch's taps."""
    import torch
    from block_speculative_decoding_dflash2_gb300.runner import DraftRunner
    cfg = S.config_of("a3b_30b_fp8", batch=batch, context=context)
    B_, k = cfg["block_size"], cfg["top_k"]
    L = context - B_                                   # context before this step's B appended rows
    seqs = sorted({0, batch // 2, batch - 1})
    W = a3b_weights()
    Wv = S.values_of(W)
    bt, n_pages = S.paged_layout(context + 1, cfg["page_size"], batch, 60 + batch)
    r = DraftRunner(cfg, S.device_weights(W), batch, context + 1, max_new=max(L, batch * B_),
                    block_table=torch.from_numpy(bt), n_pages=n_pages)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    shared = S.to_torch(S.make_taps(cfg, L, stream="a3b_shared"))
    own = {s: S.make_taps(cfg, L, stream=f"a3b_seq{s}") for s in seqs}
    zeros = np.zeros(batch, np.int32)
    for s in range(batch):                              # one sequence's context per call
        off = np.zeros(batch + 1, np.int32)
        off[s + 1:] = L
        r.append(dev(zeros), S.to_torch(own[s]) if s in own else shared, dev(off))
    del shared
    step = S.make_taps(cfg, batch * B_, stream="a3b_step")
    anchor = S.make_tokens(cfg, (batch,), stream="a3b_anchor")
    debug = torch.full((batch, B_ - 1, cfg["vocab"]), float("nan"), device="cuda")
    r.draft(dev(np.full(batch, L)), S.to_torch(step), dev(np.arange(batch + 1) * B_), dev(anchor), debug)
    torch.cuda.synchronize()
    assert r.device_status() == 0
    cid = r.cand_id.cpu().numpy()
    dbg = debug[seqs].double().cpu().numpy()
    for i, s in enumerate(seqs):                        # the GPU's own top-k, bit for bit
        ids, vals = O.topk(debug[s].double().cpu().numpy(), k)
        np.testing.assert_array_equal(cid[s], ids)
        np.testing.assert_array_equal(r.cand_logit[s].cpu().numpy(), vals.astype(np.float32))
    st = O.Store(True)
    z = []
    for s in seqs:
        ctx = O.append_context(cfg, Wv, [(np.zeros((0, cfg["n_kv_heads"], cfg["head_dim"])),) * 2
                                         for _ in range(cfg["n_layers"])], own[s].values, 0, st)
        ctx = O.append_context(cfg, Wv, ctx, step.values[s * B_:(s + 1) * B_], L, st)
        z.append(O.draft_block(cfg, Wv, int(anchor[s]), ctx, st))
    z = np.stack(z)
    err = np.max(np.abs(dbg - z))
    tol = e2e_tol(f"a3b_30b_fp8_ctx{context}")  # the bf16 pipeline's rounding-chaos floor, measured
    assert err <= tol, f"max |logit - oracle| = {err} (bound {tol})"
    near = topk_compare(cid[seqs], z, k, tol)
    print(f"[parity] fp8w b={batch} ctx={context} sampled {seqs}: max|dlogit|={err:.3e} near-tie rows={near}")
    record_near_ties(f"a3b_30b_fp8 b={batch} ctx={context}", "top-k rows", near, len(seqs) * (B_ - 1))
    # selector (factor table) and verify on the GPU's lattice, every sequence
    r.build_selector_table()
    r.select(dev(anchor))
    path = r.path.cpu().numpy()
    cz = r.cand_logit.cpu().numpy().astype(np.float64)
    near = 0
    for s in range(batch):
        p, _, sc = O.select_path(cfg, Wv, int(anchor[s]), cid[s], cz[s])
        if list(path[s]) != list(p):
            gi = [list(cid[s, i]).index(path[s, i]) for i in range(B_ - 1)]
            assert sc - O.path_score(cfg, Wv, int(anchor[s]), cid[s], cz[s], gi) < 1e-4
            near += 1
    record_near_ties(f"a3b_30b_fp8 b={batch} ctx={context}", "selector paths", near, batch)
    assert near <= max(1, batch // 8)
    target = S.make_agreeing_target(path, cfg, 0.7)
    seq = dev(np.full(batch, context))
    r.verify(dev(target), seq)
    acc = r.accept_len.cpu().numpy()
    for s in range(batch):
        assert acc[s] == O.verify_accept(path[s], target[s])[0]
    assert r.device_status() == 0
