"""The rows ranked next after the core path: DFlash (v1) drafting (no
convolution, per-position top-1 selection) and the sliding-window context
(draft_sliding_window), each against the oracle stage by stage and end to
end, on the tensor-core attention (bf16) and the SIMT attention (fp32)."""

import numpy as np
import pytest

import dflash2_synth as S
import oracle as O
from tests.helpers import Case, e2e_tol, lib
from tests.test_gpu_draft import check_case
from tests.test_gpu_stagewise import run_stagewise

pytestmark = pytest.mark.gpu


def test_dflash_v1_no_conv_stagewise_and_end_to_end():
    cfg = S.small_bf16_config(conv_kernel_size=0, n_layers=1, index=25)
    case = Case(cfg, ctx_lens=[60, 0, 150], n_new=[3, 8, 1], seed=25).run_gpu()
    assert case.status == 0
    run_stagewise(case)
    check_case(case)


def test_dflash_v1_two_layers_and_fp32():
    check_case(Case(S.small_bf16_config(conv_kernel_size=0, index=26), ctx_lens=[40, 7], n_new=[2, 8],
                    seed=26).run_gpu())
    check_case(Case(S.config_of("tiny_fp32", conv_kernel_size=0), ctx_lens=[128], n_new=[8], seed=27).run_gpu())


@pytest.mark.parametrize("window", [1, 16, 37, 200])
def test_sliding_window_bf16(window):
    # contexts shorter and longer than the window, ends mid-page, one empty
    cfg = S.small_bf16_config(sliding_window=window, n_layers=1, index=28)
    case = Case(cfg, ctx_lens=[60, 0, 150], n_new=[3, 8, 1], seed=28).run_gpu()
    assert case.status == 0
    run_stagewise(case)
    check_case(case)


def test_sliding_window_fp32_and_two_layers():
    check_case(Case(S.config_of("tiny_fp32", sliding_window=50), ctx_lens=[120], n_new=[8], seed=29).run_gpu())
    check_case(Case(S.small_bf16_config(sliding_window=33, index=30), ctx_lens=[90, 12], n_new=[4, 4],
                    seed=30).run_gpu())


@pytest.mark.slow
def test_sliding_window_qwen3_8b_shape():
    # the 8B shape with a 512-key window over a 2048-key context
    cfg = S.config_of("qwen3_8b_b1", sliding_window=512)
    case = Case(cfg, ctx_lens=[2040], n_new=[8], seed=32).run_gpu()
    run_stagewise(case)
    check_case(case, tol=e2e_tol("qwen3_8b_b1_window512"), name="qwen3_8b_b1_window512")


@pytest.mark.parametrize("n_max,p_min", [(0, 0.0), (4, 0.0), (0, 0.3), (7, 0.6), (10, 0.3)])
def test_top1_selection_with_knobs(n_max, p_min):
    """dflash2_select_top1: the per-position top-1 path, cut by the softmax
    of the candidate logits (the oracle's selector without its pairwise
    term)."""
    import torch
    B = lib()
    V, k, D, b = 500, 4, 7, 32
    cfg = S.small_bf16_config(vocab=V, top_k=k, block_size=D + 1, index=33)
    g = np.random.default_rng(33)
    cand = np.stack([np.stack([g.choice(V - 1, size=k, replace=False) for _ in range(D)]) for _ in range(b)])
    z = -np.sort(-g.standard_normal((b, D, k)).astype(np.float32), axis=2)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    c = B.make_config(cfg)
    path = torch.full((b, D), -5, dtype=torch.int32, device="cuda")
    score = torch.zeros(b, dtype=torch.float32, device="cuda")
    nd = torch.full((b,), -5, dtype=torch.int32, device="cuda")
    B.dflash2_select_top1(c, b, dev(cand.astype(np.int32)), dev(z), n_max, p_min, path, score, nd)
    torch.cuda.synchronize()
    path, score, nd = path.cpu().numpy(), score.cpu().numpy(), nd.cpu().numpy()
    W0 = {"embed": np.zeros((V, 8)), "sel": np.zeros((2 * cfg["selector_rank"], 8))}
    for s in range(b):
        p, idx, sc = O.select_path_knobs(dict(cfg, hidden=8), W0, 0, cand[s], z[s].astype(np.float64), n_max, p_min)
        probs = np.exp(z[s].astype(np.float64))[:, 0] / np.exp(z[s].astype(np.float64)).sum(1)
        if p_min > 0 and np.any(np.abs(probs - p_min) < 1e-5):
            continue
        assert nd[s] == len(p) and list(path[s, :len(p)]) == list(p) and np.all(path[s, len(p):] == -1)
        assert list(idx) == [0] * len(p)
        assert abs(score[s] - sc) < 1e-4 * max(1.0, abs(sc))
