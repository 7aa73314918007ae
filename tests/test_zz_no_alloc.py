"""dflash2_select_path_static: the selector for callers that cannot allocate
device memory (it uses the library's fixed scratch array instead of a
caller workspace).  Its output must equal dflash2_select_path's on the same
inputs, call after call, and a batch beyond the fixed scratch must be refused.

Collected last on purpose, so a run that stops at its first failure has run
every other test before it; it also passes alone in a fresh process.
"""

import numpy as np
import pytest

import dflash2_synth as S
from tests.helpers import lib

pytestmark = pytest.mark.gpu


def _inputs(cfg, b, seed):
    g = np.random.default_rng(seed)
    D, k, V = cfg["block_size"] - 1, cfg["top_k"], cfg["vocab"]
    cand = np.stack([np.stack([g.choice(V - 1, size=k, replace=False) for _ in range(D)]) for _ in range(b)])
    z = -np.sort(-g.standard_normal((b, D, k)).astype(np.float32), axis=2)
    anchor = g.integers(0, V - 1, size=b).astype(np.int32)
    return anchor, cand.astype(np.int32), z


@pytest.mark.parametrize("name,b", [("qwen3_8b_b1", 1), ("qwen3_8b_b1", 8), ("tiny_fp32", 3)])
def test_static_selector_matches_workspace_selector(name, b):
    import torch
    B = lib()
    cfg = S.config_of(name)
    W = S.make_weights(cfg)
    w = B.WeightSet({"embed": S.to_torch(W["embed"]), "sel": S.to_torch(W["sel"]), "lm_head": None, "fc": None,
                     "hidden_norm": None, "final_norm": None, "layers": []})
    c = B.make_config(cfg)
    D = cfg["block_size"] - 1
    ws = torch.zeros(B.dflash2_workspace_size(c, b, 0, 16), dtype=torch.uint8, device="cuda")
    for call in range(2):  # two calls in a row: the shared scratch must not carry state over
        anchor, cand, z = _inputs(cfg, b, seed=100 * b + call)
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        p_ref = torch.full((b, D), -3, dtype=torch.int32, device="cuda")
        s_ref = torch.zeros(b, dtype=torch.float32, device="cuda")
        p_st = torch.full((b, D), -5, dtype=torch.int32, device="cuda")
        s_st = torch.zeros(b, dtype=torch.float32, device="cuda")
        B.dflash2_select_path(c, w, b, dev(anchor), dev(cand), dev(z), p_ref, s_ref, ws)
        B.dflash2_select_path_static(c, w, b, dev(anchor), dev(cand), dev(z), p_st, s_st)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(p_st.cpu().numpy(), p_ref.cpu().numpy())
        np.testing.assert_allclose(s_st.cpu().numpy(), s_ref.cpu().numpy(), rtol=1e-5, atol=1e-5)


def test_static_selector_refuses_batches_beyond_its_scratch():
    import torch
    B = lib()
    cfg = S.config_of("qwen3_8b_b1", vocab=4096, index=30)
    W = S.make_weights(dict(cfg, n_layers=1))
    w = B.WeightSet({"embed": S.to_torch(W["embed"]), "sel": S.to_torch(W["sel"]), "lm_head": None, "fc": None,
                     "hidden_norm": None, "final_norm": None, "layers": []})
    c = B.make_config(cfg)
    assert B.dflash2_select_path_static_capacity() == 8 << 20
    b = 9  # 9 * 113 gathered rows of hidden 4096 exceed 8 MiB
    anchor, cand, z = _inputs(cfg, b, seed=7)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    path = torch.zeros((b, cfg["block_size"] - 1), dtype=torch.int32, device="cuda")
    with pytest.raises(B.DFlash2Error) as e:
        B.dflash2_select_path_static(c, w, b, dev(anchor), dev(cand), dev(z), path, None)
    assert e.value.status == -5


def test_static_selector_reports_a_bad_token_id():
    # an anchor outside the vocabulary is flagged in the fixed array's status
    # word (its gathered row reads as zeros); the read clears it, and a clean
    # call afterwards reports nothing
    import torch
    B = lib()
    cfg = S.config_of("tiny_fp32")
    W = S.make_weights(cfg)
    w = B.WeightSet({"embed": S.to_torch(W["embed"]), "sel": S.to_torch(W["sel"]), "lm_head": None, "fc": None,
                     "hidden_norm": None, "final_norm": None, "layers": []})
    c = B.make_config(cfg)
    b, D = 2, cfg["block_size"] - 1
    anchor, cand, z = _inputs(cfg, b, seed=11)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    path = torch.zeros((b, D), dtype=torch.int32, device="cuda")
    score = torch.zeros(b, dtype=torch.float32, device="cuda")
    B.dflash2_select_path_static_read_status()
    bad = anchor.copy()
    bad[1] = cfg["vocab"] + 5
    B.dflash2_select_path_static(c, w, b, dev(bad), dev(cand), dev(z), path, score)
    assert B.dflash2_select_path_static_read_status() == 0x2   # DFLASH2_DEV_BAD_TOKEN
    assert B.dflash2_select_path_static_read_status() == 0
    B.dflash2_select_path_static(c, w, b, dev(anchor), dev(cand), dev(z), path, score)
    assert B.dflash2_select_path_static_read_status() == 0
