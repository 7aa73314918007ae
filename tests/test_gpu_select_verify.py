"""Parity of the selector (factor gather + GEMM + Viterbi, or the per-token
factor table + Viterbi) and of greedy verify/accept/rollback with the oracle,
on identical inputs."""

import math

import numpy as np
import pytest

import dflash2_synth as S
import oracle as O
from tests.conftest import read_golden
from tests.helpers import lib, record_near_ties

pytestmark = pytest.mark.gpu


def sel_cfg(dtype, V, H, k, D, r):
    return dict(hidden=H, n_q_heads=2, n_kv_heads=2, head_dim=64, intermediate=64, vocab=V, n_layers=1,
                n_taps=1, block_size=D + 1, conv_kernel_size=2, conv_group_size=H, top_k=k,
                selector_rank=r, page_size=16, mask_token_id=V - 1, dtype=dtype, rms_eps=1e-6,
                rope_theta=1e6, input_embedding_scale=1.0, output_multiplier=1.0,
                final_logit_softcap=0.0)


def run_select(dtype, V, H, k, D, r, b, seed, emb_std=1.0, sel_std=0.3, logit_std=1.0, kind="gemm"):
    import torch
    B = lib()
    cfg = sel_cfg(dtype, V, H, k, D, r)
    E = S._draw(seed, "E", (V, H), emb_std / np.sqrt(H), dtype)
    Wsel = S._draw(seed, "sel", (2 * r, H), sel_std, dtype)
    g = np.random.default_rng(seed)
    cand = np.stack([np.stack([g.choice(V - 1, size=k, replace=False) for _ in range(D)]) for _ in range(b)])
    z = -np.sort(-g.standard_normal((b, D, k)).astype(np.float32) * logit_std, axis=2)
    anchor = g.integers(0, V - 1, size=b).astype(np.int32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    w = B.WeightSet({"embed": S.to_torch(E), "sel": S.to_torch(Wsel), "lm_head": None, "fc": None,
                     "hidden_norm": None, "final_norm": None, "layers": []})
    c = B.make_config(cfg)
    ws = torch.zeros(B.dflash2_workspace_size(c, b, 0, 16), dtype=torch.uint8, device="cuda")
    path = torch.full((b, D), -5, dtype=torch.int32, device="cuda")
    score = torch.zeros(b, dtype=torch.float32, device="cuda")
    if kind == "table":
        table = torch.empty(B.dflash2_selector_table_bytes(c) // 4, dtype=torch.float32, device="cuda")
        B.dflash2_build_selector_table(c, w, table)
        B.dflash2_select_path_table(c, b, dev(anchor), dev(cand.astype(np.int32)), dev(z), table, path, score, ws)
    else:
        B.dflash2_select_path(c, w, b, dev(anchor), dev(cand.astype(np.int32)), dev(z), path, score, ws)
    torch.cuda.synchronize()
    assert B.dflash2_read_device_status(ws) == 0
    Wo = {"embed": E.values, "sel": Wsel.values}
    return cfg, Wo, anchor, cand, z, path.cpu().numpy(), score.cpu().numpy()


@pytest.mark.parametrize("kind", ["gemm", "table"])
@pytest.mark.parametrize("dtype,V,H,k,D,r,b", [
    ("bf16", 4096, 256, 16, 7, 64, 4),
    ("bf16", 2000, 128, 4, 7, 16, 3),
    ("bf16", 151936, 4096, 16, 7, 64, 2),
    ("bf16", 5000, 512, 16, 15, 64, 2),
    ("f32", 4096, 256, 4, 7, 16, 3),
    # degenerate lattices: one candidate per position (the single path), one
    # draft position (the anchor's transitions only), both
    ("bf16", 1000, 128, 1, 7, 16, 3),
    ("bf16", 1000, 128, 4, 1, 16, 3),
    ("bf16", 1000, 128, 1, 1, 16, 3),
    # the largest rank (128) and the largest block (31 positions)
    ("bf16", 5000, 512, 16, 7, 128, 2),
    ("bf16", 2000, 128, 8, 31, 32, 2),
])
def test_selector_matches_oracle_viterbi(dtype, V, H, k, D, r, b, kind):
    cfg, W, anchor, cand, z, path, score = run_select(dtype, V, H, k, D, r, b, seed=V + k, kind=kind)
    near = 0
    for s in range(b):
        p, idx, sc = O.select_path(cfg, W, int(anchor[s]), cand[s], z[s].astype(np.float64))
        assert abs(score[s] - sc) < 1e-3 * max(1.0, abs(sc))
        if list(path[s]) != list(p):
            # a different path is allowed only if the oracle scores it within 1e-4
            gi = [list(cand[s, i]).index(path[s, i]) for i in range(D)]
            alt = O.path_score(cfg, W, int(anchor[s]), cand[s], z[s].astype(np.float64), gi)
            assert sc - alt < 1e-4, (s, list(path[s]), list(p))
            near += 1
    record_near_ties(f"selector {dtype} V={V} H={H} k={k} D={D} r={r} b={b} ({kind})", "selector paths", near, b)
    assert near <= max(1, b // 4)


@pytest.mark.parametrize("kind", ["gemm", "table"])
def test_selector_pairwise_term_matters_and_brute_force(kind):
    # strong factors so paths leave the per-position argmax; k=4, D=7 brute force
    cfg, W, anchor, cand, z, path, score = run_select("bf16", 1000, 128, 4, 7, 16, 6, seed=3,
                                                      emb_std=3.0, sel_std=1.0, logit_std=0.5, kind=kind)
    moved = 0
    for s in range(6):
        pb, idxb, sb = O.brute_force_path(cfg, W, int(anchor[s]), cand[s], z[s].astype(np.float64))
        assert list(path[s]) == list(pb)
        assert abs(score[s] - sb) < 1e-3 * max(1.0, abs(sb))
        moved += int(np.any(idxb != 0))
    assert moved > 0


@pytest.mark.parametrize("kind", ["gemm", "table"])
def test_selector_without_pairwise_term_is_top1(kind):
    cfg, W, anchor, cand, z, path, score = run_select("bf16", 1000, 128, 8, 7, 16, 3, seed=4, sel_std=0.0,
                                                      kind=kind)
    np.testing.assert_array_equal(path, cand[:, :, 0])


@pytest.mark.parametrize("dtype,V,H,r", [("bf16", 151936, 4096, 64), ("bf16", 1000, 128, 16),
                                         ("f32", 4096, 256, 16)])
def test_selector_table_rows_are_the_factors(dtype, V, H, r):
    """Sampled rows of the table against the oracle's factors of those tokens
    (W_a E[v], W_b E[v] in float64), every row's finiteness, and the ragged
    last tile of the vocabulary."""
    import torch
    B = lib()
    cfg = sel_cfg(dtype, V, H, 4, 7, r)
    E = S._draw(7, "E", (V, H), 1.0 / np.sqrt(H), dtype)
    Wsel = S._draw(7, "sel", (2 * r, H), 0.3, dtype)
    w = B.WeightSet({"embed": S.to_torch(E), "sel": S.to_torch(Wsel), "lm_head": None, "fc": None,
                     "hidden_norm": None, "final_norm": None, "layers": []})
    c = B.make_config(cfg)
    n = B.dflash2_selector_table_bytes(c) // 4
    assert n == V * 2 * r
    table = torch.full((n,), float("nan"), dtype=torch.float32, device="cuda")
    B.dflash2_build_selector_table(c, w, table)
    t = table.view(V, 2 * r).cpu().numpy()
    assert np.all(np.isfinite(t))
    rows = np.unique(np.concatenate([np.random.default_rng(1).integers(0, V, 64), [0, V - 1, V - 2]]))
    A, Bf = O.selector_factors(cfg, {"embed": E.values, "sel": Wsel.values}, rows)
    ref = np.concatenate([A, Bf], axis=1)
    tol = 1e-4 if dtype == "f32" else 2e-3
    np.testing.assert_allclose(t[rows], ref, atol=tol, rtol=0)


def test_selector_table_flags_bad_tokens():
    import torch
    B = lib()
    V, H, k, D, r, b = 1000, 128, 4, 7, 16, 2
    cfg = sel_cfg("bf16", V, H, k, D, r)
    E = S._draw(9, "E", (V, H), 1.0 / np.sqrt(H), "bf16")
    Wsel = S._draw(9, "sel", (2 * r, H), 0.3, "bf16")
    w = B.WeightSet({"embed": S.to_torch(E), "sel": S.to_torch(Wsel), "lm_head": None, "fc": None,
                     "hidden_norm": None, "final_norm": None, "layers": []})
    c = B.make_config(cfg)
    table = torch.empty(B.dflash2_selector_table_bytes(c) // 4, dtype=torch.float32, device="cuda")
    B.dflash2_build_selector_table(c, w, table)
    ws = torch.zeros(B.dflash2_workspace_size(c, b, 0, 16), dtype=torch.uint8, device="cuda")
    cand = torch.arange(b * D * k, dtype=torch.int32, device="cuda").reshape(b, D, k)
    z = torch.zeros((b, D, k), dtype=torch.float32, device="cuda")
    anchor = torch.tensor([3, V + 7], dtype=torch.int32, device="cuda")
    path = torch.zeros((b, D), dtype=torch.int32, device="cuda")
    B.dflash2_select_path_table(c, b, anchor, cand, z, table, path, None, ws)
    torch.cuda.synchronize()
    assert B.dflash2_read_device_status(ws) & B.DEV_BAD_TOKEN
    # without a workspace the call still runs (no status word to flag)
    B.dflash2_select_path_table(c, b, anchor, cand, z, table, path, None, None)
    torch.cuda.synchronize()


@pytest.mark.parametrize("kind", ["gemm", "table"])
@pytest.mark.parametrize("n_max,p_min", [(3, 0.0), (7, 0.2), (5, 0.35), (1, 0.0), (7, 0.99), (0, 0.5),
                                         (12, 0.35)])
def test_selector_drafting_knobs_match_oracle(kind, n_max, p_min):
    """draft_n_max / draft_p_min: the walk over positions 1..n_max and the
    cut at the first low-confidence transition, against the oracle on the
    same lattice (paths, kept counts exactly; scores to 1e-3).  A request
    above B-1 drafts is clamped to B-1."""
    import torch
    B = lib()
    V, H, k, D, r, b = 1000, 128, 4, 7, 16, 16
    cfg = sel_cfg("bf16", V, H, k, D, r)
    # factors and logits of comparable size: the pairwise term moves every
    # path off the per-position top-1, and chosen transitions span the
    # thresholds (at p_min 0.35 / 0.5 / 0.99 the oracle cuts 6 / 16 / 16 of
    # the 16 paths)
    E = S._draw(31, "E", (V, H), 1.0 / np.sqrt(H), "bf16")
    Wsel = S._draw(31, "sel", (2 * r, H), 0.3, "bf16")
    g = np.random.default_rng(31)
    cand = np.stack([np.stack([g.choice(V - 1, size=k, replace=False) for _ in range(D)]) for _ in range(b)])
    z = -np.sort(-g.standard_normal((b, D, k)).astype(np.float32), axis=2)
    anchor = g.integers(0, V - 1, size=b).astype(np.int32)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    w = B.WeightSet({"embed": S.to_torch(E), "sel": S.to_torch(Wsel), "lm_head": None, "fc": None,
                     "hidden_norm": None, "final_norm": None, "layers": []})
    c = B.make_config(cfg)
    ws = torch.zeros(B.dflash2_workspace_size(c, b, 0, 16), dtype=torch.uint8, device="cuda")
    path = torch.full((b, D), -5, dtype=torch.int32, device="cuda")
    score = torch.zeros(b, dtype=torch.float32, device="cuda")
    nd = torch.full((b,), -5, dtype=torch.int32, device="cuda")
    args = (dev(anchor), dev(cand.astype(np.int32)), dev(z))
    if kind == "table":
        table = torch.empty(B.dflash2_selector_table_bytes(c) // 4, dtype=torch.float32, device="cuda")
        B.dflash2_build_selector_table(c, w, table)
        B.dflash2_select_path_table_ex(c, b, *args, table, n_max, p_min, path, score, nd, ws)
    else:
        B.dflash2_select_path_ex(c, w, b, *args, n_max, p_min, path, score, nd, ws)
    torch.cuda.synchronize()
    path, score, nd = path.cpu().numpy(), score.cpu().numpy(), nd.cpu().numpy()
    Wo = {"embed": E.values, "sel": Wsel.values}
    cut = 0
    for s in range(b):
        zs = z[s].astype(np.float64)
        p, idx, sc = O.select_path_knobs(cfg, Wo, int(anchor[s]), cand[s], zs, n_max, p_min)
        n = len(p)
        t = O.transition_logprobs(cfg, Wo, int(anchor[s]), cand[s], zs, idx)
        walk = O.select_path_knobs(cfg, Wo, int(anchor[s]), cand[s], zs, n_max)[1]   # before the cut
        probs = np.exp(O.transition_logprobs(cfg, Wo, int(anchor[s]), cand[s], zs, walk))
        if p_min > 0 and np.any(np.abs(probs - p_min) < 1e-4):
            continue  # a transition on the threshold: fp32 and fp64 may decide it differently
        assert nd[s] == n, (s, nd[s], n)
        assert list(path[s, :n]) == list(p) and np.all(path[s, n:] == -1)
        assert abs(score[s] - sc) < 1e-3 * max(1.0, abs(sc))
        cut += int(n < (min(n_max, D) or D))
        assert np.all(t >= math.log(p_min) - 1e-9) if p_min > 0 else True
    if p_min in (0.35, 0.5, 0.99):
        assert cut > 0  # the lattice really exercises the cut


def test_verify_with_fewer_drafts_matches_oracle():
    import torch
    B = lib()
    g = np.random.default_rng(77)
    b, B_ = 400, 8
    D = B_ - 1
    nd = g.integers(0, D + 1, b)
    paths = g.integers(0, 3, (b, D))
    paths = np.where(np.arange(D)[None, :] < nd[:, None], paths, -1)
    targets = g.integers(0, 3, (b, B_))
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    acc = torch.full((b,), -9, dtype=torch.int32, device="cuda")
    out = torch.full((b, B_), -9, dtype=torch.int32, device="cuda")
    n_out = torch.zeros(b, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(b, dtype=torch.int32, device="cuda")
    seq = dev(np.zeros(b))
    counters = torch.zeros(4 + 2 * B_ - 1, dtype=torch.int64, device="cuda")
    B.dflash2_verify_accept_ex(b, B_, dev(paths), dev(nd), dev(targets), acc, out, n_out, nxt, seq, counters)
    torch.cuda.synchronize()
    acc, out, nxt, seq = acc.cpu().numpy(), out.cpu().numpy(), nxt.cpu().numpy(), seq.cpu().numpy()
    cnt = O.Counters(D)
    for s in range(b):
        a, toks, na = O.verify_accept(paths[s, :nd[s]], targets[s])
        cnt.add(a, int(nd[s]))
        assert acc[s] == a and nxt[s] == na and seq[s] == a + 1
        assert list(out[s, :a + 1]) == toks and np.all(out[s, a + 1:] == -1)
    c = counters.cpu().numpy()
    assert c[0] == cnt.steps and c[1] == cnt.drafted and c[2] == cnt.accepted and c[3] == cnt.rollback
    np.testing.assert_array_equal(c[4:4 + B_], cnt.hist)
    np.testing.assert_array_equal(c[4 + B_:], cnt.acc_pos)


@pytest.mark.parametrize("V,B_,b", [(1000, 8, 64), (151936, 8, 16), (5000, 16, 32)])
def test_sampled_verify_matches_oracle(V, B_, b):
    """Sampled (temperature > 0) verification against the oracle on the same
    target distributions and draws: accept lengths and counters exactly; the
    emitted token exactly, or, where fp32 and fp64 cumulative sums straddle
    the draw's threshold, a token the fp64 inverse CDF also admits."""
    import torch
    B = lib()
    D = B_ - 1
    g = np.random.default_rng(V + B_)
    prob = S.make_target_probs(b * B_, V, seed=V + B_).reshape(b, B_, V)
    # proposals: each position's most likely token, a kept token, or any token
    pick = g.random((b, D))
    best = prob[:, :D].argmax(axis=2)
    kept = np.array([[g.choice(np.nonzero(prob[s, i])[0]) for i in range(D)] for s in range(b)])
    paths = np.where(pick < 0.6, best, np.where(pick < 0.85, kept, g.integers(0, V, (b, D))))
    nd = np.where(g.random(b) < 0.7, D, g.integers(0, D + 1, b))
    paths = np.where(np.arange(D)[None, :] < nd[:, None], paths, -1)
    ua = g.random((b, D)).astype(np.float32)
    us = g.random(b).astype(np.float32)
    dev = lambda a, dt=np.int32: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).cuda()
    acc = torch.full((b,), -9, dtype=torch.int32, device="cuda")
    out = torch.full((b, B_), -9, dtype=torch.int32, device="cuda")
    n_out = torch.zeros(b, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(b, dtype=torch.int32, device="cuda")
    seq = dev(np.zeros(b))
    counters = torch.zeros(4 + 2 * B_ - 1, dtype=torch.int64, device="cuda")
    B.dflash2_verify_sampled(b, B_, V, dev(paths), dev(nd), dev(prob, np.float32), dev(ua, np.float32),
                             dev(us, np.float32), acc, out, n_out, nxt, seq, counters)
    torch.cuda.synchronize()
    acc, out, nxt, seq = acc.cpu().numpy(), out.cpu().numpy(), nxt.cpu().numpy(), seq.cpu().numpy()
    cnt = O.Counters(D)
    straddle = 0
    for s in range(b):
        a, toks, na = O.verify_sampled(paths[s, :nd[s]], prob[s], ua[s], us[s])
        cnt.add(a, int(nd[s]))
        assert acc[s] == a and seq[s] == a + 1
        assert list(out[s, :a]) == toks[:a] and np.all(out[s, a + 1:] == -1) and out[s, a] == nxt[s]
        if nxt[s] != na:
            row = prob[s, a].astype(np.float64).copy()
            if a < nd[s]:
                row[paths[s, a]] = 0.0
            cdf = np.cumsum(row)
            thr = float(us[s]) * cdf[-1]
            v = int(nxt[s])
            lo = cdf[v - 1] if v > 0 else 0.0
            assert row[v] > 0 and lo <= thr * (1 + 1e-5) + 1e-7 and cdf[v] >= thr * (1 - 1e-5) - 1e-7, (s, v, na)
            straddle += 1
    assert straddle <= max(1, b // 16)
    c = counters.cpu().numpy()
    assert c[0] == cnt.steps and c[1] == cnt.drafted and c[2] == cnt.accepted and c[3] == cnt.rollback
    np.testing.assert_array_equal(c[4:4 + B_], cnt.hist)
    np.testing.assert_array_equal(c[4 + B_:], cnt.acc_pos)
    assert 0 < cnt.accepted < cnt.drafted  # both outcomes occur


def test_sampled_verify_is_greedy_at_temperature_zero():
    # one-hot target rows: the sampled rule reduces to the greedy one
    import torch
    B = lib()
    g = np.random.default_rng(90)
    b, B_, V = 128, 8, 300
    D = B_ - 1
    target = g.integers(0, V, (b, B_))
    paths = np.where(g.random((b, D)) < 0.7, target[:, :D], g.integers(0, V, (b, D)))
    prob = np.zeros((b, B_, V), dtype=np.float32)
    np.put_along_axis(prob, target[:, :, None], 1.0, axis=2)
    dev = lambda a, dt=np.int32: torch.from_numpy(np.ascontiguousarray(a, dtype=dt)).cuda()
    outs = [torch.zeros(b, dtype=torch.int32, device="cuda"), torch.zeros((b, B_), dtype=torch.int32, device="cuda"),
            torch.zeros(b, dtype=torch.int32, device="cuda"), torch.zeros(b, dtype=torch.int32, device="cuda")]
    B.dflash2_verify_sampled(b, B_, V, dev(paths), None, dev(prob, np.float32),
                             dev(g.random((b, D)), np.float32), dev(g.random(b), np.float32), *outs)
    torch.cuda.synchronize()
    acc, out, _, nxt = [t.cpu().numpy() for t in outs]
    for s in range(b):
        a, toks, na = O.verify_accept(paths[s], target[s])
        assert acc[s] == a and nxt[s] == na and list(out[s, :a + 1]) == toks


def _verify(paths, targets, B_, seq_len=None, counters=None):
    import torch
    B = lib()
    b = paths.shape[0]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    acc = torch.full((b,), -9, dtype=torch.int32, device="cuda")
    out = torch.full((b, B_), -9, dtype=torch.int32, device="cuda")
    n_out = torch.zeros(b, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(b, dtype=torch.int32, device="cuda")
    sl = dev(seq_len) if seq_len is not None else None
    B.dflash2_verify_accept(b, B_, dev(paths), dev(targets), acc, out, n_out, nxt, sl, counters)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), out.cpu().numpy(), n_out.cpu().numpy(), nxt.cpu().numpy(), \
        (sl.cpu().numpy() if sl is not None else None)


def test_verify_golden_cases_on_gpu():
    for path, tgt, a, out, nxt in read_golden("verify_cases.txt"):
        p = np.array([[int(x) for x in path.split()]])
        t = np.array([[int(x) for x in tgt.split()]])
        Bsz = t.shape[1]
        acc, o, n, nx, _ = _verify(p, t, Bsz)
        assert acc[0] == int(a) and nx[0] == int(nxt) and n[0] == int(a) + 1
        exp = [int(x) for x in out.split()]
        assert list(o[0, :len(exp)]) == exp and np.all(o[0, len(exp):] == -1)


@pytest.mark.parametrize("B_", [2, 8, 16, 32])
def test_verify_and_counters_match_oracle(B_):
    import torch
    g = np.random.default_rng(B_)
    b, D = 300, B_ - 1
    paths = g.integers(0, 3, (b, D))
    targets = g.integers(0, 3, (b, B_))
    seq = g.integers(0, 1000, b)
    counters = torch.zeros(4 + 2 * B_ - 1, dtype=torch.int64, device="cuda")
    acc, out, n, nx, sl = _verify(paths, targets, B_, seq_len=seq, counters=counters)
    acc2, *_ = _verify(paths, targets, B_, counters=counters)      # accumulate a second time
    cnt = O.Counters(D)
    for s in range(b):
        a, toks, na = O.verify_accept(paths[s], targets[s])
        cnt.add(a)
        cnt.add(a)
        assert acc[s] == a and nx[s] == na and n[s] == a + 1
        assert list(out[s, :a + 1]) == toks and np.all(out[s, a + 1:] == -1)
        assert sl[s] == seq[s] + a + 1
    c = counters.cpu().numpy()
    assert c[0] == cnt.steps and c[1] == cnt.drafted and c[2] == cnt.accepted and c[3] == cnt.rollback
    np.testing.assert_array_equal(c[4:4 + B_], cnt.hist)
    np.testing.assert_array_equal(c[4 + B_:], cnt.acc_pos)
