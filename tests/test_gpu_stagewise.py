"""Stage-wise parity of the draft step: every stage of the GPU path is checked
against the oracle's same stage fed with the GPU's own stored inputs.

Why: with bf16 storage between stages the end-to-end result is sensitive to
single rounding flips (the oracle itself moves by ~0.03 in max logit at the
8B shape when its weights are nudged by 1e-6 relative), so end-to-end
agreement alone cannot separate a bug from rounding.  Fed identical inputs,
each stage must agree to about one bf16 unit in the last place (ulp).
"""

import numpy as np
import pytest

import dflash2_synth as S
import oracle as O
from tests.helpers import Case, lib

pytestmark = pytest.mark.gpu


def ulps(gpu, ref):
    """|gpu - ref| in bf16 ulps of the larger magnitude (ulp of x in
    [2^e, 2^(e+1)) is 2^(e-7)).  Magnitudes below 1e-3 of the tensor's RMS
    are measured against that floor instead: such values come from
    cancellation (a product or sum near zero), where fp32-vs-fp64 ordering
    legitimately changes many of their low bits."""
    floor = 1e-3 * np.sqrt(np.mean(np.square(ref))) + 1e-30
    m = np.maximum(np.maximum(np.abs(gpu), np.abs(ref)), floor)
    e = np.floor(np.log2(m))
    return np.abs(gpu - ref) / np.exp2(e - 7)


def check_ulps(name, gpu, ref, max_ulp, frac_over_1=0.01, slack=None):
    """At most max_ulp everywhere (or, where `slack` is given, an absolute
    error within slack plus one ulp), and at most frac_over_1 of the
    elements beyond 1 ulp."""
    assert np.all(np.isfinite(gpu)) and np.all(np.isfinite(ref)), (name, "non-finite values")
    u = ulps(gpu, ref)
    over = float(np.mean(u > 1.0 + 1e-9))
    bad = u > max_ulp
    if slack is not None:
        ulp_ref = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 1e-30))) - 7)
        bad &= np.abs(gpu - ref) > slack + ulp_ref
    w = int(np.argmax(u))
    print(f"[stage] {name:8s} max {u.max():.2f} ulp (at |ref| {abs(ref.flat[w]):.3e}, |diff| "
          f"{abs(gpu.flat[w] - ref.flat[w]):.3e}), >1ulp {over:.2e}, beyond bound {int(bad.sum())}, n={u.size}")
    assert not bad.any(), (name, float(u.max()))
    assert over <= frac_over_1, (name, over)


class Reader:
    def __init__(self, case):
        import torch
        B = lib()
        r = case.runner
        self.torch = torch
        self.ws = r.workspace
        self.bf16 = case.cfg["dtype"] != "f32"
        self.off = B.dflash2_test_layout(r.cfg, case.b, int(case.n_new.sum()),
                                         r.max_pages * case.cfg["page_size"])

    def get(self, name, shape, fp32=False):
        n = int(np.prod(shape))
        o = self.off[name]
        if fp32 or not self.bf16:
            t = self.ws[o:o + 4 * n].view(self.torch.float32)
        else:
            t = self.ws[o:o + 2 * n].view(self.torch.bfloat16)
        return t.reshape(shape).double().cpu().numpy()


def cache_rows(case, layer, s, positions):
    r = case.runner
    ps = case.cfg["page_size"]
    bt = r.block_table.cpu().numpy()
    pages = bt[s, positions // ps]
    slots = positions % ps
    k = r.k_cache[layer, pages, slots].double().cpu().numpy()
    v = r.v_cache[layer, pages, slots].double().cpu().numpy()
    return k, v


def run_stagewise(case):
    cfg = case.cfg
    assert cfg["n_layers"] == 1
    Wv = case.Wv
    Wl = Wv["layers"][0]
    st = O.Store(cfg["dtype"] != "f32")
    H, B_, nq, nkv, d, I = (cfg["hidden"], cfg["block_size"], cfg["n_q_heads"], cfg["n_kv_heads"],
                            cfg["head_dim"], cfg["intermediate"])
    D, b, eps = B_ - 1, case.b, cfg["rms_eps"]
    rows = b * B_
    R = Reader(case)
    n_new = int(case.n_new.sum())
    # (a) feature projection of the new rows and their context K/V
    if n_new:
        f = R.get("f", (n_new, H))
        check_ulps("f", f, O.project_features(cfg, Wv, case.taps_new.values, st), 2)
        n0 = 0
        for s in range(b):
            n = int(case.n_new[s])
            if n:
                pos = int(case.ctx_lens[s]) + np.arange(n)
                k_ref, v_ref = O.context_kv(cfg, Wl, f[n0:n0 + n], pos, st)
                k_gpu, v_gpu = cache_rows(case, 0, s, pos)
                check_ulps("ctx_k", k_gpu, k_ref, 2)
                check_ulps("ctx_v", v_gpu, v_ref, 2)
            n0 += n
    # (b) block forward, one stage at a time from the GPU's stored inputs
    q = R.get("q", (rows, nq, d))
    kb = R.get("kb", (rows, nkv, d))
    vb = R.get("vb", (rows, nkv, d))
    Og = R.get("O", (rows, nq * d))
    kc = cfg["conv_kernel_size"]
    win = cfg.get("sliding_window", 0)
    u_m = R.get("u", (rows, H))
    u2_m = R.get("u2", (rows, H)) if kc else u_m   # DFlash v1: no conv, u2 is u
    act = R.get("act", (rows, I))
    h = R.get("h", (rows, H), fp32=True)
    hn = R.get("hn", (b * D, H))
    ua = R.get("ua", (rows, H))
    u2a = R.get("u2a", (rows, H)) if kc else ua
    q_ref, k_ref, v_ref, O_ref, h_mid, ua_ref, u2a_ref = [], [], [], [], [], [], []
    O_slack = []
    for s in range(b):
        P = int(case.ctx_lens[s] + case.n_new[s])
        sl = slice(s * B_, (s + 1) * B_)
        toks = np.array([int(case.anchor[s])] + [cfg["mask_token_id"]] * D)
        h0 = cfg["input_embedding_scale"] * Wv["embed"][toks].astype(np.float64)
        ua_ref.append(st(O.rms_norm(h0, Wl["attn_norm"], eps)))
        u2a_ref.append(st(ua[sl] + O.dynamic_conv(ua[sl], Wl["tapgen_attn"], cfg["conv_group_size"])) if kc
                       else ua[sl])
        qkv = u2a[sl] @ Wl["qkv"].astype(np.float64).T
        pos = P + np.arange(B_)
        q_ref.append(st(O.rope(O.rms_norm(qkv[:, :nq * d].reshape(B_, nq, d), Wl["q_norm"], eps), pos,
                               cfg["rope_theta"])))
        k_ref.append(st(O.rope(O.rms_norm(qkv[:, nq * d:(nq + nkv) * d].reshape(B_, nkv, d), Wl["k_norm"], eps),
                               pos, cfg["rope_theta"])))
        v_ref.append(st(qkv[:, (nq + nkv) * d:].reshape(B_, nkv, d)))
        Kc, Vc = cache_rows(case, 0, s, np.arange(max(0, P - win) if win else 0, P))
        O_ref.append(st(O.block_attention(q[sl], Kc, Vc, kb[sl], vb[sl])).reshape(B_, nq * d))
        # fp32 (tensor-core) accumulation of the P.V sums over the L keys read:
        # a random-walk bound, 32 * 2^-24 * sqrt(L) * sum_j p_j |v_j|, the
        # magnitude sum being the same attention over |V|.  Outputs that are a
        # small remainder of large terms carry this absolute error.
        L = Kc.shape[0] + B_
        O_abs = O.block_attention(q[sl], Kc, np.abs(Vc), kb[sl], np.abs(vb[sl])).reshape(B_, nq * d)
        O_slack.append(32.0 * 2.0 ** -24 * np.sqrt(L) * O_abs)
        h_mid.append(h0 + Og[sl] @ Wl["o"].astype(np.float64).T)
    check_ulps("u_attn", ua, np.concatenate(ua_ref), 2)
    check_ulps("u2_attn", u2a, np.concatenate(u2a_ref), 2)
    check_ulps("q", q, np.concatenate(q_ref), 2)
    check_ulps("k_blk", kb, np.concatenate(k_ref), 2)
    check_ulps("v_blk", vb, np.concatenate(v_ref), 2)
    check_ulps("attn_O", Og, np.concatenate(O_ref), 2, slack=np.concatenate(O_slack))
    h_mid = np.concatenate(h_mid)
    check_ulps("u_mlp", u_m, st(O.rms_norm(h_mid, Wl["mlp_norm"], eps)), 2)
    u2_ref = np.concatenate([st(u_m[s * B_:(s + 1) * B_] + O.dynamic_conv(
        u_m[s * B_:(s + 1) * B_], Wl["tapgen_mlp"], cfg["conv_group_size"])) if kc else u_m[s * B_:(s + 1) * B_]
        for s in range(b)])
    check_ulps("u2_mlp", u2_m, u2_ref, 2)
    Wgu = Wl["gate_up"].astype(np.float64)
    gu = u2_m @ Wgu.T
    # beyond 2 ulps only where fp32 accumulation of gate or up (K terms) can
    # move SiLU(gate)*up that far: a value of up (or gate) that is a small
    # remainder of large terms carries their absolute rounding error
    acc_err = 1e-5 * (np.abs(u2_m) @ np.abs(Wgu).T)
    g, u = gu[:, :I], gu[:, I:]
    sig = 1.0 / (1.0 + np.exp(-g))
    slack = np.abs(sig * (1 + g * (1 - sig))) * np.abs(u) * acc_err[:, :I] + np.abs(g * sig) * acc_err[:, I:]
    check_ulps("act", act, st(O.silu(g) * u), 2, slack=slack)
    h_ref = h_mid + act @ Wl["down"].astype(np.float64).T
    scale = np.abs(h_mid) + np.abs(act) @ np.abs(Wl["down"].astype(np.float64)).T + np.abs(Og) @ np.abs(
        Wl["o"].astype(np.float64)).T
    assert np.all(np.abs(h - h_ref) <= 1e-5 * scale + 1e-7), float(np.max(np.abs(h - h_ref) / scale))
    keep = np.array([i % B_ != 0 for i in range(rows)])
    check_ulps("hn", hn, st(O.rms_norm(h[keep], Wv["final_norm"], eps)), 2)
    # (c) the lm_head from the GPU's hn, against the debug logits
    dbg = case.debug.double().cpu().numpy().reshape(b * D, -1)
    W = Wv["lm_head"].astype(np.float64)
    z = cfg["output_multiplier"] * (hn @ W.T)
    bound = np.abs(hn) @ np.abs(W).T
    assert np.all(np.abs(dbg - z) <= 1e-5 * bound + 1e-6), float(np.max(np.abs(dbg - z) / (bound + 1e-30)))
    print(f"[stage] logits   max |d| {np.max(np.abs(dbg - z)):.2e}")


def test_stagewise_small_bf16():
    cfg = S.small_bf16_config(n_layers=1, index=15)
    case = Case(cfg, ctx_lens=[60, 0, 150], n_new=[3, 8, 1], seed=15).run_gpu()
    run_stagewise(case)


def test_stagewise_tiny_fp32():
    cfg = S.config_of("tiny_fp32")
    case = Case(cfg, ctx_lens=[128], n_new=[8], seed=16).run_gpu()
    run_stagewise(case)


@pytest.mark.slow
def test_stagewise_qwen3_8b_shape():
    cfg = S.config_of("qwen3_8b_b1")
    case = Case(cfg, ctx_lens=[2040], n_new=[8], seed=17).run_gpu()
    run_stagewise(case)


def test_stagewise_gqa5_block16():
    # 80 query rows per kv head (5 q heads x 16 block rows), two contexts
    # that end mid-page, 16 + 4 appended rows split along K in the projection
    cfg = S.small_bf16_config(block_size=16, n_q_heads=10, n_kv_heads=2, head_dim=128, top_k=16, hidden=512,
                              n_layers=1, index=16)
    case = Case(cfg, ctx_lens=[300, 33], n_new=[16, 4], seed=18).run_gpu()
    run_stagewise(case)
