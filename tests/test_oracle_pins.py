"""Pins of the CPU oracle to facts outside itself (closed forms, special cases
that reduce to a library routine, brute force, hand-worked golden cases).

Each test names the oracle function it pins and the fact it uses.  A plausible
mistake (dropped term, wrong sign or index, transposed operand) in the pinned
function should fail at least one of them.
"""

import math

import numpy as np
import pytest
import torch

import oracle as O
from tests.conftest import read_golden


def tiny_cfg(**over):
    c = dict(hidden=64, n_q_heads=4, n_kv_heads=2, head_dim=16, intermediate=96,
             vocab=50, n_layers=1, n_taps=3, block_size=4, conv_kernel_size=2,
             conv_group_size=8, top_k=3, selector_rank=4, page_size=16,
             mask_token_id=49, rms_eps=1e-6, rope_theta=1.0e4,
             input_embedding_scale=1.0, output_multiplier=1.0,
             final_logit_softcap=0.0)
    c.update(over)
    return c


def tiny_weights(cfg, seed=0, scale=0.3):
    g = np.random.default_rng(seed)
    H, V, T = cfg["hidden"], cfg["vocab"], cfg["n_taps"]
    nq, nkv, d, I = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["intermediate"]
    G = H // cfg["conv_group_size"]
    kc, r = cfg["conv_kernel_size"], cfg["selector_rank"]
    n = lambda *s: g.standard_normal(s) * scale
    one = lambda k: 1.0 + 0.1 * g.standard_normal(k)
    W = dict(embed=n(V, H), lm_head=n(V, H), fc=n(H, T * H) / math.sqrt(T),
             hidden_norm=one(H), final_norm=one(H), sel=n(2 * r, H), layers=[])
    for _ in range(cfg["n_layers"]):
        W["layers"].append(dict(
            attn_norm=one(H), tapgen_attn=n(kc * G, H), qkv=n((nq + 2 * nkv) * d, H) / 4,
            q_norm=one(d), k_norm=one(d), o=n(H, nq * d) / 4, mlp_norm=one(H),
            tapgen_mlp=n(kc * G, H), gate_up=n(2 * I, H) / 4, down=n(H, I) / 4))
    return W


def empty_ctx(cfg):
    z = np.zeros((0, cfg["n_kv_heads"], cfg["head_dim"]))
    return [(z, z) for _ in range(cfg["n_layers"])]


# ----------------------------------------------------------------- bf16_round

def test_bf16_round_ties_to_even_exact_values():
    # 1 + 2^-8 is the midpoint of 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    assert O.bf16_round(1.0 + 2.0 ** -8) == 1.0
    # 1 + 3*2^-8 is the midpoint of 1+2^-7 (odd) and 1+2^-6 (even)
    assert O.bf16_round(1.0 + 3 * 2.0 ** -8) == 1.0 + 2.0 ** -6
    assert O.bf16_round(-(1.0 + 3 * 2.0 ** -8)) == -(1.0 + 2.0 ** -6)
    assert O.bf16_round(0.0) == 0.0
    assert O.bf16_round(3.0) == 3.0
    # just above a midpoint rounds up
    assert O.bf16_round(1.0 + 2.0 ** -8 + 2.0 ** -30) == 1.0 + 2.0 ** -7


def test_bf16_round_matches_torch_conversion():
    g = np.random.default_rng(1)
    x = np.concatenate([g.standard_normal(20000) * 10.0 ** g.integers(-30, 30, 20000),
                        g.standard_normal(1000) * 1e-39])       # bf16 subnormals
    x32 = x.astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.bf16_round(x32.astype(np.float64)), ref)


# ------------------------------------------------------------------- rms_norm

def test_rms_norm_matches_torch_and_closed_form():
    g = np.random.default_rng(2)
    x = g.standard_normal((5, 33))
    gam = g.standard_normal(33)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (33,), torch.from_numpy(gam),
                                       eps=1e-6).numpy()
    np.testing.assert_allclose(O.rms_norm(x, gam, 1e-6), ref, rtol=1e-12, atol=1e-12)
    # constant vector c*1: each entry becomes c / sqrt(c^2 + eps) * gamma
    c, eps = -0.37, 1e-3
    y = O.rms_norm(np.full(8, c), np.arange(1, 9, dtype=float), eps)
    np.testing.assert_allclose(y, c / math.sqrt(c * c + eps) * np.arange(1, 9), rtol=1e-14)


# ----------------------------------------------------------------------- rope

def test_rope_d2_is_a_plane_rotation_by_pos_radians():
    # d = 2: one frequency theta^0 = 1, so the angle is the position itself
    x = np.array([[[0.3, -1.2]]])
    for pos in (0, 1, 5, 1000):
        y = O.rope(x, np.array([pos]), 1.0e6)[0, 0]
        c, s = math.cos(pos), math.sin(pos)
        np.testing.assert_allclose(y, [0.3 * c + 1.2 * s, -1.2 * c + 0.3 * s], rtol=1e-12, atol=1e-15)


def test_rope_pair_frequencies_follow_theta_power():
    """rope: pair i rotates by pos * theta^(-2i/d).  At d = 4, theta = 100:
    pair (0, 2) by pos radians, pair (1, 3) by pos / 10 radians; a unit
    vector in x1 shows that second angle directly."""
    e1 = np.zeros((1, 1, 4)); e1[0, 0, 1] = 1.0
    for pos in (1, 3, 40):
        y = O.rope(e1, np.array([pos]), 100.0)[0, 0]
        a = pos / 10.0
        np.testing.assert_allclose(y, [0.0, math.cos(a), 0.0, math.sin(a)], rtol=1e-12, atol=1e-15)


def test_rope_relative_position_and_norm():
    g = np.random.default_rng(3)
    q = g.standard_normal((1, 1, 64))
    k = g.standard_normal((1, 1, 64))
    dot = lambda m, n: float(np.sum(O.rope(q, np.array([m]), 1e6) * O.rope(k, np.array([n]), 1e6)))
    assert abs(dot(10, 3) - dot(1010, 1003)) < 1e-9
    assert abs(dot(7, 7) - float(np.sum(q * k))) < 1e-9
    assert abs(dot(5, 9) - dot(9, 5)) > 1e-6            # the rotation has a direction
    y = O.rope(q, np.array([12345]), 1e6)
    assert abs(np.linalg.norm(y) - np.linalg.norm(q)) < 1e-12
    # pair i mixes with i + d/2 (rotate-half), not with i+1
    e0 = np.zeros((1, 1, 8)); e0[0, 0, 0] = 1.0
    y = O.rope(e0, np.array([1]), 1e4)[0, 0]
    assert np.count_nonzero(np.abs(y) > 1e-15) == 2 and abs(y[4]) > 0.5


def test_silu_matches_torch():
    x = np.linspace(-20, 20, 1001)
    np.testing.assert_allclose(O.silu(x), torch.nn.functional.silu(torch.from_numpy(x)).numpy(),
                               rtol=1e-12, atol=1e-300)


# --------------------------------------------------------------- dynamic conv

def test_dynamic_conv_zero_generator_is_two_tap_average():
    g = np.random.default_rng(4)
    u = g.standard_normal((6, 32))
    c = O.dynamic_conv(u, np.zeros((2 * 4, 32)), group_size=8)
    prev = np.vstack([np.zeros((1, 32)), u[:-1]])
    np.testing.assert_allclose(c, 0.5 * (u + prev), rtol=0, atol=1e-15)


def test_dynamic_conv_is_left_looking_and_grouped():
    g = np.random.default_rng(5)
    u = g.standard_normal((8, 32))
    w = g.standard_normal((8, 32))
    c = O.dynamic_conv(u, w, group_size=8)
    u2 = u.copy(); u2[5:] += 3.0
    c2 = O.dynamic_conv(u2, w, group_size=8)
    np.testing.assert_array_equal(c[:5], c2[:5])                 # t < 5 unchanged
    # a generator that sends group 1 hard to tap 0 and group 2 hard to tap 1
    H, gs = 32, 8
    w = np.zeros((8, H))
    u = np.abs(u) + 0.5                                          # positive so sum(u) > 0
    w[2 * 1 + 0] = 100.0                                         # group 1, tap 0 (current)
    w[2 * 2 + 1] = 100.0                                         # group 2, tap 1 (previous)
    c = O.dynamic_conv(u, w, group_size=gs)
    np.testing.assert_allclose(c[:, 8:16], u[:, 8:16], atol=1e-12)
    prev = np.vstack([np.zeros((1, H)), u[:-1]])
    np.testing.assert_allclose(c[:, 16:24], prev[:, 16:24], atol=1e-12)
    np.testing.assert_allclose(c[:, 0:8], 0.5 * (u + prev)[:, 0:8], atol=1e-12)


def test_dynamic_conv_wider_window_reads_further_back():
    # conv_kernel_size counts the taps: with three, a generator sending every
    # group hard to tap 2 returns the row two positions back (zero before the
    # block), and a zero generator the three-row average
    g = np.random.default_rng(26)
    H, gs, Kc = 16, 8, 3
    u = g.standard_normal((6, H))
    w = np.zeros((Kc * (H // gs), H))
    w[Kc * 0 + 2] = w[Kc * 1 + 2] = 100.0
    c = O.dynamic_conv(np.abs(u) + 0.5, w, gs, kernel_size=Kc)
    back2 = np.vstack([np.zeros((2, H)), (np.abs(u) + 0.5)[:-2]])
    np.testing.assert_allclose(c, back2, atol=1e-12)
    c0 = O.dynamic_conv(u, np.zeros_like(w), gs, kernel_size=Kc)
    p1 = np.vstack([np.zeros((1, H)), u[:-1]])
    p2 = np.vstack([np.zeros((2, H)), u[:-2]])
    np.testing.assert_allclose(c0, (u + p1 + p2) / 3.0, atol=1e-15)


# ------------------------------------------------------------------ attention

def test_block_attention_special_cases():
    g = np.random.default_rng(6)
    d = 8
    # one key (no context, block of one): output is that value
    q = g.standard_normal((1, 2, d)); kb = g.standard_normal((1, 1, d)); vb = g.standard_normal((1, 1, d))
    z = np.zeros((0, 1, d))
    out = O.block_attention(q, z, z, kb, vb)
    np.testing.assert_allclose(out[0, 0], vb[0, 0], rtol=1e-14)
    np.testing.assert_allclose(out[0, 1], vb[0, 0], rtol=1e-14)
    # identical keys: uniform weights, output = mean of all values (context and block)
    kc = np.tile(kb, (5, 1, 1)); vc = g.standard_normal((5, 1, d))
    kb3 = np.tile(kb, (3, 1, 1)); vb3 = g.standard_normal((3, 1, d))
    q3 = g.standard_normal((3, 2, d))
    out = O.block_attention(q3, kc, vc, kb3, vb3)
    mean = np.concatenate([vc, vb3])[:, 0].mean(0)
    np.testing.assert_allclose(out, np.broadcast_to(mean, out.shape), rtol=1e-12)


def test_block_attention_matches_sdpa_non_causal_gqa():
    g = np.random.default_rng(7)
    B, nq, nkv, d, P = 5, 6, 2, 16, 9
    q = g.standard_normal((B, nq, d)); Kc = g.standard_normal((P, nkv, d)); Vc = g.standard_normal((P, nkv, d))
    Kb = g.standard_normal((B, nkv, d)); Vb = g.standard_normal((B, nkv, d))
    out = O.block_attention(q, Kc, Vc, Kb, Vb)
    K = torch.from_numpy(np.concatenate([Kc, Kb])).permute(1, 0, 2).repeat_interleave(nq // nkv, 0)
    V = torch.from_numpy(np.concatenate([Vc, Vb])).permute(1, 0, 2).repeat_interleave(nq // nkv, 0)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).permute(1, 0, 2), K, V, is_causal=False).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    # the first block query sees the last block key (non-causal)
    Kb2 = Kb.copy(); Kb2[B - 1] += 1.0
    assert not np.allclose(O.block_attention(q, Kc, Vc, Kb2, Vb)[0], out[0])


# --------------------------------------------------------- feature projection

def test_feature_projection_identity_blocks_select_taps():
    cfg = tiny_cfg()
    W = tiny_weights(cfg)
    H, T = cfg["hidden"], cfg["n_taps"]
    g = np.random.default_rng(8)
    taps = g.standard_normal((3, T * H))
    st = O.Store(False)
    for t in range(T):
        W["fc"] = np.zeros((H, T * H)); W["fc"][:, t * H:(t + 1) * H] = np.eye(H)
        f = O.project_features(cfg, W, taps, st)
        np.testing.assert_allclose(f, O.rms_norm(taps[:, t * H:(t + 1) * H], W["hidden_norm"], 1e-6),
                                   rtol=1e-12)


def test_feature_projection_permutation_block_fixes_orientation():
    """project_features: W_fc holding a non-symmetric permutation P in tap
    block t gives x = tap_t P^T, i.e. x[:, i] = tap_t[:, pi(i)], then the
    hidden_norm gain.  A transposed operand would read pi^-1 instead (pi
    below has no fixed points and is not an involution), a wrong block
    offset another tap, and the final norm's gain a different scale."""
    cfg = tiny_cfg()
    W = tiny_weights(cfg)
    H, T = cfg["hidden"], cfg["n_taps"]
    pi = np.roll(np.arange(H), 3)  # i -> i - 3 (mod H)
    g = np.random.default_rng(18)
    taps = g.standard_normal((4, T * H))
    st = O.Store(False)
    for t in range(T):
        W["fc"] = np.zeros((H, T * H))
        W["fc"][np.arange(H), t * H + pi] = 1.0
        f = O.project_features(cfg, W, taps, st)
        want = O.rms_norm(taps[:, t * H:(t + 1) * H][:, pi], W["hidden_norm"], 1e-6)
        np.testing.assert_allclose(f, want, rtol=1e-12)
        wrong = O.rms_norm(taps[:, t * H:(t + 1) * H][:, np.argsort(pi)], W["hidden_norm"], 1e-6)
        assert not np.allclose(f, wrong)


def test_context_kv_identity_projection():
    cfg = tiny_cfg(hidden=32, n_q_heads=2, n_kv_heads=1, head_dim=16)
    H, d = 32, 16
    Wl = {"qkv": np.zeros((4 * d, H)), "k_norm": np.full(d, 2.0)}
    Wl["qkv"][2 * d:3 * d, :d] = np.eye(d)        # W_k reads f[:, :16]
    Wl["qkv"][3 * d:4 * d, d:] = np.eye(d)        # W_v reads f[:, 16:]
    f = np.random.default_rng(9).standard_normal((4, H))
    pos = np.array([0, 3, 4, 100])
    k, v = O.context_kv(cfg, Wl, f, pos, O.Store(False))
    np.testing.assert_allclose(v[:, 0], f[:, d:], rtol=1e-15)
    np.testing.assert_allclose(k[0, 0], O.rms_norm(f[0, :d], np.full(d, 2.0), 1e-6), rtol=1e-12)
    np.testing.assert_allclose(k[:, 0], O.rope(O.rms_norm(f[:, None, :d], np.full(d, 2.0), 1e-6), pos,
                                               cfg["rope_theta"])[:, 0], rtol=1e-12)


def test_context_kv_permutation_blocks_fix_orientation():
    """context_kv: permutation blocks in W_k and W_v (no fixed points, not
    involutions) give V = f[:, d + pi] and K = RoPE(RMSNorm_k(f[:, pi])): a
    transposed projection would read pi^-1."""
    cfg = tiny_cfg(hidden=32, n_q_heads=2, n_kv_heads=1, head_dim=16)
    H, d = 32, 16
    pi = np.roll(np.arange(d), 5)
    Wl = {"qkv": np.zeros((4 * d, H)), "k_norm": 0.5 + np.arange(d) / d}
    Wl["qkv"][2 * d + np.arange(d), pi] = 1.0       # W_k reads f[:, pi]
    Wl["qkv"][3 * d + np.arange(d), d + pi] = 1.0   # W_v reads f[:, 16 + pi]
    f = np.random.default_rng(29).standard_normal((5, H))
    pos = np.array([0, 1, 7, 64, 1000])
    k, v = O.context_kv(cfg, Wl, f, pos, O.Store(False))
    np.testing.assert_allclose(v[:, 0], f[:, d + pi], rtol=1e-15)
    want = O.rope(O.rms_norm(f[:, None, pi], Wl["k_norm"], 1e-6), pos, cfg["rope_theta"])[:, 0]
    np.testing.assert_allclose(k[:, 0], want, rtol=1e-12)
    assert not np.allclose(v[:, 0], f[:, d + np.argsort(pi)])


# ---------------------------------------------------------------- draft block

def test_draft_layer_residual_identity_when_outputs_zero():
    cfg = tiny_cfg()
    W = tiny_weights(cfg)
    Wl = dict(W["layers"][0]); Wl["o"] = np.zeros_like(Wl["o"]); Wl["down"] = np.zeros_like(Wl["down"])
    h = np.random.default_rng(10).standard_normal((4, cfg["hidden"]))
    out = O.draft_layer(cfg, Wl, h, *empty_ctx(cfg)[0], np.arange(4), O.Store(False))
    np.testing.assert_array_equal(out, h)


def _rms_rows(x, gamma, eps):
    # RMSNorm written out row by row for the closed forms below
    return np.stack([r / math.sqrt(float(np.dot(r, r)) / r.size + eps) for r in x]) * gamma


def _left_avg_conv_input(u):
    # a zero tap generator gives the taps 1/2, 1/2, so the sublayer reads
    # u_t + (u_t + u_{t-1}) / 2 with nothing left of the anchor
    prev = np.vstack([np.zeros_like(u[:1]), u[:-1]])
    return 1.5 * u + 0.5 * prev


@pytest.mark.parametrize("which", ["q", "k"])
def test_draft_layer_qk_norm_makes_head_scale_irrelevant(which):
    # draft_layer ([Train] "What is DFlash?", the draft's own norms; Qwen3
    # layer: per-head q/k RMSNorm before RoPE): scaling the projection rows of
    # one query head, or of one key head, by c > 0 leaves the layer output
    # unchanged, because that head's norm divides the scale out.  A dropped
    # q_norm / k_norm, or one taken over all heads together, fails this.
    cfg = tiny_cfg(rms_eps=0.0)
    W = tiny_weights(cfg, seed=3)
    nq, nkv, d = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    g = np.random.default_rng(30)
    h = g.standard_normal((4, cfg["hidden"]))
    ctxK = g.standard_normal((5, nkv, d))
    ctxV = g.standard_normal((5, nkv, d))
    pos = np.arange(5, 9)
    st = O.Store(False)
    base = O.draft_layer(cfg, W["layers"][0], h, ctxK, ctxV, pos, st)
    head_row0 = 1 * d if which == "q" else (nq + 1) * d     # q head 1, or kv head 1
    for c in (3.7, 0.25):
        Wl = dict(W["layers"][0])
        Wl["qkv"] = Wl["qkv"].copy()
        Wl["qkv"][head_row0:head_row0 + d] *= c
        out = O.draft_layer(cfg, Wl, h, ctxK, ctxV, pos, st)
        np.testing.assert_allclose(out, base, rtol=1e-11, atol=1e-11)
    # the pin has teeth: the same scaling of a v head does change the output
    Wl = dict(W["layers"][0])
    Wl["qkv"] = Wl["qkv"].copy()
    Wl["qkv"][(nq + nkv + 1) * d:(nq + nkv + 2) * d] *= 3.7
    assert np.max(np.abs(O.draft_layer(cfg, Wl, h, ctxK, ctxV, pos, st) - base)) > 1e-3


def test_draft_layer_attention_reads_u_plus_conv_closed_form():
    # draft_layer, attention sublayer ([Train] "Variants": the convolution is
    # added around the sublayer): with W_k = 0 every block key normalises to
    # 0, so (no context) each row attends uniformly to the B block values.
    # With W_v copying the first nkv*d channels of the sublayer input and W_o
    # copying head 0's output back into channels [0, d), every row gains
    # mean_t(u'_t)[0:d] with u' = u + (u + u_prev)/2.  Reading c alone (not
    # u + c), a causal mask, or a wrong V / O wiring fails this.
    cfg = tiny_cfg()
    W = tiny_weights(cfg, seed=4)
    H, nq, nkv, d, I = (cfg[k] for k in ("hidden", "n_q_heads", "n_kv_heads", "head_dim", "intermediate"))
    Wl = dict(W["layers"][0])
    Wl["tapgen_attn"] = np.zeros_like(Wl["tapgen_attn"])
    qkv = Wl["qkv"].copy()
    qkv[nq * d:(nq + nkv) * d] = 0.0
    qkv[(nq + nkv) * d:] = np.eye(nkv * d, H)
    Wl["qkv"] = qkv
    Wl["o"] = np.eye(H, nq * d) * (np.arange(H) < d)[:, None]
    Wl["gate_up"] = np.zeros((2 * I, H))
    h = np.random.default_rng(31).standard_normal((4, H))
    out = O.draft_layer(cfg, Wl, h, *empty_ctx(cfg)[0], np.arange(4), O.Store(False))
    u2 = _left_avg_conv_input(_rms_rows(h, Wl["attn_norm"], cfg["rms_eps"]))
    want = h.copy()
    want[:, :d] += u2[:, :d].mean(axis=0)
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)


def test_draft_layer_mlp_is_silu_gate_times_up_on_post_attention_rows():
    # draft_layer, MLP sublayer (Qwen3 MLP: down(SiLU(gate x) * up x)) with
    # the additive two-tap conv: one gate row e_i, one up row e_j and one down
    # column e_m give out[:, m] = h1[:, m] + SiLU(u'_i) * u'_j, where h1 is the
    # residual after the attention sublayer and u' = u + (u + u_prev)/2 of
    # RMSNorm(h1).  Swapping gate and up (SiLU(u'_j) * u'_i), norming the
    # pre-attention rows, or feeding c instead of u + c fails this.
    cfg = tiny_cfg()
    W = tiny_weights(cfg, seed=5)
    H, nq, nkv, d, I = (cfg[k] for k in ("hidden", "n_q_heads", "n_kv_heads", "head_dim", "intermediate"))
    i, j, m = 3, 11, 7
    Wl = dict(W["layers"][0])
    Wl["tapgen_attn"] = np.zeros_like(Wl["tapgen_attn"])
    Wl["tapgen_mlp"] = np.zeros_like(Wl["tapgen_mlp"])
    qkv = Wl["qkv"].copy()
    qkv[nq * d:(nq + nkv) * d] = 0.0
    qkv[(nq + nkv) * d:] = np.eye(nkv * d, H)
    Wl["qkv"] = qkv
    Wl["o"] = 0.7 * np.eye(H, nq * d) * (np.arange(H) < d)[:, None]
    gu = np.zeros((2 * I, H))
    gu[0, i] = 1.0          # gate row 0 reads channel i
    gu[I, j] = 1.0          # up row 0 reads channel j
    Wl["gate_up"] = gu
    down = np.zeros((H, I))
    down[m, 0] = 1.0
    Wl["down"] = down
    h = np.random.default_rng(32).standard_normal((4, H))
    out = O.draft_layer(cfg, Wl, h, *empty_ctx(cfg)[0], np.arange(4), O.Store(False))
    eps = cfg["rms_eps"]
    ua = _left_avg_conv_input(_rms_rows(h, Wl["attn_norm"], eps))
    h1 = h.copy()
    h1[:, :d] += 0.7 * ua[:, :d].mean(axis=0)
    um = _left_avg_conv_input(_rms_rows(h1, Wl["mlp_norm"], eps))
    want = h1.copy()
    want[:, m] += um[:, i] / (1.0 + np.exp(-um[:, i])) * um[:, j]
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)
    swapped = h1.copy()
    swapped[:, m] += um[:, j] / (1.0 + np.exp(-um[:, j])) * um[:, i]
    assert np.max(np.abs(swapped - want)) > 1e-3


def test_draft_layer_each_sublayer_uses_its_own_tap_generator():
    """draft_layer: the attention sublayer's conv reads tapgen_attn and the
    MLP's tapgen_mlp.  With a random attention generator and a zero MLP
    generator, the MLP pin above still holds with the attention rows formed
    by dynamic_conv(u, tapgen_attn) (pinned on its own) and the MLP rows by
    the two-tap average; using one generator for both sublayers fails it."""
    cfg = tiny_cfg()
    W = tiny_weights(cfg, seed=6)
    H, nq, nkv, d, I = (cfg[k] for k in ("hidden", "n_q_heads", "n_kv_heads", "head_dim", "intermediate"))
    i, j, m = 5, 2, 9
    Wl = dict(W["layers"][0])
    Wl["tapgen_attn"] = 2.0 * np.random.default_rng(40).standard_normal(Wl["tapgen_attn"].shape)
    Wl["tapgen_mlp"] = np.zeros_like(Wl["tapgen_mlp"])
    qkv = Wl["qkv"].copy()
    qkv[nq * d:(nq + nkv) * d] = 0.0
    qkv[(nq + nkv) * d:] = np.eye(nkv * d, H)
    Wl["qkv"] = qkv
    Wl["o"] = 0.7 * np.eye(H, nq * d) * (np.arange(H) < d)[:, None]
    gu = np.zeros((2 * I, H))
    gu[0, i] = 1.0
    gu[I, j] = 1.0
    Wl["gate_up"] = gu
    down = np.zeros((H, I))
    down[m, 0] = 1.0
    Wl["down"] = down
    h = np.random.default_rng(41).standard_normal((4, H))
    out = O.draft_layer(cfg, Wl, h, *empty_ctx(cfg)[0], np.arange(4), O.Store(False))
    eps = cfg["rms_eps"]
    u = _rms_rows(h, Wl["attn_norm"], eps)
    ua = u + O.dynamic_conv(u, Wl["tapgen_attn"], cfg["conv_group_size"], cfg["conv_kernel_size"])
    h1 = h.copy()
    h1[:, :d] += 0.7 * ua[:, :d].mean(axis=0)
    um = _left_avg_conv_input(_rms_rows(h1, Wl["mlp_norm"], eps))
    want = h1.copy()
    want[:, m] += um[:, i] / (1.0 + np.exp(-um[:, i])) * um[:, j]
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)


def test_v1_layer_without_conv_mixes_rows_only_through_attention():
    # conv_kernel_size 0 (DFlash v1): with the attention output switched off
    # (W_o = 0) every row is processed alone, so changing row 1 leaves rows
    # 0, 2, 3 unchanged; with the two-tap conv (DFlash 2) row 2 reads row 1
    for kc, row2_moves in [(0, False), (2, True)]:
        cfg = tiny_cfg(conv_kernel_size=kc)
        W = tiny_weights(cfg)
        Wl = dict(W["layers"][0]); Wl["o"] = np.zeros_like(Wl["o"])
        h = np.random.default_rng(20).standard_normal((4, cfg["hidden"]))
        h2 = h.copy(); h2[1] += 0.5
        a = O.draft_layer(cfg, Wl, h, *empty_ctx(cfg)[0], np.arange(4), O.Store(False))
        b = O.draft_layer(cfg, Wl, h2, *empty_ctx(cfg)[0], np.arange(4), O.Store(False))
        np.testing.assert_array_equal(a[[0, 3]], b[[0, 3]])
        assert np.any(a[1] != b[1])
        assert bool(np.any(a[2] != b[2])) == row2_moves


def test_sliding_window_reads_only_the_last_context_positions():
    cfg = tiny_cfg()
    W = tiny_weights(cfg)
    taps = np.random.default_rng(21).standard_normal((12, cfg["n_taps"] * cfg["hidden"]))
    st = O.Store(False)
    ctx = O.append_context(cfg, W, empty_ctx(cfg), taps, 0, st)
    full = O.draft_block(cfg, W, 7, ctx, st)
    for win in (0, 12, 40):     # unset, or a window covering the whole context
        np.testing.assert_array_equal(O.draft_block(dict(cfg, sliding_window=win), W, 7, ctx, st), full)
    cw = dict(cfg, sliding_window=5)
    z5 = O.draft_block(cw, W, 7, ctx, st)
    assert np.max(np.abs(z5 - full)) > 1e-6
    # keys and values older than the window do not matter; a key inside does
    K, V = ctx[0]
    old = [(np.concatenate([K[:7] * -3.0 + 1.0, K[7:]]), np.concatenate([V[:7] * 2.0, V[7:]]))]
    np.testing.assert_array_equal(O.draft_block(cw, W, 7, old, st), z5)
    inside = [(np.concatenate([K[:7], K[7:] * 1.5]), V)]
    assert np.max(np.abs(O.draft_block(cw, W, 7, inside, st) - z5)) > 1e-9


def test_context_appended_in_two_steps_equals_one_append():
    """append_context, draft_step: committing positions 0..4 and then 5..11
    leaves every layer's context rows in position order, the same as
    committing 0..11 at once (the second append starts at the context's
    length), and the step after it reads the same logits."""
    cfg = tiny_cfg(n_layers=2)
    W = tiny_weights(cfg)
    taps = np.random.default_rng(23).standard_normal((12, cfg["n_taps"] * cfg["hidden"]))
    st = O.Store(False)
    once = O.append_context(cfg, W, empty_ctx(cfg), taps, 0, st)
    first = O.append_context(cfg, W, empty_ctx(cfg), taps[:5], 0, st)
    twice = O.append_context(cfg, W, first, taps[5:], 5, st)
    c1, _, _, _ = O.draft_step(cfg, W, [empty_ctx(cfg)], [7], [taps[:5]], st)
    c2, z2, _, _ = O.draft_step(cfg, W, c1, [7], [taps[5:]], st)
    for l in range(cfg["n_layers"]):
        for i in range(2):
            np.testing.assert_allclose(twice[l][i], once[l][i], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(c2[0][l][i], once[l][i], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(z2[0], O.draft_block(cfg, W, 7, once, st), rtol=1e-10, atol=1e-12)


def test_draft_step_sequences_are_independent():
    """draft_step: a batch of sequences gives, row for row, what each
    sequence gives alone (its own anchor, context and new taps)."""
    cfg = tiny_cfg()
    W = tiny_weights(cfg)
    st = O.Store(False)
    g = np.random.default_rng(27)
    TH = cfg["n_taps"] * cfg["hidden"]
    ctxs = [O.append_context(cfg, W, empty_ctx(cfg), g.standard_normal((n, TH)), 0, st) for n in (3, 6)]
    new = [g.standard_normal((2, TH)), g.standard_normal((1, TH))]
    anchors = [7, 11]
    _, z, ids, vals = O.draft_step(cfg, W, ctxs, anchors, new, st)
    for s in range(2):
        _, z1, ids1, vals1 = O.draft_step(cfg, W, [ctxs[s]], [anchors[s]], [new[s]], st)
        np.testing.assert_array_equal(z[s], z1[0])
        np.testing.assert_array_equal(ids[s], ids1[0])
        np.testing.assert_array_equal(vals[s], vals1[0])
    assert not np.allclose(z[0], z[1])


@pytest.mark.parametrize("kc", [0, 2])
def test_block_keys_sit_where_context_keys_at_the_same_positions_would(kc):
    """draft_layer, context_kv: the block's own keys and values are the
    context's projection, norm and rotation applied to the attention input.
    Context rows built by context_kv from that input at the block's own
    positions repeat the block's keys and values exactly; every key then
    appears twice with the same value, which leaves each query's attention
    output unchanged, so the layer equals the one with an empty context.  The
    same rows one position later do change it."""
    cfg = tiny_cfg(conv_kernel_size=kc)
    W = tiny_weights(cfg)
    Wl = W["layers"][0]
    h = np.random.default_rng(24).standard_normal((cfg["block_size"], cfg["hidden"]))
    pos = 9 + np.arange(cfg["block_size"])
    st = O.Store(False)
    u = O.rms_norm(h, Wl["attn_norm"], cfg["rms_eps"])
    u2 = u + O.dynamic_conv(u, Wl["tapgen_attn"], cfg["conv_group_size"], kc) if kc else u
    alone = O.draft_layer(cfg, Wl, h, *empty_ctx(cfg)[0], pos, st)
    K, V = O.context_kv(cfg, Wl, u2, pos, st)
    np.testing.assert_allclose(O.draft_layer(cfg, Wl, h, K, V, pos, st), alone, rtol=1e-10, atol=1e-12)
    K1, V1 = O.context_kv(cfg, Wl, u2, pos + 1, st)
    assert np.max(np.abs(O.draft_layer(cfg, Wl, h, K1, V1, pos, st) - alone)) > 1e-6


def test_draft_block_invariant_to_common_position_shift():
    # scores depend on relative positions only: shifting the context's and the
    # block's positions together leaves the logits unchanged (anchor at P).
    cfg = tiny_cfg()
    W = tiny_weights(cfg)
    taps = np.random.default_rng(11).standard_normal((6, cfg["n_taps"] * cfg["hidden"]))
    st = O.Store(False)
    ctx0 = O.append_context(cfg, W, empty_ctx(cfg), taps, 0, st)
    z0 = O.draft_block(cfg, W, 7, ctx0, st)
    # context keys at positions 40..45 but the block still placed right after 6
    # context rows (draft_block puts the anchor at the context length): a
    # mismatched offset, which must change the logits
    ctx40 = O.append_context(cfg, W, empty_ctx(cfg), taps, 40, st)
    z40 = O.draft_block(cfg, W, 7, ctx40, st)
    # both context and block moved by 40, built by hand from the same pieces
    f = O.project_features(cfg, W, taps, st)
    k, v = O.context_kv(cfg, W["layers"][0], f, 40 + np.arange(6), st)
    B = cfg["block_size"]
    toks = np.array([7] + [cfg["mask_token_id"]] * (B - 1))
    h = W["embed"][toks].astype(np.float64)
    h = O.draft_layer(cfg, W["layers"][0], h, k, v, 46 + np.arange(B), st)
    z_shift = (O.rms_norm(h[1:], W["final_norm"], 1e-6) @ W["lm_head"].T)
    np.testing.assert_allclose(z_shift, z0, rtol=1e-9, atol=1e-10)
    assert not np.allclose(z40, z0, atol=1e-6)      # a mismatched offset does change it


def test_draft_block_softcap_and_multiplier():
    cfg = tiny_cfg()
    W = tiny_weights(cfg)
    st = O.Store(False)
    ctx = O.append_context(cfg, W, empty_ctx(cfg), np.ones((2, cfg["n_taps"] * cfg["hidden"])), 0, st)
    z = O.draft_block(cfg, W, 3, ctx, st)
    z2 = O.draft_block(dict(cfg, output_multiplier=2.5), W, 3, ctx, st)
    np.testing.assert_allclose(z2, 2.5 * z, rtol=1e-13)
    z3 = O.draft_block(dict(cfg, final_logit_softcap=0.5), W, 3, ctx, st)
    np.testing.assert_allclose(z3, 0.5 * np.tanh(z / 0.5), rtol=1e-13)
    assert np.all(np.abs(z3) < 0.5)
    # both set: the multiplier scales the raw logits and the cap bounds the
    # product (a cap applied first and scaled after would exceed the cap)
    z4 = O.draft_block(dict(cfg, output_multiplier=2.5, final_logit_softcap=0.5), W, 3, ctx, st)
    np.testing.assert_allclose(z4, 0.5 * np.tanh(2.5 * z / 0.5), rtol=1e-13)
    assert np.all(np.abs(z4) <= 0.5)


def test_draft_block_readout_rows_and_gain():
    """draft_block's readout z[v] = mult * sum_i lm_head[v, i] * hn[i], hn the
    final-normed rows: permuting the rows of lm_head permutes the logits the
    same way (vocab index = row index), the readout is additive in lm_head,
    and scaling final_norm's gain by c scales every logit by c."""
    cfg = tiny_cfg()
    W = tiny_weights(cfg)
    st = O.Store(False)
    ctx = O.append_context(cfg, W, empty_ctx(cfg), np.ones((2, cfg["n_taps"] * cfg["hidden"])), 0, st)
    z = O.draft_block(cfg, W, 3, ctx, st)
    perm = np.random.default_rng(19).permutation(cfg["vocab"])
    zp = O.draft_block(cfg, dict(W, lm_head=W["lm_head"][perm]), 3, ctx, st)
    np.testing.assert_allclose(zp, z[:, perm], rtol=1e-12, atol=1e-14)
    L2 = np.random.default_rng(20).standard_normal(W["lm_head"].shape)
    za = O.draft_block(cfg, dict(W, lm_head=L2), 3, ctx, st)
    zs = O.draft_block(cfg, dict(W, lm_head=W["lm_head"] + L2), 3, ctx, st)
    np.testing.assert_allclose(zs, z + za, rtol=1e-10, atol=1e-12)
    zc = O.draft_block(cfg, dict(W, final_norm=3.0 * W["final_norm"]), 3, ctx, st)
    np.testing.assert_allclose(zc, 3.0 * z, rtol=1e-12, atol=1e-14)


def test_draft_block_input_embedding_scale_scales_the_embedded_rows():
    """draft_block: input_embedding_scale c multiplies the embedded block rows,
    so the logits equal those of a table of c-scaled embeddings at scale 1
    (the residual stream carries the scale; dropping it changes the logits)."""
    cfg = tiny_cfg()
    W = tiny_weights(cfg)
    st = O.Store(False)
    ctx = O.append_context(cfg, W, empty_ctx(cfg), np.ones((2, cfg["n_taps"] * cfg["hidden"])), 0, st)
    zc = O.draft_block(dict(cfg, input_embedding_scale=3.0), W, 3, ctx, st)
    ze = O.draft_block(cfg, dict(W, embed=3.0 * W["embed"]), 3, ctx, st)
    np.testing.assert_allclose(zc, ze, rtol=1e-12, atol=1e-13)
    assert not np.allclose(zc, O.draft_block(cfg, W, 3, ctx, st))


def test_draft_block_anchor_is_the_only_non_mask_token():
    cfg = tiny_cfg()
    W = tiny_weights(cfg)
    st = O.Store(False)
    ctx = O.append_context(cfg, W, empty_ctx(cfg), np.ones((2, cfg["n_taps"] * cfg["hidden"])), 0, st)
    za = O.draft_block(cfg, W, 3, ctx, st)
    zb = O.draft_block(cfg, W, 4, ctx, st)
    assert za.shape == (cfg["block_size"] - 1, cfg["vocab"])
    assert not np.allclose(za, zb)
    # anchor == mask id gives a block of identical tokens; only the left-looking
    # conv and positions tell positions apart
    zm = O.draft_block(cfg, W, cfg["mask_token_id"], ctx, st)
    assert np.all(np.isfinite(zm))


# ----------------------------------------------------------------------- top-k

def _topk_by_selection(z, k):
    z = list(z)
    chosen = []
    for _ in range(k):
        best = None
        for i, v in enumerate(z):
            if i in chosen:
                continue
            if best is None or v > z[best]:
                best = i
        chosen.append(best)
    return chosen


def test_topk_golden_ties():
    for k, vals, exp in read_golden("topk_ties.txt"):
        z = np.array([float(x) for x in vals.split()])
        ids, v = O.topk(z, int(k))
        assert list(ids) == [int(x) for x in exp.split()]
        np.testing.assert_array_equal(v, z[ids])


def test_topk_matches_selection_with_many_ties():
    g = np.random.default_rng(12)
    for _ in range(50):
        z = g.integers(-3, 4, size=40).astype(float)        # heavy ties
        ids, _ = O.topk(z, 7)
        assert list(ids) == _topk_by_selection(z, 7)


# -------------------------------------------------------------------- selector

def _sel_case(k, D, seed, scale=1.0):
    cfg = tiny_cfg(vocab=200, hidden=32, selector_rank=4, top_k=k, block_size=D + 1)
    g = np.random.default_rng(seed)
    W = {"embed": g.standard_normal((200, 32)), "sel": g.standard_normal((8, 32)) * 0.3 * scale}
    cand = np.stack([g.choice(199, size=k, replace=False) for _ in range(D)])
    z = np.sort(g.standard_normal((D, k)), axis=1)[:, ::-1].copy()
    return cfg, W, int(g.integers(0, 199)), cand, z


@pytest.mark.parametrize("k,D,seed", [(4, 7, 0), (3, 5, 1), (3, 5, 2), (2, 6, 3), (4, 4, 4)])
def test_viterbi_equals_brute_force(k, D, seed):
    cfg, W, anchor, cand, z = _sel_case(k, D, seed)
    p, idx, s = O.select_path(cfg, W, anchor, cand, z)
    pb, idxb, sb = O.brute_force_path(cfg, W, anchor, cand, z)
    assert list(idx) == list(idxb)
    assert list(p) == list(pb)
    assert abs(s - sb) < 1e-12


def test_viterbi_pairwise_term_changes_path():
    # with N(0,1)-scale factors some lattices pick a path other than the per-
    # position argmax, so the pairwise term is really used
    changed = 0
    for seed in range(40):
        cfg, W, anchor, cand, z = _sel_case(3, 5, 100 + seed, scale=3.0)
        _, idx, _ = O.select_path(cfg, W, anchor, cand, z)
        changed += int(np.any(idx != 0))
    assert changed > 0


def test_selector_without_pairwise_term_is_per_position_top1():
    cfg, W, anchor, cand, z = _sel_case(4, 7, 5)
    W["sel"] = np.zeros_like(W["sel"])
    p, idx, s = O.select_path(cfg, W, anchor, cand, z)
    assert list(idx) == [0] * 7                       # z sorted descending per position
    lse = np.log(np.exp(z).sum(1))
    assert abs(s - float(np.sum(z[:, 0] - lse))) < 1e-12


def test_selector_two_position_hand_example():
    # k = 2, D = 2, rank 1.  E rows: token t -> [t], W_a = [1], W_b = [1],
    # so <A[p], Bf[c]> = p * c.  Anchor 1; candidates pos1 = (2, 0), pos2 = (0, 3),
    # logits all zero.  Position 1 after anchor 1: scores (2, 0).
    # Position 2 after 2: scores (0, 6); after 0: scores (0, 0).
    cfg = dict(selector_rank=1)
    W = {"embed": np.arange(5, dtype=float)[:, None], "sel": np.array([[1.0], [1.0]])}
    cand = np.array([[2, 0], [0, 3]])
    z = np.zeros((2, 2))
    p, idx, s = O.select_path(cfg, W, 1, cand, z)
    l1 = 2 - math.log(math.exp(2) + 1)
    l2 = 6 - math.log(1 + math.exp(6))
    assert list(p) == [2, 3]
    assert abs(s - (l1 + l2)) < 1e-14


def test_selector_factor_roles_are_not_swapped():
    """selector_factors: rows 0..r-1 of W_sel (W_a) factor the predecessor and
    rows r..2r-1 (W_b) the candidate.  With E[t] = [t, 1], W_a = [1, 0] and
    W_b = [0, 1] the pairwise term is the predecessor's value p, the same for
    every candidate of a position, so the path is the per-position argmax of
    the logits; with the roles swapped it would be the candidate's value and
    the larger ids would win."""
    cfg = dict(selector_rank=1)
    W = {"embed": np.stack([np.arange(10.0), np.ones(10)], 1), "sel": np.array([[1.0, 0.0], [0.0, 1.0]])}
    cand = np.array([[2, 9], [5, 8]])
    z = np.array([[1.0, 0.0], [1.0, 0.0]])
    p, idx, s = O.select_path(cfg, W, 3, cand, z)
    assert list(p) == [2, 5]
    assert abs(s - 2 * (1.0 - math.log(math.e + 1.0))) < 1e-14
    a, b = O.selector_factors(cfg, W, np.array([7]))
    assert a[0, 0] == 7.0 and b[0, 0] == 1.0


def test_selector_ties_pick_smallest_indices():
    cfg = dict(selector_rank=1)
    W = {"embed": np.zeros((10, 1)), "sel": np.zeros((2, 1))}
    cand = np.array([[4, 5, 6], [7, 8, 9]])
    p, idx, s = O.select_path(cfg, W, 0, cand, np.zeros((2, 3)))
    assert list(idx) == [0, 0]
    assert abs(s - 2 * math.log(1 / 3)) < 1e-14


@pytest.mark.parametrize("k,D,n_max,seed", [(4, 7, 3, 6), (3, 5, 1, 7), (3, 6, 4, 8)])
def test_draft_n_max_walks_the_shorter_lattice(k, D, n_max, seed):
    # the path over positions 1..n_max is the brute-force optimum of that
    # shorter lattice (not a prefix of the full-length path in general)
    cfg, W, anchor, cand, z = _sel_case(k, D, seed, scale=3.0)
    p, idx, s = O.select_path_knobs(cfg, W, anchor, cand, z, n_max=n_max)
    pb, idxb, sb = O.brute_force_path(cfg, W, anchor, cand[:n_max], z[:n_max])
    assert list(idx) == list(idxb) and abs(s - sb) < 1e-12 and len(p) == n_max


@pytest.mark.parametrize("p_min", [0.0, 0.2])
def test_draft_n_max_above_the_block_is_clamped(p_min):
    # [llama] "Configuration Notes": the engine clamps draft_n_max to
    # block_size - 1, so any request from D up walks the whole lattice
    cfg = tiny_cfg(top_k=3, selector_rank=4)
    W = tiny_weights(cfg, seed=28)
    g = np.random.default_rng(28)
    D = 5
    cand = np.stack([g.choice(cfg["vocab"] - 1, 3, replace=False) for _ in range(D)])
    z = -np.sort(-g.standard_normal((D, 3)), axis=1) + 2.0   # confident rows: few cuts
    whole = O.select_path_knobs(cfg, W, 1, cand, z, n_max=0, p_min=p_min)
    for n_max in (D, D + 1, D + 9):
        got = O.select_path_knobs(cfg, W, 1, cand, z, n_max=n_max, p_min=p_min)
        assert list(got[1]) == list(whole[1]) and got[2] == whole[2]


def test_draft_p_min_cut_closed_form():
    # no pairwise term: T_i(j) = log softmax(z_i)[j] and the path is the
    # per-position top-1.  Rows whose entries are log-probabilities already
    # (summing to 1) make exp(T_i) the printed probability exactly.
    cfg = dict(selector_rank=1)
    W = {"embed": np.zeros((50, 1)), "sel": np.zeros((2, 1))}
    top1 = [0.9, 0.8, 0.4, 0.95, 0.7]   # the top-1 entry of each row is its first
    z = np.array([[math.log(p), math.log((1 - p) / 2), math.log((1 - p) / 2)] for p in top1])
    cand = np.arange(15).reshape(5, 3)
    for p_min, keep in [(0.0, 5), (0.25, 5), (0.5, 2), (0.85, 1), (0.95, 0), (0.3, 5)]:
        p, idx, s = O.select_path_knobs(cfg, W, 0, cand, z, p_min=p_min)
        assert len(p) == keep and list(idx) == [0] * keep
        assert abs(s - sum(math.log(x) for x in top1[:keep])) < 1e-12
    # the cut and n_max together: at most n_max, then the cut
    p, idx, s = O.select_path_knobs(cfg, W, 0, cand, z, n_max=4, p_min=0.5)
    assert len(p) == 2


def test_draft_p_min_keeps_a_transition_at_the_threshold():
    """select_path_knobs: drafting stops at a transition whose probability is
    below draft_p_min, so one exactly at it is kept.  Two equal candidates
    per position make each transition exactly 1/2."""
    cfg = dict(selector_rank=1)
    W = {"embed": np.zeros((20, 1)), "sel": np.zeros((2, 1))}
    cand = np.arange(8).reshape(4, 2)
    z = np.zeros((4, 2))
    p, idx, s = O.select_path_knobs(cfg, W, 0, cand, z, p_min=0.5)
    assert len(p) == 4 and list(idx) == [0] * 4
    p, idx, s = O.select_path_knobs(cfg, W, 0, cand, z, p_min=0.5 + 1e-9)
    assert len(p) == 0


def test_transition_logprobs_match_path_score():
    cfg, W, anchor, cand, z = _sel_case(4, 6, 9, scale=2.0)
    _, idx, s = O.select_path(cfg, W, anchor, cand, z)
    t = O.transition_logprobs(cfg, W, anchor, cand, z, idx)
    assert abs(float(np.sum(t)) - s) < 1e-12 and np.all(t <= 0)


# ---------------------------------------------------------------------- verify

def test_verify_golden_cases():
    for path, tgt, a, out, nxt in read_golden("verify_cases.txt"):
        path = [int(x) for x in path.split()]
        tgt = [int(x) for x in tgt.split()]
        ga, gout, gn = O.verify_accept(path, tgt)
        assert ga == int(a)
        assert gout == [int(x) for x in out.split()]
        assert gn == int(nxt)


def test_sampled_verify_at_temperature_zero_is_greedy():
    # one-hot target rows (temperature 0): sampled verification equals the
    # greedy rule for any draws
    g = np.random.default_rng(40)
    V, D = 6, 5
    for _ in range(200):
        target = g.integers(0, V, D + 1)
        path = np.where(g.random(D) < 0.6, target[:D], g.integers(0, V, D))
        prob = np.eye(V)[target]
        got = O.verify_sampled(path, prob, g.random(D), g.random())
        assert got == O.verify_accept(path, target)


def test_sampled_verify_first_token_follows_the_target():
    # losslessness: whatever the draft proposes, the first emitted token is
    # distributed as the target's p_0 (chi-square over 40k draws, V = 6)
    g = np.random.default_rng(41)
    p0 = np.array([0.05, 0.3, 0.15, 0.25, 0.05, 0.2])
    prob = np.stack([p0, np.full(6, 1 / 6)])
    n = 40000
    for draft in (1, 4):            # a likely and an unlikely proposal
        counts = np.zeros(6)
        for _ in range(n):
            _, toks, _ = O.verify_sampled([draft], prob, [g.random()], g.random())
            counts[toks[0]] += 1
        chi2 = float(np.sum((counts - n * p0) ** 2 / (n * p0)))
        assert chi2 < 25.0, (draft, chi2, counts / n)   # 5 dof: p < 1e-4


def test_sampled_verify_hand_cases():
    prob = np.array([[0.1, 0.6, 0.3], [0.2, 0.3, 0.5], [0.2, 0.3, 0.5]])
    # both drafts accepted (u below p): the bonus draw from row 2, cdf 0.2, 0.5, 1.0
    assert O.verify_sampled([1, 2], prob, [0.59, 0.49], 0.45) == (2, [1, 2, 1], 1)
    assert O.verify_sampled([1, 2], prob, [0.59, 0.49], 0.1) == (2, [1, 2, 0], 0)
    # first draft rejected (u = 0.6 is not below 0.6): residual [0.1, 0, 0.3]
    # / 0.4, cdf 0.25, 0.25, 1.0: u 0.2 -> token 0, u 0.5 -> token 2
    assert O.verify_sampled([1, 2], prob, [0.6, 0.0], 0.2) == (0, [0], 0)
    assert O.verify_sampled([1, 2], prob, [0.6, 0.0], 0.5) == (0, [2], 2)


def test_sampled_verify_never_draws_a_zero_probability_token():
    """verify_sampled: the draw is the first token whose cumulative mass
    exceeds u times the total, so a token with no mass is never emitted, not
    even at u = 0, in a residual row and in a bonus row alike."""
    prob = np.array([[0.0, 0.0, 0.5, 0.5, 0.0], [0.0, 0.25, 0.0, 0.75, 0.0]])
    # draft 2 rejected (0.9 is not below 0.5): residual [0, 0, 0, 0.5, 0]
    assert O.verify_sampled([2], prob, [0.9], 0.0) == (0, [3], 3)
    # draft 2 accepted: the bonus from row 1, whose first token with mass is 1
    assert O.verify_sampled([2], prob, [0.1], 0.0) == (1, [2, 1], 1)
    # u just below 1 draws the last token with mass
    assert O.verify_sampled([2], prob, [0.1], 1.0 - 1e-12) == (1, [2, 3], 3)


def test_counters_with_fewer_drafts():
    # drafted counts the drafts kept; rollback = drafted - accepted
    c = O.Counters(7)
    for a, n in [(0, 0), (2, 3), (7, 7), (1, 4)]:
        c.add(a, n)
    assert c.drafted == 14 and c.accepted == 10 and c.rollback == 4 and c.steps == 4
    assert list(c.hist[:8]) == [1, 1, 1, 0, 0, 0, 0, 1]
    # acceptance rate = accepted / drafted ([NIM] "Observe Acceptance");
    # mean acceptance length counts the target's own token: 1 + 10 / 4
    assert c.acceptance_rate == 10 / 14
    assert c.mean_acceptance_length == 3.5
    assert list(c.acc_pos) == [3, 2, 1, 1, 1, 1, 1]


def test_counter_identities():
    g = np.random.default_rng(13)
    c = O.Counters(7)
    for _ in range(500):
        path = g.integers(0, 3, 7)
        tgt = g.integers(0, 3, 8)
        a, out, _ = O.verify_accept(path, tgt)
        assert 0 <= a <= 7 and len(out) == a + 1
        c.add(a)
    assert c.hist.sum() == c.steps == 500
    assert c.drafted == 7 * c.steps
    assert c.accepted + c.rollback == c.drafted
    assert 0.0 <= c.acceptance_rate <= 1.0
    assert abs(c.mean_acceptance_length - (1 + c.accepted / c.steps)) < 1e-15
    assert c.acc_pos[0] == c.steps - c.hist[0]
    assert np.all(np.diff(c.acc_pos) <= 0)
    assert c.accepted == c.acc_pos.sum()


def test_geometric_acceptance_closed_form():
    # target agrees with the proposal independently with p at each position:
    # E[a] = sum_{m=1}^{D} p^m (2.1412 for p = 0.7, D = 7)
    g = np.random.default_rng(14)
    p, D, n = 0.7, 7, 40000
    c = O.Counters(D)
    for _ in range(n):
        path = g.integers(0, 1000, D)
        agree = g.random(D) < p
        tgt = np.append(np.where(agree, path, path + 1000), 5)
        c.add(O.verify_accept(path, tgt)[0])
    expect = sum(p ** m for m in range(1, D + 1))
    sd = np.sqrt(np.sum((np.arange(D + 1) - expect) ** 2 * c.hist) / n)
    assert abs(c.accepted / n - expect) < 4 * sd / math.sqrt(n)
    assert abs(expect - 2.1412) < 1e-4


# --------------------------------------------------------------- loss decay

def test_loss_decay_golden():
    for B, gamma, k, expr in read_golden("loss_decay.txt"):
        w = O.loss_decay_weights(int(B), float(gamma))
        assert len(w) == int(B) - 1
        exact = 1.0 if expr == "1" else math.exp(eval(expr[4:-1], {}))
        assert abs(w[int(k) - 1] - exact) < 1e-15
    w = O.loss_decay_weights(16, 7.0)
    np.testing.assert_allclose(w[1:] / w[:-1], math.exp(-1 / 7), rtol=1e-14)


# ------------------------------------------------------------- lossless loop

@pytest.mark.parametrize("D,kind", [(7, "random"), (7, "perfect"), (3, "wrong"), (5, "mixed")])
def test_speculative_generation_is_lossless(D, kind):
    g = np.random.default_rng(15)
    V = 64
    table = g.integers(0, V, V)
    greedy = O.greedy_generate(table, 3, 200)

    def propose(anchor):
        if kind == "random":
            return list(g.integers(0, V, D))
        out, t = [], anchor
        for i in range(D):
            t = int(table[t])
            if kind == "wrong" or (kind == "mixed" and g.random() < 0.3):
                out.append((t + 1) % V)
                t = out[-1]
            else:
                out.append(t)
        return out

    spec, cnt = O.speculative_generate(table, 3, 200, propose)
    assert spec == greedy
    if kind == "perfect":
        assert cnt.hist[D] == cnt.steps
    if kind == "wrong":
        assert cnt.accepted == 0


def test_bf16_storage_mode_rounds_block_outputs():
    cfg = tiny_cfg()
    W = tiny_weights(cfg)
    st = O.Store(True)
    taps = O.bf16_round(np.random.default_rng(16).standard_normal((4, cfg["n_taps"] * cfg["hidden"])))
    ctx = O.append_context(cfg, W, empty_ctx(cfg), taps, 0, st)
    for K, V in ctx:
        np.testing.assert_array_equal(K, O.bf16_round(K))
        np.testing.assert_array_equal(V, O.bf16_round(V))
    z16 = O.draft_block(cfg, W, 5, ctx, st)
    z64 = O.draft_block(cfg, W, 5, O.append_context(cfg, W, empty_ctx(cfg), taps, 0, O.Store(False)),
                        O.Store(False))
    assert 0 < np.max(np.abs(z16 - z64)) < 0.2


@pytest.mark.parametrize("kc", [0, 2])
def test_storage_points_are_the_listed_tensors(kc):
    """Store: in bf16 mode the oracle rounds exactly the tensors that the
    precision reading lists, in the order the step makes them, and nothing
    else (the residual stream and the logits stay float64): the features;
    each layer's context K and V; per layer the attention input u and, with
    the conv, u'; q, k, v; the attention output; the MLP input u and u'; the
    MLP activation; then the final-normed rows."""
    shapes = []

    class Spy(O.Store):
        def __call__(self, x):
            shapes.append(np.shape(x))
            return O.Store.__call__(self, x)

    cfg = tiny_cfg(n_layers=2, conv_kernel_size=kc)
    W = tiny_weights(cfg)
    H, I, B = cfg["hidden"], cfg["intermediate"], cfg["block_size"]
    nq, nkv, d = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    taps = O.bf16_round(np.random.default_rng(25).standard_normal((5, cfg["n_taps"] * H)))
    ctx = O.append_context(cfg, W, empty_ctx(cfg), taps, 0, Spy(True))
    assert shapes == [(5, H)] + [(5, nkv, d), (5, nkv, d)] * 2
    shapes.clear()
    O.draft_block(cfg, W, 5, ctx, Spy(True))
    conv = [(B, H)] if kc else []
    layer = [(B, H)] + conv + [(B, nq, d), (B, nkv, d), (B, nkv, d), (B, nq, d)] + [(B, H)] + conv + [(B, I)]
    assert shapes == layer * 2 + [(B - 1, H)]
