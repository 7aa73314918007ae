"""The oracle's pins catch plausible mistakes.

Each case plants one single-point mistake in a copy of the oracle's source
(a dropped term or gain, a wrong sign, index, axis or offset, a transposed or
swapped operand, swapped roles, an off-by-one, a boundary moved, a bf16
storage point dropped or added), builds the
copy as a module on the CPU, and runs every pin of tests/test_oracle_pins.py
against it: at least one pin must fail.  The oracle itself is untouched.
"""

import inspect
import itertools
import os
import types

import pytest

import tests.test_oracle_pins as PINS

SRC_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "dflash2_oracle.py")

# (name, text in the oracle, the mistake put in its place)
MUTATIONS = [
    ("rms_eps_outside_sqrt", "x / np.sqrt(ms + eps) * _f64(gamma)", "x / (np.sqrt(ms) + eps) * _f64(gamma)"),
    ("rms_gain_dropped", "x / np.sqrt(ms + eps) * _f64(gamma)", "x / np.sqrt(ms + eps)"),
    ("rope_rotation_sign", "[x1 * c - x2 * s, x2 * c + x1 * s]", "[x1 * c + x2 * s, x2 * c - x1 * s]"),
    ("rope_frequency_exponent", "(-(2.0 * np.arange(half, dtype=np.float64)) / d)",
     "(-(1.0 * np.arange(half, dtype=np.float64)) / d)"),
    ("conv_looks_right", "shifted[j:] = u[: B - j]", "shifted[: B - j] = u[j:]"),
    ("conv_taps_not_normalised", "alpha = e / e.sum(axis=-1, keepdims=True)", "alpha = e"),
    ("conv_groups_interleaved", "c += np.repeat(alpha[:, :, j], group_size, axis=1) * shifted",
     "c += np.tile(alpha[:, :, j], (1, group_size)) * shifted"),
    ("conv_tap_generator_rows_transposed", "lam = (u @ _f64(w_tap).T).reshape(B, G, kernel_size)",
     "lam = (u @ _f64(w_tap).T).reshape(B, kernel_size, G).transpose(0, 2, 1)"),
    ("features_with_final_norm", 'return st(rms_norm(x, W["hidden_norm"], cfg["rms_eps"]))',
     'return st(rms_norm(x, W["final_norm"], cfg["rms_eps"]))'),
    ("context_positions_off_by_one", "pos = start_pos + np.arange(f.shape[0])",
     "pos = start_pos + 1 + np.arange(f.shape[0])"),
    ("attention_scale_1_over_d", "scale = 1.0 / math.sqrt(d)", "scale = 1.0 / d"),
    ("attention_softmax_over_queries", "p = p / p.sum(axis=1, keepdims=True)", "p = p / p.sum(axis=0, keepdims=True)"),
    ("attention_block_keys_dropped",
     "K = np.concatenate([_f64(Kc), _f64(Kb)], 0)\n    V = np.concatenate([_f64(Vc), _f64(Vb)], 0)",
     "K = np.concatenate([_f64(Kc), _f64(Kb)[:0]], 0) if Kc.shape[0] else _f64(Kb)\n"
     "    V = np.concatenate([_f64(Vc), _f64(Vb)[:0]], 0) if Vc.shape[0] else _f64(Vb)"),
    ("attention_gqa_interleaved", "g = h // grp", "g = h % nkv"),
    ("attention_residual_dropped", 'h = h + O @ _f64(Wl["o"]).T', 'h = O @ _f64(Wl["o"]).T'),
    ("attention_output_heads_transposed", "O = st(block_attention(q, ctxK, ctxV, k, v)).reshape(B, nq * d)",
     "O = st(block_attention(q, ctxK, ctxV, k, v)).transpose(0, 2, 1).reshape(B, nq * d)"),
    ("q_and_k_rows_swapped",
     "q = qkv[:, : nq * d].reshape(B, nq, d)\n    k = qkv[:, nq * d: (nq + nkv) * d].reshape(B, nkv, d)",
     "k = qkv[:, : nkv * d].reshape(B, nkv, d)\n    q = qkv[:, nkv * d: (nq + nkv) * d].reshape(B, nq, d)"),
    ("k_and_v_rows_swapped",
     "k = qkv[:, nq * d: (nq + nkv) * d].reshape(B, nkv, d)\n    v = qkv[:, (nq + nkv) * d:].reshape(B, nkv, d)",
     "v = qkv[:, nq * d: (nq + nkv) * d].reshape(B, nkv, d)\n    k = qkv[:, (nq + nkv) * d:].reshape(B, nkv, d)"),
    ('values_rotated', '    v = st(v)\n', '    v = st(rope(v, pos, cfg["rope_theta"]))\n'),
    ('q_norm_dropped', 'rms_norm(q, Wl["q_norm"], eps)', '(q)'),
    ('k_norm_dropped', 'rms_norm(k, Wl["k_norm"], eps)', '(k)'),
    ("conv_correction_without_input", 'u2 = st(u + dynamic_conv(u, Wl["tapgen_attn"]',
     'u2 = st(0 * u + dynamic_conv(u, Wl["tapgen_attn"]'),
    ("attention_conv_reads_mlp_generator", 'u2 = st(u + dynamic_conv(u, Wl["tapgen_attn"], gs, kc)) if kc else u',
     'u2 = st(u + dynamic_conv(u, Wl["tapgen_mlp"], gs, kc)) if kc else u'),
    ("mlp_conv_reads_attention_generator", 'u2 = st(u + dynamic_conv(u, Wl["tapgen_mlp"], gs, kc)) if kc else u',
     'u2 = st(u + dynamic_conv(u, Wl["tapgen_attn"], gs, kc)) if kc else u'),
    ("mlp_norm_before_attention", '    u = st(rms_norm(h, Wl["mlp_norm"], eps))',
     '    u = st(rms_norm(h - O @ _f64(Wl["o"]).T, Wl["mlp_norm"], eps))'),
    ("gate_and_up_swapped", "act = st(silu(gu[:, :I]) * gu[:, I:])", "act = st(silu(gu[:, I:]) * gu[:, :I])"),
    ('mlp_residual_dropped', 'return h + act @ _f64(Wl["down"]).T', 'return act @ _f64(Wl["down"]).T'),
    ("window_off_by_one", "ctxK[max(0, ctxK.shape[0] - win):], ctxV[max(0, ctxV.shape[0] - win):]",
     "ctxK[max(0, ctxK.shape[0] - win + 1):], ctxV[max(0, ctxV.shape[0] - win + 1):]"),
    ("block_positions_from_zero", "pos = P + np.arange(B)", "pos = np.arange(B)"),
    ("anchor_one_position_early", "pos = P + np.arange(B)", "pos = P - 1 + np.arange(B)"),
    ("embedding_scale_dropped", 'h = cfg["input_embedding_scale"] * _f64(W["embed"])[toks]',
     'h = _f64(W["embed"])[toks]'),
    ("readout_of_the_wrong_rows", 'hn = st(rms_norm(h[1:], W["final_norm"], cfg["rms_eps"]))',
     'hn = st(rms_norm(h[:-1], W["final_norm"], cfg["rms_eps"]))'),
    ("readout_with_hidden_norm", 'hn = st(rms_norm(h[1:], W["final_norm"], cfg["rms_eps"]))',
     'hn = st(rms_norm(h[1:], W["hidden_norm"], cfg["rms_eps"]))'),
    ("topk_ties_to_larger_ids", "order = np.lexsort((np.arange(V), -flat[r]))",
     "order = np.lexsort((-np.arange(V), -flat[r]))"),
    ("selector_factor_roles_swapped", "return e @ sel[:r].T, e @ sel[r:].T", "return e @ sel[r:].T, e @ sel[:r].T"),
    ("selector_normalised_over_predecessors", "T = S - _logsumexp(S, 1)", "T = S - _logsumexp(S, 0)"),
    ("selector_ignores_the_anchor", "S1 = z[0] + Bc[0] @ Aa[0]", "S1 = z[0]"),
    ("selector_ties_to_larger_predecessor", "bp = np.argmax(tot, axis=0)",
     "bp = tot.shape[0] - 1 - np.argmax(tot[::-1], axis=0)"),
    ("p_min_boundary_moved", "while keep < n and math.exp(t[keep]) >= p_min:",
     "while keep < n and math.exp(t[keep]) > p_min + 1e-3:"),
    ("verify_without_bonus_token", "return a, path[:a] + [target[a]], target[a]", "return a, path[:a], target[a]"),
    ("verify_compares_shifted_target", "while a < D and path[a] == target[a]:",
     "while a < D and path[a] == target[a + 1]:"),
    ("sampled_accept_rule", "while a < n and float(u_accept[a]) < prob[a, path[a]]:",
     "while a < n and float(u_accept[a]) <= 0.5 * prob[a, path[a]]:"),
    ("sampled_residual_keeps_the_draft", "        row[path[a]] = 0.0\n", "        pass\n"),
    ("loss_decay_offset", "return np.exp(-(k - 1.0) / gamma)", "return np.exp(-k / gamma)"),
    ("rollback_count", "self.rollback += n - a", "self.rollback += n - a - 1"),
    ("mean_acceptance_without_bonus", "return 1.0 + self.accepted / self.steps if self.steps else 0.0",
     "return self.accepted / self.steps if self.steps else 0.0"),
    ("bf16_truncates", "np.rint(np.ldexp(x, 8 - e))", "np.trunc(np.ldexp(x, 8 - e))"),
    ("bf16_one_bit_short", "np.rint(np.ldexp(x, 8 - e)), e - 8", "np.rint(np.ldexp(x, 7 - e)), e - 7"),
    ("bf16_subnormal_floor", "e = np.maximum(e, -125)", "e = np.maximum(e, -140)"),
    ("silu_sign", "return x / (1.0 + np.exp(-x))", "return x / (1.0 + np.exp(x))"),
    ("rms_over_rows", "ms = np.mean(x * x, axis=-1, keepdims=True)", "ms = np.mean(x * x, axis=0, keepdims=True)"),
    ("conv_softmax_over_groups", "alpha = e / e.sum(axis=-1, keepdims=True)",
     "alpha = e / e.sum(axis=1, keepdims=True)"),
    ('features_unnormed', 'return st(rms_norm(x, W["hidden_norm"], cfg["rms_eps"]))', 'return st(x)'),
    ("context_keys_with_q_norm",
     'k = rope(rms_norm(k, Wl["k_norm"], cfg["rms_eps"]), np.asarray(pos), cfg["rope_theta"])',
     'k = rope(rms_norm(k, Wl["q_norm"], cfg["rms_eps"]), np.asarray(pos), cfg["rope_theta"])'),
    ("context_keys_unrotated",
     'k = rope(rms_norm(k, Wl["k_norm"], cfg["rms_eps"]), np.asarray(pos), cfg["rope_theta"])',
     'k = rms_norm(k, Wl["k_norm"], cfg["rms_eps"])'),
    ("context_keys_unnormed", 'k = rope(rms_norm(k, Wl["k_norm"], cfg["rms_eps"]), np.asarray(pos), cfg["rope_theta"])',
     'k = rope(k, np.asarray(pos), cfg["rope_theta"])'),
    ("context_new_rows_prepended", "out.append((np.concatenate([K0, k], 0), np.concatenate([V0, v], 0)))",
     "out.append((np.concatenate([k, K0], 0), np.concatenate([v, V0], 0)))"),
    ("attention_reads_keys_as_values", "O[:, h, :] = p @ V[:, g, :]", "O[:, h, :] = p @ K[:, g, :]"),
    ("block_keys_one_position_late", 'k = st(rope(rms_norm(k, Wl["k_norm"], eps), pos, cfg["rope_theta"]))',
     'k = st(rope(rms_norm(k, Wl["k_norm"], eps), pos + 1, cfg["rope_theta"]))'),
    ("queries_unrotated", 'q = st(rope(rms_norm(q, Wl["q_norm"], eps), pos, cfg["rope_theta"]))',
     'q = st(rms_norm(q, Wl["q_norm"], eps))'),
    ("block_all_anchor", 'toks = np.array([anchor] + [cfg["mask_token_id"]] * (B - 1), dtype=np.int64)',
     "toks = np.array([anchor] * B, dtype=np.int64)"),
    ("block_anchor_masked", 'toks = np.array([anchor] + [cfg["mask_token_id"]] * (B - 1), dtype=np.int64)',
     'toks = np.array([cfg["mask_token_id"]] * B, dtype=np.int64)'),
    ("softcap_unscaled", "z = cap * np.tanh(z / cap)", "z = np.tanh(z / cap)"),
    ("softcap_inner_unscaled", "z = cap * np.tanh(z / cap)", "z = cap * np.tanh(z)"),
    ("multiplier_after_cap",
     'z = cfg["output_multiplier"] * (hn @ _f64(W["lm_head"]).T)\n    cap = cfg["final_logit_softcap"]\n'
     '    if cap and cap > 0:\n        z = cap * np.tanh(z / cap)',
     'z = (hn @ _f64(W["lm_head"]).T)\n    cap = cfg["final_logit_softcap"]\n'
     '    if cap and cap > 0:\n        z = cap * np.tanh(z / cap)\n    z = cfg["output_multiplier"] * z'),
    ("topk_skips_the_best", "ids[r] = order[:k]", "ids[r] = order[1:k + 1]"),
    ("draft_step_appends_at_zero", "c = append_context(cfg, W, c, new_taps[s], P0, st)",
     "c = append_context(cfg, W, c, new_taps[s], 0, st)"),
    ("selector_first_unnormalised", "delta = S1 - _logsumexp(S1, 0)", "delta = S1"),
    ("selector_pred_factor_wrong_position", "S = z[i][None, :] + Ac[i - 1] @ Bc[i].T",
     "S = z[i][None, :] + Ac[i] @ Bc[i].T"),
    ("selector_without_unary", "S = z[i][None, :] + Ac[i - 1] @ Bc[i].T", "S = Ac[i - 1] @ Bc[i].T"),
    ("transitions_keep_anchor", "        prev_tok = int(cand_id[i, idx[i]])\n    return np.array(out)",
     "        pass\n    return np.array(out)"),
    ("path_score_keep_anchor", "        prev_tok = int(cand_id[i, idx[i]])\n    return total",
     "        pass\n    return total"),
    ("sampled_inverse_cdf_left", 'v = int(np.searchsorted(cdf, float(u_sample) * cdf[-1], side="right"))',
     'v = int(np.searchsorted(cdf, float(u_sample) * cdf[-1], side="left"))'),
    ("sampled_residual_unrenormalised", 'v = int(np.searchsorted(cdf, float(u_sample) * cdf[-1], side="right"))',
     'v = int(np.searchsorted(cdf, float(u_sample), side="right"))'),
    ("sampled_bonus_from_previous_row", "row = prob[a].copy()", "row = prob[max(a - 1, 0)].copy()"),
    ("acceptance_by_position_off_by_one", "self.acc_pos[:a] += 1",
     "self.acc_pos[:a + 1 if a < self.n_spec else a] += 1"),
    ("histogram_counts_drafts", "self.hist[a] += 1", "self.hist[n - a] += 1"),
    ("acceptance_rate_over_steps", "return self.accepted / self.drafted if self.drafted else 0.0",
     "return self.accepted / self.steps if self.steps else 0.0"),
    ("knobs_n_max_off_by_one", "n = len(cand_id) if n_max == 0 else min(n_max, len(cand_id))",
     "n = len(cand_id) if n_max == 0 else min(n_max + 1, len(cand_id))"),
    ("knobs_n_max_not_clamped", "n = len(cand_id) if n_max == 0 else min(n_max, len(cand_id))",
     "n = len(cand_id) if n_max == 0 else n_max"),
    ("knobs_cut_after", "return toks[:keep], idx[:keep], float(np.sum(t[:keep]))",
     "return toks[:keep + 1], idx[:keep + 1], float(np.sum(t[:keep + 1]))"),
    ("spec_loop_anchor_not_next", "t = [toy_target_next(table, anchor)] + [toy_target_next(table, p) for p in path]",
     "t = [toy_target_next(table, p) for p in path] + [toy_target_next(table, path[-1])]"),
    ("values_not_stored", "    v = st(v)\n", ""),
    ("activation_not_stored", "act = st(silu(gu[:, :I]) * gu[:, I:])", "act = silu(gu[:, :I]) * gu[:, I:]"),
    ("readout_rows_not_stored", 'hn = st(rms_norm(h[1:], W["final_norm"], cfg["rms_eps"]))',
     'hn = rms_norm(h[1:], W["final_norm"], cfg["rms_eps"])'),
    ("residual_stored", 'h = h + O @ _f64(Wl["o"]).T', 'h = st(h + O @ _f64(Wl["o"]).T)'),
    ("features_not_stored", 'return st(rms_norm(x, W["hidden_norm"], cfg["rms_eps"]))',
     'return rms_norm(x, W["hidden_norm"], cfg["rms_eps"])'),
    ("attention_output_not_stored", "O = st(block_attention(q, ctxK, ctxV, k, v)).reshape(B, nq * d)",
     "O = block_attention(q, ctxK, ctxV, k, v).reshape(B, nq * d)"),
    ("logits_stored", 'z = cfg["output_multiplier"] * (hn @ _f64(W["lm_head"]).T)',
     'z = st(cfg["output_multiplier"] * (hn @ _f64(W["lm_head"]).T))'),
    ("mlp_input_not_stored", '    u = st(rms_norm(h, Wl["mlp_norm"], eps))',
     '    u = rms_norm(h, Wl["mlp_norm"], eps)'),
    ("context_values_not_stored", "    return st(k), st(v)", "    return st(k), v"),
    ("topk_values_of_wrong_ids", "vals = np.take_along_axis(flat, ids, axis=1)",
     "vals = -np.sort(-flat, axis=1)[:, ::-1][:, :k]"),
    ("greedy_skips_first", "        t = toy_target_next(table, t)\n        out.append(t)",
     "        out.append(t)\n        t = toy_target_next(table, t)"),
    ("spec_loop_first_anchor_is_prompt", "    anchor = toy_target_next(table, prompt_last)\n    out.append(anchor)",
     "    anchor = int(prompt_last)\n    out.append(anchor)"),
    ("verify_all_accepted_no_bonus",
     "    while a < D and path[a] == target[a]:\n        a += 1\n    return a, path[:a] + [target[a]], target[a]",
     "    while a < D and path[a] == target[a]:\n"
     "        a += 1\n"
     "    if a == D:\n"
     "        return a, path[:a], path[-1]\n"
     "    return a, path[:a] + [target[a]], target[a]"),
    ("knobs_ignore_p_min_sign", "    if p_min <= 0.0:\n        return toks, idx, score",
     "    if p_min <= 0.5:\n        return toks, idx, score"),
    ("knobs_score_not_kept", "return toks[:keep], idx[:keep], float(np.sum(t[:keep]))",
     "return toks[:keep], idx[:keep], float(np.sum(t))"),
    ("counters_fewer_drafts_ignored", "        n = self.n_spec if n_draft is None else n_draft",
     "        n = self.n_spec"),
    ("draft_step_ctx_not_updated",
     "            c = append_context(cfg, W, c, new_taps[s], P0, st)\n        out_ctx.append(c)",
     "            append_context(cfg, W, c, new_taps[s], P0, st)\n        out_ctx.append(c)"),
    ("draft_step_anchor_of_next_seq", "        logits.append(draft_block(cfg, W, int(anchor), c, st))",
     "        logits.append(draft_block(cfg, W, int(anchors[(s + 1) % len(anchors)]), c, st))"),
    ("selector_final_argmin", "    j = int(np.argmax(delta))",
     "    j = int(np.argmax(delta[::-1]))\n    j = len(delta) - 1 - j"),
    ("selector_backtrack_off_by_one", "    for bp in reversed(back):\n        j = int(bp[j])",
     "    for bp in back:\n        j = int(bp[j])"),
    ("conv_kernel_size_ignored", "    for j in range(kernel_size):", "    for j in range(2):"),
    ("rope_theta_ignored", "inv_freq = float(theta) ** (", "inv_freq = float(10000.0) ** ("),
    ("loss_decay_gamma_inverted", "return np.exp(-(k - 1.0) / gamma)", "return np.exp(-(k - 1.0) * gamma / 49.0)"),
    ("window_counts_block", "ctxK[max(0, ctxK.shape[0] - win):], ctxV[max(0, ctxV.shape[0] - win):]",
     "ctxK[max(0, ctxK.shape[0] - max(0, win - B)):], ctxV[max(0, ctxV.shape[0] - max(0, win - B)):]"),
    ("features_taps_reversed", '    x = _f64(taps) @ _f64(W["fc"]).T', '    x = _f64(taps)[:, ::-1] @ _f64(W["fc"]).T'),
    ("sampled_accept_le", "while a < n and float(u_accept[a]) < prob[a, path[a]]:",
     "while a < n and float(u_accept[a]) <= prob[a, path[a]]:"),
]


def _calls(fn):
    """Every argument tuple a pin is run with (its parametrize marks)."""
    marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
    if not marks:
        return [{}]
    grids = []
    for m in marks:
        names = [n.strip() for n in m.args[0].split(",")] if isinstance(m.args[0], str) else list(m.args[0])
        vals = [v if len(names) > 1 else (v,) for v in m.args[1]]
        grids.append([dict(zip(names, v)) for v in vals])
    out = []
    for combo in itertools.product(*grids):
        d = {}
        for c in combo:
            d.update(c)
        out.append(d)
    return out


def _some_pin_fails(module):
    saved = PINS.O
    PINS.O = module
    try:
        for name in sorted(n for n in dir(PINS) if n.startswith("test_")):
            fn = getattr(PINS, name)
            params = set(inspect.signature(fn).parameters)
            for kw in _calls(fn):
                if set(kw) != params:
                    continue  # a pin that needs fixtures: not run here
                try:
                    fn(**kw)
                except Exception:
                    return name
        return None
    finally:
        PINS.O = saved


@pytest.mark.parametrize("name,text,mistake", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_a_planted_mistake_fails_a_pin(name, text, mistake):
    src = open(SRC_PATH).read()
    assert src.count(text) >= 1, f"{name}: the text to mutate is not in the oracle"
    mod = types.ModuleType(f"oracle_with_{name}")
    exec(compile(src.replace(text, mistake, 1), f"oracle_with_{name}", "exec"), mod.__dict__)
    caught_by = _some_pin_fails(mod)
    assert caught_by is not None, f"no pin fails with the mistake '{name}' planted in the oracle"


def test_the_oracle_itself_passes_every_pin():
    mod = types.ModuleType("oracle_copy")
    exec(compile(open(SRC_PATH).read(), "oracle_copy", "exec"), mod.__dict__)
    assert _some_pin_fails(mod) is None
