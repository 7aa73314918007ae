"""Plain, slow, float64 reference of the DFlash2 draft step, selector and verify.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline and reference legs of ``bench.py``, never by the product
path.  It shares no code with the CUDA library.

Pages cited (title, then section):
  [Train]  "Train a DFlash Drafter for Speculative Decoding"
  [vLLM]   "DFlash speculative decoding with vLLM"
  [llama]  "DFlash2 Speculative Decoding" (llama-cpp-python wiki)
  [NIM]    "DFlash2 Speculative Decoding | NVIDIA NIM for Alpamayo Documentation"

Numbers are float64 throughout.  With ``bf16=True`` the oracle rounds to
bfloat16 (round to nearest, ties to even) at exactly the points where the GPU
path stores a bf16 tensor between kernels (a reading: the pages fix no precision); everything else stays
float64.  Pin status of each function is stated in its docstring; the pins
themselves live in ``tests/test_oracle_pins.py``.

Data layout used here (plain, one sequence at a time):
  weights  dict of numpy arrays, row-major [out_features, in_features]
           embed [V,H], lm_head [V,H], fc [H,T*H], hidden_norm [H],
           final_norm [H], sel [2r,H] (rows 0..r-1 = W_a, r..2r-1 = W_b),
           layers: list of dicts with attn_norm [H], tapgen_attn [Kc*G,H],
           qkv [(nq+2nkv)*d,H] (W_q rows, then W_k, then W_v), q_norm [d],
           k_norm [d], o [H,nq*d], mlp_norm [H], tapgen_mlp [Kc*G,H],
           gate_up [2I,H] (W_gate rows, then W_up), down [H,I].
  context  per sequence, per layer: (K [P,nkv,d], V [P,nkv,d]).
"""

import math

import numpy as np

__all__ = [
    "bf16_round", "Store", "rms_norm", "rope", "silu", "dynamic_conv",
    "project_features", "context_kv", "append_context", "block_attention",
    "draft_layer", "draft_block", "topk", "draft_step", "selector_factors",
    "select_path", "select_path_knobs", "transition_logprobs", "brute_force_path", "path_score", "verify_accept",
    "verify_sampled",
    "Counters", "loss_decay_weights", "toy_target_next", "greedy_generate",
    "speculative_generate",
]


# --------------------------------------------------------------------------
# storage rounding
# --------------------------------------------------------------------------

def bf16_round(x):
    """Round float64 values to the nearest bfloat16 value (ties to even).

    bfloat16 keeps 8 significant bits and the float32 exponent range.  For a
    normal value x = m * 2**e (0.5 <= |m| < 1) the spacing is 2**(e-8); below
    the smallest normal (2**-126) the spacing stays 2**-133.  Overflow is not
    handled (no value on the path comes near 3e38).
    """
    x = np.asarray(x, dtype=np.float64)
    _, e = np.frexp(x)
    e = np.maximum(e, -125)
    return np.ldexp(np.rint(np.ldexp(x, 8 - e)), e - 8)


class Store:
    """Identity in float64 mode; bf16 rounding at storage points otherwise."""

    def __init__(self, bf16):
        self.bf16 = bool(bf16)

    def __call__(self, x):
        x = np.asarray(x, dtype=np.float64)
        return bf16_round(x) if self.bf16 else x


def _f64(a):
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# primitives
# --------------------------------------------------------------------------

def rms_norm(x, gamma, eps):
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * gamma.

    [Train] "What is DFlash?": the draft trains "its norms".  Reading taken: the
    norm is RMSNorm (the Qwen3 targets the pages name in "Key Config Fields"
    use it) with learned gain gamma and no bias.
    """
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(gamma)


def rope(x, pos, theta):
    """Rotary position embedding, rotate-half layout.  (A reading where the pages are silent.)

    x has shape [..., n_heads, d]; pos has shape x.shape[:-2].  For
    i < d/2 the pair (x[i], x[i+d/2]) is rotated by pos * theta**(-2i/d).
    """
    x = _f64(x)
    d = x.shape[-1]
    half = d // 2
    inv_freq = float(theta) ** (-(2.0 * np.arange(half, dtype=np.float64)) / d)
    ang = _f64(pos)[..., None, None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x):
    x = _f64(x)
    return x / (1.0 + np.exp(-x))


def dynamic_conv(u, w_tap, group_size, kernel_size=2):
    """DFlash2 in-block dynamic grouped convolution of one block.

    [Train] "Variants": DFlash 2 wraps each sublayer of the draft in a short
    convolution along the block (two taps); "Key Config Fields":
    conv_kernel_size counts its taps and conv_group_size is how many channels
    share one set of dynamic tap weights; [vLLM] "DFlash2 inference" calls
    these convolutions dynamic.  Reading taken where the pages stop: taps are
    predicted per position and group from the normed input and normalised by
    a softmax over the taps; the window looks left and stays in the block.

    u       [B, H]  normed sublayer input of one block (position 0 = anchor)
    w_tap   [Kc*G, H]  tap generator; row Kc*g + j is tap j of group g
    returns c [B, H] with, for channel ch in group g = ch // group_size,
        alpha[t, g, :] = softmax_j( (w_tap @ u_t)[Kc*g + j] )
        c[t, ch]       = sum_j alpha[t, g, j] * u[t - j, ch]   (u[<0] = 0)
    The window looks left only, so the anchor sees itself alone.
    """
    u = _f64(u)
    B, H = u.shape
    G = H // group_size
    lam = (u @ _f64(w_tap).T).reshape(B, G, kernel_size)
    lam = lam - lam.max(axis=-1, keepdims=True)
    e = np.exp(lam)
    alpha = e / e.sum(axis=-1, keepdims=True)            # [B, G, Kc]
    c = np.zeros_like(u)
    for j in range(kernel_size):
        shifted = np.zeros_like(u)
        if j < B:
            shifted[j:] = u[: B - j]
        c += np.repeat(alpha[:, :, j], group_size, axis=1) * shifted
    return c


# --------------------------------------------------------------------------
# stage (a): feature projection and context K/V
# --------------------------------------------------------------------------

def project_features(cfg, W, taps, st):
    """f = RMSNorm_hidden(taps @ W_fc^T).  (A reading where the pages are silent.)

    [Train] "What is DFlash?": the draft reads hidden states tapped from the
    frozen target at target_layer_ids, mapped by a trained projection;
    [vLLM] "DFlash2 inference": dflash_config carries target_layer_ids.  taps [n, T*H] is the concatenation of the T tapped
    hidden states in target_layer_ids order.  Pinned by identity and
    permutation blocks (which tap, which orientation, which gain).
    """
    x = _f64(taps) @ _f64(W["fc"]).T
    return st(rms_norm(x, W["hidden_norm"], cfg["rms_eps"]))


def context_kv(cfg, Wl, f, pos, st):
    """Context keys/values of one draft layer from projected features.

    Reading taken: the features enter every draft layer as extra keys/values,
    K = RoPE(RMSNorm_k(W_k f)), V = W_v f, at their absolute positions.
    f [n, H], pos [n] -> K, V [n, nkv, d].
    """
    nq, nkv, d = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    f = _f64(f)
    n = f.shape[0]
    wkv = _f64(Wl["qkv"])[nq * d:]
    kv = f @ wkv.T
    k = kv[:, : nkv * d].reshape(n, nkv, d)
    v = kv[:, nkv * d:].reshape(n, nkv, d)
    k = rope(rms_norm(k, Wl["k_norm"], cfg["rms_eps"]), np.asarray(pos), cfg["rope_theta"])
    return st(k), st(v)


def append_context(cfg, W, ctx, taps, start_pos, st):
    """Append the committed positions start_pos.. of one sequence to its
    per-layer context K/V (stage a1 + a2).  ctx is a list of (K, V) per layer
    (possibly empty arrays); returns the new list."""
    f = project_features(cfg, W, taps, st)
    pos = start_pos + np.arange(f.shape[0])
    out = []
    for l, Wl in enumerate(W["layers"]):
        k, v = context_kv(cfg, Wl, f, pos, st)
        K0, V0 = ctx[l]
        out.append((np.concatenate([K0, k], 0), np.concatenate([V0, v], 0)))
    return out


# --------------------------------------------------------------------------
# stage (b): non-causal block forward
# --------------------------------------------------------------------------

def block_attention(q, Kc, Vc, Kb, Vb):
    """Non-causal attention of a block over [context ; block].

    [Train] "What is DFlash?": one "non-causal forward pass" over the block;
    [vLLM] "Requirements": the backend must support "the draft model's
    non-causal attention".  Reading taken: every block query sees every context
    key and every block key, no mask, scale 1/sqrt(d), grouped-query sharing
    (q head h reads kv head h // (nq/nkv)).
    q [B, nq, d]; Kc, Vc [P, nkv, d]; Kb, Vb [B, nkv, d] -> O [B, nq, d].
    """
    q = _f64(q)
    B, nq, d = q.shape
    nkv = Kb.shape[1]
    grp = nq // nkv
    K = np.concatenate([_f64(Kc), _f64(Kb)], 0)
    V = np.concatenate([_f64(Vc), _f64(Vb)], 0)
    O = np.empty_like(q)
    scale = 1.0 / math.sqrt(d)
    for h in range(nq):
        g = h // grp
        s = (q[:, h, :] @ K[:, g, :].T) * scale          # [B, P+B]
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=1, keepdims=True)
        O[:, h, :] = p @ V[:, g, :]
    return O


def draft_layer(cfg, Wl, h, ctxK, ctxV, pos, st):
    """One draft decoder layer (Reading taken: a Qwen3-style pre-norm layer
    without biases, with the DFlash2 conv around both sublayers).

    h [B, H] residual stream of one block (float64, never rounded);
    pos [B] absolute positions of the block.

    conv_kernel_size 0 is DFlash (v1): no convolution, the sublayers read
    the normed rows ([Train] "Variants": the convolution is what DFlash 2
    adds to the block-parallel baseline).  sliding_window W > 0: the block
    reads only the last W context positions ([Train] "Key Config Fields":
    draft_sliding_window bounds how far back a block reads the context;
    unset, it reads the whole prefix).  Reading taken: the window is counted
    back from the first block position and the block's own keys are always
    read.
    """
    H = cfg["hidden"]
    nq, nkv, d = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    I = cfg["intermediate"]
    gs, kc, eps = cfg["conv_group_size"], cfg["conv_kernel_size"], cfg["rms_eps"]
    B = h.shape[0]
    win = cfg.get("sliding_window", 0)
    if win and win > 0:
        ctxK, ctxV = ctxK[max(0, ctxK.shape[0] - win):], ctxV[max(0, ctxV.shape[0] - win):]

    # attention sublayer
    u = st(rms_norm(h, Wl["attn_norm"], eps))
    u2 = st(u + dynamic_conv(u, Wl["tapgen_attn"], gs, kc)) if kc else u
    qkv = u2 @ _f64(Wl["qkv"]).T
    q = qkv[:, : nq * d].reshape(B, nq, d)
    k = qkv[:, nq * d: (nq + nkv) * d].reshape(B, nkv, d)
    v = qkv[:, (nq + nkv) * d:].reshape(B, nkv, d)
    q = st(rope(rms_norm(q, Wl["q_norm"], eps), pos, cfg["rope_theta"]))
    k = st(rope(rms_norm(k, Wl["k_norm"], eps), pos, cfg["rope_theta"]))
    v = st(v)
    O = st(block_attention(q, ctxK, ctxV, k, v)).reshape(B, nq * d)
    h = h + O @ _f64(Wl["o"]).T

    # MLP sublayer
    u = st(rms_norm(h, Wl["mlp_norm"], eps))
    u2 = st(u + dynamic_conv(u, Wl["tapgen_mlp"], gs, kc)) if kc else u
    gu = u2 @ _f64(Wl["gate_up"]).T
    act = st(silu(gu[:, :I]) * gu[:, I:])
    return h + act @ _f64(Wl["down"]).T


def draft_block(cfg, W, anchor, ctx, st):
    """Logits of block positions 1..B-1 for one sequence.

    [Train] "What is DFlash?": position 0 holds the anchor (a real token),
    the rest are MASK (mask_token_id from the config), the block is
    embedded with the target's shared, frozen embed_tokens and read out with
    its lm_head.  "Key Config Fields": input_embedding_scale scales the
    embedded block; output_multiplier / final_logit_softcapping are the
    target's logit transform (Reading taken: z = m*logit, then cap*tanh(z/cap)
    when cap > 0).  Reading taken: with P committed context positions the anchor
    sits at position P and block position i at P+i.
    Returns z [B-1, V] (float64).
    """
    B = cfg["block_size"]
    toks = np.array([anchor] + [cfg["mask_token_id"]] * (B - 1), dtype=np.int64)
    h = cfg["input_embedding_scale"] * _f64(W["embed"])[toks]
    P = ctx[0][0].shape[0]
    pos = P + np.arange(B)
    for l, Wl in enumerate(W["layers"]):
        h = draft_layer(cfg, Wl, h, ctx[l][0], ctx[l][1], pos, st)
    hn = st(rms_norm(h[1:], W["final_norm"], cfg["rms_eps"]))
    z = cfg["output_multiplier"] * (hn @ _f64(W["lm_head"]).T)
    cap = cfg["final_logit_softcap"]
    if cap and cap > 0:
        z = cap * np.tanh(z / cap)
    return z


# --------------------------------------------------------------------------
# stage (c): top-k candidates
# --------------------------------------------------------------------------

def topk(z, k):
    """The k largest entries of z (last axis), sorted by value descending,
    equal values by smaller token id first.  (A reading where the pages are silent.)

    [llama] "Configuration Notes" / [Train] "Key Config Fields":
    selector_top_k candidates are scored per position.
    Returns (ids [..., k] int64, values [..., k] float64).
    """
    z = _f64(z)
    flat = z.reshape(-1, z.shape[-1])
    V = z.shape[-1]
    ids = np.empty((flat.shape[0], k), dtype=np.int64)
    for r in range(flat.shape[0]):
        order = np.lexsort((np.arange(V), -flat[r]))
        ids[r] = order[:k]
    vals = np.take_along_axis(flat, ids, axis=1)
    return ids.reshape(z.shape[:-1] + (k,)), vals.reshape(z.shape[:-1] + (k,))


def draft_step(cfg, W, ctxs, anchors, new_taps, st):
    """Stages (a)-(c) for a batch of sequences.

    ctxs      list over sequences of per-layer (K, V) context (before append)
    anchors   [b] anchor token per sequence
    new_taps  list over sequences of [n_b, T*H] taps of the newly committed
              positions (n_b may be 0)
    Returns (new ctxs, logits [b, B-1, V], cand_id [b, B-1, k], cand_z).
    """
    out_ctx, logits = [], []
    for s, anchor in enumerate(anchors):
        P0 = ctxs[s][0][0].shape[0]
        c = ctxs[s]
        if new_taps[s] is not None and len(new_taps[s]) > 0:
            c = append_context(cfg, W, c, new_taps[s], P0, st)
        out_ctx.append(c)
        logits.append(draft_block(cfg, W, int(anchor), c, st))
    z = np.stack(logits)
    ids, vals = topk(z, cfg["top_k"])
    return out_ctx, z, ids, vals


# --------------------------------------------------------------------------
# stage (d): selector
# --------------------------------------------------------------------------

def selector_factors(cfg, W, tokens):
    """Low-rank factors of tokens: A = W_a E[tok], Bf = W_b E[tok].

    [Train] "Key Config Fields": selector_rank sets the selector's width;
    "Objective": the selector's loss conditions each position on its true
    predecessor, so a transition pairs a predecessor token with a candidate
    token.  Reading: the factors read the shared embedding.
    tokens [...] -> A, Bf [..., r].
    """
    r = cfg["selector_rank"]
    e = _f64(W["embed"])[np.asarray(tokens, dtype=np.int64)]
    sel = _f64(W["sel"])
    return e @ sel[:r].T, e @ sel[r:].T


def _logsumexp(x, axis):
    m = np.max(x, axis=axis, keepdims=True)
    return (m + np.log(np.sum(np.exp(x - m), axis=axis, keepdims=True)))


def select_path(cfg, W, anchor, cand_id, cand_z):
    """Max-score path through the candidate lattice (Viterbi).

    [Train] "Variants": the DFlash 2 selector scores pairs of consecutive
    choices and picks one candidate per position so the picks form a single
    consistent sequence; [llama] "Configuration Notes": the selector's
    transitions carry a confidence (draft_p_min).

    Score of choosing candidate j at position i after predecessor token p:
        S_i(p, j) = z_i[j] + <A[p], Bf[c_{i,j}]>
        T_i(p, j) = S_i(p, j) - logsumexp_j' S_i(p, j')
    The predecessor of position 1 is the anchor.  The path maximises the sum
    of T.  Ties: the smaller predecessor index wins each max, the smaller
    candidate index wins the final argmax.
    cand_id, cand_z [D, k].  Returns (path tokens [D], indices [D], score).
    """
    cand_id = np.asarray(cand_id, dtype=np.int64)
    z = _f64(cand_z)
    D, k = cand_id.shape
    Aa, _ = selector_factors(cfg, W, np.array([anchor]))
    Ac, Bc = selector_factors(cfg, W, cand_id)            # [D, k, r]
    S1 = z[0] + Bc[0] @ Aa[0]                              # [k]
    delta = S1 - _logsumexp(S1, 0)
    back = []
    for i in range(1, D):
        S = z[i][None, :] + Ac[i - 1] @ Bc[i].T            # [p, j]
        T = S - _logsumexp(S, 1)
        tot = delta[:, None] + T
        bp = np.argmax(tot, axis=0)                        # first max: smallest p
        delta = tot[bp, np.arange(k)]
        back.append(bp)
    j = int(np.argmax(delta))
    score = float(delta[j])
    idx = [j]
    for bp in reversed(back):
        j = int(bp[j])
        idx.append(j)
    idx = np.array(idx[::-1], dtype=np.int64)
    return cand_id[np.arange(D), idx], idx, score


def transition_logprobs(cfg, W, anchor, cand_id, cand_z, idx):
    """T_i(prev, chosen) along one path, i = 1..len(idx): the log-probability
    of each chosen transition (the selector's confidence in it)."""
    cand_id = np.asarray(cand_id, dtype=np.int64)
    z = _f64(cand_z)
    out = []
    prev_tok = int(anchor)
    for i in range(len(idx)):
        a_prev, _ = selector_factors(cfg, W, np.array([prev_tok]))
        _, b_all = selector_factors(cfg, W, cand_id[i])
        s = z[i] + b_all @ a_prev[0]
        m = s.max()
        out.append(s[idx[i]] - (m + math.log(np.exp(s - m).sum())))
        prev_tok = int(cand_id[i, idx[i]])
    return np.array(out)


def select_path_knobs(cfg, W, anchor, cand_id, cand_z, n_max=0, p_min=0.0):
    """The selector with the drafting knobs ([llama] "Configuration Notes":
    draft_n_max bounds the drafts of a step; drafting stops at a transition
    whose confidence is below draft_p_min).  (A reading where the pages are
    silent.)

    The max-score path over positions 1..n_max only (n_max = 0: all D; a
    request above D is clamped to D, as the same section says the engine
    clamps draft_n_max to block_size - 1), then cut before the first
    position whose chosen transition has probability exp(T_i) < p_min.
    Returns (kept tokens, kept indices, the kept positions' summed
    log-probability)."""
    n = len(cand_id) if n_max == 0 else min(n_max, len(cand_id))
    toks, idx, score = select_path(cfg, W, anchor, np.asarray(cand_id)[:n], np.asarray(cand_z)[:n])
    if p_min <= 0.0:
        return toks, idx, score
    t = transition_logprobs(cfg, W, anchor, np.asarray(cand_id)[:n], np.asarray(cand_z)[:n], idx)
    keep = 0
    while keep < n and math.exp(t[keep]) >= p_min:
        keep += 1
    return toks[:keep], idx[:keep], float(np.sum(t[:keep]))


def path_score(cfg, W, anchor, cand_id, cand_z, idx):
    """Sum of transition log-probabilities of one path, computed directly
    from its definition (used by the brute-force search)."""
    cand_id = np.asarray(cand_id, dtype=np.int64)
    z = _f64(cand_z)
    D, k = cand_id.shape
    total = 0.0
    prev_tok = int(anchor)
    for i in range(D):
        a_prev, _ = selector_factors(cfg, W, np.array([prev_tok]))
        _, b_all = selector_factors(cfg, W, cand_id[i])
        s = z[i] + b_all @ a_prev[0]
        m = s.max()
        total += s[idx[i]] - (m + math.log(np.exp(s - m).sum()))
        prev_tok = int(cand_id[i, idx[i]])
    return total


def brute_force_path(cfg, W, anchor, cand_id, cand_z):
    """Exhaustive search over all k**D paths (tiny lattices only).  Ties go to
    the lexicographically smallest index sequence, scanning the last position
    fastest -- the same order the Viterbi tie rule produces."""
    cand_id = np.asarray(cand_id, dtype=np.int64)
    D, k = cand_id.shape
    best, best_idx = -np.inf, None
    for flat in range(k ** D):
        idx = []
        x = flat
        for _ in range(D):
            idx.append(x % k)
            x //= k
        idx = idx[::-1]
        s = path_score(cfg, W, anchor, cand_id, cand_z, idx)
        if s > best:
            best, best_idx = s, idx
    best_idx = np.array(best_idx, dtype=np.int64)
    return cand_id[np.arange(D), best_idx], best_idx, best


# --------------------------------------------------------------------------
# verify / accept / rollback and counters
# --------------------------------------------------------------------------

def verify_accept(path, target):
    """Greedy verification of one proposal.  (A reading where the pages are silent.)

    [llama] "Prerequisites": the target verifies [id_last, draft...] in one
    batch; t_i is the target's greedy token after [anchor, path_1..path_{i-1}],
    i = 1..B.  The accepted length is the longest prefix with path_i == t_i;
    the output is path_1..path_a followed by the target's own token t_{a+1},
    which becomes the next anchor ([vLLM] "Validation": generated token ids
    must equal plain greedy decoding).
    path [D], target [D+1] -> (a, out tokens [a+1], next anchor).
    """
    path = [int(x) for x in path]
    target = [int(x) for x in target]
    D = len(path)
    a = 0
    while a < D and path[a] == target[a]:
        a += 1
    return a, path[:a] + [target[a]], target[a]


def verify_sampled(path, prob, u_accept, u_sample):
    """Sampled (temperature > 0) verification of one proposal.  (A reading
    where the pages are silent on the mechanics.)

    [Train] (spec_generate): temperature, top_p and top_k truncate the
    target's distribution, the one rejection sampling verifies against, so
    sampled decoding stays lossless with respect to the target sampling on
    its own; [llama] "Configuration Notes": DFlash2 proposes through its
    selector lattice, not by sampling the vocabulary.  Reading taken: the
    proposal is a point mass on the selector's path, so the rejection rule
    min(1, p/q) becomes "accept draft i when u_accept[i] < p_i(path_i)"; at
    the first rejection the emitted token is drawn from p_i with path_i
    removed and renormalised (the residual max(0, p - q)); when every draft
    is accepted the bonus token is drawn from p_D.  A draw is the inverse
    CDF in token-id order: the first token whose cumulative mass exceeds
    u_sample times the total.
    path [n] kept drafts; prob [>= n+1, V] rows p_0..p_n; u_accept [>= n];
    u_sample scalar.  Returns (a, emitted tokens [a+1], next anchor).
    """
    path = [int(x) for x in path]
    prob = np.asarray(prob, dtype=np.float64)
    n = len(path)
    a = 0
    while a < n and float(u_accept[a]) < prob[a, path[a]]:
        a += 1
    row = prob[a].copy()
    if a < n:
        row[path[a]] = 0.0
    cdf = np.cumsum(row)
    v = int(np.searchsorted(cdf, float(u_sample) * cdf[-1], side="right"))
    v = min(v, len(row) - 1)
    return a, path[:a] + [v], v


class Counters:
    """Speculative-decoding counters ([NIM] "Observe Acceptance":
    num_spec_steps, num_draft_tokens, num_accepted_draft_tokens,
    acceptance_histogram; [llama] "Compare With Ordinary Decoding":
    acceptance by position and rollback counts)."""

    def __init__(self, n_spec):
        self.n_spec = n_spec
        self.steps = 0
        self.drafted = 0
        self.accepted = 0
        self.rollback = 0
        self.hist = np.zeros(n_spec + 1, dtype=np.int64)
        self.acc_pos = np.zeros(n_spec, dtype=np.int64)

    def add(self, a, n_draft=None):
        """One verified step with a accepted of n_draft drafted tokens (all
        n_spec unless the drafting knobs kept fewer)."""
        n = self.n_spec if n_draft is None else n_draft
        self.steps += 1
        self.drafted += n
        self.accepted += a
        self.rollback += n - a
        self.hist[a] += 1
        self.acc_pos[:a] += 1

    @property
    def acceptance_rate(self):
        return self.accepted / self.drafted if self.drafted else 0.0

    @property
    def mean_acceptance_length(self):
        return 1.0 + self.accepted / self.steps if self.steps else 0.0


def loss_decay_weights(block_size, gamma):
    """w_k = exp(-(k-1)/gamma) for block positions k = 1..block_size-1.

    [Train] "Objective": only positions 1..block_size-1 are supervised and
    weighted by this decay."""
    k = np.arange(1, block_size, dtype=np.float64)
    return np.exp(-(k - 1.0) / gamma)


# --------------------------------------------------------------------------
# lossless loop with a toy deterministic target (oracle-only integration)
# --------------------------------------------------------------------------

def toy_target_next(table, tok):
    """Toy greedy target: the next token is a fixed function of the last."""
    return int(table[int(tok)])


def greedy_generate(table, prompt_last, n):
    out, t = [], int(prompt_last)
    for _ in range(n):
        t = toy_target_next(table, t)
        out.append(t)
    return out


def speculative_generate(table, prompt_last, n, propose):
    """Draft -> verify -> accept loop against the toy target.

    propose(anchor) returns D draft tokens.  The target's greedy tokens for
    [anchor, path...] are t_1 = next(anchor), t_{i+1} = next(path_i).
    Returns (tokens, Counters)."""
    out = []
    anchor = toy_target_next(table, prompt_last)
    out.append(anchor)
    cnt = None
    while len(out) < n:
        path = list(propose(anchor))
        if cnt is None:
            cnt = Counters(len(path))
        t = [toy_target_next(table, anchor)] + [toy_target_next(table, p) for p in path]
        a, toks, nxt = verify_accept(path, t)
        cnt.add(a)
        out.extend(toks)
        anchor = nxt
    return out[:n], cnt
