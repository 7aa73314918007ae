"""Seeded synthetic inputs for the DFlash2 draft step.

This module only draws random numbers and converts storage formats.  It
holds none of the method's arithmetic and imports neither the oracle nor the
CUDA library; both the tests and ``bench.py`` take their inputs from here.

Recipe (per workload, seed = 1000 + workload index):
  * matrices ~ N(0, 0.02), norm gains ~ 1 + N(0, 0.1);
  * target-layer taps ~ N(0, 1), each row divided by its RMS for the bf16
    workloads (plain N(0, 1) for the tiny fp32 one);
  * bf16 workloads round every drawn value to bfloat16 (nearest, ties to
    even) before either side sees it, so both sides read identical values.
Each tensor has its own PCG64 stream keyed by (seed, tensor name).
"""

import hashlib

import numpy as np

# ---------------------------------------------------------------------------
# workloads (shapes from the pages' targets: a tiny fp32 case, an 8B-class
# Qwen3 shape at batch 1 and batch 32, a 27B-class shape, a 30B-A3B-class
# shape with fp8 weights)
# ---------------------------------------------------------------------------

_COMMON = dict(n_taps=3, conv_kernel_size=2, conv_group_size=32, page_size=16,
               rms_eps=1e-6, rope_theta=1.0e6, input_embedding_scale=1.0,
               output_multiplier=1.0, final_logit_softcap=0.0)

WORKLOADS = {
    "tiny_fp32": dict(_COMMON, index=0, dtype="f32", hidden=256, n_q_heads=4,
                      n_kv_heads=4, head_dim=64, intermediate=1024, vocab=4096,
                      n_layers=1, block_size=8, top_k=4, selector_rank=16,
                      batch=1, context=128),
    "qwen3_8b_b1": dict(_COMMON, index=1, dtype="bf16", hidden=4096, n_q_heads=32,
                        n_kv_heads=8, head_dim=128, intermediate=12288,
                        vocab=151936, n_layers=1, block_size=8, top_k=16,
                        selector_rank=64, batch=1, context=2048),
    "qwen3_8b_b32_paged": dict(_COMMON, index=2, dtype="bf16", hidden=4096,
                               n_q_heads=32, n_kv_heads=8, head_dim=128,
                               intermediate=12288, vocab=151936, n_layers=1,
                               block_size=8, top_k=16, selector_rank=64,
                               batch=32, context=(512, 4096), accept_p=0.7),
    "qwen3_27b_b8": dict(_COMMON, index=3, dtype="bf16", hidden=5120, n_q_heads=40,
                         n_kv_heads=8, head_dim=128, intermediate=17408,
                         vocab=151936, n_layers=1, block_size=16, top_k=16,
                         selector_rank=64, batch=8, context=8192),
    # 30B-A3B-shaped throughput sweep: batch {1, 8, 64, 256} x context {1k, 8k}
    # (config_of(..., batch=b, context=c)); the draft attention is sized on
    # its own (32 q / 4 kv heads x 128), MLP 3H, groups of 32 channels
    "a3b_30b_fp8": dict(_COMMON, index=4, dtype="fp8w", hidden=2688, n_q_heads=32,
                        n_kv_heads=4, head_dim=128, intermediate=8064,
                        vocab=131072, n_layers=2, block_size=7, top_k=16,
                        selector_rank=32, batch=1, context=1024),
}
A3B_SWEEP = [(b, c) for b in (1, 8, 64, 256) for c in (1024, 8192)]


def config_of(name, **over):
    """Model/config dict of a workload (mask token = vocab - 1)."""
    c = dict(WORKLOADS[name])
    c.update(over)
    c.setdefault("mask_token_id", c["vocab"] - 1)
    return c


# ---------------------------------------------------------------------------
# format conversion (storage only)
# ---------------------------------------------------------------------------

def to_bf16_bits(x):
    """float32 array -> uint16 bfloat16 bit patterns, nearest-even rounding."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits):
    """uint16 bfloat16 bit patterns -> float32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


class Tensor:
    """A drawn tensor: exact values plus its stored form: bf16 bit patterns,
    or, for an fp8 matrix, e4m3 codes `q` with per-row float32 scales (then
    `values` = decoded code * scale, exactly, in float64)."""

    __slots__ = ("values", "bits", "q", "scale")

    def __init__(self, values, bits=None, q=None, scale=None):
        self.values = values
        self.bits = bits
        self.q = q
        self.scale = scale

    @property
    def shape(self):
        return self.values.shape


# ---------------------------------------------------------------------------
# fp8 e4m3 weights (the format: 1 sign bit, 4 exponent bits with bias 7, 3
# mantissa bits; exponent field 0 holds the subnormals m/8 * 2^-6; the
# largest finite magnitude is 448; code 0x7f / 0xff is NaN, never produced)
# ---------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_encode(x):
    """float array -> e4m3 codes (uint8), round to nearest, ties to even;
    magnitudes above 448 saturate to 448."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.uint8) << np.uint8(7)
    a = np.minimum(np.abs(x), E4M3_MAX)
    e = np.clip(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6, 8)
    m = np.rint(a / np.exp2(e - 3))          # spacing 2^(e-3); exact quotient, half-even rounding
    carry = m >= 16                          # rounded up to the next power of two
    e = np.where(carry, e + 1, e)
    m = np.where(carry, m / 2, m)
    code = np.where(m >= 8, ((e + 7).astype(np.int64) << 3) | (m - 8).astype(np.int64), m.astype(np.int64))
    return code.astype(np.uint8) | sign


def e4m3_decode(q):
    """e4m3 codes -> float64 values (NaN codes -> nan)."""
    q = np.asarray(q, dtype=np.uint8).astype(np.int64)
    s, e, m = (q >> 7) & 1, (q >> 3) & 15, q & 7
    v = np.where(e == 0, m * 2.0 ** -9, (8 + m) * np.exp2(e.astype(np.float64) - 10))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return np.where(s == 1, -v, v)


def quantize_rows_e4m3(w):
    """Per-output-channel quantisation of a [rows, cols] matrix: scale =
    max|row| / 448 (float32), q = e4m3(w / scale).  Returns a Tensor whose
    values are the dequantised q * scale (float64, exact)."""
    w = np.asarray(w, dtype=np.float32)
    amax = np.max(np.abs(w), axis=1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    q = e4m3_encode(w.astype(np.float64) / scale.astype(np.float64)[:, None])
    values = e4m3_decode(q) * scale.astype(np.float64)[:, None]
    return Tensor(values, q=q, scale=scale)


def _rng(seed, name):
    h = int.from_bytes(hashlib.sha256(name.encode()).digest()[:8], "little")
    return np.random.Generator(np.random.PCG64([seed, h]))


_CHUNK = 1 << 22  # elements per independent stream of a large tensor


def _fill(out, bits, seed, name, lo, hi, std, mean, dtype):
    x = _rng(seed, f"{name}#{lo // _CHUNK}").standard_normal(size=hi - lo, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    if dtype in ("bf16", "fp8w"):
        b = to_bf16_bits(x)
        bits[lo:hi] = b
        out[lo:hi] = bf16_bits_to_f32(b)
    else:
        out[lo:hi] = x


def _draw(seed, name, shape, std, dtype, mean=0.0):
    """N(mean, std) draws; large tensors are cut into chunks of _CHUNK
    elements, each from its own stream (seed, name#chunk), filled in parallel."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    bits = np.empty(n, dtype=np.uint16) if dtype in ("bf16", "fp8w") else None
    bounds = [(lo, min(n, lo + _CHUNK)) for lo in range(0, n, _CHUNK)]
    if len(bounds) > 1:
        import concurrent.futures
        import os
        with concurrent.futures.ThreadPoolExecutor(min(32, os.cpu_count() or 4)) as ex:
            list(ex.map(lambda b: _fill(out, bits, seed, name, b[0], b[1], std, mean, dtype), bounds))
    else:
        for lo, hi in bounds:
            _fill(out, bits, seed, name, lo, hi, std, mean, dtype)
    return Tensor(out.reshape(shape), None if bits is None else bits.reshape(shape))


def make_weights(cfg, seed=None):
    """All draft weights of a workload, as a dict of Tensor (layers: list).
    With dtype "fp8w" the matrices other than the embedding are drawn in
    float32 and quantised per output channel to e4m3 (quantize_rows_e4m3);
    the embedding and the norm gains are bf16."""
    seed = 1000 + cfg["index"] if seed is None else seed
    dt = cfg["dtype"]
    if dt == "fp8w":
        def mat(name, shape):
            return quantize_rows_e4m3(_draw(seed, name, shape, 0.02, "f32").values)
        dt = "bf16"
    else:
        def mat(name, shape):
            return _draw(seed, name, shape, 0.02, dt)
    H, V, T = cfg["hidden"], cfg["vocab"], cfg["n_taps"]
    nq, nkv, d, I = cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["intermediate"]
    G = H // cfg["conv_group_size"]
    kc, r = cfg["conv_kernel_size"], cfg["selector_rank"]
    w = {
        "embed": _draw(seed, "embed", (V, H), 0.02, dt),
        "lm_head": mat("lm_head", (V, H)),
        "fc": mat("fc", (H, T * H)),
        "hidden_norm": _draw(seed, "hidden_norm", (H,), 0.1, dt, 1.0),
        "final_norm": _draw(seed, "final_norm", (H,), 0.1, dt, 1.0),
        "sel": mat("sel", (2 * r, H)),
        "layers": [],
    }
    for l in range(cfg["n_layers"]):
        p = f"layer{l}."
        w["layers"].append({
            "attn_norm": _draw(seed, p + "attn_norm", (H,), 0.1, dt, 1.0),
            "tapgen_attn": mat(p + "tapgen_attn", (kc * G, H)),
            "qkv": mat(p + "qkv", ((nq + 2 * nkv) * d, H)),
            "q_norm": _draw(seed, p + "q_norm", (d,), 0.1, dt, 1.0),
            "k_norm": _draw(seed, p + "k_norm", (d,), 0.1, dt, 1.0),
            "o": mat(p + "o", (H, nq * d)),
            "mlp_norm": _draw(seed, p + "mlp_norm", (H,), 0.1, dt, 1.0),
            "tapgen_mlp": mat(p + "tapgen_mlp", (kc * G, H)),
            "gate_up": mat(p + "gate_up", (2 * I, H)),
            "down": mat(p + "down", (H, I)),
        })
    return w


def values_of(w):
    """Weight dict of Tensor -> weight dict of float32 value arrays."""
    out = {k: v.values for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: v.values for k, v in L.items()} for L in w["layers"]]
    return out


def make_taps(cfg, n_rows, seed=None, stream="taps"):
    """[n_rows, T*H] target-layer taps (row-RMS-normalised for bf16)."""
    seed = 1000 + cfg["index"] if seed is None else seed
    x = _rng(seed, stream).standard_normal(size=(n_rows, cfg["n_taps"] * cfg["hidden"]),
                                           dtype=np.float32)
    if cfg["dtype"] != "f32":  # bf16 activations (also with fp8 weights)
        x /= np.sqrt(np.mean(x.astype(np.float64) ** 2, axis=1, keepdims=True)).astype(np.float32)
        bits = to_bf16_bits(x)
        return Tensor(bf16_bits_to_f32(bits), bits)
    return Tensor(x)


def make_context_lengths(cfg, seed=None):
    """Per-sequence context lengths (fixed, or uniform in [lo, hi])."""
    seed = 1000 + cfg["index"] if seed is None else seed
    c = cfg["context"]
    if isinstance(c, tuple):
        return _rng(seed, "ctx_len").integers(c[0], c[1] + 1, size=cfg["batch"]).astype(np.int32)
    return np.full(cfg["batch"], c, dtype=np.int32)


def make_tokens(cfg, shape, seed=None, stream="tokens"):
    """Uniform random token ids in [0, vocab - 1) (never the mask id)."""
    seed = 1000 + cfg["index"] if seed is None else seed
    return _rng(seed, stream).integers(0, cfg["vocab"] - 1, size=shape).astype(np.int32)


def make_target_logits(cfg, seed=None, stream="target_logits"):
    """[b, B, V] float32 N(0,1) logits whose argmax is the toy target's token."""
    seed = 1000 + cfg["index"] if seed is None else seed
    return _rng(seed, stream).standard_normal(
        size=(cfg["batch"], cfg["block_size"], cfg["vocab"]), dtype=np.float32)


def make_agreeing_target(path, cfg, p, seed=None, stream="agree"):
    """Target tokens that agree with the proposed path at each position with
    probability p (else a different random token); the bonus slot is random.
    path [b, D] -> target [b, D+1]."""
    seed = 1000 + cfg["index"] if seed is None else seed
    g = _rng(seed, stream)
    b, D = path.shape
    V = cfg["vocab"]
    t = g.integers(0, V - 1, size=(b, D + 1)).astype(np.int32)
    agree = g.random(size=(b, D)) < p
    other = t[:, :D]
    other = np.where(other == path, (other + 1) % (V - 1), other)
    t[:, :D] = np.where(agree, path, other)
    return t


def make_target_probs(n_rows, V, seed, stream="target_probs", temperature=1.0, top_p=0.95, top_k=20, scale=3.0):
    """Synthetic target distributions for sampled verification: N(0, scale)
    logits, temperature, then the target's own truncation (top-k, then the
    smallest top-p nucleus in probability order), renormalised; float32
    [n_rows, V] with zeros outside the kept tokens.  The settings default to
    the ones the DFlash 2 evaluations quote (1.0, 0.95, 20)."""
    z = _rng(seed, stream).standard_normal((n_rows, V)) * scale / temperature
    order = np.argsort(-z, axis=1, kind="stable")
    zs = np.take_along_axis(z, order, axis=1)
    keep = np.zeros_like(zs, dtype=bool)
    keep[:, :min(top_k, V)] = True
    ps = np.exp(zs - zs[:, :1]) * keep
    ps /= ps.sum(axis=1, keepdims=True)
    cum = np.cumsum(ps, axis=1)
    keep &= (cum - ps) < top_p               # a token is kept while the mass before it is below top_p
    ps = ps * keep
    ps /= ps.sum(axis=1, keepdims=True)
    out = np.zeros_like(ps)
    np.put_along_axis(out, order, ps, axis=1)
    return out.astype(np.float32)


def paged_layout(ctx_cap, page_size, batch, seed, spare_pages=0):
    """Block table [batch, max_pages] as a seeded random permutation of
    physical pages; returns (block_table int32, n_pages)."""
    max_pages = -(-int(ctx_cap) // page_size)
    n_pages = batch * max_pages + spare_pages
    perm = _rng(seed, "pages").permutation(n_pages).astype(np.int32)
    return perm[: batch * max_pages].reshape(batch, max_pages), n_pages


# ---------------------------------------------------------------------------
# torch placement (format conversion only)
# ---------------------------------------------------------------------------

def to_torch(t, device="cuda"):
    """Tensor -> torch tensor on `device` (bf16 from its bit patterns; an fp8
    matrix as its uint8 e4m3 codes)."""
    import torch
    if t.q is not None:
        return torch.from_numpy(np.ascontiguousarray(t.q)).to(device)
    if t.bits is not None:
        return torch.from_numpy(t.bits.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(t.values)).to(device)


def device_weights(w, device="cuda"):
    """Weight dict of Tensor -> weight dict of torch device tensors; with fp8
    matrices, also "scales": their per-row float32 scales in the same nesting."""
    import torch
    out = {k: to_torch(v, device) for k, v in w.items() if k != "layers"}
    out["layers"] = [{k: to_torch(v, device) for k, v in L.items()} for L in w["layers"]]
    if w["lm_head"].q is not None:
        sc = lambda t: torch.from_numpy(t.scale).to(device)
        out["scales"] = {k: sc(w[k]) for k in ("lm_head", "fc", "sel")}
        out["scales"]["layers"] = [{k: sc(v) for k, v in L.items() if v.q is not None} for L in w["layers"]]
    return out


def small_bf16_config(**over):
    """A small bf16 shape that still spans several tiles with ragged edges:
    V = 1000 (7 full 128-row tiles + 104), 2 layers, GQA 4:2."""
    c = dict(_COMMON, index=10, dtype="bf16", hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64,
             intermediate=704, vocab=1000, n_layers=2, block_size=8, top_k=8, selector_rank=16,
             batch=3, context=(40, 200))
    c.update(over)
    c.setdefault("mask_token_id", c["vocab"] - 1)
    return c
