"""Shared helpers of the GPU parity tests: build the library, place seeded
inputs on the device, run the same case through the oracle."""

import numpy as np

import dflash2_synth as S
import oracle as O

TOL = {"f32": 1e-4, "bf16": 2e-2, "fp8w": 2e-2}


def e2e_tol(case):
    """End-to-end logit bound of a full-size case: max(2e-2, 1.6 x the
    oracle's own bf16 rounding-chaos floor at that case), the floor measured
    by tests/golden/make_bf16_chaos_floor.py (oracle only) and stored in
    tests/golden/bf16_chaos_floor.txt."""
    from tests.conftest import read_golden
    floors = {k: float(v) for k, v in read_golden("bf16_chaos_floor.txt")}
    return max(2e-2, 1.6 * floors[case])


# Near-ties allowed by the discrete checks, recorded per case and written to
# tests/near_tie_counts.txt when the session ends (tests/conftest.py).
NEAR_TIES = {}


def record_near_ties(case, kind, count, total):
    NEAR_TIES[(case, kind)] = (count, total)


def lib():
    from block_speculative_decoding_dflash2_gb300 import build as bld
    bld.build()
    from block_speculative_decoding_dflash2_gb300 import binding
    binding.lib()
    return binding


def empty_ctx(cfg):
    z = np.zeros((0, cfg["n_kv_heads"], cfg["head_dim"]))
    return [(z, z) for _ in range(cfg["n_layers"])]


def topk_compare(cand_gpu, z_ref, k, tol):
    """End-to-end top-k parity against the oracle's own logits.  A row may
    differ from the oracle's top-k only where the oracle itself rates the GPU's
    pick within 4*tol of its own pick at that rank (a near-tie); those rows
    are counted and returned, anything else fails."""
    ids_ref, _ = O.topk(z_ref, k)
    g = np.asarray(cand_gpu).reshape(-1, k)
    o = ids_ref.reshape(-1, k)
    z = np.asarray(z_ref).reshape(g.shape[0], -1)
    near = 0
    for r in range(g.shape[0]):
        if np.array_equal(g[r], o[r]):
            continue
        bad = [j for j in range(k) if g[r, j] != o[r, j] and abs(z[r, g[r, j]] - z[r, o[r, j]]) >= 4 * tol]
        if bad:
            raise AssertionError(f"row {r}: top-k {list(g[r])} vs oracle {list(o[r])}")
        near += 1
    return near


class Case:
    """One batch: weights, paged prefill, a draft step's new rows and anchors."""

    def __init__(self, cfg, weights=None, ctx_lens=None, n_new=None, seed=7, spare_pages=3):
        import torch
        from block_speculative_decoding_dflash2_gb300.runner import DraftRunner

        self.cfg = cfg
        self.W = weights if weights is not None else S.make_weights(cfg)
        self.Wv = S.values_of(self.W)
        b = len(ctx_lens)
        self.b = b
        self.ctx_lens = np.asarray(ctx_lens, dtype=np.int32)
        self.n_new = np.asarray(n_new, dtype=np.int32)
        ps = cfg["page_size"]
        max_ctx = int(np.max(self.ctx_lens + self.n_new)) + 1
        bt, n_pages = S.paged_layout(max_ctx, ps, b, seed, spare_pages=spare_pages)
        self.taps_pre = S.make_taps(cfg, int(self.ctx_lens.sum()), stream=f"prefill{seed}")
        self.taps_new = S.make_taps(cfg, int(self.n_new.sum()), stream=f"step{seed}")
        self.anchor = S.make_tokens(cfg, (b,), stream=f"anchor{seed}")
        self.runner = DraftRunner(cfg, S.device_weights(self.W), b, max_ctx,
                                  max_new=int(max(self.ctx_lens.sum(), self.n_new.sum(), 1)),
                                  block_table=torch.from_numpy(bt), n_pages=n_pages)
        self.torch = torch

    def dev(self, a, dtype=None):
        t = self.torch.from_numpy(np.ascontiguousarray(a)).cuda()
        return t if dtype is None else t.to(dtype)

    def run_gpu(self, debug=True):
        torch = self.torch
        cfg = self.cfg
        pre_off = np.concatenate([[0], np.cumsum(self.ctx_lens)]).astype(np.int32)
        zeros = np.zeros(self.b, dtype=np.int32)
        r = self.runner
        if self.taps_pre.shape[0] > 0:
            r.append(self.dev(zeros), S.to_torch(self.taps_pre), self.dev(pre_off))
        new_off = np.concatenate([[0], np.cumsum(self.n_new)]).astype(np.int32)
        D, V = cfg["block_size"] - 1, cfg["vocab"]
        self.debug = torch.full((self.b, D, V), float("nan"), device="cuda") if debug else None
        taps = S.to_torch(self.taps_new) if self.taps_new.shape[0] > 0 else None
        r.draft(self.dev(self.ctx_lens), taps, self.dev(new_off), self.dev(self.anchor), self.debug)
        torch.cuda.synchronize()
        self.status = r.device_status()
        return self

    def oracle_logits(self, seqs=None):
        """The oracle's logits of every sequence, or of the sampled `seqs`
        (sequences are independent: each is computed from its own rows)."""
        cfg = self.cfg
        st = O.Store(cfg["dtype"] != "f32")
        pre = np.concatenate([[0], np.cumsum(self.ctx_lens)])
        new = np.concatenate([[0], np.cumsum(self.n_new)])
        out = []
        for s in (range(self.b) if seqs is None else seqs):
            L, n = int(self.ctx_lens[s]), int(self.n_new[s])
            p0, n0 = int(pre[s]), int(new[s])
            ctx = empty_ctx(cfg)
            if L:
                ctx = O.append_context(cfg, self.Wv, ctx, self.taps_pre.values[p0:p0 + L], 0, st)
            if n:
                ctx = O.append_context(cfg, self.Wv, ctx, self.taps_new.values[n0:n0 + n], L, st)
            out.append(O.draft_block(cfg, self.Wv, int(self.anchor[s]), ctx, st))
        return np.stack(out)
