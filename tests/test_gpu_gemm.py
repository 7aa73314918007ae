"""Parity of the dense contraction (tcgen05 + TMA path for bf16, SIMT path for
fp32) and of the lm_head's streaming top-k against a float64 matrix product
and the oracle's top-k."""

import numpy as np
import pytest

import dflash2_synth as S
import oracle as O
from tests.helpers import lib

pytestmark = pytest.mark.gpu


def _mat(rows, cols, seed, std, dtype):
    return S._draw(seed, f"m{rows}x{cols}", (rows, cols), std, dtype)


@pytest.mark.parametrize("M,N,K,ctas", [
    (128, 16, 64, 0),        # one tile, one K chunk
    (256, 8, 4096, 0),       # the library's stream-K schedule
    (1000, 7, 256, 5),       # ragged M tile, N below the MMA width, pieces across tiles
    (1000, 17, 520, 3),      # ragged M and ragged K tail, N -> 32-wide tile
    (384, 100, 1024, 7),     # 128-wide activation tile
    (512, 256, 512, -1),     # 256-wide activation tile, whole tiles
    (300, 300, 128, 11),     # two activation tiles, ragged everywhere
    (4096, 8, 12288, 0),     # feature projection shape (8B)
    (6144, 8, 4096, 0),      # QKV shape (8B)
    (24576, 8, 4096, 0),     # gate/up shape (8B): 1.26 tiles per CTA
    (4096, 8, 4096, 256),    # 8 K chunks per CTA: 8 pieces per tile
    (4096, 8, 4096, 1),      # one CTA streams every tile whole
    (1000, 7, 256, -1),      # whole tiles round-robin
    (1000, 7, 256, -2),      # cluster split-K: 2 slices of 2 K chunks, ragged M tile
    (1000, 17, 520, -3),     # cluster split-K: 9 chunks in 3 slices, ragged K tail, 32-wide tile
    (300, 40, 640, -8),      # cluster split-K: 8 slices, 64-wide ragged activation tile
    (4096, 8, 4096, -8),     # 32 clusters x 8 CTAs > the SM count: clusters queue
    (128, 16, 64, -2),       # one K chunk: too short to split, whole tiles instead
    (384, 100, 1024, -4),    # 100 columns in 16-wide tiles (at most 4 row tiles): split
    (640, 100, 1024, -4),    # 128-wide activation tile: 4-slice cluster split of wide partial tiles
    (512, 256, 2048, -4),    # 256-wide activation tile: 4 slices summed through distributed shared memory
    (4096, 256, 12288, 0),   # the down / feature shape at 256 rows (batch 32): the library's cluster schedule
    (6144, 256, 4096, 0),    # the QKV shape at 256 rows
])
@pytest.mark.parametrize("accumulate", [False, True])
def test_bf16_gemm_matches_float64_product(M, N, K, ctas, accumulate):
    import torch
    B = lib()
    W = _mat(M, K, 1, 0.05, "bf16")
    X = _mat(N, K, 2, 1.0, "bf16")
    base = np.random.default_rng(3).standard_normal((N, M)).astype(np.float32)
    out = torch.from_numpy(base).cuda() if accumulate else torch.full((N, M), float("nan"), device="cuda")
    ws = torch.zeros(B.dflash2_test_gemm_workspace(M, N), dtype=torch.uint8, device="cuda")
    for rep in range(2):  # twice: the arrival counters must come back to zero
        if accumulate and rep == 1:
            out.copy_(torch.from_numpy(base))
        used = B.dflash2_test_gemm(B.BF16, S.to_torch(W), S.to_torch(X), ctas, out, ws, accumulate)
        torch.cuda.synchronize()
        assert 1 <= used <= 256 and (ctas <= 0 or used <= ctas)
        if ctas <= -2:
            # the cluster schedule ran where it applies (at least -ctas K chunks):
            # -ctas CTAs for each whole tile, else one
            tiles = B.dflash2_test_gemm(B.BF16, S.to_torch(W), S.to_torch(X), -1, torch.empty_like(out), ws)
            split = (K + 63) // 64 >= -ctas
            assert used == tiles * (-ctas if split else 1)
        got = out.double().cpu().numpy() - (base if accumulate else 0.0)
        w64, x64 = W.values.astype(np.float64), X.values.astype(np.float64)
        ref = x64 @ w64.T
        bound = np.abs(x64) @ np.abs(w64).T + (np.abs(base) if accumulate else 0.0)
        err = np.abs(got - ref)
        assert np.all(np.isfinite(got))
        assert np.all(err <= 1e-4 * bound + 1e-6), float(np.max(err / (bound + 1e-30)))
        assert int(ws[:4 * 256].view(torch.int32).abs().sum()) == 0


@pytest.mark.parametrize("M,N,K,ctas", [
    (128, 16, 64, 0),        # one tile, one K chunk
    (1000, 7, 512, 5),       # ragged M tile, pieces across tiles
    (384, 70, 1024, -1),     # 128-wide activation tile, whole tiles
    (2688, 7, 8064, 0),      # the 30B-A3B down / feature projection shape
    (5120, 14, 2688, 0),     # the 30B-A3B QKV shape with appended rows
    (1000, 7, 512, -4),      # cluster split-K with the converter warps
    (2688, 7, 8064, -8),     # 21 clusters x 8 slices
])
@pytest.mark.parametrize("accumulate", [False, True])
def test_fp8_gemm_matches_dequantised_product(M, N, K, ctas, accumulate):
    """e4m3 weights with per-row scales against the float64 product of the
    dequantised weights (the converters' e4m3 -> bf16 step is exact, so the
    error is fp32 accumulation and the final scaling only)."""
    import torch
    B = lib()
    W = S.quantize_rows_e4m3(_mat(M, K, 11, 0.05, "f32").values)
    X = _mat(N, K, 12, 1.0, "bf16")
    base = np.random.default_rng(13).standard_normal((N, M)).astype(np.float32)
    out = torch.from_numpy(base).cuda() if accumulate else torch.full((N, M), float("nan"), device="cuda")
    ws = torch.zeros(B.dflash2_test_gemm_workspace(M, N), dtype=torch.uint8, device="cuda")
    used = B.dflash2_test_gemm_fp8(torch.from_numpy(W.q).cuda(), torch.from_numpy(W.scale).cuda(), S.to_torch(X),
                                   ctas, out, ws, accumulate)
    torch.cuda.synchronize()
    assert 1 <= used <= 256
    if ctas <= -2:
        assert used == -(-M // 128) * -ctas
    got = out.double().cpu().numpy() - (base if accumulate else 0.0)
    x64 = X.values.astype(np.float64)
    ref = x64 @ W.values.T
    bound = np.abs(x64) @ np.abs(W.values).T + (np.abs(base) if accumulate else 0.0)
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got))
    assert np.all(err <= 1e-4 * bound + 1e-6), float(np.max(err / (bound + 1e-30)))
    assert int(ws[:4 * 256].view(torch.int32).abs().sum()) == 0


def test_fp8_gemm_reads_every_code_exactly():
    """Every finite e4m3 code through the converters: W8 row m holds the 256
    codes (NaN codes replaced by 0) shifted by m, X = one-hot rows, scale 1,
    so out[n][m] is the decoded code itself, bit for bit."""
    import torch
    B = lib()
    M, K = 128, 256
    codes = (np.arange(K)[None, :] + np.arange(M)[:, None]) % 256
    codes = np.where((codes & 0x7F) == 0x7F, 0, codes).astype(np.uint8)
    X = np.zeros((K, K), dtype=np.float32)
    X[np.arange(K), np.arange(K)] = 1.0
    Xb = torch.from_numpy(S.to_bf16_bits(X).view(np.int16)).cuda().view(torch.bfloat16)
    out = torch.full((K, M), float("nan"), device="cuda")
    ws = torch.zeros(B.dflash2_test_gemm_workspace(M, K), dtype=torch.uint8, device="cuda")
    B.dflash2_test_gemm_fp8(torch.from_numpy(codes).cuda(), torch.ones(M, device="cuda"), Xb, -1, out, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), S.e4m3_decode(codes).T.astype(np.float32))


def test_bf16_gemm_is_deterministic():
    # pieces of shared tiles are summed in CTA order: bit-identical reruns
    import torch
    B = lib()
    M, N, K = 4096, 8, 12288
    W = S.to_torch(_mat(M, K, 5, 0.05, "bf16"))
    X = S.to_torch(_mat(N, K, 6, 1.0, "bf16"))
    ws = torch.zeros(B.dflash2_test_gemm_workspace(M, N), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(3):
        out = torch.empty((N, M), device="cuda")
        B.dflash2_test_gemm(B.BF16, W, X, 0, out, ws)
        outs.append(out.cpu())
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])


@pytest.mark.parametrize("M,N,K", [(1000, 7, 256), (4096, 8, 768), (130, 40, 64)])
def test_f32_gemm_matches_float64_product(M, N, K):
    import torch
    B = lib()
    W = _mat(M, K, 3, 0.05, "f32")
    X = _mat(N, K, 4, 1.0, "f32")
    out = torch.full((N, M), float("nan"), device="cuda")
    ws = torch.zeros(B.dflash2_test_gemm_workspace(M, N), dtype=torch.uint8, device="cuda")
    assert B.dflash2_test_gemm(B.F32, S.to_torch(W), S.to_torch(X), 0, out, ws) == 1
    torch.cuda.synchronize()
    got = out.double().cpu().numpy()
    ref = X.values.astype(np.float64) @ W.values.astype(np.float64).T
    bound = np.abs(X.values.astype(np.float64)) @ np.abs(W.values.astype(np.float64)).T
    assert np.all(np.abs(got - ref) <= 1e-5 * bound + 1e-7)


def _topk_run(dtype, W, X, k, mult=1.0, cap=0.0):
    import torch
    B = lib()
    M, N = W.shape[0], X.shape[0]
    ws = torch.zeros(B.dflash2_test_topk_workspace(dtype, M, N), dtype=torch.uint8, device="cuda")
    cid = torch.full((N, k), -7, dtype=torch.int32, device="cuda")
    cz = torch.zeros((N, k), dtype=torch.float32, device="cuda")
    dbg = torch.full((N, M), float("nan"), device="cuda")
    B.dflash2_test_gemm_topk(dtype, S.to_torch(W), S.to_torch(X), k, mult, cap, cid, cz, dbg, ws)
    torch.cuda.synchronize()
    return cid.cpu().numpy(), cz.cpu().numpy(), dbg.cpu().numpy()


@pytest.mark.parametrize("dtype,M,N,k", [
    ("bf16", 1000, 7, 4), ("bf16", 1000, 16, 16), ("bf16", 4096 + 50, 40, 16), ("bf16", 2000, 300, 8),
    ("bf16", 151936, 7, 16), ("f32", 4096, 7, 4), ("f32", 3000, 9, 16),
    # 209..224 rows in one 256-wide tile (224 = the 8B batch-32 block; 209
    # ragged), K = 1024: 16 chunks a tile, so the ring wraps within a tile;
    # 20000 rows: 157 tiles, some CTAs take two
    ("bf16", 20000, 224, 16), ("bf16", 2500, 209, 8),
])
def test_lm_head_topk_component_parity(dtype, M, N, k):
    K = 1024 if N > 208 else 256
    W = _mat(M, K, 5, 0.05, dtype)
    X = _mat(N, K, 6, 1.0, dtype)
    cid, cz, dbg = _topk_run(1 if dtype == "bf16" else 0, W, X, k)
    assert np.all(np.isfinite(dbg))
    # the logits the kernel scored agree with the float64 product
    ref = X.values.astype(np.float64) @ W.values.astype(np.float64).T
    bound = np.abs(X.values.astype(np.float64)) @ np.abs(W.values.astype(np.float64)).T
    assert np.all(np.abs(dbg - ref) <= 1e-4 * bound + 1e-6)
    # component parity: the oracle's top-k of the GPU's own logits, bit-exact
    ids, vals = O.topk(dbg.astype(np.float64), k)
    np.testing.assert_array_equal(cid, ids)
    np.testing.assert_array_equal(cz, vals.astype(np.float32))


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_lm_head_topk_exact_ties_take_smaller_ids(dtype):
    # rows repeat with period 5, so every logit value appears many times
    base = _mat(5, 128, 7, 0.05, dtype)
    reps = 700
    vals = np.tile(base.values, (reps, 1))
    if dtype == "bf16":
        W = S.Tensor(vals, np.tile(base.bits, (reps, 1)))
    else:
        W = S.Tensor(np.ascontiguousarray(vals))
    X = _mat(6, 128, 8, 1.0, dtype)
    cid, _, dbg = _topk_run(1 if dtype == "bf16" else 0, W, X, 16)
    ids, _ = O.topk(dbg.astype(np.float64), 16)
    np.testing.assert_array_equal(cid, ids)
    # all ties: the best value's 16 smallest ids come first
    for r in range(6):
        best = int(np.argmax(dbg[r, :5]))
        assert list(cid[r]) == [best + 5 * j for j in range(16)]


def test_lm_head_multiplier_and_softcap():
    K, M, N = 128, 1000, 7
    W = _mat(M, K, 9, 0.5, "bf16")
    X = _mat(N, K, 10, 1.0, "bf16")
    cid, cz, dbg = _topk_run(1, W, X, 8, mult=2.0, cap=3.0)
    ref = X.values.astype(np.float64) @ W.values.astype(np.float64).T
    z = 3.0 * np.tanh(2.0 * ref / 3.0)
    assert np.max(np.abs(dbg - z)) < 1e-4
    assert np.all(np.abs(dbg) <= 3.0)
    ids, _ = O.topk(dbg.astype(np.float64), 8)
    np.testing.assert_array_equal(cid, ids)
