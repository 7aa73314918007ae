"""Runs one hot kernel of the library a few times on a fixed shape, for
profiler captures (ncu) and quick timing.

  python -m block_speculative_decoding_dflash2_gb300.kernel_bench --kernel lm_head [--launches 3]

Kernels:
  lm_head   the lm_head contraction with its fused streaming top-k
            (vocab 151936 x hidden 4096 bf16, 7 block rows, top-16) through
            the dflash2_test_gemm_topk hook, then the top-k merge;
  gate_up   the MLP gate/up contraction (24576 x 4096, 8 rows);
  fc, qkv, kv, down, o   the other contractions of the 8B-shaped draft step;
  fc27, kv27, qkv27, o27, gate_up27, down27   the 27B-shaped step's contractions
            at 128 rows (batch 8 x block 16);
  select    the selector on a factor table (vocab 151936, rank 64, 7
            positions x top-16, one sequence) through
            dflash2_select_path_table.
Weights are seeded N(0, 0.02) bf16 drawn on the device (timing only; no
parity is checked here).  L2 is flushed (a 256 MiB write) before every
launch; prints the mean CUDA-event time per launch.
"""

import argparse

import torch

from . import binding as B
from .build import build

SHAPES = {"lm_head": (151936, 4096, 7), "gate_up": (24576, 4096, 8), "fc": (4096, 12288, 8),
          "qkv": (6144, 4096, 8), "down": (4096, 12288, 8), "o": (4096, 4096, 8),
          "kv": (2048, 4096, 8),
          # the 27B-shaped draft at batch 8 x block 16 (128 rows)
          "fc27": (5120, 15360, 128), "kv27": (2048, 5120, 128), "qkv27": (7168, 5120, 128),
          "gate_up27": (34816, 5120, 128), "down27": (5120, 17408, 128), "o27": (5120, 5120, 128)}


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--kernel", default="lm_head", choices=sorted(SHAPES) + ["select"])
    p.add_argument("--launches", type=int, default=3)
    p.add_argument("--rows", type=int, default=0,
                   help="activation rows (N); 0 = the batch-1 block's rows of the 8B-shaped step")
    p.add_argument("--ctas", type=int, default=0,
                   help="contraction schedule: 0 = the library's, >0 = stream-K over that many CTAs, <0 = whole tiles")
    a = p.parse_args()
    build()
    if a.kernel == "select":
        return bench_select(a)
    M, K, N = SHAPES[a.kernel]
    N = a.rows or N
    g = torch.Generator(device="cuda")
    g.manual_seed(1234)
    W = (torch.randn((M, K), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    X = torch.randn((N, K), generator=g, device="cuda").to(torch.bfloat16)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if a.kernel == "lm_head":
        ws = torch.zeros(B.dflash2_test_topk_workspace(B.BF16, M, N), dtype=torch.uint8, device="cuda")
        cid = torch.empty((N, 16), dtype=torch.int32, device="cuda")
        cz = torch.empty((N, 16), dtype=torch.float32, device="cuda")
        run = lambda: B.dflash2_test_gemm_topk(B.BF16, W, X, 16, 1.0, 0.0, cid, cz, None, ws)
    else:
        out = torch.empty((N, M), dtype=torch.float32, device="cuda")
        ws = torch.zeros(B.dflash2_test_gemm_workspace(M, N), dtype=torch.uint8, device="cuda")
        run = lambda: B.dflash2_test_gemm(B.BF16, W, X, a.ctas, out, ws)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    run()
    torch.cuda.synchronize()
    total = 0.0
    for _ in range(a.launches):
        flush.zero_()
        e0.record()
        run()
        e1.record()
        e1.synchronize()
        total += e0.elapsed_time(e1)
    ms = total / a.launches
    gb = M * K * 2 / 1e9
    print(f"{a.kernel}: M={M} K={K} N={N} ctas={a.ctas}: {ms * 1e3:.1f} us per call, "
          f"{gb / (ms / 1e3):.0f} GB/s of weights")


def bench_select(a):
    V, r, D, k = 151936, 64, 7, 16
    cfg = B.make_config(dict(hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128, intermediate=12288, vocab=V,
                             n_layers=1, n_taps=3, block_size=D + 1, conv_kernel_size=2, conv_group_size=32,
                             top_k=k, selector_rank=r, page_size=16, mask_token_id=V - 1, dtype="bf16",
                             rms_eps=1e-6, rope_theta=1e6, input_embedding_scale=1.0, output_multiplier=1.0,
                             final_logit_softcap=0.0))
    g = torch.Generator(device="cuda")
    g.manual_seed(99)
    table = torch.randn((V * 2 * r,), generator=g, device="cuda") * 0.1
    cand = torch.randint(0, V - 1, (1, D, k), generator=g, device="cuda", dtype=torch.int32)
    z = torch.sort(torch.randn((1, D, k), generator=g, device="cuda"), dim=2, descending=True).values
    anchor = torch.randint(0, V - 1, (1,), generator=g, device="cuda", dtype=torch.int32)
    path = torch.empty((1, D), dtype=torch.int32, device="cuda")
    score = torch.empty((1,), dtype=torch.float32, device="cuda")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run = lambda: B.dflash2_select_path_table(cfg, 1, anchor, cand, z, table, path, score)
    run()
    torch.cuda.synchronize()
    e0.record()
    for _ in range(a.launches):
        run()
    e1.record()
    e1.synchronize()
    print(f"select: {e0.elapsed_time(e1) * 1e3 / a.launches:.1f} us per call (back to back)")


if __name__ == "__main__":
    main()
