"""The tcgen05 block attention (head dimension 128, 16-key pages) against the
oracle, stage by stage, next to the mma.sync cluster kernel on the same
inputs: every query-row count it is built for (16 .. 80 rows per kv head,
the 56-row shape padded to 64), contexts that span several 128-key tiles per
CTA (up to eight) and end mid-page, an empty context, sliding windows whose first key is
not on a page boundary (every row then takes the cp.async path), and the
end-to-end step."""

import pytest

import dflash2_synth as S
from tests.helpers import Case, lib
from tests.test_gpu_draft import check_case
from tests.test_gpu_stagewise import run_stagewise

pytestmark = pytest.mark.gpu

# query rows per kv head = (n_q_heads / n_kv_heads) x block_size
SHAPES = {
    "r16": dict(n_q_heads=4, n_kv_heads=2, block_size=8),
    "r32": dict(n_q_heads=8, n_kv_heads=2, block_size=8),
    "r48": dict(n_q_heads=12, n_kv_heads=2, block_size=8),
    "r56": dict(n_q_heads=16, n_kv_heads=2, block_size=7),
    "r80": dict(n_q_heads=10, n_kv_heads=2, block_size=16),
}


def _cfg(name, i, **over):
    return S.small_bf16_config(head_dim=128, hidden=512, n_layers=1, top_k=8, index=40 + i, **SHAPES[name],
                               **over)


def _run(cfg, mode, ctx_lens, n_new, seed):
    B = lib()
    B.dflash2_test_force_attention(mode)
    try:
        case = Case(cfg, ctx_lens=ctx_lens, n_new=n_new, seed=seed).run_gpu()
    finally:
        B.dflash2_test_force_attention(0)
    assert case.status == 0
    return case


@pytest.mark.parametrize("mode", [2, 1])
@pytest.mark.parametrize("name", list(SHAPES))
def test_attention_kernels_stagewise(name, mode):
    # 3000 + 8 keys in 8 chunks of 384: three 128-key tiles per CTA; 1234
    # ends mid-page; the empty context reads the block's own keys only
    i = list(SHAPES).index(name)
    B_ = SHAPES[name]["block_size"]
    case = _run(_cfg(name, i), mode, [3000, 0, 333, 1234], [B_, 3, 1, 5], 60 + i)
    run_stagewise(case)


@pytest.mark.parametrize("window", [37, 200, 1000])
@pytest.mark.parametrize("name", ["r56", "r80"])
def test_tc_attention_sliding_window(name, window):
    i = list(SHAPES).index(name)
    case = _run(_cfg(name, i, sliding_window=window), 2, [3000, 60, 0, 777], [4, 2, 8, 1], 70 + i)
    run_stagewise(case)


@pytest.mark.parametrize("name", ["r32", "r56", "r80"])
def test_tc_attention_long_chunks(name):
    # one long sequence and a shorter one: 8 chunks of ~1000 keys, eight
    # 128-key tiles per CTA, so the double-buffered P and the K/V stages
    # each go round several times
    i = list(SHAPES).index(name)
    case = _run(_cfg(name, i), 2, [8000, 5100], [3, 2], 90 + i)
    run_stagewise(case)


def test_tc_attention_flags_bad_page():
    """A block-table entry outside [0, n_pages) is flagged, not read: a whole
    page inside a chunk (the TMA path) and the last, partial page (the row
    path); the kernel zero-fills those rows and the step completes."""
    import torch
    B = lib()
    B.dflash2_test_force_attention(2)
    try:
        case = Case(_cfg("r80", 4), ctx_lens=[700, 300], n_new=[2, 2], seed=98)
        case.run_gpu()
        assert case.status == 0
        r = case.runner
        r.block_table[0, 3] = r.n_pages + 5  # keys 48..63 of sequence 0
        r.block_table[1, 18] = -7             # keys 288..303 of sequence 1 (its last page)
        case.run_gpu()
        assert case.status & B.DEV_BAD_PAGE
        torch.cuda.synchronize()
    finally:
        B.dflash2_test_force_attention(0)


def test_library_attention_choice():
    """The library's own choice: tcgen05 for more than 32 rows per kv head
    and chunks of at least 1024 keys per CTA, else the mma.sync kernel."""
    B = lib()
    # 80 rows, one 9000-key sequence (8 chunks of ~1130 keys): tcgen05
    case = Case(_cfg("r80", 4), ctx_lens=[9000], n_new=[2], seed=95).run_gpu()
    assert case.status == 0 and B.dflash2_test_last_attention() == 2
    run_stagewise(case)
    # 80 rows, short context (chunks of ~130 keys): mma.sync
    case = Case(_cfg("r80", 4), ctx_lens=[1000], n_new=[2], seed=96).run_gpu()
    assert case.status == 0 and B.dflash2_test_last_attention() == 1
    # 32 rows, long context: mma.sync
    case = Case(_cfg("r32", 1), ctx_lens=[9000], n_new=[2], seed=97).run_gpu()
    assert case.status == 0 and B.dflash2_test_last_attention() == 1


def test_tc_attention_end_to_end():
    case = _run(_cfg("r80", 4), 2, [2047, 16, 500], [16, 1, 7], 80)
    run_stagewise(case)
    check_case(case)
