"""The C ABI loads, exports every declared symbol, and its host-side checks
behave (no GPU needed: only calls that return before touching CUDA)."""

import ctypes
import os
import re

import pytest

from tests.conftest import ROOT

pytestmark = pytest.mark.skipif(
    not (os.path.exists("/usr/local/cuda/bin/nvcc") or __import__("shutil").which("nvcc")),
    reason="nvcc is needed to build the library")


@pytest.fixture(scope="module")
def B():
    from block_speculative_decoding_dflash2_gb300 import build as bld
    bld.build()
    from block_speculative_decoding_dflash2_gb300 import binding
    binding.lib()
    return binding


def declared(header):
    text = open(os.path.join(ROOT, "include", header)).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash2_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(B):
    names = declared("dflash2.h")
    assert "dflash2_draft_step" in names and "dflash2_select_path" in names
    assert "dflash2_verify_accept" in names
    lib = ctypes.CDLL(B.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    # the test hooks come from their own library, not the product one
    hooks = declared("dflash2_testing.h")
    tlib = ctypes.CDLL(B.TEST_LIB_PATH)
    for n in hooks:
        assert hasattr(tlib, n), n
        assert not hasattr(lib, n), n


def test_struct_sizes_match_header(B):
    # 16 ints + 5 floats + 1 int; 10 and 6+1+1 pointers; fp8 scales: 6 and 3+1
    assert ctypes.sizeof(B.Config) == 22 * 4
    assert ctypes.sizeof(B.LayerWeights) == 10 * 8
    assert ctypes.sizeof(B.Weights) == 8 * 8
    assert ctypes.sizeof(B.LayerScales) == 6 * 8
    assert ctypes.sizeof(B.Scales) == 4 * 8


def _cfg(B, name, **over):
    import dflash2_synth as S
    return B.make_config(S.config_of(name, **over))


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen3_8b_b1", "qwen3_8b_b32_paged", "qwen3_27b_b8", "a3b_30b_fp8"])
def test_workload_configs_validate(B, name):
    assert B.dflash2_validate_config(_cfg(B, name)) == 0


@pytest.mark.parametrize("over,code", [
    (dict(block_size=1), -3), (dict(block_size=33), -3), (dict(dtype=7), -4),
    (dict(head_dim=96), -2), (dict(conv_kernel_size=3), -2), (dict(top_k=17), -2),
    (dict(conv_group_size=33), -2), (dict(n_q_heads=6, n_kv_heads=4), -2),
    (dict(mask_token_id=4096), -2), (dict(selector_rank=0), -2), (dict(page_size=0), -2),
])
def test_bad_configs_are_rejected(B, over, code):
    assert B.dflash2_validate_config(_cfg(B, "tiny_fp32", **over)) == code
    assert B.dflash2_workspace_size(_cfg(B, "tiny_fp32", **over), 1, 8, 128) == 0


def test_null_config_and_status_strings(B):
    assert B.lib().dflash2_validate_config(None) == -1
    for s in (0, -1, -2, -3, -4, -5, -6, -7):
        assert B.dflash2_status_string(s)
    assert B.dflash2_version() >= 10000


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen3_8b_b1", "qwen3_27b_b8"])
def test_workspace_size_is_monotone(B, name):
    c = _cfg(B, name)
    prev = 0
    for b, n, ctx in [(1, 0, 16), (1, 8, 128), (2, 8, 128), (2, 64, 512), (4, 64, 2048), (8, 300, 4096)]:
        s = B.dflash2_workspace_size(c, b, n, ctx)
        assert s >= prev > -1
        prev = s
    for b in range(1, 9):
        for n in (0, 1, 8, 17, 64):
            assert B.dflash2_workspace_size(c, b, n, 512) <= B.dflash2_workspace_size(c, 8, 64, 512)


@pytest.mark.parametrize("name", ["tiny_fp32", "qwen3_8b_b1", "qwen3_27b_b8"])
def test_counter_regions_do_not_move_between_calls(B, name):
    # split-K tile counters are left at zero by one call and must be zero at
    # the next: their offsets may not depend on the call's shape (the
    # context append plans its workspace with batch 0)
    c = _cfg(B, name)
    seen = {(o["cnt"], o["cnta"]) for o in (B.dflash2_test_layout(c, b, n, ctx)
                                           for b, n, ctx in [(0, 333, 0), (0, 1, 0), (1, 8, 2048),
                                                             (2, 20, 512), (8, 300, 4096)])}
    assert len(seen) == 1
    cnt, cnta = seen.pop()
    assert cnt < cnta and cnta - cnt >= 128 * 4


def test_fp8_weights_need_their_scales(B):
    # fp8 configs: the bf16-activation workspace, and weights without row
    # scales are refused before any CUDA call
    L = B.lib()
    c8 = _cfg(B, "a3b_30b_fp8")
    cb = _cfg(B, "a3b_30b_fp8", dtype="bf16")
    assert B.dflash2_workspace_size(c8, 8, 56, 1024) == B.dflash2_workspace_size(cb, 8, 56, 1024) > 0
    w = B.Weights()
    for f in ("embed", "lm_head", "fc", "hidden_norm", "final_norm", "sel"):
        setattr(w, f, 16)
    layers = (B.LayerWeights * 2)()
    for l in range(2):
        for f in B._LAYER_FIELDS:
            setattr(layers[l], f, 16)
    w.layers = ctypes.cast(layers, ctypes.POINTER(B.LayerWeights))
    assert L.dflash2_draft_step(ctypes.byref(c8), ctypes.byref(w), 1, 1, 1, 1, 1, 1, 1, 0, None, 1, 1, 1, 1,
                                None, 1, 1 << 30, None) == -1
    assert L.dflash2_build_selector_table(ctypes.byref(c8), ctypes.byref(w), 16, None) == -1


def test_host_side_error_paths_return_before_cuda(B):
    L = B.lib()
    # verify: bad block size / batch / null pointers
    assert L.dflash2_verify_accept(1, 1, 1, 1, 1, 1, 1, 1, None, None, None) == -3
    assert L.dflash2_verify_accept(0, 8, 1, 1, 1, 1, 1, 1, None, None, None) == -2
    assert L.dflash2_verify_accept(1, 8, None, 1, 1, 1, 1, 1, None, None, None) == -1
    c = _cfg(B, "tiny_fp32")
    w = B.Weights()  # all null
    assert L.dflash2_draft_step(ctypes.byref(c), ctypes.byref(w), 1, 1, 1, 1, 1, 1, 1, 0, None, 1, 1, 1, 1,
                                None, 1, 1 << 30, None) == -1
    bad = _cfg(B, "tiny_fp32", block_size=40)
    assert L.dflash2_draft_step(ctypes.byref(bad), ctypes.byref(w), 1, 1, 1, 1, 1, 1, 1, 0, None, 1, 1, 1, 1,
                                None, 1, 1 << 30, None) == -3
    assert L.dflash2_select_path(ctypes.byref(c), ctypes.byref(w), 1, 1, 1, 1, 1, None, 1, 1 << 30,
                                 None) == -1
    assert L.dflash2_read_device_status(None, 0, None) == -5


def test_sampled_verify_and_cluster_switch_host_checks(B):
    L = B.lib()
    # sampled verification: block size, vocabulary bounds and null pointers are
    # checked on the host, before any launch (dummy non-null pointers are never
    # dereferenced)
    args = (1, 1, 1, 1, 1, 1, 1, 1, 1, None, None, None)
    assert L.dflash2_verify_sampled(1, 40, 1000, *args) == -3
    assert L.dflash2_verify_sampled(1, 8, 1, *args) == -2
    assert L.dflash2_verify_sampled(1, 8, 1_536_001, *args) == -2  # segment sums exceed shared memory
    assert L.dflash2_verify_sampled(1, 8, 1000, None, *args[1:]) == -1
    # the test switch of cluster split-K: 0 or 2..8 slices, nothing else
    T = B.testing_lib()
    for cs in (1, 9, -2):
        assert T.dflash2_test_force_cluster_split(cs) == -1
    for cs in (2, 8, 0):
        assert T.dflash2_test_force_cluster_split(cs) == 0
