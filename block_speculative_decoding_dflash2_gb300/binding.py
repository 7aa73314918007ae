"""ctypes binding of libdflash2.so: argument marshalling only.

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it turns torch tensors into device pointers, Python
numbers into C ints/floats, and raises ``DFlash2Error`` on a non-OK status.
There is no fallback: without the built library, loading raises.
"""

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libdflash2.so")
TEST_LIB_PATH = os.path.join(_PKG, "libdflash2_testing.so")

F32 = 0
BF16 = 1
FP8W = 2

STATUS = {0: "ok", -1: "invalid argument", -2: "shape", -3: "block size", -4: "dtype",
          -5: "workspace", -6: "cuda", -7: "unsupported"}
DEV_BAD_PAGE, DEV_BAD_TOKEN, DEV_WAIT_TIMEOUT, DEV_BAD_LENGTH = 0x1, 0x2, 0x4, 0x8


class DFlash2Error(RuntimeError):
    def __init__(self, fn, status, text):
        super().__init__(f"{fn} failed: status {status} ({text})")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "hidden", "n_q_heads", "n_kv_heads", "head_dim", "intermediate", "vocab",
        "n_layers", "n_taps", "block_size", "conv_kernel_size", "conv_group_size",
        "top_k", "selector_rank", "page_size", "mask_token_id", "dtype")] + \
        [(n, ctypes.c_float) for n in (
            "rms_eps", "rope_theta", "input_embedding_scale", "output_multiplier",
            "final_logit_softcap")] + [("sliding_window", ctypes.c_int)]


_LAYER_FIELDS = ("attn_norm", "tapgen_attn", "qkv", "q_norm", "k_norm", "o", "mlp_norm",
                 "tapgen_mlp", "gate_up", "down")


class LayerWeights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _LAYER_FIELDS]


_TOP_FIELDS = ("embed", "lm_head", "fc", "hidden_norm", "final_norm", "sel")


_LAYER_SCALE_FIELDS = ("tapgen_attn", "qkv", "o", "tapgen_mlp", "gate_up", "down")


class LayerScales(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _LAYER_SCALE_FIELDS]


class Scales(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("lm_head", "fc", "sel")] + \
        [("layers", ctypes.POINTER(LayerScales))]


class Weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in _TOP_FIELDS] + [("layers", ctypes.POINTER(LayerWeights)),
                                                              ("scales", ctypes.POINTER(Scales))]


_lib = None
_tlib = None


def testing_lib():
    """The test-hook library (include/dflash2_testing.h), loaded after the
    product library it links against."""
    global _tlib
    if _tlib is None:
        lib()
        if not os.path.exists(TEST_LIB_PATH):
            raise ImportError(f"{TEST_LIB_PATH} is missing: build it with __graft_entry__.build()")
        T = ctypes.CDLL(TEST_LIB_PATH)
        P, I, S, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.POINTER
        T.dflash2_test_last_schedule.restype = I
        T.dflash2_test_last_schedule.argtypes = []
        T.dflash2_test_gemm_workspace.restype = S
        T.dflash2_test_gemm_workspace.argtypes = [I, I]
        T.dflash2_test_gemm.restype = I
        T.dflash2_test_gemm.argtypes = [I, P, I, I, P, I, I, I, P, P, S, P]
        T.dflash2_test_gemm_fp8.restype = I
        T.dflash2_test_force_cluster_split.restype = I
        T.dflash2_test_force_cluster_split.argtypes = [I]
        T.dflash2_test_force_attention.restype = I
        T.dflash2_test_force_attention.argtypes = [I]
        T.dflash2_test_last_attention.restype = I
        T.dflash2_test_last_attention.argtypes = []
        T.dflash2_test_gemm_fp8.argtypes = [P, P, I, I, P, I, I, I, P, P, S, P]
        T.dflash2_test_layout.restype = I
        T.dflash2_test_layout.argtypes = [F(Config), I, I, I, F(ctypes.c_size_t), I]
        T.dflash2_test_topk_workspace.restype = S
        T.dflash2_test_topk_workspace.argtypes = [I, I, I]
        T.dflash2_test_gemm_topk.restype = I
        T.dflash2_test_gemm_topk.argtypes = [I, P, I, I, P, I, I, ctypes.c_float, ctypes.c_float, P, P, P,
                                             P, S, P]
        _tlib = T
    return _tlib


def lib():
    """The loaded library (raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                              "(the product path has no fallback)")
        L = ctypes.CDLL(LIB_PATH)
        P, I, S, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.POINTER
        L.dflash2_status_string.restype = ctypes.c_char_p
        L.dflash2_status_string.argtypes = [I]
        L.dflash2_version.restype = I
        L.dflash2_validate_config.restype = I
        L.dflash2_validate_config.argtypes = [F(Config)]
        L.dflash2_workspace_size.restype = S
        L.dflash2_workspace_size.argtypes = [F(Config), I, I, I]
        L.dflash2_append_context.restype = I
        L.dflash2_append_context.argtypes = [F(Config), F(Weights), P, P, I, P, I, I, P, I, P, P, P, S, P]
        L.dflash2_draft_step.restype = I
        L.dflash2_draft_step.argtypes = [F(Config), F(Weights), P, P, I, P, I, I, P, I, P, P, P,
                                         P, P, P, P, S, P]
        L.dflash2_select_path.restype = I
        L.dflash2_select_path.argtypes = [F(Config), F(Weights), I, P, P, P, P, P, P, S, P]
        L.dflash2_verify_accept.restype = I
        L.dflash2_verify_accept.argtypes = [I, I, P, P, P, P, P, P, P, P, P]
        L.dflash2_read_device_status.restype = I
        L.dflash2_read_device_status.argtypes = [P, S, P]
        L.dflash2_select_path_static.restype = I
        L.dflash2_select_path_static.argtypes = [F(Config), F(Weights), I, P, P, P, P, P, P]
        L.dflash2_select_path_static_capacity.restype = S
        L.dflash2_select_path_static_read_status.restype = I
        L.dflash2_select_path_static_read_status.argtypes = [P]
        L.dflash2_selector_table_bytes.restype = S
        L.dflash2_selector_table_bytes.argtypes = [F(Config)]
        L.dflash2_build_selector_table.restype = I
        L.dflash2_build_selector_table.argtypes = [F(Config), F(Weights), P, P]
        L.dflash2_select_path_table.restype = I
        L.dflash2_select_path_table.argtypes = [F(Config), I, P, P, P, P, P, P, P, P]
        L.dflash2_select_path_table_ex.restype = I
        L.dflash2_select_path_table_ex.argtypes = [F(Config), I, P, P, P, P, F(DraftOpts), P, P, P, P, P]
        L.dflash2_select_path_ex.restype = I
        L.dflash2_select_path_ex.argtypes = [F(Config), F(Weights), I, P, P, P, F(DraftOpts), P, P, P, P, S, P]
        L.dflash2_select_top1.restype = I
        L.dflash2_select_top1.argtypes = [F(Config), I, P, P, F(DraftOpts), P, P, P, P, P]
        L.dflash2_verify_sampled.restype = I
        L.dflash2_verify_sampled.argtypes = [I, I, I, P, P, P, P, P, P, P, P, P, P, P, P]
        L.dflash2_verify_accept_ex.restype = I
        L.dflash2_verify_accept_ex.argtypes = [I, I, P, P, P, P, P, P, P, P, P, P]
        L.dflash2_launch_count.restype = ctypes.c_int64
        L.dflash2_set_stage_events.restype = None
        L.dflash2_set_stage_events.argtypes = [P]
        _lib = L
    return _lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, rc):
    if rc != 0:
        raise DFlash2Error(fn, rc, lib().dflash2_status_string(rc).decode())
    return rc


def make_config(d):
    """Config struct from a dict with the header's field names (extra keys ignored)."""
    c = Config()
    for name, _ in Config._fields_:
        v = d.get(name, 0) if name == "sliding_window" else d[name]
        if name == "dtype" and isinstance(v, str):
            v = {"f32": F32, "bf16": BF16, "fp8w": FP8W}[v]
        setattr(c, name, v)
    return c


class DraftOpts(ctypes.Structure):
    _fields_ = [("n_max", ctypes.c_int), ("p_min", ctypes.c_float)]


class WeightSet:
    """Holds a Weights struct over torch device tensors (kept alive here);
    tensors["scales"] (fp8 weights) fills its Scales struct."""

    def __init__(self, tensors):
        self.tensors = tensors
        n = len(tensors["layers"])
        self._layers = (LayerWeights * n)()
        for i, L in enumerate(tensors["layers"]):
            for f in _LAYER_FIELDS:
                setattr(self._layers[i], f, _ptr(L[f]))
        scales = None
        sc = tensors.get("scales")
        if sc is not None:
            self._layer_scales = (LayerScales * n)()
            for i, L in enumerate(sc["layers"]):
                for f in _LAYER_SCALE_FIELDS:
                    setattr(self._layer_scales[i], f, _ptr(L[f]))
            self._scales = Scales(*[_ptr(sc[f]) for f in ("lm_head", "fc", "sel")],
                                  ctypes.cast(self._layer_scales, ctypes.POINTER(LayerScales)))
            scales = ctypes.pointer(self._scales)
        self.struct = Weights(*[_ptr(tensors[f]) for f in _TOP_FIELDS],
                              ctypes.cast(self._layers, ctypes.POINTER(LayerWeights)), scales)


def dflash2_status_string(status):
    return lib().dflash2_status_string(status).decode()


def dflash2_version():
    return lib().dflash2_version()


def dflash2_validate_config(cfg):
    return lib().dflash2_validate_config(ctypes.byref(cfg))


def dflash2_workspace_size(cfg, max_batch, max_new_rows, max_ctx):
    return lib().dflash2_workspace_size(ctypes.byref(cfg), max_batch, max_new_rows, max_ctx)


def dflash2_append_context(cfg, w, k_cache, v_cache, n_pages, block_table, max_pages, batch, ctx_len,
                           n_new, new_taps, new_off, workspace, stream=None):
    return _check("dflash2_append_context", lib().dflash2_append_context(
        ctypes.byref(cfg), ctypes.byref(w.struct), _ptr(k_cache), _ptr(v_cache), n_pages,
        _ptr(block_table), max_pages, batch, _ptr(ctx_len), n_new, _ptr(new_taps), _ptr(new_off),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def dflash2_draft_step(cfg, w, k_cache, v_cache, n_pages, block_table, max_pages, batch, ctx_len,
                       n_new, new_taps, new_off, anchor, cand_id, cand_logit, debug_logits,
                       workspace, stream=None):
    return _check("dflash2_draft_step", lib().dflash2_draft_step(
        ctypes.byref(cfg), ctypes.byref(w.struct), _ptr(k_cache), _ptr(v_cache), n_pages,
        _ptr(block_table), max_pages, batch, _ptr(ctx_len), n_new, _ptr(new_taps), _ptr(new_off),
        _ptr(anchor), _ptr(cand_id), _ptr(cand_logit), _ptr(debug_logits),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def dflash2_select_path(cfg, w, batch, anchor, cand_id, cand_logit, path, path_score, workspace,
                        stream=None):
    return _check("dflash2_select_path", lib().dflash2_select_path(
        ctypes.byref(cfg), ctypes.byref(w.struct), batch, _ptr(anchor), _ptr(cand_id),
        _ptr(cand_logit), _ptr(path), _ptr(path_score), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def dflash2_selector_table_bytes(cfg):
    return lib().dflash2_selector_table_bytes(ctypes.byref(cfg))


def dflash2_build_selector_table(cfg, w, table, stream=None):
    return _check("dflash2_build_selector_table", lib().dflash2_build_selector_table(
        ctypes.byref(cfg), ctypes.byref(w.struct), _ptr(table), _stream(stream)))


def dflash2_select_path_table(cfg, batch, anchor, cand_id, cand_logit, table, path, path_score,
                              workspace=None, stream=None):
    return _check("dflash2_select_path_table", lib().dflash2_select_path_table(
        ctypes.byref(cfg), batch, _ptr(anchor), _ptr(cand_id), _ptr(cand_logit), _ptr(table), _ptr(path),
        _ptr(path_score), _ptr(workspace), _stream(stream)))


def _opts(n_max, p_min):
    return ctypes.byref(DraftOpts(int(n_max), float(p_min)))


def dflash2_select_path_ex(cfg, w, batch, anchor, cand_id, cand_logit, n_max, p_min, path, path_score, n_draft,
                           workspace, stream=None):
    return _check("dflash2_select_path_ex", lib().dflash2_select_path_ex(
        ctypes.byref(cfg), ctypes.byref(w.struct), batch, _ptr(anchor), _ptr(cand_id), _ptr(cand_logit),
        _opts(n_max, p_min), _ptr(path), _ptr(path_score), _ptr(n_draft), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))


def dflash2_select_path_table_ex(cfg, batch, anchor, cand_id, cand_logit, table, n_max, p_min, path, path_score,
                                 n_draft, workspace=None, stream=None):
    return _check("dflash2_select_path_table_ex", lib().dflash2_select_path_table_ex(
        ctypes.byref(cfg), batch, _ptr(anchor), _ptr(cand_id), _ptr(cand_logit), _ptr(table), _opts(n_max, p_min),
        _ptr(path), _ptr(path_score), _ptr(n_draft), _ptr(workspace), _stream(stream)))


def dflash2_select_top1(cfg, batch, cand_id, cand_logit, n_max, p_min, path, path_score, n_draft, workspace=None,
                        stream=None):
    return _check("dflash2_select_top1", lib().dflash2_select_top1(
        ctypes.byref(cfg), batch, _ptr(cand_id), _ptr(cand_logit), _opts(n_max, p_min), _ptr(path),
        _ptr(path_score), _ptr(n_draft), _ptr(workspace), _stream(stream)))


def dflash2_verify_sampled(batch, block_size, vocab, path, n_draft, target_prob, u_accept, u_sample, accept_len,
                           out_tok, n_out, next_anchor, seq_len=None, counters=None, stream=None):
    return _check("dflash2_verify_sampled", lib().dflash2_verify_sampled(
        batch, block_size, vocab, _ptr(path), _ptr(n_draft), _ptr(target_prob), _ptr(u_accept), _ptr(u_sample),
        _ptr(accept_len), _ptr(out_tok), _ptr(n_out), _ptr(next_anchor), _ptr(seq_len), _ptr(counters),
        _stream(stream)))


def dflash2_verify_accept_ex(batch, block_size, path, n_draft, target, accept_len, out_tok, n_out, next_anchor,
                             seq_len=None, counters=None, stream=None):
    return _check("dflash2_verify_accept_ex", lib().dflash2_verify_accept_ex(
        batch, block_size, _ptr(path), _ptr(n_draft), _ptr(target), _ptr(accept_len), _ptr(out_tok), _ptr(n_out),
        _ptr(next_anchor), _ptr(seq_len), _ptr(counters), _stream(stream)))


def dflash2_verify_accept(batch, block_size, path, target, accept_len, out_tok, n_out, next_anchor,
                          seq_len=None, counters=None, stream=None):
    return _check("dflash2_verify_accept", lib().dflash2_verify_accept(
        batch, block_size, _ptr(path), _ptr(target), _ptr(accept_len), _ptr(out_tok), _ptr(n_out),
        _ptr(next_anchor), _ptr(seq_len), _ptr(counters), _stream(stream)))


def dflash2_read_device_status(workspace, stream=None):
    rc = lib().dflash2_read_device_status(_ptr(workspace), workspace.numel() * workspace.element_size(),
                                          _stream(stream))
    if rc < 0:
        _check("dflash2_read_device_status", rc)
    return rc


# --------------------------------------------------------------- test hooks
# (include/dflash2_testing.h: the internal contraction and the lm_head top-k
# path on their own, for parity tests)

def dflash2_test_gemm_workspace(M, N):
    return testing_lib().dflash2_test_gemm_workspace(M, N)


def dflash2_test_gemm(dtype, W, X, ctas, out, workspace, accumulate=False, stream=None):
    """ctas: 0 = the library's schedule, > 0 = stream-K over that many CTAs,
    -1 = whole tiles, -2..-8 = cluster split-K of -ctas slices per tile.
    Returns the CTA count launched."""
    M, K = W.shape
    N = X.shape[0]
    rc = testing_lib().dflash2_test_gemm(dtype, _ptr(W), M, K, _ptr(X), N, ctas, int(accumulate), _ptr(out),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if rc < 0:
        _check("dflash2_test_gemm", rc)
    return rc


def dflash2_test_force_cluster_split(cs):
    """Force cluster split-K of cs slices on the library's own contractions
    (0 = its own schedule)."""
    _check("dflash2_test_force_cluster_split", testing_lib().dflash2_test_force_cluster_split(int(cs)))


def dflash2_test_force_attention(mode):
    """Attention kernel of later draft steps: 0 the library's choice, 1 the
    mma.sync cluster kernel, 2 the tcgen05 kernel wherever it applies."""
    _check("dflash2_test_force_attention", testing_lib().dflash2_test_force_attention(int(mode)))


def dflash2_test_last_attention():
    """Attention kernel of the last draft step: 1 mma.sync cluster, 2
    tcgen05, 3 SIMT (0 before any)."""
    return int(testing_lib().dflash2_test_last_attention())


def dflash2_test_gemm_fp8(W8, scale, X, ctas, out, workspace, accumulate=False, stream=None):
    """W8: uint8 e4m3 codes [M, K]; scale: float32 [M]; X: bf16 [N, K]."""
    M, K = W8.shape
    N = X.shape[0]
    rc = testing_lib().dflash2_test_gemm_fp8(_ptr(W8), _ptr(scale), M, K, _ptr(X), N, ctas, int(accumulate), _ptr(out),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if rc < 0:
        _check("dflash2_test_gemm_fp8", rc)
    return rc


def dflash2_test_topk_workspace(dtype, M, N):
    return testing_lib().dflash2_test_topk_workspace(dtype, M, N)


def dflash2_test_gemm_topk(dtype, W, X, k, mult, cap, cand_id, cand_logit, debug, workspace, stream=None):
    M, K = W.shape
    N = X.shape[0]
    return _check("dflash2_test_gemm_topk", testing_lib().dflash2_test_gemm_topk(
        dtype, _ptr(W), M, K, _ptr(X), N, k, mult, cap, _ptr(cand_id), _ptr(cand_logit), _ptr(debug),
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream)))


def dflash2_test_layout(cfg, batch, n_new, max_ctx):
    """Workspace byte offsets of {f, h, u, u2, q, kb, vb, O, act, hn, ua, u2a, cnt, cnta}."""
    out = (ctypes.c_size_t * 14)()
    _check("dflash2_test_layout", testing_lib().dflash2_test_layout(ctypes.byref(cfg), batch, n_new, max_ctx, out, 14))
    return dict(zip(("f", "h", "u", "u2", "q", "kb", "vb", "O", "act", "hn", "ua", "u2a", "cnt", "cnta"),
                    list(out)))


SCHED_FUSED_PROLOGUE, SCHED_SPLIT_SMS, SCHED_FUSED_QKV, SCHED_KV_BESIDE_QKV, SCHED_MERGED = 1, 2, 4, 8, 16


def dflash2_test_last_schedule():
    """Schedule bits (SCHED_*) of the last draft step in this process."""
    return testing_lib().dflash2_test_last_schedule()


def dflash2_launch_count():
    return lib().dflash2_launch_count()


def dflash2_set_stage_events(events):
    """events: None, or 5 torch.cuda.Event(enable_timing=True) already recorded once.

    Returns a holder that the caller keeps alive for as long as the library
    (or a graph captured while the events were set) may record into them."""
    if events is None:
        lib().dflash2_set_stage_events(None)
        return None
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    lib().dflash2_set_stage_events(ctypes.cast(arr, ctypes.c_void_p))
    # a graph captured with these events records into them at every replay:
    # the holder keeps the event objects (not only their handles) alive
    return (arr, tuple(events))


def dflash2_select_path_static(cfg, w, batch, anchor, cand_id, cand_logit, path, path_score, stream=None):
    """dflash2_select_path for callers that cannot allocate device memory: the
    library's own fixed scratch array replaces the workspace (see the header)."""
    return _check("dflash2_select_path_static", lib().dflash2_select_path_static(
        ctypes.byref(cfg), ctypes.byref(w.struct), batch, _ptr(anchor), _ptr(cand_id), _ptr(cand_logit),
        _ptr(path), _ptr(path_score), _stream(stream)))


def dflash2_select_path_static_capacity():
    return lib().dflash2_select_path_static_capacity()


def dflash2_select_path_static_read_status(stream=None):
    """Device status word (DFLASH2_DEV_* bits) of the last static selector
    call on the current device, read and cleared; synchronises the stream."""
    rc = lib().dflash2_select_path_static_read_status(_stream(stream))
    if rc < 0:
        _check("dflash2_select_path_static_read_status", rc)
    return rc
