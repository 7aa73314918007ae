"""Host-side owner of the device buffers of one batch of sequences.

``DraftRunner`` allocates the paged context cache, the block table, the
workspace and the output tensors once, and calls the library's entry points
in step order on one stream.  It performs no arithmetic of the method; every
stage runs in libdflash2.so.
"""

import torch

from . import binding as B


class DraftRunner:
    def __init__(self, cfg, weights, batch, max_ctx, max_new, block_table=None, n_pages=None,
                 device="cuda"):
        """cfg: dict with the dflash2_config fields; weights: dict of device tensors
        (layers: list of dicts) in the layouts of include/dflash2.h."""
        self.cfgd = dict(cfg)
        self.cfg = B.make_config(cfg)
        rc = B.dflash2_validate_config(self.cfg)
        if rc != 0:
            raise B.DFlash2Error("dflash2_validate_config", rc, B.dflash2_status_string(rc))
        self.w = B.WeightSet(weights)
        self.batch = batch
        self.device = device
        c = self.cfgd
        self.dtype = torch.float32 if self.cfg.dtype == B.F32 else torch.bfloat16  # activations and cache
        ps = c["page_size"]
        self.max_pages = -(-max_ctx // ps)
        if block_table is None:
            block_table = torch.arange(batch * self.max_pages, dtype=torch.int32).reshape(batch, self.max_pages)
            n_pages = batch * self.max_pages
        self.block_table = block_table.to(device=device, dtype=torch.int32).contiguous()
        self.max_pages = self.block_table.shape[1]
        self.n_pages = int(n_pages)
        shape = (c["n_layers"], self.n_pages, ps, c["n_kv_heads"], c["head_dim"])
        self.k_cache = torch.zeros(shape, dtype=self.dtype, device=device)
        self.v_cache = torch.zeros(shape, dtype=self.dtype, device=device)
        self.ws_bytes = B.dflash2_workspace_size(self.cfg, batch, max_new, self.max_pages * ps)
        if self.ws_bytes == 0:
            raise B.DFlash2Error("dflash2_workspace_size", -2, "invalid config")
        self.workspace = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)
        D, k = c["block_size"] - 1, c["top_k"]
        i32 = dict(dtype=torch.int32, device=device)
        self.cand_id = torch.zeros((batch, D, k), **i32)
        self.cand_logit = torch.zeros((batch, D, k), dtype=torch.float32, device=device)
        # the step's int32 results share one buffer (`results`), so a caller
        # reads them back to the host in one copy
        self.results = torch.zeros((batch * (2 * D + 4),), **i32)
        parts = torch.split(self.results, [batch * D, batch, batch * (D + 1), batch, batch])
        self.path = parts[0].view(batch, D)
        self.accept_len = parts[1]
        self.out_tok = parts[2].view(batch, D + 1)
        self.n_out = parts[3]
        self.next_anchor = parts[4]
        self.path_score = torch.zeros((batch,), dtype=torch.float32, device=device)
        self.counters = torch.zeros((4 + 2 * (D + 1) - 1,), dtype=torch.int64, device=device)

    def append(self, ctx_len, taps, new_off, stream=None):
        n_new = int(taps.shape[0]) if taps is not None else 0
        B.dflash2_append_context(self.cfg, self.w, self.k_cache, self.v_cache, self.n_pages, self.block_table,
                                 self.max_pages, self.batch, ctx_len, n_new, taps, new_off, self.workspace,
                                 stream)

    def draft(self, ctx_len, taps, new_off, anchor, debug_logits=None, stream=None):
        n_new = int(taps.shape[0]) if taps is not None else 0
        B.dflash2_draft_step(self.cfg, self.w, self.k_cache, self.v_cache, self.n_pages, self.block_table,
                             self.max_pages, self.batch, ctx_len, n_new, taps, new_off, anchor, self.cand_id,
                             self.cand_logit, debug_logits, self.workspace, stream)

    def build_selector_table(self, stream=None):
        """Factors of every vocabulary token (built once; select() then looks
        its rows up instead of contracting per step)."""
        n = B.dflash2_selector_table_bytes(self.cfg) // 4
        self.sel_table = torch.empty((n,), dtype=torch.float32, device=self.device)
        B.dflash2_build_selector_table(self.cfg, self.w, self.sel_table, stream)

    def select(self, anchor, stream=None):
        if getattr(self, "sel_table", None) is not None:
            B.dflash2_select_path_table(self.cfg, self.batch, anchor, self.cand_id, self.cand_logit,
                                        self.sel_table, self.path, self.path_score, self.workspace, stream)
        else:
            B.dflash2_select_path(self.cfg, self.w, self.batch, anchor, self.cand_id, self.cand_logit,
                                  self.path, self.path_score, self.workspace, stream)

    def verify(self, target, seq_len=None, stream=None):
        B.dflash2_verify_accept(self.batch, self.cfgd["block_size"], self.path, target, self.accept_len,
                                self.out_tok, self.n_out, self.next_anchor, seq_len, self.counters, stream)

    def device_status(self, stream=None):
        return B.dflash2_read_device_status(self.workspace, stream)
