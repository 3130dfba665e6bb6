"""One DSA layer (or IndexShare group) as a user runs it: buffers plus the C-ABI calls.

    layer = DsaLayer(case_on_gpu)
    layer.run()          # indexer -> top-k -> sparse MLA, all in libdsa's kernels
                         # (decode: top-k and sparse MLA in one call)
    layer.run_shared()   # IndexShare: indexer and top-k once, MLA for every layer

Only allocation and argument marshalling happen here.
"""
from __future__ import annotations

import torch

from . import capi as libdsa


def layout_for(case) -> libdsa.CacheLayout:
    return libdsa.make_layout(case.n_phys, seq_start=case.seq_start,
                              block_table=case.block_table, page_size=case.page_size)


class DsaLayer:
    def __init__(self, case, stream=None):
        if not case.k8.is_cuda:
            raise ValueError("DsaLayer needs the case on a CUDA device")
        self.case = case
        self.stream = stream
        dev = case.k8.device
        rows = case.rows
        self.layout = layout_for(case)
        self.scores = torch.empty((rows, case.Lmax), dtype=torch.float32, device=dev)
        self.idx = torch.empty((rows, case.k), dtype=torch.int32, device=dev)
        self.out = [torch.empty((rows, case.H, case.d), dtype=torch.bfloat16, device=dev)
                    for _ in range(case.layers)]
        self.lse = [torch.empty((rows, case.H), dtype=torch.float32, device=dev)
                    for _ in range(case.layers)]
        ws1 = libdsa.dsa_workspace_bytes(libdsa.DSA_OP_SPARSE_MLA, case.B, case.T, case.H,
                                         case.d, case.k, 1)
        wsg = libdsa.dsa_workspace_bytes(libdsa.DSA_OP_SPARSE_MLA, case.B, case.T, case.H,
                                         case.d, case.k, case.layers)
        self.ws_bytes = max(ws1, wsg)
        self.workspace = (torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
                          if self.ws_bytes else None)
        self.sel_ws = None  # dsa_indexer_topk's workspace, allocated on first use

    # -- the three calls ----------------------------------------------------------------
    def indexer(self):
        c = self.case
        libdsa.dsa_indexer_scores(c.q8, c.q_scale, c.w, c.k8, c.k_scale, self.layout, c.q_pos,
                                  c.B, c.T, c.Hi, c.Di, c.Lmax, self.scores, self.stream)

    def topk(self):
        c = self.case
        libdsa.dsa_topk(self.scores, c.q_pos, c.rows, c.Lmax, c.k, self.idx, self.stream)

    def indexer_topk(self):
        """The fused indexer + top-k (chunked prefill): the index set without the scores."""
        c = self.case
        if self.sel_ws is None:
            n = libdsa.dsa_indexer_topk_workspace_bytes(c.B, c.T, c.Lmax)
            self.sel_ws = torch.empty(n, dtype=torch.uint8, device=c.k8.device)
        libdsa.dsa_indexer_topk(c.q8, c.q_scale, c.w, c.k8, c.k_scale, self.layout, c.q_pos,
                                c.B, c.T, c.Hi, c.Di, c.Lmax, c.k, self.idx, self.sel_ws,
                                self.sel_ws.numel(), self.stream)

    def mla(self, layer=0, idx=None):
        c = self.case
        idx = self.idx if idx is None else idx
        if c.T == 1:
            libdsa.dsa_sparse_mla_decode(c.q[layer], c.kv[layer], self.layout, idx, c.B, c.H,
                                         c.d, c.r, c.k, c.softmax_scale, self.out[layer],
                                         self.lse[layer], self.workspace, self.ws_bytes,
                                         self.stream)
        else:
            libdsa.dsa_sparse_mla_prefill(c.q[layer], c.kv[layer], self.layout, idx, c.B, c.T,
                                          c.H, c.d, c.r, c.k, c.softmax_scale, self.out[layer],
                                          self.lse[layer], self.workspace, self.ws_bytes,
                                          self.stream)

    def topk_mla(self, layer=0):
        """Top-k and sparse MLA decode in one call (one kernel where the row fits)."""
        c = self.case
        libdsa.dsa_topk_sparse_mla_decode(self.scores, c.q_pos, c.Lmax, c.q[layer], c.kv[layer],
                                          self.layout, self.idx, c.B, c.H, c.d, c.r, c.k,
                                          c.softmax_scale, self.out[layer], self.lse[layer],
                                          self.workspace, self.ws_bytes, self.stream)

    def mla_shared(self, idx=None):
        c = self.case
        idx = self.idx if idx is None else idx
        libdsa.dsa_sparse_mla_shared(c.q, c.kv, self.layout, idx, c.B, c.T, c.H, c.d, c.r, c.k,
                                     c.softmax_scale, self.out, self.lse, self.workspace,
                                     self.ws_bytes, self.stream)

    # -- whole steps --------------------------------------------------------------------
    def run(self, layer=0):
        self.indexer()
        if self.case.T == 1:
            self.topk_mla(layer)
        else:
            self.topk()
            self.mla(layer)

    def run_shared(self):
        self.indexer()
        self.topk()
        self.mla_shared()

    def run_fused(self, layer=0):
        """Chunked prefill with the fused indexer + top-k, then sparse MLA."""
        self.indexer_topk()
        self.mla(layer)

    def check_device_error(self):
        st, code = libdsa.dsa_device_error(self.stream)
        if st != libdsa.DSA_OK:
            raise libdsa.DsaError(f"device check (code {code:#x})", st)
