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


class HostTierGroup:
    """The latent caches of an IndexShare group behind the host tier.

    Per layer the full history stays in pinned host memory and the device keeps a working
    set of C slots per sequence, least recently used (dsa_hisparse_init / _fetch); the
    sparse MLA reads a layer's working set as a cache of one-token pages.  step() runs one
    decode step of the group over its shared index set: each layer's fetch, then its sparse
    MLA.  With `overlap`, the fetches run in order on a second stream and layer l + 1's
    fetch proceeds while layer l attends (the host tier's layer-wise overlap); a layer's
    MLA waits only for its own fetch, and a step's fetches wait for the previous step's
    attention, which still reads the slots they refill.

        group = HostTierGroup(host_kv_layers, host_seq_start, B, Lmax, D, C)
        group.reset()
        group.step(idx, k, step_no, q_layers, out_layers, lse_layers, H, d, r, scale,
                   workspace, ws_bytes)
    """

    def __init__(self, host_kv_layers, host_seq_start, B, Lmax, D, C, device="cuda"):
        self.host_kv = list(host_kv_layers)  # pinned host tensors [rows, D] of bf16 bits
        self.host_seq_start = host_seq_start  # device int32 [B]: first host row of each sequence
        self.B, self.Lmax, self.D, self.C = B, Lmax, D, C
        L = len(self.host_kv)
        i32 = dict(dtype=torch.int32, device=device)
        self.res = [torch.empty((B, Lmax), **i32) for _ in range(L)]
        self.stok = [torch.empty((B, C), **i32) for _ in range(L)]
        self.use = [torch.empty((B, C), **i32) for _ in range(L)]
        self.pool = [torch.empty((B * C, D), dtype=torch.int16, device=device) for _ in range(L)]
        self.stats = [torch.zeros((B, 2), **i32) for _ in range(L)]
        self.layouts = [libdsa.make_layout(B * C, block_table=r, page_size=1) for r in self.res]
        self.fetch_stream = torch.cuda.Stream(device=device)
        self.fetched = [torch.cuda.Event() for _ in range(L)]

    def reset(self):
        for g in range(len(self.host_kv)):
            libdsa.dsa_hisparse_init(self.res[g], self.B, self.Lmax, self.stok[g], self.use[g],
                                     self.C)

    def fetch(self, g, idx, k, step_no, stream=None):
        libdsa.dsa_hisparse_fetch(idx, self.B, k, step_no, self.host_kv[g], self.host_seq_start,
                                  self.D, self.res[g], self.Lmax, self.stok[g], self.use[g],
                                  self.C, self.pool[g], self.stats[g], stream)

    def mla(self, g, idx, k, q, out, lse, H, d, r, scale, workspace, ws_bytes, stream=None):
        libdsa.dsa_sparse_mla_decode(q, self.pool[g].view(torch.bfloat16), self.layouts[g], idx,
                                     self.B, H, d, r, k, scale, out, lse, workspace, ws_bytes,
                                     stream)

    def step(self, idx, k, step_no, q_layers, out_layers, lse_layers, H, d, r, scale,
             workspace, ws_bytes, overlap=True):
        L = len(self.host_kv)
        main = torch.cuda.current_stream()
        if not overlap:
            for g in range(L):
                self.fetch(g, idx, k, step_no)
                self.mla(g, idx, k, q_layers[g], out_layers[g], lse_layers[g], H, d, r, scale,
                         workspace, ws_bytes)
            return
        fs = self.fetch_stream
        fs.wait_stream(main)  # the previous step's attention is done with the slots
        for g in range(L):
            self.fetch(g, idx, k, step_no, fs.cuda_stream)
            self.fetched[g].record(fs)
        for g in range(L):
            main.wait_event(self.fetched[g])
            self.mla(g, idx, k, q_layers[g], out_layers[g], lse_layers[g], H, d, r, scale,
                     workspace, ws_bytes)
        main.wait_stream(fs)
