"""Full-size parity at the benchmark workloads (GPU).

Each workload is generated on the device with the benchmark's own seeds and run through
the same calls bench.py times (DsaLayer.run / run_shared: indexer, top-k, sparse MLA in
their launch configuration).  The fp64 oracle then recomputes a few sampled query rows
one by one -- their scores, their top-k set and their attention outputs (fed the GPU's
index set) -- on a compact CPU copy that holds only the sampled sequences' cache rows.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import check_mla, check_scores, check_topk_sets, cpu
from sparse_attention_29_b300 import build, capi, inputs
from sparse_attention_29_b300.pipeline import DsaLayer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    capi.load()
    oracle.build()
    assert torch.cuda.is_available()


def compact(case, seqs, rows_in_seq):
    """CPU case of the sampled sequences (contiguous caches holding only their tokens) and
    the sampled rows of each; returns it with the GPU row numbers of its rows."""
    dev = case.k8.device
    src = []
    for b in seqs:
        s = torch.arange(case.lengths[b], device=dev)
        if case.page_size:
            bt = case.block_table[b].long()
            src.append(bt[s // case.page_size] * case.page_size + s % case.page_size)
        else:
            src.append(case.seq_start[b].long() + s)
    src = torch.cat(src)
    rows = [b * case.T + i for b in seqs for i in rows_in_seq]
    ri = torch.tensor(rows, device=dev)
    lengths = [case.lengths[b] for b in seqs]
    out = inputs.Case(name=case.name + "-sample", kind=case.kind, seed=case.seed, B=len(seqs),
                      T=len(rows_in_seq), lengths=lengths, Hi=case.Hi, Di=case.Di, H=case.H,
                      d=case.d, r=case.r, k=case.k, softmax_scale=case.softmax_scale,
                      layers=case.layers, page_size=0)
    out.q8 = case.q8[ri].cpu()
    out.q_scale = case.q_scale[ri].cpu()
    out.w = case.w[ri].cpu()
    out.q_pos = case.q_pos[ri].cpu()
    out.q = [q[ri].cpu() for q in case.q]
    out.k8 = case.k8[src].cpu()
    out.k_scale = case.k_scale[src].cpu()
    out.kv = [kv[src].cpu() for kv in case.kv]
    out.seq_start = torch.tensor(np.cumsum([0] + lengths[:-1]), dtype=torch.int32)
    out.block_table = None
    return out, rows


def run_and_check(name, seqs, rows_in_seq):
    case = inputs.preset(name, device="cuda")
    lay = DsaLayer(case)
    if case.layers > 1:
        lay.run_shared()
    else:
        lay.run()
    torch.cuda.synchronize()
    lay.check_device_error()
    sub, rows = compact(case, seqs, rows_in_seq)
    ri = torch.tensor(rows, device="cuda")
    ref_scores, abs_terms = oracle.indexer_scores(sub, with_abs=True)
    check_scores(lay.scores[ri, :sub.Lmax], ref_scores, sub.q_pos, abs_terms, Hi=sub.Hi, Di=sub.Di)
    gidx = cpu(lay.idx[ri])
    check_topk_sets(gidx, ref_scores, sub.q_pos, case.k)
    for g in range(case.layers):
        ref_out, ref_lse = oracle.sparse_mla(sub, gidx, layer=g)
        check_mla(lay.out[g][ri], lay.lse[g][ri], ref_out, ref_lse)
    return case, sub


def test_decode_32k_every_row():
    run_and_check("decode_32k", seqs=range(32), rows_in_seq=[0])


def test_ragged_decode_every_row():
    lengths = inputs.ragged_lengths(16, 1024, 200000, inputs.PRESETS["ragged_decode"]["seed"])
    case, sub = run_and_check("ragged_decode", seqs=range(16), rows_in_seq=[0])
    assert max(sub.lengths) > 100000 and min(sub.lengths) < 2048  # long tail and dense rows


# chunked prefill rows at q_pos = 57344 + i: groups of four rows share a tensor-core tile
# (edges between rows 3|4 and 4095|4096), and a row's causal edge falls on a 128-key tile
# boundary when 57345 + i is a multiple of 128 (i = 127, 255, ...)
PREFILL_ROWS = [0, 1, 2, 3, 4, 126, 127, 128, 129, 2047, 2048, 4095, 4096, 6143, 8188, 8189,
                8190, 8191]


def test_prefill_8k_sampled_rows():
    run_and_check("prefill_8k", seqs=[0], rows_in_seq=PREFILL_ROWS)


def test_indexshare_paged_sampled_rows():
    run_and_check("indexshare_paged", seqs=[0, 1, 31, 32, 62, 63], rows_in_seq=[0])
