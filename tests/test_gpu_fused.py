"""GPU parity of dsa_indexer_topk, the fused indexer + top-k of chunked prefill.

The fused call must select exactly what the oracle's full sort selects on the oracle's
scores where those are exact (integer-valued inputs), and exactly what the two separate
calls (dsa_indexer_scores, dsa_topk) select on realistic inputs: both evaluate every
score with the same fp32 arithmetic and apply the same order and tie rule, so their index
rows are identical bit for bit.  The cases cover ragged query groups, rows that see at
most k tokens (dense), a paged cache, and a bin holding thousands of exact ties (the
radix path of the final selection, ties going to the lower token index).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import check_topk_sets, cpu
from sparse_attention_29_b300 import build, capi, inputs
from sparse_attention_29_b300.pipeline import DsaLayer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    capi.load()
    oracle.build()
    assert torch.cuda.is_available()


def fused_and_separate(case):
    lay = DsaLayer(case.to("cuda"))
    lay.indexer()
    lay.topk()
    torch.cuda.synchronize()
    lay.check_device_error()
    sep = lay.idx.clone()
    lay.idx.fill_(-7)
    lay.indexer_topk()
    torch.cuda.synchronize()
    lay.check_device_error()
    return lay, sep


def test_fused_integer_prefill_bit_exact():
    case = inputs.make_case(kind="int", seed=71, lengths=[8192], T=67)
    lay, sep = fused_and_separate(case)
    ref = oracle.topk(oracle.indexer_scores(case), case.q_pos, case.k)
    assert np.array_equal(cpu(lay.idx).numpy(), ref)
    assert torch.equal(lay.idx, sep)


@pytest.mark.parametrize("lengths,T,paged", [
    ([20000], 45, 0),            # realistic prefill rows, ragged last group
    ([9000, 5000], 37, 64),      # two sequences, paged cache
    ([2100], 100, 0),            # rows at positions 2000..2099: dense and sparse rows
])
def test_fused_equals_separate_calls(lengths, T, paged):
    case = inputs.make_case(kind="planted", seed=72 + T, lengths=lengths, T=T, page_size=paged)
    lay, sep = fused_and_separate(case)
    assert torch.equal(lay.idx, sep)
    ref_scores = oracle.indexer_scores(case)
    check_topk_sets(lay.idx, ref_scores, case.q_pos, case.k)


def test_fused_many_exact_ties_take_the_lower_indices():
    # every key the same: every row's scores are all equal, so one coarse bin holds every
    # candidate (more than the direct ranking holds) and the k lowest indices win
    case = inputs.make_case(kind="int", seed=73, lengths=[9000], T=8)
    case.k8[:] = case.k8[0]
    case.k_scale[:] = 1.0
    lay, sep = fused_and_separate(case)
    ref = oracle.topk(oracle.indexer_scores(case), case.q_pos, case.k)
    got = cpu(lay.idx).numpy()
    assert np.array_equal(got, ref)
    assert np.array_equal(got[0], np.arange(case.k))
    assert torch.equal(lay.idx, sep)


def test_fused_prefill_8k_sampled_rows():
    """The chunked-prefill workload at full size: fused index rows equal the separate
    calls' rows everywhere, and sampled rows agree with the oracle's selection."""
    case = inputs.preset("prefill_8k", device="cuda")
    lay = DsaLayer(case)
    lay.indexer()
    lay.topk()
    torch.cuda.synchronize()
    sep = lay.idx.clone()
    lay.idx.fill_(-7)
    lay.indexer_topk()
    torch.cuda.synchronize()
    lay.check_device_error()
    assert torch.equal(lay.idx, sep)
    rows = [0, 3, 4, 127, 128, 4095, 8191]
    ri = torch.tensor(rows, device="cuda")
    sub = inputs.Case(name="prefill-sample", kind=case.kind, seed=case.seed, B=1, T=len(rows),
                      lengths=case.lengths, Hi=case.Hi, Di=case.Di, H=case.H, d=case.d,
                      r=case.r, k=case.k, softmax_scale=case.softmax_scale, layers=1,
                      page_size=0)
    sub.q8, sub.q_scale, sub.w = case.q8[ri].cpu(), case.q_scale[ri].cpu(), case.w[ri].cpu()
    sub.q_pos = case.q_pos[ri].cpu()
    sub.q = [case.q[0][ri].cpu()]
    sub.k8, sub.k_scale, sub.kv = case.k8.cpu(), case.k_scale.cpu(), [case.kv[0].cpu()]
    sub.seq_start = case.seq_start.cpu()
    check_topk_sets(lay.idx[ri], oracle.indexer_scores(sub), sub.q_pos, case.k)
