"""Integer-valued workloads at the production shapes (GPU): bit-exact scores and indices.

Every indexer input is an integer in [-4, 4] (exact in e4m3), every weight is 0.5, 1 or 2
and every scale is 1, with Hi = 64 heads of Di = 128: a head's dot product is an integer
of magnitude at most 128 * 16 = 2048 and a score a multiple of 0.5 below 64 * 2 * 2048 =
2^18, so every product and partial sum is exact in fp32 and the kernels' scores must equal
the oracle's fp64 scores bit for bit.  Scores this coarse tie often; the top-k must break
every tie toward the lower token index exactly as the oracle's full sort does.  The shapes
run the launch paths of the realistic workloads: the decode form (one query row of 64
heads per tensor-core tile), the chunked-prefill form (four rows of 64 heads per tile) and
IndexShare over a paged cache.  Attention outputs are compared with the oracle fed the
same index set within one bf16 ulp of the correctly rounded value plus the fp32 bound of
forming the weighted mean, and of merging split rows from bf16 partials (tests/parity.py).
"""
import numpy as np
import pytest
import torch

import oracle
from parity import check_mla_integer, cpu
from sparse_attention_29_b300 import build, capi, inputs
from sparse_attention_29_b300.pipeline import DsaLayer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    capi.load()
    oracle.build()
    assert torch.cuda.is_available()


def exact_scores_and_indices(lay, case):
    g = cpu(lay.scores).double().numpy()
    ref = oracle.indexer_scores(case)
    vis = np.arange(case.Lmax)[None, :] <= case.q_pos.numpy()[:, None]
    bad = np.nonzero(g[vis] != ref[vis])[0]
    assert bad.size == 0, f"{bad.size} scores differ"
    ref_idx = oracle.topk(ref, case.q_pos, case.k)
    gi = cpu(lay.idx).numpy()
    rows_bad = [t for t in range(case.rows) if not np.array_equal(gi[t], ref_idx[t])]
    assert not rows_bad, f"index rows differ: {rows_bad[:5]}"
    # the case does exercise ties at the k-th score
    ties = 0
    for t in range(case.rows):
        n = int(case.q_pos[t]) + 1
        if n > case.k:
            kth = np.sort(ref[t, :n])[-case.k]
            ties += int(np.sum(ref[t, :n] == kth) > 1)
    return ref_idx, ties


def test_integer_decode_production_shape():
    # 32 rows x 8192 context, plus rows at 2048 / 2049 (the dense edge) and a ragged one
    lengths = [8192] * 29 + [2048, 2049, 5000]
    case = inputs.make_case(kind="int", seed=61, lengths=lengths, T=1)
    lay = DsaLayer(case.to("cuda"))
    lay.run()
    torch.cuda.synchronize()
    lay.check_device_error()
    ref_idx, ties = exact_scores_and_indices(lay, case)
    assert ties > 0
    ref_out, ref_lse = oracle.sparse_mla(case, ref_idx)
    check_mla_integer(lay.out[0], lay.lse[0], case, lay.idx, ref_out, ref_lse, split_exchange=True)


def test_integer_chunked_prefill_production_shape():
    # 67 query rows at the end of an 8192-token context: 16 full groups of four rows and a
    # ragged group of three; the causal edge of every row falls at a different key
    case = inputs.make_case(kind="int", seed=62, lengths=[8192], T=67)
    lay = DsaLayer(case.to("cuda"))
    lay.run()
    torch.cuda.synchronize()
    lay.check_device_error()
    ref_idx, ties = exact_scores_and_indices(lay, case)
    assert ties > 0
    ref_out, ref_lse = oracle.sparse_mla(case, ref_idx)
    check_mla_integer(lay.out[0], lay.lse[0], case, lay.idx, ref_out, ref_lse, split_exchange=True)


def test_integer_indexshare_paged_production_shape():
    case = inputs.make_case(kind="int", seed=63, lengths=[8192, 6000, 8192, 3000], T=1,
                            layers=4, page_size=64)
    lay = DsaLayer(case.to("cuda"))
    lay.run_shared()
    torch.cuda.synchronize()
    lay.check_device_error()
    ref_idx, _ = exact_scores_and_indices(lay, case)
    for g in range(case.layers):
        ref_out, ref_lse = oracle.sparse_mla(case, ref_idx, layer=g)
        check_mla_integer(lay.out[g], lay.lse[g], case, lay.idx, ref_out, ref_lse, layer=g,
                          split_exchange=True)
    # the paged run equals the contiguous run of the same tokens, bit for bit
    flat = DsaLayer(inputs.unpage(case).to("cuda"))
    flat.run_shared()
    torch.cuda.synchronize()
    assert torch.equal(flat.idx, lay.idx)
    for g in range(case.layers):
        assert torch.equal(flat.out[g], lay.out[g])
