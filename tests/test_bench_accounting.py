"""bench.py's byte and FLOP accounting and its choice of the headline roofline (host logic,
no GPU): the kernel with the largest share of the step's kernel time is the headline, its
figures are its algorithmic work over its duration against the peak, and the one-call
top-k + sparse MLA launch counts its index set once."""
import importlib.util
import math
import os
import types

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_acct", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _decode(rows=32, L=32768, k=2048):
    return types.SimpleNamespace(lengths=[L] * rows, T=1, d=512, r=64, k=k, Di=128, Hi=64,
                                 H=64, layers=1, rows=rows,
                                 q_pos=torch.full((rows,), L - 1, dtype=torch.int32))


def test_per_query_bytes_decode_32k(bench):
    case = _decode()
    b_idx, b_topk, b_mla = bench.per_query_bytes(case)
    L, k, D = 32768, 2048, 576
    # indexer: keys + scales of every visible token, the query group, the scores written
    assert b_idx == 32 * (L * (128 + 4) + 64 * 128 + 4 + 64 * 4 + 4 + 4 * L)
    # top-k: scores read, indices written (+ the row's position)
    assert b_topk == 32 * (4 * L + 4 * k + 4)
    # sparse MLA: the selected rows, the query, the output and lse, the indices read
    assert b_mla == 32 * (k * D * 2 + 64 * D * 2 + 64 * 512 * 2 + 64 * 4 + 4 * k)
    # the whole step leaves out the score round trip between the two-call form's kernels
    step = b_idx + b_topk + b_mla - bench.scores_in_step(case)
    assert step == 219_169_152


def test_one_call_counts_the_index_set_once(bench):
    case = _decode()
    _, b_topk, b_mla = bench.per_query_bytes(case)
    assert bench.one_call_bytes(case) == b_topk + b_mla - 4 * case.k * case.rows
    assert bench.one_call_bytes(case) == 84_418_688


def test_headline_is_the_kernel_with_the_largest_share(bench):
    case = _decode()
    args = types.SimpleNamespace(workload="decode_32k")
    head, allk = bench.step_rooflines(case, args, 0.035, 0.0135, 0.0324, 0.0446, False,
                                      6494.9, 1801.9, "measured")
    assert set(allk) == {"indexer", "topk_and_sparse_mla_one_call"}
    assert head is allk["topk_and_sparse_mla_one_call"]
    assert head["achieved"] == pytest.approx(84_418_688 / 44.6e-6 / 1e9)
    assert head["frac"] == pytest.approx(head["achieved"] / 6494.9)
    # a faster one-call launch hands the headline to the indexer
    head2, _ = bench.step_rooflines(case, args, 0.035, 0.0135, 0.0324, 0.030, False,
                                    6494.9, 1801.9, "measured")
    assert head2["kernel"] == "indexer"
    # the two-call form lists the top-k and the sparse MLA separately
    head3, allk3 = bench.step_rooflines(case, args, 0.035, 0.0135, 0.0324, None, False,
                                        6494.9, 1801.9, "measured")
    assert set(allk3) == {"indexer", "topk", "sparse_mla"} and head3["kernel"] == "indexer"


def test_prefill_rooflines_are_tensor_bound(bench):
    pos = torch.arange(57344, 65536, dtype=torch.int32)
    case = types.SimpleNamespace(lengths=[65536], T=8192, d=512, r=64, k=2048, Di=128, Hi=64,
                                 H=64, layers=1, rows=8192, q_pos=pos)
    args = types.SimpleNamespace(workload="prefill_8k")
    head, allk = bench.step_rooflines(case, args, 6.74, 2.18, 5.12, None, False,
                                      6494.9, 1801.9, "measured")
    flops = float((pos.long() + 1).sum()) * 64 * 128 * 2
    assert head["kernel"] == "indexer" and head["bound"] == "tensor"
    assert head["algorithmic_flops"] == flops
    assert head["peak"] == pytest.approx(2 * 1801.9)  # fp8 taken as twice the bf16 burst
    assert allk["sparse_mla"]["peak"] == pytest.approx(1801.9)
    assert allk["sparse_mla"]["algorithmic_flops"] == 8192 * 2048 * 64 * (2.0 * 576 + 2.0 * 512)


def test_profile_run_without_times_falls_back_to_the_indexer(bench):
    case = _decode()
    args = types.SimpleNamespace(workload="decode_32k")
    nan = float("nan")
    head, allk = bench.step_rooflines(case, args, nan, nan, nan, None, False,
                                      6494.9, 1801.9, "measured")
    assert head["kernel"] == "indexer" and math.isnan(head["frac"])
