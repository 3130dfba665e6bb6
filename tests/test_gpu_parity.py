"""GPU parity: libdsa's CUDA path (through the C ABI) against the fp64 oracle.

Small cases span several 128-key tiles with ragged tails; the integer-valued workload is
checked bit-exactly.  Tolerances are defined in tests/parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import (check_case_scores, check_mla, check_mla_integer, check_topk_sets, cpu)
from sparse_attention_29_b300 import build, capi, inputs
from sparse_attention_29_b300.pipeline import DsaLayer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    capi.load()
    assert torch.cuda.is_available()


def gpu_layer(case):
    return DsaLayer(case.to("cuda"))


def assert_no_device_error(layer):
    layer.check_device_error()


# ---- integer-valued workload: exact -------------------------------------------------------

def test_tiny_int_exact():
    case = inputs.preset("tiny_int")
    lay = gpu_layer(case)
    lay.run()
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    ref_scores = oracle.indexer_scores(case)
    g = cpu(lay.scores).double().numpy()
    vis = np.arange(case.Lmax)[None, :] <= case.q_pos.numpy()[:, None]
    assert np.array_equal(g[vis], ref_scores[vis])          # bit-exact scores
    ref_idx = oracle.topk(ref_scores, case.q_pos, case.k)
    assert np.array_equal(cpu(lay.idx).numpy(), ref_idx)     # bit-exact indices (with ties)
    ref_out, ref_lse = oracle.sparse_mla(case, ref_idx)
    # within one bf16 ulp of the correctly rounded value (plus the fp32 bound near zero)
    check_mla_integer(lay.out[0], lay.lse[0], case, lay.idx, ref_out, ref_lse)


# ---- indexer ------------------------------------------------------------------------------

@pytest.mark.parametrize("lengths,T,paged", [
    ([3000, 700, 2048 + 131, 77], 1, 0),     # decode, ragged, one context under one tile
    ([2500], 37, 0),                         # prefill form, ragged row group
    ([1500, 900], 5, 64),                    # prefill form on a paged cache
    ([4100, 129, 2048], 1, 64),              # decode on a paged cache
])
def test_indexer_matches_oracle(lengths, T, paged):
    case = inputs.make_case(seed=101 + T, lengths=lengths, T=T, page_size=paged)
    lay = gpu_layer(case)
    lay.indexer()
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    check_case_scores(lay.scores, case)


@pytest.mark.parametrize("Hi,Di,T", [
    (128, 128, 1),   # decode, 128 heads: one row of N = 128 per tile
    (128, 128, 5),   # two rows of 128 heads per tile, a ragged last group
    (256, 64, 2),    # the widest query group: one row of N = 256
    (100, 128, 3),   # heads padded to 112, two rows per tile
    (1, 32, 20),     # one head padded to 16: sixteen rows per tile
])
def test_indexer_wide_and_narrow_heads(Hi, Di, T):
    """Head counts away from 64 (up to the 256 columns of one tensor-core tile), where the
    epilogue takes the general path, in decode and prefill form, against the oracle."""
    case = inputs.make_case(seed=31 + Hi + T, lengths=[1500, 777], T=T, Hi=Hi, Di=Di, H=4,
                            d=64, r=16, k=256)
    lay = gpu_layer(case)
    lay.indexer()
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    check_case_scores(lay.scores, case)


@pytest.mark.parametrize("Hi,Di", [(4, 32), (16, 64), (24, 128), (64, 32)])
def test_indexer_head_shapes(Hi, Di):
    case = inputs.make_case(seed=7 + Hi, lengths=[1000, 301], T=3, Hi=Hi, Di=Di, H=4, d=64,
                            r=16, k=256)
    lay = gpu_layer(case)
    lay.indexer()
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    check_case_scores(lay.scores, case)


# ---- top-k on fixed fp32 scores (bit-exact; both sides compare fp32 values) -----------------

def _scores_with_ties(rows, Lmax, seed, levels=None):
    g = torch.Generator().manual_seed(seed)
    if levels:
        return (torch.randint(0, levels, (rows, Lmax), generator=g).float() * 0.5 - 3.0)
    return torch.randn((rows, Lmax), generator=g)


@pytest.mark.parametrize("Lmax,k,levels", [
    (3000, 2048, None), (3000, 2048, 7), (40960, 2048, None), (41000, 2048, 13),
    (65536, 2048, None), (200000, 2048, None), (5000, 100, 3), (9000, 8192, None),
    (1000, 1, None), (70000, 2048, 1),
])
def test_topk_exact_on_fixed_scores(Lmax, k, levels):
    rows = 6
    s = _scores_with_ties(rows, Lmax, seed=Lmax + k, levels=levels)
    # positions: dense (n <= k), exactly k, k + 1, and long rows
    q_pos = torch.tensor([min(k - 1, Lmax - 1), min(k, Lmax - 1), Lmax - 1, Lmax // 2,
                          max(0, Lmax - 3), Lmax - 1], dtype=torch.int32)
    if levels is None:
        s[5, : Lmax // 3] = 0.0                    # a run of exact zeros
        s[5, 7] = -0.0
    out = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    capi.dsa_topk(s.cuda(), q_pos.cuda(), rows, Lmax, k, out)
    torch.cuda.synchronize()
    ref = oracle.topk(s.numpy(), q_pos.numpy(), k)
    assert np.array_equal(cpu(out).numpy(), ref)


def test_topk_exact_on_extreme_scores():
    """Scores the fp16-based bins cannot separate: beyond the fp16 range (every one in the
    infinity bin), +inf and -inf runs, subnormals (all in the zero bin with +-0), and
    distinct fp32 values inside one fp16 step; the selection stays exact, ties to the
    lower index."""
    Lmax, k, rows = 20000, 2048, 6
    g = torch.Generator().manual_seed(77)
    s = torch.randn((rows, Lmax), generator=g)
    s[0] *= 1e30                                   # beyond fp16: one bin holds all
    s[1, torch.randperm(Lmax, generator=g)[:100]] = float("inf")
    s[2] *= 1e-40                                  # subnormal: the zero bin, with +-0
    s[2, 10:20] = 0.0
    s[2, 20:30] = -0.0
    s[3, torch.randperm(Lmax, generator=g)[: Lmax // 2]] = float("-inf")
    s[4] = 1.0 + torch.arange(Lmax, dtype=torch.float32) * 2.0 ** -20  # one fp16 step wide
    s[4, ::7] = 1.0 + 2.0 ** -20 * 19990              # and ~2900 exact ties near the top
    q_pos = torch.full((rows,), Lmax - 1, dtype=torch.int32)
    q_pos[5] = Lmax // 3
    out = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    capi.dsa_topk(s.cuda(), q_pos.cuda(), rows, Lmax, k, out)
    torch.cuda.synchronize()
    ref = oracle.topk(s.numpy(), q_pos.numpy(), k)
    assert np.array_equal(cpu(out).numpy(), ref)


# ---- sparse MLA ---------------------------------------------------------------------------

def _random_idx(case, seed, frac_invalid=0.0):
    g = np.random.default_rng(seed)
    rows = case.rows
    idx = np.full((rows, case.k), -1, np.int32)
    for t in range(rows):
        n = int(case.q_pos[t]) + 1
        m = min(n, case.k)
        sel = np.sort(g.choice(n, size=m, replace=False))
        idx[t, :m] = sel
        if frac_invalid:
            kill = g.random(case.k) < frac_invalid
            idx[t, kill] = -1
    return torch.from_numpy(idx)


@pytest.mark.parametrize("lengths,T,k,paged", [
    ([5000, 3000, 2100], 1, 2048, 0),   # decode: few rows -> split-KV path
    ([700, 300], 1, 2048, 0),           # dense rows (fewer tokens than k), -1 padding
    ([1200], 24, 512, 0),               # prefill form
    ([2600, 1900], 1, 1000, 64),        # paged, k not a multiple of the tile
])
def test_sparse_mla_matches_oracle(lengths, T, k, paged):
    case = inputs.make_case(seed=200 + k, lengths=lengths, T=T, k=k, page_size=paged)
    lay = gpu_layer(case)
    idx = _random_idx(case, seed=k, frac_invalid=0.02)
    lay.mla(idx=idx.cuda())
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    ref_out, ref_lse = oracle.sparse_mla(case, idx)
    check_mla(lay.out[0], lay.lse[0], ref_out, ref_lse)


@pytest.mark.parametrize("k", [1, 33, 4096, 8192])
def test_topk_and_mla_edge_k(k):
    """k at the ends of the supported range: one key, a partial tile, and 64 / 128 tiles
    (a row then needs more splits' worth of tiles); a sparse and a dense row.  The index
    set from the GPU's own top-k equals the oracle's (scores fixed by the oracle), the
    attention matches the oracle fed it, and the one-call form equals the two calls."""
    case = inputs.make_case(seed=500 + k, lengths=[12000, 300, 9000], T=1, k=k)
    lay = gpu_layer(case)
    lay.indexer()
    lay.topk()
    lay.mla()
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    ref_scores = oracle.indexer_scores(case)
    check_topk_sets(lay.idx, ref_scores, case.q_pos, case.k)
    gidx = cpu(lay.idx)
    ref_out, ref_lse = oracle.sparse_mla(case, gidx)
    check_mla(lay.out[0], lay.lse[0], ref_out, ref_lse)
    idx_sep, out_sep, lse_sep = lay.idx.clone(), lay.out[0].clone(), lay.lse[0].clone()
    lay.idx.fill_(-7)
    lay.out[0].zero_()
    lay.topk_mla()
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    assert torch.equal(lay.idx, idx_sep)
    assert torch.equal(lay.out[0], out_sep) and torch.equal(lay.lse[0], lse_sep)


@pytest.mark.parametrize("H,d,r,T", [
    (32, 256, 0, 1),    # no rope dims: the key is the latent part alone
    (64, 448, 64, 1),   # seven latent chunks: the last value M-block is half used
    (16, 384, 32, 3),   # prefill form, six latent chunks, 16 heads
    (48, 192, 8, 1),    # three latent chunks, a rope part one 16-byte granule wide
])
def test_sparse_mla_other_shapes(H, d, r, T):
    """Shapes inside the supported range (H <= 64, d a multiple of 64 up to 512, r <= 64)
    that the production and tiny cases do not reach, decode (split-KV) and prefill, with
    2 % invalid indices, against the oracle fed the same index set."""
    case = inputs.make_case(seed=700 + d + r, lengths=[3000, 900], T=T, Hi=4, Di=32, H=H,
                            d=d, r=r, k=512)
    lay = gpu_layer(case)
    idx = _random_idx(case, seed=d + r, frac_invalid=0.02)
    lay.mla(idx=idx.cuda())
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    ref_out, ref_lse = oracle.sparse_mla(case, idx)
    check_mla(lay.out[0], lay.lse[0], ref_out, ref_lse)


def test_sparse_mla_small_heads_and_dims():
    case = inputs.make_case(seed=9, lengths=[900, 400], T=2, Hi=4, Di=32, H=12, d=128, r=32,
                            k=300, softmax_scale=0.1)
    lay = gpu_layer(case)
    idx = _random_idx(case, seed=3)
    lay.mla(idx=idx.cuda())
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.sparse_mla(case, idx)
    check_mla(lay.out[0], lay.lse[0], ref_out, ref_lse)


def test_sparse_mla_all_invalid_row():
    case = inputs.make_case(seed=10, lengths=[500, 600], T=1, k=256)
    lay = gpu_layer(case)
    idx = _random_idx(case, seed=4)
    idx[1] = -1
    lay.mla(idx=idx.cuda())
    torch.cuda.synchronize()
    out = cpu(lay.out[0]).float()
    assert torch.all(out[1] == 0)
    assert torch.all(torch.isneginf(cpu(lay.lse[0])[1]))
    ref_out, ref_lse = oracle.sparse_mla(case, idx)
    check_mla(lay.out[0][:1], lay.lse[0][:1], ref_out[:1], ref_lse[:1])


# ---- whole layer and IndexShare ------------------------------------------------------------

@pytest.mark.parametrize("lengths,T,paged", [
    ([6000, 1000, 2049], 1, 0),
    ([3000], 16, 0),
])
def test_dsa_layer_end_to_end(lengths, T, paged):
    case = inputs.make_case(kind="planted", seed=300 + T, lengths=lengths, T=T,
                            page_size=paged)
    lay = gpu_layer(case)
    lay.run()
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    ref_scores = check_case_scores(lay.scores, case)
    check_topk_sets(lay.idx, ref_scores, case.q_pos, case.k)
    ref_out, ref_lse = oracle.sparse_mla(case, cpu(lay.idx))
    check_mla(lay.out[0], lay.lse[0], ref_out, ref_lse)


def test_indexshare_paged_group():
    case = inputs.make_case(seed=400, lengths=[3000, 2200, 700], T=1, layers=4, page_size=64)
    lay = gpu_layer(case)
    lay.run_shared()
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    ref_idx, per_layer = oracle.indexshare_group(case)
    ref_scores = oracle.indexer_scores(case)
    check_topk_sets(lay.idx, ref_scores, case.q_pos, case.k)
    gidx = cpu(lay.idx)
    for g in range(4):
        ref_out, ref_lse = oracle.sparse_mla(case, gidx, layer=g)
        check_mla(lay.out[g], lay.lse[g], ref_out, ref_lse)
    # paged == contiguous on the un-paged copy, bit for bit
    flat = gpu_layer(inputs.unpage(case))
    flat.run_shared()
    torch.cuda.synchronize()
    assert torch.equal(flat.idx, lay.idx)
    for g in range(4):
        assert torch.equal(flat.out[g], lay.out[g])


def test_shared_layers_match_the_oracle_and_separate_calls():
    """An IndexShare launch plans its split for all layers' rows at once, so with few rows
    it splits them less than separate per-layer calls do: every layer of the launch and
    of the separate calls matches the oracle, the two agree to the merge's rounding, and
    the launch is deterministic."""
    case = inputs.make_case(seed=401, lengths=[2500, 4000], T=1, layers=3)
    lay = gpu_layer(case)
    lay.run_shared()
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    shared = [o.clone() for o in lay.out]
    shared_lse = [x.clone() for x in lay.lse]
    gidx = cpu(lay.idx)
    for g in range(3):
        ref_out, ref_lse = oracle.sparse_mla(case, gidx, layer=g)
        check_mla(shared[g], shared_lse[g], ref_out, ref_lse)
        lay.mla(layer=g)
        torch.cuda.synchronize()
        check_mla(lay.out[g], lay.lse[g], ref_out, ref_lse)
        assert (lay.out[g].float() - shared[g].float()).abs().max().item() <= 2e-2
    lay.mla_shared()
    torch.cuda.synchronize()
    for g in range(3):
        assert torch.equal(lay.out[g], shared[g]) and torch.equal(lay.lse[g], shared_lse[g])


@pytest.mark.parametrize("lengths", [
    [3000] * 32,            # 4 splits per row: the row's cluster selects, then attends
    [5000, 3000, 2100],     # more splits than a cluster holds: a separate top-k launch first
    [2600] * 160,           # one CTA per row selects and attends
    [1500, 2049, 2048] * 12,  # dense rows and the dense edge
])
def test_topk_and_mla_in_one_call_equal_the_two_calls(lengths):
    case = inputs.make_case(kind="planted", seed=len(lengths), lengths=lengths, T=1)
    lay = gpu_layer(case)
    lay.indexer()
    lay.topk()
    lay.mla()
    torch.cuda.synchronize()
    idx_sep, out_sep, lse_sep = lay.idx.clone(), lay.out[0].clone(), lay.lse[0].clone()
    lay.idx.fill_(-7)
    lay.out[0].zero_()
    lay.topk_mla()
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    assert torch.equal(lay.idx, idx_sep)
    assert torch.equal(lay.out[0], out_sep) and torch.equal(lay.lse[0], lse_sep)


def test_one_call_on_extreme_scores():
    """The one-call decode form on scores that force the radix passes and the tie rules
    inside the sparse MLA kernel's tile buffers: the index sets equal the oracle's, and
    index sets and attention equal the two calls bit for bit."""
    case = inputs.make_case(seed=88, lengths=[20000] * 6, T=1)
    lay = gpu_layer(case)
    g = torch.Generator().manual_seed(78)
    s = torch.randn((6, case.Lmax), generator=g)
    s[0] *= 1e30                                   # one fp16 bin holds half the row
    s[1, torch.randperm(case.Lmax, generator=g)[:100]] = float("inf")
    s[2] *= 1e-40                                  # subnormals and +-0
    s[2, 10:20] = 0.0
    s[2, 20:30] = -0.0
    s[4] = 1.0 + torch.arange(case.Lmax, dtype=torch.float32) * 2.0 ** -20
    s[4, ::7] = 1.0 + 2.0 ** -20 * 19990           # ~2900 exact ties near the top
    lay.scores.copy_(s.cuda())
    lay.topk()
    lay.mla()
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    ref = oracle.topk(s.numpy(), cpu(case.q_pos).numpy(), case.k)
    assert np.array_equal(cpu(lay.idx).numpy(), ref)
    idx_sep, out_sep, lse_sep = lay.idx.clone(), lay.out[0].clone(), lay.lse[0].clone()
    lay.idx.fill_(-7)
    lay.out[0].zero_()
    lay.topk_mla()
    torch.cuda.synchronize()
    assert_no_device_error(lay)
    assert torch.equal(lay.idx, idx_sep)
    assert torch.equal(lay.out[0], out_sep) and torch.equal(lay.lse[0], lse_sep)


def test_concurrent_streams_equal_sequential_runs():
    """Calls on different streams with their own buffers may run at once: three layers (a
    decode batch in one call, a decode batch as two calls, a prefill chunk) stepped
    concurrently on three streams, several times, give what each gives alone."""
    cases = [inputs.make_case(seed=601, lengths=[3000] * 8, T=1),
             inputs.make_case(seed=602, lengths=[5000, 2600, 900], T=1),
             inputs.make_case(seed=603, lengths=[2500], T=16)]
    steps = [lambda l: l.run(), lambda l: (l.indexer(), l.topk(), l.mla()), lambda l: l.run()]
    alone = []
    for c, st in zip(cases, steps):
        lay = gpu_layer(c)
        st(lay)
        torch.cuda.synchronize()
        assert_no_device_error(lay)
        alone.append((lay.idx.clone(), lay.out[0].clone(), lay.lse[0].clone()))
    streams = [torch.cuda.Stream() for _ in cases]
    lays = [DsaLayer(c.to("cuda"), stream=s) for c, s in zip(cases, streams)]
    torch.cuda.synchronize()
    for _ in range(3):
        for lay, st in zip(lays, steps):
            st(lay)
        torch.cuda.synchronize()
        for lay, (idx, out, lse) in zip(lays, alone):
            assert_no_device_error(lay)
            assert torch.equal(lay.idx, idx)
            assert torch.equal(lay.out[0], out) and torch.equal(lay.lse[0], lse)
