"""GPU parity of dsa_cache_append (new tokens into the caches) against the oracle.

The e4m3 codes, the fp32 scales and the copied latent rows are integer/byte results, so
the comparison is bit-exact; rows that no token targets must stay untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import check_case_scores
from sparse_attention_29_b300 import build, capi

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    capi.load()
    assert torch.cuda.is_available()


def make_tokens(seed, n, Di, D):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(n, Di, generator=g)
    # spread of magnitudes: tiny keys (subnormal codes), huge keys, an all-zero key
    k *= torch.exp(torch.randn(n, 1, generator=g) * 3)
    if n > 2:
        k[1] = 0.0
        k[2] *= 1e-6
    c = torch.randint(-32768, 32767, (n, D), generator=g, dtype=torch.int16).view(torch.uint16)
    return k.contiguous(), c.contiguous()


def run_both(k, c, seq, pos, B, num_rows, Di, D, seq_start=None, block_table=None, ps=0):
    """GPU append into sentinel-filled caches vs the oracle on copies of the same caches."""
    fill = np.random.default_rng(7)
    k8_0 = fill.integers(0, 256, (num_rows, Di), dtype=np.uint8)
    ks_0 = fill.standard_normal(num_rows).astype(np.float32)
    kv_0 = fill.integers(0, 65536, (num_rows, D), dtype=np.uint16) if D else None
    k8_ref, ks_ref = k8_0.copy(), ks_0.copy()
    kv_ref = None if kv_0 is None else kv_0.copy()
    skipped = oracle.cache_append(k, c, seq, pos, B, k8_ref, ks_ref, kv_ref,
                                  seq_start=seq_start, block_table=block_table, page_size=ps)
    dev = "cuda"
    k8 = torch.from_numpy(k8_0).to(dev)
    ks = torch.from_numpy(ks_0).to(dev)
    kv = None if kv_0 is None else torch.from_numpy(kv_0.view(np.int16)).to(dev)
    ss = None if seq_start is None else torch.from_numpy(seq_start).to(dev)
    bt = None if block_table is None else torch.from_numpy(block_table).to(dev)
    layout = capi.make_layout(num_rows, seq_start=ss, block_table=bt, page_size=ps)
    kd, cd = k.to(dev), (None if c is None else c.view(torch.int16).to(dev))
    sq, pq = torch.from_numpy(seq).to(dev), torch.from_numpy(pos).to(dev)
    capi.dsa_cache_append(kd, cd, sq, pq, len(seq), B, Di, D, layout, k8, ks, kv)
    st, code = capi.dsa_device_error()
    assert np.array_equal(k8.cpu().numpy(), k8_ref)
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), ks_ref.view(np.uint32))
    if kv is not None:
        assert np.array_equal(kv.cpu().numpy().view(np.uint16), kv_ref)
    return skipped, st, code


@pytest.mark.parametrize("Di", [32, 64, 128])
def test_contiguous_append_bit_exact(Di):
    B, D, per = 3, 576, 37            # 111 tokens: 14 full blocks of 8 warps and a tail
    n = B * per
    k, c = make_tokens(Di, n, Di, D)
    seq = np.repeat(np.arange(B, dtype=np.int32), per)
    pos = np.tile(np.arange(100, 100 + per, dtype=np.int32), B)
    seq_start = np.array([0, 200, 400], np.int32)
    skipped, st, _ = run_both(k, c, seq, pos, B, 600, Di, D, seq_start=seq_start)
    assert skipped == 0 and st == capi.DSA_OK


def test_paged_append_bit_exact_and_bad_tokens_reported():
    B, Di, D, ps, pps = 4, 128, 576, 64, 8
    n = 300
    k, c = make_tokens(5, n, Di, D)
    rng = np.random.default_rng(5)
    bt = rng.permutation(B * pps).astype(np.int32).reshape(B, pps)
    seq = rng.integers(0, B, n).astype(np.int32)
    # distinct (seq, pos) pairs so that no two tokens share a row
    pos = np.zeros(n, np.int32)
    for b in range(B):
        idx = np.nonzero(seq == b)[0]
        pos[idx] = rng.choice(ps * pps, len(idx), replace=False)
    pos[7] = ps * pps + 3      # past the block table: skipped, reported
    skipped, st, code = run_both(k, c, seq, pos, B, B * pps * ps, Di, D, block_table=bt, ps=ps)
    assert skipped == 1
    assert st == capi.DSA_ERR_DEVICE and code == (5 << 16) | 4


def test_keys_only_and_empty_calls():
    B, Di = 2, 64
    k, _ = make_tokens(9, 20, Di, 8)
    seq = np.array([0] * 10 + [1] * 10, np.int32)
    pos = np.array(list(range(10)) * 2, np.int32)
    seq_start = np.array([0, 10], np.int32)
    skipped, st, _ = run_both(k, None, seq, pos, B, 20, Di, 0, seq_start=seq_start)
    assert skipped == 0 and st == capi.DSA_OK
    # n == 0 launches nothing and succeeds
    ss = torch.zeros(1, dtype=torch.int32, device="cuda")  # kept alive: the layout holds its address
    layout = capi.make_layout(4, seq_start=ss)
    k8 = torch.zeros(4, Di, dtype=torch.uint8, device="cuda")
    ks = torch.zeros(4, dtype=torch.float32, device="cuda")
    e = torch.zeros(0, dtype=torch.int32, device="cuda")
    capi.dsa_cache_append(torch.zeros(1, Di, device="cuda"), None, e, e, 0, 1, Di, 0, layout,
                          k8, ks, None)
    assert capi.dsa_device_error()[0] == capi.DSA_OK


def test_appended_keys_score_like_the_definition():
    """Keys appended through the library, then scored by the library's indexer, match the
    oracle's scores of the oracle-appended cache (bit-exact codes make this the indexer's
    own parity on freshly written rows)."""
    B, Di, Hi, L = 1, 128, 64, 256
    k, _ = make_tokens(11, L, Di, 8)
    seq = np.zeros(L, np.int32)
    pos = np.arange(L, dtype=np.int32)
    seq_start = np.zeros(1, np.int32)
    k8_ref = np.zeros((L, Di), np.uint8)
    ks_ref = np.zeros(L, np.float32)
    oracle.cache_append(k, None, seq, pos, B, k8_ref, ks_ref, None, seq_start=seq_start)
    dev = "cuda"
    k8 = torch.zeros(L, Di, dtype=torch.uint8, device=dev)
    ks = torch.zeros(L, dtype=torch.float32, device=dev)
    ss = torch.from_numpy(seq_start).to(dev)
    layout = capi.make_layout(L, seq_start=ss)
    capi.dsa_cache_append(k.to(dev), None, torch.from_numpy(seq).to(dev),
                          torch.from_numpy(pos).to(dev), L, B, Di, 0, layout, k8, ks, None)
    assert np.array_equal(k8.cpu().numpy(), k8_ref)
    g = torch.Generator().manual_seed(12)
    q8 = torch.randn(1, Hi, Di, generator=g).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    q_scale = torch.ones(1)
    w = torch.randn(1, Hi, generator=g) / 8
    q_pos = torch.tensor([L - 1], dtype=torch.int32)
    scores = torch.full((1, L), float("nan"), device=dev)
    capi.dsa_indexer_scores(q8.to(dev), q_scale.to(dev), w.to(dev), k8, ks, layout,
                            q_pos.to(dev), B, 1, Hi, Di, L, scores)
    torch.cuda.synchronize()

    class Sub:  # the oracle's case fields for this one-row workload
        pass
    sub = Sub()
    sub.q8, sub.q_scale, sub.w, sub.q_pos = q8, q_scale, w, q_pos
    sub.k8, sub.k_scale = torch.from_numpy(k8_ref), torch.from_numpy(ks_ref)
    sub.seq_start, sub.block_table, sub.page_size, sub.pages_per_seq = torch.from_numpy(seq_start), None, 0, 0
    sub.B, sub.T, sub.Hi, sub.Di, sub.Lmax, sub.lengths = B, 1, Hi, Di, L, [L]
    check_case_scores(scores, sub)



def test_codes_round_the_exact_quotient_once():
    """Keys planted so that the fp32 quotient x / scale sits exactly on an e4m3 midpoint
    while the exact quotient lies on the other neighbour's side: the codes must be those
    of the exact quotient rounded once (the oracle's reading), bit for bit."""
    from planted import double_rounding_keys
    Di, n = 128, 8
    k = torch.from_numpy(double_rounding_keys(n, Di, seed=21))
    seq = np.zeros(n, np.int32)
    pos = np.arange(n, dtype=np.int32)
    skipped, st, _ = run_both(k, None, seq, pos, 1, n, Di, 0, seq_start=np.zeros(1, np.int32))
    assert skipped == 0 and st == capi.DSA_OK
