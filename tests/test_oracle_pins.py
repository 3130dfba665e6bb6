"""Pins of the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each check is chosen so that a plausible slip in the oracle (a dropped ReLU or weight,
a wrong index, a transposed operand, a missing scale, a wrong tie-break or causal bound,
a softmax without its shift) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

import oracle
from sparse_attention_29_b300 import inputs


# ---- number formats -------------------------------------------------------------------

def test_e4m3_decode_matches_library_for_all_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for code in range(256):
        got = oracle.e4m3_to_double(code)
        want = ref[code].item()
        if math.isnan(want):
            assert math.isnan(got), code
        else:
            assert got == want, (code, got, want)


def test_bf16_decode_matches_library():
    g = torch.Generator().manual_seed(11)
    bits = torch.randint(-32768, 32767, (4096,), generator=g, dtype=torch.int16)
    vals = bits.view(torch.bfloat16).to(torch.float64)
    for b, v in zip(bits.tolist(), vals.tolist()):
        got = oracle.bf16_to_double(b)
        assert (math.isnan(got) and math.isnan(v)) or got == v


# ---- helpers ----------------------------------------------------------------------------

def _manual_case(q_heads, w, keys, q_pos, q_scale=1.0, k_scale=None, k=2):
    """One sequence, one query row; small integer values stored as e4m3 codes."""
    q = torch.tensor([q_heads], dtype=torch.float32)            # [1, Hi, Di]
    kk = torch.tensor(keys, dtype=torch.float32)                # [L, Di]
    L, Di = kk.shape
    case = inputs.Case(name="manual", kind="int", seed=0, B=1, T=1, lengths=[L],
                       Hi=q.shape[1], Di=Di, H=1, d=1, r=0, k=k, softmax_scale=1.0,
                       layers=1, page_size=0)
    case.q8 = q.to(torch.float8_e4m3fn).view(torch.uint8)
    case.k8 = kk.to(torch.float8_e4m3fn).view(torch.uint8)
    case.q_scale = torch.tensor([q_scale], dtype=torch.float32)
    case.k_scale = (torch.ones(L) if k_scale is None else torch.tensor(k_scale)).float()
    case.w = torch.tensor([w], dtype=torch.float32)
    case.q_pos = torch.tensor([q_pos], dtype=torch.int32)
    case.seq_start = torch.tensor([0], dtype=torch.int32)
    return case


def _hand():
    from conftest import read_golden
    g = read_golden("indexer_hand_example.txt")
    keys = [g[f"k{i}"] for i in range(5)]
    return g, keys


# ---- 1. lightning indexer ---------------------------------------------------------------

def test_indexer_hand_worked_example():
    g, keys = _hand()
    case = _manual_case([g["q_head0"], g["q_head1"]], g["w"], keys, int(g["q_pos"]))
    s = oracle.indexer_scores(case)[0]
    assert list(s[:4]) == g["scores"]
    assert s[4] == -np.inf          # causal: key 4 is after position 3


def test_indexer_scales_factor_out():
    g, keys = _hand()
    ks = [1.0, 1.0, 4.0, 1.0, 1.0]
    case = _manual_case([g["q_head0"], g["q_head1"]], g["w"], keys, int(g["q_pos"]),
                        q_scale=0.5, k_scale=ks)
    s = oracle.indexer_scores(case)[0]
    assert s[2] == g["scaled_score_k2"]
    assert list(s[[0, 1, 3]]) == [0.5 * x for x in (1.0, 0.5, 6.0)]


def test_indexer_single_head_is_relu_of_library_dot():
    c = inputs.make_case(kind="normal", seed=21, lengths=[300], Hi=1, Di=128, H=4, d=64, r=16)
    c.w = torch.ones_like(c.w)
    s = oracle.indexer_scores(c)[0]
    q = c.q8.view(torch.float8_e4m3fn).double()[0, 0] * c.q_scale.double()[0]
    k = c.k8.view(torch.float8_e4m3fn).double() * c.k_scale.double()[:, None]
    want = np.maximum(k.numpy() @ q.numpy(), 0.0)
    np.testing.assert_allclose(s, want, rtol=1e-13, atol=1e-300)


def test_indexer_linear_in_weights_and_head_order_free():
    c = inputs.make_case(kind="normal", seed=22, lengths=[257, 140], Hi=8, Di=32, H=4, d=64,
                         r=16)
    base = oracle.indexer_scores(c)
    w0 = c.w.clone()
    c.w = 2.0 * w0
    np.testing.assert_array_equal(oracle.indexer_scores(c), 2.0 * base)
    perm = torch.randperm(8, generator=torch.Generator().manual_seed(3))
    c.w = w0[:, perm].contiguous()
    q8 = c.q8
    c.q8 = q8[:, perm].contiguous()
    np.testing.assert_allclose(oracle.indexer_scores(c), base, rtol=1e-12)


def test_indexer_causal_ignores_future_keys():
    c = inputs.make_case(kind="normal", seed=23, lengths=[200], T=3, Hi=4, Di=32, H=4,
                         d=64, r=16)
    s0 = oracle.indexer_scores(c)
    c.k8[198:] = 0x38            # 1.0 in e4m3 on tokens 198, 199 (future of rows 0/1)
    s1 = oracle.indexer_scores(c)
    assert np.array_equal(s0[0], s1[0])          # row 0 sits at position 197
    assert not np.array_equal(s0[2], s1[2])      # row 2 sees token 199
    assert np.all(np.isinf(s0[0, 198:]))


def test_indexer_paged_equals_contiguous():
    c = inputs.make_case(kind="normal", seed=24, lengths=[300, 129, 64], T=2, Hi=4, Di=32,
                         H=4, d=64, r=16, page_size=64)
    u = inputs.unpage(c)
    np.testing.assert_array_equal(oracle.indexer_scores(c), oracle.indexer_scores(u))


# ---- 2. top-k -------------------------------------------------------------------------

def _brute_topk(row, n, k):
    order = sorted(range(n), key=lambda s: (-row[s], s))
    sel = sorted(order[:k]) if n > k else list(range(n))
    return sel + [-1] * (k - len(sel))


def test_topk_hand_worked_example():
    g, _ = _hand()
    scores = np.array([g["scores"] + [-np.inf]])
    qp = np.array([3], dtype=np.int32)
    for kk in (2, 3, 4, 5):
        want = g[f"top{kk}"]
        want = [int(x) for x in (want if isinstance(want, list) else [want])]
        assert oracle.topk(scores, qp, kk)[0].tolist() == want


@pytest.mark.parametrize("seed", range(6))
def test_topk_matches_full_sort_with_ties(seed):
    rng = np.random.default_rng(seed)
    rows, Lmax, k = 9, 70, 16
    # few distinct values so that ties are everywhere
    scores = rng.integers(-3, 4, size=(rows, Lmax)).astype(np.float32) * 0.25
    q_pos = rng.integers(0, Lmax, size=rows).astype(np.int32)
    q_pos[0], q_pos[1] = k - 1, k          # the dense edge and one past it
    got = oracle.topk(scores, q_pos, k)
    for t in range(rows):
        assert got[t].tolist() == _brute_topk(scores[t].tolist(), q_pos[t] + 1, k)


def test_topk_all_equal_takes_lowest_indices():
    scores = np.full((1, 100), 1.5)
    assert oracle.topk(scores, np.array([99], np.int32), 10)[0].tolist() == list(range(10))


def test_topk_dense_below_k_and_monotone():
    rng = np.random.default_rng(5)
    s = rng.standard_normal((1, 500))
    assert oracle.topk(s, np.array([40], np.int32), 64)[0].tolist() == \
        list(range(41)) + [-1] * 23
    sel = oracle.topk(s, np.array([499], np.int32), 64)[0]
    s2 = s.copy()
    s2[0, sel[5]] += 10.0                       # raising a selected score keeps it selected
    assert np.array_equal(oracle.topk(s2, np.array([499], np.int32), 64)[0], sel)
    unsel = sorted(set(range(500)) - set(sel.tolist()))[0]
    s2[0, unsel] = s.max() + 1.0                # a new maximum enters the set
    assert unsel in oracle.topk(s2, np.array([499], np.int32), 64)[0]


# ---- 3. sparse MLA --------------------------------------------------------------------

def _mla_case(seed, lengths, T=1, H=4, d=64, r=16, kind="normal", page_size=0, layers=1):
    return inputs.make_case(kind=kind, seed=seed, lengths=lengths, T=T, Hi=4, Di=32, H=H,
                            d=d, r=r, k=max(lengths), softmax_scale=0.125,
                            page_size=page_size, layers=layers)


def test_sparse_with_all_tokens_equals_dense():
    c = _mla_case(31, [90, 37], T=2)
    rows = c.rows
    K = 96
    idx = np.full((rows, K), -1, np.int32)
    for t in range(rows):
        n = int(c.q_pos[t]) + 1
        idx[t, :n] = np.arange(n)
    o_s, l_s = oracle.sparse_mla(c, idx)
    o_d, l_d = oracle.dense_mla(c)
    np.testing.assert_allclose(o_s, o_d, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(l_s, l_d, rtol=1e-13)


def test_single_token_gives_its_value_row():
    c = _mla_case(32, [50])
    idx = np.full((1, 8), -1, np.int32)
    idx[0, 3] = 17
    out, lse = oracle.sparse_mla(c, idx)
    q = c.q[0].double()[0]                        # [H, D]
    row = c.kv[0].double()[17]                    # [D]
    np.testing.assert_array_equal(out[0], np.broadcast_to(row[: c.d].numpy(), (c.H, c.d)))
    np.testing.assert_allclose(lse[0], 0.125 * (q @ row).numpy(), rtol=1e-14)


def test_zero_query_gives_mean_of_values():
    c = _mla_case(33, [64])
    c.q[0] = torch.zeros_like(c.q[0])
    sel = np.array([[3, 9, 10, 40, 63, -1, -1, 1]], np.int32)
    out, lse = oracle.sparse_mla(c, sel)
    v = c.kv[0].double()[[3, 9, 10, 40, 63, 1], : c.d].numpy()
    np.testing.assert_allclose(out[0], np.broadcast_to(v.mean(0), (c.H, c.d)), rtol=1e-13)
    np.testing.assert_allclose(lse[0], math.log(6.0), rtol=1e-15)


def test_two_token_closed_form():
    # logits 0 and 1: weights 1/(1+e) and e/(1+e)
    c = _mla_case(34, [4], H=1, d=64, r=0)
    D = c.D
    q = torch.zeros((1, 1, D))
    q[0, 0, 0] = 1.0
    kv = torch.zeros((4, D))
    kv[0, 1:] = 2.0
    kv[1, 0] = 8.0                               # logit = 0.125 * 8 = 1
    kv[1, 1:] = -3.0
    c.q[0] = q.to(torch.bfloat16)
    c.kv[0] = kv.to(torch.bfloat16)
    out, lse = oracle.sparse_mla(c, np.array([[0, 1]], np.int32))
    a, b = 1.0 / (1.0 + math.e), math.e / (1.0 + math.e)
    want = a * kv[0].double().numpy() + b * kv[1].double().numpy()
    np.testing.assert_allclose(out[0, 0], want, rtol=1e-15, atol=1e-15)
    assert abs(lse[0, 0] - math.log(1.0 + math.e)) < 1e-15


def test_index_order_and_padding_do_not_matter():
    c = _mla_case(35, [300])
    rng = np.random.default_rng(1)
    sel = rng.choice(300, size=40, replace=False).astype(np.int32)
    a = np.full((1, 64), -1, np.int32)
    a[0, :40] = sel
    b = np.full((1, 64), -1, np.int32)
    b[0, rng.permutation(64)[:40]] = sel[::-1]
    oa, la = oracle.sparse_mla(c, a)
    ob, lb = oracle.sparse_mla(c, b)
    np.testing.assert_allclose(oa, ob, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(la, lb, rtol=1e-14)


def test_sparse_mla_against_library_softmax():
    c = _mla_case(36, [120], H=3)
    sel = np.random.default_rng(2).choice(120, size=50, replace=False).astype(np.int32)
    out, lse = oracle.sparse_mla(c, sel[None, :])
    Q = c.q[0].double()[0].numpy()                     # [H, D]
    C = c.kv[0].double()[sel].numpy()                  # [50, D]
    S = 0.125 * Q @ C.T
    np.testing.assert_allclose(out[0], softmax(S, axis=1) @ C[:, : c.d], rtol=1e-12,
                               atol=1e-13)
    np.testing.assert_allclose(lse[0], logsumexp(S, axis=1), rtol=1e-13)


def test_sparse_mla_rejects_future_index():
    c = _mla_case(37, [40], T=2)
    idx = np.array([[0, 39], [0, 39]], np.int32)       # row 0 sits at position 38
    with pytest.raises(ValueError):
        oracle.sparse_mla(c, idx)


def test_sparse_mla_paged_equals_contiguous():
    c = _mla_case(38, [200, 70], T=1, page_size=64)
    u = inputs.unpage(c)
    rows = [np.r_[np.arange(0, 200, 3)], np.arange(70)]
    K = max(len(x) for x in rows)
    idx = np.full((2, K), -1, np.int32)
    for t, x in enumerate(rows):
        idx[t, : len(x)] = x
    o1, l1 = oracle.sparse_mla(c, idx)
    o2, l2 = oracle.sparse_mla(u, idx)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ---- 4. IndexShare ----------------------------------------------------------------------

def test_indexshare_identical_layers_identical_outputs():
    c = inputs.make_case(kind="normal", seed=41, lengths=[700, 300], Hi=4, Di=32, H=4, d=64,
                         r=16, k=128, softmax_scale=0.125, layers=4)
    for g in range(1, 4):
        c.q[g] = c.q[0].clone()
        c.kv[g] = c.kv[0].clone()
    idx, per_layer = oracle.indexshare_group(c)
    for out, lse in per_layer[1:]:
        np.testing.assert_array_equal(out, per_layer[0][0])
        np.testing.assert_array_equal(lse, per_layer[0][1])
    # the shared index set is layer 0's own top-k, and row 1 (context 300 > 128) is sparse
    assert np.array_equal(idx, oracle.topk(oracle.indexer_scores(c), c.q_pos, 128))
    assert (idx[1] >= 0).all()


def test_indexshare_layers_differ_only_through_their_caches():
    c = inputs.make_case(kind="normal", seed=42, lengths=[500], Hi=4, Di=32, H=4, d=64,
                         r=16, k=64, softmax_scale=0.125, layers=4)
    idx, per_layer = oracle.indexshare_group(c)
    for g in range(4):
        out, lse = oracle.sparse_mla(c, idx, layer=g)
        np.testing.assert_array_equal(out, per_layer[g][0])
    assert not np.array_equal(per_layer[0][0], per_layer[1][0])


# ---- accounting -------------------------------------------------------------------------

def test_accounting_reproduces_printed_numbers(golden):
    g = golden("accounting.txt")
    ai = oracle.mqa_decode_intensity(int(g["heads_glm5"]), 512, 64, 2)
    assert math.floor(ai * 10) / 10 == g["intensity_H64_d512_r64_b2"]
    assert oracle.mqa_decode_intensity(int(g["heads_dsv32"]), 512, 64, 2) == 2 * ai
    ridge = g["h800_tflops"] / g["h800_tbs"]
    assert round(ridge, 1) == g["h800_ridge"]
    h = oracle.heads_at_ridge(ridge, 512, 64, 2)
    # "H about 128": the nearest power of two to the solved head count
    assert 2 ** round(math.log2(h)) == g["heads_at_h800_ridge_approx"]
    before = oracle.sdpa_score_flops(int(g["heads_dsv32"]), int(g["head_dim_before"]))
    after = oracle.sdpa_score_flops(int(g["heads_glm5"]), int(g["head_dim_after"]))
    assert round(100 * (1 - after / before)) == g["flop_cut_percent"]
    assert oracle.indexshare_indexer_cut(int(g["indexshare_group"])) * 100 == \
        g["indexshare_cut_percent"]
    assert g["top_k"] == 2048


def test_decode_bytes_per_query_of_the_32k_workload():
    # the per-query algorithmic bytes the decode benchmark counts (B=32, L=32768)
    L, k, Hi, Di, H, d, r = 32768, 2048, 64, 128, 64, 512, 64
    indexer = L * Di + L * 4 + Hi * Di + 4 + Hi * 4          # keys, key scales, q8, sq, w
    kv = k * oracle.mqa_decode_bytes_per_token(d, r, 2)
    assert indexer == 4_333_828
    assert kv == 2_359_296
    assert oracle.indexer_flops(Hi, Di, L) == 536_870_912


# ---- cache append (the step that feeds the path) -------------------------------------------

def _finite_codes():
    return [c for c in range(256) if c not in (0x7F, 0xFF)]


def test_e4m3_encode_inverts_decode_on_every_code():
    for c in _finite_codes():
        assert oracle.e4m3_encode(oracle.e4m3_to_double(c)) == c, hex(c)


def test_e4m3_encode_ties_go_to_even_and_neighbours_to_nearest():
    for c in range(0, 0x7E):  # adjacent non-negative finite codes c, c + 1
        lo, hi = oracle.e4m3_to_double(c), oracle.e4m3_to_double(c + 1)
        mid = (lo + hi) / 2  # exact in fp32: e4m3 values carry 4 significant bits
        assert float(np.float32(mid)) == mid
        assert oracle.e4m3_encode(mid) == (c if c % 2 == 0 else c + 1), hex(c)
        assert oracle.e4m3_encode(-mid) == 0x80 | (c if c % 2 == 0 else c + 1)
        below = float(np.nextafter(np.float32(mid), np.float32(0)))
        above = float(np.nextafter(np.float32(mid), np.float32(1e9)))
        assert oracle.e4m3_encode(below) == c and oracle.e4m3_encode(above) == c + 1, hex(c)


def test_e4m3_encode_saturates_at_448():
    for x, code in ((448.0, 0x7E), (460.0, 0x7E), (464.0, 0x7E), (1e30, 0x7E), (-1e30, 0xFE),
                    (-449.0, 0xFE), (0.0, 0x00), (-0.0, 0x80)):
        assert oracle.e4m3_encode(x) == code, x


def test_e4m3_encode_matches_library_cast():
    g = torch.Generator().manual_seed(21)
    x = torch.cat([torch.randn(20000, generator=g) * s for s in (1e-3, 0.05, 1.0, 30.0, 300.0)])
    ref = x.clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    for v, c in zip(x.tolist(), ref.tolist()):
        assert oracle.e4m3_encode(v) == c, v


def _append_inputs(seed, n, Di, D):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(n, Di, generator=g)
    k[0] *= 1e-4                          # small keys: subnormal codes
    k[1] = 0.0                            # an all-zero key: scale from the 1e-30 floor
    c = torch.randint(-32768, 32767, (n, D), generator=g, dtype=torch.int16).view(torch.uint16)
    return k, c


def test_cache_append_scale_and_codes_follow_the_definition():
    n, Di, D, B = 6, 128, 64, 2
    k, c = _append_inputs(3, n, Di, D)
    seq = np.array([0, 0, 1, 1, 0, 1], np.int32)
    pos = np.array([0, 1, 0, 1, 2, 2], np.int32)
    seq_start = np.array([0, 10], np.int32)
    k8 = np.zeros((20, Di), np.uint8)
    ks = np.zeros(20, np.float32)
    kv = np.zeros((20, D), np.uint16)
    assert oracle.cache_append(k, c, seq, pos, B, k8, ks, kv, seq_start=seq_start) == 0
    for i in range(n):
        r = seq_start[seq[i]] + pos[i]
        amax = np.float32(np.abs(k[i].numpy()).max())
        scale = np.float32(max(amax, np.float32(1e-30))) / np.float32(448)
        assert ks[r] == scale
        if amax > 0:  # the largest key maps to +-448 exactly
            j = int(np.abs(k[i].numpy()).argmax())
            assert k8[r, j] & 0x7F == 0x7E
        dq = np.array([oracle.e4m3_to_double(int(b)) for b in k8[r]]) * float(scale)
        step = np.abs(k[i].numpy().astype(np.float64)) * 2.0 ** -4 + 2.0 ** -9 * float(scale)
        assert np.all(np.abs(dq - k[i].numpy()) <= step)  # within half an e4m3 step
        assert np.array_equal(kv[r], c[i].numpy())
    untouched = [r for r in range(20) if r not in set((seq_start[seq] + pos).tolist())]
    assert not k8[untouched].any() and not ks[untouched].any() and not kv[untouched].any()


def test_cache_append_paged_equals_contiguous_and_skips_bad_tokens():
    n, Di, D, B, ps, pps = 9, 64, 16, 2, 4, 3
    k, c = _append_inputs(4, n, Di, D)
    seq = np.array([0, 0, 0, 0, 0, 1, 1, 1, 1], np.int32)
    pos = np.array([0, 3, 4, 7, 11, 0, 5, 6, 12], np.int32)  # last: past the block table
    bt = np.array([[5, 1, 3], [0, 4, 2]], np.int32)
    num = 6 * ps
    k8p, ksp, kvp = np.zeros((num, Di), np.uint8), np.zeros(num, np.float32), np.zeros((num, D), np.uint16)
    assert oracle.cache_append(k, c, seq, pos, B, k8p, ksp, kvp, block_table=bt, page_size=ps) == 1
    seq_start = np.array([0, 12], np.int32)
    k8c, ksc, kvc = np.zeros((24, Di), np.uint8), np.zeros(24, np.float32), np.zeros((24, D), np.uint16)
    assert oracle.cache_append(k[:8], c[:8], seq[:8], pos[:8], B, k8c, ksc, kvc, seq_start=seq_start) == 0
    for b in range(B):
        for s in range(12):
            rp = bt[b, s // ps] * ps + s % ps
            rc = seq_start[b] + s
            assert np.array_equal(k8p[rp], k8c[rc]) and ksp[rp] == ksc[rc]
            assert np.array_equal(kvp[rp], kvc[rc])


def test_cache_append_codes_round_the_exact_quotient_once():
    """Every code is the e4m3 value nearest the exact rational x / scale (brute force over
    all codes), including keys planted where a second rounding of the fp32 quotient
    would pick the other neighbour."""
    from fractions import Fraction
    from planted import double_rounding_keys, nearest_e4m3_code
    n, Di = 6, 128
    k = np.concatenate([double_rounding_keys(n, Di, seed=3),
                        (np.random.default_rng(4).standard_normal((2, Di)) * 3).astype(np.float32)])
    n = k.shape[0]
    seq = np.zeros(n, np.int32)
    pos = np.arange(n, dtype=np.int32)
    k8 = np.zeros((n, Di), np.uint8)
    ks = np.zeros(n, np.float32)
    assert oracle.cache_append(k, None, seq, pos, 1, k8, ks, None,
                               seq_start=np.zeros(1, np.int32)) == 0
    differs = 0
    for i in range(n):
        scale = Fraction(float(ks[i]))
        for c in range(Di):
            want = nearest_e4m3_code(Fraction(float(k[i, c])) / scale)
            assert k8[i, c] == want, (i, c)
            twice = oracle.e4m3_encode(np.float32(k[i, c]) / ks[i])
            differs += int(twice != want)
    assert differs >= 3 * 6  # the planted keys do separate the two readings


def test_hisparse_lru_hand_worked_example(golden):
    g = golden("hisparse_lru.txt")
    st = oracle.HiSparseState(int(g["Lmax"]), int(g["C"]))
    hits = []
    for s in (1, 2, 3):
        row = np.atleast_1d(np.asarray(g[f"step{s}"], dtype=np.int32))
        h, loaded = st.step(row, s)
        hits.append(h)
        want = np.atleast_1d(np.asarray(g[f"loaded{s}"], dtype=np.int64)).reshape(-1, 2)
        assert loaded == [tuple(x) for x in want.tolist()], s
    assert hits == [int(x) for x in g["hits"]]
    assert st.res.tolist() == [int(x) for x in g["final_residency"]]
    assert st.slot_tok.tolist() == [int(x) for x in g["final_slot_token"]]
    assert st.slot_use.tolist() == [int(x) for x in g["final_slot_use"]]


def test_hisparse_policy_invariants():
    """Over random steps: every selected token is resident afterwards, residency and slot
    tokens stay inverse maps, the set of evicted tokens were never used later than any
    non-selected resident token that stayed, and the hit count is the overlap with the
    tokens resident before the step."""
    rng = np.random.default_rng(5)
    Lmax, C, k = 300, 40, 25
    st = oracle.HiSparseState(Lmax, C)
    for step in range(1, 30):
        sel = np.sort(rng.choice(Lmax if step % 3 else 60, size=k, replace=False)).astype(np.int32)
        before = {int(t): int(st.res[t]) for t in np.nonzero(st.res >= 0)[0]}
        use_before = st.slot_use.copy()
        hits, loaded = st.step(sel, step)
        assert hits == sum(int(t) in before for t in sel)
        assert all(st.res[t] >= 0 for t in sel)
        for s, t in enumerate(st.slot_tok):
            if t >= 0:
                assert st.res[t] == s
        assert int((st.res >= 0).sum()) == int((st.slot_tok >= 0).sum()) <= C
        victims = {v for _, v in loaded}
        kept = [s for s in range(C) if s not in victims and use_before[s] < step
                and st.slot_use[s] < step]
        if victims and kept:
            assert max(use_before[v] for v in victims) <= min(use_before[s] for s in kept)


def _mha_inputs(seed, H, d, r, dn, vd, lengths, T, k):
    """Integer-valued weights and queries: with w_uk and q_nope in {-1, 0, 1} the absorbed
    query w_uk[h]^T q_nope is an integer of magnitude <= dn, exact in bf16."""
    case = inputs.make_case(kind="int", seed=seed, lengths=lengths, T=T, Hi=4, Di=32, H=H, d=d,
                            r=r, k=k, softmax_scale=1.0 / 8.0)
    g = torch.Generator().manual_seed(seed)
    w_uk = torch.randint(-1, 2, (H, dn, d), generator=g).to(torch.bfloat16)
    w_uv = torch.randint(-2, 3, (H, vd, d), generator=g).to(torch.bfloat16)
    q_nope = torch.randint(-1, 2, (case.rows, H, dn), generator=g).float()
    q_rope = case.q[0][:, :, d:].float()
    q_mha = torch.cat([q_nope, q_rope], dim=2).to(torch.bfloat16)
    q_abs = torch.einsum("hie,thi->the", w_uk.float(), q_nope)
    assert torch.equal(q_abs.to(torch.bfloat16).float(), q_abs)  # exact in bf16
    case.q = [torch.cat([q_abs, q_rope], dim=2).to(torch.bfloat16)]
    return case, w_uk, w_uv, q_mha


def test_mha_mode_equals_absorbed_mqa_then_value_projection():
    """MLA's MHA and MQA modes compute one attention [GLM53 §Sparse MLA]: the MHA-mode oracle
    equals the (independently pinned) MQA oracle fed the absorbed query, followed by the
    value up-projection, to fp64 round-off -- for sparse index sets with -1 holes."""
    H, d, r, dn, vd, k = 3, 64, 16, 32, 48, 24
    case, w_uk, w_uv, q_mha = _mha_inputs(11, H, d, r, dn, vd, [50, 37], 3, k)
    rng = np.random.default_rng(3)
    idx = np.full((case.rows, k), -1, np.int32)
    for t in range(case.rows):
        n = int(case.q_pos[t]) + 1
        m = min(n, k - 3)
        idx[t, :m] = np.sort(rng.choice(n, size=m, replace=False))
    o_lat, lse_mqa = oracle.sparse_mla(case, idx)
    want = np.einsum("hve,the->thv", w_uv.double().numpy(), o_lat)
    got, lse_mha = oracle.sparse_mha(case, idx, w_uk, w_uv, q_mha)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-9 * np.abs(want).max())
    np.testing.assert_allclose(lse_mha, lse_mqa, rtol=1e-13, atol=1e-12)


def test_mha_mode_one_selected_token_gives_its_value():
    H, d, r, dn, vd, k = 2, 64, 16, 32, 32, 8
    case, w_uk, w_uv, q_mha = _mha_inputs(12, H, d, r, dn, vd, [20], 1, k)
    idx = np.full((1, k), -1, np.int32)
    idx[0, 3] = 7
    got, lse = oracle.sparse_mha(case, idx, w_uk, w_uv, q_mha)
    c = case.kv[0][int(case.seq_start[0]) + 7, :d].double().numpy()
    want = np.einsum("hve,e->hv", w_uv.double().numpy(), c)
    np.testing.assert_array_equal(got[0], want)
