"""The seeded input generator: deterministic, well-formed, layouts consistent (CPU)."""
import numpy as np
import torch

from sparse_attention_29_b300 import inputs


def test_same_seed_same_bytes():
    a = inputs.make_case(seed=9, lengths=[130, 70], Hi=4, Di=32, H=4, d=64, r=16)
    b = inputs.make_case(seed=9, lengths=[130, 70], Hi=4, Di=32, H=4, d=64, r=16)
    for f in ("q8", "q_scale", "w", "k8", "k_scale", "q_pos", "seq_start"):
        assert torch.equal(getattr(a, f), getattr(b, f))
    assert torch.equal(a.kv[0].view(torch.int16), b.kv[0].view(torch.int16))


def test_fp8_codes_are_finite_and_scales_positive():
    c = inputs.make_case(kind="planted", seed=3, lengths=[2000], Hi=8, Di=128, H=4, d=64, r=16)
    for codes in (c.k8, c.q8):
        assert not ((codes & 0x7F) == 0x7F).any()       # no NaN code
    assert (c.k_scale > 0).all() and (c.q_scale > 0).all()
    # every row reaches the top of the e4m3 range (scale = amax / 448)
    amax = c.k8.view(torch.float8_e4m3fn).float().abs().amax(dim=1)
    assert (amax == 448.0).all()


def test_int_case_is_exact():
    c = inputs.preset("tiny_int")
    assert c.q8.view(torch.float8_e4m3fn).float().abs().max() <= 4
    assert set(c.w.unique().tolist()) <= {0.5, 1.0, 2.0}
    assert c.q_pos.tolist() == [508, 509, 510, 511]
    kv = c.kv[0].float()
    assert torch.equal(kv, kv.round()) and kv.abs().max() <= 4


def test_paged_layout_is_a_page_permutation():
    c = inputs.make_case(seed=4, lengths=[300, 129], page_size=64, Hi=4, Di=32, H=4, d=64,
                         r=16, layers=2)
    bt = c.block_table
    assert sorted(bt.flatten().tolist()) == list(range(bt.numel()))
    u = inputs.unpage(c)
    for b, L in enumerate(c.lengths):
        for s in (0, 63, 64, L - 1):
            p = int(bt[b, s // 64]) * 64 + s % 64
            assert torch.equal(c.k8[p], u.k8[int(u.seq_start[b]) + s])
            assert torch.equal(c.kv[1][p].view(torch.int16),
                               u.kv[1][int(u.seq_start[b]) + s].view(torch.int16))


def test_ragged_lengths_span_the_dense_threshold():
    L = inputs.ragged_lengths(16, 1024, 200000, 3)
    assert min(L) >= 1024 and max(L) <= 200000
    assert any(x <= 2048 for x in L) and any(x > 100000 for x in L)
