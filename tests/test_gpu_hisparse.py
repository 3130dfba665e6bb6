"""GPU parity of the host-tier working set (dsa_hisparse_init / dsa_hisparse_fetch).

Over several decode steps with overlapping selections, the device's residency table, slot
tokens, last uses and hit/miss counts must equal the oracle's LRU simulation bit for bit;
every resident slot must hold its token's row of the host cache; and the sparse MLA read
through the working set (a block table of one-token pages) must equal, bit for bit, the
sparse MLA over the full device cache: moving rows between tiers changes nothing.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_29_b300 import build, capi, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    capi.load()
    oracle.build()
    assert torch.cuda.is_available()


def selections(lengths, k, steps, seed):
    """Per step a [B, k] index row: ascending tokens, about half of them repeated from the
    previous step, a few -1 entries at the end."""
    rng = np.random.default_rng(seed)
    out, prev = [], None
    for s in range(steps):
        rows = np.full((len(lengths), k), -1, np.int32)
        for b, L in enumerate(lengths):
            n = k - int(rng.integers(0, 8))
            if prev is None:
                sel = rng.choice(L, size=n, replace=False)
            else:
                old = prev[b][prev[b] >= 0]
                keep = rng.choice(old, size=min(len(old), n // 2), replace=False)
                rest = np.setdiff1d(np.arange(L), keep)
                sel = np.concatenate([keep, rng.choice(rest, size=n - len(keep), replace=False)])
            rows[b, :n] = np.sort(sel)
        out.append(rows)
        prev = rows
    return out


@pytest.mark.parametrize("lengths,C,k", [([6000, 4000, 5000], 1024, 512), ([3000], 2048, 2048)])
def test_working_set_matches_oracle_and_attention_is_unchanged(lengths, C, k):
    case = inputs.make_case(seed=81, lengths=lengths, T=1, k=k)
    B, D, Lmax = case.B, case.D, case.Lmax
    dev = "cuda"
    host_kv = case.kv[0].view(torch.int16).pin_memory()        # the full history, pinned
    host_start = case.seq_start.to(dev)
    full = case.to(dev)                                         # the same rows, all on device
    res = torch.empty((B, Lmax), dtype=torch.int32, device=dev)
    stok = torch.empty((B, C), dtype=torch.int32, device=dev)
    use = torch.empty((B, C), dtype=torch.int32, device=dev)    # uint32 bits
    pool = torch.zeros((B * C, D), dtype=torch.int16, device=dev)
    stats = torch.zeros((B, 2), dtype=torch.int32, device=dev)
    capi.dsa_hisparse_init(res, B, Lmax, stok, use, C)
    states = [oracle.HiSparseState(Lmax, C) for _ in range(B)]
    full_layout = capi.make_layout(full.n_phys, seq_start=full.seq_start)
    tier_layout = capi.make_layout(B * C, block_table=res, page_size=1)
    for step, rows in enumerate(selections(lengths, k, 6, seed=C), start=1):
        idx = torch.from_numpy(rows).to(dev)
        capi.dsa_hisparse_fetch(idx, B, k, step, host_kv, host_start, D, res, Lmax, stok, use, C,
                                pool, stats)
        torch.cuda.synchronize()
        st, code = capi.dsa_device_error()
        assert st == capi.DSA_OK, hex(code)
        r_dev, t_dev = res.cpu().numpy(), stok.cpu().numpy()
        u_dev = use.cpu().numpy().view(np.uint32)
        s_dev = stats.cpu().numpy()
        for b in range(B):
            hits, loaded = states[b].step(rows[b], step)
            want_res = np.where(states[b].res >= 0, states[b].res + b * C, -1)
            assert np.array_equal(r_dev[b], want_res), (step, b)
            assert np.array_equal(t_dev[b], states[b].slot_tok), (step, b)
            assert np.array_equal(u_dev[b], states[b].slot_use), (step, b)
            assert (s_dev[b, 0], s_dev[b, 1]) == (hits, len(loaded)), (step, b)
        # every resident slot holds its token's host row
        resident = np.nonzero(t_dev >= 0)
        host = case.kv[0].view(torch.int16)
        rows_host = torch.from_numpy(case.seq_start.numpy()[resident[0]] + t_dev[resident]).long()
        slots = torch.from_numpy(resident[0] * C + resident[1]).long()
        assert torch.equal(pool.cpu()[slots], host[rows_host])
        # attention through the working set equals attention over the full device cache
        outs = []
        for layout, kv in ((full_layout, full.kv[0]), (tier_layout, pool.view(torch.bfloat16))):
            o = torch.empty((B, case.H, case.d), dtype=torch.bfloat16, device=dev)
            l = torch.empty((B, case.H), dtype=torch.float32, device=dev)
            ws = capi.dsa_workspace_bytes(capi.DSA_OP_SPARSE_MLA, B, 1, case.H, case.d, k, 1)
            w = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)
            capi.dsa_sparse_mla_decode(full.q[0], kv, layout, idx, B, case.H, case.d, case.r, k,
                                       case.softmax_scale, o, l, w, ws)
            outs.append((o, l))
        torch.cuda.synchronize()
        assert capi.dsa_device_error()[0] == capi.DSA_OK
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1]), step


def test_layer_ahead_overlap_equals_sequential_and_full_cache():
    """An IndexShare group of 3 layers behind the host tier, 3 decode steps: with the
    fetches on a second stream (layer l + 1's fetch while layer l attends) every layer's
    output and log-sum-exp equal those of the one-stream schedule and of the sparse MLA
    over the full device cache, bit for bit."""
    from sparse_attention_29_b300.pipeline import HostTierGroup
    case = inputs.make_case(seed=85, lengths=[5000, 3000, 4200], T=1, layers=3, k=512)
    B, D, Lmax, k, L, C = case.B, case.D, case.Lmax, case.k, case.layers, 1024
    dev = "cuda"
    full = case.to(dev)
    host = [case.kv[g].view(torch.int16).pin_memory() for g in range(L)]
    host_start = case.seq_start.to(dev)
    full_layout = capi.make_layout(full.n_phys, seq_start=full.seq_start)
    ws = capi.dsa_workspace_bytes(capi.DSA_OP_SPARSE_MLA, B, 1, case.H, case.d, k, 1)
    w = torch.empty(max(ws, 16), dtype=torch.uint8, device=dev)

    def buffers():
        return ([torch.empty((B, case.H, case.d), dtype=torch.bfloat16, device=dev) for _ in range(L)],
                [torch.empty((B, case.H), dtype=torch.float32, device=dev) for _ in range(L)])

    sel = [torch.from_numpy(r).to(dev) for r in selections(case.lengths, k, 3, seed=9)]
    results = {}
    for overlap in (False, True):
        grp = HostTierGroup(host, host_start, B, Lmax, D, C)
        grp.reset()
        per_step = []
        for s, idx in enumerate(sel, start=1):
            out, lse = buffers()
            grp.step(idx, k, s, full.q, out, lse, case.H, case.d, case.r, case.softmax_scale,
                     w, ws, overlap=overlap)
            torch.cuda.synchronize()
            assert capi.dsa_device_error()[0] == capi.DSA_OK
            per_step.append(([o.clone() for o in out], [x.clone() for x in lse]))
        results[overlap] = per_step
    for s, idx in enumerate(sel):
        ref_out, ref_lse = buffers()
        for g in range(L):
            capi.dsa_sparse_mla_decode(full.q[g], full.kv[g], full_layout, idx, B, case.H, case.d,
                                       case.r, k, case.softmax_scale, ref_out[g], ref_lse[g], w, ws)
        torch.cuda.synchronize()
        for g in range(L):
            for ov in (False, True):
                assert torch.equal(results[ov][s][0][g], ref_out[g]), (s, g, ov)
                assert torch.equal(results[ov][s][1][g], ref_lse[g]), (s, g, ov)
