"""Shared comparison rules for the GPU-vs-oracle parity tests.

Tolerances (restating the acceptance bars, with the readings taken where they are open):
  * integer-valued workload: indexer scores and top-k indices bit-exact;
  * indexer scores elsewhere: |gpu - ref| <= 1e-3 * max(|ref|, 1e-2 * rms(row)).  The floor
    reads "1e-3 relative" for scores near zero, where a relative error is undefined; it
    still sits an order of magnitude above the fp32 round-off of the kernel's sums;
  * top-k sets equal, except tokens whose oracle score lies within 1e-3 relative of the
    oracle's k-th score;
  * attention outputs, against the oracle fed the GPU's own index set: max-abs <= 1e-2 and
    relative Frobenius error <= 5e-3; lse within 2.5e-3 (probabilities enter the second
    product as bf16, a relative error of at most 2^-9 on their sum);
  * integer-valued workload outputs: |gpu - ref| <= 0.5 ulp_bf16(ref) + 2^-8 * max_j
    |v_j - ref| (bf16 probabilities perturb the convex weights by at most 2^-9 each).
"""
import numpy as np
import torch

import oracle
from sparse_attention_29_b300 import inputs

SCORE_RTOL = 1e-3
SCORE_FLOOR = 1e-2
TOPK_RTOL = 1e-3
OUT_MAX_ABS = 1e-2
OUT_REL_FRO = 5e-3
LSE_ABS = 2.5e-3


def cpu(t):
    return t.detach().cpu()


def visible_mask(q_pos, Lmax):
    s = np.arange(Lmax)[None, :]
    return s <= np.asarray(q_pos)[:, None]


def check_scores(gpu_scores, ref, q_pos):
    g = cpu(gpu_scores).double().numpy()
    vis = visible_mask(cpu(q_pos).numpy(), ref.shape[1])
    worst = 0.0
    for t in range(ref.shape[0]):
        m = vis[t]
        r, x = ref[t, m], g[t, m]
        rms = np.sqrt(np.mean(r * r)) if r.size else 0.0
        tol = SCORE_RTOL * np.maximum(np.abs(r), SCORE_FLOOR * rms)
        err = np.abs(x - r)
        bad = np.nonzero(err > tol)[0]
        assert bad.size == 0, (f"row {t}: {bad.size} scores off, first at s={bad[0]}: "
                               f"gpu {x[bad[0]]!r} oracle {r[bad[0]]!r}")
        if r.size:
            worst = max(worst, float(np.max(err / np.maximum(tol, 1e-300))))
    return worst


def check_topk_sets(gpu_idx, ref_scores, q_pos, k):
    """GPU index rows against the oracle's scores (tolerant at the threshold)."""
    gi = cpu(gpu_idx).numpy()
    qp = cpu(q_pos).numpy()
    ref_idx = oracle.topk(ref_scores, qp, k)
    n_diff = 0
    for t in range(gi.shape[0]):
        n = int(qp[t]) + 1
        got = gi[t]
        # well-formed: ascending valid indices then -1 padding, nothing past the position
        valid = got[got >= 0]
        assert np.all(got[len(valid):] == -1), f"row {t}: padding not at the end"
        assert np.all(np.diff(valid) > 0), f"row {t}: indices not ascending/unique"
        assert valid.size == min(n, k) and (valid.size == 0 or valid[-1] < n)
        want = ref_idx[t][ref_idx[t] >= 0]
        if n <= k:
            assert np.array_equal(valid, np.arange(n))
            continue
        a, b = set(valid.tolist()), set(want.tolist())
        diff = a ^ b
        if diff:
            row = ref_scores[t, :n]
            kth = np.sort(row)[-k]
            for s in diff:
                assert abs(row[s] - kth) <= TOPK_RTOL * abs(kth), (
                    f"row {t}: token {s} (score {row[s]}) differs; k-th score {kth}")
            n_diff += len(diff)
    return n_diff


def check_mla(gpu_out, gpu_lse, ref_out, ref_lse):
    g = cpu(gpu_out).double().numpy()
    r = ref_out
    err = np.abs(g - r)
    max_abs = float(err.max()) if err.size else 0.0
    fro = float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-300))
    assert max_abs <= OUT_MAX_ABS, f"max-abs {max_abs}"
    assert fro <= OUT_REL_FRO, f"relative Frobenius {fro}"
    if gpu_lse is not None:
        gl = cpu(gpu_lse).double().numpy()
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(gl), fin)
        dl = float(np.max(np.abs(gl[fin] - ref_lse[fin]))) if fin.any() else 0.0
        assert dl <= LSE_ABS, f"lse off by {dl}"
    return max_abs, fro


def bf16_ulp(x):
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return 2.0 ** (e - 7)


def check_mla_integer(gpu_out, case, idx, ref_out, layer=0):
    """Bound from the arithmetic for exactly representable inputs (see module doc)."""
    g = cpu(gpu_out).double().numpy()
    kv = cpu(case.kv[layer]).double().numpy()
    ix = cpu(idx).numpy()
    rows, H, d = ref_out.shape
    for t in range(rows):
        b = t // case.T
        sel = ix[t][ix[t] >= 0]
        if case.block_table is None:
            phys = int(case.seq_start[b]) + sel
        else:
            bt = cpu(case.block_table).numpy()
            phys = bt[b, sel // case.page_size] * case.page_size + sel % case.page_size
        V = kv[phys, :d]                                    # [n, d]
        for h in range(H):
            o = ref_out[t, h]
            spread = np.max(np.abs(V - o[None, :]), axis=0)
            tol = 0.5 * bf16_ulp(o) + 2.0 ** -8 * spread + 1e-12
            err = np.abs(g[t, h] - o)
            assert np.all(err <= tol), (t, h, float(np.max(err - tol)))


def subcase(case, seqs=None, rows_in_seq=None):
    """A CPU case restricted to some sequences and/or some rows of each sequence (views of
    the same caches), for oracle runs on sampled outputs."""
    seqs = list(range(case.B)) if seqs is None else list(seqs)
    rows_in_seq = list(range(case.T)) if rows_in_seq is None else list(rows_in_seq)
    rows = [b * case.T + i for b in seqs for i in rows_in_seq]
    sub = inputs.Case(name=case.name + "-sub", kind=case.kind, seed=case.seed, B=len(seqs),
                      T=len(rows_in_seq), lengths=[case.lengths[b] for b in seqs], Hi=case.Hi,
                      Di=case.Di, H=case.H, d=case.d, r=case.r, k=case.k,
                      softmax_scale=case.softmax_scale, layers=case.layers,
                      page_size=case.page_size)
    sub.q8 = case.q8[rows]
    sub.q_scale = case.q_scale[rows]
    sub.w = case.w[rows]
    sub.q_pos = case.q_pos[rows]
    sub.q = [q[rows] for q in case.q]
    sub.k8, sub.k_scale, sub.kv = case.k8, case.k_scale, case.kv
    sub.seq_start = None if case.seq_start is None else case.seq_start[seqs]
    sub.block_table = None if case.block_table is None else case.block_table[seqs]
    return sub, rows
