"""Shared comparison rules for the GPU-vs-oracle parity tests.

Tolerances (restating the acceptance bars, with the readings taken where they are open):
  * integer-valued workloads: indexer scores and top-k indices bit-exact;
  * indexer scores elsewhere: |gpu - ref| <= 1e-3 * max(|ref|, 1e-3 * rms(row)), the
    "1e-3 relative" bar with a floor for scores near zero -- except where the score is
    a near-cancellation of large terms, where no fp32 evaluation can meet a relative bar:
    there the bar is the textbook round-off bound of the fp32 sums themselves,
    (Di + Hi + 2) * 2^-23 * A, with A = sum_h |w_h| sum_c |q_hc k_c| (the oracle's
    `abs_terms`; Higham, Accuracy and Stability of Numerical Algorithms, eq. 3.5, with
    the unit 2^-23 so that truncating accumulation is covered too);
  * top-k sets equal, except tokens whose oracle score lies within 1e-3 relative of the
    oracle's k-th score;
  * attention outputs, against the oracle fed the GPU's own index set: max-abs <= 1e-2 and
    relative Frobenius error <= 5e-3; lse within 2.5e-3;
  * integer-valued workload outputs: within one bf16 ulp of the correctly rounded oracle
    value, plus the fp32 error of forming the weighted mean before that rounding,
    (2^-14 + 2 n 2^-23) * max_j |v_j| for n selected keys (softmax weights to a relative
    2^-16 from the hi/lo bf16 split, 2^-21 from the exponential, and fp32 accumulation
    of 2n products); lse within fp32 round-off, 2^-16 + 2^-20 |lse|.  Rows whose keys
    are split over a thread-block cluster exchange their unnormalised partial outputs
    in bf16 (relative 2^-8 each), which adds at most 2^-8 * max_j |v_j| (the merge is a
    convex combination of the partial means).
"""
import numpy as np
import torch

import oracle
from sparse_attention_29_b300 import inputs

SCORE_RTOL = 1e-3
SCORE_FLOOR = 1e-3
FP32_UNIT = 2.0 ** -23
TOPK_RTOL = 1e-3
OUT_MAX_ABS = 1e-2
OUT_REL_FRO = 5e-3
LSE_ABS = 2.5e-3


def cpu(t):
    return t.detach().cpu()


def visible_mask(q_pos, Lmax):
    s = np.arange(Lmax)[None, :]
    return s <= np.asarray(q_pos)[:, None]


def check_scores(gpu_scores, ref, q_pos, abs_terms=None, Hi=64, Di=128):
    """`ref` and `abs_terms` from oracle.indexer_scores(case, with_abs=True)."""
    g = cpu(gpu_scores).double().numpy()
    vis = visible_mask(cpu(q_pos).numpy(), ref.shape[1])
    worst = 0.0
    gamma = (Di + Hi + 2) * FP32_UNIT
    for t in range(ref.shape[0]):
        m = vis[t]
        r, x = ref[t, m], g[t, m]
        rms = np.sqrt(np.mean(r * r)) if r.size else 0.0
        tol = SCORE_RTOL * np.maximum(np.abs(r), SCORE_FLOOR * rms)
        if abs_terms is not None:
            tol = np.maximum(tol, gamma * abs_terms[t, m])
        err = np.abs(x - r)
        bad = np.nonzero(err > tol)[0]
        assert bad.size == 0, (f"row {t}: {bad.size} scores off, first at s={bad[0]}: "
                               f"gpu {x[bad[0]]!r} oracle {r[bad[0]]!r}")
        if r.size:
            worst = max(worst, float(np.max(err / np.maximum(tol, 1e-300))))
    return worst


def check_case_scores(gpu_scores, case):
    """GPU scores of every row of `case` against the oracle; returns the oracle scores."""
    ref, absum = oracle.indexer_scores(case, with_abs=True)
    check_scores(gpu_scores, ref, case.q_pos, absum, Hi=case.Hi, Di=case.Di)
    return ref


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


def bf16_round(x):
    """Round float64 values to the nearest bf16 value (8 significant bits, ties to even),
    directly from float64 (no intermediate fp32 rounding)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def bf16_ulp(x):
    """Spacing of bf16 values at |x| (2^(E-7) for |x| in [2^E, 2^(E+1)))."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.maximum(a, 2.0 ** -126))
    return np.ldexp(1.0, e - 8)


def check_mla_integer(gpu_out, gpu_lse, case, idx, ref_out, ref_lse, layer=0,
                      split_exchange=False):
    """Outputs within one bf16 ulp of the correctly rounded oracle value plus the bound on
    forming the weighted mean in fp32 (module doc); lse within fp32 round-off.
    split_exchange: the rows may be merged from bf16 partials (module doc)."""
    g = cpu(gpu_out).double().numpy()
    kv = cpu(case.kv[layer]).double().numpy()
    ix = cpu(idx).numpy()
    rows, H, d = ref_out.shape
    worst_ulps = 0.0
    for t in range(rows):
        b = t // case.T
        sel = ix[t][ix[t] >= 0]
        if case.block_table is None:
            phys = int(case.seq_start[b]) + sel
        else:
            bt = cpu(case.block_table).numpy()
            phys = bt[b, sel // case.page_size] * case.page_size + sel % case.page_size
        vmax = float(np.abs(kv[phys, :d]).max()) if sel.size else 0.0
        pre = (2.0 ** -14 + 2 * sel.size * FP32_UNIT + (2.0 ** -8 if split_exchange else 0.0)) * vmax
        rn = bf16_round(ref_out[t])                         # [H, d]
        err = np.abs(g[t] - rn)
        tol = bf16_ulp(rn) + pre
        assert np.all(err <= tol), (t, float(np.max(err - tol)))
        worst_ulps = max(worst_ulps, float(np.max(err / bf16_ulp(rn))))
    gl = cpu(gpu_lse).double().numpy()
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(gl), fin)
    dl = np.abs(gl[fin] - ref_lse[fin])
    assert np.all(dl <= 2.0 ** -16 + 2.0 ** -20 * np.abs(ref_lse[fin])), float(dl.max())
    return worst_ulps


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
