"""fp64 CPU oracle of the DSA hot path (ctypes wrapper over dsa_oracle.c).

TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg
may import this package.  The CUDA library (sparse_attention_29_b300) never does, and
this package never imports it.

Every function takes numpy arrays or torch CPU tensors and returns numpy arrays (float64
for real values).  The C file cites, for each step, the page and section it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_LIB = os.path.join(_HERE, "liborc_dsa.so")
_lock = threading.Lock()
_lib = None

# Plain code: no fused multiply-add contraction, no fast-math; OpenMP only over
# independent output rows.
CFLAGS = ["-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-shared", "-Wall"]


def build(force: bool = False) -> str:
    """Compile dsa_oracle.c into liborc_dsa.so (if missing or older than the source)."""
    with _lock:
        stale = (not os.path.exists(_LIB) or
                 os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
        if force or stale:
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        lib.orc_e4m3_to_double.restype = D
        lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_cache_append.restype = I
        lib.orc_cache_append.argtypes = [P, P, P, P, I, I, I, I, P, P, I, I, ctypes.c_int64,
                                         P, P, P]
        lib.orc_bf16_to_double.restype = D
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_indexer_scores.restype = I
        lib.orc_indexer_scores.argtypes = [P, P, P, P, P, P, P, I, I, P, I, I, I, I, I, P, P]
        lib.orc_topk.restype = I
        lib.orc_topk.argtypes = [P, P, I, I, I, P]
        lib.orc_sparse_mla.restype = I
        lib.orc_sparse_mla.argtypes = [P, P, P, P, I, I, P, P, I, I, I, I, I, I, D, P, P]
        lib.orc_dense_mla.restype = I
        lib.orc_dense_mla.argtypes = [P, P, P, P, I, I, P, I, I, I, I, I, D, P, P]
        for name in ("orc_mqa_decode_flops_per_token",):
            getattr(lib, name).restype = D
            getattr(lib, name).argtypes = [I, I, I]
        lib.orc_mqa_decode_bytes_per_token.restype = D
        lib.orc_mqa_decode_bytes_per_token.argtypes = [I, I, I]
        lib.orc_mqa_decode_intensity.restype = D
        lib.orc_mqa_decode_intensity.argtypes = [I, I, I, I]
        lib.orc_heads_at_ridge.restype = D
        lib.orc_heads_at_ridge.argtypes = [D, I, I, I]
        lib.orc_sdpa_score_flops.restype = D
        lib.orc_sdpa_score_flops.argtypes = [I, I]
        lib.orc_indexshare_indexer_cut.restype = D
        lib.orc_indexshare_indexer_cut.argtypes = [I]
        lib.orc_indexer_flops.restype = D
        lib.orc_indexer_flops.argtypes = [I, I, D]
        lib.orc_num_threads.restype = I
        lib.orc_num_threads.argtypes = []
        lib.orc_sparse_mha.restype = I
        lib.orc_sparse_mha.argtypes = [P, P, ctypes.c_int64, P, P, P, P, I, I, P, I, I, I, I, I, I, I, I, D, P, P]
        lib.orc_hisparse_step.restype = I
        lib.orc_hisparse_step.argtypes = [P, I, ctypes.c_uint32, P, I, P, P, I, P, P]
        _lib = lib
    return _lib


def _np(x, dtype):
    """Contiguous numpy view/copy of a numpy array or torch CPU tensor, as `dtype`."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        t = x.detach().cpu()
        if t.dtype == torch.bfloat16:
            t = t.view(torch.int16)
        x = t.numpy()
    a = np.ascontiguousarray(x)
    if a.dtype != np.dtype(dtype):
        if a.dtype.itemsize == np.dtype(dtype).itemsize and a.dtype.kind in "iu" and \
                np.dtype(dtype).kind in "iu":
            a = a.view(dtype)
        else:
            a = a.astype(dtype)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return _load().orc_num_threads()


def e4m3_to_double(code: int) -> float:
    return _load().orc_e4m3_to_double(int(code))


def e4m3_encode(x: float) -> int:
    """e4m3 code of the fp32 value x (nearest, ties to even, saturating at 448)."""
    return int(_load().orc_e4m3_encode(float(np.float32(x))))


def cache_append(k_new, c_new, seq, pos, B, k8, k_scale, kv, seq_start=None, block_table=None,
                 page_size=0):
    """New tokens into copies of the caches (step 0 of the C file).  k8 [num_rows, Di] uint8,
    k_scale [num_rows] float32 and kv [num_rows, D] uint16 are modified in place (numpy
    arrays); returns the number of tokens whose row did not resolve."""
    k_new = _np(k_new, np.float32)
    n, Di = k_new.shape
    c = None if c_new is None else _np(c_new, np.uint16)
    D = 0 if c is None else c.shape[1]
    seq = _np(seq, np.int32)
    pos = _np(pos, np.int32)
    ss = None if seq_start is None else _np(seq_start, np.int32)
    bt = None if block_table is None else _np(block_table, np.int32)
    pps = 0 if bt is None else bt.shape[-1]
    for a, t in ((k8, np.uint8), (k_scale, np.float32)):
        assert a.dtype == t and a.flags.c_contiguous
    assert kv is None or (kv.dtype == np.uint16 and kv.flags.c_contiguous)
    return int(_load().orc_cache_append(_ptr(k_new), None if c is None else _ptr(c), _ptr(seq),
                                        _ptr(pos), n, B, Di, D,
                                        None if ss is None else _ptr(ss),
                                        None if bt is None else _ptr(bt), int(page_size),
                                        int(pps), k8.shape[0], _ptr(k8), _ptr(k_scale),
                                        None if kv is None else _ptr(kv)))


def bf16_to_double(bits: int) -> float:
    return _load().orc_bf16_to_double(int(bits) & 0xFFFF)


def _addressing(case):
    seq_start = _np(case.seq_start, np.int32)
    bt = _np(case.block_table, np.int32)
    return seq_start, bt, int(case.page_size or 0), int(case.pages_per_seq)


def indexer_scores(case, with_abs=False):
    """[rows, Lmax] float64 indexer scores; -inf beyond each row's position.

    with_abs: also return the [rows, Lmax] sums of the magnitudes of every term of each
    score, sum_h |w| * sum_c |q * k| (0 beyond the position), as (scores, abs_terms)."""
    lib = _load()
    seq_start, bt, ps, pps = _addressing(case)
    q8 = _np(case.q8, np.uint8)
    qs = _np(case.q_scale, np.float32)
    w = _np(case.w, np.float32)
    qp = _np(case.q_pos, np.int32)
    B, T = case.B, case.T
    Lmax = case.Lmax
    out = np.empty((B * T, Lmax), dtype=np.float64)
    absum = np.empty((B * T, Lmax), dtype=np.float64) if with_abs else None
    rc = lib.orc_indexer_scores(_ptr(q8), _ptr(qs), _ptr(w), _ptr(_np(case.k8, np.uint8)),
                                _ptr(_np(case.k_scale, np.float32)), _ptr(seq_start), _ptr(bt),
                                ps, pps, _ptr(qp), B, T, case.Hi, case.Di, Lmax, _ptr(out),
                                _ptr(absum))
    if rc != 0:
        raise ValueError("oracle indexer: bad argument")
    return (out, absum) if with_abs else out


def topk(scores, q_pos, k):
    """[rows, k] int32: causal top-k (ascending token order, -1 padded).

    `scores` may be float32 or float64; float32 values are widened exactly, so every
    comparison is the one fp32 would make."""
    lib = _load()
    s = _np(scores, np.float64)
    qp = _np(q_pos, np.int32)
    rows, Lmax = s.shape
    out = np.empty((rows, k), dtype=np.int32)
    if lib.orc_topk(_ptr(s), _ptr(qp), rows, Lmax, int(k), _ptr(out)) != 0:
        raise ValueError("oracle top-k: bad argument")
    return out


def sparse_mla(case, idx, layer=0, check_causal=True):
    """(out [rows, H, d] float64, lse [rows, H] float64) of sparse MQA-mode MLA."""
    lib = _load()
    seq_start, bt, ps, pps = _addressing(case)
    q = _np(case.q[layer], np.uint16)
    kv = _np(case.kv[layer], np.uint16)
    ix = _np(idx, np.int32)
    rows = case.B * case.T
    K = ix.shape[1]
    out = np.empty((rows, case.H, case.d), dtype=np.float64)
    lse = np.empty((rows, case.H), dtype=np.float64)
    qp = _np(case.q_pos, np.int32) if check_causal else None
    rc = lib.orc_sparse_mla(_ptr(q), _ptr(kv), _ptr(seq_start), _ptr(bt), ps, pps, _ptr(ix),
                            _ptr(qp), case.B, case.T, case.H, case.d, case.r, K,
                            float(case.softmax_scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle sparse MLA: bad argument or index outside the causal window")
    return out, lse


def sparse_mha(case, idx, w_uk, w_uv, q_mha, layer=0):
    """(out [rows, H, vd] float64, lse [rows, H]) of MLA in MHA mode (step of the C file):
    w_uk [H, dn, d] and w_uv [H, vd, d] bf16 up-projections, q_mha [rows, H, dn + r] bf16."""
    lib = _load()
    seq_start, bt, ps, pps = _addressing(case)
    wk = _np(w_uk, np.uint16)
    wv = _np(w_uv, np.uint16)
    H, dn, d = wk.shape
    vd = wv.shape[1]
    ix = _np(idx, np.int32)
    rows = case.B * case.T
    out = np.empty((rows, H, vd), dtype=np.float64)
    lse = np.empty((rows, H), dtype=np.float64)
    kv = _np(case.kv[layer], np.uint16)
    rc = lib.orc_sparse_mha(_ptr(_np(q_mha, np.uint16)), _ptr(kv), kv.shape[0],
                            _ptr(wk), _ptr(wv), _ptr(seq_start), _ptr(bt), ps, pps, _ptr(ix),
                            case.B, case.T, H, d, case.r, dn, vd, ix.shape[1],
                            float(case.softmax_scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle sparse MHA: bad argument")
    return out, lse


def dense_mla(case, layer=0):
    """(out, lse) of dense causal MQA-mode attention over tokens 0..q_pos[t]."""
    lib = _load()
    seq_start, bt, ps, pps = _addressing(case)
    rows = case.B * case.T
    out = np.empty((rows, case.H, case.d), dtype=np.float64)
    lse = np.empty((rows, case.H), dtype=np.float64)
    rc = lib.orc_dense_mla(_ptr(_np(case.q[layer], np.uint16)), _ptr(_np(case.kv[layer], np.uint16)),
                           _ptr(seq_start), _ptr(bt), ps, pps, _ptr(_np(case.q_pos, np.int32)),
                           case.B, case.T, case.H, case.d, case.r, float(case.softmax_scale),
                           _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle dense MLA: bad argument")
    return out, lse


def dsa_layer(case, layer=0):
    """One DSA layer: indexer -> top-k -> sparse MLA.  Returns (scores, idx, out, lse)."""
    scores = indexer_scores(case)
    idx = topk(scores, case.q_pos, case.k)
    out, lse = sparse_mla(case, idx, layer=layer)
    return scores, idx, out, lse


def indexshare_group(case):
    """IndexShare over the case's layers [GLM53 §IndexShare]: layer 0 runs the indexer and
    the top-k once; every layer of the group attends over that one index set with its
    own query and latent cache.  Returns (idx, [(out, lse) per layer])."""
    scores = indexer_scores(case)
    idx = topk(scores, case.q_pos, case.k)
    return idx, [sparse_mla(case, idx, layer=g) for g in range(case.layers)]


# ---- accounting ------------------------------------------------------------------------

def mqa_decode_intensity(H, d, r, b):
    return _load().orc_mqa_decode_intensity(H, d, r, b)


def mqa_decode_flops_per_token(H, d, r):
    return _load().orc_mqa_decode_flops_per_token(H, d, r)


def mqa_decode_bytes_per_token(d, r, b):
    return _load().orc_mqa_decode_bytes_per_token(d, r, b)


def heads_at_ridge(ridge, d, r, b):
    return _load().orc_heads_at_ridge(float(ridge), d, r, b)


def sdpa_score_flops(H, dh):
    return _load().orc_sdpa_score_flops(H, dh)


def indexshare_indexer_cut(G):
    return _load().orc_indexshare_indexer_cut(G)


def indexer_flops(Hi, Di, n_keys):
    return _load().orc_indexer_flops(Hi, Di, float(n_keys))


# ---- HiSparse host tier ------------------------------------------------------------------

class HiSparseState:
    """One sequence's device working set under the oracle's LRU policy (step of the C file):
    res [Lmax] slot or -1, slot_tok [C] token or -1, slot_use [C] last use (0: never)."""

    def __init__(self, Lmax, C):
        self.res = np.full(Lmax, -1, np.int32)
        self.slot_tok = np.full(C, -1, np.int32)
        self.slot_use = np.zeros(C, np.uint32)

    def step(self, idx_row, step):
        """Apply one step; returns (hits, [(token, slot) loaded])."""
        lib = _load()
        row = np.ascontiguousarray(np.asarray(idx_row, np.int32))
        k = row.size
        loaded = np.empty(2 * max(k, 1), np.int32)
        hits = ctypes.c_int(0)
        m = lib.orc_hisparse_step(_ptr(row), k, int(step), _ptr(self.res), self.res.size,
                                  _ptr(self.slot_tok), _ptr(self.slot_use), self.slot_tok.size,
                                  _ptr(loaded), ctypes.byref(hits))
        if m < 0:
            raise ValueError("oracle HiSparse step: index out of range or too few slots")
        return hits.value, [(int(loaded[2 * i]), int(loaded[2 * i + 1])) for i in range(m)]
