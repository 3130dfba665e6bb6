"""ctypes binding of libdsa.so: argument marshalling only.

Each function has the name of the C entry point it calls and takes torch CUDA tensors
(or None) where the C function takes device pointers; every step of the computation runs
in the library's CUDA kernels.  A non-OK status raises DsaError.  There is no fallback:
if libdsa.so is missing or cannot be loaded, `load()` raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdsa.so")

DSA_OK = 0
DSA_ERR_DEVICE = 5
STATUS = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED", 3: "DSA_ERR_CUDA",
          4: "DSA_ERR_WORKSPACE", 5: "DSA_ERR_DEVICE", 6: "DSA_ERR_SCRATCH_LIMIT"}
DSA_OP_INDEXER, DSA_OP_TOPK, DSA_OP_SPARSE_MLA = 0, 1, 2
DSA_NOALLOC_SCRATCH_BYTES = 20 << 20

# every symbol include/dsa.h declares
EXPORTS = ("dsa_version", "dsa_status_string", "dsa_indexer_scores", "dsa_topk",
           "dsa_sparse_mla_decode", "dsa_sparse_mla_decode_noalloc", "dsa_sparse_mla_prefill",
           "dsa_sparse_mla_shared", "dsa_cache_append", "dsa_workspace_bytes",
           "dsa_device_error", "dsa_indexer_topk", "dsa_indexer_topk_workspace_bytes",
           "dsa_hisparse_init", "dsa_hisparse_fetch", "dsa_mla_up_project",
           "dsa_mha_workspace_bytes", "dsa_sparse_mha_prefill", "dsa_topk_sparse_mla_decode",
           "dsa_wait_probe")


class DsaError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")


class CacheLayout(ctypes.Structure):
    """dsa_cache_layout_t"""
    _fields_ = [("seq_start", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("page_size", ctypes.c_int32), ("pages_per_seq", ctypes.c_int32),
                ("num_rows", ctypes.c_int64)]


_lib = None


def load(path: str = LIB_PATH):
    """Load libdsa.so (built by sparse_attention_29_b300.build); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libdsa.so not found at {path}: run "
                           "`python -m sparse_attention_29_b300.build`")
    lib = ctypes.CDLL(path)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    LP = ctypes.POINTER(CacheLayout)
    lib.dsa_version.restype = ctypes.c_char_p
    lib.dsa_version.argtypes = []
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_status_string.argtypes = [I]
    lib.dsa_indexer_scores.restype = I
    lib.dsa_indexer_scores.argtypes = [P, P, P, P, P, LP, P, I, I, I, I, I, P, P]
    lib.dsa_topk.restype = I
    lib.dsa_topk.argtypes = [P, P, I, I, I, P, P]
    lib.dsa_indexer_topk.restype = I
    lib.dsa_indexer_topk.argtypes = [P, P, P, P, P, LP, P, I, I, I, I, I, I, P, P, S, P]
    lib.dsa_indexer_topk_workspace_bytes.restype = S
    lib.dsa_indexer_topk_workspace_bytes.argtypes = [I, I, I]
    lib.dsa_mla_up_project.restype = I
    lib.dsa_mla_up_project.argtypes = [P, ctypes.c_int64, I, I, P, I, P, P]
    lib.dsa_mha_workspace_bytes.restype = S
    lib.dsa_mha_workspace_bytes.argtypes = [I, I, I]
    lib.dsa_sparse_mha_prefill.restype = I
    lib.dsa_sparse_mha_prefill.argtypes = [P, P, P, P, LP, P, P, I, I, I, I, I, I, I, I, I, F, P,
                                           P, P, S, P]
    lib.dsa_hisparse_init.restype = I
    lib.dsa_hisparse_init.argtypes = [P, I, I, P, P, I, P]
    lib.dsa_hisparse_fetch.restype = I
    lib.dsa_hisparse_fetch.argtypes = [P, I, I, ctypes.c_uint32, P, P, I, P, I, P, P, I, P, P, P]
    lib.dsa_sparse_mla_decode.restype = I
    lib.dsa_sparse_mla_decode.argtypes = [P, P, LP, P, I, I, I, I, I, F, P, P, P, S, P]
    lib.dsa_topk_sparse_mla_decode.restype = I
    lib.dsa_topk_sparse_mla_decode.argtypes = [P, P, I, P, P, LP, P, I, I, I, I, I, F, P, P, P, S, P]
    lib.dsa_sparse_mla_decode_noalloc.restype = I
    lib.dsa_sparse_mla_decode_noalloc.argtypes = [P, P, LP, P, I, I, I, I, I, F, P, P, P]
    lib.dsa_sparse_mla_prefill.restype = I
    lib.dsa_sparse_mla_prefill.argtypes = [P, P, LP, P, I, I, I, I, I, I, F, P, P, P, S, P]
    lib.dsa_sparse_mla_shared.restype = I
    lib.dsa_sparse_mla_shared.argtypes = [P, P, I, LP, P, I, I, I, I, I, I, F, P, P, P, S, P]
    lib.dsa_cache_append.restype = I
    lib.dsa_cache_append.argtypes = [P, P, P, P, I, I, I, I, LP, P, P, P, P]
    lib.dsa_workspace_bytes.restype = S
    lib.dsa_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
    lib.dsa_device_error.restype = I
    lib.dsa_device_error.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    lib.dsa_wait_probe.restype = I
    lib.dsa_wait_probe.argtypes = [P, P]
    _lib = lib
    return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn, status):
    if status != DSA_OK:
        raise DsaError(fn, status)


def version() -> str:
    return load().dsa_version().decode()


def make_layout(num_rows, seq_start=None, block_table=None, page_size=0) -> CacheLayout:
    """dsa_cache_layout_t over device tensors; the structure keeps the tensors alive, since
    it holds only their addresses."""
    pps = 0 if block_table is None else int(block_table.shape[-1])
    layout = CacheLayout(_ptr(seq_start), _ptr(block_table), int(page_size), pps, int(num_rows))
    layout._tensors = (seq_start, block_table)
    return layout


def dsa_indexer_scores(q8, q_scale, w, k8_cache, k_scale, layout, q_pos, B, T, Hi, Di, Lmax,
                       scores, stream=None):
    st = load().dsa_indexer_scores(_ptr(q8), _ptr(q_scale), _ptr(w), _ptr(k8_cache),
                                   _ptr(k_scale), ctypes.byref(layout), _ptr(q_pos), B, T, Hi,
                                   Di, Lmax, _ptr(scores), _stream(stream))
    _check("dsa_indexer_scores", st)


def dsa_topk(scores, q_pos, rows, Lmax, k, idx, stream=None):
    st = load().dsa_topk(_ptr(scores), _ptr(q_pos), rows, Lmax, k, _ptr(idx), _stream(stream))
    _check("dsa_topk", st)


def dsa_indexer_topk(q8, q_scale, w, k8_cache, k_scale, layout, q_pos, B, T, Hi, Di, Lmax, k,
                     idx, workspace, workspace_bytes, stream=None):
    st = load().dsa_indexer_topk(_ptr(q8), _ptr(q_scale), _ptr(w), _ptr(k8_cache), _ptr(k_scale),
                                 ctypes.byref(layout), _ptr(q_pos), B, T, Hi, Di, Lmax, k,
                                 _ptr(idx), _ptr(workspace), int(workspace_bytes),
                                 _stream(stream))
    _check("dsa_indexer_topk", st)


def dsa_indexer_topk_workspace_bytes(B, T, Lmax) -> int:
    n = load().dsa_indexer_topk_workspace_bytes(B, T, Lmax)
    if n == ctypes.c_size_t(-1).value:
        raise DsaError("dsa_indexer_topk_workspace_bytes", 1)
    return n


def dsa_mla_up_project(latent, n, ld, d, w, N, out, stream=None):
    st = load().dsa_mla_up_project(_ptr(latent), int(n), ld, d, _ptr(w), N, _ptr(out),
                                   _stream(stream))
    _check("dsa_mla_up_project", st)


def dsa_mha_workspace_bytes(B, T, Lmax) -> int:
    n = load().dsa_mha_workspace_bytes(B, T, Lmax)
    if n == ctypes.c_size_t(-1).value:
        raise DsaError("dsa_mha_workspace_bytes", 1)
    return n


def dsa_sparse_mha_prefill(q, k_up, v_up, kv_cache, layout, idx, q_pos, B, T, H, d, r, dn, vd, k,
                           Lmax, scale, out, lse, workspace, workspace_bytes, stream=None):
    st = load().dsa_sparse_mha_prefill(_ptr(q), _ptr(k_up), _ptr(v_up), _ptr(kv_cache),
                                       ctypes.byref(layout), _ptr(idx), _ptr(q_pos), B, T, H, d, r,
                                       dn, vd, k, Lmax, float(scale), _ptr(out), _ptr(lse),
                                       _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check("dsa_sparse_mha_prefill", st)


def dsa_hisparse_init(residency, B, Lmax, slot_token, slot_use, C, stream=None):
    st = load().dsa_hisparse_init(_ptr(residency), B, Lmax, _ptr(slot_token), _ptr(slot_use), C,
                                  _stream(stream))
    _check("dsa_hisparse_init", st)


def dsa_hisparse_fetch(idx, B, k, step, host_kv, host_seq_start, D, residency, Lmax, slot_token,
                       slot_use, C, pool, stats=None, stream=None):
    """host_kv: a pinned host tensor (its address is device-accessible under unified
    addressing) or a device-accessible address."""
    st = load().dsa_hisparse_fetch(_ptr(idx), B, k, int(step), _ptr(host_kv), _ptr(host_seq_start),
                                   D, _ptr(residency), Lmax, _ptr(slot_token), _ptr(slot_use), C,
                                   _ptr(pool), _ptr(stats), _stream(stream))
    _check("dsa_hisparse_fetch", st)


def dsa_cache_append(k_new, c_new, seq, pos, n, B, Di, D, layout, k8_cache, k_scale, kv_cache,
                     stream=None):
    st = load().dsa_cache_append(_ptr(k_new), _ptr(c_new), _ptr(seq), _ptr(pos), n, B, Di, D,
                                 ctypes.byref(layout), _ptr(k8_cache), _ptr(k_scale),
                                 _ptr(kv_cache), _stream(stream))
    _check("dsa_cache_append", st)


def dsa_workspace_bytes(op, B, T, H, d, k, n_layers=1) -> int:
    n = load().dsa_workspace_bytes(op, B, T, H, d, k, n_layers)
    if n == ctypes.c_size_t(-1).value:
        raise DsaError("dsa_workspace_bytes", 1)
    return n


def dsa_sparse_mla_decode(q, kv_cache, layout, idx, B, H, d, r, k, scale, out, lse, workspace,
                          workspace_bytes, stream=None):
    st = load().dsa_sparse_mla_decode(_ptr(q), _ptr(kv_cache), ctypes.byref(layout), _ptr(idx),
                                      B, H, d, r, k, float(scale), _ptr(out), _ptr(lse),
                                      _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check("dsa_sparse_mla_decode", st)


def dsa_topk_sparse_mla_decode(scores, q_pos, Lmax, q, kv_cache, layout, idx, B, H, d, r, k,
                               scale, out, lse, workspace, workspace_bytes, stream=None):
    st = load().dsa_topk_sparse_mla_decode(_ptr(scores), _ptr(q_pos), Lmax, _ptr(q),
                                           _ptr(kv_cache), ctypes.byref(layout), _ptr(idx), B, H,
                                           d, r, k, float(scale), _ptr(out), _ptr(lse),
                                           _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check("dsa_topk_sparse_mla_decode", st)


def dsa_sparse_mla_decode_noalloc(q, kv_cache, layout, idx, B, H, d, r, k, scale, out, lse,
                                  stream=None):
    st = load().dsa_sparse_mla_decode_noalloc(_ptr(q), _ptr(kv_cache), ctypes.byref(layout),
                                              _ptr(idx), B, H, d, r, k, float(scale),
                                              _ptr(out), _ptr(lse), _stream(stream))
    _check("dsa_sparse_mla_decode_noalloc", st)


def dsa_sparse_mla_prefill(q, kv_cache, layout, idx, B, T, H, d, r, k, scale, out, lse,
                           workspace, workspace_bytes, stream=None):
    st = load().dsa_sparse_mla_prefill(_ptr(q), _ptr(kv_cache), ctypes.byref(layout),
                                       _ptr(idx), B, T, H, d, r, k, float(scale), _ptr(out),
                                       _ptr(lse), _ptr(workspace), int(workspace_bytes),
                                       _stream(stream))
    _check("dsa_sparse_mla_prefill", st)


def _ptr_array(ts):
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = _ptr(t)
    return arr


def dsa_sparse_mla_shared(q_layers, kv_layers, layout, idx, B, T, H, d, r, k, scale,
                          out_layers, lse_layers, workspace, workspace_bytes, stream=None):
    n = len(q_layers)
    qa, kva, oa = _ptr_array(q_layers), _ptr_array(kv_layers), _ptr_array(out_layers)
    la = _ptr_array(lse_layers) if lse_layers is not None else None
    st = load().dsa_sparse_mla_shared(ctypes.cast(qa, ctypes.c_void_p),
                                      ctypes.cast(kva, ctypes.c_void_p), n, ctypes.byref(layout),
                                      _ptr(idx), B, T, H, d, r, k, float(scale),
                                      ctypes.cast(oa, ctypes.c_void_p),
                                      None if la is None else ctypes.cast(la, ctypes.c_void_p),
                                      _ptr(workspace), int(workspace_bytes), _stream(stream))
    _check("dsa_sparse_mla_shared", st)


def dsa_wait_probe(result, stream=None):
    """Diagnostics: a bounded wait that runs out on purpose (result: 4 uint64 on the device)."""
    _check("dsa_wait_probe", load().dsa_wait_probe(_ptr(result), _stream(stream)))


def dsa_device_error(stream=None):
    """(status, first error code) after synchronising the stream; clears the word."""
    code = ctypes.c_uint32(0)
    st = load().dsa_device_error(_stream(stream), ctypes.byref(code))
    return st, code.value
