"""Benchmark of the DSA decode hot path on B300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode_32k|ragged_decode|prefill_8k|indexshare_paged]

A step is one pass of the whole hot path over one batch: lightning indexer -> top-k ->
sparse MLA (for the IndexShare workload: indexer and top-k once, MLA for 4 layers).
The default workload is the decode batch the metric is quoted on: 32 sequences x 32768
cached tokens, one query each, Hi=64 x Di=128 fp8 indexer, k=2048, H=64, d=512 + r=64
bf16 latent.  Inputs are synthetic (seeded, drawn on the device) and resident in HBM;
three independent input sets rotate so that each step's ~220 MB of reads miss L2.

Multi-GPU: every sequence is independent, so N ranks run N replicas on their own
batches (weak scaling, no collective on the data path); value = all ranks' query
tokens / max-over-ranks time.

--impl reference times the fp64 CPU oracle (the only other implementation there is) on a
bounded sample of the same workload, on the host's cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "DSA decode query-tokens/s at 32K ctx; achieved HBM TB/s vs B300 peak"
UNIT = "query-tok/s"

WORKLOADS = {
    "decode_32k": "32 seq x 32768 ctx, 1 decode query each; indexer 64x128 e4m3; top-2048; "
                  "MLA H=64 d=512 r=64 bf16",
    "ragged_decode": "16 seq, ctx log-uniform 1024..200000 (5% planted keys), 1 decode query each",
    "prefill_8k": "1 seq, 8192 query rows after a 57344-token prefix (65536 total)",
    "indexshare_paged": "IndexShare group of 4 layers, 64 seq x 16384 ctx, 64-token pages",
}


def per_query_bytes(case):
    """Algorithmic HBM bytes of one step, per workload: every byte the path must move once.

    Indexer: the fp8 keys and their scales of every visible token, the query (q8, scale,
    weights, position) and the written scores.  Top-k: the scores read, the indices
    written.  Sparse MLA: the selected latent rows (d+r bf16 each), the query, the
    indices read, the output written (and lse)."""
    tot_idx = tot_topk = tot_mla = 0
    D = case.d + case.r
    for b, L in enumerate(case.lengths):
        for i in range(case.T):
            n = L - case.T + 1 + i
            m = min(n, case.k)
            tot_idx += n * (case.Di + 4) + case.Hi * case.Di + 4 + case.Hi * 4 + 4 + 4 * n
            tot_topk += 4 * n + 4 * case.k + 4
            tot_mla += case.layers * (m * D * 2 + case.H * D * 2 + case.H * case.d * 2 +
                                      case.H * 4) + 4 * case.k
    return tot_idx, tot_topk, tot_mla


def scores_in_step(case):
    """Bytes of the score round trip (written by the indexer, read by top-k): part of the
    API's two-call form, not of the method, so excluded from the whole-step figure."""
    return sum(8 * (L - case.T + 1 + i) for L in case.lengths for i in range(case.T))


def one_call_bytes(case):
    """Algorithmic bytes of the one-call top-k + sparse MLA launch: the scores read and the
    index set written once (the kernel reads its own index set back from L2), plus the
    sparse MLA's selected rows, query and output."""
    _, b_topk, b_mla = per_query_bytes(case)
    return b_topk + b_mla - 4 * case.k * case.rows


IDX_FILES = ["sparse_attention_29_b300/csrc/indexer.cu", "sparse_attention_29_b300/csrc/ptx.cuh"]
MLA_FILES = ["sparse_attention_29_b300/csrc/sparse_mla.cu", "sparse_attention_29_b300/csrc/ptx.cuh",
             "sparse_attention_29_b300/csrc/topk_core.cuh", "sparse_attention_29_b300/csrc/keys.cuh"]
TOPK_FILES = ["sparse_attention_29_b300/csrc/topk.cu", "sparse_attention_29_b300/csrc/topk_core.cuh",
              "sparse_attention_29_b300/csrc/ptx.cuh", "sparse_attention_29_b300/csrc/keys.cuh"]


def step_rooflines(case, args, k_idx, k_topk, k_mla, k_fused, shared, hbm_peak, bf16_peak,
                   peak_src):
    """The roofline of every kernel of the step (warm per-launch times), and that of the
    kernel with the largest share of the step's kernel time, which is the headline one.

    Decode: each kernel against the measured copy bandwidth, with its algorithmic bytes.
    Chunked prefill: the indexer against the fp8 tensor peak (the measured bf16 burst peak
    x 2, the nominal fp8:bf16 ratio), over the q.k dot products of every visible key; the
    sparse MLA against the bf16 peak, over its two products per selected key; the top-k
    against the copy bandwidth."""
    b_idx, b_topk, b_mla = per_query_bytes(case)
    wl = args.workload

    def hbm(name, nbytes, ms, traffic=None):
        ach = nbytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "kernel": name, "achieved": ach, "peak": hbm_peak,
                "unit": "GB/s", "frac": ach / hbm_peak, "traffic": traffic,
                "algorithmic_bytes": nbytes, "ms": ms, "peak_source": peak_src}

    def tensor(name, flops, ms, peak, src):
        tf = flops / (ms * 1e-3) / 1e12
        return {"bound": "tensor", "kernel": name, "achieved": tf, "peak": peak,
                "unit": "TFLOP/s", "frac": tf / peak, "traffic": None,
                "algorithmic_flops": flops, "ms": ms, "peak_source": src}

    out = {}
    if case.T > 1:
        pos = case.q_pos.long().add(1)
        flops = float(pos.sum().item()) * case.Hi * case.Di * 2.0
        out["indexer"] = tensor("indexer", flops, k_idx, 2.0 * bf16_peak,
                                f"{peak_src} bf16 burst x 2 (nominal fp8:bf16 ratio)")
        out["topk"] = hbm("topk", b_topk, k_topk)
        nsel = float(pos.clamp(max=case.k).sum().item()) * case.layers
        mla_flops = nsel * case.H * (2.0 * (case.d + case.r) + 2.0 * case.d)
        out["sparse_mla"] = tensor("sparse_mla", mla_flops, k_mla, bf16_peak,
                                   f"{peak_src} bf16 burst")
    else:
        out["indexer"] = hbm("indexer", b_idx, k_idx, traffic_for(IDX_FILES, "indexer", wl))
        if k_fused:
            out["topk_and_sparse_mla_one_call"] = hbm(
                "topk_and_sparse_mla_one_call", one_call_bytes(case), k_fused,
                traffic_for(MLA_FILES, "sparse_mla", wl))
        else:
            out["topk"] = hbm("topk", b_topk, k_topk, traffic_for(TOPK_FILES, "topk", wl))
            out["sparse_mla_shared" if shared else "sparse_mla"] = hbm(
                "sparse_mla_shared" if shared else "sparse_mla", b_mla, k_mla)
    timed = [r for r in out.values() if r["ms"] == r["ms"]]  # NaN in a profile run
    head = max(timed, key=lambda r: r["ms"]) if timed else out["indexer"]
    return head, out


def src_sha(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs"), d.get("bf16_tflops"), "measured"
    return 6400.0, 1800.0, "fallback"


def traffic_for(kernel_files, kernel, workload):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on this
    workload and the kernel is unchanged since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(kernel)
    if not d or d.get("source_sha") != src_sha(kernel_files) or d.get("workload_key") != workload:
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 200 ms into a file while the
    block runs (a load pre-roll plus the timed region)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        import tempfile
        self.gpu = gpu_index
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="dsa_clocks_", suffix=".csv")
        os.close(fd)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                lines = f.read().splitlines()
            os.unlink(self.path)
        except OSError:
            lines = []
        for ln in lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm),
                "window": "1 s load pre-roll + timed region"}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value, world, device=None):
    """The largest of every rank's value: a job's time is that of its slowest rank.  With
    one rank, the value itself; else an all-reduce (MAX) on the current process group."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, world, ms):
    """Whole-job throughput: every rank processed `units_per_rank` in `ms` (the slowest
    rank's time), so the job processed world x units_per_rank."""
    return world * units_per_rank / (ms * 1e-3)


def pack_io(lay):
    """Lay the step's per-query inputs (q8, q_scale, w, q_pos and every layer's q) and its
    outputs (every layer's out and lse) out as views of two contiguous device buffers, so
    that a step's upload and download are one copy each.  Returns (in_buf, out_buf)."""
    import torch
    c = lay.case
    dev = c.k8.device

    def layout(tensors):
        offs, n = [], 0
        for t in tensors:
            n = (n + 255) // 256 * 256
            offs.append(n)
            n += t.numel() * t.element_size()
        return offs, n

    ins = [c.q8, c.q_scale, c.w, c.q_pos] + list(c.q)
    offs, n = layout(ins)
    in_buf = torch.empty(n, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(ins, offs):
        v = in_buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    c.q8, c.q_scale, c.w, c.q_pos = views[:4]
    c.q = views[4:]
    outs = list(lay.out) + list(lay.lse)
    offs, n = layout(outs)
    out_buf = torch.empty(n, dtype=torch.uint8, device=dev)
    ov = [out_buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
          for t, o in zip(outs, offs)]
    lay.out, lay.lse = ov[:len(lay.out)], ov[len(lay.out):]
    return in_buf, out_buf


def kernel_times(layers, stream, steps, fns):
    """Average device time of each call type: `steps` launches of one call (inputs rotating
    over the layers' input sets) captured into one CUDA graph and replayed between two
    events on the launching stream, so that host submission does not read as device time.
    An eager loop stands in where capture is unavailable."""
    import torch
    out = []
    for fn in fns:
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        try:
            cap = torch.cuda.Stream()
            cap.wait_stream(stream)
            with torch.cuda.stream(cap):
                for lay in layers:
                    lay.stream = cap
                fn(layers[0])
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap):
                    for i in range(steps):
                        fn(layers[i % len(layers)])
            for lay in layers:
                lay.stream = None
            g.replay()
            torch.cuda.synchronize()
            a.record(stream)
            g.replay()
            b.record(stream)
            torch.cuda.synchronize()
        except Exception:
            for lay in layers:
                lay.stream = None
            torch.cuda.synchronize()
            a.record(stream)
            for i in range(steps):
                fn(layers[i % len(layers)])
            b.record(stream)
            torch.cuda.synchronize()
        out.append(a.elapsed_time(b) / steps)
    return out


class HostBuffer:
    """Page-locked host memory from cudaHostAlloc with a CPU tensor view; copies to and
    from device tensors are single cudaMemcpyAsync calls on a given stream."""

    def __init__(self, numel, dtype):
        import ctypes
        import numpy as np
        import torch
        from cuda.bindings import runtime as rt
        self.rt = rt
        self.nbytes = numel * torch.empty(0, dtype=dtype).element_size()
        err, self.ptr = rt.cudaHostAlloc(self.nbytes, rt.cudaHostAllocDefault)
        if err != rt.cudaError_t.cudaSuccess:
            raise RuntimeError(f"cudaHostAlloc: {err}")
        raw = np.frombuffer((ctypes.c_uint8 * self.nbytes).from_address(self.ptr), dtype=np.uint8)
        self.tensor = torch.from_numpy(raw).view(dtype)

    def fill_from(self, src):
        import ctypes
        assert src.is_contiguous() and src.numel() * src.element_size() == self.nbytes
        ctypes.memmove(self.ptr, src.data_ptr(), self.nbytes)

    def _copy(self, dst, src, kind, stream):
        err, = self.rt.cudaMemcpyAsync(dst, src, self.nbytes, kind, stream.cuda_stream)
        if err != self.rt.cudaError_t.cudaSuccess:
            raise RuntimeError(f"cudaMemcpyAsync: {err}")

    def upload(self, dev_tensor, stream):
        assert dev_tensor.numel() * dev_tensor.element_size() == self.nbytes
        self._copy(dev_tensor.data_ptr(), self.ptr, self.rt.cudaMemcpyKind.cudaMemcpyHostToDevice, stream)

    def download(self, dev_tensor, stream):
        assert dev_tensor.numel() * dev_tensor.element_size() == self.nbytes
        self._copy(self.ptr, dev_tensor.data_ptr(), self.rt.cudaMemcpyKind.cudaMemcpyDeviceToHost, stream)

    def __del__(self):
        try:
            self.rt.cudaFreeHost(self.ptr)
        except Exception:
            pass


def flush_host_caches(nbytes=512 << 20):
    """Write (then drop) a scratch buffer larger than the host caches, so that lines written
    earlier are back in memory."""
    import ctypes
    buf = ctypes.create_string_buffer(nbytes)
    ctypes.memset(buf, 1, nbytes)
    del buf


def kernels_in_graph(graph):
    """Kernel nodes of a captured CUDA graph (the launches one replay makes), or None."""
    try:
        from cuda.bindings import runtime as rt
        raw = rt.cudaGraph_t(init_value=graph.raw_cuda_graph())
        err, _, n = rt.cudaGraphGetNodes(raw, 0)
        if err != rt.cudaError_t.cudaSuccess:
            return None
        err, nodes, n = rt.cudaGraphGetNodes(raw, n)
        if err != rt.cudaError_t.cudaSuccess:
            return None
        count = 0
        for node in nodes[:n]:
            err, t = rt.cudaGraphNodeGetType(node)
            if err == rt.cudaError_t.cudaSuccess and t == rt.cudaGraphNodeType.cudaGraphNodeTypeKernel:
                count += 1
        return count
    except Exception:
        return None


def step_of(case):
    return (lambda lay: lay.run_shared()) if case.layers > 1 else (lambda lay: lay.run())


def time_steps(layers, stream, steps, warmup, step):
    """Milliseconds per whole step: `steps` steps back to back between two events."""
    import torch
    for i in range(warmup):
        step(layers[i % len(layers)])
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(steps):
        step(layers[i % len(layers)])
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def measure_other_workload(name, dev, steps, warmup, hbm_peak, bf16_peak):
    """One of the other serving workloads, measured beside the headline one (not part of
    `value`): whole-step time, per-kernel times and the roofline that bounds the step."""
    import torch
    from sparse_attention_29_b300.pipeline import DsaLayer
    n_sets = 1 if name in ("prefill_8k", "indexshare_paged") else 2
    sets = [make_workload(name, dev, seed_offset=17 * i) for i in range(n_sets)]
    layers = [DsaLayer(c) for c in sets]
    case = sets[0]
    stream = torch.cuda.current_stream()
    step = step_of(case)
    ms = time_steps(layers, stream, steps, warmup, step)
    mla = (lambda lay: lay.mla_shared()) if case.layers > 1 else (lambda lay: lay.mla())
    k_idx, k_topk, k_mla = kernel_times(layers, stream, steps,
                                        [lambda lay: lay.indexer(), lambda lay: lay.topk(), mla])
    layers[0].check_device_error()
    b_idx, b_topk, b_mla = per_query_bytes(case)
    res = {"workload": name + ": " + WORKLOADS[name], "rows": case.rows, "steps": steps,
           "ms_per_step": ms, "query_tok_per_s": case.rows / (ms * 1e-3),
           "kernel_ms": {"indexer": k_idx, "topk": k_topk, "sparse_mla": k_mla}}
    if case.T > 1:
        # chunked prefill: the indexer is a dense fp8 contraction (every visible key's q.k
        # dot products), the sparse MLA two bf16 contractions per selected key
        flops = float(case.q_pos.long().add(1).sum().item()) * case.Hi * case.Di * 2.0
        fp8_peak = 2.0 * bf16_peak
        tf = flops / (k_idx * 1e-3) / 1e12
        nsel = float(case.q_pos.long().add(1).clamp(max=case.k).sum().item())
        mla_flops = nsel * case.H * (2.0 * (case.d + case.r) + 2.0 * case.d)
        mtf = mla_flops / (k_mla * 1e-3) / 1e12
        res["roofline"] = {"bound": "tensor", "kernel": "indexer", "achieved": tf,
                           "peak": fp8_peak, "unit": "TFLOP/s", "frac": tf / fp8_peak,
                           "algorithmic_flops": flops,
                           "peak_source": "measured bf16 burst x 2 (nominal fp8:bf16 ratio)"}
        res["sparse_mla_roofline"] = {"bound": "tensor", "achieved": mtf, "peak": bf16_peak,
                                      "unit": "TFLOP/s", "frac": mtf / bf16_peak,
                                      "algorithmic_flops": mla_flops}
        res["score_round_trip_bytes"] = scores_in_step(case)
        # the same step with the fused indexer + top-k (no score matrix in memory)
        ms_f = time_steps(layers, stream, steps, warmup, lambda lay: lay.run_fused())
        (k_f,) = kernel_times(layers, stream, steps, [lambda lay: lay.indexer_topk()])
        layers[0].check_device_error()
        tf_f = flops / (k_f * 1e-3) / 1e12
        res["fused_indexer_topk"] = {
            "ms_per_step": ms_f, "query_tok_per_s": case.rows / (ms_f * 1e-3),
            "indexer_topk_ms": k_f,
            "roofline": {"bound": "tensor", "kernel": "indexer + top-k (fused)",
                         "achieved": tf_f, "peak": fp8_peak, "unit": "TFLOP/s",
                         "frac": tf_f / fp8_peak, "algorithmic_flops": flops}}
    else:
        step_bytes = b_idx + b_topk + b_mla - scores_in_step(case)
        tbs = step_bytes / (ms * 1e-3) / 1e12
        res["roofline"] = {"bound": "hbm", "kernel": "whole step", "achieved": tbs * 1e3,
                           "peak": hbm_peak, "unit": "GB/s", "frac": tbs * 1e3 / hbm_peak,
                           "algorithmic_bytes": step_bytes}
        res["us_per_step"] = ms * 1e3
    del layers, sets
    torch.cuda.empty_cache()
    return res


def measure_hisparse(lay, dev, hbm_peak, C=4096, reps=10):
    """The host-tier working set on the decode batch: the full latent cache in pinned host
    memory, C device slots per sequence (LRU), the step's own top-k selection.  Times the
    fetch of a cold step (every selected row comes from the host), of a step whose
    selection is already resident (all hits) and of one with half the selection new, and
    the sparse MLA reading the working set against the MLA over the full device cache."""
    import torch
    from sparse_attention_29_b300 import capi
    c = lay.case
    B, D, Lmax, k = c.B, c.D, c.Lmax, c.k
    host_kv = c.kv[0].view(torch.int16).cpu().pin_memory()
    res = torch.empty((B, Lmax), dtype=torch.int32, device=dev)
    stok = torch.empty((B, C), dtype=torch.int32, device=dev)
    use = torch.empty((B, C), dtype=torch.int32, device=dev)
    pool = torch.empty((B * C, D), dtype=torch.int16, device=dev)
    stats = torch.zeros((B, 2), dtype=torch.int32, device=dev)
    lay.indexer()
    lay.topk()
    idx = lay.idx.clone()
    # a second selection sharing half of each row (the other half: the rows' next tokens
    # outside the first selection), still ascending
    idx2 = idx.clone()
    for b in range(B):
        row = idx[b]
        free = torch.ones(Lmax, dtype=torch.bool, device=dev)
        free[row[row >= 0].long()] = False
        free[c.lengths[b]:] = False
        new = torch.nonzero(free).flatten()[: k // 2].to(torch.int32)
        idx2[b] = torch.sort(torch.cat([row[: k - new.numel()], new])).values
    layout = capi.make_layout(B * C, block_table=res, page_size=1)
    ev = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))  # noqa: E731

    def fetch_ms(sel, step):
        a, e = ev()
        a.record()
        capi.dsa_hisparse_fetch(sel, B, k, step, host_kv, c.seq_start, D, res, Lmax, stok, use, C,
                                pool, stats)
        e.record()
        torch.cuda.synchronize()
        return a.elapsed_time(e)

    cold, warm, half = [], [], []
    step = 0
    for _ in range(reps):
        capi.dsa_hisparse_init(res, B, Lmax, stok, use, C)
        step += 1
        cold.append(fetch_ms(idx, step))
        step += 1
        warm.append(fetch_ms(idx, step))
        st_warm = stats.sum(0).tolist()
        step += 1
        half.append(fetch_ms(idx2, step))
        st_half = stats.sum(0).tolist()
    out = torch.empty_like(lay.out[0])
    lse = torch.empty_like(lay.lse[0])

    def mla_ms(kv, lay_):
        times = []
        for _ in range(reps):
            a, e = ev()
            a.record()
            capi.dsa_sparse_mla_decode(c.q[0], kv, lay_, idx2, B, c.H, c.d, c.r, k, c.softmax_scale,
                                       out, lse, lay.workspace, lay.ws_bytes)
            e.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(e))
        return sorted(times)[len(times) // 2]

    mla_pool = mla_ms(pool.view(torch.bfloat16), layout)
    mla_full = mla_ms(c.kv[0], lay.layout)
    overlap = measure_layer_overlap(lay, dev, host_kv, idx, C=C, reps=reps)
    st, code = capi.dsa_device_error()
    med = lambda x: sorted(x)[len(x) // 2]  # noqa: E731
    cold_bytes = B * k * D * 2
    return {"workload": f"decode_32k with the latent cache in pinned host memory and {C} device "
                        f"slots per sequence ({C / c.lengths[0]:.3f} of the context), LRU",
            "fetch_us": {"cold": med(cold) * 1e3, "all_hits": med(warm) * 1e3,
                         "half_new": med(half) * 1e3},
            "hits_misses": {"all_hits": st_warm, "half_new": st_half},
            "host_link_gbs_cold": cold_bytes / (med(cold) * 1e-3) / 1e9,
            "sparse_mla_us": {"through_working_set": mla_pool * 1e3, "full_device_cache": mla_full * 1e3},
            "device_bytes": {"working_set": B * C * D * 2, "full_cache": c.n_phys * D * 2},
            "layer_ahead_overlap": overlap,
            "device_check": "ok" if st == capi.DSA_OK else f"code {code:#x}",
            "timing": "CUDA events around single launches, median of %d" % reps}


def measure_layer_overlap(lay, dev, host_kv, idx, C, reps, L=4, frac_new=0.05):
    """The host tier's layer-wise overlap on an IndexShare group of L layers over the decode
    batch (each layer with its own working set; the timing does not depend on the rows'
    contents, so the layers share one pinned history): a decode step whose shared
    selection differs from the previous step's in `frac_new` of each row, run with every
    layer's fetch before its attention on one stream, and with the fetches on a second
    stream so that layer l + 1's fetch runs while layer l attends."""
    import torch
    from sparse_attention_29_b300.pipeline import HostTierGroup
    c = lay.case
    B, k, Lmax = c.B, c.k, c.Lmax
    idx2 = idx.clone()
    n_new = int(k * frac_new)
    for b in range(B):
        row = idx[b]
        free = torch.ones(Lmax, dtype=torch.bool, device=dev)
        free[row[row >= 0].long()] = False
        free[c.lengths[b]:] = False
        cand = torch.nonzero(free).flatten()
        new = cand[torch.randperm(cand.numel(), device=dev)[:n_new]].to(torch.int32)
        keep = row[torch.randperm(k, device=dev)[: k - n_new]]
        idx2[b] = torch.sort(torch.cat([keep, new])).values
    grp = HostTierGroup([host_kv] * L, c.seq_start, B, Lmax, c.D, C, device=dev)
    outs = [torch.empty_like(lay.out[0]) for _ in range(L)]
    lses = [torch.empty_like(lay.lse[0]) for _ in range(L)]
    qs = [c.q[0]] * L
    args = (c.H, c.d, c.r, c.softmax_scale, lay.workspace, lay.ws_bytes)

    def step_ms(overlap):
        times = []
        for _ in range(reps):
            grp.reset()
            grp.step(idx, k, 1, qs, outs, lses, *args, overlap=overlap)  # the previous step
            torch.cuda.synchronize()
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            grp.step(idx2, k, 2, qs, outs, lses, *args, overlap=overlap)
            e.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(e))
        return sorted(times)[len(times) // 2]

    def one_ms(fn):
        times = []
        for _ in range(reps):
            grp.reset()
            grp.step(idx, k, 1, qs, outs, lses, *args, overlap=False)
            torch.cuda.synchronize()
            a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            e.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(e))
        return sorted(times)[len(times) // 2]

    seq = step_ms(False)
    ov = step_ms(True)
    fetch = one_ms(lambda: grp.fetch(0, idx2, k, 2))
    misses = int(grp.stats[0][:, 1].sum().item())  # of that fetch
    mla = one_ms(lambda: grp.mla(0, idx, k, qs[0], outs[0], lses[0], *args))
    return {"layers": L, "selection_new_per_row": n_new,
            "step_us": {"fetch_then_attend": seq * 1e3, "layer_ahead_overlap": ov * 1e3},
            "per_layer_us": {"fetch": fetch * 1e3, "sparse_mla": mla * 1e3},
            "rows_fetched_per_layer": misses}


def measure_mha_vs_mqa(dev, contexts=(2048, 4096, 8192), T=1024, H=64, reps=5):
    """MLA's two modes on short-context chunked prefill: T query rows at the end of one
    sequence, each with k = 2048 selected tokens (all of them when it sees fewer), the
    GLM-5 shapes (latent 512 + rope 64; MHA mode: nope 192 + rope 64 per head, values of
    128).  MHA mode: up-projection of the context's keys and values, then the masked
    attention; MQA mode: the sparse MLA over the latent rows."""
    import torch
    from sparse_attention_29_b300 import capi, inputs
    d, r, dn, vd, k = 512, 64, 192, 128, 2048
    g = torch.Generator(device=dev).manual_seed(7)
    w_uk = (torch.randn(H * dn, d, device=dev, generator=g) / 16).to(torch.bfloat16)
    w_uv = (torch.randn(H * vd, d, device=dev, generator=g) / 16).to(torch.bfloat16)
    out = {}
    for L in contexts:
        case = inputs.make_case(f"mha-{L}", seed=L, lengths=[L], T=T, H=H, k=k, device=dev)
        n = L
        idx = torch.full((T, k), -1, dtype=torch.int32, device=dev)
        for t in range(T):
            nv = int(case.q_pos[t]) + 1
            m = min(nv, k)
            idx[t, :m] = torch.sort(torch.randperm(nv, device=dev, generator=g)[:m]).values.to(torch.int32)
        kv = case.kv[0]
        q_mha = torch.randn(T, H, dn + r, device=dev, generator=g).to(torch.bfloat16)
        k_up = torch.empty((n, H * dn), dtype=torch.bfloat16, device=dev)
        v_up = torch.empty((n, H * vd), dtype=torch.bfloat16, device=dev)
        o_mha = torch.empty((T, H, vd), dtype=torch.bfloat16, device=dev)
        o_mqa = torch.empty((T, H, d), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((T, H), dtype=torch.float32, device=dev)
        ws = capi.dsa_mha_workspace_bytes(1, T, L)
        wbuf = torch.empty(ws, dtype=torch.uint8, device=dev)
        wsm = capi.dsa_workspace_bytes(capi.DSA_OP_SPARSE_MLA, 1, T, H, d, k, 1)
        wbm = torch.empty(max(wsm, 16), dtype=torch.uint8, device=dev)
        layout = capi.make_layout(n, seq_start=case.seq_start)

        def up():
            capi.dsa_mla_up_project(kv, n, d + r, d, w_uk, H * dn, k_up)
            capi.dsa_mla_up_project(kv, n, d + r, d, w_uv, H * vd, v_up)

        def attn():
            capi.dsa_sparse_mha_prefill(q_mha, k_up, v_up, kv, layout, idx, case.q_pos, 1, T, H, d,
                                        r, dn, vd, k, L, case.softmax_scale, o_mha, lse, wbuf, ws)

        def mqa():
            capi.dsa_sparse_mla_prefill(case.q[0], kv, layout, idx, 1, T, H, d, r, k,
                                        case.softmax_scale, o_mqa, lse, wbm, wsm)

        def ms(fn):
            fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                fn()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / reps

        t_up, t_attn, t_mqa = ms(up), ms(attn), ms(mqa)
        nsel = float(case.q_pos.long().add(1).clamp(max=k).sum().item())
        out[str(L)] = {"mha_ms": t_up + t_attn, "mha_up_project_ms": t_up, "mha_attention_ms": t_attn,
                       "mqa_sparse_mla_ms": t_mqa,
                       "flops_per_pair": {"mha": 2 * H * (dn + r + vd), "mqa": 2 * H * (2 * d + r)},
                       "selected_pairs": nsel}
        del case, k_up, v_up
    torch.cuda.empty_cache()
    return {"rows": T, "heads": H, "shapes": "latent 512 + rope 64; MHA nope 192 + rope 64, values 128",
            "by_context": out}


def make_workload(name, device, seed_offset=0, rows=0):
    from sparse_attention_29_b300 import inputs
    if rows and inputs.PRESETS[name]["T"] > 1:
        p = dict(inputs.PRESETS[name])
        p["seed"] += seed_offset
        p["T"] = rows
        return inputs.make_case(name, device=device, **p)
    return inputs.preset(name, seed=inputs.PRESETS[name]["seed"] + seed_offset, device=device)


def run_reference(args, world, rank):
    """The oracle, timed on the host's cores on a bounded sample of the workload."""
    if rank != 0:
        return 0
    import oracle
    from sparse_attention_29_b300 import inputs
    oracle.build()
    p = dict(inputs.PRESETS[args.workload])
    # a bounded sample: one sequence (one query row) of the workload per step
    if args.workload == "ragged_decode":
        p["lengths"] = [inputs.ragged_lengths(16, 1024, 200000, p["seed"])[0]]
    elif args.workload == "prefill_8k":
        p["lengths"] = [65536]
        p["T"] = 1
    else:
        p["lengths"] = p["lengths"][:1]
    case = inputs.make_case(args.workload + "-sample", **p)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        if case.layers > 1:
            oracle.indexshare_group(case)
        else:
            oracle.dsa_layer(case)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    per_step = sum(times) / len(times)
    value = case.rows / per_step
    cores = oracle.num_threads()
    sample = (f"{case.rows} query row(s) of {args.workload} per step "
              f"(context {case.lengths[0]}, full indexer + top-k + MLA"
              f"{' x4 layers' if case.layers > 1 else ''})")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "value_scope": ("rank 0 alone: the oracle on this host's cores; the other ranks "
                            "do no work, so the value does not grow with n_gpus"),
            "config": {"workload": args.workload + ": " + WORKLOADS[args.workload]},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def time_cache_append(dev, hbm_peak, launches=40):
    """The cache-append step (new tokens into the caches) on a prefill chunk: 8192 tokens of
    Di = 128 fp32 indexer keys and 576-wide bf16 latent rows into a contiguous 65536-row
    cache, eight input sets rotating over disjoint rows so that each launch's ~24 MB miss
    L2; CUDA events around a graph replay of `launches` launches after warm-up."""
    import torch
    from sparse_attention_29_b300 import capi
    n, Di, D, sets = 8192, 128, 576, 8
    g = torch.Generator(device=dev).manual_seed(5)
    k_new = [torch.randn(n, Di, device=dev, generator=g) for _ in range(sets)]
    c_new = [torch.randint(-32768, 32767, (n, D), device=dev, dtype=torch.int16, generator=g)
             for _ in range(sets)]
    seq = torch.zeros(n, dtype=torch.int32, device=dev)
    pos = [torch.arange(i * n, (i + 1) * n, dtype=torch.int32, device=dev) for i in range(sets)]
    rows = n * sets
    k8 = torch.zeros(rows, Di, dtype=torch.uint8, device=dev)
    ks = torch.zeros(rows, dtype=torch.float32, device=dev)
    kv = torch.zeros(rows, D, dtype=torch.int16, device=dev)
    seq_start = torch.zeros(1, dtype=torch.int32, device=dev)
    layout = capi.make_layout(rows, seq_start=seq_start)

    def launch(i):
        j = i % sets
        capi.dsa_cache_append(k_new[j], c_new[j], seq, pos[j], n, 1, Di, D, layout, k8, ks, kv)
    for i in range(2 * sets):
        launch(i)
    torch.cuda.synchronize()
    # the launches are captured into one CUDA graph and replayed, so that the host's
    # per-call cost does not read as device time
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap):
        with torch.cuda.graph(graph, stream=cap):
            for i in range(launches):
                launch(i)
    graph.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    graph.replay()
    b.record()
    torch.cuda.synchronize()
    st, code = capi.dsa_device_error()
    us = a.elapsed_time(b) / launches * 1e3
    per_token = Di * 4 + D * 2 + 8 + Di + 4 + D * 2
    gbs = n * per_token / (us * 1e-6) / 1e9
    return {"tokens": n, "Di": Di, "D": D, "us_per_launch": us, "bytes_per_token": per_token,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak},
            "device_check": "ok" if st == capi.DSA_OK else f"code {code:#x}",
            "timing": "CUDA-graph replay of the launches between events, inputs rotating "
                      "over 8 sets (> L2)"}


def cpu_baseline(workload, budget_s=12.0):
    """The oracle as it stands, on a bounded sample of the workload (rank 0, N=1)."""
    import oracle
    from sparse_attention_29_b300 import inputs
    oracle.build()
    p = dict(inputs.PRESETS[workload])
    if workload == "ragged_decode":
        p["lengths"] = [inputs.ragged_lengths(16, 1024, 200000, p["seed"])[0]]
    elif workload == "prefill_8k":
        p["T"] = 1
    else:
        p["lengths"] = p["lengths"][:1]
    case = inputs.make_case(workload + "-sample", **p)
    t0 = time.perf_counter()
    n = 0
    while True:
        if case.layers > 1:
            oracle.indexshare_group(case)
        else:
            oracle.dsa_layer(case)
        n += case.rows
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} query row(s) of {workload} (context {case.lengths[0]}), "
                      f"fp64 indexer + top-k + MLA, {dt:.1f} s"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_32k", choices=sorted(WORKLOADS))
    ap.add_argument("--sets", type=int, default=3, help="rotating input sets")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the other workloads measured beside the decode batch")
    ap.add_argument("--profile", action="store_true",
                    help="lean run for profiler captures: one input set, no clock pre-roll, "
                         "no per-kernel loops, graph replay, e2e or CPU baseline")
    ap.add_argument("--rows", type=int, default=0,
                    help="prefill workloads: query rows per sequence (the last ROWS positions; "
                         "a smaller case of the same kernel, e.g. for profiler captures)")
    ap.add_argument("--fused", action="store_true",
                    help="prefill workloads: the step uses the fused indexer + top-k")
    ap.add_argument("--two-call", action="store_true",
                    help="decode: the step runs top-k and sparse MLA as two calls (the "
                         "API's other form) instead of the one-call decode")
    ap.add_argument("--append-only", action="store_true",
                    help="only the cache-append measurement (one JSON object; for profiler "
                         "captures of that kernel)")
    args = ap.parse_args()
    world, rank, local = dist_setup()
    if args.warmup < 3:
        args.warmup = 3

    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    import torch.distributed as dist
    from sparse_attention_29_b300 import build as libbuild
    from sparse_attention_29_b300 import capi
    from sparse_attention_29_b300.pipeline import DsaLayer

    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    libbuild.build()
    capi.load()
    if args.append_only:
        hbm_peak = load_peaks()[0]
        print(json.dumps({"cache_append": time_cache_append(dev, hbm_peak)}), flush=True)
        return 0

    # baseline CPU timing first (before the GPU is busy; host cores only)
    cpu_base = None
    if args.profile:
        args.sets, args.no_cpu_baseline, args.no_e2e = 1, True, True
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu_base = cpu_baseline(args.workload)

    sets = [make_workload(args.workload, dev, seed_offset=1000 * rank + 17 * i, rows=args.rows)
            for i in range(args.sets)]
    layers = [DsaLayer(c) for c in sets]
    # every set's per-query inputs and outputs as views of one device buffer each (the
    # end-to-end measurement moves each with one copy)
    packed = [pack_io(lay) for lay in layers]
    case = sets[0]
    shared = case.layers > 1
    stream = torch.cuda.current_stream()

    def step(lay):
        if shared:
            lay.run_shared()
        elif args.fused and case.T > 1:
            lay.run_fused()
        elif args.two_call:
            lay.indexer()
            lay.topk()
            lay.mla()
        else:
            lay.run()

    # launches per step: counted below from the kernel nodes of a captured step; before
    # that (and if capture is unavailable) the calls' nominal count: the indexer, the top-k
    # (inside the sparse MLA kernel in decode when the row fits), the sparse MLA, and a
    # merge kernel when a row needs more splits than a cluster holds
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    launches_per_step = 3 + (1 if layers[0].ws_bytes and case.rows * 8 < sms else 0)
    for i in range(args.warmup):
        step(layers[i % len(layers)])
    torch.cuda.synchronize()
    layers[0].check_device_error()

    # ---- timed region: K whole steps, bracketed by a barrier and synchronize ------------
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        # untimed pre-roll of the same steps, so that the clock samples see this load
        t_stop, i = time.time() + (0.0 if args.profile else 1.0), 0
        while time.time() < t_stop:
            step(layers[i % len(layers)])
            i += 1
            if i % 16 == 0:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        for i in range(args.steps):
            step(layers[i % len(layers)])
        end.record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    total_ms = max_over_ranks(start.elapsed_time(end), world, dev)
    ms_per_step = total_ms / args.steps
    layers[0].check_device_error()

    # ---- per-kernel durations: each call type launched K times back to back (its inputs
    # are the previous steps' outputs), graph-replayed between events (kernel_times) ------
    if args.profile:  # no further launches after the timed steps
        k_idx = k_topk = k_mla = float("nan")
        k_fused = None
    else:
        mla_call = (lambda lay: lay.mla_shared()) if shared else (lambda lay: lay.mla())
        k_idx, k_topk, k_mla = kernel_times(
            layers, stream, args.steps, [lambda lay: lay.indexer(), lambda lay: lay.topk(), mla_call])
        k_fused = None
        if case.T == 1 and not shared:  # top-k and sparse MLA in one call, as the step runs them
            (k_fused,) = kernel_times(layers, stream, args.steps, [lambda lay: lay.topk_mla()])

    # ---- the same K steps replayed from a CUDA graph of the C-ABI calls ----------------
    graph_ms = None
    graphs = None
    try:
        if args.profile:
            raise RuntimeError("skipped in a profile run")
        graphs = []
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            for lay in layers:
                lay.stream = cap
                step(lay)  # warm the per-kernel attribute set-up outside capture
            torch.cuda.synchronize()
            for lay in layers:
                g = torch.cuda.CUDAGraph(keep_graph=True)  # kept for the node count below
                with torch.cuda.graph(g, stream=cap):
                    step(lay)
                g.instantiate()
                graphs.append(g)
        for lay in layers:
            lay.stream = None
        for i in range(args.warmup):
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for i in range(args.steps):
            graphs[i % len(graphs)].replay()
        g1.record(stream)
        torch.cuda.synchronize()
        graph_ms = g0.elapsed_time(g1) / args.steps
        layers[0].check_device_error()
        counted = kernels_in_graph(graphs[0])
        if counted:
            launches_per_step = counted
    except Exception as exc:  # graphs are an extra measurement; the step time stands
        graph_ms = f"unavailable: {type(exc).__name__}: {exc}"[:200]
        graphs = None
        for lay in layers:
            lay.stream = None

    b_idx, b_topk, b_mla = per_query_bytes(case)
    step_bytes = b_idx + b_topk + b_mla - scores_in_step(case)
    q_tokens = case.rows
    value = job_rate(q_tokens, world, ms_per_step)

    # ---- e2e: host (pinned) inputs -> C-ABI calls -> host result, every step ----------
    # A serving loop's pipeline: each input set's per-query inputs live in one pinned host
    # buffer and one device buffer (views of it feed the calls), its outputs likewise, so
    # a step is one upload, the C-ABI calls and one download.  As a serving loop does, the
    # C-ABI calls of each input set's step are captured once into a CUDA graph and the
    # graph is replayed per step (host submission per step: one launch instead of three
    # calls).  The upload of a step runs on one copy stream and the download of the
    # previous one on another while a step computes; events keep a set's buffers from
    # being reused before the step that last used them (and the download of its outputs)
    # is done.
    e2e = None
    if not args.no_e2e:
        # Page-locked host buffers from cudaHostAlloc, filled by one thread (memmove), then
        # the host caches are flushed by writing a larger scratch buffer: on this machine
        # an upload whose source lines are still dirty in other cores' caches (written by
        # torch's multi-threaded copy) ran at 10-12 GB/s, from memory at ~50 GB/s.
        host_in = [HostBuffer(ib.numel(), ib.dtype) for ib, _ in packed]
        host_out = [HostBuffer(ob.numel(), ob.dtype) for _, ob in packed]
        for hb, (ib, _) in zip(host_in, packed):
            hb.fill_from(ib.cpu().contiguous())
        flush_host_caches()
        h2d = packed[0][0].numel() * packed[0][0].element_size()
        d2h = packed[0][1].numel() * packed[0][1].element_size()
        n_sets = len(layers)
        h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
        computed = [torch.cuda.Event() for _ in range(n_sets)]
        uploaded = [torch.cuda.Event() for _ in range(n_sets)]
        downloaded = [torch.cuda.Event() for _ in range(n_sets)]
        used = [False] * n_sets

        def e2e_step(i):
            j = i % n_sets
            (in_dev, out_dev), lay = packed[j], layers[j]
            if used[j]:
                h2d_stream.wait_event(computed[j])
            host_in[j].upload(in_dev, h2d_stream)
            uploaded[j].record(h2d_stream)
            stream.wait_event(uploaded[j])
            if used[j]:
                stream.wait_event(downloaded[j])
            if graphs is not None:
                graphs[j].replay()
            else:
                step(lay)
            computed[j].record(stream)
            d2h_stream.wait_event(computed[j])
            host_out[j].download(out_dev, d2h_stream)
            downloaded[j].record(d2h_stream)
            used[j] = True

        for i in range(args.warmup):
            e2e_step(i)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        h2d_stream.wait_stream(stream)
        d2h_stream.wait_stream(stream)
        t_host = time.perf_counter()
        for i in range(args.steps):
            e2e_step(i)
        host_us = (time.perf_counter() - t_host) / args.steps * 1e6
        stream.wait_stream(d2h_stream)
        e2.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(s2.elapsed_time(e2), world, dev) / args.steps
        layers[0].check_device_error()
        # the host link on its own: one upload and one download of a step's buffers
        def copy_us(copy, n=10):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            copy()
            torch.cuda.synchronize()
            a.record(stream)
            for _ in range(n):
                copy()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) / n * 1e3
        up_us = copy_us(lambda: host_in[0].upload(packed[0][0], stream))
        down_us = copy_us(lambda: host_out[0].download(packed[0][1], stream))
        e2e = {"value": job_rate(q_tokens, world, e2e_ms), "unit": UNIT,
               "host_link": {"h2d_us": up_us, "h2d_gbs": h2d / up_us / 1e3,
                             "d2h_us": down_us, "d2h_gbs": d2h / down_us / 1e3},
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "host_submit_us_per_step": host_us,
               "pipelined": "one packed upload and one packed download per step (page-locked "
                            "host buffers from cudaHostAlloc), on two copy streams while a "
                            "step computes",
               "step_submission": ("the C-ABI calls of each input set's step captured once "
                                   "into a CUDA graph, replayed per step") if graphs is not None
                                  else "the C-ABI calls, eagerly"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    hbm_peak, bf16_peak, peak_src = load_peaks()
    roof, rooflines = step_rooflines(case, args, k_idx, k_topk, k_mla, k_fused, shared,
                                     hbm_peak, bf16_peak, peak_src)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3+bf16 (fp32 accumulate)",
        "data": "synthetic (seeded, drawn on device)",
        "config": {"workload": args.workload + ": " + WORKLOADS[args.workload],
                   "batch": case.B, "rows": case.rows, "context": case.lengths[0] if len(set(case.lengths)) == 1 else "ragged",
                   "k": case.k, "layers": case.layers, "page_size": case.page_size,
                   "l2": f"inputs larger than L2, {args.sets} rotating input sets",
                   "parallelism": f"replicas x{world}",
                   "step_calls": ("indexer, top-k and MLA over shared layers" if shared else
                                  "fused indexer + top-k, then MLA" if args.fused and case.T > 1
                                  else "indexer, top-k, MLA" if args.two_call or case.T > 1
                                  else "indexer, then top-k + MLA in one call")},
        "hbm_tbs": step_bytes / (ms_per_step * 1e-3) / 1e12,
        **({"hbm_note": "per-row algorithmic bytes: the rows of one sequence share its keys "
                        "and many selected rows, so much of this is served from L2"}
           if case.T > 1 else {}),
        "hbm_frac": step_bytes / (ms_per_step * 1e-3) / 1e9 / hbm_peak,
        "step_bytes": step_bytes,
        "kernel_ms": {"indexer": k_idx, "topk": k_topk, "sparse_mla": k_mla,
                      **({"topk_and_sparse_mla_one_call": k_fused} if k_fused else {})},
        "roofline": roof,
        "rooflines": rooflines,
        "gpu_launches": launches_per_step * args.steps,
        "graph_replay": (graph_ms if isinstance(graph_ms, str) else
                         {"ms_per_step": graph_ms,
                          "value": job_rate(q_tokens, world, graph_ms), "unit": UNIT}),
        "clocks": clocks.summary(),
    }
    if e2e:
        line["e2e"] = e2e
    if not args.profile and world == 1:
        try:  # the step that feeds the path, measured beside it (not part of `value`)
            line["cache_append"] = time_cache_append(dev, hbm_peak)
        except Exception as exc:
            line["cache_append"] = f"unavailable: {type(exc).__name__}: {exc}"[:200]
    if not args.profile and world == 1 and not args.no_extras and args.workload == "decode_32k":
        # the other serving workloads, each measured on its own (not part of `value`)
        others = {}
        for name in ("prefill_8k", "ragged_decode", "indexshare_paged"):
            try:
                others[name] = measure_other_workload(name, dev, max(5, min(args.steps, 20)),
                                                      3, hbm_peak, bf16_peak)
            except Exception as exc:
                others[name] = f"unavailable: {type(exc).__name__}: {exc}"[:200]
        line["other_workloads"] = others
        try:  # MLA's two modes on short-context chunked prefill
            line["mha_vs_mqa"] = measure_mha_vs_mqa(dev)
        except Exception as exc:
            line["mha_vs_mqa"] = f"unavailable: {type(exc).__name__}: {exc}"[:200]
        try:  # the host-tier working set on the decode batch
            line["hisparse"] = measure_hisparse(layers[0], dev, hbm_peak)
        except Exception as exc:
            line["hisparse"] = f"unavailable: {type(exc).__name__}: {exc}"[:200]
    if cpu_base:
        line["cpu_baseline"] = cpu_base
    if args.profile:
        line["note"] = "profile run (lean, for profiler captures): not a measurement"
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
