"""Seeded synthetic inputs for the DSA hot path.

This module draws random numbers and lays them out in memory. It holds none of the
method's arithmetic: no scoring, no selection, no attention. It is the one piece of code
that both the CUDA path (tests, bench) and the oracle (tests) use, so that both sides
see the same bytes.

What the inputs stand for (titles of the source pages):
  * "Inside GLM-5.3: How Sparse Attention Affects DRAM Memory TAM", §Lightning Indexer:
    multi-head indexer queries, single-head indexer keys cached like KV, a weight per
    query head.  Here: q8 [rows, Hi, Di] and k8 [tokens, Di] in fp8 e4m3 with one fp32
    scale per token, w [rows, Hi] fp32.
  * same page, §Sparse MLA and §MLA changes: MQA (absorbed) mode over a cached latent
    of d=512 plus a rope part of r=64, b=2 bytes (bf16).  Here: kv [tokens, d+r] bf16
    and q [rows, H, d+r] bf16.
  * same page, §IndexShare: several layers share one indexer; each layer keeps its own
    latent cache.  Here: `layers` copies of (q, kv), one indexer cache.
  * the pages speak of page management for the cache; the page size is not given.
    Here: an optional paged layout with a randomly permuted int32 block table.

The pages publish no dataset; every tensor is synthetic with the shapes of their
long-context serving workload.  Recipes (the seed defaults to the preset's number):
  * "int": every q/k/latent value an integer drawn uniformly from [-4, 4], indexer
    weights from {0.5, 1, 2}, all fp8 scales 1.0.  Every value is exact in e4m3 and bf16.
  * "normal": indexer q and k drawn from N(0, 1), stored as e4m3 (round to nearest even,
    saturated at +-448) with a per-token scale amax/448; weights N(0, 1)/8 in fp32;
    latent q and kv drawn from N(0, 1) and rounded to bf16.
  * "planted": as "normal", but a seeded 5% of the tokens get indexer-key coordinates
    drawn from N(3, 1), so that the top-k is not uniform over the context.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

E4M3_MAX = 448.0


@dataclass
class Case:
    """One synthetic workload, laid out as the library consumes it.

    Rows are grouped by sequence: rows b*T .. b*T+T-1 belong to sequence b, and row t
    sits at position q_pos[t] (it may look at tokens 0..q_pos[t]).  Token s of sequence
    b sits at physical row seq_start[b] + s (contiguous layout), or at
    block_table[b, s // page_size] * page_size + s % page_size (paged layout).
    """

    name: str
    kind: str
    seed: int
    B: int
    T: int
    lengths: list
    Hi: int
    Di: int
    H: int
    d: int
    r: int
    k: int
    softmax_scale: float
    layers: int
    page_size: int  # 0: contiguous
    q8: torch.Tensor = None        # [rows, Hi, Di] uint8 (e4m3 codes)
    q_scale: torch.Tensor = None   # [rows] float32
    w: torch.Tensor = None         # [rows, Hi] float32
    k8: torch.Tensor = None        # [n_phys, Di] uint8 (e4m3 codes)
    k_scale: torch.Tensor = None   # [n_phys] float32
    q: list = field(default_factory=list)   # per layer: [rows, H, d+r] bfloat16
    kv: list = field(default_factory=list)  # per layer: [n_phys, d+r] bfloat16
    q_pos: torch.Tensor = None     # [rows] int32
    seq_start: torch.Tensor = None  # [B] int32 (contiguous layout) else None
    block_table: torch.Tensor = None  # [B, pages_per_seq] int32 (paged layout) else None

    @property
    def rows(self) -> int:
        return self.B * self.T

    @property
    def D(self) -> int:
        return self.d + self.r

    @property
    def Lmax(self) -> int:
        return int(max(self.lengths))

    @property
    def pages_per_seq(self) -> int:
        return 0 if self.block_table is None else int(self.block_table.shape[1])

    @property
    def n_phys(self) -> int:
        return int(self.k8.shape[0])

    def to(self, device) -> "Case":
        """A copy with every tensor moved to `device`."""
        out = Case(**{f: getattr(self, f) for f in (
            "name", "kind", "seed", "B", "T", "lengths", "Hi", "Di", "H", "d", "r", "k",
            "softmax_scale", "layers", "page_size")})
        for f in ("q8", "q_scale", "w", "k8", "k_scale", "q_pos", "seq_start", "block_table"):
            v = getattr(self, f)
            setattr(out, f, None if v is None else v.to(device))
        out.q = [x.to(device) for x in self.q]
        out.kv = [x.to(device) for x in self.kv]
        return out


def _generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _to_e4m3_per_token(x: torch.Tensor):
    """Store float32 rows as e4m3 codes with one scale per row (amax/448), RNE, satfinite."""
    flat = x.reshape(x.shape[0], -1)
    amax = flat.abs().amax(dim=1).clamp_min(1e-30)
    scale = (amax / E4M3_MAX).to(torch.float32)
    y = (flat / scale[:, None]).clamp(-E4M3_MAX, E4M3_MAX)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(x.shape)
    return codes.contiguous(), scale.contiguous()


def _ints(shape, g, device):
    return torch.randint(-4, 5, shape, generator=g, device=device, dtype=torch.int32).to(torch.float32)


def make_case(name="custom", *, kind="normal", seed=0, lengths, T=1, Hi=64, Di=128, H=64,
              d=512, r=64, k=2048, softmax_scale=None, layers=1, page_size=0,
              device="cpu") -> Case:
    """Draw one workload.

    lengths: context length of each sequence (tokens 0..L-1 are cached).  With T query
    rows per sequence the rows sit at positions L-T .. L-1 (T=1: a decode step).
    """
    lengths = [int(x) for x in lengths]
    B = len(lengths)
    if any(L < T for L in lengths):
        raise ValueError("every context must hold its T query positions")
    if softmax_scale is None:
        # the SDPA head dim of the absorbed model: qk-nope 192 + rope 64 = 256
        softmax_scale = 1.0 / 16.0
    g = _generator(seed, device)
    rows = B * T
    D = d + r

    # Logical token layout.  Contiguous: sequences back to back.  Paged: every sequence
    # owns pages_per_seq pages of page_size tokens; the block table then permutes pages.
    if page_size:
        pps = max(1, -(-max(lengths) // page_size))
        n_log = B * pps * page_size
        log_start = [b * pps * page_size for b in range(B)]
    else:
        n_log = sum(lengths)
        log_start = list(np.cumsum([0] + lengths[:-1]))

    # Indexer keys and queries.
    if kind == "int":
        k_f = _ints((n_log, Di), g, device)
        q_f = _ints((rows, Hi, Di), g, device)
        k8 = k_f.to(torch.float8_e4m3fn).view(torch.uint8)
        q8 = q_f.to(torch.float8_e4m3fn).view(torch.uint8)
        k_scale = torch.ones(n_log, dtype=torch.float32, device=device)
        q_scale = torch.ones(rows, dtype=torch.float32, device=device)
        choice = torch.tensor([0.5, 1.0, 2.0], device=device)
        w = choice[torch.randint(0, 3, (rows, Hi), generator=g, device=device)]
    elif kind in ("normal", "planted"):
        k_f = torch.randn((n_log, Di), generator=g, device=device)
        if kind == "planted":
            # 5% of tokens (seeded choice) carry keys drawn from N(3, 1).
            n_plant = int(round(0.05 * n_log))
            pick = torch.randperm(n_log, generator=g, device=device)[:n_plant]
            k_f[pick] = torch.randn((n_plant, Di), generator=g, device=device) + 3.0
        q_f = torch.randn((rows, Hi, Di), generator=g, device=device)
        k8, k_scale = _to_e4m3_per_token(k_f)
        q8, q_scale = _to_e4m3_per_token(q_f)
        w = torch.randn((rows, Hi), generator=g, device=device) / 8.0
    else:
        raise ValueError(f"unknown kind {kind!r}")
    del k_f, q_f

    # Latent caches and absorbed queries, one pair per layer.
    qs, kvs = [], []
    for _ in range(layers):
        if kind == "int":
            kv = _ints((n_log, D), g, device).to(torch.bfloat16)
            q = _ints((rows, H, D), g, device).to(torch.bfloat16)
        else:
            kv = torch.randn((n_log, D), generator=g, device=device).to(torch.bfloat16)
            q = torch.randn((rows, H, D), generator=g, device=device).to(torch.bfloat16)
        qs.append(q.contiguous())
        kvs.append(kv.contiguous())

    q_pos = torch.tensor([L - T + i for L in lengths for i in range(T)], dtype=torch.int32,
                         device=device)

    case = Case(name=name, kind=kind, seed=seed, B=B, T=T, lengths=lengths, Hi=Hi, Di=Di,
                H=H, d=d, r=r, k=k, softmax_scale=float(softmax_scale), layers=layers,
                page_size=page_size, q8=q8.contiguous(), q_scale=q_scale.contiguous(),
                w=w.to(torch.float32).contiguous(), q=qs, q_pos=q_pos)
    if page_size:
        pps = n_log // (B * page_size)
        n_pages = B * pps
        perm = torch.randperm(n_pages, generator=g, device=device).to(torch.int32)
        block_table = perm.reshape(B, pps).contiguous()
        # physical page perm[j] holds logical page j
        inv = torch.empty_like(perm)
        inv[perm.long()] = torch.arange(n_pages, dtype=torch.int32, device=device)
        src_rows = (inv.long()[:, None] * page_size +
                    torch.arange(page_size, device=device)[None, :]).reshape(-1)
        case.k8 = k8[src_rows].contiguous()
        case.k_scale = k_scale[src_rows].contiguous()
        case.kv = [kv[src_rows].contiguous() for kv in kvs]
        case.block_table = block_table
    else:
        case.k8 = k8.contiguous()
        case.k_scale = k_scale.contiguous()
        case.kv = kvs
        case.seq_start = torch.tensor(log_start, dtype=torch.int32, device=device)
    return case


def unpage(case: Case) -> Case:
    """The same workload in the contiguous layout (sequences back to back).

    Moves bytes only: token s of sequence b is copied from its physical paged row.
    """
    if not case.page_size:
        return case
    dev = case.k8.device
    bt = case.block_table.long()
    rows = []
    for b, L in enumerate(case.lengths):
        s = torch.arange(L, device=dev)
        rows.append(bt[b, s // case.page_size] * case.page_size + s % case.page_size)
    src = torch.cat(rows)
    out = Case(**{f: getattr(case, f) for f in (
        "name", "kind", "seed", "B", "T", "lengths", "Hi", "Di", "H", "d", "r", "k",
        "softmax_scale", "layers")}, page_size=0)
    out.q8, out.q_scale, out.w, out.q, out.q_pos = case.q8, case.q_scale, case.w, case.q, case.q_pos
    out.k8 = case.k8[src].contiguous()
    out.k_scale = case.k_scale[src].contiguous()
    out.kv = [kv[src].contiguous() for kv in case.kv]
    out.seq_start = torch.tensor(np.cumsum([0] + case.lengths[:-1]), dtype=torch.int32,
                                 device=dev)
    return out


def ragged_lengths(B: int, lo: int, hi: int, seed: int):
    """Context lengths drawn log-uniformly from [lo, hi] (seeded PCG64)."""
    rng = np.random.default_rng(seed)
    return [int(round(math.exp(x))) for x in rng.uniform(math.log(lo), math.log(hi), B)]


# The five workloads of the method's serving scenario, by name.  The number in each
# entry is its default seed.
PRESETS = {
    # 1 sequence, context 512, the last 4 positions query; indexer 4 heads x 32;
    # top-64; MLA 4 heads, latent 64 + rope 16, softmax scale 1/8; integer values.
    "tiny_int": dict(seed=1, kind="int", lengths=[512], T=4, Hi=4, Di=32, H=4, d=64, r=16,
                     k=64, softmax_scale=1.0 / 8.0),
    # 32 sequences x 32768 context, one decode query each.
    "decode_32k": dict(seed=2, kind="normal", lengths=[32768] * 32, T=1),
    # 16 sequences, contexts log-uniform in [1024, 200000]; 5% planted keys.
    "ragged_decode": dict(seed=3, kind="planted", lengths=None, T=1),
    # chunked prefill: 8192 new rows after a 57344-token prefix (65536 in total).
    "prefill_8k": dict(seed=4, kind="normal", lengths=[65536], T=8192),
    # IndexShare group of 4 layers, 64 sequences x 16384, 64-token pages.
    "indexshare_paged": dict(seed=5, kind="normal", lengths=[16384] * 64, T=1, layers=4,
                             page_size=64),
}


def preset(name: str, seed=None, device="cpu") -> Case:
    p = dict(PRESETS[name])
    if seed is not None:
        p["seed"] = seed
    if p.get("lengths") is None:
        p["lengths"] = ragged_lengths(16, 1024, 200000, p["seed"])
    return make_case(name, device=device, **p)
