"""GPU parity of MLA in MHA mode (dsa_mla_up_project, dsa_sparse_mha_prefill).

The up-projection is checked element by element against an fp64 product of the same bf16
inputs (within the bf16 rounding of the result plus the fp32 accumulation bound); the
attention against the fp64 oracle of MHA mode fed the same index sets, within the
attention bounds of tests/parity.py.  Cases: a chunked-prefill tail with rows that see
more than k tokens (sparse) and rows that see fewer (dense), a ragged row tile, two
sequences, both value widths.
"""
import numpy as np
import pytest
import torch

import oracle
from parity import check_mla, cpu
from sparse_attention_29_b300 import build, capi, inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    capi.load()
    oracle.build()
    assert torch.cuda.is_available()


def random_idx(case, k, seed):
    g = np.random.default_rng(seed)
    idx = np.full((case.rows, k), -1, np.int32)
    for t in range(case.rows):
        n = int(case.q_pos[t]) + 1
        m = min(n, k)
        idx[t, :m] = np.sort(g.choice(n, size=m, replace=False))
    return idx


@pytest.mark.parametrize("lengths,T,H,vd,k", [
    ([3000], 40, 4, 128, 2048),        # sparse rows (3000 > k) in one ragged row tile
    ([2100, 1500], 150, 2, 256, 2048),  # two sequences; 150 rows: two row tiles; dense rows
])
def test_mha_mode_matches_oracle(lengths, T, H, vd, k):
    d, r, dn = 512, 64, 192
    case = inputs.make_case(seed=91 + T, lengths=lengths, T=T, H=H, k=k)
    g = torch.Generator().manual_seed(T)
    w_uk = (torch.randn(H, dn, d, generator=g) / 16).to(torch.bfloat16)
    w_uv = (torch.randn(H, vd, d, generator=g) / 16).to(torch.bfloat16)
    q_mha = torch.randn(case.rows, H, dn + r, generator=g).to(torch.bfloat16)
    idx = random_idx(case, k, seed=T)
    dev = "cuda"
    kv = case.kv[0].to(dev)
    n = kv.shape[0]
    k_up = torch.empty((n, H * dn), dtype=torch.bfloat16, device=dev)
    v_up = torch.empty((n, H * vd), dtype=torch.bfloat16, device=dev)
    capi.dsa_mla_up_project(kv, n, d + r, d, w_uk.reshape(H * dn, d).to(dev), H * dn, k_up)
    capi.dsa_mla_up_project(kv, n, d + r, d, w_uv.reshape(H * vd, d).to(dev), H * vd, v_up)
    torch.cuda.synchronize()
    # the up-projection against an fp64 product of the same bf16 values
    lat = case.kv[0][:, :d].double()
    for got, w in ((k_up, w_uk.reshape(H * dn, d)), (v_up, w_uv.reshape(H * vd, d))):
        ref = lat @ w.double().T
        bound = (lat.abs() @ w.double().abs().T) * (d * 2.0 ** -23)
        err = (cpu(got).double() - ref).abs()
        assert torch.all(err <= 2.0 ** -8 * ref.abs() + bound + 1e-30)
    ws = capi.dsa_mha_workspace_bytes(case.B, case.T, case.Lmax)
    w_buf = torch.empty(ws, dtype=torch.uint8, device=dev)
    out = torch.full((case.rows, H, vd), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((case.rows, H), float("nan"), dtype=torch.float32, device=dev)
    layout = capi.make_layout(n, seq_start=case.seq_start.to(dev))
    capi.dsa_sparse_mha_prefill(q_mha.to(dev), k_up, v_up, kv, layout, torch.from_numpy(idx).to(dev),
                                case.q_pos.to(dev), case.B, case.T, H, d, r, dn, vd, k, case.Lmax,
                                case.softmax_scale, out, lse, w_buf, ws)
    torch.cuda.synchronize()
    st, code = capi.dsa_device_error()
    assert st == capi.DSA_OK, hex(code)
    ref_out, ref_lse = oracle.sparse_mha(case, idx, w_uk, w_uv, q_mha)
    check_mla(out, lse, ref_out, ref_lse)
