"""dsa_sparse_mla_decode_noalloc (split-KV partials in the library's fixed static scratch,
no allocation, no workspace) against dsa_sparse_mla_decode with a caller workspace.

Both entry points run the same kernels with the same split of the keys, so their outputs
must be identical bit for bit.  Two calls in a row on the same inputs must each reproduce
the workspace entry point: the second shows that nothing left in the scratch by the first
call (or by an earlier call of another shape) changes the result.  This file sorts last
so that it also runs after every other GPU test in one session.
"""
import numpy as np
import pytest
import torch

from sparse_attention_29_b300 import build, capi, inputs
from sparse_attention_29_b300.pipeline import DsaLayer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    capi.load()
    assert torch.cuda.is_available()


def _random_idx(case, seed, frac_invalid=0.02):
    g = np.random.default_rng(seed)
    idx = np.full((case.rows, case.k), -1, np.int32)
    for t in range(case.rows):
        n = int(case.q_pos[t]) + 1
        m = min(n, case.k)
        idx[t, :m] = np.sort(g.choice(n, size=m, replace=False))
        idx[t, g.random(case.k) < frac_invalid] = -1
    return torch.from_numpy(idx)


@pytest.mark.parametrize("lengths,k,splits", [
    ([5000, 3000, 2100], 2048, True),   # three rows: more splits than a cluster holds
    ([2500] * 32, 2048, True),          # 32 rows x 4 splits, merged in a cluster through the scratch
    ([700] * 150, 512, False),          # more rows than SMs: no split, no scratch used
])
def test_noalloc_decode_matches_workspace_entry(lengths, k, splits):
    case = inputs.make_case(seed=500 + len(lengths), lengths=lengths, T=1, k=k)
    idx = _random_idx(case, seed=len(lengths)).cuda()
    lay = DsaLayer(case.to("cuda"))
    c = lay.case
    assert (lay.ws_bytes > 0) == splits
    assert lay.ws_bytes <= capi.DSA_NOALLOC_SCRATCH_BYTES
    lay.mla(idx=idx)  # the workspace entry point
    torch.cuda.synchronize()
    lay.check_device_error()
    ref_lse = lay.lse[0]
    for call in range(2):
        out = torch.full((c.rows, c.H, c.d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((c.rows, c.H), float("nan"), dtype=torch.float32, device="cuda")
        capi.dsa_sparse_mla_decode_noalloc(c.q[0], c.kv[0], lay.layout, idx, c.B, c.H, c.d,
                                           c.r, c.k, c.softmax_scale, out, lse)
        torch.cuda.synchronize()
        st, code = capi.dsa_device_error()
        assert st == capi.DSA_OK, (call, hex(code))
        assert torch.isfinite(out.float()).all() and not torch.isnan(lse).any(), call
        assert torch.equal(out, lay.out[0]), call
        assert torch.equal(lse, ref_lse), call
