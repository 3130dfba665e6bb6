"""The bounded waits on the GPU: a wait that runs out ends its kernel with a status the
host reads, and the device stays usable.  The probe waits on a barrier that nothing
completes (no fault, no trap, no endless loop); both of its waiters give up after the
time limit, the device error word holds the probe's code, and an exact decode step run
afterwards still matches the oracle bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from parity import cpu
from sparse_attention_29_b300 import build, capi, inputs
from sparse_attention_29_b300.pipeline import DsaLayer

pytestmark = pytest.mark.gpu

DSA_OK, DSA_ERR_DEVICE = 0, 5
KID_PROBE, ERR_WAIT_TIMEOUT = 8, 1
LIMIT_NS = 2_000_000_000  # the time limit of every in-kernel wait


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    capi.load()
    oracle.build()
    assert torch.cuda.is_available()


def test_wait_runs_out_reports_and_the_device_stays_usable():
    torch.cuda.synchronize()
    assert capi.dsa_device_error()[0] in (DSA_OK, DSA_ERR_DEVICE)  # start from a clear word
    res = torch.full((4,), 7, dtype=torch.int64, device="cuda")
    capi.dsa_wait_probe(res)
    st, code = capi.dsa_device_error()
    assert st == DSA_ERR_DEVICE and code == (KID_PROBE << 16) | ERR_WAIT_TIMEOUT
    done0, done1, ns0, ns1 = cpu(res).tolist()
    assert done0 == 0 and done1 == 0          # neither barrier completed
    assert LIMIT_NS <= ns0 < LIMIT_NS + 500_000_000
    assert LIMIT_NS - 1_000_000 <= ns1 < LIMIT_NS + 500_000_000  # stopped by the flag or its own limit
    assert capi.dsa_device_error() == (DSA_OK, 0)  # read and cleared

    # an exact decode step afterwards: integer inputs, so scores and index sets are exact
    case = inputs.preset("tiny_int")
    lay = DsaLayer(case.to("cuda"))
    lay.run()
    torch.cuda.synchronize()
    lay.check_device_error()
    ref = oracle.indexer_scores(case)
    g = cpu(lay.scores).double().numpy()
    vis = np.arange(case.Lmax)[None, :] <= case.q_pos.numpy()[:, None]
    assert np.array_equal(g[vis], ref[vis])
    assert np.array_equal(cpu(lay.idx).numpy(), oracle.topk(ref, case.q_pos.numpy(), case.k))
