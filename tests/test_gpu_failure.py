"""The failure path on the GPU, without a fault: every wait inside the kernels is
bounded, and past its limit it records DSA_ERR_TIMEOUT and returns.  The
diagnostic entry point runs that same bounded wait on a barrier that nothing
completes, with a short limit (a fraction of a millisecond), so the wait really
runs out; the status must say so, and the device must still run a layer step
correctly afterwards."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dsa_sparse_attention_gb300.build import build
    build()


def test_bounded_wait_runs_out_and_reports_timeout():
    import dsa_sparse_attention_gb300 as dsa
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    for limit in (100_000, 2_000_000):
        dsa.dsa_selftest_wait_timeout(ws, limit, stream)
        assert dsa.dsa_check(ws, stream) == -5        # DSA_ERR_TIMEOUT
        assert dsa.dsa_check(ws, stream) == 0         # read and cleared


def test_device_usable_after_a_timeout():
    import dsa_sparse_attention_gb300 as dsa
    from dsa_sparse_attention_gb300 import workloads as W
    from dsa_sparse_attention_gb300.harness import DeviceWorkload
    from tests.parity import OracleCache, check_mla, check_topk
    wl = W.make_workload([3000, 700], 1, seed=61, permute=True, pool_rows=70)
    dw = DeviceWorkload(wl)
    dsa.dsa_selftest_wait_timeout(dw.ws, 100_000)
    idx, out, lse = dw.layer_step()
    assert dsa.dsa_check(dw.ws) == -5                 # the earlier timeout, nothing else
    idx, out, lse = dw.layer_step()
    assert dsa.dsa_check(dw.ws) == 0
    oc = OracleCache(wl)
    g = idx.cpu().numpy()
    check_topk(oc, g, [0, 1], dw.topk)
    check_mla(oc, g, out.float().cpu().numpy(), lse.cpu().numpy(), [0, 1])
