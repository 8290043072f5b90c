"""dsa_topk_noalloc: the top-k entry point that takes no workspace.

It is for callers that cannot allocate device memory; its scratch is a fixed
array inside the library.  Called through the C ABI, it must give exactly what
dsa_topk (with a caller workspace) gives, on two calls in a row (the second call
finds the first call's leftovers in the shared array).  This file is collected
last so that a run stopping at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    import dsa_sparse_attention_gb300 as dsa
    fn = dsa.library().dsa_topk_noalloc
    P = ctypes.POINTER
    fn.restype = ctypes.c_int32
    fn.argtypes = [P(dsa.dsa_kv_layout), P(dsa.dsa_batch), ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                   ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return fn


def test_noalloc_topk_matches_workspace_topk_twice():
    from dsa_sparse_attention_gb300.build import build
    build()
    from dsa_sparse_attention_gb300 import workloads as W
    from dsa_sparse_attention_gb300.harness import DeviceWorkload
    fn = _noalloc_fn()
    stream = torch.cuda.current_stream()
    wl = W.make_workload([9000, 700, 3001, 4097], [1, 1, 6, 1], seed=31, permute=True, pool_rows=400)
    dw = DeviceWorkload(wl)
    scores = dw.indexer_scores()
    ref_idx, ref_phys = dw.topk_of(scores, with_phys=True)
    torch.cuda.synchronize()
    for call in range(2):
        idx = torch.full_like(ref_idx, -7)
        phys = torch.full_like(ref_phys, -7)
        st = fn(ctypes.byref(dw.layout), ctypes.byref(dw.batch), scores.data_ptr(), scores.shape[1], dw.topk,
                idx.data_ptr(), phys.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), ref_idx.cpu().numpy()), f"call {call}: indices differ"
        assert np.array_equal(phys.cpu().numpy(), ref_phys.cpu().numpy()), f"call {call}: slots differ"
    # a batch needing more scratch than the fixed array is refused up front
    big = dw.batch
    big_batch = type(big)(4096, big.num_reqs, big.q_req, big.q_pos, big.ctx_lens, big.block_table,
                          big.bt_stride, 0, 1 << 20)
    big_batch.bt_stride = (1 << 20) // 64
    st = fn(None, ctypes.byref(big_batch), scores.data_ptr(), 1 << 20, dw.topk, idx.data_ptr(), None,
            ctypes.c_void_p(stream.cuda_stream))
    assert st == -4      # DSA_ERR_WORKSPACE
