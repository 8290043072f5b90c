"""dsa_topk_noalloc: the top-k entry point that takes no workspace.

It is for callers that cannot allocate device memory; the scratch of its long
rows is a fixed array inside the library.  Called through the C ABI, it must
give exactly what dsa_topk (with a caller workspace) gives.  Rows of at most
65,536 scores take the one-launch cluster kernel and use none of the array;
longer rows take the three-pass path, whose histograms, candidate lists and
per-chunk counts live in the array, so the workloads here have rows above
65,536.  Two calls in a row on one stream must both be exact: the second finds
the first call's histograms and counts in the array and must clear them.  This
file is collected last so that a run stopping at the first failure has already
run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    import dsa_sparse_attention_gb300 as dsa
    return dsa.library().dsa_topk_noalloc


def _case(ctx, qpr, seed, ties=False):
    """A batch over synthetic scores (no cache pool: only block ids are needed).
    Request b has ctx[b] tokens and its last qpr[b] positions are queries."""
    import dsa_sparse_attention_gb300 as dsa
    rng = np.random.default_rng(seed)
    bs = 64
    nblk = [(c + bs - 1) // bs for c in ctx]
    bt_stride = max(nblk)
    perm = rng.permutation(sum(nblk) + 5).astype(np.int32)
    bt = np.full((len(ctx), bt_stride), -1, np.int32)
    off = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = perm[off:off + n]
        off += n
    q_req = np.concatenate([np.full(q, b, np.int32) for b, q in enumerate(qpr)])
    q_pos = np.concatenate([np.arange(c - q, c, dtype=np.int32) for c, q in zip(ctx, qpr)])
    ld = (max(ctx) + 3) // 4 * 4
    scores = rng.standard_normal((q_req.size, ld)).astype(np.float32)
    if ties:   # thousands of equal scores around the threshold of one row
        scores[-1, 1::7] = np.float32(1.875)
    dev = {k: torch.from_numpy(v).cuda() for k, v in
           dict(bt=bt, ctx=np.asarray(ctx, np.int32), q_req=q_req, q_pos=q_pos, scores=scores).items()}
    layout = dsa.make_layout(None, perm.size, 64 * (132 + 576), 0, 64 * 132, bs)
    batch = dsa.make_batch(dev["q_req"], dev["q_pos"], dev["ctx"], dev["bt"], max(ctx))
    return layout, batch, dev, scores, q_pos


def _ref(layout, batch, dev, topk=2048):
    import dsa_sparse_attention_gb300 as dsa
    ws = dsa.alloc_workspace(layout, batch, topk)
    T, ld = dev["scores"].shape
    idx = torch.empty(T, topk, dtype=torch.int32, device="cuda")
    phys = torch.empty_like(idx)
    dsa.dsa_topk(layout, batch, dev["scores"], ld, topk, idx, phys, ws=ws)
    torch.cuda.synchronize()
    return idx.cpu().numpy(), phys.cpu().numpy()


def _noalloc(layout, batch, dev, stream, topk=2048):
    T, ld = dev["scores"].shape
    idx = torch.full((T, topk), -7, dtype=torch.int32, device="cuda")
    phys = torch.full_like(idx, -7)
    st = _noalloc_fn()(ctypes.byref(layout), ctypes.byref(batch), dev["scores"].data_ptr(), ld, topk,
                       idx.data_ptr(), phys.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
    return st, idx, phys


def test_noalloc_long_rows_match_workspace_topk_twice():
    from dsa_sparse_attention_gb300.build import build
    build()
    from oracle import dsa_oracle as O
    stream = torch.cuda.Stream()
    # one 1-token request at 70,000 tokens, one 6-token request at 131,072 (ties in its last row)
    layout, batch, dev, scores, q_pos = _case([70000, 131072], [1, 6], seed=31, ties=True)
    ref_idx, ref_phys = _ref(layout, batch, dev)
    for t in (0, 6):   # the oracle's exact top-k on a row of each request
        n = int(q_pos[t]) + 1
        assert np.array_equal(ref_idx[t], O.topk_select(scores[t, :n].astype(np.float64), 2048))
    got = []
    for call in range(2):   # back to back on one stream: the second call finds the first's leftovers
        st, idx, phys = _noalloc(layout, batch, dev, stream)
        assert st == 0, f"call {call}: status {st}"
        got.append((idx, phys))
    stream.synchronize()
    for call, (idx, phys) in enumerate(got):
        assert np.array_equal(idx.cpu().numpy(), ref_idx), f"call {call}: indices differ"
        assert np.array_equal(phys.cpu().numpy(), ref_phys), f"call {call}: slots differ"
    # other scores after those two: the array's contents from before must not leak in
    l2, b2, d2, _, _ = _case([90000], [3], seed=32)
    r2_idx, r2_phys = _ref(l2, b2, d2)
    st, idx, phys = _noalloc(l2, b2, d2, stream)
    assert st == 0
    stream.synchronize()
    assert np.array_equal(idx.cpu().numpy(), r2_idx) and np.array_equal(phys.cpu().numpy(), r2_phys)


def test_noalloc_short_rows_need_no_scratch():
    # 150 query tokens of one request at 65,536 tokens: the long-row scratch
    # would exceed the fixed array, but these rows take the cluster kernel,
    # which needs none, so the call is accepted and exact.
    from dsa_sparse_attention_gb300.build import build
    build()
    stream = torch.cuda.Stream()
    layout, batch, dev, _, _ = _case([65536], [150], seed=33)
    ref_idx, ref_phys = _ref(layout, batch, dev)
    st, idx, phys = _noalloc(layout, batch, dev, stream)
    assert st == 0
    stream.synchronize()
    assert np.array_equal(idx.cpu().numpy(), ref_idx) and np.array_equal(phys.cpu().numpy(), ref_phys)


def test_noalloc_refuses_long_row_batches_beyond_the_array():
    import dsa_sparse_attention_gb300 as dsa
    layout = dsa.make_layout(None, 20000, 64 * 708, 0, 64 * 132, 64)
    big = dsa.dsa_batch(98, 1, 0x1000, 0x2000, 0x3000, 0x4000, (1 << 20) // 64, 0, 1 << 20)
    st = _noalloc_fn()(None, ctypes.byref(big), 0x10000, 1 << 20, 2048, 0x20000, None, None)
    assert st == -4      # DSA_ERR_WORKSPACE: 98 tokens at 1M context need more than 4 MiB
