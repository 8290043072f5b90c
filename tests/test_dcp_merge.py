"""The exact one-round top-k merge across context-parallel ranks (the vLLM post,
"An exact top-k merge with 10x less traffic"), on the CPU: W ranks each hold a
contiguous 1/W of a row's tokens, send their best ceil(1.5 k / W) BF16 candidates
packed into 32-bit words through a mailbox, radix-select the same global top-k,
and resend a full local top-k for a row where they hold more of it than they
sent.  The merged set must equal the single-rank exact top-k of the BF16 scores
(the oracle's top-k, ties to the lower position) bit for bit, the resend path
must run, and a rank that posts nothing in time must make the bounded waits
return DSA_ERR_TIMEOUT."""
import os
import socket
import threading
import time

import numpy as np
import pytest
import torch

from dsa_sparse_attention_gb300 import dcp_merge as M
from oracle import dsa_oracle as O


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _reference(row_f32, k):
    """Single-rank exact top-k of the BF16-rounded scores (torch's cast, the oracle's select)."""
    vals = torch.from_numpy(np.ascontiguousarray(row_f32, dtype=np.float32)).to(torch.bfloat16).double().numpy()
    sel = O.topk_select(vals, k)
    out = np.full(k, -1, np.int64)
    out[:sel.size] = sel
    return out


def _shards(n, world):
    """Contiguous shards of n positions: (offset, size) per rank (the last ones may be shorter)."""
    per = -(-n // world)
    return [(min(r * per, n), max(0, min(per, n - r * per))) for r in range(world)]


def _run_threads(rows, world, k, limit=5.0, mutate=None):
    """Every rank's merge_rows in its own thread over a shared in-process mailbox."""
    T, n = rows.shape
    box = M.ThreadMailbox(world, limit)
    res = [None] * world
    per = -(-n // world)

    def go(r):
        lo, hi = r * per, min(n, (r + 1) * per)
        local = np.full((T, per), -np.inf, np.float32)
        local[:, :hi - lo] = rows[:, lo:hi]
        if mutate:
            mutate(r)
        res[r] = M.merge_rows(box.view(r), r, world, local, lo, k)

    th = [threading.Thread(target=go, args=(r,)) for r in range(world)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    return res


# ------------------------------------------------------------- the pieces

def test_bf16_rounding_matches_torch_and_order_key_is_monotone():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(5000).astype(np.float32) * 10, np.float32([0.0, -0.0, 1.0, -1.0]),
                        np.float32([1.00390625, 1.01171875, -3.0078125])])   # exact ties at half an ulp
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(M.bf16_bits(x), want)
    v = M.bf16_value(M.bf16_bits(x))
    key = M.order_key16(M.bf16_bits(x)).astype(np.int64)
    for i in range(0, x.size - 1):
        a, b = v[i], v[i + 1]
        assert (a < b) == (key[i] < key[i + 1]) and (a == b) == (key[i] == key[i + 1])


@pytest.mark.parametrize("seed", range(4))
def test_radix_select_is_the_k_largest(seed):
    rng = np.random.default_rng(seed)
    w = rng.choice(1 << 32, size=3000, replace=False).astype(np.uint32)
    w[:50] = (w[:50] & 0xFFFF0000) | np.arange(50)   # shared high digits
    for k in (1, 2, 999, 2999, 3000, 4000):
        sel = M.radix_select_top(w, k)
        want = np.zeros(w.size, bool)
        want[np.argsort(w)[::-1][:min(k, w.size)]] = True
        assert np.array_equal(sel, want)


# -------------------------------------------- the merge, ranks as threads

@pytest.mark.parametrize("world", [2, 4, 8])
def test_merge_equals_single_rank_topk(world):
    rng = np.random.default_rng(world)
    T, n = 5, 9000
    rows = rng.standard_normal((T, n)).astype(np.float32)
    rows[1] = rng.integers(-3, 4, size=n).astype(np.float32)          # thousands of exact ties
    rows[2, ::2] = -0.0
    rows[3] = np.float32(1.0) + rng.integers(0, 4, size=n).astype(np.float32) * np.float32(2.0 ** -9)  # ties after bf16
    for k in (1, 100, 2048):
        for r, (st, idx, stats) in enumerate(_run_threads(rows, world, k)):
            assert st == M.DSA_OK
            for t in range(T):
                assert np.array_equal(idx[t], _reference(rows[t], k)), (world, k, r, t)
            assert stats["candidates_per_rank"] == -(-3 * k // (2 * world))


def test_rank_holding_most_of_the_topk_resends():
    # rank 0 of 4 holds every one of the best 2048 tokens: it sent only 768, all of
    # them selected, so it must resend its full local top-k and the result stays exact
    world, k, n = 4, 2048, 12000
    rng = np.random.default_rng(7)
    rows = rng.standard_normal((3, n)).astype(np.float32)
    rows[0, :3000] += 100.0
    rows[2] = 0.0                                                      # all tied: lowest positions win
    res = _run_threads(rows, world, k)
    for st, idx, stats in res:
        assert st == M.DSA_OK and stats["resent_rows"] >= 2
        for t in range(3):
            assert np.array_equal(idx[t], _reference(rows[t], k))


def test_short_rows_and_empty_shards():
    # fewer tokens than k (all selected, -1 padded), and ranks whose shard is empty
    world, k = 4, 2048
    rng = np.random.default_rng(9)
    rows = np.full((3, 3000), -np.inf, np.float32)
    rows[0, :1500] = rng.standard_normal(1500)
    rows[1, :3] = [1.0, 1.0, -2.0]
    rows[2, :3000] = rng.standard_normal(3000)
    for st, idx, _ in _run_threads(rows, world, k):
        assert st == M.DSA_OK
        for t, n in enumerate((1500, 3, 3000)):
            assert np.array_equal(idx[t], _reference(rows[t, :n], k))


def test_silent_rank_times_out_in_threads():
    world = 2
    rows = np.random.default_rng(1).standard_normal((2, 4000)).astype(np.float32)
    box = M.ThreadMailbox(world, limit_s=0.3)
    t0 = time.perf_counter()
    st, idx, _ = M.merge_rows(box.view(0), 0, world, rows[:, :2000], 0, 2048)   # rank 1 never posts
    assert st == M.DSA_ERR_TIMEOUT and idx is None and time.perf_counter() - t0 < 5


# -------------------------------------------- ranks as processes (TCPStore)

def _proc(rank, world, port, rows, k, limit, delays, out):
    from datetime import timedelta
    import torch.distributed as dist
    store = dist.TCPStore("127.0.0.1", port, world, rank == 0, timedelta(seconds=120), wait_for_workers=False)
    # every process has started before the merge's own (short) waits begin
    store.set(f"up/{rank}", "1")
    store.wait([f"up/{r}" for r in range(world)], timedelta(seconds=120))
    n = rows.shape[1]
    per = -(-n // world)
    lo, hi = rank * per, min(n, (rank + 1) * per)
    local = np.full((rows.shape[0], per), -np.inf, np.float32)
    local[:, :hi - lo] = rows[:, lo:hi]
    box = M.StoreMailbox(store, rank, world, limit)
    for step, delay in enumerate(delays[rank]):
        if delay is None:          # this rank leaves before the step (it never posts)
            break
        time.sleep(delay)
        st, idx, _ = M.merge_rows(box, rank, world, local, lo, k, step=step)
        out[(rank, step)] = (st, None if idx is None else idx.tolist())
    store.set(f"done/{rank}", "1")
    if rank == 0:                  # the store's server lives in rank 0: wait for the others
        try:
            store.wait([f"done/{r}" for r in range(world)], timedelta(seconds=120))
        except Exception:
            pass


def _spawn(world, rows, k, limit, delays):
    import torch.multiprocessing as mp
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_proc, args=(world, _free_port(), rows, k, limit, delays, out), nprocs=world, join=True)
    return dict(out)


@pytest.mark.parametrize("world", [2, 4])
def test_merge_across_processes(world):
    rng = np.random.default_rng(40 + world)
    rows = rng.standard_normal((3, 7000)).astype(np.float32)
    rows[1, :2500] += 50.0                                             # one rank holds the top-k: resend
    k = 2048
    out = _spawn(world, rows, k, 10.0, [[0.0]] * world)
    for r in range(world):
        st, idx = out[(r, 0)]
        assert st == M.DSA_OK
        for t in range(3):
            assert np.array_equal(np.asarray(idx[t]), _reference(rows[t], k))


def test_dropped_and_delayed_ranks_time_out():
    # step 0: rank 1 posts 0.2 s late (inside the 1.5 s limit): exact;
    # step 1: rank 1 posts 3 s late: rank 0's bounded wait gives up with DSA_ERR_TIMEOUT;
    # a third run where rank 1 leaves before the step: rank 0 times out as well
    rows = np.random.default_rng(5).standard_normal((2, 5000)).astype(np.float32)
    out = _spawn(2, rows, 2048, 1.5, [[0.0, 0.0], [0.2, 3.0]])
    st0, idx0 = out[(0, 0)]
    assert st0 == M.DSA_OK and np.array_equal(np.asarray(idx0[1]), _reference(rows[1], 2048))
    assert out[(0, 1)][0] == M.DSA_ERR_TIMEOUT
    out = _spawn(2, rows, 2048, 1.0, [[0.0], [None]])
    assert out[(0, 0)] == (M.DSA_ERR_TIMEOUT, None)
