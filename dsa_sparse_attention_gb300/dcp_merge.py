"""Exact one-round top-k merge across context-parallel ranks (host protocol).

vLLM K3.1 Pro day-0 post, "An exact top-k merge with 10x less traffic": under
decode context parallelism each of W ranks holds 1/W of a request's tokens and
can rank only those.  Instead of sending its whole local top-2048, each rank
sends its best ceil(1.5 * 2048 / W) candidates taken straight from the BF16
scores, each packed with its score into 32 bits.  Every rank radix-selects the
same global top-k from the gathered candidates.  The merge stays exact: when a
rank holds more of the global top-k than it sent, the select detects it and that
rank resends its full local top-k for that row.  "Low-latency decode: a fused
DSA decode path" moves these messages through mailboxes inside the kernels, with
no collective on the path; here the mailbox is a key-value store (a
torch.distributed TCPStore) and every wait on it is bounded: a rank that posts
nothing in time makes the merge return DSA_ERR_TIMEOUT instead of hanging.

Readings taken where the post is silent:
 * Ranks hold contiguous position ranges (rank r before rank r + 1), so the
   lower-position tie rule is "lower rank, then lower local position".
 * The 32-bit word is (order-preserving 16-bit key of the BF16 score) << 16 |
   (0xFFFF - g), g = the candidate's rank-major, position-ascending index in the
   gathered set, so a larger word is a better candidate and equal scores go to
   the lower position; the ids stay local (g indexes the sender's list).
 * A rank that may hold more top-k members than it sent is detected as: every candidate the rank sent was
   selected and the rank has tokens it did not send.  Then none of its unsent
   tokens can be excluded, so it resends its full local top-k for that row; a
   rank with an unselected candidate cannot hold a better unsent one.
 * Exactness is with respect to the BF16-rounded scores the candidates carry.

Everything here is host code over numpy arrays: the component is the protocol
(packing, radix select, overflow detection and resend, bounded mailbox waits),
exercised by multi-process tests on the CPU.
"""
import math
import pickle
from datetime import timedelta

import numpy as np

DSA_OK = 0
DSA_ERR_TIMEOUT = -5


# -------------------------------------------------------------- score words

def bf16_bits(scores):
    """float scores -> bf16 bit patterns (round to nearest even), uint16."""
    f = np.ascontiguousarray(np.asarray(scores, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_value(bits):
    """bf16 bit patterns -> float64 values."""
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def order_key16(bits):
    """Order-preserving 16-bit key of a bf16 value (-0 and +0 share a key)."""
    b = np.asarray(bits, dtype=np.uint16)
    b = np.where(b == 0x8000, np.uint16(0), b)
    neg = (b & 0x8000) != 0
    return np.where(neg, ~b, b | 0x8000).astype(np.uint16)


def pack_words(keys16, g):
    """Candidate words: key in the high half, 0xFFFF - g in the low half."""
    return (np.asarray(keys16, np.uint32) << 16) | (0xFFFF - np.asarray(g, np.uint32))


def radix_select_top(words, k):
    """Boolean mask of the k largest of distinct uint32 words, by radix select
    (most significant 8-bit digit first, one histogram per digit)."""
    w = np.asarray(words, dtype=np.uint32)
    n = w.size
    if k >= n:
        return np.ones(n, dtype=bool)
    if k <= 0:
        return np.zeros(n, dtype=bool)
    prefix, mask, need = 0, 0, k
    for shift in (24, 16, 8, 0):
        live = (w & np.uint32(mask)) == np.uint32(prefix)
        digits = ((w[live] >> shift) & 0xFF).astype(np.int64)
        hist = np.bincount(digits, minlength=256)
        above = 0
        for d in range(255, -1, -1):
            if above + hist[d] >= need:
                break
            above += hist[d]
        need -= above
        prefix |= d << shift
        mask |= 0xFF << shift
    # words are distinct: exactly k are >= the threshold word `prefix`
    sel = w >= np.uint32(prefix)
    assert int(sel.sum()) == k
    return sel


# ------------------------------------------------------------ one rank's side

def local_order(keys16):
    """Local indices ordered best first: key descending, position ascending."""
    n = keys16.size
    return np.lexsort((np.arange(n), -keys16.astype(np.int64)))


def candidates_per_rank(k, world):
    return int(math.ceil(1.5 * k / world))


# --------------------------------------------------------------- the merge

class StoreMailbox:
    """Per-(step, round, rank) messages in a key-value store; `gather` waits for
    every rank's message for at most `limit_s` seconds."""

    def __init__(self, store, rank, world, limit_s=1.0):
        self.store, self.rank, self.world, self.limit = store, rank, world, float(limit_s)

    def _key(self, step, rnd, r):
        return f"dsa_merge/{step}/{rnd}/{r}"

    def post(self, step, rnd, payload):
        self.store.set(self._key(step, rnd, self.rank), pickle.dumps(payload))

    def gather(self, step, rnd):
        """List of every rank's payload, or None when a rank posted nothing in time."""
        keys = [self._key(step, rnd, r) for r in range(self.world)]
        try:
            self.store.wait(keys, timedelta(seconds=self.limit))
        except Exception:   # the store's timeout (RuntimeError / DistStoreError)
            return None
        return [pickle.loads(self.store.get(k)) for k in keys]


class ThreadMailbox:
    """In-process mailbox for W simulated ranks running in threads; `gather`
    waits (bounded, like StoreMailbox) until every rank has posted."""

    def __init__(self, world, limit_s=1.0):
        import threading
        self.world, self.limit = world, float(limit_s)
        self.box = {}
        self.cv = threading.Condition()

    def view(self, rank):
        outer = self

        class _View:
            def post(self, step, rnd, payload):
                with outer.cv:
                    outer.box[(step, rnd, rank)] = payload
                    outer.cv.notify_all()

            def gather(self, step, rnd):
                keys = [(step, rnd, r) for r in range(outer.world)]
                with outer.cv:
                    if not outer.cv.wait_for(lambda: all(k in outer.box for k in keys), timeout=outer.limit):
                        return None
                    return [outer.box[k] for k in keys]
        return _View()


def _select(lists, k):
    """Global selection from per-rank candidate lists.

    lists[r] = (keys16 [n_r], local positions [n_r]) sorted by position.
    Returns (selected: list over ranks of boolean masks, rank_all_selected flags)."""
    sizes = [len(lst[0]) for lst in lists]
    stride = max(sizes + [1])
    keys = np.concatenate([lst[0] for lst in lists]) if sizes else np.zeros(0, np.uint16)
    g = np.concatenate([r * stride + np.arange(n) for r, n in enumerate(sizes)]).astype(np.int64)
    if g.size and g.max() > 0xFFFF:
        raise ValueError("candidate ids do not fit 16 bits")
    sel = radix_select_top(pack_words(keys, g), k)
    out, off = [], 0
    for n in sizes:
        out.append(sel[off:off + n])
        off += n
    return out


def merge_rows(mailbox, rank, world, scores_local, offset, k, step=0):
    """This rank's part of the exact merge for T rows.

    scores_local: float [T, n_local] scores of this rank's tokens (positions
    offset .. offset + n_local - 1; -inf marks positions beyond a row's context).
    Returns (status, idx [T, k] global positions ascending, -1 padded, stats)."""
    bits = bf16_bits(scores_local)
    T, n_local = bits.shape
    valid = np.isfinite(np.asarray(scores_local, dtype=np.float32))
    m = candidates_per_rank(k, world)
    keys_all = order_key16(bits)
    orders = []
    round1 = []
    for t in range(T):
        nv = int(valid[t].sum())
        kt = keys_all[t, :nv]
        order = local_order(kt)
        orders.append(order)
        sent = np.sort(order[:m])                      # best m, listed by position
        round1.append((kt[sent], sent + offset, nv))
    mailbox.post(step, 1, {"offset": offset, "rows": round1})
    got = mailbox.gather(step, 1)
    if got is None:
        return DSA_ERR_TIMEOUT, None, None
    # every rank evaluates the same selection and the same overflow flags
    lists = [[(g["rows"][t][0], g["rows"][t][1]) for g in got] for t in range(T)]
    counts = [[g["rows"][t][2] for g in got] for t in range(T)]
    flags = np.zeros((T, world), dtype=bool)
    for t in range(T):
        sel = _select(lists[t], k)
        for r in range(world):
            n_sent = len(lists[t][r][0])
            flags[t, r] = n_sent > 0 and bool(sel[r].all()) and counts[t][r] > n_sent
    resends = int(flags.sum())
    if resends:
        full = {}
        for t in np.nonzero(flags[:, rank])[0]:
            nv = int(valid[t].sum())
            kt = keys_all[t, :nv]
            sent = np.sort(orders[t][:min(k, nv)])     # the full local top-k
            full[int(t)] = (kt[sent], sent + offset)
        mailbox.post(step, 2, full)
        got2 = mailbox.gather(step, 2)
        if got2 is None:
            return DSA_ERR_TIMEOUT, None, None
        for r in range(world):
            for t, lst in got2[r].items():
                lists[t][r] = lst
    idx = np.full((T, k), -1, dtype=np.int64)
    for t in range(T):
        sel = _select(lists[t], k)
        pos = np.concatenate([lists[t][r][1][sel[r]] for r in range(world)])
        pos = np.sort(pos)
        idx[t, :pos.size] = pos
    stats = {"candidates_per_rank": m, "resent_rows": resends,
             "words_sent_round1": int(sum(len(r[0]) for r in round1))}
    return DSA_OK, idx, stats
