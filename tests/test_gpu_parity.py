"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Small cases span several key tiles, ragged tails and the degenerate cases
(context 1, contexts straddling a 64-token block and the 2048 boundary, fewer
tokens than k); the full-size decode configuration runs in the launch
configuration the benchmark times.
"""
import numpy as np
import pytest
import torch

from dsa_sparse_attention_gb300 import workloads as W
from tests.parity import OracleCache, check_mla, check_scores, check_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dsa_sparse_attention_gb300.build import build
    build()


def _dev(wl, topk=None, flags=0):
    from dsa_sparse_attention_gb300.harness import DeviceWorkload
    return DeviceWorkload(wl, topk=topk, flags=flags)


def _np(x):
    return x.float().cpu().numpy() if x.dtype == torch.bfloat16 else x.cpu().numpy()


def _run_all(wl, topk=None, tokens=None, check_split=True):
    from dsa_sparse_attention_gb300 import dsa_check
    dw = _dev(wl, topk)
    k = dw.topk
    idx, out, lse = dw.layer_step()
    torch.cuda.synchronize()
    assert dsa_check(dw.ws) == 0
    oc = OracleCache(wl)
    tokens = list(range(wl.num_tokens)) if tokens is None else tokens
    g_idx, g_out, g_lse = _np(idx), _np(out), _np(lse)
    scores = dw.indexer_scores()
    torch.cuda.synchronize()
    worst_s = check_scores(oc, _np(scores), tokens)
    subs = check_topk(oc, g_idx, tokens, k)
    worst_m = check_mla(oc, g_idx, g_out, g_lse, tokens)
    if check_split:
        # the three separate calls give exactly what the fused step gives
        idx2 = dw.topk_of(scores)
        out2, lse2 = dw.sparse_mla_of(idx2)
        torch.cuda.synchronize()
        assert np.array_equal(_np(idx2), g_idx)
        assert np.array_equal(_np(out2), g_out) and np.array_equal(_np(lse2), g_lse)
    assert dsa_check(dw.ws) == 0
    return dict(score_err=worst_s, tie_subs=subs, mla=worst_m)


def test_cfg0_tiny_decode():
    r = _run_all(W.config(0))
    print(r)


def test_ragged_multi_request_decode():
    lens = [5000, 1, 64, 65, 2047, 2048, 2049, 3000, 129]
    wl = W.make_workload(lens, 1, seed=11, permute=True, pool_rows=300)
    _run_all(wl)


def test_decode_batch_planned_by_kernel():
    # 160 single-token requests: more than the scorer plans inside itself, so the
    # planning kernel lays out the tiles; the layer step's histogram hand-off and the
    # separate calls must agree, and sampled tokens match the oracle.
    rng = np.random.default_rng(41)
    lens = [int(x) for x in rng.integers(1, 4000, size=160)]
    lens[:4] = [1, 2048, 2049, 3999]
    wl = W.make_workload(lens, 1, seed=41, permute=True)
    _run_all(wl, tokens=[0, 1, 2, 3, 50, 99, 159])


def test_mtp_groups_of_six():
    wl = W.make_workload([3000, 5000, 9001], 6, seed=12, permute=True, pool_rows=300)
    _run_all(wl)


def test_prefill_chunk():
    base, new = 3000, 300
    wl = W.make_workload([base + new], new, seed=13, permute=True)
    _run_all(wl, tokens=[0, 1, 2, 7, 8, 150, 298, 299])


@pytest.mark.parametrize("bs", [16, 32, 128, 256])
def test_block_sizes(bs):
    wl = W.make_workload([3001, 700], 1, seed=14, block_size=bs, permute=True, pool_rows=400)
    _run_all(wl)


@pytest.mark.parametrize("bs,frac", [(64, 0.5), (256, 0.5), (64, 1.0)])
def test_mixed_sign_key_scales(bs, frac):
    # The key scale multiplies the decoded key, so a negative scale turns
    # ReLU(q . code * scale) into scale * min(q . code, 0); the scorer takes that
    # branch per key.  Half (or all) of the keys get a negative scale.
    wl = W.make_workload([5000, 700, 2049, 129], 1, seed=44, block_size=bs, permute=True,
                         pool_rows=(5000 + 700 + 2049 + 129) // bs + 8, negative_scale_frac=frac)
    _run_all(wl)


def test_mixed_sign_key_scales_mtp_groups():
    # the same through the grouped scorer (six query tokens share each key tile)
    wl = W.make_workload([3000, 4100], 6, seed=45, permute=True, pool_rows=120, negative_scale_frac=0.5)
    _run_all(wl)


@pytest.mark.parametrize("k", [1, 7, 100, 300, 700, 1000])
def test_topk_sizes(k):
    wl = W.make_workload([4000, 90, 5], 1, seed=15, permute=True)
    _run_all(wl, topk=k)


def test_all_scores_tied_takes_lowest_positions():
    # w = 0 makes every score exactly 0: the top-k is then positions 0..k-1.
    wl = W.make_workload([3000, 2500], 1, seed=16)
    wl.w[:] = 0
    dw = _dev(wl)
    idx, out, lse = dw.layer_step()
    g = _np(idx)
    assert np.array_equal(g[0], np.arange(2048)) and np.array_equal(g[1], np.arange(2048))
    check_mla(OracleCache(wl), g, _np(out), _np(lse), [0, 1])


@pytest.mark.parametrize("lens", [[65536, 40000, 9000], [6000, 8000]])
def test_layer_step_all_scores_tied_long_rows(lens):
    # w = 0: every score is 0, so the whole row shares the threshold key.  Inside a
    # layer step the top-k starts from the scorer's histogram (one full bin), finds more
    # candidates than it gathers and resolves the cut through the cluster (or, for rows
    # of at most 8,192 scores, inside one CTA); the result is the lowest k positions.
    wl = W.make_workload(lens, 1, seed=29)
    wl.w[:] = 0
    dw = _dev(wl)
    toks = list(range(len(lens)))
    for _ in range(2):   # the second step starts from the histograms the first left zeroed
        idx, out, lse = dw.layer_step()
        g = _np(idx)
        for t in toks:
            assert np.array_equal(g[t], np.arange(2048)), f"token {t}"
    check_mla(OracleCache(wl), g, _np(out), _np(lse), toks)


@pytest.mark.parametrize("lens", [[65536, 40000, 9000, 3000, 2049], [70000, 12345, 5, 66000]])
def test_layer_step_dirty_workspace_hint(lens):
    # Inside a layer step the top-k starts from top-digit histograms the scorer
    # leaves in the workspace, and leaves them zeroed.  A workspace whose bytes
    # past the status word hold garbage (here all ones) gives the top-k a wrong
    # hint, which it must detect and replace; the next step starts clean.  All
    # three steps must equal the separate calls exactly.  The second case takes the
    # multi-pass path (rows over 65,536 scores), with a row selected whole.
    wl = W.make_workload(lens, 1, seed=23)
    dw = _dev(wl)
    ref_scores = dw.indexer_scores()
    ref_idx = _np(dw.topk_of(ref_scores))
    ref_out, ref_lse = (_np(x) for x in dw.sparse_mla_of(torch.from_numpy(ref_idx).cuda()))
    for dirty in (True, False, True):
        if dirty:
            dw.ws[256:].fill_(255)
        idx, out, lse = dw.layer_step()
        torch.cuda.synchronize()
        assert np.array_equal(_np(idx), ref_idx)
        assert np.array_equal(_np(out), ref_out) and np.array_equal(_np(lse), ref_lse)
    check_topk(OracleCache(wl), ref_idx, list(range(wl.num_tokens)), dw.topk)


def _copy_key(wl, b, src, dsts):
    """Give positions `dsts` of request b the FP8 index key (codes and scale) of position `src`."""
    rows = wl.pool.reshape(wl.num_rows, wl.row_stride)
    bs = wl.block_size

    def loc(pos):
        return int(wl.block_table[b, pos // bs]), pos % bs

    r, sl = loc(src)
    page = rows[r, wl.idx_page_offset:]
    codes = page[sl * 128: sl * 128 + 128].copy()
    scale = page[bs * 128 + sl * 4: bs * 128 + sl * 4 + 4].copy()
    for d in dsts:
        r, sl = loc(int(d))
        page = rows[r, wl.idx_page_offset:]
        page[sl * 128: sl * 128 + 128] = codes
        page[bs * 128 + sl * 4: bs * 128 + sl * 4 + 4] = scale


@pytest.mark.parametrize("n_tied", [150, 400])
def test_layer_step_threshold_ties(n_tied):
    # Many positions of a row share the exact key whose score sits at the k-th
    # place: the layer step's top-k (starting from the scorer's histogram) must cut
    # them at the lowest positions, spread over several CTAs of the row, and equal
    # the exact selection over the GPU's own scores.
    from oracle import dsa_oracle as O
    wl = W.make_workload([65536, 30000, 5000], 1, seed=61, permute=True)
    oc = OracleCache(wl)
    rng = np.random.default_rng(61)
    for b in range(2):
        t = int(np.nonzero(wl.q_req == b)[0][0])
        n = int(wl.q_pos[t]) + 1
        sc = oc.scores(t)
        src = int(np.argsort(-sc, kind="stable")[wl.topk - 40])
        _copy_key(wl, b, src, rng.choice(np.setdiff1d(np.arange(n), [src]), n_tied, replace=False))
    dw = _dev(wl)
    for _ in range(3):   # the first step may start from an unzeroed workspace; the next ones not
        idx, out, lse = dw.layer_step()
        torch.cuda.synchronize()
        scores = _np(dw.indexer_scores())
        g_idx = _np(idx)
        for t in range(wl.num_tokens):
            n = int(wl.q_pos[t]) + 1
            ref = O.topk_select(scores[t, :n].astype(np.float64), dw.topk)
            assert np.array_equal(g_idx[t, :ref.size], ref), f"token {t}"
            assert np.all(g_idx[t, ref.size:] == -1)


@pytest.mark.parametrize("lens", [[65536, 9000, 3000, 1, 2048, 2049, 40000], [70000, 12345, 5]])
def test_topk_heavy_ties_exact(lens):
    # Scores with five distinct values (and both signs of zero): the threshold
    # key is shared by thousands of positions spread over several CTAs of a row,
    # so the lowest-position cut decides the selection, which must equal the
    # oracle's exactly.  Rows up to 65,536 scores take the one-launch cluster
    # path; the second case also runs the multi-pass path.
    from oracle import dsa_oracle as O
    wl = W.make_workload(lens, 1, seed=51, permute=True)
    dw = _dev(wl)
    rng = np.random.default_rng(51)
    sc = rng.integers(-2, 3, size=(wl.num_tokens, dw.ld)).astype(np.float32)
    sc[(sc == 0) & (rng.random(sc.shape) < 0.5)] = -0.0
    idx = _np(dw.topk_of(torch.from_numpy(sc).cuda()))
    for t in range(wl.num_tokens):
        n = int(wl.q_pos[t]) + 1
        ref = O.topk_select(sc[t, :n].astype(np.float64), dw.topk)
        assert np.array_equal(idx[t, :ref.size], ref), f"token {t} (n={n})"
        assert np.all(idx[t, ref.size:] == -1)


def _embed(big, b, alone):
    """Give request b of `big` exactly the cache and queries of request 0 of `alone`."""
    nb = (int(alone.ctx_lens[0]) + 63) // 64
    rb = big.pool.reshape(big.num_rows, big.row_stride)
    ra = alone.pool.reshape(alone.num_rows, alone.row_stride)
    rb[big.block_table[b, :nb]] = ra[alone.block_table[0, :nb]]
    t = int(np.nonzero(big.q_req == b)[0][0])
    big.q_idx[t], big.w[t], big.q[t] = alone.q_idx[0], alone.w[0], alone.q[0]
    return t


@pytest.mark.parametrize("flags", [0, 1])
def test_batch_invariance_bitwise(flags):
    # Selection never depends on the batch; with DSA_BATCH_INVARIANT (flags=1)
    # the output does not either, even when the batch size changes the default
    # split plan (40 tokens -> 8 splits by default, 1 token -> 16).
    alone = W.make_workload([3000], 1, seed=17, permute=False)
    lens = [3000 + 37 * i for i in range(40)]
    lens[5] = 3000
    big = W.make_workload(lens, 1, seed=27, permute=True)
    t = _embed(big, 5, alone)
    i1, o1, l1 = [_np(x).copy() for x in _dev(big, flags=flags).layer_step()]
    i2, o2, l2 = [_np(x).copy() for x in _dev(alone, flags=flags).layer_step()]
    assert np.array_equal(i1[t], i2[0])
    if flags:
        assert np.array_equal(o1[t], o2[0]) and np.array_equal(l1[t], l2[0])
    else:
        oc = OracleCache(alone)
        check_mla(oc, i1[t:t + 1].repeat(1, 0), o1[t:t + 1], l1[t:t + 1], [0])


def test_batch_invariance_same_split_plan_default_mode():
    # With the same split plan (batch sizes 3 and 1 both use 16 splits) the
    # default mode is bit-identical as well.
    alone = W.make_workload([3000], 1, seed=17, permute=False)
    big = W.make_workload([6000, 3000, 7000], 1, seed=37, permute=True)
    t = _embed(big, 1, alone)
    i1, o1, l1 = [_np(x).copy() for x in _dev(big).layer_step()]
    i2, o2, l2 = [_np(x).copy() for x in _dev(alone).layer_step()]
    assert np.array_equal(i1[t], i2[0])
    assert np.array_equal(o1[t], o2[0]) and np.array_equal(l1[t], l2[0])


def test_block_table_permutation_bitwise():
    a = W.make_workload([5000, 3000], 2, seed=18, permute=False, pool_rows=200)
    b = W.make_workload([5000, 3000], 2, seed=18, permute=True, pool_rows=200)
    ra = [_np(x).copy() for x in _dev(a).layer_step()]
    rb = [_np(x).copy() for x in _dev(b).layer_step()]
    for x, y in zip(ra, rb):
        assert np.array_equal(x, y)


def test_phys_slots():
    wl = W.make_workload([3000, 100], 1, seed=19, permute=True, pool_rows=100)
    dw = _dev(wl)
    scores = dw.indexer_scores()
    idx, phys = dw.topk_of(scores, with_phys=True)
    gi, gp = _np(idx), _np(phys)
    for t in range(2):
        b = wl.q_req[t]
        v = gi[t] >= 0
        exp = wl.block_table[b][gi[t][v] // 64] * 64 + gi[t][v] % 64
        assert np.array_equal(gp[t][v], exp) and np.all(gp[t][~v] == -1)


def test_bad_block_id_is_reported_not_faulted():
    from dsa_sparse_attention_gb300 import dsa_check
    wl = W.make_workload([3000], 1, seed=20, pool_rows=60)
    wl.block_table[0, 5] = wl.num_rows + 7          # outside the pool
    dw = _dev(wl)
    dw.layer_step()
    assert dsa_check(dw.ws) == -6                    # DSA_ERR_DEVICE_CHECK
    assert dsa_check(dw.ws) == 0                     # cleared


@pytest.mark.slow
def test_full_cfg1_decode_b8_64k():
    wl = W.config(1)
    r = _run_all(wl, check_split=False)
    print(r)


@pytest.mark.slow
def test_full_cfg2_mtp_b32x6_sampled():
    # 32 requests x 6 speculative query tokens, contexts log-uniform in [16K, 256K];
    # oracle on every request's first and last query token.
    wl = W.config(2)
    toks = sorted(set(int(np.nonzero(wl.q_req == b)[0][i]) for b in range(wl.num_reqs) for i in (0, -1)))
    r = _run_all(wl, tokens=toks, check_split=False)
    print(r)


@pytest.mark.slow
def test_full_cfg4_prefill_8192_on_131072_sampled():
    # 8192 new queries on a 131,072-token cache; oracle on 64 seeded positions
    # including the first two and the last.
    wl = W.config(4)
    rng = np.random.default_rng(4)
    toks = sorted(set([0, 1, 8191] + list(rng.choice(8192, 61, replace=False))))
    r = _run_all(wl, tokens=toks, check_split=False)
    print(r)


# ------------------------------------------------- MXFP4 keys / NVFP4 latents

def test_mxfp4_keys_fp8_latents():
    wl = W.make_workload([5000, 700, 2049], 1, seed=41, idx_fmt=W.IDX_MXFP4, permute=True, pool_rows=200)
    _run_all(wl)


def test_fp8_keys_nvfp4_latents():
    wl = W.make_workload([5000, 700, 2049], 1, seed=42, lat_fmt=W.LAT_NVFP4, permute=True, pool_rows=200)
    _run_all(wl)


def test_combine_split_count_not_a_multiple_of_four():
    # 48 query tokens with NVFP4 latents: the attention runs 6 splits per token, so
    # the combine's last 4-split copy of each token reaches past its splits (into the
    # next token's, and past the end of the partials for the last token)
    wl = W.make_workload([1500 + 211 * i for i in range(8)], 6, seed=46, lat_fmt=W.LAT_NVFP4, permute=True,
                         pool_rows=400)
    assert wl.num_tokens == 48
    _run_all(wl, tokens=[0, 5, 17, 30, 46, 47])


def test_mxfp4_nvfp4_mtp_groups():
    wl = W.make_workload([3000, 4100], 6, seed=43, idx_fmt=W.IDX_MXFP4, lat_fmt=W.LAT_NVFP4, permute=True,
                         pool_rows=200)
    _run_all(wl)


def test_mxfp4_queries_and_keys():
    # MXFP4 index queries (codes through the 4-bit tensor copy, exponents as the
    # MMA's B scales) against MXFP4 keys, one token per request; 165 key tiles over
    # 152 CTAs, so some CTAs cross from one token's tiles to the next (the second
    # query buffer and its scale columns)
    wl = W.make_workload([5000, 700, 2049, 129, 3000, 3000, 4000, 2500], 1, seed=51, idx_fmt=W.IDX_MXFP4,
                         q_fmt=W.Q_MXFP4, permute=True, pool_rows=400)
    _run_all(wl)


def test_mxfp4_queries_wide_exponents_mtp_groups():
    # every (token, head, block) exponent redrawn over 2^-9 .. 2^9: a wrong head,
    # block or token column of the B scales would show; six tokens per request
    # (groups of two tokens in the scorer) and NVFP4 latents
    wl = W.make_workload([3000, 4100, 333], 6, seed=52, idx_fmt=W.IDX_MXFP4, lat_fmt=W.LAT_NVFP4, q_fmt=W.Q_MXFP4,
                         permute=True, pool_rows=200)
    T = wl.num_tokens
    rng = np.random.default_rng(3)
    wl.q_idx[T * 32 * 64:] = rng.integers(118, 137, size=T * 32 * 4).astype(np.uint8)
    _run_all(wl)


@pytest.mark.slow
def test_full_cfg3_decode_1m_mxfp4_nvfp4():
    # one request, 1,048,576-token context, MXFP4 index keys and NVFP4 latents
    wl = W.config(3)
    r = _run_all(wl, check_split=False)
    print(r)


@pytest.mark.parametrize("packed,pinned,misalign,lens", [
    (True, True, 0, [5000, 1, 2049, 300]),
    (False, True, 0, [5000, 1, 2049, 300]),
    (False, False, 0, [5000, 1, 2049, 300]),
    (True, True, 0, [700, 3001, 1]),
    (False, True, 4, [700, 3001, 1]),
    (True, True, 4, [700, 3001, 1]),
])
def test_layer_step_from_host_buffers(packed, pinned, misalign, lens):
    # the host-buffer call copies in, runs the same step and copies out: its host
    # results equal the device call's bit for bit.  Inputs packed into one buffer
    # each side (one copy) or each in its own allocation; page-locked host memory
    # (moved by the library's copy kernel) or pageable (cudaMemcpyAsync); host
    # arrays 16-byte aligned or 4 bytes off; three tokens leave byte tails (12-byte
    # position arrays, a packed total that is not a multiple of 16)
    from dsa_sparse_attention_gb300 import dsa_check
    from dsa_sparse_attention_gb300.harness import HostStep
    wl = W.make_workload(lens, 1, seed=17, permute=True, pool_rows=120)
    dw = _dev(wl)
    idx, out, lse = (_np(x) for x in dw.layer_step())
    hs = HostStep(dw, packed=packed, pinned=pinned, misalign=misalign)
    for t in hs.dev:   # the step must read what the call copied in, not what was there
        t.zero_()
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    for _ in range(2):
        hs.out_host.zero_()
        hs.step(stream)
        stream.synchronize()
        assert np.array_equal(hs.idx_host.numpy(), idx)
        assert np.array_equal(hs.out_host.float().numpy(), out)
        assert np.array_equal(hs.lse_host.numpy(), lse)
    assert dsa_check(dw.ws) == 0
