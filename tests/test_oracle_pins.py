"""Pins of the float64 oracle to facts fixed outside it.

Each test checks the oracle against something the vLLM post on Kimi K3.1 Pro
or mathematics fix: format tables (OCP definitions, cross-checked with torch's
own casts), the post's byte arithmetic (*KV cache footprint*), a hand-worked example with closed-form answers, brute
force on tiny inputs, a library routine for the dense special case, and
invariants.  None of them retypes the oracle's own formula.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import dsa_oracle as O
from dsa_sparse_attention_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def oracle_layout(wl):
    return O.Layout(wl.pool, wl.row_stride, wl.idx_page_offset, wl.lat_page_offset,
                    wl.block_size, wl.idx_fmt, wl.lat_fmt)


# ------------------------------------------------------------------ formats

def test_e4m3_table_matches_ocp_and_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode_e4m3(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}           # S.1111.111 only
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x38] == 1.0
    assert ours[0x80] == 0.0 and math.copysign(1, ours[0x80]) == -1


def test_e2m1_table_is_the_ocp_fp4_set():
    vals = oracle.decode_e2m1(np.arange(16, dtype=np.uint8))
    assert list(vals[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(vals[8:]) == [-v for v in vals[:8]]


def test_e8m0_and_bf16():
    e = oracle.decode_e8m0(np.array([0, 1, 126, 127, 128, 254, 255], dtype=np.uint8))
    assert list(e[:6]) == [2.0 ** -127, 2.0 ** -126, 0.5, 1.0, 2.0, 2.0 ** 127]
    assert np.isnan(e[6])
    x = torch.randn(1000, dtype=torch.float32).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.decode_bf16(bits), x.to(torch.float64).numpy())


def test_nibble_order_low_first():
    from oracle.formats import unpack_nibbles
    assert list(unpack_nibbles(np.array([0x21, 0xF7], dtype=np.uint8))) == [1, 2, 7, 15]


def test_mxfp4_and_nvfp4_roundtrip_of_representable_vectors():
    # MXFP4 key whose values are exactly representable: block j holds
    # e2m1 magnitudes times 2^(j-1); quantise with the generator and decode with
    # the oracle: the vector must come back exactly.
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -6, -4, -3, -2, -1.5, -1, -.5, 0], np.float32)
    x = np.concatenate([np.tile(grid, 2) * 2.0 ** (j - 1) for j in range(4)])[None, :]
    packed, e8 = W.quantize_mxfp4(x)
    bs = 64
    page = np.zeros(bs * 68, np.uint8)
    page[:64] = packed[0]
    page[bs * 64:bs * 64 + 4] = e8[0]
    lay = O.Layout(page, bs * 68, 0, 0, bs, O.IDX_MXFP4, O.LAT_FP8)
    got = O.gather_index_keys(lay, np.array([0]), 1)[0]
    assert np.array_equal(got, x[0].astype(np.float64))
    # NVFP4 latent: blocks of 16 with amax 6 * 2^k -> e4m3 scale 2^k exactly.
    y = np.concatenate([grid * 2.0 ** ((j % 9) - 4) for j in range(36)])[None, :]
    rec = W.quantize_nvfp4_latent(y)
    lpage = np.zeros(bs * 352, np.uint8)
    lpage[:352] = rec[0]
    lay2 = O.Layout(lpage, bs * 352, 0, 0, bs, O.IDX_FP8, O.LAT_NVFP4)
    got2 = O.gather_latents(lay2, np.array([0]), np.array([0]))[0]
    assert np.array_equal(got2, y[0].astype(np.float64))
    assert not rec[0, 324:].any()        # 28 bytes of padding are zero


def test_mxfp4_index_page_read_from_hand_written_bytes():
    # Block of 16 tokens, token in slot 1 (so slot offsets matter): its 64 value
    # bytes start at byte 64, its four E8M0 scales at 16 * 64 + 4.  Byte 0 = 0x21:
    # elements 0, 1 = e2m1 codes 1, 2 = 0.5, 1.0; byte 16 = 0xF7: elements 32, 33 =
    # codes 7, 15 = 6.0, -6.0.  Scales: block 0 = 127 (x1), block 1 = 129 (x4).
    bs = 16
    page = np.zeros(bs * 68, np.uint8)
    page[64 + 0] = 0x21
    page[64 + 16] = 0xF7
    page[bs * 64 + 4 * 1 + 0] = 127
    page[bs * 64 + 4 * 1 + 1] = 129
    page[bs * 64 + 4 * 1 + 2] = 127
    page[bs * 64 + 4 * 1 + 3] = 127
    lay = O.Layout(page, bs * 68, 0, 0, bs, O.IDX_MXFP4, O.LAT_FP8)
    keys = O.gather_index_keys(lay, np.array([0]), 2)
    want = np.zeros(128)
    want[[0, 1, 32, 33]] = [0.5, 1.0, 24.0, -24.0]
    assert np.array_equal(keys[1], want)
    assert not keys[0].any()                 # slot 0 is all zero codes


def test_nvfp4_latent_record_read_from_hand_written_bytes():
    # Token in slot 1 of a 16-token block: record at byte 352.  Byte 0 = 0x3A:
    # elements 0, 1 = codes 0xA, 0x3 = -1.0, 1.5; element 16 (byte 8, low nibble)
    # = code 0x7 = 6.0.  Scales (e4m3, per 16 values) at record byte 288: block 0 =
    # 0x40 = 2.0, block 1 = 0x30 = 0.5.
    bs = 16
    page = np.zeros(bs * 352, np.uint8)
    rec = 352
    page[rec + 0] = 0x3A
    page[rec + 8] = 0x07
    page[rec + 288 + 0] = 0x40
    page[rec + 288 + 1] = 0x30
    lay = O.Layout(page, bs * 352, 0, 0, bs, O.IDX_FP8, O.LAT_NVFP4)
    lat = O.gather_latents(lay, np.array([0]), np.array([1]))[0]
    want = np.zeros(576)
    want[[0, 1, 16]] = [-2.0, 3.0, 3.0]
    assert np.array_equal(lat, want)


# --------------------------------------------------------- byte arithmetic

def test_per_token_widths():
    # an FP8 index key takes 132 B with its scale, an MXFP4 one 68 B with its scales; latents 576 / 352 B
    assert O.idx_bytes_per_token(O.IDX_FP8) == 132 == 128 + 4
    assert O.idx_bytes_per_token(O.IDX_MXFP4) == 68 == 64 + 4
    assert O.lat_bytes_per_token(O.LAT_FP8) == 576
    assert O.lat_bytes_per_token(O.LAT_NVFP4) == 352 >= 288 + 36
    assert 352 % 16 == 0 and 8448 % 16 == 0 and 4352 % 16 == 0


def test_kv_footprint_table():
    # "KV cache footprint" table: 13,824 / 16,992 / 10,080 bytes per token (24 layers)
    assert O.kv_bytes_per_token_all_layers(None, O.LAT_FP8) == 13824
    assert O.kv_bytes_per_token_all_layers(O.IDX_FP8, O.LAT_FP8) == 16992
    assert O.kv_bytes_per_token_all_layers(O.IDX_MXFP4, O.LAT_NVFP4) == 10080
    # MXFP4 keys need 48.5% less index storage; the MXFP4 + NVFP4 cache holds 1.7x the tokens of FP8
    assert round(100 * (1 - 68 / 132), 1) == 48.5
    assert round(16992 / 10080, 1) == 1.7


def test_decode_byte_ratio_about_23_percent():
    # at long context a decode step reads about 23% of the bytes dense MLA would, per layer
    r = lambda L: O.decode_bytes_model(L) / O.dense_mla_bytes(L)
    assert abs(r(65536) - 0.2604) < 1e-4
    assert abs(r(1 << 20) - 0.2311) < 1e-4
    assert abs(r(1 << 30) - 132 / 576) < 1e-5 and round(132 / 576, 2) == 0.23
    assert O.decode_bytes_model(1000) == 1000 * 132 + 1000 * 576      # L < k: all latents


# ------------------------------------------------------- worked example

def _golden():
    vals = {}
    with open(os.path.join(GOLDEN, "four_token_example.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split("=")
                vals[k.strip()] = [float(x) for x in v.split()]
    return vals


def _four_token_layout():
    g = _golden()
    bs = 64
    idx_pb, lat_pb = bs * 132, bs * 576
    pool = np.zeros(idx_pb + lat_pb, np.uint8)
    keys = np.tile(np.array([7.0, -3.0], np.float32), 64)[None, :].repeat(4, 0)
    keys[:, 0] = g["key_d0"]
    pool[:4 * 128] = W.to_e4m3(keys).reshape(-1)
    pool[bs * 128:bs * 128 + 16] = np.array(g["key_scale"], np.float32).view(np.uint8)
    lat = np.zeros((4, 576), np.float32)
    lat[0, 1] = 2
    lat[2, 0], lat[2, 1] = 1, -1
    lat[1, :] = lat[3, :] = 4
    pool[idx_pb:idx_pb + 4 * 576] = W.to_e4m3(lat).reshape(-1)
    q_idx = np.zeros((32, 128), np.float32)
    q_idx[0, 0], q_idx[1, 0] = 1, -1
    w = np.full(32, g["w_h0_h1_rest"][2], np.float32)
    w[0], w[1] = g["w_h0_h1_rest"][:2]
    q = np.zeros((96, 576), np.float32)
    q[0, 0] = 24.0
    lay = O.Layout(pool, idx_pb + lat_pb, 0, idx_pb, bs, O.IDX_FP8, O.LAT_FP8)
    return g, lay, W.to_e4m3(q_idx), w, W.to_bf16_bits(q)


@pytest.mark.parametrize("k", [2, 3])
def test_four_token_example(k):
    g, lay, q_idx, w, q = _four_token_layout()
    bt = np.array([[0]], np.int32)
    res = O.layer_step(lay, bt, np.array([4]), np.array([0]), np.array([3]),
                       q_idx[None], w[None], q[None], topk=k, sm_scale=1 / 24)
    assert np.array_equal(res["scores"][0], g["expect_scores"])
    assert list(res["idx"][0]) == [int(v) for v in g[f"expect_top{k}"]]
    out, lse = res["out"][0], res["lse"][0]
    if k == 2:
        np.testing.assert_allclose(out[0, :2], g["top2_h0_out01"], rtol=0, atol=1e-14)
        assert np.all(out[0, 2:] == 0)
        np.testing.assert_allclose(lse[0], g["top2_h0_lse"][0], atol=1e-14)
        np.testing.assert_allclose(out[1:, :2], np.broadcast_to(g["top2_other_out01"], (95, 2)), atol=1e-14)
        np.testing.assert_allclose(lse[1:], g["top2_other_lse"][0], atol=1e-14)
    else:
        h0 = g["top3_h0_out012"]
        np.testing.assert_allclose(out[0, :3], h0, atol=1e-13)
        np.testing.assert_allclose(out[0, 3:], h0[2], atol=1e-13)
        np.testing.assert_allclose(lse[0], g["top3_h0_lse"][0], atol=1e-13)
        oth = g["top3_other_out012"]
        np.testing.assert_allclose(out[1:, :3], np.broadcast_to(oth, (95, 3)), atol=1e-13)
        np.testing.assert_allclose(lse[1:], g["top3_other_lse"][0], atol=1e-13)


def test_causal_inclusive_range():
    # A query at position p scores exactly tokens 0..p of its request.
    g, lay, q_idx, w, q = _four_token_layout()
    sc = O.indexer_scores(lay, np.array([[0]]), np.array([0, 0]), np.array([1, 3]),
                          np.stack([q_idx, q_idx]), np.stack([w, w]))
    assert [len(s) for s in sc] == [2, 4]
    assert np.array_equal(sc[0], sc[1][:2])


# ------------------------------------------------------------ brute force

def _dominates(scores, a, b):
    return scores[a] > scores[b] or (scores[a] == scores[b] and a < b)


@pytest.mark.parametrize("seed", range(12))
def test_topk_brute_force_tiny(seed):
    # Definition of exact top-k with the lower-index tie rule: S (|S| = k) such that
    # every member beats every non-member.  Enumerate all subsets; exactly one
    # qualifies and it must be the oracle's choice.  Small integer scores force ties.
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 10))
    scores = rng.integers(-2, 3, size=n).astype(np.float64)
    for k in range(1, n + 2):
        want = []
        for S in itertools.combinations(range(n), min(k, n)):
            rest = [j for j in range(n) if j not in S]
            if all(_dominates(scores, a, b) for a in S for b in rest):
                want.append(S)
        assert len(want) == 1
        assert tuple(O.topk_select(scores, k)) == want[0]


# ------------------------------------------------------- the tie band's anchor

def test_kth_score_hand_values():
    # kth_score sets where the parity bar's tie band lies (scores within 1e-5 of
    # the k-th best may be swapped).  Values worked out by hand: sorted
    # descending [3, 2, 2, 1, -1]; k past n gives the lowest score.
    s = np.array([3.0, 1.0, 2.0, 2.0, -1.0])
    want = {1: 3.0, 2: 2.0, 3: 2.0, 4: 1.0, 5: -1.0, 6: -1.0, 2048: -1.0}
    for k, v in want.items():
        assert O.kth_score(s, k) == v, k
    # signed zeros compare equal; negatives order below them
    z = np.array([-0.0, 0.0, -2.0, -1.0])
    assert [O.kth_score(z, k) for k in (1, 2, 3, 4, 7)] == [0.0, 0.0, -1.0, -2.0, -2.0]
    assert O.kth_score(np.array([5.0]), 1) == 5.0 and O.kth_score(np.array([5.0]), 2048) == 5.0


@pytest.mark.parametrize("seed", range(6))
def test_kth_score_is_the_order_statistic(seed):
    # The k-th largest x of a list is defined by: fewer than k entries exceed x
    # and at least k entries are >= x; it is also the smallest score the exact
    # top-k keeps (topk_select is pinned by brute force above).
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 400))
    s = rng.integers(-20, 21, size=n).astype(np.float64) / 4.0
    for k in sorted({1, 2, n // 2 + 1, n, n + 3}):
        x = O.kth_score(s, k)
        kk = min(k, n)
        assert np.count_nonzero(s > x) < kk <= np.count_nonzero(s >= x)
        assert x == s[O.topk_select(s, k)].min()


# ------------------------------------------------- dense special case (library)

@pytest.mark.parametrize("L", [1, 64, 65, 200])
def test_k_at_least_L_equals_dense_attention(L):
    # With k >= L every token is kept, so the step must equal dense softmax
    # attention over the whole context: torch's scaled_dot_product_attention in
    # float64 (value = first 512 latent dims) and scipy's logsumexp.
    from scipy.special import logsumexp
    wl = W.make_workload([L], 1, seed=L, permute=True, pool_rows=(L + 63) // 64 + 3)
    lay = oracle_layout(wl)
    res = O.layer_step(lay, wl.block_table, wl.ctx_lens, wl.q_req, wl.q_pos, wl.q_idx,
                       wl.w, wl.q, topk=2048, sm_scale=1 / 24)
    assert list(res["idx"][0]) == list(range(L))
    c = torch.from_numpy(O.gather_latents(lay, wl.block_table[0], np.arange(L)))
    qf = torch.from_numpy(oracle.decode_bf16(wl.q[0]).reshape(96, 576))
    # the 96 heads act as 96 query rows that all attend the same L keys
    ref = torch.nn.functional.scaled_dot_product_attention(
        qf[None], c[None], c[None, :, :512], scale=1 / 24)[0]
    np.testing.assert_allclose(res["out"][0], ref.numpy(), rtol=1e-12, atol=1e-12)
    lse = logsumexp((qf.numpy() @ c.numpy().T) / 24, axis=1)
    np.testing.assert_allclose(res["lse"][0], lse, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- invariants

def _small(seed=3, L=300, **kw):
    wl = W.make_workload([L], 1, seed=seed, pool_rows=(L + 63) // 64 + 2, **kw)
    return wl, oracle_layout(wl)


def test_relu_identity_and_linearity_in_w():
    # ReLU(x) - ReLU(-x) = x  =>  score(q) - score(-q) = sum_h w_h (q_h . k_s), a
    # plain bilinear form; and scores are linear in the head weights.
    wl, lay = _small()
    keys = O.gather_index_keys(lay, wl.block_table[0], 300)
    qc = wl.q_idx[0]
    neg = qc ^ np.uint8(0x80)                       # flip every sign bit
    w = wl.w[0].astype(np.float64)
    d = O.indexer_scores_for_token(keys, qc, w) - O.indexer_scores_for_token(keys, neg, w)
    bil = np.einsum("sd,hd,h->s", keys, oracle.decode_e4m3(qc), w)
    np.testing.assert_allclose(d, bil, rtol=1e-12, atol=1e-12)
    w2 = np.random.default_rng(0).standard_normal(32)
    np.testing.assert_allclose(O.indexer_scores_for_token(keys, qc, w + w2),
                               O.indexer_scores_for_token(keys, qc, w)
                               + O.indexer_scores_for_token(keys, qc, w2), rtol=1e-12, atol=1e-12)
    assert np.all(O.indexer_scores_for_token(keys, qc, np.abs(w)) >= 0)


def test_key_scale_scales_score():
    wl, lay = _small()
    base = O.indexer_scores(lay, wl.block_table, wl.q_req, wl.q_pos, wl.q_idx, wl.w)[0]
    pool = wl.pool.copy()
    row = wl.block_table[0, 1]
    off = row * wl.row_stride + 64 * 128 + 5 * 4        # token 64+5
    s = pool[off:off + 4].view(np.float32)[0]
    pool[off:off + 4] = np.array([s * 4.0], np.float32).view(np.uint8)
    lay2 = O.Layout(pool, wl.row_stride, 0, wl.lat_page_offset)
    new = O.indexer_scores(lay2, wl.block_table, wl.q_req, wl.q_pos, wl.q_idx, wl.w)[0]
    assert new[69] == 4.0 * base[69]
    mask = np.ones(300, bool)
    mask[69] = False
    assert np.array_equal(new[mask], base[mask])


def test_negative_key_scale_reads_as_a_negated_key():
    # A negative fp32 scale multiplies the decoded key: with the scale of token 69
    # negated, its score equals the score of the unchanged key against the negated
    # query codes (e4m3 negation flips the sign bit, an exact operation).
    wl, lay = _small()
    keys = O.gather_index_keys(lay, wl.block_table[0], 300)
    pool = wl.pool.copy()
    row = wl.block_table[0, 1]
    off = row * wl.row_stride + 64 * 128 + 5 * 4        # token 64+5
    s = pool[off:off + 4].view(np.float32)[0]
    pool[off:off + 4] = np.array([-s], np.float32).view(np.uint8)
    lay2 = O.Layout(pool, wl.row_stride, 0, wl.lat_page_offset)
    new = O.indexer_scores(lay2, wl.block_table, wl.q_req, wl.q_pos, wl.q_idx, wl.w)[0]
    flipped = O.indexer_scores_for_token(keys, wl.q_idx[0] ^ np.uint8(0x80), wl.w[0])[69]
    assert new[69] == flipped
    base = O.indexer_scores(lay, wl.block_table, wl.q_req, wl.q_pos, wl.q_idx, wl.w)[0]
    assert new[69] != base[69]


def test_block_table_permutation_changes_nothing():
    # The same logical cache stored under two different row permutations.
    a = W.make_workload([700, 300], 2, seed=9, permute=False, pool_rows=20)
    b = W.make_workload([700, 300], 2, seed=9, permute=True, pool_rows=20)
    ra = O.layer_step(oracle_layout(a), a.block_table, a.ctx_lens, a.q_req, a.q_pos,
                      a.q_idx, a.w, a.q, topk=128)
    rb = O.layer_step(oracle_layout(b), b.block_table, b.ctx_lens, b.q_req, b.q_pos,
                      b.q_idx, b.w, b.q, topk=128)
    assert not np.array_equal(a.block_table, b.block_table)
    for x, y in zip(ra["idx"], rb["idx"]):
        assert np.array_equal(x, y)
    assert np.array_equal(ra["out"], rb["out"]) and np.array_equal(ra["lse"], rb["lse"])


def test_softmax_weights_sum_to_one():
    # Identical value rows -> every head returns that row exactly (weights sum to 1);
    # zero query -> uniform weights, lse = log n.
    rng = np.random.default_rng(1)
    n = 37
    lat = np.repeat(rng.standard_normal((1, 576)), n, 0)
    q = W.to_bf16_bits(rng.standard_normal((96, 576)).astype(np.float32))
    out, _ = O.sparse_mla(q, lat, 1 / 24)
    np.testing.assert_allclose(out, np.broadcast_to(lat[0, :512], (96, 512)), rtol=1e-13, atol=1e-13)
    lat2 = rng.standard_normal((n, 576))
    out2, lse2 = O.sparse_mla(np.zeros((96, 576), np.uint16), lat2, 1 / 24)
    np.testing.assert_allclose(out2, np.broadcast_to(lat2[:, :512].mean(0), (96, 512)), atol=1e-13)
    np.testing.assert_allclose(lse2, math.log(n), atol=1e-13)


def test_fewer_tokens_than_k_selects_all():
    wl, lay = _small(L=100)
    res = O.layer_step(lay, wl.block_table, wl.ctx_lens, wl.q_req, wl.q_pos, wl.q_idx,
                       wl.w, wl.q, topk=2048)
    assert list(res["idx"][0]) == list(range(100))


def test_mtp_positions_are_causal_among_new_tokens():
    wl = W.make_workload([500], 6, seed=4, pool_rows=10)
    assert list(wl.q_pos) == list(range(494, 500))
    sc = O.indexer_scores(oracle_layout(wl), wl.block_table, wl.q_req, wl.q_pos, wl.q_idx, wl.w)
    assert [len(s) for s in sc] == list(range(495, 501))
