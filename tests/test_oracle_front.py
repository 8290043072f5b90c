"""Pins of the fused indexer front and cache-write oracle (oracle/front.py)
against what the post and the formats fix, independent of the CUDA path:
the e4m3 / e2m1 encoders against torch's float8 cast and hand-worked ties,
RMSNorm against torch's rms_norm, a hand-worked projection and quantization, the
head-weight folding identity, and the writes read back through the oracle's own
(already pinned) page readers."""
import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from oracle import front as F
from oracle.formats import E4M3_TABLE, decode_e4m3
from dsa_sparse_attention_gb300 import workloads as W


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_encode_e4m3_matches_torch_and_saturates():
    finite = E4M3_TABLE[:127]
    mids = (finite[:-1] + finite[1:]) / 2                        # exact ties: even code wins
    grid = np.concatenate([finite, mids, mids * (1 + 1e-6), mids * (1 - 1e-6), np.linspace(0, 448, 4001)])
    x = np.concatenate([grid, -grid]).astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.encode_e4m3(x.astype(np.float64)), want)
    assert F.encode_e4m3(np.array([1000.0, -1e9, 448.0]))[:3].tolist() == [0x7E, 0xFE, 0x7E]
    assert F.encode_e4m3(np.array([-0.0, -1e-30]))[:2].tolist() == [0x80, 0x80]


def test_encode_e2m1_ties_to_even_and_saturates():
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 100.0, -0.75, -5.0, 0.0, 0.5, 3.0])
    # hand-worked: ties between neighbours go to the even code (codes 0..7 = 0,.5,1,1.5,2,3,4,6)
    assert F.encode_e2m1(x).tolist() == [0, 2, 2, 4, 4, 6, 6, 7, 7, 0x8 | 2, 0x8 | 6, 0, 1, 5]


def test_rmsnorm_matches_torch_and_closed_form():
    rng = np.random.default_rng(0)
    x, g = rng.standard_normal(1536), rng.standard_normal(1536)
    want = torch.nn.functional.rms_norm(torch.from_numpy(x), (1536,), torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(F.rmsnorm(x, g, 1e-6), want, rtol=1e-13)
    # a constant vector c with eps = 0 normalises to sign(c) * gamma
    np.testing.assert_array_equal(F.rmsnorm(np.full(8, -3.0), np.arange(8.0), 0.0), -np.arange(8.0))


def test_front_hand_worked():
    # d_q = 4: c = (1, 2, 2, 4), gamma = 1, eps = 0 -> rms = 2.5, y = (0.4, 0.8, 0.8, 1.6).
    # W picks y0 into (head 0, dim 0) and y3 into (head 0, dim 1), (head 5, dim 7) = -y1.
    c, gam = _bf16([1, 2, 2, 4]), _bf16([1, 1, 1, 1])
    w = np.zeros((32 * 128, 4), np.float32)
    w[0, 0], w[1, 3], w[5 * 128 + 7, 1] = 1.0, 1.0, -1.0
    head_w = np.full(32, 0.5)
    codes, wf, s, q = F.indexer_front(c, gam, _bf16(w), head_w, 0.0)
    assert q[0, 0] == pytest.approx(0.4) and q[0, 1] == pytest.approx(1.6) and q[5, 7] == pytest.approx(-0.8)
    assert s[0] == pytest.approx(1.6 / 448) and s[5] == pytest.approx(0.8 / 448) and s[1] == 1.0
    assert codes[0, 1] == 0x7E and codes[0, 0] == 0x6E            # 448 and 112 = 1.75 * 2^6
    assert codes[5, 7] == 0xFE and np.count_nonzero(codes) == 3
    assert wf[0] == pytest.approx(0.5 * 1.6 / 448) and wf[1] == 0.5


def test_folded_weights_give_the_unquantized_score():
    # With a query whose per-head values are exact multiples of e4m3 values, the
    # quantized query with folded weights scores every key exactly like the original.
    rng = np.random.default_rng(3)
    codes0 = rng.integers(0, 0x7E, size=(32, 128)).astype(np.uint8) | (rng.integers(0, 2, size=(32, 128)) << 7).astype(np.uint8)
    codes0[:, 0] = 0x7E                                           # each head's amax is 448 code units
    s_true = np.exp2(rng.integers(-8, 4, size=32)).astype(np.float64)
    q = decode_e4m3(codes0) * s_true[:, None]
    codes, s = F.quantize_query_fp8(q)
    assert np.array_equal(codes, codes0) and np.allclose(s, s_true, rtol=0, atol=0)
    keys = rng.standard_normal((50, 128))
    w = rng.standard_normal(32)
    direct = np.maximum(keys @ q.T, 0) @ w
    np.testing.assert_allclose(O.indexer_scores_for_token(keys, codes, w * s), direct, rtol=1e-12, atol=1e-12)


def test_index_key_and_latent_writes_read_back():
    from dsa_sparse_attention_gb300 import workloads as W
    wl = W.make_workload([300], 1, seed=5, pool_rows=8, permute=True)
    lay = O.Layout(wl.pool, wl.row_stride, wl.idx_page_offset, wl.lat_page_offset, wl.block_size)
    pos = 130                                                     # block 2, slot 2
    row = wl.block_table[0, pos // 64]
    k = np.zeros(128, np.float32)
    k[:4] = [1.0, -2.0, 3.0, 0.5]
    codes, s = F.index_key_fp8(_bf16(k))
    assert s == np.float32(np.float32(3.0) / np.float32(448.0)) and codes[2] == 0x7E and codes[1] & 0x80
    pool = wl.pool.copy()
    F.write_index_key(pool, wl.row_stride, wl.idx_page_offset, 64, row, pos % 64, codes, s)
    lay2 = O.Layout(pool, wl.row_stride, wl.idx_page_offset, wl.lat_page_offset, 64)
    got = O.gather_index_keys(lay2, wl.block_table[0], 300)
    np.testing.assert_array_equal(got[pos], decode_e4m3(codes) * np.float64(s))
    np.testing.assert_array_equal(np.delete(got, pos, 0), np.delete(O.gather_index_keys(lay, wl.block_table[0], 300), pos, 0))
    assert np.allclose(got[pos][:4], k[:4], rtol=0.07)
    zc, zs = F.index_key_fp8(_bf16(np.zeros(128)))
    assert zs == 1.0 and not zc.any()
    # FP8 latent: representable values are kept; NVFP4: a block with amax 6 has scale 1.0
    x = np.zeros(576, np.float32)
    x[:4] = [1.5, -448.0, 0.0078125, 3.0]
    rec8 = F.latent_record(_bf16(x), 0)
    np.testing.assert_array_equal(decode_e4m3(rec8), x)
    y = np.zeros(576, np.float32)
    y[:6] = [6.0, -3.0, 1.5, 0.5, 4.0, -0.0]
    y[16:18] = [0.75, 0.375]                                      # block 1: amax 0.75 -> scale e4m3(0.125)
    rec4 = F.latent_record(_bf16(y), 1)
    assert rec4.size == 352 and rec4[288] == 0x38 and rec4[289] == 0x20 and not rec4[324:].any()
    wl4 = W.make_workload([300], 1, seed=6, pool_rows=8, permute=True, lat_fmt=W.LAT_NVFP4)
    pool4 = wl4.pool.copy()
    row4 = wl4.block_table[0, pos // 64]
    F.write_latent(pool4, wl4.row_stride, wl4.lat_page_offset, row4, pos % 64, rec4)
    lay4 = O.Layout(pool4, wl4.row_stride, wl4.idx_page_offset, wl4.lat_page_offset, 64, lat_fmt=1)
    back = O.gather_latents(lay4, wl4.block_table[0], np.array([pos]))[0]
    np.testing.assert_array_equal(back[:18], y[:18].astype(np.float64))


# ------------------------------------------------------------------ MXFP4

def test_mx_exponent_rule_hand_worked():
    # OCP MX: E = floor(log2 max|x|) - 2 + 127 per 32 values (2 = the largest e2m1
    # exponent, so the block's largest value lands in [4, 8) before saturation at 6)
    x = np.zeros(128)
    x[0], x[1], x[2] = 0.75, 0.3, -0.1875          # block 0: floor(log2 .75) = -1 -> E = 124, scale 1/8
    x[32] = 6.0                                      # block 1: E = 127, 6 exactly
    x[64] = -7.0                                     # block 2: E = 127, 7 saturates to 6
    packed, e = F.quantize_mxfp4(x)                  # block 3: all zero -> E = 0
    assert e.tolist() == [124, 127, 127, 0]
    # 0.75 * 8 = 6 -> code 7; 0.3 * 8 = 2.4 -> 2 (code 4); -0.1875 * 8 = -1.5 -> code 0x8 | 3
    assert packed[0] == (7 | 4 << 4) and packed[1] == (0x8 | 3)
    assert packed[16] == 7 and packed[32] == 0x8 | 7 and np.count_nonzero(packed) == 4
    # powers of two at the boundary: max|x| = 4 -> E = 127; just below 4 -> E = 126 (scale 2)
    assert F.mx_exponents(np.r_[4.0, np.zeros(31)]).tolist() == [127]
    assert F.mx_exponents(np.r_[np.nextafter(4.0, 0), np.zeros(31)]).tolist() == [126]
    assert F.mx_exponents(np.r_[1e-45, np.zeros(31)]).tolist() == [0]    # clamped at the bottom


def test_mxfp4_quantizer_roundtrips_representable_blocks():
    # a block of e2m1 values times 2^j, whose largest magnitude is 4 or 6, comes back
    # exactly with E = 127 + j (decoded by the oracle's own, separately pinned readers)
    rng = np.random.default_rng(5)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    for j in (-20, -3, 0, 5, 40):
        v = rng.choice(grid, size=(32, 128)) * rng.choice([-1, 1], size=(32, 128))
        v[:, ::32] = 6.0                                          # each block's max
        tok = F.quantize_query_mxfp4(np.ldexp(v, j))
        assert np.all(tok[:, 64:] == 127 + j)
        np.testing.assert_array_equal(O.decode_query(tok, O.Q_MXFP4), np.ldexp(v, j))


def test_mxfp4_query_error_within_half_a_step():
    # scaled by 2^(127-E) every value lies in [0, 8); the e2m1 grid spacing is 0.5 below
    # 2, 1 below 4 and 2 up to 6, so rounding errs by at most half of it, and values in
    # (6, 8) saturate to 6; large random queries over a wide range of magnitudes
    rng = np.random.default_rng(6)
    q = rng.standard_normal((32, 128)) * np.exp(rng.uniform(-5, 5, size=(32, 1)))
    tok = F.quantize_query_mxfp4(q)
    back = O.decode_query(tok, O.Q_MXFP4)
    unit = np.repeat(np.ldexp(1.0, tok[:, 64:].astype(int) - 127), 32, axis=1)
    v = np.abs(q) / unit
    assert np.all(v < 8)
    bound = np.where(v < 2, 0.25, np.where(v < 4, 0.5, np.where(v <= 6, 1.0, v - 6)))
    assert np.all(np.abs(back - q) <= bound * unit * (1 + 1e-12))


def test_mxfp4_query_buffer_layout_and_score():
    # the library's buffer: T x 32 x 64 code bytes, then T x 32 x 4 exponents; a
    # hand-worked score: head 0 = 1.5 * 2^-2 at dim 0 and head 1 = -3 at dim 40,
    # key = (2, 0, ..., dim 40 = 0.5), w = (1, 0.25, 0 ...): score = 1 * ReLU(0.75)
    # + 0.25 * ReLU(-1.5) = 0.75
    T = 2
    codes = np.zeros((T, 32, 64), np.uint8)
    e8 = np.full((T, 32, 4), 127, np.uint8)
    codes[1, 0, 0] = 3                               # token 1, head 0, dim 0: e2m1 1.5
    e8[1, 0, 0] = 125                                #   block 0 of head 0: 2^-2
    codes[1, 1, 20] = 0x8 | 5                        # head 1, dim 40 (low nibble of byte 20): -3
    buf = np.concatenate([codes.reshape(-1), e8.reshape(-1)])
    tok = O.mxfp4_query_tokens(buf, T)
    assert tok.shape == (T, 32, 68) and np.all(tok[0] == np.r_[np.zeros(64), np.full(4, 127)])
    key = np.zeros((1, 128))
    key[0, 0], key[0, 40] = 2.0, 0.5
    w = np.zeros(32)
    w[0], w[1] = 1.0, 0.25
    assert O.indexer_scores_for_token(key, tok[1], w, O.Q_MXFP4).tolist() == [0.75]
    assert O.indexer_scores_for_token(key, tok[0], w, O.Q_MXFP4).tolist() == [0.0]


def test_mxfp4_key_write_reads_back():
    # the new token's MXFP4 key written into a page and read back by the page reader
    wl = W.make_workload([200], 1, seed=9, idx_fmt=W.IDX_MXFP4)
    pool = wl.pool.copy()
    k = np.random.default_rng(3).standard_normal(128).astype(np.float32)
    kb = _bf16(k)
    packed, e8 = F.index_key_mxfp4(kb)
    row, slot = int(wl.block_table[0, 3]), 7
    F.write_index_key_mxfp4(pool, wl.row_stride, wl.idx_page_offset, 64, row, slot, packed, e8)
    lay = O.Layout(pool, wl.row_stride, wl.idx_page_offset, wl.lat_page_offset, 64, idx_fmt=O.IDX_MXFP4)
    got = O.gather_index_keys(lay, wl.block_table[0], 200)[3 * 64 + slot]
    want = O.decode_query(np.r_[packed, e8].reshape(1, 68).repeat(32, 0), O.Q_MXFP4)[0]
    np.testing.assert_array_equal(got, want)
    kf = torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    unit = np.repeat(np.ldexp(1.0, e8.astype(int) - 127), 32)
    assert np.all(np.abs(got - kf) <= unit)
