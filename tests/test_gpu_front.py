"""GPU parity of the fused indexer front and of the new tokens' cache writes,
through the C ABI, against the float64 oracle (oracle/front.py):

* the folded head weights within 1e-5 relative; the query's e4m3 codes equal
  except where the oracle's scaled value x = q / s lies within tau of the
  midpoint between two neighbouring codes.  The kernel multiplies W by y carried
  as two bf16 terms (hi = bf16(y), lo = bf16(y - hi): within 2^-17 |y| of y) and
  sums the d_q products in fp32 on the tensor cores, so its q differs from the
  exact one by about (2^-17 + sqrt(d_q) * 2^-24) * sqrt(sum of the squared
  products) (errors of random sign); tau is 8 times that, in units of x, plus
  2^-20 |x| for the fp32 division by s;
* the pool after the call equals the oracle's pool byte for byte (the new index
  keys, and for dsa_write_latent the new FP8 / NVFP4 latent records: those are
  computed in fp32 on both sides, so the bytes are exact);
* the front's outputs feed the layer step, which then matches the oracle on the
  written cache (the new key is scored like every other);
* a block id outside the pool is reported and nothing is written for it.
"""
import numpy as np
import pytest
import torch

from dsa_sparse_attention_gb300 import workloads as W
from oracle import dsa_oracle as O
from oracle import front as F
from oracle.formats import decode_e4m3
from tests.parity import OracleCache, check_mla, check_scores, check_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dsa_sparse_attention_gb300.build import build
    build()


def _bf16(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _dev_u16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


def _codes_match(got, want, x, tau):
    """e4m3 codes equal, or neighbours around a midpoint within tau of x."""
    if np.array_equal(got, want):
        return 0
    diff = np.nonzero(got != want)
    a, b, v = decode_e4m3(got[diff]), decode_e4m3(want[diff]), x[diff]
    mid = (a + b) / 2
    ok = np.abs(v - mid) <= tau[diff]
    assert np.all(ok), f"{np.count_nonzero(~ok)} codes differ away from a rounding midpoint"
    return diff[0].size


def _tau(c_q, gamma, w_qi, eps, s, x):
    """Tolerance of x = q / s for the fp32 sums of the kernel (see the module docstring)."""
    from oracle.formats import decode_bf16
    y = F.rmsnorm(decode_bf16(c_q), decode_bf16(gamma), eps)
    wd = decode_bf16(w_qi).reshape(32 * 128, -1)
    rss = np.sqrt(((wd * y) ** 2).sum(axis=1)).reshape(32, 128)
    return 8 * (2.0 ** -17 + np.sqrt(wd.shape[1]) * 2.0 ** -24) * rss / s[:, None] + 2.0 ** -20 * np.abs(x)


def _front_case(lens, d_q, seed, mx=False):
    rng = np.random.default_rng(seed)
    fmt = dict(idx_fmt=W.IDX_MXFP4, q_fmt=W.Q_MXFP4) if mx else {}
    wl = W.make_workload(lens, 1, seed=seed, permute=True, pool_rows=sum((n + 63) // 64 for n in lens) + 3, **fmt)
    T = wl.num_tokens
    c_q = _bf16(rng.standard_normal((T, d_q)))
    gamma = _bf16(1.0 + 0.1 * rng.standard_normal(d_q))
    w_qi = _bf16(rng.standard_normal((32 * 128, d_q)) / np.sqrt(d_q))
    head_w = (rng.standard_normal((T, 32)) / np.sqrt(32)).astype(np.float32)
    k_new = _bf16(rng.standard_normal((T, 128)))
    return wl, c_q, gamma, w_qi, head_w, k_new


@pytest.mark.parametrize("lens,d_q", [([3000 + 41 * i for i in range(8)], 1536), ([700 + 97 * i for i in range(13)], 512),
                                      ([2500, 1900, 129], 4096)])
def test_indexer_front_and_new_keys(lens, d_q):
    import dsa_sparse_attention_gb300 as dsa
    from dsa_sparse_attention_gb300.harness import DeviceWorkload
    eps = 1e-6
    wl, c_q, gamma, w_qi, head_w, k_new = _front_case(lens, d_q, seed=len(lens) + d_q)
    T = wl.num_tokens
    dw = DeviceWorkload(wl)
    q_idx = torch.zeros(T, 32, 128, dtype=torch.uint8, device="cuda")
    w_out = torch.zeros(T, 32, dtype=torch.float32, device="cuda")
    dsa.dsa_indexer_front(dw.layout, dw.batch, _dev_u16(c_q), _dev_u16(gamma), eps, _dev_u16(w_qi),
                          torch.from_numpy(head_w).cuda(), q_idx, w_out, k_new=_dev_u16(k_new), ws=dw.ws)
    torch.cuda.synchronize()
    assert dsa.dsa_check(dw.ws) == 0
    pool_ref = wl.pool.copy()
    flips = 0
    g_codes, g_w = q_idx.cpu().numpy(), w_out.cpu().numpy()
    for t in range(T):
        codes, wf, s, q = F.indexer_front(c_q[t], gamma, w_qi, head_w[t], eps)
        np.testing.assert_allclose(g_w[t], wf, rtol=1e-5, atol=1e-30)
        x = q / s[:, None]
        flips += _codes_match(g_codes[t], codes, x, _tau(c_q[t], gamma, w_qi, eps, s, x))
        kc, ks = F.index_key_fp8(k_new[t])
        p = int(wl.q_pos[t])
        F.write_index_key(pool_ref, wl.row_stride, wl.idx_page_offset, wl.block_size,
                          wl.block_table[wl.q_req[t], p // 64], p % 64, kc, ks)
    assert flips <= T * 4096 // 1000            # ties at a midpoint are rare
    assert np.array_equal(dw.pool.cpu().numpy(), pool_ref), "pool bytes differ from the oracle's writes"

    # the front's outputs drive the layer step over the written cache
    wl.pool[:] = pool_ref
    wl.q_idx[:] = g_codes
    wl.w[:] = g_w
    dw2 = DeviceWorkload(wl)
    idx, out, lse = dw2.layer_step()
    scores = dw2.indexer_scores()
    torch.cuda.synchronize()
    oc = OracleCache(wl)
    toks = list(range(T))
    check_scores(oc, scores.cpu().numpy(), toks)
    check_topk(oc, idx.cpu().numpy(), toks, dw2.topk)
    check_mla(oc, idx.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy(), toks)


@pytest.mark.parametrize("lat_fmt", [W.LAT_FP8, W.LAT_NVFP4])
def test_write_latent_bytes(lat_fmt):
    import dsa_sparse_attention_gb300 as dsa
    from dsa_sparse_attention_gb300.harness import DeviceWorkload
    rng = np.random.default_rng(70 + lat_fmt)
    wl = W.make_workload([3000, 65, 1, 2049, 700], 1, seed=71, permute=True, pool_rows=100, lat_fmt=lat_fmt)
    T = wl.num_tokens
    x = (rng.standard_normal((T, 576)) * 3).astype(np.float32)
    x[0, :16] = 0.0                                   # a zero block (NVFP4 scale 0)
    x[1, 16:32] = 1000.0                              # saturation
    x[2, 32] = -0.0
    lat = _bf16(x)
    dw = DeviceWorkload(wl)
    dsa.dsa_write_latent(dw.layout, dw.batch, _dev_u16(lat), ws=dw.ws)
    torch.cuda.synchronize()
    assert dsa.dsa_check(dw.ws) == 0
    pool_ref = wl.pool.copy()
    for t in range(T):
        p = int(wl.q_pos[t])
        F.write_latent(pool_ref, wl.row_stride, wl.lat_page_offset, wl.block_table[wl.q_req[t], p // 64], p % 64,
                       F.latent_record(lat[t], lat_fmt))
    assert np.array_equal(dw.pool.cpu().numpy(), pool_ref)


def test_bad_block_is_reported_and_not_written():
    import dsa_sparse_attention_gb300 as dsa
    from dsa_sparse_attention_gb300.harness import DeviceWorkload
    wl, c_q, gamma, w_qi, head_w, k_new = _front_case([3000, 700], 512, seed=5)
    wl.block_table[1, 699 // 64] = wl.num_rows + 3     # the second token's block is outside the pool
    dw = DeviceWorkload(wl)
    before = dw.pool.cpu().numpy()
    q_idx = torch.zeros(2, 32, 128, dtype=torch.uint8, device="cuda")
    w_out = torch.zeros(2, 32, dtype=torch.float32, device="cuda")
    dsa.dsa_indexer_front(dw.layout, dw.batch, _dev_u16(c_q), _dev_u16(gamma), 1e-6, _dev_u16(w_qi),
                          torch.from_numpy(head_w).cuda(), q_idx, w_out, k_new=_dev_u16(k_new), ws=dw.ws)
    lat = _bf16(np.ones((2, 576)))
    dsa.dsa_write_latent(dw.layout, dw.batch, _dev_u16(lat), ws=dw.ws)
    torch.cuda.synchronize()
    assert dsa.dsa_check(dw.ws) == -6                   # DSA_ERR_DEVICE_CHECK
    after = dw.pool.cpu().numpy()
    rows = after.reshape(wl.num_rows, wl.row_stride) != before.reshape(wl.num_rows, wl.row_stride)
    changed = np.nonzero(rows.any(axis=1))[0]
    assert changed.tolist() == [wl.block_table[0, 2999 // 64]]   # only the first token's block was written


_E2M1_MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


@pytest.mark.parametrize("lens,d_q", [([3000 + 41 * i for i in range(8)], 1536), ([2500, 1900, 129], 4096)])
def test_indexer_front_mxfp4(lens, d_q):
    # MXFP4 queries (DSA_BATCH_QIDX_MXFP4) and MXFP4 new keys.  The exponent of a
    # block equals the oracle's unless the block's max lies within tau of a power of
    # two; with equal exponents a code may differ only where the scaled value lies
    # within tau (scaled) of an e2m1 rounding midpoint, or where both decode to zero.
    # The new keys are exact (bf16 inputs, power-of-two scaling): pool bytes equal.
    import dsa_sparse_attention_gb300 as dsa
    from dsa_sparse_attention_gb300.harness import DeviceWorkload
    from oracle.formats import decode_e2m1
    eps = 1e-6
    wl, c_q, gamma, w_qi, head_w, k_new = _front_case(lens, d_q, seed=len(lens) + d_q + 5, mx=True)
    T = wl.num_tokens
    dw = DeviceWorkload(wl)
    assert dw.batch.flags & dsa.DSA_BATCH_QIDX_MXFP4
    q_idx = torch.zeros(T * 32 * 68, dtype=torch.uint8, device="cuda")
    w_out = torch.zeros(T, 32, dtype=torch.float32, device="cuda")
    dsa.dsa_indexer_front(dw.layout, dw.batch, _dev_u16(c_q), _dev_u16(gamma), eps, _dev_u16(w_qi),
                          torch.from_numpy(head_w).cuda(), q_idx, w_out, k_new=_dev_u16(k_new), ws=dw.ws)
    torch.cuda.synchronize()
    assert dsa.dsa_check(dw.ws) == 0
    g_buf, g_w = q_idx.cpu().numpy(), w_out.cpu().numpy()
    assert np.array_equal(g_w, head_w)
    g_tok = O.mxfp4_query_tokens(g_buf, T)
    pool_ref = wl.pool.copy()
    e_flips = c_flips = 0
    for t in range(T):
        tok, wf, _, q = F.indexer_front(c_q[t], gamma, w_qi, head_w[t], eps, q_fmt=1)
        tau = _tau(c_q[t], gamma, w_qi, eps, np.ones(32), q)
        ge, we = g_tok[t, :, 64:].astype(int), tok[:, 64:].astype(int)
        amax = np.abs(q.reshape(32, 4, 32)).max(axis=2)
        tmax = tau.reshape(32, 4, 32).max(axis=2)
        near_pow2 = np.abs(amax - np.exp2(np.round(np.log2(np.maximum(amax, 1e-300))))) <= tmax
        assert np.all((ge == we) | near_pow2), f"token {t}: exponents differ away from a power of two"
        e_flips += np.count_nonzero(ge != we)
        same = np.repeat(ge == we, 32, axis=1)
        gc = np.stack([g_tok[t, :, :64] & 0xF, g_tok[t, :, :64] >> 4], axis=2).reshape(32, 128)
        wc = np.stack([tok[:, :64] & 0xF, tok[:, :64] >> 4], axis=2).reshape(32, 128)
        scale = np.repeat(np.exp2(127.0 - we), 32, axis=1)
        v = np.abs(q) * scale
        near_mid = np.abs(v[..., None] - _E2M1_MIDS).min(axis=-1) <= tau * scale
        zero_both = (decode_e2m1(gc) == 0) & (decode_e2m1(wc) == 0)
        bad = same & (gc != wc) & ~near_mid & ~zero_both
        assert not bad.any(), f"token {t}: {np.count_nonzero(bad)} codes differ away from a rounding midpoint"
        c_flips += np.count_nonzero(same & (gc != wc) & ~zero_both)
        packed, e8 = F.index_key_mxfp4(k_new[t])
        p = int(wl.q_pos[t])
        F.write_index_key_mxfp4(pool_ref, wl.row_stride, wl.idx_page_offset, wl.block_size,
                                wl.block_table[wl.q_req[t], p // 64], p % 64, packed, e8)
    assert c_flips <= T * 4096 // 1000 and e_flips <= T
    assert np.array_equal(dw.pool.cpu().numpy(), pool_ref), "pool bytes differ from the oracle's MXFP4 key writes"

    # the front's outputs drive the layer step over the written cache
    wl.pool[:] = pool_ref
    wl.q_idx[:] = g_buf
    wl.w[:] = g_w
    dw2 = DeviceWorkload(wl)
    idx, out, lse = dw2.layer_step()
    scores = dw2.indexer_scores()
    torch.cuda.synchronize()
    oc = OracleCache(wl)
    toks = list(range(T))
    check_scores(oc, scores.cpu().numpy(), toks)
    check_topk(oc, idx.cpu().numpy(), toks, dw2.topk)
    check_mla(oc, idx.cpu().numpy(), out.float().cpu().numpy(), lse.cpu().numpy(), toks)
