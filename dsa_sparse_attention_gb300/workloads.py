"""Seeded synthetic DSA workloads: query tensors, a packed paged KV pool, block tables.

This module only draws random numbers and writes them into the storage formats
and the byte layout of the cache; it computes nothing of the method.  Both the
CUDA path's tests/benchmark and the CPU oracle consume its output.

Layout written (one DSA layer's pair of pages per cache row, as in "A KV cache
for three kinds of state" of the vLLM Kimi K3.1 Pro day-0 post):
  row = [index page | latent page]  (``idx_page_offset`` = 0, ``lat_page_offset`` =
  index page bytes), padded up to ``row_stride``.
  FP8 index page  : bs x 128 e4m3, then bs x fp32 scale          (132 B/token)
  MXFP4 index page: bs x 64 packed e2m1, then bs x 4 E8M0         (68 B/token)
  FP8 latent page : bs x 576 e4m3                                  (576 B/token)
  NVFP4 latent    : per token 288 packed e2m1, 36 e4m3 scales, 28 zero bytes (352 B)

Value distributions (the decode, MTP and prefill workloads of the vLLM post
on Kimi K3.1 Pro, at the sizes of the five benchmark configurations): q_idx and FP8 index keys are N(0,1) clamped to
[-8, 8] and rounded to e4m3; key scales U(0.5, 2); head weights N(0, 1/32);
absorbed queries N(0,1) rounded to bf16; latents N(0,1) rounded to e4m3, or
quantised to NVFP4 (e4m3 scale per 16 = amax/6); MXFP4 keys quantised with one
E8M0 exponent per 32 (floor(log2 amax) - 2).  Every tensor has its own random
stream spawned in a fixed order from ``numpy.random.SeedSequence(seed)``.
"""
from dataclasses import dataclass, field

import numpy as np
import torch

IDX_FP8, IDX_MXFP4 = 0, 1
Q_FP8, Q_MXFP4 = 0, 1               # index-query formats
LAT_FP8, LAT_NVFP4 = 0, 1
_IDX_TOKEN_BYTES = {IDX_FP8: 132, IDX_MXFP4: 68}
_LAT_TOKEN_BYTES = {LAT_FP8: 576, LAT_NVFP4: 352}


# ------------------------------------------------------------ format encoders

def to_e4m3(x: np.ndarray) -> np.ndarray:
    """float -> e4m3 codes (round to nearest even), via torch's cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    """e4m3 codes -> float32, via torch's cast (generator-side helper)."""
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float32).numpy()


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float -> bf16 bit patterns (round to nearest even), via torch's cast."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)


def to_e2m1(x: np.ndarray) -> np.ndarray:
    """float -> 4-bit e2m1 codes (nearest, ties to the even code, saturating at 6)."""
    x = np.asarray(x, dtype=np.float32)
    mag = np.minimum(np.abs(x), 6.0)
    lo = np.clip(np.searchsorted(_E2M1_GRID, mag, side="right") - 1, 0, 7)
    hi = np.minimum(lo + 1, 7)
    dlo = mag - _E2M1_GRID[lo]
    dhi = _E2M1_GRID[hi] - mag
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0) & (hi != lo))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    sign = ((x < 0) & (code != 0)).astype(np.uint8)
    return code | (sign << 3)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """4-bit codes [..., 2n] -> bytes [..., n]; element 2i goes to the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def quantize_mxfp4(x: np.ndarray):
    """[n, 128] float -> (packed e2m1 [n, 64], E8M0 [n, 4]), one scale per 32."""
    x = np.asarray(x, dtype=np.float32)
    blocks = x.reshape(x.shape[0], 4, 32)
    amax = np.abs(blocks).max(axis=2)
    with np.errstate(divide="ignore"):
        e = np.where(amax > 0, np.floor(np.log2(np.maximum(amax, 1e-38))) - 2, -127)
    e = np.clip(e, -127, 127).astype(np.int32)
    scaled = blocks / np.exp2(e.astype(np.float32))[:, :, None]
    codes = to_e2m1(scaled).reshape(x.shape[0], 128)
    return pack_nibbles(codes), (e + 127).astype(np.uint8)


def quantize_nvfp4_latent(x: np.ndarray) -> np.ndarray:
    """[n, 576] float -> [n, 352] records: 288 packed e2m1, 36 e4m3 scales, 28 zeros."""
    x = np.asarray(x, dtype=np.float32)
    n = x.shape[0]
    blocks = x.reshape(n, 36, 16)
    amax = np.abs(blocks).max(axis=2)
    scode = to_e4m3(amax / 6.0)
    sval = e4m3_values(scode)
    safe = np.where(sval > 0, sval, 1.0)
    codes = to_e2m1(np.where(sval[:, :, None] > 0, blocks / safe[:, :, None], 0.0))
    rec = np.zeros((n, 352), dtype=np.uint8)
    rec[:, :288] = pack_nibbles(codes.reshape(n, 576))
    rec[:, 288:324] = scode
    return rec


# ----------------------------------------------------------------- workload

@dataclass
class Workload:
    name: str
    pool: np.ndarray            # uint8 [num_rows * row_stride]
    num_rows: int
    row_stride: int
    idx_page_offset: int
    lat_page_offset: int
    block_size: int
    idx_fmt: int
    lat_fmt: int
    block_table: np.ndarray     # int32 [B, bt_stride]
    ctx_lens: np.ndarray        # int32 [B]
    q_req: np.ndarray           # int32 [T]
    q_pos: np.ndarray           # int32 [T]
    q_idx: np.ndarray           # uint8 e4m3 [T, 32, 128]; MXFP4 queries: [T * 32 * 68] (codes, then E8M0)
    w: np.ndarray               # float32 [T, 32]
    q: np.ndarray               # uint16 bf16 bits [T, 96, 576]
    topk: int = 2048
    sm_scale: float = 1.0 / 24.0
    meta: dict = field(default_factory=dict)
    q_fmt: int = Q_FP8

    @property
    def num_tokens(self):
        return int(self.q_req.shape[0])

    @property
    def num_reqs(self):
        return int(self.ctx_lens.shape[0])

    @property
    def max_ctx_len(self):
        return int(self.ctx_lens.max()) if self.ctx_lens.size else 0


def _streams(seed: int, n: int = 10):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def make_workload(ctx_lens, q_per_req=1, *, name="custom", seed=0, idx_fmt=IDX_FP8,
                  lat_fmt=LAT_FP8, block_size=64, pool_rows=None, row_stride=None,
                  permute=True, topk=2048, q_pos=None, bt_stride=None, negative_scale_frac=0.0, q_fmt=Q_FP8):
    """Build a workload.

    ctx_lens: tokens in cache per request (including that request's query tokens).
    q_per_req: query tokens per request (int or list); by default they are the
      last ones of the context, causal among themselves (positions L-n .. L-1).
    pool_rows: rows in the pool (default: exactly the blocks needed).
    permute: map blocks to a random permutation of pool rows (else identity).
    q_pos: optional explicit positions (list of arrays, one per request).
    negative_scale_frac: fraction of FP8 index keys whose fp32 scale is negated
      (magnitudes still U(0.5, 2)); 0 keeps every scale positive.  The signs come
      from their own random stream, so the other tensors do not change with it.
    q_fmt: Q_MXFP4 draws the index queries N(0,1) and stores them MXFP4 in the
      library's query layout: T x 32 x 64 packed e2m1 bytes, then T x 32 x 4 E8M0.
    """
    rs = _streams(seed)
    ctx_lens = np.asarray(ctx_lens, dtype=np.int64)
    B = ctx_lens.size
    bs = int(block_size)
    qpr = [int(q_per_req)] * B if np.isscalar(q_per_req) else [int(v) for v in q_per_req]
    nblk = (ctx_lens + bs - 1) // bs
    need = int(nblk.sum())
    pool_rows = need if pool_rows is None else int(pool_rows)
    if pool_rows < need:
        raise ValueError("pool too small")
    idx_pb = bs * _IDX_TOKEN_BYTES[idx_fmt]
    lat_pb = bs * _LAT_TOKEN_BYTES[lat_fmt]
    row_stride = idx_pb + lat_pb if row_stride is None else int(row_stride)
    if row_stride < idx_pb + lat_pb or row_stride % 16:
        raise ValueError("bad row stride")
    bt_stride = int(nblk.max()) if bt_stride is None else int(bt_stride)

    perm = rs[0].permutation(pool_rows) if permute else np.arange(pool_rows)
    bt = np.full((B, bt_stride), -1, dtype=np.int32)
    cursor = 0
    for b in range(B):
        bt[b, :nblk[b]] = perm[cursor:cursor + nblk[b]]
        cursor += nblk[b]

    pool = np.zeros(pool_rows * row_stride, dtype=np.uint8)
    rows2d = pool.reshape(pool_rows, row_stride)
    g_key, g_scale, g_lat, g_sign = rs[1], rs[2], rs[3], rs[7]
    chunk_blocks = 512
    for b in range(B):
        for j0 in range(0, int(nblk[b]), chunk_blocks):
            j1 = min(int(nblk[b]), j0 + chunk_blocks)
            nb = j1 - j0
            ntok = nb * bs
            rows = bt[b, j0:j1]
            if idx_fmt == IDX_FP8:
                k = np.clip(g_key.standard_normal((ntok, 128), dtype=np.float32), -8, 8)
                page_v = to_e4m3(k).reshape(nb, bs * 128)
                sc = g_scale.uniform(0.5, 2.0, size=ntok).astype(np.float32)
                if negative_scale_frac > 0:
                    sc[g_sign.random(ntok) < negative_scale_frac] *= -1.0
                page_s = sc.view(np.uint8).reshape(nb, bs * 4)
                rows2d[rows, 0:bs * 128] = page_v
                rows2d[rows, bs * 128:bs * 132] = page_s
            else:
                k = g_key.standard_normal((ntok, 128), dtype=np.float32)
                packed, e8 = quantize_mxfp4(k)
                rows2d[rows, 0:bs * 64] = packed.reshape(nb, bs * 64)
                rows2d[rows, bs * 64:bs * 68] = e8.reshape(nb, bs * 4)
            c = g_lat.standard_normal((ntok, 576), dtype=np.float32)
            if lat_fmt == LAT_FP8:
                rec = to_e4m3(c).reshape(nb, bs * 576)
            else:
                rec = quantize_nvfp4_latent(c).reshape(nb, bs * 352)
            rows2d[rows, idx_pb:idx_pb + lat_pb] = rec

    if q_pos is None:
        q_req = np.concatenate([np.full(qpr[b], b, dtype=np.int32) for b in range(B)])
        q_pos_arr = np.concatenate([np.arange(ctx_lens[b] - qpr[b], ctx_lens[b]) for b in range(B)])
    else:
        q_req = np.concatenate([np.full(len(q_pos[b]), b, dtype=np.int32) for b in range(B)])
        q_pos_arr = np.concatenate([np.asarray(q_pos[b]) for b in range(B)])
    q_pos_arr = q_pos_arr.astype(np.int32)
    T = q_req.size
    qd = rs[4].standard_normal((T, 32, 128), dtype=np.float32)
    if q_fmt == Q_MXFP4:
        packed, e8 = quantize_mxfp4(qd.reshape(T * 32, 128))
        q_idx = np.concatenate([packed.reshape(-1), e8.reshape(-1)])
    else:
        q_idx = to_e4m3(np.clip(qd, -8, 8))
    w = (rs[5].standard_normal((T, 32)) * np.sqrt(1.0 / 32.0)).astype(np.float32)
    q = to_bf16_bits(rs[6].standard_normal((T, 96, 576), dtype=np.float32))
    return Workload(name=name, pool=pool, num_rows=pool_rows, row_stride=row_stride,
                    idx_page_offset=0, lat_page_offset=idx_pb, block_size=bs,
                    idx_fmt=idx_fmt, lat_fmt=lat_fmt, block_table=bt,
                    ctx_lens=ctx_lens.astype(np.int32), q_req=q_req, q_pos=q_pos_arr,
                    q_idx=q_idx, w=w, q=q, topk=int(topk), q_fmt=int(q_fmt))


# --------------------------------------------------- the five configurations

GIB = 1 << 30


def config(n: int, seed: int = 0) -> Workload:
    """The five benchmark configurations (sizes from the benchmark definition):

    0  tiny decode: 1 request, 1 query, context 8192, identity block table.
    1  batch-8 decode, context 65,536 each, block table a random permutation
       across a 1 GiB packed pool (rows of index page + latent page).
    2  batch-32 MTP decode: 6 query tokens per request, causal among them,
       contexts log-uniform in [16384, 262144].
    3  single-request 1,048,576-token decode, MXFP4 keys + NVFP4 latents.
    4  chunked prefill: 8192 new queries appended to a 131,072-token cache.
    """
    if n == 0:
        return make_workload([8192], 1, name="cfg0_decode_b1_L8192", seed=seed, permute=False)
    if n == 1:
        rs = 64 * (132 + 576)
        return make_workload([65536] * 8, 1, name="cfg1_decode_b8_L65536", seed=seed,
                             pool_rows=GIB // rs, row_stride=rs, permute=True)
    if n == 2:
        g = _streams(seed + 1000, 1)[0]
        lens = np.round(np.exp(g.uniform(np.log(16384), np.log(262144), size=32))).astype(np.int64)
        return make_workload(lens, 6, name="cfg2_mtp_b32x6", seed=seed, permute=True)
    if n == 3:
        return make_workload([1 << 20], 1, name="cfg3_decode_L1M_mxfp4_nvfp4", seed=seed,
                             idx_fmt=IDX_MXFP4, lat_fmt=LAT_NVFP4, permute=True)
    if n == 4:
        base, new = 131072, 8192
        return make_workload([base + new], new, name="cfg4_prefill_8192_on_131072",
                             seed=seed, permute=True)
    raise ValueError(n)
