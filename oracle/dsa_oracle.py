"""Float64 reference of one DSA layer step over a packed, paged KV pool.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain numpy in float64;
a matrix product or a sort from numpy is used as a single step where the
definition calls for one, with no blocking or reordering beyond the definition.

The method (vLLM blog post "vLLM delivers day-0 support for Kimi K3.1 Pro"):

* "Sparse Attention in K3.1 Pro": an indexer keeps one FP8 key per token
  (128 e4m3 values plus a 4-byte scale, 132 bytes) and scores every earlier
  token for each query with 32 light heads; the 2,048 best tokens are kept and
  exact MLA attention reads only their 576-byte latents.
  The score is  score(t, s) = sum_h w[t, h] * ReLU(q_idx[t, h, :] . k_idx[s, :])
  with k_idx the dequantised key (code * scale).  Causal and inclusive: token t
  at position p scores s = 0 .. p.
* "What's new in Kimi K3.1 Pro" (table): 32 indexer heads x 128 dims, top-2048,
  NoPE.  MLA runs over 96 heads with absorbed 576-dim queries; the value is the
  first 512 latent dims and the softmax scale is 1/sqrt(576).
* "KV cache footprint" and "A KV cache for three kinds of state": per-token
  widths 576 B (FP8 latent) / 352 B (NVFP4 latent) and 132 B (FP8 index key) /
  68 B (MXFP4 index key); one contiguous row per cache block holds that block's
  pages at fixed offsets; block tables are translated to page addresses.
* "AMD / Quantization: Native MXFP4 indexer": MXFP4 index keys are 68 bytes
  including scales (128 e2m1 values, one E8M0 scale per 32 values).

Byte layout read here (the same contract the library header states):

  row r of the pool starts at  pool + r * row_stride.
  index page at  row + idx_page_offset, for a block of ``bs`` tokens:
     FP8  : bs x 128 e4m3 value bytes, then bs x 4-byte little-endian fp32 scales
     MXFP4: bs x 64 packed e2m1 bytes (element 2i in the low nibble of byte i),
            then bs x 4 E8M0 bytes (scale j covers dims 32j .. 32j+31)
  latent page at  row + lat_page_offset:
     FP8  : bs x 576 e4m3 bytes
     NVFP4: bs x 352 bytes per token = 288 packed e2m1 bytes, 36 e4m3 scales
            (scale j covers dims 16j .. 16j+15), 28 zero bytes of padding
  token s of request b lives in row block_table[b, s // bs], slot s % bs.

Index queries ("Low-latency decode: a fused DSA decode path": the indexer query
is quantized to FP8 or MXFP4):
     FP8  : e4m3 codes [T, 32, 128], used as-is (a per-head scale is folded
            into the head weights)
     MXFP4: T x 32 x 64 packed e2m1 bytes (element 2i in the low nibble), then
            T x 32 x 4 E8M0 bytes (scale j covers dims 32j .. 32j+31); per token
            the oracle takes them as [32, 68]: a head's 64 code bytes, then its 4
            exponents (``mxfp4_query_tokens``).
"""
import numpy as np

from .formats import decode_e4m3, decode_e2m1, decode_e8m0, decode_bf16, unpack_nibbles

IDX_FP8, IDX_MXFP4 = 0, 1
LAT_FP8, LAT_NVFP4 = 0, 1
Q_FP8, Q_MXFP4 = 0, 1
H_IDX, D_IDX = 32, 128          # indexer heads x dims
H_MLA, D_LAT, D_V = 96, 576, 512  # MLA heads, latent dims, value dims


# ---------------------------------------------------------------- byte model

def idx_bytes_per_token(idx_fmt: int) -> int:
    """132 = 128 e4m3 + 4-byte scale ("Sparse Attention in K3.1 Pro": one FP8 key
    of 132 bytes with its scale); 68 = 64 packed e2m1 + 4 E8M0 ("AMD /
    Quantization: Native MXFP4 indexer": 68 bytes including scales)."""
    return {IDX_FP8: D_IDX + 4, IDX_MXFP4: D_IDX // 2 + D_IDX // 32}[idx_fmt]


def lat_bytes_per_token(lat_fmt: int) -> int:
    """576 e4m3, or 288 packed e2m1 + 36 e4m3 scales padded to 352 ("KV cache
    footprint": 576 B FP8 and 352 B NVFP4 latents per token and layer)."""
    return {LAT_FP8: D_LAT, LAT_NVFP4: 352}[lat_fmt]


def idx_page_bytes(idx_fmt: int, bs: int) -> int:
    """Bytes of one block's index page ("A KV cache for three kinds of state": each
    block's pages sit at fixed offsets in its row)."""
    return bs * idx_bytes_per_token(idx_fmt)


def lat_page_bytes(lat_fmt: int, bs: int) -> int:
    """Bytes of one block's latent page (same section)."""
    return bs * lat_bytes_per_token(lat_fmt)


def kv_bytes_per_token_all_layers(idx_fmt, lat_fmt, n_layers=24) -> int:
    """Per-token KV bytes over the 24 DSA layers ("KV cache footprint" table).
    ``idx_fmt`` None means no index keys (the dense-MLA model)."""
    idx = 0 if idx_fmt is None else idx_bytes_per_token(idx_fmt)
    return n_layers * (lat_bytes_per_token(lat_fmt) + idx)


def decode_bytes_model(ctx_len: int, topk: int = 2048, idx_fmt=IDX_FP8, lat_fmt=LAT_FP8) -> int:
    """Bytes one decode query reads from the cache in one DSA layer: every index
    key of the context plus the latents of the selected tokens ("Sparse Attention
    in K3.1 Pro": the indexer scans every key, attention reads 2,048 latents)."""
    return ctx_len * idx_bytes_per_token(idx_fmt) + min(topk, ctx_len) * lat_bytes_per_token(lat_fmt)


def dense_mla_bytes(ctx_len: int, lat_fmt=LAT_FP8) -> int:
    """Bytes dense MLA reads per query per layer: the latent of every token (the
    dense baseline the same section compares against)."""
    return ctx_len * lat_bytes_per_token(lat_fmt)


# ------------------------------------------------------------ page reading

class Layout:
    """One DSA layer's view of a packed pool held in host memory (uint8): one
    contiguous row per cache block with that block's index-key and latent pages at
    fixed offsets ("A KV cache for three kinds of state")."""

    def __init__(self, pool, row_stride, idx_page_offset, lat_page_offset,
                 block_size=64, idx_fmt=IDX_FP8, lat_fmt=LAT_FP8):
        self.pool = np.asarray(pool, dtype=np.uint8).reshape(-1)
        self.row_stride = int(row_stride)
        self.idx_off = int(idx_page_offset)
        self.lat_off = int(lat_page_offset)
        self.bs = int(block_size)
        self.idx_fmt = int(idx_fmt)
        self.lat_fmt = int(lat_fmt)

    def _page(self, row, off, nbytes):
        start = int(row) * self.row_stride + off
        if row < 0 or start + nbytes > self.pool.size:
            raise IndexError(f"block id {row} outside the pool")
        return self.pool[start:start + nbytes]


def _decode_index_page(layout: Layout, page: np.ndarray, n: int) -> np.ndarray:
    """First ``n`` keys of one index page -> float64 [n, 128].  FP8: e4m3 code times
    the token's fp32 scale ("Sparse Attention in K3.1 Pro"); MXFP4: e2m1 code times
    2^(E-127), one E8M0 exponent per 32 dims ("AMD / Quantization: Native MXFP4
    indexer").  The byte order inside the page is the layout stated above."""
    bs = layout.bs
    if layout.idx_fmt == IDX_FP8:
        vals = decode_e4m3(page[:bs * D_IDX].reshape(bs, D_IDX)[:n])
        scales = page[bs * D_IDX:bs * (D_IDX + 4)].view("<f4").astype(np.float64)[:n]
        return vals * scales[:, None]
    if layout.idx_fmt == IDX_MXFP4:
        codes = unpack_nibbles(page[:bs * D_IDX // 2].reshape(bs, D_IDX // 2)[:n])
        vals = decode_e2m1(codes)
        e8 = page[bs * D_IDX // 2:bs * (D_IDX // 2 + 4)].reshape(bs, 4)[:n]
        scale = np.repeat(decode_e8m0(e8), 32, axis=1)
        return vals * scale
    raise ValueError("unknown index-key format")


def _decode_latent_page(layout: Layout, page: np.ndarray, slots: np.ndarray) -> np.ndarray:
    """Latents of the given slots of one latent page -> float64 [len(slots), 576].
    FP8: 576 e4m3 values with no scale ("KV cache footprint": 576 bytes); NVFP4:
    e2m1 code times an e4m3 scale per 16 values (352-byte records)."""
    bs = layout.bs
    if layout.lat_fmt == LAT_FP8:
        return decode_e4m3(page.reshape(bs, D_LAT)[slots])
    if layout.lat_fmt == LAT_NVFP4:
        rec = page.reshape(bs, 352)[slots]
        vals = decode_e2m1(unpack_nibbles(rec[:, :288]))
        scale = np.repeat(decode_e4m3(rec[:, 288:324]), 16, axis=1)
        return vals * scale
    raise ValueError("unknown latent format")


def gather_index_keys(layout: Layout, bt_row: np.ndarray, n_tokens: int) -> np.ndarray:
    """Dequantised index keys of tokens 0 .. n_tokens-1 of one request -> [n, 128].
    Page translation ("A KV cache for three kinds of state": block tables are
    translated into page addresses): token s is slot s % bs of row bt_row[s // bs]."""
    bs = layout.bs
    out = np.empty((n_tokens, D_IDX), dtype=np.float64)
    pb = idx_page_bytes(layout.idx_fmt, bs)
    for j in range((n_tokens + bs - 1) // bs):
        n = min(bs, n_tokens - j * bs)
        page = layout._page(bt_row[j], layout.idx_off, pb)
        out[j * bs:j * bs + n] = _decode_index_page(layout, page, n)
    return out


def gather_latents(layout: Layout, bt_row: np.ndarray, tokens: np.ndarray) -> np.ndarray:
    """Dequantised latents of the given token positions of one request -> [n, 576]
    (page translation as in gather_index_keys)."""
    bs = layout.bs
    tokens = np.asarray(tokens, dtype=np.int64)
    out = np.empty((tokens.size, D_LAT), dtype=np.float64)
    pb = lat_page_bytes(layout.lat_fmt, bs)
    blocks = tokens // bs
    for blk in np.unique(blocks):
        sel = np.nonzero(blocks == blk)[0]
        page = layout._page(bt_row[blk], layout.lat_off, pb)
        out[sel] = _decode_latent_page(layout, page, tokens[sel] % bs)
    return out


# ------------------------------------------------------------------ indexer

def mxfp4_query_tokens(buf: np.ndarray, T: int) -> np.ndarray:
    """The library's MXFP4 query buffer (T x 32 x 64 code bytes, then T x 32 x 4
    E8M0 bytes) -> per token [T, 32, 68]: each head's 64 code bytes, then its 4
    exponents."""
    buf = np.asarray(buf, dtype=np.uint8).reshape(-1)
    codes = buf[:T * H_IDX * 64].reshape(T, H_IDX, 64)
    e8 = buf[T * H_IDX * 64:T * H_IDX * 68].reshape(T, H_IDX, 4)
    return np.concatenate([codes, e8], axis=2)


def decode_query(q_idx_token: np.ndarray, q_fmt: int = Q_FP8) -> np.ndarray:
    """One token's index query -> float64 [32, 128].  FP8: the e4m3 codes [32, 128]
    as-is; MXFP4: [32, 68] per head 64 packed e2m1 bytes and 4 E8M0 exponents, the
    value e2m1(code) * 2^(E - 127) with exponent j covering dims 32j .. 32j+31 (the
    MX block format the post names for the indexer, as for the MXFP4 keys)."""
    if q_fmt == Q_FP8:
        return decode_e4m3(np.asarray(q_idx_token).reshape(H_IDX, D_IDX))
    if q_fmt == Q_MXFP4:
        t = np.asarray(q_idx_token, dtype=np.uint8).reshape(H_IDX, 68)
        vals = decode_e2m1(unpack_nibbles(t[:, :64]))
        return vals * np.repeat(decode_e8m0(t[:, 64:68]), 32, axis=1)
    raise ValueError("unknown index-query format")


def indexer_scores_for_token(keys: np.ndarray, q_idx_codes: np.ndarray, w: np.ndarray,
                             q_fmt: int = Q_FP8) -> np.ndarray:
    """score[s] = sum_h w[h] * max(0, q_idx[h] . k[s]) for every row of ``keys``
    ("Sparse Attention in K3.1 Pro": each earlier token is scored with 32 light
    heads against its index key; the formula is the plain reading of that prose).

    keys: float64 [n, 128] dequantised index keys; q_idx_codes: one token's index
    query in format q_fmt (see decode_query; FP8 codes are used as-is: any
    query-side scale is folded into w); w: [32]."""
    q = decode_query(q_idx_codes, q_fmt)
    dots = keys @ q.T                       # [n, 32]
    return np.maximum(dots, 0.0) @ np.asarray(w, dtype=np.float64).reshape(H_IDX)


def indexer_scores(layout: Layout, block_table, q_req, q_pos, q_idx, w, q_fmt=Q_FP8):
    """Scores of every token of a batch: list over query tokens of float64 arrays
    of length q_pos[t] + 1 (positions 0 .. q_pos[t] of its request: "every earlier
    token", inclusive because the new token's key is written before scoring, per
    "Low-latency decode: a fused DSA decode path")."""
    out = []
    cache = {}
    for t in range(len(q_req)):
        b, p = int(q_req[t]), int(q_pos[t])
        if b not in cache or cache[b].shape[0] < p + 1:
            cache[b] = gather_index_keys(layout, block_table[b], p + 1)
        out.append(indexer_scores_for_token(cache[b][:p + 1], q_idx[t], w[t], q_fmt))
    return out


# -------------------------------------------------------------------- top-k

def topk_select(scores: np.ndarray, k: int) -> np.ndarray:
    """Exact top-k ("Sparse Attention in K3.1 Pro": the 2,048 best tokens are
    kept): the k highest scores, equal scores ordered by lower token index first
    (the tie rule of the benchmark definition).  Returns the selected token
    indices in ascending order; when fewer than k tokens exist every token is
    selected."""
    scores = np.asarray(scores, dtype=np.float64)
    n = scores.size
    order = np.lexsort((np.arange(n), -scores))   # primary: score desc; then index asc
    return np.sort(order[:min(k, n)])


def kth_score(scores: np.ndarray, k: int) -> float:
    """The k-th highest score (the selection threshold, around which the parity
    bar's tie band lies); the lowest if n <= k."""
    s = np.sort(np.asarray(scores, dtype=np.float64))[::-1]
    return float(s[min(k, s.size) - 1])


# --------------------------------------------------------------- sparse MLA

def sparse_mla(q_bf16: np.ndarray, latents: np.ndarray, sm_scale: float):
    """Exact softmax attention of each of the 96 heads over the given latents
    ("Sparse Attention in K3.1 Pro": MLA runs exactly, but only over the selected
    tokens; "What's new in Kimi K3.1 Pro": 96 absorbed heads, 576-dim latent, NoPE,
    so the value is the first 512 dims and no part of the product is rotary).

    q_bf16: uint16 bf16 bit patterns [96, 576]; latents: float64 [n, 576].
    logits[h, s] = sm_scale * q[h] . c[s]  (all 576 dims, no rotary part);
    out[h] = sum_s softmax_s(logits[h]) * c[s, :512];  lse[h] = log sum_s exp(logits[h, s]).
    """
    q = decode_bf16(q_bf16).reshape(H_MLA, D_LAT)
    logits = sm_scale * (q @ latents.T)          # [96, n]
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    z = p.sum(axis=1, keepdims=True)
    out = (p @ latents[:, :D_V]) / z
    lse = (m + np.log(z))[:, 0]
    return out, lse


# --------------------------------------------------------------- layer step

def layer_step(layout: Layout, block_table, ctx_lens, q_req, q_pos, q_idx, w, q,
               topk=2048, sm_scale=1.0 / 24.0, tokens=None, q_fmt=Q_FP8):
    """One DSA layer for the query tokens listed in ``tokens`` (default: all):
    indexer scores, exact top-k, sparse MLA, in the order of Figure 1 of "Sparse
    Attention in K3.1 Pro".

    Returns dict with per-token lists: 'scores' (float64 arrays), 'idx' (selected
    positions, ascending), and arrays 'out' [n, 96, 512], 'lse' [n, 96].
    q_idx holds one entry per token in format q_fmt (MXFP4: [T, 32, 68], see
    mxfp4_query_tokens)."""
    T = len(q_req)
    tokens = list(range(T)) if tokens is None else list(tokens)
    res = {"tokens": tokens, "scores": [], "idx": [], "out": [], "lse": []}
    key_cache = {}
    for t in tokens:
        b, p = int(q_req[t]), int(q_pos[t])
        if not (0 <= p < int(ctx_lens[b])):
            raise ValueError(f"token {t}: position {p} outside context {ctx_lens[b]}")
        if b not in key_cache or key_cache[b].shape[0] < p + 1:
            key_cache[b] = gather_index_keys(layout, block_table[b], p + 1)
        sc = indexer_scores_for_token(key_cache[b][:p + 1], q_idx[t], w[t], q_fmt)
        sel = topk_select(sc, topk)
        lat = gather_latents(layout, block_table[b], sel)
        o, l = sparse_mla(q[t], lat, sm_scale)
        res["scores"].append(sc)
        res["idx"].append(sel)
        res["out"].append(o)
        res["lse"].append(l)
    res["out"] = np.stack(res["out"]) if res["out"] else np.zeros((0, H_MLA, D_V))
    res["lse"] = np.stack(res["lse"]) if res["lse"] else np.zeros((0, H_MLA))
    return res
