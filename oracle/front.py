"""Float64 reference of the fused indexer front and of the new token's cache writes.

TEST INFRASTRUCTURE ONLY (see the package docstring).

vLLM K3.1 Pro day-0 post, "Low-latency decode: a fused DSA decode path": a DSA
layer runs one packed input projection (query, KV latent, output gate, the
indexer's key and head weights), then one kernel that normalises the query,
projects the indexer query, quantizes it (FP8 or MXFP4) with the scales absorbed
by the head weights, and writes the new token's index key; the new token's
latent enters the KV cache from the MLA query side.  The post gives no shapes or
formulas for these steps.  Readings taken (stated in the
library's header as well):

* query norm: RMSNorm, y = x / sqrt(mean(x^2) + eps) * gamma, over the
  compressed query of width d_q (a parameter; no width is printed);
* indexer query projection: q = W . y, W of shape [32 heads * 128 dims, d_q];
* FP8 quantization per (token, head): s = max|q_h| / 448 (1 for an all-zero
  head), codes = e4m3(q_h / s); the scale is folded into the head weight,
  w'[h] = w[h] * s, because ReLU(s x) = s ReLU(x) for s > 0;
* the new token's index key: FP8 with one fp32 scale, s_k = max|k| / 448
  computed in fp32 (1 when zero), codes = e4m3(fp32(k) / s_k), written at the
  token's slot of its block's index page (132 bytes: 128 codes, then the scale
  in the page's scale area);
* MXFP4 quantization (of the query per (token, head), and of the new token's
  index key when the pool holds MXFP4 keys), per block of 32 dims with the OCP MX
  rule: E = floor(log2(max|x|)) - 2 + 127 (2 is the largest e2m1 exponent),
  clamped to 0 .. 254, E = 0 for an all-zero block; codes = e2m1(x * 2^(127 - E))
  rounded to nearest even and saturated at +-6; the exponents travel with the
  codes (E8M0), so the head weights stay as given;
* the new token's latent: FP8 pages hold e4m3(x) (no scale); NVFP4 records hold,
  per 16 values, the scale e4m3(max|x| / 6) and e2m1(x / scale), packed two per
  byte (element 2i in the low nibble), 36 scale bytes, 28 zero bytes.

The key and latent writes are stated in fp32 arithmetic (IEEE division, round to
nearest even) because their bytes are compared exactly; the query path is float64.
"""
import numpy as np

from .formats import E4M3_TABLE, E2M1_TABLE, decode_bf16

_E4M3_POS = E4M3_TABLE[:127]          # codes 0x00 .. 0x7E, ascending, 0 .. 448
_E2M1_POS = E2M1_TABLE[:8]            # codes 0 .. 7, ascending, 0 .. 6


def _encode_rne(x, table, sign_bit, top):
    """Nearest code of a sign-magnitude format whose non-negative codes 0..len-1
    list ascending values (ties to the even code, saturating at the largest)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), top)
    hi = np.clip(np.searchsorted(table, a, side="left"), 0, table.size - 1)
    lo = np.clip(hi - 1, 0, table.size - 1)
    d_lo, d_hi = a - table[lo], table[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    neg = np.signbit(x)
    return code | (neg.astype(np.uint8) << sign_bit)


def encode_e4m3(x):
    """float -> e4m3 codes, round to nearest (ties to the even code), saturating
    at +-448, the sign kept on zero (OCP FP8 E4M3 from its value table)."""
    return _encode_rne(x, _E4M3_POS, 7, 448.0)


def encode_e2m1(x):
    """float -> 4-bit e2m1 codes, round to nearest (ties to the even code),
    saturating at +-6 (OCP MX FP4 E2M1 from its value table)."""
    return _encode_rne(x, _E2M1_POS, 3, 6.0) & np.uint8(0xF)


# --------------------------------------------------------------- the front

def rmsnorm(x, gamma, eps):
    """RMSNorm of one vector (float64)."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x) + eps) * np.asarray(gamma, dtype=np.float64)


def indexer_query(c_q_bf16, gamma_bf16, w_qi_bf16, eps):
    """The indexer query of one token before quantization: W . rmsnorm(c_q),
    float64 [32, 128].  Inputs are bf16 bit patterns (uint16)."""
    y = rmsnorm(decode_bf16(c_q_bf16), decode_bf16(gamma_bf16), eps)
    w = decode_bf16(w_qi_bf16).reshape(32 * 128, -1)
    return (w @ y).reshape(32, 128)


def quantize_query_fp8(q):
    """Per-head FP8 quantization of q [32, 128]: (codes uint8 [32, 128], scales
    float64 [32]); s = max|q_h| / 448, or 1 for an all-zero head."""
    amax = np.abs(q).max(axis=1)
    s = np.where(amax > 0, amax / 448.0, 1.0)
    return encode_e4m3(q / s[:, None]), s


def mx_exponents(x):
    """E8M0 exponents of the 32-value blocks along the last axis of x [..., 32 m]:
    floor(log2(max|x|)) - 2 + 127 clamped to 0 .. 254, 0 for an all-zero block."""
    x = np.asarray(x, dtype=np.float64)
    blocks = x.reshape(x.shape[:-1] + (x.shape[-1] // 32, 32))
    amax = np.abs(blocks).max(axis=-1)
    _, ex = np.frexp(amax)                 # amax = f * 2^ex, 0.5 <= f < 1: floor(log2 amax) = ex - 1
    e = np.where(amax > 0, ex - 1 - 2 + 127, 0)
    return np.clip(e, 0, 254).astype(np.uint8)


def quantize_mxfp4(x):
    """MXFP4 of x [..., 128] (float64 or float32 values): (packed codes [..., 64],
    element 2i in the low nibble; E8M0 [..., 4]).  The scaling by 2^(127 - E) is
    exact, so the arithmetic's width does not matter."""
    x = np.asarray(x, dtype=np.float64)
    e = mx_exponents(x)
    scale = np.repeat(np.ldexp(1.0, 127 - e.astype(np.int64)), 32, axis=-1)
    codes = encode_e2m1(x * scale)
    return (codes[..., 0::2] & 0xF) | ((codes[..., 1::2] & 0xF) << 4), e


def quantize_query_mxfp4(q):
    """Per-(head, 32-dim block) MXFP4 quantization of q [32, 128]: the library's
    per-token query form [32, 68] (each head's 64 code bytes, then its 4 E8M0)."""
    packed, e = quantize_mxfp4(q)
    return np.concatenate([packed, e], axis=1).astype(np.uint8)


def indexer_front(c_q_bf16, gamma_bf16, w_qi_bf16, head_w, eps, q_fmt=0):
    """One token's index query and head weights, plus the scales and the
    unquantized query for the parity check.  FP8 (q_fmt 0): codes [32, 128], w'
    = w * s folded (float64), s [32].  MXFP4 (q_fmt 1): [32, 68] (codes and E8M0),
    w unchanged, s = None."""
    q = indexer_query(c_q_bf16, gamma_bf16, w_qi_bf16, eps)
    if q_fmt == 1:
        return quantize_query_mxfp4(q), np.asarray(head_w, dtype=np.float64), None, q
    codes, s = quantize_query_fp8(q)
    return codes, np.asarray(head_w, dtype=np.float64) * s, s, q


def index_key_fp8(k_bf16):
    """The new token's FP8 index key in fp32 arithmetic: (codes uint8 [128],
    scale float32)."""
    k = decode_bf16(k_bf16).astype(np.float32)
    amax = np.float32(np.abs(k).max())
    s = np.float32(amax / np.float32(448.0)) if amax > 0 else np.float32(1.0)
    return encode_e4m3((k / s).astype(np.float64)), s


def index_key_mxfp4(k_bf16):
    """The new token's MXFP4 index key: (packed codes uint8 [64], E8M0 uint8 [4]).
    bf16 inputs are exact in fp32 and the scaling is by a power of two, so this
    equals the fp32 computation."""
    return quantize_mxfp4(decode_bf16(k_bf16).reshape(128))


def latent_record(x_bf16, lat_fmt):
    """The new token's latent record: FP8 (576 e4m3 bytes) or NVFP4 (352 bytes),
    in fp32 arithmetic."""
    x = decode_bf16(x_bf16).astype(np.float32)
    if lat_fmt == 0:
        return encode_e4m3(x.astype(np.float64))
    blocks = x.reshape(36, 16)
    amax = np.abs(blocks).max(axis=1).astype(np.float32)
    scode = encode_e4m3((amax / np.float32(6.0)).astype(np.float64))
    sval = E4M3_TABLE[scode].astype(np.float32)
    safe = np.where(sval > 0, sval, np.float32(1.0)).astype(np.float32)
    ratio = np.where(sval[:, None] > 0, blocks / safe[:, None], np.float32(0.0)).astype(np.float32)
    codes = encode_e2m1(ratio.astype(np.float64)).reshape(576)
    rec = np.zeros(352, dtype=np.uint8)
    rec[:288] = (codes[0::2] & 0xF) | ((codes[1::2] & 0xF) << 4)
    rec[288:324] = scode
    return rec


# ----------------------------------------------------------- cache writes

def write_index_key(pool, row_stride, idx_page_offset, bs, row, slot, codes, scale):
    """Place an FP8 key in its block's index page: codes at slot * 128, the fp32
    scale at bs * 128 + slot * 4 (the library's index-page layout)."""
    base = int(row) * row_stride + idx_page_offset
    pool[base + slot * 128: base + slot * 128 + 128] = codes
    pool[base + bs * 128 + slot * 4: base + bs * 128 + slot * 4 + 4] = np.float32(scale).reshape(1).view(np.uint8)


def write_index_key_mxfp4(pool, row_stride, idx_page_offset, bs, row, slot, packed, e8):
    """Place an MXFP4 key in its block's index page: 64 code bytes at slot * 64,
    the 4 exponents at bs * 64 + slot * 4 (the library's index-page layout)."""
    base = int(row) * row_stride + idx_page_offset
    pool[base + slot * 64: base + slot * 64 + 64] = packed
    pool[base + bs * 64 + slot * 4: base + bs * 64 + slot * 4 + 4] = e8


def write_latent(pool, row_stride, lat_page_offset, row, slot, record):
    """Place a latent record (576 or 352 bytes) at its slot of the latent page."""
    n = record.size
    base = int(row) * row_stride + lat_page_offset + slot * n
    pool[base: base + n] = record
