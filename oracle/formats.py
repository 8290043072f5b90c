"""Element formats decoded from their definitions (float64 results).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Formats used on the DSA path (vLLM K3.1 Pro day-0 post, "KV cache footprint" and
"A KV cache for three kinds of state": FP8 index keys and latents, MXFP4 index
keys, NVFP4 latents):

* e4m3 (OCP FP8 "fn" variant): 1 sign, 4 exponent bits with bias 7, 3 mantissa
  bits; exponent field 0 is subnormal (m/8 * 2^-6); 0bS.1111.111 is NaN; there is
  no infinity; the largest finite magnitude is 448.
* e2m1 (OCP FP4): 1 sign, 2 exponent bits with bias 1, 1 mantissa bit; exponent
  field 0 is subnormal (m * 0.5).  Magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}.
* E8M0 (OCP MX block scale): an unsigned biased exponent, value 2^(e-127);
  e = 255 is NaN.
* bf16: the top 16 bits of an IEEE binary32.

Each decoder is a 2^bits table computed once from the field definitions above.
"""
import numpy as np


def _e4m3_value(code: int) -> float:
    """Value of an e4m3 code from its fields (OCP 8-bit floating point
    specification, E4M3 encoding: bias 7, no infinity, S.1111.111 is NaN)."""
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        mag = (m / 8.0) * 2.0 ** (1 - 7)
    else:
        mag = (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return -mag if s else mag


def _e2m1_value(code: int) -> float:
    """Value of an e2m1 code from its fields (OCP Microscaling Formats v1.0, FP4
    E2M1 element: bias 1, no infinity or NaN)."""
    s = (code >> 3) & 1
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        mag = m * 0.5
    else:
        mag = (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if s else mag


E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
E2M1_TABLE = np.array([_e2m1_value(c) for c in range(16)], dtype=np.float64)
_E8M0_TABLE = np.array([2.0 ** (c - 127) if c != 255 else float("nan")
                        for c in range(256)], dtype=np.float64)


def decode_e4m3(b: np.ndarray) -> np.ndarray:
    """uint8 codes -> float64 values."""
    return E4M3_TABLE[np.asarray(b, dtype=np.uint8)]


def decode_e2m1(nibbles: np.ndarray) -> np.ndarray:
    """4-bit codes held in uint8 (0..15) -> float64 values."""
    return E2M1_TABLE[np.asarray(nibbles, dtype=np.uint8) & 0xF]


def decode_e8m0(b: np.ndarray) -> np.ndarray:
    """uint8 biased exponents -> float64 scale factors 2^(b-127) (OCP Microscaling
    Formats v1.0, E8M0 shared scale; 255 is NaN)."""
    return _E8M0_TABLE[np.asarray(b, dtype=np.uint8)]


def decode_bf16(u16: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float64 values (bfloat16 is the upper half of
    an IEEE 754 binary32)."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """Packed e2m1 bytes -> codes, element 2i from the low nibble of byte i (the
    post gives sizes only; this order is the layout reading the library's header
    states, pinned by a hand-written byte test)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out
