"""FP4 E2M1 codec for indexer keys, written from the format definition.

[AgentX "Hybrid KV cache management"]: with the FP4 indexer enabled, the
packed KV layout uses a smaller allocation unit and saves about 10% of KV
memory.  The pages fix no FP4 format; this oracle takes the OCP Microscaling
(MX) element type FP4 E2M1:

[OCP-MX] E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit.
  exponent field 0     : subnormal, value = (-1)^s * 2^0 * (m/2)   (0, 0.5)
  exponent field 1..3  : normal,    value = (-1)^s * 2^(e-1) * (1 + m/2)
  No infinities and no NaN; max magnitude 6.0, min normal 1.0, min subnormal 0.5.

reading (packing): a key of D elements is D/2 bytes; element 2i is the low
nibble (bits 0-3) of byte i and element 2i+1 its high nibble (bits 4-7).

reading (scale): the key's existing fp32 indexer scale s_I multiplies the
score after the head sum, exactly as for E4M3 keys; there is no per-block MX
scale.

Encoding (used only to build test inputs and pins) rounds to the nearest
E2M1 value, ties to the even mantissa, and saturates to +-6 ("satfinite");
the sign of x is kept, including for results that round to zero.
"""

import numpy as np

E2M1_MAX = 6.0


def _decode_one(code: int) -> float:
    s = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    if e == 0:
        return s * (m / 2.0)
    return s * 2.0 ** (e - 1) * (1.0 + m / 2.0)


_TABLE = np.array([_decode_one(c) for c in range(16)], dtype=np.float64)


def e2m1_decode(codes) -> np.ndarray:
    """Decode 4-bit E2M1 codes (held one per uint8, values 0..15) to float64 (exact)."""
    c = np.asarray(codes, dtype=np.uint8)
    if np.any(c > 15):
        raise ValueError("E2M1 codes are 4-bit values 0..15")
    return _TABLE[c]


def e2m1_unpack(packed) -> np.ndarray:
    """Packed bytes [..., D/2] -> codes [..., D]: low nibble first."""
    b = np.asarray(packed, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0x0F
    out[..., 1::2] = b >> 4
    return out


def e2m1_pack(codes) -> np.ndarray:
    """Codes [..., D] (D even, values 0..15) -> packed bytes [..., D/2]: low nibble first."""
    c = np.asarray(codes, dtype=np.uint8)
    if c.shape[-1] % 2 or np.any(c > 15):
        raise ValueError("E2M1 packing takes an even number of 4-bit codes")
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def e2m1_encode(x) -> np.ndarray:
    """Round values to E2M1 codes (RNE, satfinite).  Returns uint8 codes 0..15.

    The E2M1 magnitudes are the multiples of 0.5 up to 2, of 1 up to 4 and of 2
    up to 6 (spacing 0.5 below 2, 1 in [2, 4), 2 in [4, 6]); each value is
    rounded once to the nearest of them, ties to the code with the even mantissa
    bit.
    """
    a = np.asarray(x, dtype=np.float64)
    if np.any(np.isnan(a)):
        raise ValueError("E2M1 has no NaN encoding")
    sign = np.where(np.signbit(a), 0x8, 0).astype(np.uint8)
    mag = np.minimum(np.abs(a), E2M1_MAX)
    best = np.zeros(a.shape, dtype=np.uint8)
    best_err = np.full(a.shape, np.inf)
    for c in range(8):                       # the eight magnitudes, nearest wins, ties to even m
        err = np.abs(mag - _TABLE[c])
        take = (err < best_err) | ((err == best_err) & (c % 2 == 0))
        best = np.where(take, c, best).astype(np.uint8)
        best_err = np.where(take, err, best_err)
    return (best | sign).astype(np.uint8)
