"""FP8 E4M3 codec written from the format definition.

[OCP-FP8] E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits.
  exponent field 0      : subnormal, value = (-1)^s * 2^-6 * m/8
  exponent field 1..15  : normal,    value = (-1)^s * 2^(e-7) * (1 + m/8)
  S.1111.111 (0x7F/0xFF): NaN.  There are no infinities; max finite = 448.
[GLM-5.3 "How to try"]: the KV cache is FP8 in every configuration.

Encoding used by the store is round-to-nearest-even with saturation to the
largest finite magnitude ("satfinite"): every finite |x| > 448 and +-inf map
to +-448, NaN maps to 0x7F.  The sign of x is kept, including for results
that round to zero.
"""

import numpy as np

E4M3_MAX = 448.0
_MIN_NORMAL = 2.0 ** -6
_SUB_QUANTUM = 2.0 ** -9


def _decode_one(code: int) -> float:
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * _MIN_NORMAL * (m / 8.0)
    return s * 2.0 ** (e - 7) * (1.0 + m / 8.0)


_TABLE = np.array([_decode_one(c) for c in range(256)], dtype=np.float64)


def e4m3_decode(codes) -> np.ndarray:
    """Decode uint8 E4M3 codes to float64 (exact)."""
    return _TABLE[np.asarray(codes, dtype=np.uint8)]


def _floor_log2(a: np.ndarray) -> np.ndarray:
    """floor(log2(a)) for normal float64 a > 0: the unbiased exponent field of its IEEE bits."""
    return ((a.view(np.uint64) >> np.uint64(52)) & np.uint64(0x7FF)).astype(np.int64) - 1023


def _pow2(e: np.ndarray) -> np.ndarray:
    """2.0 ** e for integer e in the normal float64 range, built from the exponent field."""
    return ((e + 1023).astype(np.uint64) << np.uint64(52)).view(np.float64)


def e4m3_encode(x) -> np.ndarray:
    """Round float32 values to E4M3 codes (RNE, satfinite).  Returns uint8.

    Each value is rounded once, from its exact value to the nearest E4M3 value,
    ties to the even mantissa: the spacing of E4M3 values is 2^-9 below 2^-6
    (subnormals) and 2^(floor(log2|x|) - 3) above.
    """
    shape = np.shape(x)
    flat = np.asarray(x, dtype=np.float64).reshape(-1)
    out = np.empty(flat.size, dtype=np.uint8)
    for c0 in range(0, flat.size, 1 << 20):       # bounded temporaries
        out[c0:c0 + (1 << 20)] = _encode_flat(flat[c0:c0 + (1 << 20)])
    return out.reshape(shape)


def _encode_flat(arr: np.ndarray) -> np.ndarray:
    arr = np.ascontiguousarray(arr)
    nan = np.isnan(arr)
    sign = np.where(np.signbit(arr), 0x80, 0).astype(np.int64)
    a = np.minimum(np.abs(np.where(nan, 0.0, arr)), E4M3_MAX)   # satfinite clamp
    normal_in = a >= _MIN_NORMAL
    safe_a = np.where(normal_in, a, 1.0)
    quantum = np.where(normal_in, _pow2(_floor_log2(safe_a) - 3), _SUB_QUANTUM)
    v = np.rint(a / quantum) * quantum          # np.rint: round half to even; exact product
    v = np.minimum(v, E4M3_MAX)
    normal_out = v >= _MIN_NORMAL
    safe_v = np.where(normal_out, v, 1.0)
    e = _floor_log2(safe_v)
    m = np.rint((safe_v / _pow2(e) - 1.0) * 8.0).astype(np.int64)
    code_normal = ((e + 7) << 3) | m
    code_sub = np.rint(v / _SUB_QUANTUM).astype(np.int64)
    code = np.where(normal_out, code_normal, code_sub) | sign
    code = np.where(nan, 0x7F, code)
    return code.astype(np.uint8)
