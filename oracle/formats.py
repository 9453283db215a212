"""Number formats the oracle reads, decoded from their bit-field definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

- bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits; the upper half of
  an IEEE binary32.
- e2m1 (FP4): 1 sign, 2 exponent (bias 1), 1 mantissa bit; no inf/NaN.
- e4m3 (FP8, finite-only variant): 1 sign, 4 exponent (bias 7), 3 mantissa
  bits; S.1111.111 is NaN, there is no infinity; max 448.
- NVFP4 weight = e2m1 value x e4m3 block scale (one per 16 consecutive values
  along the reduction dimension) x float32 tensor scale.  The pages name the
  NVFP4 checkpoint (evermx.com review, section "Quantization"; futurpulse.com,
  section "How did Recursive use AI to build Flint?") without a layout; this
  is the plainest reading of the format's name.
"""
import numpy as np


def bf16_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values, decoded field by field."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where((b >> 15) & 1, -1.0, 1.0)
    exp = (b >> 7) & 0xFF
    man = (b & 0x7F).astype(np.float64)
    normal = sign * (1.0 + man / 128.0) * np.exp2(exp.astype(np.float64) - 127.0)
    sub = sign * (man / 128.0) * 2.0 ** -126
    out = np.where(exp == 0, sub, normal)
    special = exp == 0xFF
    if np.any(special):
        out = np.where(special & (man == 0), sign * np.inf, out)
        out = np.where(special & (man != 0), np.nan, out)
    return out


def round_to_bf16(v) -> np.ndarray:
    """float64 -> nearest bfloat16 value (ties to even), returned as float64.

    One rounding step straight from float64 (no detour through float32).
    Finite inputs beyond the bf16 range become +-inf; subnormals are kept.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros_like(v)
    nz = (v != 0) & np.isfinite(v)
    a = np.abs(v[nz])
    _, e = np.frexp(a)                 # a = m * 2^e, m in [0.5, 1)
    e = np.maximum(e - 1, -126)        # exponent of the leading bit, clamped to bf16's normal min
    ulp = np.exp2(e - 7.0)             # 8 significant bits (subnormals: fixed 2^-133)
    r = np.rint(a / ulp) * ulp         # np.rint is round-half-to-even
    r = np.where(r > (2.0 - 2.0 ** -7) * 2.0 ** 127, np.inf, r)
    out[nz] = np.sign(v[nz]) * r
    out[~np.isfinite(v)] = v[~np.isfinite(v)]
    return out


def e2m1_value(code) -> np.ndarray:
    """FP4 e2m1 codes (low 4 bits) -> float64."""
    c = np.asarray(code).astype(np.int64) & 0xF
    sign = np.where(c & 8, -1.0, 1.0)
    e = (c >> 1) & 3
    m = (c & 1).astype(np.float64)
    mag = np.where(e == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(e - 1.0))
    return sign * mag


def e4m3_value(code) -> np.ndarray:
    """FP8 e4m3 (finite-only) codes -> float64; the two NaN codes give nan."""
    c = np.asarray(code).astype(np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return sign * mag


def nvfp4_to_f64(packed, scales, tscale) -> np.ndarray:
    """Decode one NVFP4 matrix: packed uint8 [rows][K/2] (element 2i in the low
    nibble), e4m3 block scales uint8 [rows][K/16], float32 tensor scale."""
    packed = np.asarray(packed, dtype=np.uint8)
    rows, half = packed.shape
    K = half * 2
    codes = np.empty((rows, K), dtype=np.uint8)
    codes[:, 0::2] = packed & 0xF
    codes[:, 1::2] = packed >> 4
    vals = e2m1_value(codes).reshape(rows, K // 16, 16)
    sb = e4m3_value(np.asarray(scales, dtype=np.uint8)).reshape(rows, K // 16, 1)
    return (vals * sb * float(np.float32(tscale))).reshape(rows, K)
