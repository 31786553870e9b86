"""FP8 (E4M3, "fn" variant) codec used for Recent and Anchor pages.

Source of the format: the OCP 8-bit floating point specification (E4M3:
1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
S.1111.111 is NaN, largest finite value 448, smallest subnormal 2^-9).

The Minima-KV pages (abstract, mlsanity.com paper page; "Technical Deep
Dive" on the setupai.cc summary) only say that Recent and Anchor pages stay
"in FP8".  The reading taken here, fixed in ``include/mkv.h``:

* one fp16 scale per (token, kv head, K-or-V) row:
  ``s = fp16_rn(fp32_rn(max_i |x_i| / 448))``;
* ``code_i = e4m3_rn_satfinite(fp32_rn(x_i / s))`` (IEEE fp32 division, then
  round-to-nearest-even onto the E4M3 grid, saturating at +-448);
* a row whose scale is 0 stores all codes as +0;
* dequantisation ``x_hat_i = value(code_i) * s`` (exact in fp32).

The quantiser's decision is taken in IEEE fp32 on both sides (the precision
the spec fixes), so the oracle's codes are bit-exact by construction.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_MIN_SUBNORMAL = 2.0 ** -9


def e4m3_value(code: int) -> float:
    """Value of one E4M3 code byte, from the bit-field definition."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * man * 2.0 ** -9          # subnormal: 0.mmm * 2^-6
    return sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)


E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def _round_half_even(x: float) -> int:
    # np.rint rounds half-way cases to the even integer (IEEE default mode)
    return int(np.rint(x))


def e4m3_round(v: float) -> int:
    """Round a finite real to the nearest E4M3 code, ties to even, saturating.

    Works from the exponent/mantissa structure (not by table search); the
    tests pin it against a brute-force nearest-value search and against
    ``torch.float8_e4m3fn`` conversion.
    """
    v = float(v)
    if np.isnan(v):
        raise ValueError("non-finite input to the FP8 quantiser")
    sign = 0x80 if np.signbit(v) else 0x00
    a = abs(v)
    if a >= E4M3_MAX:
        return sign | 0x7E
    if a < E4M3_MIN_NORMAL:
        m = _round_half_even(a / E4M3_MIN_SUBNORMAL)   # exact power-of-two scaling
        return sign | m                                  # m == 8 is the min normal 0x08
    e = int(np.floor(np.log2(a)))
    # guard against log2 rounding at exact powers of two
    if 2.0 ** e > a:
        e -= 1
    elif 2.0 ** (e + 1) <= a:
        e += 1
    m = _round_half_even(a / 2.0 ** (e - 3)) - 8
    if m == 8:
        e += 1
        m = 0
    code = ((e + 7) << 3) | m
    if code > 0x7E:          # rounded past 448: saturate (satfinite)
        code = 0x7E
    return sign | code


def round_to_fp16(v: float) -> float:
    """IEEE binary16 round-to-nearest-even of a float64, from the format
    definition (10 mantissa bits, bias 15, subnormals down to 2^-24)."""
    return float(round_to_fp16_array(np.array([v], dtype=np.float64))[0])


def round_to_fp16_array(v) -> np.ndarray:
    """Vectorised binary16 RNE (values returned as float64)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, E = np.frexp(a)                    # a = f * 2^E, f in [0.5, 1): exact
    e = np.maximum(E - 1, -14)            # binade of a; subnormals share -14
    q = np.ldexp(1.0, e - 10)             # spacing of binary16 values near a
    r = np.rint(a / q) * q                # exact scaling, ties to even
    r = np.where(r > 65504.0, np.inf, r)  # 65520 and above round to infinity
    out = np.copysign(r, v)
    return np.where(a == 0.0, v, out)


def fp32(v) -> np.float32:
    return np.float32(v)


def fp8_scale(x_row: np.ndarray) -> float:
    """s = fp16_rn(fp32_rn(max|x| / 448)); x is already fp32-representable."""
    amax = float(np.max(np.abs(np.asarray(x_row, dtype=np.float64))))
    q32 = np.float32(np.float32(amax) / np.float32(E4M3_MAX))   # IEEE fp32 division
    return round_to_fp16(float(q32))


def e4m3_round_array(v) -> np.ndarray:
    """Vectorised form of ``e4m3_round`` (same steps, numpy arrays)."""
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("non-finite input to the FP8 quantiser")
    sign = np.where(np.signbit(v), 0x80, 0x00).astype(np.int64)
    a = np.abs(v)
    _, E = np.frexp(a)
    e = E.astype(np.int64) - 1
    sub = a < E4M3_MIN_NORMAL
    m_sub = np.rint(a / E4M3_MIN_SUBNORMAL).astype(np.int64)
    e_n = np.where(sub, 0, e)
    m_n = np.rint(a / np.ldexp(1.0, e_n - 3)).astype(np.int64) - 8
    carry = m_n == 8
    e_n = np.where(carry, e_n + 1, e_n)
    m_n = np.where(carry, 0, m_n)
    code_n = ((e_n + 7) << 3) | m_n
    code = np.where(sub, m_sub, code_n)
    code = np.where((a >= E4M3_MAX) | (code > 0x7E), 0x7E, code)
    return (sign | code).astype(np.uint8)


def fp8_quantize_row(x_row) -> tuple[np.ndarray, float]:
    """Quantise one row (values exactly representable in fp32) to FP8.

    Returns (codes uint8[d], scale as float64 holding an fp16 value)."""
    x = np.asarray(x_row, dtype=np.float32)
    s = fp8_scale(x)
    if s == 0.0:
        return np.zeros(x.shape[0], dtype=np.uint8), 0.0
    q = (x / np.float32(s)).astype(np.float32)      # IEEE fp32 division, per element
    return e4m3_round_array(q.astype(np.float64)), s


def fp8_quantize_rows(x) -> tuple[np.ndarray, np.ndarray]:
    """Row-wise ``fp8_quantize_row`` over the last axis of ``x``."""
    x = np.asarray(x, dtype=np.float32)
    flat = x.reshape(-1, x.shape[-1])
    amax = np.max(np.abs(flat), axis=1)
    s = round_to_fp16_array((amax / np.float32(E4M3_MAX)).astype(np.float32).astype(np.float64))
    codes = np.zeros(flat.shape, dtype=np.uint8)
    nz = s != 0.0
    if np.any(nz):
        q = (flat[nz] / s[nz, None].astype(np.float32)).astype(np.float32)
        codes[nz] = e4m3_round_array(q.astype(np.float64))
    return codes.reshape(x.shape), s.reshape(x.shape[:-1])


def fp8_dequant_row(codes, scale: float) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)] * float(scale)
