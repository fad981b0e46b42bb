"""Oracle number formats: bf16, fp8 e4m3fn and e8m0, written from their bit-field definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring): nothing on the CUDA path imports this.

Everything is computed in float64 on numpy arrays. Every bf16, e4m3 and e8m0 value, and every
product of a bf16 pair, is exact in float64, so the only rounding anywhere is the one each
function names.
"""
from __future__ import annotations

import numpy as np

# ----------------------------------------------------------------------------------------- bf16


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Value of bf16 storage bits: the top half of a binary32 word."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def _round_half_even_to_quantum(a: np.ndarray, quantum: np.ndarray) -> np.ndarray:
    # a / quantum is exact (quantum is a power of two); np.rint rounds half to even.
    return np.rint(a / quantum) * quantum


def f64_to_bf16(v: np.ndarray) -> np.ndarray:
    """bf16 bits of float64 values, rounded ONCE to nearest, ties to even.

    bf16 keeps 8 significant bits (1 implicit + 7 stored), the binary32 exponent range and
    subnormals down to 2^-133. Rounding the float64 value directly (no detour through binary32)
    is the correctly rounded result. Values beyond the largest finite bf16 after rounding become
    +-inf; NaN stays NaN (quiet, 0x7FC0 with its sign).
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty(v.shape, dtype=np.uint16)
    a = np.abs(v)
    sign = np.signbit(v)
    nan = np.isnan(v)
    finite = np.isfinite(v)
    _, e = np.frexp(np.where(finite & (a > 0), a, 1.0))  # a = m * 2^e, m in [0.5, 1)
    # spacing of bf16 numbers in a's binade: 2^(e-1-7), never below the subnormal step 2^-133
    qexp = np.maximum(e.astype(np.int64) - 8, -133)
    quantum = np.ldexp(1.0, qexp)
    r = np.where(finite, _round_half_even_to_quantum(np.where(finite, a, 0.0), quantum), np.inf)
    max_bf16 = float(np.ldexp(255.0, 120))  # (2 - 2^-7) * 2^127
    r = np.where(r > max_bf16, np.inf, r)
    # r is now exactly a bf16 value (or inf); binary32 holds it exactly, so its top half is it.
    bits32 = r.astype(np.float32).view(np.uint32)
    out[...] = (bits32 >> np.uint32(16)).astype(np.uint16)
    out |= np.where(sign, np.uint16(0x8000), np.uint16(0))
    out[nan] = np.where(sign[nan], np.uint16(0xFFC0), np.uint16(0x7FC0))
    return out


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |v| (2^(floor(log2|v|) - 7), at least 2^-133)."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(np.where(a > 0, a, 1.0))
    q = np.ldexp(1.0, np.maximum(e.astype(np.int64) - 8, -133))
    return np.where(a > 0, q, np.ldexp(1.0, -133))


# ---------------------------------------------------------------------------------------- e4m3
# float8 e4m3fn: 1 sign, 4 exponent (bias 7), 3 mantissa bits. No infinities; S.1111.111 is NaN.
# Largest finite magnitude 448 = 1.75 * 2^8; subnormals are m/8 * 2^-6 (step 2^-9).

E4M3_MAX = 448.0


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Value of fp8 e4m3fn codes, decoded from the bit fields ("Module engram": e4m3_to_f32)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    E = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.ldexp(1.0, E - 7)
    subnormal = (m / 8.0) * np.ldexp(1.0, -6)
    val = sign * np.where(E == 0, subnormal, normal)
    return np.where((E == 0xF) & (m == 0x7), np.nan, val)


def f32_to_e4m3_rne(v: np.ndarray) -> np.ndarray:
    """Encode to e4m3fn: round to nearest, ties to even; magnitudes that round above 448 give 448.

    Follows "Module engram", function f32_to_e4m3_rne: round-to-nearest-even as a float8_e4m3fn
    cast does, saturating above 448. NaN encodes as 0x7F (with the input's sign bit).
    """
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    nan = np.isnan(v)
    a0 = np.where(nan, 0.0, a)
    _, e = np.frexp(np.where(a0 > 0, a0, 1.0))
    # spacing in a's binade: 2^(floor(log2 a) - 3) for normals, 2^-9 in the subnormal range
    qexp = np.maximum(e.astype(np.int64) - 4, -9)
    q = _round_half_even_to_quantum(np.where(np.isinf(a0), E4M3_MAX, a0), np.ldexp(1.0, qexp))
    q = np.minimum(q, E4M3_MAX)
    # bits of the (now representable) magnitude q
    _, eq = np.frexp(np.where(q > 0, q, 1.0))
    E = eq.astype(np.int64) - 1 + 7
    is_sub = (q < np.ldexp(1.0, -6))
    m_sub = np.rint(q / np.ldexp(1.0, -9)).astype(np.int64)
    m_nrm = np.rint((q / np.ldexp(1.0, E - 7) - 1.0) * 8.0).astype(np.int64)
    mag = np.where(is_sub, m_sub, (E << 3) | m_nrm)
    code = (mag | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)
    code[nan] = np.where(np.signbit(v[nan]), 0xFF, 0x7F)
    return code


# ---------------------------------------------------------------------------------------- e8m0
# e8m0: an unsigned power-of-two scale, value 2^(code - 127); code 255 is NaN; there is no zero.


def e8m0_to_f64(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    return np.where(c == 255, np.nan, np.ldexp(1.0, c - 127))


def f32_to_e8m0_rne(v: np.ndarray) -> np.ndarray:
    """Nearest power of two; a tie (exactly 1.5 * 2^e) goes to the EVEN exponent of {e, e+1}.

    Follows "Module engram", function f32_to_e8m0_rne. Exponents are clamped to the code range
    [-127, 127]; non-positive inputs (not given a meaning there) map to the smallest code 0 and
    NaN to 255.
    """
    v = np.asarray(v, dtype=np.float64)
    pos = v > 0
    m, e = np.frexp(np.where(pos & np.isfinite(v), v, 1.0))   # v = m * 2^e, m in [0.5, 1)
    e = e.astype(np.int64) - 1                                # v = (2m) * 2^e, 2m in [1, 2)
    mant = 2.0 * m
    up = (mant > 1.5) | ((mant == 1.5) & ((e + 1) % 2 == 0))
    ex = np.clip(e + up.astype(np.int64), -127, 127)
    code = (ex + 127).astype(np.int64)
    code = np.where(np.isinf(v) & pos, 254, code)
    code = np.where(pos, code, 0)
    code = np.where(np.isnan(v), 255, code)
    return code.astype(np.uint8)
