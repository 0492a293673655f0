"""fp8 (e4m3) copy of the state for the attend's read (test infrastructure
only; the same import rules as ``oracle.block_hybrid``).

The pages keep the state S in full precision and read it at every step
([GIST] technical summary, state-compression bullet; [PITH] "What carries the
argument": the read is O(Fd) per query). This library can also keep a copy of
S in 8 bits per value for that read; the copy is its own storage format, not
the pages'. This module is the plain definition of that copy, written from
the e4m3 format itself (1 sign bit, 4 exponent bits with bias 7, 3 mantissa
bits; no infinities; the largest finite value 448 = 1.75 * 2^8; subnormals
m/8 * 2^-6 for m = 1..7; codes 0x7F and 0xFF are NaN):

* per head: scale = max|S| / 448, in fp32 and rounded to nearest, as the
  library computes it (the quantised code is an integer that floating point
  decides, so both sides decide it in the same precision);
* code = e4m3(S / scale): the quotient rounded to nearest in fp32, then to
  the nearest e4m3 value, ties to even, magnitudes above 448 to 448;
* a head whose S is all zero gets scale 0 and zero codes;
* the dequantised state is scale * value(code), exact in fp64.
"""

from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
_MIN_NORMAL = 2.0 ** -6   # smallest normal e4m3 magnitude
_SUB_STEP = 2.0 ** -9     # spacing of the subnormals (and of [2^-6, 2^-5))


def e4m3_round(x) -> np.ndarray:
    """The nearest e4m3 value of each element (ties to even), saturated to
    +-448, as float64. Exact for any float32 input."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # quantum: 2^(e - 3) for a in [2^e, 2^(e+1)) with e >= -6; 2^-9 below
    _, ex = np.frexp(np.where(a > 0, a, 1.0))  # a = m 2^ex, m in [0.5, 1)
    e = ex - 1
    quantum = np.where(a >= _MIN_NORMAL, np.ldexp(1.0, e - 3), _SUB_STEP)
    r = np.rint(a / quantum) * quantum  # rint: round half to even
    r = np.minimum(r, E4M3_MAX)
    return np.where(np.signbit(x), -r, r)


def e4m3_value(codes) -> np.ndarray:
    """Value of each e4m3 code (uint8) as float64; NaN for 0x7F and 0xFF."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(r) -> np.ndarray:
    """Code (uint8) of each value already on the e4m3 grid (``e4m3_round``)."""
    r = np.asarray(r, dtype=np.float64)
    a = np.abs(r)
    _, ex = np.frexp(np.where(a > 0, a, 1.0))
    e = ex - 1                                   # a in [2^e, 2^(e+1))
    normal = a >= _MIN_NORMAL
    e_field = np.where(normal, e + 7, 0)
    m_field = np.where(normal, np.rint((a / np.ldexp(1.0, e) - 1.0) * 8.0),
                       np.rint(a / _SUB_STEP))
    code = (e_field.astype(np.int64) << 3) | m_field.astype(np.int64)
    code = np.where(np.signbit(r), code | 0x80, code)
    return code.astype(np.uint8)


def quantize_state_fp8(S):
    """One request's S [H, F, d] (the fp32 master's values) to its fp8 copy:
    codes [H, F, d] uint8 and scales [H] float32."""
    S32 = np.asarray(S, dtype=np.float32)
    H = S32.shape[0]
    codes = np.zeros(S32.shape, dtype=np.uint8)
    scales = np.zeros(H, dtype=np.float32)
    for h in range(H):
        amax = np.float32(np.max(np.abs(S32[h])))
        if amax == 0:
            continue
        scale = np.float32(amax / np.float32(E4M3_MAX))
        scales[h] = scale
        q = (S32[h] / scale).astype(np.float32)  # fp32 quotient, rounded to nearest
        codes[h] = e4m3_encode(e4m3_round(q))
    return codes, scales


def dequantize_state_fp8(codes, scales) -> np.ndarray:
    """scale * value(code), per head, as float64 [H, F, d]."""
    v = e4m3_value(codes)
    return v * np.asarray(scales, dtype=np.float64)[:, None, None]
