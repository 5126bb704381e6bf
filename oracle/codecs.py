"""Number-format codecs of the oracle, written from the formats' definitions.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module; only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.

Every function maps stored codes to exact real values (float64) or rounds a real value to
the nearest code of a format. The formats are the ones the Ascend ``mega_moe`` page
(p1, "Computation Process" and "Parameters") and the DeepGEMM MegaMoE page (p2, §4 step 5)
name:

* BFLOAT16: the upper 16 bits of an IEEE binary32 value.
* FLOAT8_E4M3FN: 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,
  NaN only at S.1111.111, largest finite 448.
* FLOAT8_E5M2: 1 sign, 5 exponent bits (bias 15), 2 mantissa bits, IEEE-style: exponent field
  31 holds the infinities (mantissa 0) and NaNs; largest finite 1.75 * 2^15 = 57344.
* FLOAT4_E2M1 (packed two per byte): 1 sign, 2 exponent bits (bias 1), 1 mantissa bit;
  magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* FLOAT8_E8M0 / UE8M0 scale: unsigned exponent byte s meaning 2^(s-127); 255 is NaN.
* INT8 in the symmetric range Z8sym = [-127, 127] (p1, "Conventions").

Rounding is round-to-nearest, ties to even, the rule of the IEEE formats and of
``torch.round`` that p1's own example uses (p1, "Example", per_channel_cast_to_int8).
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------------------
# bfloat16
# ---------------------------------------------------------------------------------------


def bf16_decode(bits: np.ndarray) -> np.ndarray:
    """uint16 bf16 codes -> float64 values (bf16 is the high half of a binary32 word)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even); returns float64.

    bf16 keeps 8 significant bits. For |v| in [2^e, 2^(e+1)) the spacing is 2^(e-7); below
    the smallest normal 2^-126 the spacing stays 2^-133 (subnormals). A value at or beyond
    the largest finite bf16 plus half a spacing rounds to infinity.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty_like(v)
    finite = np.isfinite(v)
    out[~finite] = v[~finite]
    vf = v[finite]
    _, ex = np.frexp(vf)  # vf = m * 2^ex with 0.5 <= |m| < 1, so |vf| in [2^(ex-1), 2^ex)
    e = np.maximum(ex - 1, -126)
    quantum = np.ldexp(1.0, e - 7)
    r = np.rint(vf / quantum) * quantum  # np.rint rounds half to even
    bf16_max = (2.0 - 2.0 ** -7) * 2.0 ** 127
    r = np.where(np.abs(r) > bf16_max, np.copysign(np.inf, vf), r)
    out[finite] = r
    return out


def bf16_encode(v: np.ndarray) -> np.ndarray:
    """float64 values that are exactly bf16 -> uint16 codes."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


# ---------------------------------------------------------------------------------------
# float8 e4m3fn
# ---------------------------------------------------------------------------------------


def _e4m3_table() -> np.ndarray:
    """Value of each of the 256 e4m3fn codes, built from the field definition."""
    t = np.empty(256, dtype=np.float64)
    for c in range(256):
        s = -1.0 if (c >> 7) & 1 else 1.0
        e = (c >> 3) & 0xF
        m = c & 0x7
        if e == 0xF and m == 0x7:
            t[c] = np.nan
        elif e == 0:
            t[c] = s * (m / 8.0) * 2.0 ** (1 - 7)  # subnormal
        else:
            t[c] = s * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return t


E4M3_VALUES = _e4m3_table()
E4M3_MAX = 448.0


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return E4M3_VALUES[np.asarray(codes, dtype=np.uint8)]


# Non-negative finite e4m3 magnitudes in code order 0x00..0x7E (increasing with the code).
_E4M3_POS = E4M3_VALUES[:0x7F]


def e4m3_encode_rne_satfinite(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest e4m3fn code, ties to the even code, and clamp
    magnitudes above 448 to 448 (saturating finite conversion). The sign is kept, also when
    the magnitude rounds to zero (a negative value gives -0, code 0x80, as a rounding
    conversion does). Returns uint8 codes."""
    v = np.asarray(v, dtype=np.float64)
    mag = np.minimum(np.abs(v), E4M3_MAX)
    # index of the first table magnitude >= mag
    hi = np.searchsorted(_E4M3_POS, mag, side="left")
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - _E4M3_POS[lo]
    d_hi = _E4M3_POS[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    sign = np.signbit(v).astype(np.uint8) << np.uint8(7)
    return code | sign


# ---------------------------------------------------------------------------------------
# float8 e5m2
# ---------------------------------------------------------------------------------------


def _e5m2_table() -> np.ndarray:
    """Value of each of the 256 e5m2 codes, built from the field definition."""
    t = np.empty(256, dtype=np.float64)
    for c in range(256):
        s = -1.0 if (c >> 7) & 1 else 1.0
        e = (c >> 2) & 0x1F
        m = c & 0x3
        if e == 0x1F:
            t[c] = s * np.inf if m == 0 else np.nan
        elif e == 0:
            t[c] = s * (m / 4.0) * 2.0 ** (1 - 15)  # subnormal
        else:
            t[c] = s * (1.0 + m / 4.0) * 2.0 ** (e - 15)
    return t


E5M2_VALUES = _e5m2_table()
E5M2_MAX = 57344.0


def e5m2_decode(codes: np.ndarray) -> np.ndarray:
    return E5M2_VALUES[np.asarray(codes, dtype=np.uint8)]


# Non-negative finite e5m2 magnitudes in code order 0x00..0x7B (increasing with the code).
_E5M2_POS = E5M2_VALUES[:0x7C]


def e5m2_encode_rne_satfinite(v: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest e5m2 code, ties to the even code, magnitudes above
    57344 clamped to 57344 (saturating finite conversion); the sign is kept, also on zero."""
    v = np.asarray(v, dtype=np.float64)
    mag = np.minimum(np.abs(v), E5M2_MAX)
    hi = np.minimum(np.searchsorted(_E5M2_POS, mag, side="left"), 0x7B)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - _E5M2_POS[lo]
    d_hi = _E5M2_POS[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    return code | (np.signbit(v).astype(np.uint8) << np.uint8(7))


# ---------------------------------------------------------------------------------------
# float4 e2m1 (two codes per byte)
# ---------------------------------------------------------------------------------------

E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _e2m1_table() -> np.ndarray:
    t = np.empty(16, dtype=np.float64)
    for c in range(16):
        s = -1.0 if (c >> 3) & 1 else 1.0
        e = (c >> 1) & 0x3
        m = c & 0x1
        if e == 0:
            t[c] = s * (m / 2.0)  # subnormal: m * 2^-1 * 2^(1-1)
        else:
            t[c] = s * (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return t


E2M1_VALUES = _e2m1_table()


def e2m1_unpack_decode(packed: np.ndarray) -> np.ndarray:
    """Packed bytes [..., K/2] -> float64 values [..., K]; element 2j sits in the low
    nibble of byte j and element 2j+1 in the high nibble."""
    p = np.asarray(packed, dtype=np.uint8)
    lo = E2M1_VALUES[p & 0xF]
    hi = E2M1_VALUES[p >> 4]
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.float64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def int4_unpack(packed: np.ndarray) -> np.ndarray:
    """Packed bytes [..., K/2] of signed 4-bit integers (two's complement nibbles, element 2j in
    the low nibble of byte j) -> int8 values [..., K] in [-8, 7]."""
    p = np.asarray(packed, dtype=np.uint8)
    nib = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.int16)
    nib[..., 0::2] = p & 0xF
    nib[..., 1::2] = p >> 4
    return np.where(nib >= 8, nib - 16, nib).astype(np.int8)


# ---------------------------------------------------------------------------------------
# UE8M0 scale byte
# ---------------------------------------------------------------------------------------


def ue8m0_decode(s: np.ndarray) -> np.ndarray:
    s = np.asarray(s, dtype=np.uint8).astype(np.int32)
    out = np.ldexp(1.0, s - 127)
    return np.where(s == 255, np.nan, out)
