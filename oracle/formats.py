"""Element and scale formats, enumerated code by code (oracle; test infrastructure).

The pages name the formats but do not define their bits: jax.nn.scaled_matmul,
Notes (cuDNN on Blackwell) names float8_e4m3fn / float8_e5m2 elements with
float8_e8m0fnu scales for MXFP8 and float4_e2m1fn elements with float8_e4m3fn
scales for NVFP4.  The bit layouts below are the standard OCP 8-bit / MX
definitions:

    E4M3 (e4m3fn): 1 sign, 4 exponent (bias 7), 3 mantissa; no infinity;
                   S.1111.111 is NaN; largest finite 448.
    E5M2:          1 sign, 5 exponent (bias 15), 2 mantissa; IEEE-like, exponent
                   31 is Inf (mantissa 0) or NaN; largest finite 57344.
    E2M1:          1 sign, 2 exponent (bias 1), 1 mantissa; no Inf/NaN;
                   magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}.
    UE8M0:         8-bit biased exponent, value 2**(e - 127); 0xFF is NaN.
    UE4M3:         the non-negative half of E4M3 (sign bit always 0), used as
                   the NVFP4 block scale.

Every table is built by evaluating the definition for every code; nothing is
hard-coded except the field widths.

Encoding is round-to-nearest, ties to the code whose lowest bit is 0 (this is
IEEE round-half-even: the code's lowest bit is the significand's lowest bit),
with saturation of finite magnitudes above the largest finite value to that
value ("satfinite").  The sign of the input, including that of -0.0, is kept.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Format:
    name: str
    bits: int          # total storage bits of one code
    signed: bool
    exp_bits: int
    man_bits: int
    bias: int
    ieee_special: bool  # all-ones exponent is Inf/NaN (E5M2)
    fn_nan: bool        # only all-ones exponent+mantissa is NaN (E4M3 "fn")

    @property
    def n_codes(self) -> int:
        return 1 << self.bits


def _value_of(fmt: Format, code: int) -> float:
    """Evaluate one code from the sign/exponent/mantissa definition."""
    if fmt.exp_bits == 8 and fmt.man_bits == 0:  # UE8M0: pure exponent
        return math.nan if code == 0xFF else math.ldexp(1.0, code - fmt.bias)
    sign = 0
    mag_code = code
    if fmt.signed:
        sign = (code >> (fmt.bits - 1)) & 1
        mag_code = code & ((1 << (fmt.bits - 1)) - 1)
    e = (mag_code >> fmt.man_bits) & ((1 << fmt.exp_bits) - 1)
    m = mag_code & ((1 << fmt.man_bits) - 1)
    e_all_ones = e == (1 << fmt.exp_bits) - 1
    if fmt.ieee_special and e_all_ones:
        v = math.inf if m == 0 else math.nan
    elif fmt.fn_nan and e_all_ones and m == (1 << fmt.man_bits) - 1:
        v = math.nan
    elif e == 0:  # subnormal: 0.m * 2**(1 - bias)
        v = math.ldexp(m / (1 << fmt.man_bits), 1 - fmt.bias)
    else:         # normal: 1.m * 2**(e - bias)
        v = math.ldexp(1.0 + m / (1 << fmt.man_bits), e - fmt.bias)
    return -v if sign else v


E4M3 = Format("e4m3", 8, True, 4, 3, 7, False, True)
E5M2 = Format("e5m2", 8, True, 5, 2, 15, True, False)
E2M1 = Format("e2m1", 4, True, 2, 1, 1, False, False)
UE8M0 = Format("ue8m0", 8, False, 8, 0, 127, False, False)
# UE4M3 has 7 significant bits (no sign); stored in a byte whose top bit is 0.
UE4M3 = Format("ue4m3", 7, False, 4, 3, 7, False, True)

FORMATS = {f.name: f for f in (E4M3, E5M2, E2M1, UE8M0, UE4M3)}


def get(fmt) -> Format:
    return FORMATS[fmt] if isinstance(fmt, str) else fmt


_TABLES: dict[str, np.ndarray] = {}


def table(fmt) -> np.ndarray:
    """float64 value of every code, index = code (NaN where the code is NaN)."""
    fmt = get(fmt)
    if fmt.name not in _TABLES:
        _TABLES[fmt.name] = np.array([_value_of(fmt, c) for c in range(fmt.n_codes)],
                                     dtype=np.float64)
    return _TABLES[fmt.name]


def _positive_finite(fmt: Format):
    """(codes, values) of the non-negative finite codes, ascending by value."""
    vals = table(fmt)
    n_mag = fmt.n_codes // 2 if fmt.signed else fmt.n_codes
    codes = np.arange(n_mag)
    v = vals[:n_mag]
    keep = np.isfinite(v)
    codes, v = codes[keep], v[keep]
    order = np.argsort(v, kind="stable")
    return codes[order], v[order]


def max_finite(fmt) -> float:
    return float(_positive_finite(get(fmt))[1][-1])


def decode(codes, fmt) -> np.ndarray:
    """Codes (integer array) -> float64 values."""
    fmt = get(fmt)
    c = np.asarray(codes).astype(np.int64) & (fmt.n_codes - 1 if fmt.bits < 8 else 0xFF)
    return table(fmt)[c]


def encode(values, fmt) -> np.ndarray:
    """Round binary32 values to the nearest code of ``fmt`` (ties to even code),
    saturating finite overflow to the largest finite value.  Returns uint8 codes.
    NaN inputs are rejected: the quantizer never produces them."""
    fmt = get(fmt)
    v = np.asarray(values, dtype=np.float32).astype(np.float64)
    if np.isnan(v).any():
        raise ValueError("NaN input to encode")
    neg = np.signbit(v)
    if not fmt.signed and (neg & (v != 0)).any():
        raise ValueError(f"negative input to unsigned format {fmt.name}")
    mag = np.abs(v)
    codes, vals = _positive_finite(fmt)
    top = vals[-1]
    mag = np.minimum(mag, top)                      # satfinite
    hi = np.searchsorted(vals, mag, side="left")    # vals[hi] >= mag
    hi = np.minimum(hi, len(vals) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = mag - vals[lo]                           # exact in float64
    d_hi = vals[hi] - mag
    exact = vals[hi] == mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0))
    mag_code = np.where(exact, codes[hi], np.where(pick_hi, codes[hi], codes[lo]))
    if fmt.signed:
        mag_code = mag_code | (neg.astype(np.int64) << (fmt.bits - 1))
    return mag_code.astype(np.uint8)


def pack_e2m1(codes) -> np.ndarray:
    """Pack 4-bit codes two per byte along the last axis, even element in the
    low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    if c.shape[-1] % 2:
        raise ValueError("E2M1 packing needs an even last dimension")
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> the binary32 values they denote."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)
