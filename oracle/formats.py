"""Number formats of the cache and the indexer query, decoded in float64.

Test infrastructure only (see the package docstring).

The formats are those the vLLM Kimi K3.1 Pro article names in "面向三种状态的
KV 缓存" and "KV 缓存占用" (FP8 E4M3 keys and latents, NVFP4 latents, MXFP4 index
keys). Their bit layouts are the OCP definitions:

* E4M3 (OCP 8-bit floating point, "FN" variant): 1 sign, 4 exponent (bias 7),
  3 mantissa bits; exponent 0 is subnormal (2**-6 * m/8); no infinities;
  S.1111.111 is NaN; largest finite 448.
* E2M1 (OCP MX FP4): 1 sign, 2 exponent (bias 1), 1 mantissa bit; exponent 0
  is subnormal (m/2); magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}.
* E8M0 (OCP MX scale): 2**(e - 127); 0xFF is NaN.
* bf16: the upper 16 bits of an IEEE binary32.
"""
from __future__ import annotations

import numpy as np


def e4m3_table() -> np.ndarray:
    """Value of each of the 256 E4M3 codes, float64 (NaN for 0x7F and 0xFF)."""
    t = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        exp = (code >> 3) & 0xF
        man = code & 0x7
        if exp == 0xF and man == 0x7:
            t[code] = np.nan
        elif exp == 0:
            t[code] = sign * (man / 8.0) * 2.0 ** (1 - 7)
        else:
            t[code] = sign * (1.0 + man / 8.0) * 2.0 ** (exp - 7)
    return t


E4M3 = e4m3_table()


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    return E4M3[np.asarray(codes, dtype=np.uint8)]


def e2m1_table() -> np.ndarray:
    """Value of each of the 16 E2M1 codes (sign in bit 3), float64."""
    t = np.empty(16, dtype=np.float64)
    for code in range(16):
        sign = -1.0 if code & 0x8 else 1.0
        exp = (code >> 1) & 0x3
        man = code & 0x1
        t[code] = sign * (man / 2.0 if exp == 0 else (1.0 + man / 2.0) * 2.0 ** (exp - 1))
    return t


E2M1 = e2m1_table()


def e2m1_unpack(packed: np.ndarray) -> np.ndarray:
    """Bytes holding two E2M1 codes (element 2i in the low nibble) -> float64, twice as long."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.float64)
    out[..., 0::2] = E2M1[p & 0xF]
    out[..., 1::2] = E2M1[p >> 4]
    return out


def e8m0_decode(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.int64)
    return np.where(c == 0xFF, np.nan, np.ldexp(1.0, c - 127))


def bf16_decode(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def f32_from_bytes(raw: np.ndarray) -> np.ndarray:
    """Little-endian fp32 values from a uint8 array whose last axis is 4*n bytes."""
    r = np.ascontiguousarray(raw, dtype=np.uint8)
    return r.view("<f4").astype(np.float32)


def e4m3_encode_rne_satfinite(x: np.ndarray) -> np.ndarray:
    """fp32 values -> E4M3 codes, round to nearest (ties to the even code), saturating.

    Magnitudes above 448 become +-448 (the saturating "satfinite" conversion);
    NaN becomes 0x7F. Each value is compared against the exact code values, so
    the result is the correctly rounded code.
    """
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    pos = E4M3[:127]                      # codes 0..126, increasing
    a = np.minimum(np.abs(x), 448.0)
    hi = np.clip(np.searchsorted(pos, a, side="left"), 1, 126)
    lo = hi - 1
    d_lo = a - pos[lo]
    d_hi = pos[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo)
    code = np.where(a == pos[hi], hi, code)
    code = np.where(a == 0.0, 0, code).astype(np.uint8)
    code = code | np.where(np.signbit(x), 0x80, 0).astype(np.uint8)
    return np.where(np.isnan(x), 0x7F, code).astype(np.uint8)
