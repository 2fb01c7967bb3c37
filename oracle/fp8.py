"""fp8 (E4M3) attention forward (oracle; test infrastructure only: tests, the
smoke check and the bench's CPU baseline use it).

The USP README ("3. Test", the Sage/SpargeAttention test) runs a forward-only
fp8 attention backend (sage_fp8) under the same sequence-parallel wrappers;
the pages give no arithmetic for it. This module fixes the plainest reading:

  * q, k, v are stored as 8-bit E4M3 codes, each tensor with one descale
    factor: the real value of code c in a tensor with descale d is
    decode(c) * d;
  * the attention is the plain definition of oracle.attention (masks, GQA,
    varlen, LSE in natural log) applied to those real values.

E4M3 (the OCP 8-bit floating-point format, E4M3 variant): 1 sign bit, 4
exponent bits with bias 7, 3 mantissa bits. Exponent field e > 0 holds
(1 + m/8) * 2^(e-7); e = 0 holds the subnormals (m/8) * 2^-6. The largest
finite magnitude is 448 (e = 15, m = 6); e = 15, m = 7 is NaN; there are no
infinities. Encoding rounds to the nearest value, ties to the even code, and
saturates finite magnitudes beyond 448 to 448 (NaN stays NaN).

quantize(x, inv_scale) is the encoding of x * inv_scale computed in fp32 (a
product rounded to nearest), so that the codes are fixed bit for bit.
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

from oracle import attention

E4M3_MAX = 448.0
E4M3_NAN = 0x7F


def _magnitudes() -> np.ndarray:
    """Values of the non-negative finite codes 0x00 .. 0x7E, in code order."""
    out = np.zeros(0x7F, dtype=np.float64)
    for c in range(0x7F):
        e, m = c >> 3, c & 7
        out[c] = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


_MAG = _magnitudes()


def e4m3_decode(codes) -> np.ndarray:
    """uint8 codes -> float64 values (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.uint8)
    mag = np.where((c & 0x7F) == E4M3_NAN, np.nan, _MAG[np.minimum(c & 0x7F, 0x7E)])
    return np.where(c & 0x80, -mag, mag)


def e4m3_encode(x) -> np.ndarray:
    """Values -> uint8 codes: round to nearest, ties to the even code,
    saturate beyond 448, NaN -> 0x7F (sign kept)."""
    v = np.asarray(x, dtype=np.float64)
    a = np.abs(v)
    sign = np.where(np.signbit(v), 0x80, 0).astype(np.uint8)
    # the neighbouring representable magnitudes lo <= a <= hi (codes are
    # monotonic in value for a non-negative sign)
    hi = np.searchsorted(_MAG, np.minimum(a, E4M3_MAX), side="left")
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    exact = _MAG[hi] == a
    d_lo = a - _MAG[lo]
    d_hi = _MAG[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(exact, hi, np.where(pick_hi, hi, lo))
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    code = np.where(np.isnan(v), E4M3_NAN, code).astype(np.uint8)
    return code | sign


def quantize(x, inv_scale: float) -> np.ndarray:
    """Codes of x * inv_scale, the product taken in fp32."""
    p = np.asarray(x, dtype=np.float32) * np.float32(inv_scale)
    return e4m3_encode(p.astype(np.float32))


def dequantize(codes, descale: float) -> np.ndarray:
    return e4m3_decode(codes) * float(np.float32(descale))


def attn_fwd_fp8(q8, k8, v8, q_descale: float, k_descale: float, v_descale: float,
                 scale: float, causal: bool = True, window: int = 0, sink_tokens: int = 0,
                 cu_seqlens=None, heads=None) -> Tuple[np.ndarray, np.ndarray]:
    """(O, LSE) of oracle.attention.attn_fwd on the real values of the codes
    (`heads`: as there, a subset of query heads)."""
    return attention.attn_fwd(dequantize(q8, q_descale), dequantize(k8, k_descale),
                              dequantize(v8, v_descale), scale, causal, window,
                              sink_tokens, cu_seqlens=cu_seqlens, heads=heads)
