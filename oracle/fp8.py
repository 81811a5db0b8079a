"""The e4m3 (FN) 8-bit float format, written from its definition (TEST INFRASTRUCTURE ONLY).

Format: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits.  Exponent
field 0 holds the subnormals ``m * 2**-9``; the pattern ``S.1111.111`` is NaN;
there are no infinities; the largest finite magnitude is ``1.75 * 2**8 = 448``.

The pages name an fp8 scheme for batch-invariant scores ("spinf-serve"
man page, DESCRIPTION and PARAMETERS ``--quant``); its calibration needs data
that is not available, so the scale reading used here is per-row dynamic:
``scale = absmax / 448`` in fp32, values divided by the scale in fp32, then
rounded to nearest-even and saturated to +-448.
"""
from __future__ import annotations

import numpy as np


def decode(codes):
    """Values of e4m3 codes (uint8 array) as fp64."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float64)
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 15) & ((c & 7) == 7), np.nan, val)
    return sign * val


_POS_CODES = np.arange(127, dtype=np.uint8)          # 0x00 .. 0x7E: every non-negative finite value
_POS_VALUES = decode(_POS_CODES)                       # increasing with the code


def encode_rne_sat(x):
    """e4m3 code nearest to ``x`` (ties to even code), magnitudes above 448 saturated."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    d_hi = np.abs(_POS_VALUES[hi] - a)
    d_lo = np.abs(a - _POS_VALUES[lo])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    mag = np.where(pick_lo, lo, hi).astype(np.uint8)
    mag = np.where(a >= 448.0, np.uint8(126), mag)
    sign = np.where(np.signbit(x), np.uint8(0x80), np.uint8(0))
    out = (mag | sign).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), out)


def quantize_rows(x):
    """Per-row dynamic e4m3 quantisation of an fp32-representable matrix.

    Returns ``(codes uint8 [R, C], scale float32 [R])`` with
    ``scale = absmax / 448`` (fp32 division; 1 for an all-zero row) and
    ``codes = encode_rne_sat(x / scale)`` (fp32 division).
    """
    x = np.asarray(x, dtype=np.float32)
    absmax = np.max(np.abs(x), axis=1)
    scale = (absmax / np.float32(448.0)).astype(np.float32)
    scale = np.where(absmax == 0, np.float32(1.0), scale).astype(np.float32)
    scaled = (x / scale[:, None]).astype(np.float32)
    return encode_rne_sat(scaled), scale
