"""A compact 656-byte latent row for the host link, and its value.

TEST INFRASTRUCTURE ONLY.  Only the tests may import this module.  It shares
no code with the CUDA library.

The "ESS: Latent-Cache Offload" page (foosynaptic tech notes) names the
latent entry c^KV[512] + k^R[64], says in its summary that the indexer cache
is about 16.8% and the latent cache about 83.2% of the per-token bytes, and
in its table of mechanisms (the FlashTrans + UVA row) quotes host transfers
of about 656 bytes.  A 656-byte latent entry beside a 132-byte indexer entry
(128 e4m3 values and a float32 scale) gives exactly that split.  The pages
do not lay the 656 bytes out; the reading taken here (656 = 512 + 16 + 128):

  bytes   0..511  the 512 latent values as FP8 e4m3, four tiles of 128;
  bytes 512..527  one float32 scale per tile (little-endian);
  bytes 528..655  the 64 RoPE values, bf16 as they were.

Encoding a tile: its scale is the smallest power of two at or above
fl32(amax / 448) (1 when the tile is all zero), where amax is the largest
magnitude in the tile and 448 the largest finite e4m3 value; a power of two,
like the shared block exponents of the OCP microscaling (MX) formats, so that
every decoded value code * scale is exact in bf16 and a GPU can widen a row
into the bf16 operands of its attention without rounding.  Each value becomes
e4m3(x / scale) (exact division), rounded to nearest with ties to the even
code; the largest magnitude lands in (224, 448], and anything at or above 448
saturates there; the sign of a value that rounds to zero is kept.  The row's
value is code * scale, exact in float64 and in bf16.
"""
from __future__ import annotations

import numpy as np

ROW_BYTES = 656
LATENT = 512
ROPE = 64
TILE = 128
E4M3_MAX = 448.0


def e4m3_value(code: int) -> float:
    """Value of an e4m3 byte: 1 sign bit, 4 exponent bits (bias 7), 3
    mantissa bits; exponent 0 is subnormal; 0x7F and 0xFF are NaN."""
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_POS_CODES = np.arange(0x7F)                            # 0x00..0x7E: +0 .. 448
_POS_VALUES = np.array([e4m3_value(int(c)) for c in _POS_CODES])


def e4m3_encode(v: float) -> int:
    """Round v to the nearest e4m3 value (ties to the even code), saturating
    at +-448; returns the byte."""
    sign = 0x80 if (v < 0 or (v == 0 and np.signbit(v))) else 0
    a = abs(float(v))
    if a >= E4M3_MAX:
        return sign | 0x7E
    i = int(np.searchsorted(_POS_VALUES, a))            # first level >= a
    if _POS_VALUES[i] == a:
        return sign | int(_POS_CODES[i])
    lo, hi = i - 1, i
    dlo, dhi = a - _POS_VALUES[lo], _POS_VALUES[hi] - a
    if dlo < dhi or (dlo == dhi and _POS_CODES[lo] % 2 == 0):
        return sign | int(_POS_CODES[lo])
    return sign | int(_POS_CODES[hi])


def tile_scale(amax: np.float32) -> np.float32:
    """The smallest power of two >= fl32(amax / 448); 1 for amax = 0."""
    if not amax > 0:
        return np.float32(1.0)
    q = np.float32(np.float32(amax) / np.float32(E4M3_MAX))
    m, e = np.frexp(q)                                  # q = m * 2^e, m in [0.5, 1)
    return np.float32(np.ldexp(1.0, int(e) - 1) if m == 0.5 else np.ldexp(1.0, int(e)))


def encode_row(bits: np.ndarray) -> np.ndarray:
    """bf16 bits [576] of one latent row -> uint8 [656]."""
    bits = np.asarray(bits, dtype=np.uint16)
    x = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    out = np.zeros(ROW_BYTES, dtype=np.uint8)
    scales = np.zeros(LATENT // TILE, dtype=np.float32)
    for j in range(LATENT // TILE):
        tile = x[j * TILE:(j + 1) * TILE]
        scale = tile_scale(np.float32(np.max(np.abs(tile))))
        scales[j] = scale
        q = (tile / scale).astype(np.float32)           # exact: the scale is a power of two
        out[j * TILE:(j + 1) * TILE] = [e4m3_encode(float(v)) for v in q]
    out[LATENT:LATENT + 16] = scales.astype("<f4").view(np.uint8)
    out[LATENT + 16:] = bits[LATENT:].astype("<u2").view(np.uint8)
    return out


def decode_row(row: np.ndarray) -> np.ndarray:
    """uint8 [656] -> float64 [576], the value the compact row stands for."""
    row = np.asarray(row, dtype=np.uint8)
    scales = row[LATENT:LATENT + 16].view("<f4").astype(np.float64)
    codes = row[:LATENT]
    lat = np.array([e4m3_value(int(c)) for c in codes]) * np.repeat(scales, TILE)
    rope_bits = row[LATENT + 16:].view("<u2").astype(np.uint32) << np.uint32(16)
    rope = rope_bits.view(np.float32).astype(np.float64)
    return np.concatenate([lat, rope])


_CODE_VALUES = np.array([e4m3_value(c) for c in range(256)])   # NaN for 0x7F, 0xFF


def decode_rows(rows: np.ndarray) -> np.ndarray:
    """uint8 [n][656] -> float64 [n][576]: decode_row for many rows at once
    (a table lookup of the codes times each tile's scale)."""
    rows = np.ascontiguousarray(rows, dtype=np.uint8).reshape(-1, ROW_BYTES)
    scales = rows[:, LATENT:LATENT + 16].copy().view("<f4").astype(np.float64)   # [n][4]
    lat = _CODE_VALUES[rows[:, :LATENT]] * np.repeat(scales, TILE, axis=1)
    rope_bits = rows[:, LATENT + 16:].copy().view("<u2").astype(np.uint32) << np.uint32(16)
    rope = rope_bits.view(np.float32).astype(np.float64)
    return np.concatenate([lat, rope], axis=1)
