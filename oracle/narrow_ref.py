"""Plain restatement of the narrow KV formats (fp6 e3m2 / e2m3, fp4 e2m1).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: the "mjolnir/t5_decode.py" page, "Narrow KV formats: value tables,
quantization and bit packing" (module helpers) and the KV-format constants.
Each format is sign | exponent | mantissa with a bias, a subnormal binade at
exponent 0 and no infinities or NaN:

    e3m2: 3 exponent bits, 2 mantissa bits, bias 3   (largest 28)
    e2m3: 2 exponent bits, 3 mantissa bits, bias 1   (largest 7.5)
    e2m1: 2 exponent bits, 1 mantissa bit,  bias 1   (largest 6)

The page's quantiser rounds |x| (clamped to the largest value) to the
nearer of its two neighbours in the non-negative table, a tie going to the
smaller one, and gives the code the sign bit only when the magnitude is not
zero.  Codes are packed little-endian into a bit stream (fp4: element 2i in
the low nibble of byte i; fp6: four elements in three bytes).

Every value of the three formats is also an e4m3 value, so an attention
problem with narrow KV is the same problem with the equal e4m3 codes:
`to_e4m3_codes` maps them exactly, and the fp64 attention oracle then
applies unchanged.  Written from the format definition; shares nothing
with any encoder of the CUDA path or of the input generator.
"""

from __future__ import annotations

from typing import Dict, Tuple

import numpy as np

# format: (exponent bits, mantissa bits, bias)
FORMATS: Dict[str, Tuple[int, int, int]] = {"e3m2": (3, 2, 3), "e2m3": (2, 3, 1), "e2m1": (2, 1, 1)}
BITS = {"e3m2": 6, "e2m3": 6, "e2m1": 4}


def minifloat_value(code: int, fmt: str) -> float:
    eb, mb, bias = FORMATS[fmt]
    sign = -1.0 if (code >> (eb + mb)) & 1 else 1.0
    e = (code >> mb) & ((1 << eb) - 1)
    m = code & ((1 << mb) - 1)
    if e == 0:
        mag = (m / (1 << mb)) * 2.0 ** (1 - bias)
    else:
        mag = (1.0 + m / (1 << mb)) * 2.0 ** (e - bias)
    return sign * mag


def minifloat_table(fmt: str) -> np.ndarray:
    """float64 value of every code (2^bits entries; the upper half negative)."""
    return np.array([minifloat_value(c, fmt) for c in range(1 << BITS[fmt])], dtype=np.float64)


def minifloat_encode(x: np.ndarray, fmt: str) -> np.ndarray:
    """Codes of x: round to nearest, ties to the smaller magnitude,
    saturating at the largest value; zero (either sign) -> code 0."""
    table = minifloat_table(fmt)
    half = len(table) // 2
    pos = table[:half]  # 0 .. largest, ascending
    xs = np.asarray(x, dtype=np.float64)
    out = np.empty(xs.shape, dtype=np.uint8)
    flat, res = xs.reshape(-1), out.reshape(-1)
    for i, v in enumerate(flat):
        a = min(abs(v), pos[-1])
        hi = int(np.searchsorted(pos, a, side="left"))  # first value >= a
        if hi == 0:
            mag = 0
        else:
            lo = hi - 1
            hi = min(hi, half - 1)
            mag = lo if (a - pos[lo]) <= (pos[hi] - a) else hi
        neg = v < 0 and pos[mag] > 0
        res[i] = mag + (half if neg else 0)
    return out


def pack_bits(codes: np.ndarray, bits: int) -> np.ndarray:
    """Little-endian bit stream of the last axis: element i at bits
    [bits*i, bits*(i+1)).  fp4 needs an even length, fp6 a multiple of 4."""
    c = np.asarray(codes, dtype=np.uint64)
    d = c.shape[-1]
    if bits == 4:
        assert d % 2 == 0
        c = c.reshape(*c.shape[:-1], d // 2, 2)
        return (c[..., 0] | (c[..., 1] << np.uint64(4))).astype(np.uint8)
    assert bits == 6 and d % 4 == 0
    c = c.reshape(*c.shape[:-1], d // 4, 4)
    w = c[..., 0] | (c[..., 1] << np.uint64(6)) | (c[..., 2] << np.uint64(12)) | (c[..., 3] << np.uint64(18))
    out = np.stack([w & np.uint64(0xFF), (w >> np.uint64(8)) & np.uint64(0xFF), (w >> np.uint64(16)) & np.uint64(0xFF)], axis=-1)
    return out.reshape(*c.shape[:-2], d // 4 * 3).astype(np.uint8)


def unpack_bits(packed: np.ndarray, bits: int, d: int) -> np.ndarray:
    """Inverse of pack_bits for a last axis of d codes."""
    p = np.asarray(packed, dtype=np.uint64)
    if bits == 4:
        lo, hi = p & np.uint64(0xF), p >> np.uint64(4)
        return np.stack([lo, hi], axis=-1).reshape(*p.shape[:-1], d).astype(np.uint8)
    assert bits == 6
    p = p.reshape(*p.shape[:-1], d // 4, 3)
    w = p[..., 0] | (p[..., 1] << np.uint64(8)) | (p[..., 2] << np.uint64(16))
    parts = [(w >> np.uint64(6 * k)) & np.uint64(0x3F) for k in range(4)]
    return np.stack(parts, axis=-1).reshape(*p.shape[:-2], d).astype(np.uint8)


def to_e4m3_codes(codes: np.ndarray, fmt: str, e4m3_table: np.ndarray) -> np.ndarray:
    """The e4m3 code of equal value for every narrow code (exact: each
    narrow value is an e4m3 value; zero maps to +0)."""
    table = minifloat_table(fmt)
    lut = np.zeros(len(table), dtype=np.uint8)
    for c, v in enumerate(table):
        hits = [k for k in range(256) if k not in (0x7F, 0xFF, 0x80) and e4m3_table[k] == v]
        if len(hits) != 1:
            raise ValueError(f"{fmt} code {c} ({v}) has no unique e4m3 equal")
        lut[c] = hits[0]
    return lut[np.asarray(codes, dtype=np.int64)]
