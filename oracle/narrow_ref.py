"""Plain restatement of the narrow KV formats (fp6 e3m2 / e2m3, fp4 e2m1).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: the "mjolnir/t5_decode.py" page, "Narrow KV formats: value tables,
quantization and bit packing" (module helpers) and the KV-format constants.
Each format is sign | exponent | mantissa with a bias, a subnormal binade at
exponent 0 and no infinities or NaN:

    e3m2: 3 exponent bits, 2 mantissa bits, bias 3   (largest 28)
    e2m3: 2 exponent bits, 3 mantissa bits, bias 1   (largest 7.5)
    e2m1: 2 exponent bits, 1 mantissa bit,  bias 1   (largest 6)

Quantisation picks the representable magnitude nearest to |x| (the
page's quantiser settles a tie on the smaller magnitude and saturates at
the largest), with the sign bit only on a non-zero magnitude.  Codes are
laid out as one little-endian bit stream per row (so fp4 puts element 2i in
the low nibble of byte i, and fp6 fills three bytes with four elements).

nvfp4 (the same page's fourth narrow format) stores e2m1 codes with one e4m3
scale per 16 consecutive elements of a row; the value the attention uses is
the code's value times its scale times 2^-3, rounded to e4m3 (nearest, ties
to even).  The product is exact (at most six significant bits), so only that
one rounding defines the format's e4m3 view (`nvfp4_to_e4m3_codes`).

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
    """Codes of x by exhaustive nearest search: the non-negative magnitude
    at the least distance from |x|, two equally near magnitudes resolved
    to the smaller one (the tie rule of the page's `minifloat_quantize`);
    anything beyond the largest magnitude is nearest to it, so the search
    saturates by itself.  The sign bit is set for negative x whose chosen
    magnitude is not zero (no negative-zero codes)."""
    table = minifloat_table(fmt)
    half = len(table) // 2
    xs = np.asarray(x, dtype=np.float64)
    out = np.empty(xs.shape, dtype=np.uint8)
    flat, res = xs.reshape(-1), out.reshape(-1)
    for i, v in enumerate(flat):
        best, best_dist = 0, None
        for c in range(half):  # non-negative codes: magnitudes ascending
            dist = abs(abs(v) - table[c])
            if best_dist is None or dist < best_dist:  # a tie keeps the smaller
                best, best_dist = c, dist
        res[i] = best + (half if (v < 0 and table[best] != 0) else 0)
    return out


def pack_bits(codes: np.ndarray, bits: int) -> np.ndarray:
    """Little-endian bit stream of the last axis: bit k of element i is
    stream bit bits*i + k, and stream bit j is bit j % 8 of byte j // 8.
    fp4 needs an even length, fp6 a multiple of 4 (whole bytes).  One pass
    per (element, bit), over every row at once."""
    c = np.asarray(codes, dtype=np.int64)
    d = c.shape[-1]
    assert (d * bits) % 8 == 0
    flat = c.reshape(-1, d)
    out = np.zeros((flat.shape[0], d * bits // 8), dtype=np.int64)
    for i in range(d):
        for k in range(bits):
            j = bits * i + k
            out[:, j // 8] |= ((flat[:, i] >> k) & 1) << (j % 8)
    return out.astype(np.uint8).reshape(*c.shape[:-1], d * bits // 8)


def unpack_bits(packed: np.ndarray, bits: int, d: int) -> np.ndarray:
    """Inverse of pack_bits for a last axis of d codes: code i gathers
    stream bits bits*i .. bits*i + bits - 1, least significant first."""
    p = np.asarray(packed, dtype=np.int64)
    flat = p.reshape(-1, p.shape[-1])
    out = np.zeros((flat.shape[0], d), dtype=np.int64)
    for i in range(d):
        for k in range(bits):
            j = bits * i + k
            out[:, i] |= ((flat[:, j // 8] >> (j % 8)) & 1) << k
    return out.astype(np.uint8).reshape(*p.shape[:-1], d)


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


NVFP4_GROUP = 16  # elements of a row that share one e4m3 scale
NVFP4_SHIFT = 2.0**-3  # folded into the scale on the page; undone by the descale


def nvfp4_to_e4m3_codes(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """e4m3 codes of an nvfp4 row block: codes (..., d) e2m1 codes (one per
    element), scales (..., d / 16) e4m3 codes; element i takes scale
    i // 16.  Each result is the e4m3 rounding (nearest, ties to even, via
    the oracle's own encoder) of value(code) * value(scale) * 2^-3, computed
    once per (code, scale) pair; a NaN scale gives the NaN code."""
    from .quant_ref import e4m3_encode_rne
    from . import e4m3_table

    e2m1 = minifloat_table("e2m1")
    e4 = e4m3_table()
    products = np.array([[e2m1[c] * e4[sc] * NVFP4_SHIFT for sc in range(256)] for c in range(16)])
    lut = e4m3_encode_rne(products.astype(np.float32))  # exact: the products fit fp32
    c = np.asarray(codes, dtype=np.int64)
    sc = np.repeat(np.asarray(scales, dtype=np.int64), NVFP4_GROUP, axis=-1)
    return lut[c, sc]
