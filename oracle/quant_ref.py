"""Plain numpy restatement of the fp8 query quantisation (fused with the pack).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: the "mjolnir/t5_decode.py" page, `quantize_q_fp8` and `pack_q` (host
helpers section).  Per sequence b and kv head g the page takes the largest
magnitude of Q over the group's q_len tokens, its h_r query heads and d,
raises it to at least 1e-6, divides it by 448 (the largest e4m3 value) to
get the group's fp32 descale, and stores e4m3(q / descale) for every element
of the group; the kernel layout then packs the group's rows qi-major,
(b, h_k, q_len*h_r, d).  Everything is fp32, as on the page (`q.float()`,
an fp32 amax and fp32 divisions); the encoder below rounds to nearest with
ties to even and saturates at +-448 (the page's values never exceed 448, as
|q| <= amax).

The encoder is written here from the format definition (sign, 4-bit
exponent with bias 7, 3-bit mantissa, exponent 0 subnormal, S.1111.111 NaN)
and shares nothing with the input generator's encoder or the CUDA path.
"""

from __future__ import annotations

from typing import Tuple

import numpy as np

from .layout_ref import pack_q_ref

E4M3_MAX = 448.0
AMAX_FLOOR = np.float32(1e-6)


def e4m3_encode_rne(x: np.ndarray) -> np.ndarray:
    """e4m3 (FN) codes of fp32 values: round to nearest, ties to even,
    saturate finite overflow to +-448, NaN -> 0x7F."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)  # exact copy
    out = np.zeros(x.shape, dtype=np.uint8)
    flat, res = x.reshape(-1), out.reshape(-1)
    for i, v in enumerate(flat):
        if np.isnan(v):
            res[i] = 0x7F
            continue
        sign = 0x80 if np.signbit(v) else 0x00
        a = abs(v)
        if a >= E4M3_MAX:
            res[i] = sign | 0x7E  # saturate (448 itself included)
            continue
        # the representable grid near a: spacing 2^(e-3) for a in [2^e, 2^(e+1)),
        # e >= -6; subnormals share the spacing 2^-9 below 2^-6
        if a < 2.0**-6:
            step = 2.0**-9
        else:
            e = int(np.floor(np.log2(a)))
            # guard log2's rounding at exact powers of two
            if 2.0**e > a:
                e -= 1
            elif 2.0 ** (e + 1) <= a:
                e += 1
            step = 2.0 ** (e - 3)
        q = a / step  # exact: a power-of-two scaling
        lo = np.floor(q)
        frac = q - lo
        n = lo + 1 if (frac > 0.5 or (frac == 0.5 and int(lo) % 2 == 1)) else lo
        mag = n * step
        if mag > E4M3_MAX:
            mag = E4M3_MAX
        res[i] = sign | _code_of_magnitude(mag)
    return out


def _code_of_magnitude(m: float) -> int:
    """Bits of a non-negative representable magnitude m <= 448."""
    if m == 0.0:
        return 0
    if m < 2.0**-6:  # subnormal: m = k 2^-9, k in 1..7
        return int(round(m / 2.0**-9))
    e = int(np.floor(np.log2(m)))
    if 2.0**e > m:
        e -= 1
    mant = int(round((m / 2.0**e - 1.0) * 8))
    if mant == 8:  # rounded up into the next binade
        e, mant = e + 1, 0
    return ((e + 7) << 3) | mant


def quantize_pack_q_ref(
    q_vllm: np.ndarray, num_seqs: int, q_len: int, h_k: int, h_r: int
) -> Tuple[np.ndarray, np.ndarray]:
    """q_vllm: float32 values (num_seqs * q_len, h_k * h_r, d) (bf16 inputs
    converted exactly).  Returns (codes uint8 (num_seqs, h_k, q_len * h_r, d),
    descale float32 (num_seqs, h_k))."""
    q = np.asarray(q_vllm, dtype=np.float32)
    d = q.shape[-1]
    qg = q.reshape(num_seqs, q_len, h_k, h_r, d)
    amax = np.abs(qg).max(axis=(1, 3, 4)).astype(np.float32)  # (b, h_k), exact
    amax = np.maximum(amax, AMAX_FLOOR)
    descale = (amax / np.float32(E4M3_MAX)).astype(np.float32)  # fp32 division
    x = (qg / descale[:, None, :, None, None]).astype(np.float32)  # fp32 divisions
    codes = e4m3_encode_rne(x).reshape(num_seqs * q_len, h_k * h_r, d)
    return pack_q_ref(codes, num_seqs, q_len, h_k, h_r), descale
