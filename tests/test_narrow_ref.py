"""Pins of the oracle's narrow KV formats (oracle/narrow_ref.py), CPU only.

What fixes each part, independently of the oracle's own code:
* the value tables: the fp4 e2m1 magnitudes are the set the page's nvfp4
  comment relies on (codes up to 6); the fp6 tables' largest values, the
  subnormal steps and the number of distinct magnitudes follow from the
  exponent / mantissa widths and biases the page lists; e2m1 against
  torch's float4_e2m1fn_x2 where the installed torch can decode it;
* the encoder: every table value to its own code, midpoints to the smaller
  neighbour (the page's tie rule), saturation, no negative-zero codes;
* the packing: hand-written bytes for a few codes, and round trips;
* the e4m3 view: each narrow value equals the e4m3 value of its mapped code.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle.narrow_ref import (
    BITS,
    FORMATS,
    minifloat_encode,
    minifloat_table,
    pack_bits,
    to_e4m3_codes,
    unpack_bits,
)


def test_e2m1_values():
    t = minifloat_table("e2m1")
    assert list(t[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(t[8:]) == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


@pytest.mark.parametrize("fmt,largest,step", [("e3m2", 28.0, 2.0**-4), ("e2m3", 7.5, 2.0**-3), ("e2m1", 6.0, 0.5)])
def test_table_shape(fmt, largest, step):
    eb, mb, bias = FORMATS[fmt]
    t = minifloat_table(fmt)
    pos = t[: len(t) // 2]
    assert len(t) == 1 << BITS[fmt] == 1 << (1 + eb + mb)
    assert pos[-1] == largest
    assert pos[1] == step  # smallest subnormal: 2^(1 - bias - mb)
    assert np.all(np.diff(pos) > 0)  # strictly ascending: every code distinct
    assert np.array_equal(t[len(t) // 2 :], -pos)


def test_e2m1_against_torch_if_available():
    dt = getattr(torch, "float4_e2m1fn_x2", None)
    if dt is None:
        pytest.skip("torch has no float4_e2m1fn_x2")
    try:
        packed = torch.arange(256, dtype=torch.uint8).view(dt)
        lo_hi = packed.to(torch.float32)
    except Exception:
        pytest.skip("this torch cannot convert float4_e2m1fn_x2 to float32")
    t = minifloat_table("e2m1")
    ref = np.array([[t[c & 0xF], t[c >> 4]] for c in range(256)], dtype=np.float32).reshape(-1)
    assert np.array_equal(lo_hi.reshape(-1).numpy(), ref)


@pytest.mark.parametrize("fmt", list(FORMATS))
def test_encoder_round_trip_ties_and_saturation(fmt):
    t = minifloat_table(fmt)
    half = len(t) // 2
    for c in range(len(t)):
        want = 0 if t[c] == 0 else c  # negative zero is never produced
        assert int(minifloat_encode(np.array([t[c]]), fmt)[0]) == want
    pos = t[:half]
    for i in range(half - 1):
        mid = (pos[i] + pos[i + 1]) / 2
        assert int(minifloat_encode(np.array([mid]), fmt)[0]) == i  # tie: the smaller one
        assert int(minifloat_encode(np.array([np.nextafter(mid, np.inf)]), fmt)[0]) == i + 1
        assert int(minifloat_encode(np.array([-mid]), fmt)[0]) == (i + half if pos[i] > 0 else 0)
    assert int(minifloat_encode(np.array([1e9]), fmt)[0]) == half - 1
    assert int(minifloat_encode(np.array([-1e9]), fmt)[0]) == len(t) - 1


def test_packing_bytes_by_hand():
    assert list(pack_bits(np.array([1, 2, 0xF, 0x0]), 4)) == [0x21, 0x0F]
    # 1 | 2 << 6 | 3 << 12 | 4 << 18 = 0x103081, little-endian
    assert list(pack_bits(np.array([1, 2, 3, 4]), 6)) == [0x81, 0x30, 0x10]


@pytest.mark.parametrize("bits", [4, 6])
def test_packing_round_trip(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, size=(3, 5, 128)).astype(np.uint8)
    packed = pack_bits(codes, bits)
    assert packed.shape == (3, 5, 128 * bits // 8)
    assert np.array_equal(unpack_bits(packed, bits, 128), codes)


@pytest.mark.parametrize("fmt", list(FORMATS))
def test_e4m3_view_is_exact(fmt):
    e4 = oracle.e4m3_table()
    t = minifloat_table(fmt)
    codes = np.arange(len(t))
    mapped = to_e4m3_codes(codes, fmt, e4)
    assert np.array_equal(e4[mapped], np.where(t == 0, 0.0, t))
    # quantising through the narrow format and reading it as e4m3 is a
    # value-preserving round trip for random inputs
    rng = np.random.default_rng(3)
    x = rng.normal(0, 2, 1000)
    c = minifloat_encode(x, fmt)
    assert np.array_equal(e4[to_e4m3_codes(c, fmt, e4)], t[c] + 0.0)
