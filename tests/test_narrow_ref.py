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
* the e4m3 view: each narrow value equals the e4m3 value of its mapped code;
* nvfp4: hand-worked (code, scale) pairs (tests/golden/nvfp4_examples.json),
  every one of the 16 x 256 pairs within half an e4m3 step of the exact
  product (brute force), and the scale of element i being that of group
  i // 16.

Each pin is a function of the module under test, so that
tests/test_oracle_mutations.py can run the same pins against copies of the
module with planted mistakes.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.narrow_ref as narrow_ref

TABLE_SHAPES = [("e3m2", 28.0, 2.0**-4), ("e2m3", 7.5, 2.0**-3), ("e2m1", 6.0, 0.5)]
FMTS = ["e3m2", "e2m3", "e2m1"]


def pin_e2m1_values(m):
    t = m.minifloat_table("e2m1")
    assert list(t[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(t[8:]) == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


def pin_table_shape(m, fmt, largest, step):
    eb, mb, bias = m.FORMATS[fmt]
    t = m.minifloat_table(fmt)
    pos = t[: len(t) // 2]
    assert len(t) == 1 << m.BITS[fmt] == 1 << (1 + eb + mb)
    assert pos[-1] == largest
    assert pos[1] == step  # smallest subnormal: 2^(1 - bias - mb)
    assert np.all(np.diff(pos) > 0)  # strictly ascending: every code distinct
    assert np.array_equal(t[len(t) // 2 :], -pos)


def pin_encoder(m, fmt):
    t = m.minifloat_table(fmt)
    half = len(t) // 2
    for c in range(len(t)):
        want = 0 if t[c] == 0 else c  # negative zero is never produced
        assert int(m.minifloat_encode(np.array([t[c]]), fmt)[0]) == want
    pos = t[:half]
    for i in range(half - 1):
        mid = (pos[i] + pos[i + 1]) / 2
        assert int(m.minifloat_encode(np.array([mid]), fmt)[0]) == i  # tie: the smaller one
        assert int(m.minifloat_encode(np.array([np.nextafter(mid, np.inf)]), fmt)[0]) == i + 1
        assert int(m.minifloat_encode(np.array([-mid]), fmt)[0]) == (i + half if pos[i] > 0 else 0)
    assert int(m.minifloat_encode(np.array([1e9]), fmt)[0]) == half - 1
    assert int(m.minifloat_encode(np.array([-1e9]), fmt)[0]) == len(t) - 1


def pin_packing_bytes(m):
    assert list(m.pack_bits(np.array([1, 2, 0xF, 0x0]), 4)) == [0x21, 0x0F]
    # 1 | 2 << 6 | 3 << 12 | 4 << 18 = 0x103081, little-endian
    assert list(m.pack_bits(np.array([1, 2, 3, 4]), 6)) == [0x81, 0x30, 0x10]


def pin_packing_round_trip(m, bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 1 << bits, size=(3, 5, 128)).astype(np.uint8)
    packed = m.pack_bits(codes, bits)
    assert packed.shape == (3, 5, 128 * bits // 8)
    assert np.array_equal(m.unpack_bits(packed, bits, 128), codes)


def pin_e4m3_view(m, fmt):
    e4 = oracle.e4m3_table()
    t = m.minifloat_table(fmt)
    mapped = m.to_e4m3_codes(np.arange(len(t)), fmt, e4)
    assert np.array_equal(e4[mapped], np.where(t == 0, 0.0, t))
    rng = np.random.default_rng(3)
    c = m.minifloat_encode(rng.normal(0, 2, 1000), fmt)
    assert np.array_equal(e4[m.to_e4m3_codes(c, fmt, e4)], t[c] + 0.0)


GOLDEN_NVFP4 = os.path.join(os.path.dirname(__file__), "golden", "nvfp4_examples.json")


def pin_nvfp4_golden(m):
    for c in json.load(open(GOLDEN_NVFP4))["cases"]:
        got = m.nvfp4_to_e4m3_codes(np.full((1, 16), c["code"]), np.array([[c["scale"]]]))
        assert np.all(got == c["expect"]), c["why"]


def pin_nvfp4_rounding_bound(m):
    e4 = oracle.e4m3_table()
    e2 = m.minifloat_table("e2m1")
    codes = np.repeat(np.arange(16), 16)[None, :]  # group g holds code g
    for sc in range(256):
        if sc in (0x7F, 0xFF):
            continue
        got = e4[m.nvfp4_to_e4m3_codes(codes, np.full((1, 16), sc))][0, ::16]
        exact = e2 * e4[sc] / 8.0
        # half a step of e4m3 at the exact value (2^-10 below the normal range)
        mag = np.maximum(np.abs(exact), 2.0**-6)
        half = 2.0 ** (np.floor(np.log2(mag)) - 4)
        assert np.all(np.abs(got - exact) <= half * (1 + 1e-12)), sc


def pin_nvfp4_groups(m):
    codes = np.full((2, 128), 4)  # 2.0 everywhere
    scales = np.arange(16).reshape(2, 8) * 8 + 0x38  # distinct scales per group
    e4 = oracle.e4m3_table()
    got = e4[m.nvfp4_to_e4m3_codes(codes, scales)]
    for r in range(2):
        for i in range(128):
            assert got[r, i] == e4[m.nvfp4_to_e4m3_codes(np.full((1, 16), 4), scales[r : r + 1, i // 16 : i // 16 + 1])][0, 0]
    assert len(set(got[0, ::16])) == 8


def all_pins(m):
    """Every pin against module m (raises on the first that fails)."""
    pin_e2m1_values(m)
    for case in TABLE_SHAPES:
        pin_table_shape(m, *case)
    for fmt in FMTS:
        pin_encoder(m, fmt)
        pin_e4m3_view(m, fmt)
    pin_packing_bytes(m)
    for bits in (4, 6):
        pin_packing_round_trip(m, bits)
    pin_nvfp4_golden(m)
    pin_nvfp4_rounding_bound(m)
    pin_nvfp4_groups(m)


def test_e2m1_values():
    pin_e2m1_values(narrow_ref)


@pytest.mark.parametrize("fmt,largest,step", TABLE_SHAPES)
def test_table_shape(fmt, largest, step):
    pin_table_shape(narrow_ref, fmt, largest, step)


def test_e2m1_against_torch_if_available():
    dt = getattr(torch, "float4_e2m1fn_x2", None)
    if dt is None:
        pytest.skip("torch has no float4_e2m1fn_x2")
    try:
        vals = torch.arange(256, dtype=torch.uint8).view(dt).to(torch.float32)
    except Exception:
        pytest.skip("this torch cannot convert float4_e2m1fn_x2 to float32")
    t = narrow_ref.minifloat_table("e2m1")
    ref = np.array([[t[c & 0xF], t[c >> 4]] for c in range(256)], dtype=np.float32).reshape(-1)
    assert np.array_equal(vals.reshape(-1).numpy(), ref)


@pytest.mark.parametrize("fmt", FMTS)
def test_encoder_round_trip_ties_and_saturation(fmt):
    pin_encoder(narrow_ref, fmt)


def test_packing_bytes_by_hand():
    pin_packing_bytes(narrow_ref)


@pytest.mark.parametrize("bits", [4, 6])
def test_packing_round_trip(bits):
    pin_packing_round_trip(narrow_ref, bits)


@pytest.mark.parametrize("fmt", FMTS)
def test_e4m3_view_is_exact(fmt):
    pin_e4m3_view(narrow_ref, fmt)


def test_nvfp4_hand_worked_examples():
    pin_nvfp4_golden(narrow_ref)


def test_nvfp4_rounding_bound_over_every_pair():
    pin_nvfp4_rounding_bound(narrow_ref)


def test_nvfp4_scale_groups():
    pin_nvfp4_groups(narrow_ref)
