"""Pins of the oracle's fp8 query quantisation (oracle/quant_ref.py), CPU only.

What fixes each part, independently of the oracle's own code:
* the encoder: every finite e4m3 value (from the oracle's decode table,
  itself pinned against the format and torch) encodes to its own code;
  midpoints between neighbours go to the even code; saturation and NaN;
  agreement with torch's float8_e4m3fn cast (a library routine) on random
  in-range values, the subnormal range included;
* the quantisation: a hand-worked example of the page's definition
  (tests/golden/quantize_q_example.json), the group maximum landing on
  +-448, an all-zero group, the error bound of round-to-nearest, and every
  element's placement checked by a brute-force loop over the vLLM layout.

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
import oracle.quant_ref as quant_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def pin_round_trip(m):
    tab = oracle.e4m3_table()
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        v = np.float32(tab[c])
        assert int(m.e4m3_encode_rne(np.array([v]))[0]) == c, hex(c)


def pin_midpoints(m):
    tab = oracle.e4m3_table()
    for c in range(0x7E):  # positive neighbours c, c + 1
        lo, hi = tab[c], tab[c + 1]
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2  # exact in fp32
        even = c if c % 2 == 0 else c + 1
        assert int(m.e4m3_encode_rne(np.array([mid]))[0]) == even
        assert int(m.e4m3_encode_rne(np.array([-mid]))[0]) == (even | 0x80)
        # just off the midpoint: the nearer neighbour
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(1000))
        assert int(m.e4m3_encode_rne(np.array([below]))[0]) == c
        assert int(m.e4m3_encode_rne(np.array([above]))[0]) == c + 1


def pin_saturation_and_specials(m):
    vals = np.array([448.0, 460.0, 464.0, 1e6, np.inf], dtype=np.float32)
    assert list(m.e4m3_encode_rne(vals)) == [0x7E] * 5
    assert list(m.e4m3_encode_rne(-vals)) == [0xFE] * 5
    assert int(m.e4m3_encode_rne(np.array([np.nan], dtype=np.float32))[0]) == 0x7F
    assert int(m.e4m3_encode_rne(np.array([-0.0], dtype=np.float32))[0]) == 0x80
    # below half the smallest subnormal: zero; exactly half: ties to even (0)
    assert list(m.e4m3_encode_rne(np.array([2.0**-11, 2.0**-10], dtype=np.float32))) == [0, 0]
    assert int(m.e4m3_encode_rne(np.array([2.0**-10 * 1.01], dtype=np.float32))[0]) == 1


def pin_torch_cast(m):
    rng = np.random.default_rng(11)
    x = np.concatenate(
        [rng.normal(0, 1, 4000), rng.normal(0, 100, 2000), rng.uniform(-448, 448, 2000), rng.normal(0, 1e-3, 2000)]
    ).astype(np.float32)
    ours = m.e4m3_encode_rne(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def pin_hand_worked_example(m):
    g = json.load(open(os.path.join(GOLDEN, "quantize_q_example.json")))
    sh = g["shape"]
    q = np.array(g["q"], dtype=np.float32).reshape(sh["num_seqs"] * sh["q_len"], sh["h_k"] * sh["h_r"], sh["d"])
    codes, descale = m.quantize_pack_q_ref(q, sh["num_seqs"], sh["q_len"], sh["h_k"], sh["h_r"])
    assert descale.dtype == np.float32
    assert hex(descale.view(np.uint32)[0, 0]) == g["descale_fp32_hex"]
    assert [hex(c) for c in codes.reshape(-1)] == g["codes"]


def pin_layout_bound_and_group_maximum(m, num_seqs, q_len, h_k, h_r, d):
    rng = np.random.default_rng(num_seqs * 100 + q_len)
    q = rng.normal(0, 1, (num_seqs * q_len, h_k * h_r, d)).astype(np.float32)
    q[:q_len, :h_r, :] = 0.0  # sequence 0, kv head 0: an all-zero group
    codes, descale = m.quantize_pack_q_ref(q, num_seqs, q_len, h_k, h_r)
    tab = oracle.e4m3_table()
    assert codes.shape == (num_seqs, h_k, q_len * h_r, d) and descale.shape == (num_seqs, h_k)
    assert descale[0, 0] == np.float32(1e-6) / np.float32(448.0)
    for b in range(num_seqs):
        for g in range(h_k):
            grp = q.reshape(num_seqs, q_len, h_k, h_r, d)[b, :, g]
            amax = np.float32(np.abs(grp).max())
            if amax == 0:
                assert not codes[b, g].any()
                continue
            assert descale[b, g] == amax / np.float32(448.0)
            # brute force over the vLLM layout: token qi, head g*h_r + hr
            for qi in range(q_len):
                for hr in range(h_r):
                    row = codes[b, g, qi * h_r + hr]
                    src = q[b * q_len + qi, g * h_r + hr]
                    back = tab[row] * float(descale[b, g])
                    err = np.abs(back - src.astype(np.float64))
                    # round to nearest: half a step, 2^-4 relative for normals,
                    # 2^-10 descale absolute below the normal range
                    assert np.all(err <= np.abs(src) * 2.0**-4 + float(descale[b, g]) * 2.0**-10 * 1.0001)
                    top = np.abs(src) == amax
                    assert np.all((row[top] & 0x7F) == 0x7E)


LAYOUT_CASES = [(2, 1, 1, 16, 128), (3, 4, 2, 8, 16), (2, 5, 3, 2, 32)]


def all_pins(m):
    """Every pin against module m (raises on the first that fails)."""
    pin_round_trip(m)
    pin_midpoints(m)
    pin_saturation_and_specials(m)
    pin_torch_cast(m)
    pin_hand_worked_example(m)
    for case in LAYOUT_CASES:
        pin_layout_bound_and_group_maximum(m, *case)


def test_encoder_round_trips_every_finite_code():
    pin_round_trip(quant_ref)


def test_encoder_midpoints_go_to_the_even_code():
    pin_midpoints(quant_ref)


def test_encoder_saturates_and_maps_nan():
    pin_saturation_and_specials(quant_ref)


def test_encoder_matches_torch_cast_in_range():
    pin_torch_cast(quant_ref)


def test_hand_worked_example():
    pin_hand_worked_example(quant_ref)


@pytest.mark.parametrize("num_seqs,q_len,h_k,h_r,d", LAYOUT_CASES)
def test_quantise_layout_bound_and_group_maximum(num_seqs, q_len, h_k, h_r, d):
    pin_layout_bound_and_group_maximum(quant_ref, num_seqs, q_len, h_k, h_r, d)
