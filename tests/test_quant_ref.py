"""Pins of the oracle's fp8 query quantisation (oracle/quant_ref.py), CPU only.

What fixes each part, independently of the oracle's own code:
* the encoder: every finite e4m3 value (from the oracle's decode table,
  itself pinned against the format and torch) encodes to its own code;
  midpoints between neighbours go to the even code; saturation and NaN;
  agreement with torch's float8_e4m3fn cast (a library routine) on random
  in-range values;
* the quantisation: a hand-worked example of the page's definition
  (tests/golden/quantize_q_example.json), the group maximum landing on
  +-448, an all-zero group, the error bound of round-to-nearest, and every
  element's placement checked by a brute-force loop over the vLLM layout.
"""

import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle.quant_ref import e4m3_encode_rne, quantize_pack_q_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _table():
    return oracle.e4m3_table()


def test_encoder_round_trips_every_finite_code():
    tab = _table()
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        v = np.float32(tab[c])
        assert int(e4m3_encode_rne(np.array([v]))[0]) == c, hex(c)


def test_encoder_midpoints_go_to_the_even_code():
    tab = _table()
    for c in range(0x7E):  # positive neighbours c, c + 1
        lo, hi = tab[c], tab[c + 1]
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2  # exact in fp32
        even = c if c % 2 == 0 else c + 1
        assert int(e4m3_encode_rne(np.array([mid]))[0]) == even
        assert int(e4m3_encode_rne(np.array([-mid]))[0]) == (even | 0x80)
        # just off the midpoint: the nearer neighbour
        below = np.nextafter(mid, np.float32(0))
        above = np.nextafter(mid, np.float32(1000))
        assert int(e4m3_encode_rne(np.array([below]))[0]) == c
        assert int(e4m3_encode_rne(np.array([above]))[0]) == c + 1


def test_encoder_saturates_and_maps_nan():
    vals = np.array([448.0, 460.0, 464.0, 1e6, np.inf], dtype=np.float32)
    assert list(e4m3_encode_rne(vals)) == [0x7E] * 5
    assert list(e4m3_encode_rne(-vals)) == [0xFE] * 5
    assert int(e4m3_encode_rne(np.array([np.nan], dtype=np.float32))[0]) == 0x7F
    assert int(e4m3_encode_rne(np.array([-0.0], dtype=np.float32))[0]) == 0x80
    # below half the smallest subnormal: zero; exactly half: ties to even (0)
    assert list(e4m3_encode_rne(np.array([2.0**-11, 2.0**-10], dtype=np.float32))) == [0, 0]
    assert int(e4m3_encode_rne(np.array([2.0**-10 * 1.01], dtype=np.float32))[0]) == 1


def test_encoder_matches_torch_cast_in_range():
    rng = np.random.default_rng(11)
    x = np.concatenate(
        [rng.normal(0, 1, 4000), rng.normal(0, 100, 2000), rng.uniform(-448, 448, 2000), rng.normal(0, 1e-3, 2000)]
    ).astype(np.float32)
    ours = e4m3_encode_rne(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "quantize_q_example.json")))
    sh = g["shape"]
    q = np.array(g["q"], dtype=np.float32).reshape(sh["num_seqs"] * sh["q_len"], sh["h_k"] * sh["h_r"], sh["d"])
    codes, descale = quantize_pack_q_ref(q, sh["num_seqs"], sh["q_len"], sh["h_k"], sh["h_r"])
    assert descale.dtype == np.float32
    assert hex(descale.view(np.uint32)[0, 0]) == g["descale_fp32_hex"]
    assert [hex(c) for c in codes.reshape(-1)] == g["codes"]


@pytest.mark.parametrize("num_seqs,q_len,h_k,h_r,d", [(2, 1, 1, 16, 128), (3, 4, 2, 8, 16), (2, 5, 3, 2, 32)])
def test_quantise_layout_bound_and_group_maximum(num_seqs, q_len, h_k, h_r, d):
    rng = np.random.default_rng(num_seqs * 100 + q_len)
    q = rng.normal(0, 1, (num_seqs * q_len, h_k * h_r, d)).astype(np.float32)
    q[0, 0, 0] = 0.0
    q[:q_len, :h_r, :] = 0.0  # sequence 0, kv head 0: an all-zero group
    codes, descale = quantize_pack_q_ref(q, num_seqs, q_len, h_k, h_r)
    tab = _table()
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
