"""Pins of the oracle's query / output row permutation (oracle/layout_ref.py),
CPU only.

Source: the "mjolnir/t5_decode.py" page, `pack_q` / `unpack_o` and the
module docstring: packed row n = qi * h_r + hr of kv head g holds query
token qi of query head g * h_r + hr.  What fixes the functions,
independently of their reshapes:
* an element-by-element loop over that placement rule, with distinct
  values in every cell (so a swapped axis or a wrong factor moves a value);
* unpack(pack(x)) == x and pack(unpack(y)) == y on shapes whose axes all
  differ in length;
* q_len == 1: packing is the identity on the memory (vLLM's (b, h_q, d)
  rows are already packed).

Each pin is a function of the module under test, so that
tests/test_oracle_mutations.py can run the same pins against copies of the
module with planted mistakes.
"""

import numpy as np
import pytest

import oracle.layout_ref as layout_ref

# (num_seqs, q_len, h_k, h_r, d): every axis of a different length
SHAPES = [(2, 3, 5, 4, 7), (3, 4, 2, 5, 6), (1, 2, 3, 1, 4), (4, 1, 3, 2, 5)]


def distinct(shape, seed):
    rng = np.random.default_rng(seed)
    return rng.permutation(int(np.prod(shape))).reshape(shape).astype(np.int64)


def pin_unpack_placement(m, num_seqs, q_len, h_k, h_r, d):
    packed = distinct((num_seqs, h_k, q_len * h_r, d), 1)
    o = m.unpack_o_ref(packed, num_seqs, q_len, h_k, h_r)
    assert o.shape == (num_seqs * q_len, h_k * h_r, d)
    for b in range(num_seqs):
        for qi in range(q_len):
            for g in range(h_k):
                for hr in range(h_r):
                    assert np.array_equal(o[b * q_len + qi, g * h_r + hr], packed[b, g, qi * h_r + hr])


def pin_pack_placement(m, num_seqs, q_len, h_k, h_r, d):
    q = distinct((num_seqs * q_len, h_k * h_r, d), 2)
    p = m.pack_q_ref(q, num_seqs, q_len, h_k, h_r)
    assert p.shape == (num_seqs, h_k, q_len * h_r, d)
    for b in range(num_seqs):
        for g in range(h_k):
            for n in range(q_len * h_r):
                qi, hr = divmod(n, h_r)
                assert np.array_equal(p[b, g, n], q[b * q_len + qi, g * h_r + hr])


def pin_round_trips(m, num_seqs, q_len, h_k, h_r, d):
    q = distinct((num_seqs * q_len, h_k * h_r, d), 3)
    assert np.array_equal(m.unpack_o_ref(m.pack_q_ref(q, num_seqs, q_len, h_k, h_r), num_seqs, q_len, h_k, h_r), q)
    y = distinct((num_seqs, h_k, q_len * h_r, d), 4)
    assert np.array_equal(m.pack_q_ref(m.unpack_o_ref(y, num_seqs, q_len, h_k, h_r), num_seqs, q_len, h_k, h_r), y)


def pin_single_token_is_identity(m):
    q = distinct((3, 4 * 2, 5), 5)  # num_seqs 3, q_len 1, h_k 4, h_r 2
    assert np.array_equal(m.pack_q_ref(q, 3, 1, 4, 2).reshape(-1), q.reshape(-1))
    assert np.array_equal(m.unpack_o_ref(q.reshape(3, 4, 2, 5), 3, 1, 4, 2).reshape(-1), q.reshape(-1))


def all_pins(m):
    """Every pin against module m (raises on the first that fails)."""
    for sh in SHAPES:
        pin_unpack_placement(m, *sh)
        pin_pack_placement(m, *sh)
        pin_round_trips(m, *sh)
    pin_single_token_is_identity(m)


@pytest.mark.parametrize("shape", SHAPES)
def test_unpack_places_every_element(shape):
    pin_unpack_placement(layout_ref, *shape)


@pytest.mark.parametrize("shape", SHAPES)
def test_pack_places_every_element(shape):
    pin_pack_placement(layout_ref, *shape)


@pytest.mark.parametrize("shape", SHAPES)
def test_round_trips(shape):
    pin_round_trips(layout_ref, *shape)


def test_single_token_is_identity():
    pin_single_token_is_identity(layout_ref)
