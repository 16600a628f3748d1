"""The seeded input generator: storage-format rounding and cache structure."""

import numpy as np
import pytest
import torch

from paged_fp8_kv_gb300 import synthetic as syn


def test_e4m3_encoder_matches_torch_in_range():
    x = np.random.default_rng(0).standard_normal(2_000_000).astype(np.float32)
    x = np.concatenate([x * 40, x * 0.003, np.float32(2.0) ** np.arange(-12, 9, dtype=np.float32)])
    x = x[np.abs(x) < 448]
    ours = syn.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(ours, ref)


def test_e4m3_encoder_saturates_and_keeps_nan():
    x = np.array([448, 460, 464, 500, 1e30, np.inf, -np.inf, -1000, np.nan], dtype=np.float32)
    codes = syn.e4m3_encode(x)
    assert codes.tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F]


def test_e4m3_encoder_ties_to_even():
    # 1 + 1/16 lies halfway between 1 (mantissa 000) and 1.125 (001): even -> 1
    # 1 + 3/16 lies halfway between 1.125 (001) and 1.25 (010): even -> 1.25
    # 2^-10 lies halfway between 0 and 2^-9: even -> 0
    x = np.array([1.0625, 1.1875, 2.0**-10, 3 * 2.0**-10], dtype=np.float32)
    assert syn.e4m3_encode(x).tolist() == [0x38, 0x3A, 0x00, 0x02]


def test_bf16_encoder_matches_torch():
    x = np.random.default_rng(1).standard_normal(1_000_000).astype(np.float32) * 10
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(syn.bf16_encode(x), ref)


def test_workload_structure_and_poison():
    w = syn.config(1)
    assert w.num_pages == 16 and w.seq_lens.tolist() == [37, 100]
    owned = set()
    for b, L in enumerate(w.seq_lens):
        n = -(-int(L) // w.page_size)
        pages = w.block_table[b, :n].tolist()
        assert len(set(pages)) == n and all(0 <= p < w.num_pages for p in pages)
        owned |= set(pages)
        # garbage past the last page
        assert all(v in (-1, 2**31 - 1) for v in w.block_table[b, n:].tolist())
        # rows past L in the last page are poisoned
        last = pages[-1]
        tail = int(L) - (n - 1) * w.page_size
        assert np.all(w.k_cache[last, tail:] == syn.E4M3_NAN)
    assert len(owned) == 10
    for p in range(w.num_pages):
        if p not in owned:
            assert np.all(w.k_cache[p] == syn.E4M3_NAN) and np.all(w.v_cache[p] == syn.E4M3_NAN)


def test_generation_is_deterministic():
    a = syn.config(2, num_seqs=3, len_range=(100, 400))
    b = syn.config(2, num_seqs=3, len_range=(100, 400))
    for f in ("k_cache", "v_cache", "q", "block_table", "seq_lens", "k_descale"):
        np.testing.assert_array_equal(getattr(a, f), getattr(b, f))


@pytest.mark.parametrize("fmt", ["e3m2", "e2m3", "e2m1"])
def test_narrow_generator_agrees_with_the_oracle_encoder(fmt):
    # two independent implementations of the same rounding (the generator's
    # midpoint search and the oracle's exhaustive nearest search, ties to the
    # smaller magnitude) and of the same little-endian packing
    from oracle import narrow_ref

    rng = np.random.default_rng(11)
    x = np.concatenate([rng.normal(0, 3, 5000), narrow_ref.minifloat_table(fmt), [1e6, -1e6, 0.0, -0.0]])
    assert np.array_equal(syn.narrow_encode(x, fmt), narrow_ref.minifloat_encode(x, fmt))
    bits = syn.KV_FORMAT_BITS[fmt]
    codes = rng.integers(0, 1 << bits, size=(3, 4, 128)).astype(np.uint8)
    assert np.array_equal(syn.pack_codes(codes, bits), narrow_ref.pack_bits(codes, bits))


def test_narrow_workload_layout():
    w = syn.config(2, num_seqs=3, len_range=(100, 400), kv_format="e2m1")
    assert w.name.endswith("_kve2m1") and w.kv_format == "e2m1"
    assert w.k_cache.shape[-1] == 64 and w.v_cache.shape[-1] == 64
    assert w.kv_bytes() == int(w.seq_lens.sum()) * w.h_k * 64 * 2
