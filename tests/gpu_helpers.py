"""Shared helpers of the GPU parity tests: run a workload through the C ABI
and compare it with the fp64 oracle element by element."""

from __future__ import annotations

import numpy as np

import oracle

# Parity tolerances, |o - ref| <= atol + rtol |ref| and |lse - ref| <= LSE_TOL:
# bf16 Q (hi + lo e4m3 parts) and the fully-fp8 path (e4m3 Q and P).
O_TOL_BF16 = (2e-2, 2e-2)
O_TOL_FP8 = (5e-2, 5e-2)
LSE_TOL = 2e-3


def o_tol(w):
    return O_TOL_FP8 if w.q_is_e4m3 else O_TOL_BF16


def compare(w, o_gpu, lse_gpu, units=None, threads=0):
    """o_gpu (b, h_k, n_q, d) float, lse_gpu (b, h_k, n_q) float: assert
    |o - ref| <= atol + rtol |ref| and |lse - ref| <= 2e-3 on the given (b, g)
    units (all when None).  Returns the worst errors for reporting.  A
    narrow-KV workload is compared through its e4m3 view."""
    if getattr(w, "kv_format", "e4m3") != "e4m3":
        w = e4m3_view(w, None if units is None else sorted({b for b, _ in units}))
    if units is None:
        ref_o, ref_lse = oracle.attention(w, threads=threads)
        got_o, got_lse = o_gpu, lse_gpu
    else:
        ref_o, ref_lse = oracle.attention(w, units=units, threads=threads)
        got_o = np.stack([o_gpu[b, g] for b, g in units])
        got_lse = np.stack([lse_gpu[b, g] for b, g in units])
    atol, rtol = o_tol(w)
    assert not np.isnan(got_o).any(), "NaN in O (stray read of a poisoned row?)"
    err_o = np.abs(got_o - ref_o)
    bound = atol + rtol * np.abs(ref_o)
    bad = err_o > bound
    assert not bad.any(), f"O mismatch at {np.argwhere(bad)[:5].tolist()}: max err {err_o.max():.3g}"
    both_inf = np.isneginf(ref_lse) & np.isneginf(got_lse)
    with np.errstate(invalid="ignore"):
        err_l = np.where(both_inf, 0.0, np.abs(got_lse - ref_lse))
    assert not np.isnan(err_l).any(), "NaN LSE"
    assert err_l.max() <= LSE_TOL, f"LSE mismatch: max err {err_l.max():.3g}"
    return float(err_o.max()), float(err_l.max())


def sample_units(w, n, seed=0, include=()):
    rng = np.random.default_rng(seed)
    units = set(tuple(u) for u in include)
    while len(units) < min(n, w.num_seqs * w.h_k):
        units.add((int(rng.integers(w.num_seqs)), int(rng.integers(w.h_k))))
    return sorted(units)


def e4m3_view(w, seqs=None):
    """A narrow-KV workload as the same attention problem over e4m3 pools:
    every narrow value is an e4m3 value, so the oracle's unpacking and its
    exact code map (oracle.narrow_ref) turn the packed rows into e4m3 rows of
    equal value.  Only the pages of `seqs` (all when None) are converted; the
    rest of the view stays zero (the oracle never reads them)."""
    import copy

    from oracle import narrow_ref

    if w.kv_format == "e4m3":
        return w
    e4 = oracle.e4m3_table()
    v = copy.copy(w)
    v.kv_format = "e4m3"
    for name, sname in (("k_cache", "k_scales"), ("v_cache", "v_scales")):
        src = getattr(w, name)
        dst = np.zeros(src.shape[:3] + (w.head_dim,), dtype=np.uint8)
        bs = range(w.num_seqs) if seqs is None else seqs
        pages = sorted({int(p) for b in bs for p in w.block_table[b, : -(-int(w.seq_lens[b]) // w.page_size)]})
        if pages and w.kv_format == "nvfp4":
            codes = narrow_ref.unpack_bits(src[pages], 4, w.head_dim)
            scales = getattr(w, sname)[pages].transpose(0, 2, 1, 3)  # (page, row, head, group)
            dst[pages] = narrow_ref.nvfp4_to_e4m3_codes(codes, scales)
        elif pages:
            codes = narrow_ref.unpack_bits(src[pages], narrow_ref.BITS[w.kv_format], w.head_dim)
            dst[pages] = narrow_ref.to_e4m3_codes(codes, w.kv_format, e4)
        setattr(v, name, dst)
    return v
