"""Seeded synthetic workloads for paged fp8-KV decode attention.

This module produces HOST arrays only (numpy) and holds none of the decode
method's arithmetic: it draws random numbers, rounds them into the storage
formats the cache and the queries use (e4m3 and bf16, round to nearest even,
e4m3 saturating at +-448), lays the cache out in pages and fills the block
table.  Both the CUDA path and the CPU oracle read the same bytes from it.

Input recipe (numpy PCG64 streams, seed fixed per config):

* sequence lengths from the config (uniform integers where it says so);
* a block table that hands each sequence ceil(L / PS) pages taken in order
  from a seeded permutation of the pool; entries past a sequence's last page
  are garbage (-1 / INT32_MAX alternating) and must never be read;
* K and V: x ~ N(0, 1) in float32, divided by the (seq, kv-head) descale and
  rounded to e4m3; pages no sequence owns, and the rows of a sequence's last
  page at or past L, hold the e4m3 NaN code 0x7F (poison: any stray read that
  reaches the output turns it into NaN);
* descales uniform in [0.5, 2) per (seq, kv head) where the config asks for
  them, else 1.0;
* Q ~ N(0, 1) rounded to bf16, or (fully-fp8 configs) divided by its
  (seq, kv-head) descale and rounded to e4m3; Q is in vLLM's layout
  (num_seqs * q_len, h_q, d).

The five named configs are the workloads the decode path is tested and
measured on: tiny reference, GQA decode, skewed varlen fully-fp8,
speculative verify (causal, and a non-causal block variant) and the
small-live-head sweep.
"""

from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

E4M3_NAN = 0x7F
HEAD_DIM = 128

# ------------------------------------------------------------ storage formats


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Round float values to e4m3 (E4M3FN) codes: nearest, ties to even,
    saturating at +-448; NaN maps to 0x7F.

    Works on the float32 bit pattern: in the normal range the 23-bit mantissa
    is rounded to 3 bits (drop 20 bits, ties to even) and the exponent is
    rebiased from 127 to 7; below 2^-6 the value is an integer multiple of the
    subnormal step 2^-9.  (int32 arithmetic: numpy's uint32 shifts are slow.)
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.int32)
    mag = bits & np.int32(0x7FFFFFFF)
    neg = bits < 0
    lsb = (mag // np.int32(1 << 20)) & np.int32(1)
    code = (mag + np.int32(0x7FFFF) + lsb) // np.int32(1 << 20) - np.int32((127 - 7) << 3)
    small = mag < np.int32(0x3C800000)  # |x| < 2^-6
    if small.any():
        scaled = np.where(small, mag, np.int32(0)).view(np.float32) * np.float32(512.0)
        sub = np.rint(scaled).astype(np.int32)
        code = np.where(small, sub, code)
    code = np.minimum(code, np.int32(0x7E)).astype(np.uint8)
    code |= np.where(neg, np.uint8(0x80), np.uint8(0))
    nan = mag > np.int32(0x7F800000)
    if nan.any():
        code[nan] = E4M3_NAN
    return code


# Narrow KV formats: (exponent bits, mantissa bits, bias); sign bit on top,
# a subnormal binade at exponent 0, no infinities or NaN.
NARROW_FORMATS = {"e3m2": (3, 2, 3), "e2m3": (2, 3, 1), "e2m1": (2, 1, 1)}
KV_FORMAT_CODE = {"e4m3": 0, "e3m2": 1, "e2m3": 2, "e2m1": 3, "nvfp4": 4}
KV_FORMAT_BITS = {"e4m3": 8, "e3m2": 6, "e2m3": 6, "e2m1": 4, "nvfp4": 4}
NVFP4_GROUP = 16  # elements of a row sharing one e4m3 scale


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """float32 values of e4m3 (E4M3FN) codes (0x7F / 0xFF -> NaN)."""
    c = np.asarray(codes, dtype=np.int32)
    e = (c >> 3) & 0xF
    m = (c & 7).astype(np.float32)
    mag = np.where(e == 0, m * np.float32(2.0**-9), (np.float32(1.0) + m / np.float32(8.0)) * np.exp2(e - 7).astype(np.float32))
    mag = np.where((c & 0x7F) == 0x7F, np.float32(np.nan), mag)
    return np.where(c & 0x80, -mag, mag).astype(np.float32)


def nvfp4_encode(v: np.ndarray):
    """nvfp4 storage of values v (..., d): per group of 16 elements an e4m3
    scale code = e4m3(8 * amax / 6) (so the group's largest magnitude lands on
    e2m1's largest, 6, after the 2^-3 the format folds into its scale), and
    e2m1 codes of v * 8 / scale (nearest, ties to the smaller magnitude).
    Returns (codes (..., d) uint8, scale codes (..., d / 16) uint8)."""
    v = np.asarray(v, dtype=np.float32)
    g = v.reshape(*v.shape[:-1], v.shape[-1] // NVFP4_GROUP, NVFP4_GROUP)
    amax = np.abs(g).max(axis=-1)
    sc = e4m3_encode(amax * np.float32(8.0 / 6.0))
    scv = e4m3_decode(sc)
    denom = np.where(scv > 0, scv, np.float32(1.0))[..., None]
    q = np.where(scv[..., None] > 0, g * np.float32(8.0) / denom, np.float32(0.0))
    codes = narrow_encode(q, "e2m1").reshape(v.shape)
    return codes, sc


def _narrow_magnitudes(fmt: str) -> np.ndarray:
    """The non-negative values of a narrow format, indexed by magnitude code
    (ascending)."""
    eb, mb, bias = NARROW_FORMATS[fmt]
    e = np.arange(1 << (eb + mb)) >> mb
    m = np.arange(1 << (eb + mb)) & ((1 << mb) - 1)
    frac = m.astype(np.float64) / (1 << mb)
    return np.where(e == 0, frac * 2.0 ** (1 - bias), (1.0 + frac) * 2.0 ** (e - bias))


def narrow_encode(x: np.ndarray, fmt: str) -> np.ndarray:
    """Round float values to a narrow format's codes: nearest value, a value
    half-way between two taking the smaller magnitude (the rounding of the
    narrow-format quantiser on the "mjolnir/t5_decode.py" page), saturating at
    the largest; the sign bit only on a non-zero magnitude."""
    mags = _narrow_magnitudes(fmt)
    eb, mb, _ = NARROW_FORMATS[fmt]
    mids = (mags[:-1] + mags[1:]) / 2.0
    a = np.abs(np.asarray(x, dtype=np.float64))
    mag = np.searchsorted(mids, a, side="left").astype(np.uint8)  # ties stay below the midpoint
    neg = (np.asarray(x) < 0) & (mag > 0)
    return mag | np.where(neg, np.uint8(1 << (eb + mb)), np.uint8(0))


def pack_codes(codes: np.ndarray, bits: int) -> np.ndarray:
    """Little-endian packing of the last axis (fp4: element 2i in the low
    nibble of byte i; fp6: each four elements in three bytes, element j of the
    group at bits 6j .. 6j + 5 of the little-endian 24-bit word)."""
    c = np.asarray(codes, dtype=np.uint32)
    d = c.shape[-1]
    if bits == 4:
        c = c.reshape(*c.shape[:-1], d // 2, 2)
        return (c[..., 0] | (c[..., 1] << 4)).astype(np.uint8)
    c = c.reshape(*c.shape[:-1], d // 4, 4)
    word = c[..., 0] | (c[..., 1] << 6) | (c[..., 2] << 12) | (c[..., 3] << 18)
    out = np.stack([word & 0xFF, (word >> 8) & 0xFF, (word >> 16) & 0xFF], axis=-1)
    return out.reshape(*c.shape[:-2], d // 4 * 3).astype(np.uint8)


def bf16_encode(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 bit patterns (nearest, ties to even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    bits = x.view(np.uint32).astype(np.int64)
    rounded = (bits + 0x7FFF + ((bits // 65536) & 1)) // 65536
    out = rounded.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out = np.where(nan, np.uint16(0x7FC0), out)
    return out


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------------ workload


@dataclass
class Workload:
    name: str
    num_seqs: int
    q_len: int
    h_k: int
    h_r: int
    page_size: int
    causal: bool
    q_is_e4m3: bool
    seq_lens: np.ndarray  # int32 (b,)
    block_table: np.ndarray  # int32 (b, max_blocks)
    k_cache: np.ndarray  # uint8 (num_pages, PS, h_k, d) e4m3 codes
    v_cache: np.ndarray
    q: np.ndarray  # uint16 bf16 bits or uint8 e4m3, (b * q_len, h_q, d)
    q_descale: np.ndarray  # float32 (b, h_k)
    k_descale: np.ndarray
    v_descale: np.ndarray
    softmax_scale: float
    scale_o: float = 1.0
    max_splits: int = 16
    head_dim: int = HEAD_DIM
    kv_format: str = "e4m3"  # e4m3, or a narrow format packed little-endian
    # nvfp4 only: e4m3 scale codes, (num_pages, h_k, PS, d / 16) (a page's
    # scales of one head together, 8 bytes a row)
    k_scales: Optional[np.ndarray] = None
    v_scales: Optional[np.ndarray] = None
    meta: Dict[str, object] = field(default_factory=dict)

    @property
    def n_q(self) -> int:
        return self.q_len * self.h_r

    @property
    def h_q(self) -> int:
        return self.h_k * self.h_r

    @property
    def num_pages(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    # Element strides in the forms the oracle and the library take.
    @property
    def q_strides(self) -> Tuple[int, int, int]:
        """(seq, token, head) strides of q in elements."""
        tok = self.q.strides[0] // self.q.itemsize
        return (self.q_len * tok, tok, self.q.strides[1] // self.q.itemsize)

    @staticmethod
    def _kv_strides(t: np.ndarray) -> Tuple[int, int, int]:
        return tuple(s // t.itemsize for s in t.strides[:3])  # type: ignore[return-value]

    @property
    def k_strides(self) -> Tuple[int, int, int]:
        return self._kv_strides(self.k_cache)

    @property
    def v_strides(self) -> Tuple[int, int, int]:
        return self._kv_strides(self.v_cache)

    @staticmethod
    def _descale_strides(t: np.ndarray) -> Tuple[int, int]:
        if t.size == 1:
            return (0, 0)
        if t.ndim == 1:
            return (0, t.strides[0] // t.itemsize)
        return (t.strides[0] // t.itemsize, t.strides[1] // t.itemsize)

    @property
    def qd_strides(self):
        return self._descale_strides(self.q_descale)

    @property
    def kd_strides(self):
        return self._descale_strides(self.k_descale)

    @property
    def vd_strides(self):
        return self._descale_strides(self.v_descale)

    def kv_bytes(self) -> int:
        """K + V bytes of the rows the attention reads (rows < L), nvfp4's
        scales included."""
        row = self.head_dim * KV_FORMAT_BITS[self.kv_format] // 8
        if self.kv_format == "nvfp4":
            row += self.head_dim // NVFP4_GROUP
        return int(self.seq_lens.astype(np.int64).sum()) * self.h_k * row * 2


def _fill_kv(
    seed: int,
    tag: int,
    cache: np.ndarray,
    block_table: np.ndarray,
    seq_lens: np.ndarray,
    descale: np.ndarray,
    kv_format: str = "e4m3",
    scales: Optional[np.ndarray] = None,
) -> None:
    """Quantised N(0,1)/descale rows for every (seq, page, row < L); the rest
    of the pool keeps the poison code it was created with.  Sequence b draws
    from its own stream, SeedSequence([seed, tag, b]), so sequences can be
    filled in parallel threads with a result that does not depend on the
    thread count.  Narrow formats are packed (d * bits / 8 bytes a row)."""
    PS, h_k = cache.shape[1], cache.shape[2]
    d = HEAD_DIM

    def one(b: int) -> None:
        L = int(seq_lens[b])
        n_pages = -(-L // PS)
        if n_pages == 0:
            return
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, b])))
        pages = block_table[b, :n_pages]
        x = rng.standard_normal((n_pages * PS, h_k, d), dtype=np.float32)
        x /= descale[b].astype(np.float32)[None, :, None]
        if kv_format == "e4m3":
            codes = e4m3_encode(x)
        elif kv_format == "nvfp4":
            c4, sc = nvfp4_encode(x)
            codes = pack_codes(c4, 4)
            sc[L:] = E4M3_NAN  # rows past the sequence end: a NaN scale
            # the scale plane is (page, head, row, group)
            scales[pages] = sc.reshape(n_pages, PS, h_k, -1).transpose(0, 2, 1, 3)
        else:
            codes = pack_codes(narrow_encode(x, kv_format), KV_FORMAT_BITS[kv_format])
        codes[L:] = E4M3_NAN  # rows past the sequence end (poison bytes)
        cache[pages] = codes.reshape(n_pages, PS, h_k, cache.shape[3])

    workers = min(len(seq_lens), os.cpu_count() or 1)
    if workers <= 1:
        for b in range(len(seq_lens)):
            one(b)
    else:
        with ThreadPoolExecutor(max_workers=workers) as ex:
            list(ex.map(one, range(len(seq_lens))))


def make_workload(
    name: str,
    seq_lens: Sequence[int],
    q_len: int,
    h_k: int,
    h_r: int,
    page_size: int,
    *,
    seed: int,
    causal: bool = True,
    q_is_e4m3: bool = False,
    random_descales: bool = True,
    max_splits: int = 16,
    spare_pages: Optional[int] = None,
    num_pages: Optional[int] = None,
    scale_o: float = 1.0,
    softmax_scale: Optional[float] = None,
    kv_format: str = "e4m3",
) -> Workload:
    rng = np.random.Generator(np.random.PCG64(seed))
    b = len(seq_lens)
    seq = np.asarray(seq_lens, dtype=np.int32)
    d = HEAD_DIM
    pages_per_seq = [-(-int(L) // page_size) for L in seq]
    used = sum(pages_per_seq)
    if num_pages is None:
        spare = max(4, used // 4) if spare_pages is None else spare_pages
        num_pages = used + spare
    assert num_pages >= used
    perm = rng.permutation(num_pages).astype(np.int32)
    max_blocks = max(pages_per_seq + [0]) + 1  # one garbage column at least
    bt = np.empty((b, max_blocks), dtype=np.int32)
    garbage = np.where(np.arange(max_blocks) % 2 == 0, np.int32(-1), np.int32(2**31 - 1))
    cursor = 0
    for i, n in enumerate(pages_per_seq):
        bt[i] = garbage
        bt[i, :n] = perm[cursor : cursor + n]
        cursor += n

    def descales() -> np.ndarray:
        if random_descales:
            return rng.uniform(0.5, 2.0, size=(b, h_k)).astype(np.float32)
        return np.ones((b, h_k), dtype=np.float32)

    k_desc = descales()
    v_desc = descales()
    q_desc = descales() if q_is_e4m3 else np.ones((b, h_k), dtype=np.float32)
    row_bytes = d * KV_FORMAT_BITS[kv_format] // 8
    k_cache = np.full((num_pages, page_size, h_k, row_bytes), E4M3_NAN, dtype=np.uint8)
    v_cache = np.full((num_pages, page_size, h_k, row_bytes), E4M3_NAN, dtype=np.uint8)
    k_scales = v_scales = None
    if kv_format == "nvfp4":
        k_scales = np.full((num_pages, h_k, page_size, d // NVFP4_GROUP), E4M3_NAN, dtype=np.uint8)
        v_scales = np.full((num_pages, h_k, page_size, d // NVFP4_GROUP), E4M3_NAN, dtype=np.uint8)
    _fill_kv(seed, 1, k_cache, bt, seq, k_desc, kv_format, k_scales)
    _fill_kv(seed, 2, v_cache, bt, seq, v_desc, kv_format, v_scales)
    h_q = h_k * h_r
    qx = rng.standard_normal((b * q_len, h_q, d), dtype=np.float32)
    if q_is_e4m3:
        # query head h belongs to kv head h // h_r
        div = np.repeat(q_desc, q_len, axis=0)  # (b * q_len, h_k)
        div = np.repeat(div, h_r, axis=1)  # (b * q_len, h_q)
        q = e4m3_encode(qx / div[:, :, None])
    else:
        q = bf16_encode(qx)
    return Workload(
        name=name,
        num_seqs=b,
        q_len=q_len,
        h_k=h_k,
        h_r=h_r,
        page_size=page_size,
        causal=causal,
        q_is_e4m3=q_is_e4m3,
        seq_lens=seq,
        block_table=bt,
        k_cache=k_cache,
        v_cache=v_cache,
        q=q,
        q_descale=q_desc,
        k_descale=k_desc,
        v_descale=v_desc,
        softmax_scale=1.0 / math.sqrt(d) if softmax_scale is None else softmax_scale,
        scale_o=scale_o,
        max_splits=max_splits,
        kv_format=kv_format,
        k_scales=k_scales,
        v_scales=v_scales,
        meta={"seed": seed},
    )


# --------------------------------------------------------------- the configs

CONFIG_NAMES = {
    1: "tiny_ref",
    2: "gqa_decode",
    3: "skewed_fp8",
    4: "spec_verify",
    5: "swapab_sweep",
}

SWEEP_POINTS: List[Tuple[int, int]] = [(h_r, ql) for h_r in (16, 32) for ql in (1, 2, 4, 8, 16)]


def config(
    idx: int,
    *,
    variant: Optional[str] = None,
    num_seqs: Optional[int] = None,
    len_range: Optional[Tuple[int, int]] = None,
    h_r: Optional[int] = None,
    q_len: Optional[int] = None,
    max_splits: Optional[int] = None,
    seed: Optional[int] = None,
    kv_format: str = "e4m3",
) -> Workload:
    """Workload of a named config (1..5).  Keyword overrides shrink it for
    parity tests (fewer sequences, shorter lengths) while keeping its
    structure; ``variant="noncausal"`` gives config 4's q_len = 5 block
    attention variant."""
    def mk(name, *args, **kw):
        suffix = "" if kv_format == "e4m3" else "_kv" + kv_format
        return make_workload(name + suffix, *args, kv_format=kv_format, **kw)

    seed = 1111 + idx if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    if idx == 1:
        return mk(
            CONFIG_NAMES[1],
            [37, 100] if len_range is None else list(rng.integers(len_range[0], len_range[1] + 1, num_seqs or 2)),
            1,
            1,
            8,
            16,
            seed=seed,
            random_descales=False,
            max_splits=1 if max_splits is None else max_splits,
            num_pages=16 if len_range is None else None,
        )
    if idx == 2:
        b = 64 if num_seqs is None else num_seqs
        lo, hi = (512, 8192) if len_range is None else len_range
        lens = rng.integers(lo, hi + 1, size=b)
        return mk(CONFIG_NAMES[2], lens, 1, 8, 4, 16, seed=seed, max_splits=max_splits or 16)
    if idx == 3:
        b = 8 if num_seqs is None else num_seqs
        long_len, short = (131072, 1024) if len_range is None else len_range
        lens = [long_len] + list(short + rng.integers(-64, 65, size=b - 1))
        return mk(
            CONFIG_NAMES[3], lens, 1, 1, 16, 128, seed=seed, q_is_e4m3=True, max_splits=max_splits or 256
        )
    if idx == 4:
        b = 32 if num_seqs is None else num_seqs
        lo, hi = (2048, 32768) if len_range is None else len_range
        lens = rng.integers(lo, hi + 1, size=b)
        noncausal = variant == "noncausal"
        ql = (5 if noncausal else 4) if q_len is None else q_len
        return mk(
            CONFIG_NAMES[4] + ("_noncausal" if noncausal else ""),
            lens,
            ql,
            8,
            8,
            64,
            seed=seed,
            causal=not noncausal,
            max_splits=max_splits or 16,
        )
    if idx == 5:
        b = 128 if num_seqs is None else num_seqs
        L = 16384 if len_range is None else len_range[1]
        hr = 16 if h_r is None else h_r
        ql = 1 if q_len is None else q_len
        return mk(
            f"{CONFIG_NAMES[5]}_hr{hr}_q{ql}",
            [L] * b,
            ql,
            1,
            hr,
            128,
            seed=seed,
            max_splits=max_splits or 16,
        )
    raise ValueError(f"unknown config {idx}")
