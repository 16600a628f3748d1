"""Narrow KV formats on the GPU (fp6 e3m2 / e2m3 and fp4 e2m1 pools read by
the tensor-core kernels' kind::f8f6f4 MMAs as they are).

* The page gather: the TMA boxes the decode kernels issue for a packed pool
  land each 16-code group in 16 bytes of shared memory; the hook's rows are
  compared byte for byte with the packed bytes of the group (the oracle's
  little-endian packing of the generator's codes), the group's padding
  ignored.
* Attention: against the fp64 oracle on the workload's e4m3 view (every
  narrow value is an e4m3 value), element by element on small cases of the
  configurations (swap-AB and query-rows kernels, bf16 and e4m3 Q, split and
  merged sequences) and on sampled units at full size.
"""

import numpy as np
import pytest
import torch

import oracle
import paged_fp8_kv_gb300 as mj
from oracle import narrow_ref
from paged_fp8_kv_gb300 import synthetic as syn
from paged_fp8_kv_gb300.session import DecodeSession
from tests.gpu_helpers import compare, sample_units

pytestmark = pytest.mark.gpu

FORMATS = ["e3m2", "e2m3", "e2m1"]


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_fp8_kv_gb300.build import build

    build()


def run(w, **kw):
    s = DecodeSession(w, **kw)
    s.fill_workspace(float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s.step(status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return s


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("page_size", [16, 128])
def test_gather_lands_each_group_in_16_bytes(fmt, page_size):
    w = syn.make_workload("narrow_gather", [1, 17, 130, 300], 1, 2, 4, page_size, seed=61, kv_format=fmt)
    s = DecodeSession(w)
    bits = narrow_ref.BITS[fmt]
    gbytes = 16 * bits // 8  # packed bytes of a 16-code group
    rows = int(w.seq_lens.max())
    for values, cache in ((False, w.k_cache), (True, w.v_cache)):
        out = torch.zeros((w.num_seqs, w.h_k, rows, 128), dtype=torch.uint8, device="cuda")
        mj.check_gather_kv(s.params, s.k_cache, s.v_cache, s.block_table, s.seq_lens, values, out)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        for b in range(w.num_seqs):
            L = int(w.seq_lens[b])
            j = np.arange(L)
            packed = cache[w.block_table[b, j // page_size], j % page_size]  # (L, h_k, packed bytes)
            for g in range(w.h_k):
                want = packed[:, g].reshape(L, 8, gbytes)
                have = got[b, g, :L].reshape(L, 8, 16)[:, :, :gbytes]
                assert np.array_equal(have, want), f"{fmt} values={values} b={b} g={g}"


SMALL = [
    ("gqa_swapab", lambda f: syn.config(2, num_seqs=5, len_range=(300, 2500), kv_format=f)),
    ("fp8q_split", lambda f: syn.config(3, num_seqs=3, len_range=(6000, 500), kv_format=f)),
    ("spec_qrows", lambda f: syn.config(4, num_seqs=3, len_range=(500, 1800), kv_format=f)),
    ("sweep_qrows128", lambda f: syn.config(5, h_r=32, q_len=4, num_seqs=2, len_range=(0, 1500), kv_format=f)),
]


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("name,make", SMALL, ids=[c[0] for c in SMALL])
def test_attention_small(name, make, fmt):
    w = make(fmt)
    s = run(w)
    assert s.kernel.endswith("_kv" + fmt), s.kernel
    compare(w, s.o_host(), s.lse_host())


@pytest.mark.parametrize("fmt", ["e2m3", "e2m1"])
def test_forced_splits_and_kernels(fmt):
    # the swap-AB kernel at 32 rows and the query-rows kernel at 16, with
    # every sequence cut and merged
    w = syn.config(4, num_seqs=3, len_range=(700, 2600), kv_format=fmt)
    for kernel in (mj.MJ_KERNEL_TENSOR_CORE, mj.MJ_KERNEL_TENSOR_CORE_QROWS):
        s = run(w, kernel=kernel, force_splits=3)
        assert s.plan.max_n_splits == 3
        compare(w, s.o_host(), s.lse_host())


def test_narrow_refused_by_other_kernels():
    w = syn.config(2, num_seqs=2, len_range=(100, 200), kv_format="e2m1")
    for kernel in (mj.MJ_KERNEL_CUDA_CORE, mj.MJ_KERNEL_TENSOR_CORE_GROUPED):
        with pytest.raises(mj.MjError):
            DecodeSession(w, kernel=kernel)


@pytest.mark.parametrize("cfg,opts,fmt", [(2, {}, "e2m1"), (4, {}, "e3m2"), (3, {}, "e2m3")], ids=["gqa_e2m1", "spec_e3m2", "skewed_e2m3"])
def test_full_size_sampled(cfg, opts, fmt):
    w = syn.config(cfg, kv_format=fmt, **opts)
    s = run(w)
    longest = int(np.argmax(w.seq_lens))
    units = sample_units(w, 6, seed=cfg, include=[(longest, w.h_k - 1), (w.num_seqs - 1, 0)])
    compare(w, s.o_host(), s.lse_host(), units=units)


# --------------------------------------------------------------------- nvfp4


@pytest.mark.parametrize("page_size", [16, 64, 128])
def test_nvfp4_conversion_is_bit_exact(page_size):
    # the kernel's conversion of each 16-code group and its scale, through the
    # block table and the scale plane, against the oracle's definition
    w = syn.make_workload("nv_gather", [1, 17, 130, 300], 1, 2, 4, page_size, seed=62, q_is_e4m3=True,
                          kv_format="nvfp4")
    s = DecodeSession(w)
    rows = int(w.seq_lens.max())
    for values, cache, scales in ((False, w.k_cache, w.k_scales), (True, w.v_cache, w.v_scales)):
        out = torch.zeros((w.num_seqs, w.h_k, rows, 128), dtype=torch.uint8, device="cuda")
        mj.check_gather_kv(s.params, s.k_cache, s.v_cache, s.block_table, s.seq_lens, values, out,
                           k_scales=s.k_scales, v_scales=s.v_scales)
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        for b in range(w.num_seqs):
            L = int(w.seq_lens[b])
            j = np.arange(L)
            pg, rw = w.block_table[b, j // page_size], j % page_size
            for g in range(w.h_k):
                codes = narrow_ref.unpack_bits(cache[pg, rw, g], 4, 128)
                want = narrow_ref.nvfp4_to_e4m3_codes(codes, scales[pg, g, rw])
                assert np.array_equal(got[b, g, :L], want), f"values={values} b={b} g={g}"


NV_SMALL = [
    ("skewed_split", lambda: syn.config(3, num_seqs=3, len_range=(6000, 500), kv_format="nvfp4")),
    ("gqa_rows8", lambda: syn.make_workload("nv_gqa", [1, 300, 1000, 2500, 129], 1, 8, 4, 16, seed=63,
                                            q_is_e4m3=True, kv_format="nvfp4")),
    ("spec_rows32", lambda: syn.make_workload("nv_spec", [500, 1800, 3], 4, 8, 8, 64, seed=64, q_is_e4m3=True,
                                              kv_format="nvfp4")),
]


@pytest.mark.parametrize("name,make", NV_SMALL, ids=[c[0] for c in NV_SMALL])
def test_nvfp4_attention_small(name, make):
    w = make()
    s = run(w)
    assert s.kernel.startswith("tc_") and s.kernel.endswith("_kvnvfp4"), s.kernel
    compare(w, s.o_host(), s.lse_host())
    s2 = run(w, force_splits=3)
    compare(w, s2.o_host(), s2.lse_host())


def test_nvfp4_full_size_sampled():
    w = syn.config(3, kv_format="nvfp4")
    s = run(w)
    assert s.plan.n_splits[0] > 1
    compare(w, s.o_host(), s.lse_host(), units=[(0, 0), (3, 0), (7, 0)])
