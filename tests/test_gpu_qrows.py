"""GPU parity of the query-rows tensor-core kernel
(MJ_KERNEL_TENSOR_CORE_QROWS; the automatic choice for more than 32 packed
rows): 128 packed query rows of one kv head on the MMA's M, 128 keys of a
tile on N, one softmax thread per query row.

Against the fp64 oracle element by element: every sweep shape of the small-
live-head workload (packed rows 16 to 512, so one to four q tiles and a
partly filled last tile), bf16 and e4m3 Q, causal and non-causal, every page
size, empty and ragged lengths, forced splits with the merge, every KV
layout, descale broadcasts, and the full-size sweep extremes on sampled
units; plus determinism and graph replay.
"""

import copy

import numpy as np
import pytest
import torch

from paged_fp8_kv_gb300 import synthetic as syn
from paged_fp8_kv_gb300.session import DecodeSession
from tests.gpu_helpers import compare, sample_units

pytestmark = pytest.mark.gpu

QROWS = 4  # MJ_KERNEL_TENSOR_CORE_QROWS


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_fp8_kv_gb300.build import build

    build()


def run(w, nan_workspace=True, kernel=QROWS, **kw):
    s = DecodeSession(w, kernel=kernel, **kw)
    assert s.kernel.startswith("qm_"), s.kernel
    if nan_workspace:
        s.fill_workspace(float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    s.step(status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return s


def check(w, units=None, **kw):
    s = run(w, **kw)
    return s, compare(w, s.o_host(), s.lse_host(), units=units)


@pytest.mark.parametrize("h_r,q_len", syn.SWEEP_POINTS)
def test_sweep_small(h_r, q_len):
    w = syn.config(5, h_r=h_r, q_len=q_len, num_seqs=3, len_range=(0, 700))
    check(w)


@pytest.mark.parametrize("h_r,q_len", [(16, 4), (32, 4), (32, 16)])
def test_sweep_full_sampled(h_r, q_len):
    w = syn.config(5, h_r=h_r, q_len=q_len)
    s = run(w, kernel=0)  # the automatic choice
    compare(w, s.o_host(), s.lse_host(), units=[(0, 0), (77, 0), (127, 0)])


def test_spec_verify_noncausal_small():
    w = syn.config(4, variant="noncausal", num_seqs=5, len_range=(200, 1300))
    s, _ = check(w)  # 40 packed rows in one q tile
    assert s.plan.opts.n_q_tiles == 1


@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
@pytest.mark.parametrize("q_is_e4m3", [False, True])
def test_page_sizes_and_q_dtype(page_size, q_is_e4m3):
    lens = [1, 100, 127, 128, 129, 300, 1000]
    w = syn.make_workload("qrows", lens, 3, 2, 24, page_size, seed=91 + page_size, q_is_e4m3=q_is_e4m3,
                          max_splits=4)
    check(w, force_splits=2)


@pytest.mark.parametrize("q_len,h_r", [(3, 48), (16, 16), (5, 64)], ids=["rows144", "rows256", "rows320"])
@pytest.mark.parametrize("page_size", [16, 128])
@pytest.mark.parametrize("q_is_e4m3", [False, True])
def test_paired_q_tiles(q_len, h_r, page_size, q_is_e4m3):
    """More than 128 packed rows: two q tiles per CTA, each KV tile taken by
    both softmax groups.  144 rows leave the second group's tile mostly
    empty; 320 rows make a second CTA whose second group has no live row."""
    lens = [1, 100, 127, 128, 129, 300, 1000, 2500]
    causal = q_len != 5
    w = syn.make_workload("pair", lens, q_len, 2, h_r, page_size, seed=71 + q_len * h_r + page_size,
                          q_is_e4m3=q_is_e4m3, causal=causal, max_splits=4)
    s, _ = check(w, force_splits=2)
    assert s.kernel == ("qm_pair_e4m3" if q_is_e4m3 else "qm_pair_bf16")
    assert s.plan.opts.n_q_tiles == (q_len * h_r + 255) // 256
    check(w)  # unsplit


@pytest.mark.parametrize("q_len,causal", [(1, True), (4, True), (3, False)])
def test_empty_short_and_aligned_lengths(q_len, causal):
    lens = [0, 1, 2, 3, 16, 127, 128, 129, 256, 300]
    w = syn.make_workload("edge", lens, q_len, 2, 48, 16, seed=52, causal=causal, max_splits=4)
    s, _ = check(w, force_splits=2)
    assert np.all(np.isneginf(s.lse_host()[0]))  # L = 0
    assert np.all(s.o_host()[0] == 0.0)


def test_descale_broadcasts_and_unused_pages():
    w = syn.config(5, h_r=32, q_len=4, num_seqs=3, len_range=(200, 900))
    w.k_descale = np.array([1.375], dtype=np.float32)
    w.v_descale = np.array([0.625], dtype=np.float32)
    a, _ = check(w)
    w2 = copy.deepcopy(w)
    owned = set()
    for bi, L in enumerate(w.seq_lens):
        owned |= set(w.block_table[bi, : -(-int(L) // w.page_size)].tolist())
    free = [p for p in range(w.num_pages) if p not in owned]
    w2.k_cache[free] = 0x3F
    w2.v_cache[free] = 0x40
    b = run(w2)
    assert torch.equal(a.o_packed, b.o_packed) and torch.equal(a.lse, b.lse)


@pytest.mark.parametrize("layout", ["hnd", "interleaved", "flashinfer"])
def test_kv_layouts_match_nhd(layout):
    w = syn.make_workload("qrows_layout", [200, 513, 900], 2, 4, 32, 32, seed=93)
    a = run(w)
    b = run(w, kv_layout=layout)
    assert torch.equal(a.o_packed, b.o_packed) and torch.equal(a.lse, b.lse)


def test_determinism_and_graph_replay():
    w = syn.config(5, h_r=16, q_len=8, num_seqs=4, len_range=(500, 3000))
    s = run(w)
    o0, l0 = s.o_vllm.clone(), s.lse.clone()
    for _ in range(3):
        s.step()
    torch.cuda.synchronize()
    assert torch.equal(o0, s.o_vllm) and torch.equal(l0, s.lse)
    stream = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    s.o_vllm.zero_()
    with torch.cuda.graph(g, stream=stream):
        s.step(stream=stream)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(o0, s.o_vllm) and torch.equal(l0, s.lse)


# ---- rows held two or four times (64 or 32 packed rows per q tile): every
# copy takes a share of each tile's keys, the copies of a row share its
# reference maximum and GEMM2 runs transposed on the packed rows


@pytest.mark.parametrize("q_len,h_r,causal", [(3, 8, True), (1, 24, False), (4, 16, True), (2, 5, False)])
@pytest.mark.parametrize("page_size", [16, 128])
def test_row_copies_lengths_and_masks(q_len, h_r, causal, page_size):
    lens = [0, 1, 2, 5, 31, 32, 33, 127, 128, 129, 300, 1100]
    w = syn.make_workload("copies", lens, q_len, 2, h_r, page_size, seed=61 + q_len * h_r, causal=causal, max_splits=4)
    s, _ = check(w, force_splits=2)
    n_q = q_len * h_r
    assert s.kernel == ("qm_r32_bf16" if n_q <= 32 else "qm_r64_bf16")
    assert np.all(np.isneginf(s.lse_host()[0]))  # L = 0
    assert np.all(s.o_host()[0] == 0.0)


def test_row_copies_e4m3_q_and_determinism():
    w = syn.make_workload("copies_e4m3", [400, 2000, 3100], 2, 2, 16, 64, seed=67, q_is_e4m3=True)
    a, _ = check(w)
    assert a.kernel == "qm_r32_e4m3"
    o0, l0 = a.o_vllm.clone(), a.lse.clone()
    for _ in range(3):
        a.step()
    torch.cuda.synchronize()
    assert torch.equal(o0, a.o_vllm) and torch.equal(l0, a.lse)


@pytest.mark.parametrize("h_r,q_len", [(32, 1), (32, 4)], ids=["rows32_x4", "rows128"])
def test_softmax_stress_identical_keys_long_rows(h_r, q_len):
    # every key of a 16384-key row identical: all probabilities equal, the
    # row sum is as large as it gets (L terms of the same size), and O is the
    # plain mean of V; LSE = z + ln L within 2e-3 asks for an accurate sum
    w = syn.config(5, h_r=h_r, q_len=q_len, num_seqs=2, len_range=(0, 16384))
    for b in range(w.num_seqs):
        L = int(w.seq_lens[b])
        pages = w.block_table[b, : -(-L // w.page_size)]
        row = w.k_cache[pages[0], 0].copy()
        w.k_cache[pages] = row[None, None]
        w.k_cache[pages[-1], (L % w.page_size) or w.page_size :] = 0x7F  # keep the tail poison
    check(w)


@pytest.mark.parametrize("h_r,q_len", [(32, 1), (32, 4)], ids=["rows32_x4", "rows128"])
def test_softmax_stress_wide_logit_spread(h_r, q_len):
    # queries scaled by 6: logits spread over about +-16 around their
    # maximum, so most probabilities sit far below the largest and the
    # reference maximum moves late in a row
    w = syn.config(5, h_r=h_r, q_len=q_len, num_seqs=3, len_range=(0, 9000))
    w.q = syn.bf16_encode(syn.bf16_bits_to_float(w.q) * 6.0)
    check(w)


@pytest.mark.parametrize("h_r,q_len", [(32, 1), (16, 4)], ids=["rows32_x4", "rows64_x2"])
def test_row_copies_late_maximum_in_one_slice(h_r, q_len):
    """The keys of one copy's slice (the last 32 / 64 keys of a tile) grow
    from tile 3 on, so the row maximum moves late and from a single copy: the
    shared maximum must rescale the O^T column that every copy has added to."""
    w = syn.config(5, h_r=h_r, q_len=q_len, num_seqs=3, len_range=(1500, 4000))
    kr = 128 // (128 // (h_r * q_len))  # keys per copy slice
    for b in range(w.num_seqs):
        L = int(w.seq_lens[b])
        for key in range(3 * 128, L):
            if key % 128 < 128 - kr:
                continue
            pg, off = w.block_table[b, key // w.page_size], key % w.page_size
            v = syn.e4m3_decode(w.k_cache[pg, off]) * 4.0
            w.k_cache[pg, off] = syn.e4m3_encode(v)
    check(w)

