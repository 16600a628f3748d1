"""GPU parity of the head-grouped tensor-core kernel
(MJ_KERNEL_TENSOR_CORE_GROUPED): one CTA serves 2, 4 or 8 kv heads, whose
rows of every page it fetches together.

The kernel's arithmetic is the per-head tensor-core kernel's; what is new is
the tile shape (G heads x 128/G keys on the MMA's M side, every head's query
rows on N, P block-diagonal), the per-head masking, maxima and descales
inside one tile, and the smaller key step.  So these cases compare it with
the fp64 oracle element by element on: every instance (8 heads x 4 rows,
4 heads x 8 rows, 2 heads x 32 rows with a head's keys in a warp pair),
every page size (a page is 1, 2, 4 or 8 steps, or two
pages one step), bf16 and e4m3 Q, causal and non-causal, empty and ragged
lengths, forced splits with the merge, per-head descales that differ inside
one CTA, every KV layout, determinism and graph replay.
"""

import copy

import numpy as np
import pytest
import torch

from paged_fp8_kv_gb300 import synthetic as syn
from paged_fp8_kv_gb300.session import DecodeSession
from tests.gpu_helpers import compare, sample_units

pytestmark = pytest.mark.gpu

TCG = 3  # MJ_KERNEL_TENSOR_CORE_GROUPED


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_fp8_kv_gb300.build import build

    build()


def run(w, nan_workspace=True, **kw):
    s = DecodeSession(w, kernel=TCG, **kw)
    assert s.kernel.startswith("tcg_"), s.kernel
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


@pytest.mark.parametrize("force", [0, 3])
def test_gqa_decode_small(force):
    w = syn.config(2, num_seqs=6, len_range=(300, 1500))
    s, _ = check(w, force_splits=force)
    assert s.kernel == "tcg_g8r4_bf16"


def test_gqa_decode_full_sampled():
    w = syn.config(2)
    s = run(w)
    units = sample_units(w, 24, seed=2, include=[(int(np.argmax(w.seq_lens)), 0), (0, 7)])
    compare(w, s.o_host(), s.lse_host(), units=units)


@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
@pytest.mark.parametrize("h_k,h_r,q_len", [(8, 4, 1), (8, 2, 2), (4, 8, 1), (12, 3, 2)])
def test_instances_and_page_sizes(page_size, h_k, h_r, q_len):
    lens = [1, 15, 16, 17, 100, 250, 511, 700]
    w = syn.make_workload("grouped", lens, q_len, h_k, h_r, page_size, seed=71 + page_size, max_splits=4)
    s, _ = check(w, force_splits=2)
    g = 8 if (h_k % 8 == 0 and q_len * h_r <= 4) else 4
    assert s.kernel.startswith(f"tcg_g{g}")


@pytest.mark.parametrize("q_is_e4m3", [False, True])
@pytest.mark.parametrize("causal", [True, False])
def test_q_dtype_and_masking(q_is_e4m3, causal):
    lens = [5, 64, 333, 1029]
    w = syn.make_workload("grouped_q", lens, 2, 8, 4, 16, seed=83, q_is_e4m3=q_is_e4m3, causal=causal, max_splits=8)
    check(w)  # n_q = 8: the 4-head x 8-row instance
    w1 = syn.make_workload("grouped_q1", lens, 1, 8, 4, 16, seed=84, q_is_e4m3=q_is_e4m3, causal=causal)
    check(w1)  # n_q = 4: the 8-head x 4-row instance


@pytest.mark.parametrize("q_len,causal", [(1, True), (4, True), (3, False)])
def test_empty_short_and_aligned_lengths(q_len, causal):
    lens = [0, 1, 2, 3, 16, 127, 128, 129, 256, 300]
    w = syn.make_workload("edge", lens, q_len, 8, 2, 16, seed=51, causal=causal, max_splits=4)
    s, _ = check(w, force_splits=2)
    assert np.all(np.isneginf(s.lse_host()[0]))  # L = 0
    assert np.all(s.o_host()[0] == 0.0)


def test_descales_differ_per_head():
    w = syn.config(2, num_seqs=3, len_range=(200, 700))
    w.q_descale = np.linspace(0.5, 2.0, w.h_k).astype(np.float32)
    w.k_descale = np.geomspace(0.25, 4.0, w.num_seqs * w.h_k).reshape(w.num_seqs, w.h_k).astype(np.float32)
    w.v_descale = np.linspace(2.0, 0.5, w.num_seqs * w.h_k).reshape(w.num_seqs, w.h_k).astype(np.float32)
    check(w)


def test_padded_work_list_and_unused_pages():
    w = syn.config(2, num_seqs=5, len_range=(200, 900))
    a = run(w)
    b = run(w, pad_to=a.plan.num_work + 37)
    assert torch.equal(a.o_packed, b.o_packed) and torch.equal(a.lse, b.lse)
    w2 = copy.deepcopy(w)
    owned = set()
    for bi, L in enumerate(w.seq_lens):
        owned |= set(w.block_table[bi, : -(-int(L) // w.page_size)].tolist())
    free = [p for p in range(w.num_pages) if p not in owned]
    w2.k_cache[free] = 0x3F
    w2.v_cache[free] = 0x40
    c = run(w2)
    assert torch.equal(a.o_packed, c.o_packed) and torch.equal(a.lse, c.lse)


@pytest.mark.parametrize("layout", ["hnd", "interleaved", "flashinfer"])
def test_kv_layouts_match_nhd(layout):
    w = syn.config(2, num_seqs=3, len_range=(200, 900))
    a = run(w)
    b = run(w, kv_layout=layout)
    assert torch.equal(a.o_packed, b.o_packed) and torch.equal(a.lse, b.lse)


def test_determinism_and_graph_replay():
    w = syn.config(2, num_seqs=8, len_range=(500, 4000))
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


# ---- 2 heads x 32 rows: a head's 64 keys of a step span two warps, which
# exchange column maxima and row sums; one S buffer per warpgroup.


@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
@pytest.mark.parametrize("h_k,h_r,q_len", [(8, 8, 4), (2, 8, 3), (6, 4, 4), (4, 16, 1)])
def test_pair_instance_page_sizes(page_size, h_k, h_r, q_len):
    lens = [1, 63, 64, 65, 100, 250, 511, 700, 1300]
    w = syn.make_workload("grouped_pair", lens, q_len, h_k, h_r, page_size, seed=171 + page_size, max_splits=4)
    s, _ = check(w, force_splits=2)
    assert s.kernel == "tcg_g2r32_bf16"


@pytest.mark.parametrize("force", [0, 3])
def test_spec_verify_small_pair(force):
    w = syn.config(4, num_seqs=4, len_range=(300, 3000))
    s, _ = check(w, force_splits=force)
    assert s.kernel == "tcg_g2r32_bf16"


def test_spec_verify_full_sampled_pair():
    w = syn.config(4)
    s = run(w)
    units = sample_units(w, 16, seed=4, include=[(int(np.argmax(w.seq_lens)), 0), (int(np.argmin(w.seq_lens)), 7)])
    compare(w, s.o_host(), s.lse_host(), units=units)


@pytest.mark.parametrize("q_is_e4m3", [False, True])
@pytest.mark.parametrize("causal", [True, False])
def test_pair_q_dtype_and_masking(q_is_e4m3, causal):
    lens = [5, 64, 333, 1029]
    w = syn.make_workload("grouped_pair_q", lens, 4, 4, 8, 64, seed=183, q_is_e4m3=q_is_e4m3, causal=causal,
                          max_splits=8)
    s, _ = check(w)
    assert s.kernel.startswith("tcg_g2r32")


@pytest.mark.parametrize("q_len,causal", [(4, True), (3, False)])
def test_pair_empty_short_and_aligned_lengths(q_len, causal):
    lens = [0, 1, 2, 3, 16, 63, 64, 65, 127, 128, 129, 256, 300]
    w = syn.make_workload("edge_pair", lens, q_len, 2, 8, 16, seed=151, causal=causal, max_splits=4)
    s, _ = check(w, force_splits=2)
    assert s.kernel == "tcg_g2r32_bf16"
    assert np.all(np.isneginf(s.lse_host()[0]))  # L = 0
    assert np.all(s.o_host()[0] == 0.0)


def test_pair_determinism_and_layouts():
    # more units than CTAs: which CTA runs which unit varies between launches
    w = syn.config(4, num_seqs=12, len_range=(500, 6000))
    a = run(w)
    assert a.plan.num_work * (w.h_k // 2) > torch.cuda.get_device_properties(0).multi_processor_count
    o0, l0 = a.o_vllm.clone(), a.lse.clone()
    for _ in range(3):
        a.step()
    torch.cuda.synchronize()
    assert torch.equal(o0, a.o_vllm) and torch.equal(l0, a.lse)
    b = run(w, kv_layout="hnd")
    assert torch.equal(a.o_packed, b.o_packed) and torch.equal(a.lse, b.lse)


# ---- 1 head x 32 rows: a head's 128 keys of a step over the four warps of
# a group (an odd number of kv heads, or h_k = 1)


@pytest.mark.parametrize("page_size", [16, 64, 128])
@pytest.mark.parametrize("h_k,h_r,q_len", [(1, 32, 1), (1, 16, 2), (3, 8, 3)])
def test_one_head_instance(page_size, h_k, h_r, q_len):
    lens = [1, 63, 127, 128, 129, 250, 511, 700, 1300]
    w = syn.make_workload("grouped_one", lens, q_len, h_k, h_r, page_size, seed=271 + page_size, max_splits=4)
    s, _ = check(w, force_splits=2)
    assert s.kernel == "tcg_g1r32_bf16"


@pytest.mark.parametrize("q_is_e4m3", [False, True])
@pytest.mark.parametrize("causal", [True, False])
def test_one_head_q_dtype_masks_and_edges(q_is_e4m3, causal):
    lens = [0, 1, 2, 3, 16, 127, 128, 129, 300, 2100]
    w = syn.make_workload("edge_one", lens, 2, 1, 16, 32, seed=283, causal=causal, q_is_e4m3=q_is_e4m3, max_splits=8)
    s, _ = check(w)
    assert s.kernel.startswith("tcg_g1r32")
    assert np.all(np.isneginf(s.lse_host()[0]))  # L = 0
    assert np.all(s.o_host()[0] == 0.0)


def test_one_head_sweep_full_sampled_and_determinism():
    w = syn.config(5, h_r=32, q_len=1)
    s = run(w)
    compare(w, s.o_host(), s.lse_host(), units=[(0, 0), (64, 0), (127, 0)])
    o0, l0 = s.o_vllm.clone(), s.lse.clone()
    for _ in range(2):
        s.step()
    torch.cuda.synchronize()
    assert torch.equal(o0, s.o_vllm) and torch.equal(l0, s.lse)
