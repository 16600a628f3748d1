"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, on
the same seeded inputs, element by element.

Small cases (several KV tiles and a ragged tail, every row checked) cover
each config; full-size cases (the benchmark's sizes and launch
configuration) are checked on sampled (sequence, kv head) units.  Edge
cases: empty and shorter-than-q_len sequences, padded work lists, an
uninitialised (NaN) workspace, poisoned unused pages and garbage block-table
padding, forced splits, every KV layout the strides allow, descale
broadcasts, determinism and CUDA-graph replay.
"""

import copy

import numpy as np
import pytest
import torch

import oracle
from oracle.layout_ref import pack_q_ref, unpack_o_ref
from paged_fp8_kv_gb300 import synthetic as syn
from paged_fp8_kv_gb300.session import DecodeSession
from tests.gpu_helpers import compare, sample_units

pytestmark = pytest.mark.gpu

CC, TC = 1, 2  # MJ_KERNEL_CUDA_CORE, MJ_KERNEL_TENSOR_CORE
KERNELS = pytest.mark.parametrize("kernel", [CC, TC], ids=["cuda_core", "tensor_core"])


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_fp8_kv_gb300.build import build

    build()


def run(w, nan_workspace=True, **kw):
    s = DecodeSession(w, **kw)
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


# ------------------------------------------------------------------ configs


@KERNELS
def test_config1_tiny_full(kernel):
    w = syn.config(1)
    s, errs = check(w, kernel=kernel)
    assert s.plan.max_n_splits == 1


@KERNELS
@pytest.mark.parametrize("force", [0, 3])
def test_config2_small(force, kernel):
    w = syn.config(2, num_seqs=6, len_range=(300, 1500))
    check(w, force_splits=force, kernel=kernel)


@KERNELS
def test_config2_full_sampled(kernel):
    w = syn.config(2)
    s = run(w, kernel=kernel)
    units = sample_units(w, 24, seed=2, include=[(int(np.argmax(w.seq_lens)), 0)])
    compare(w, s.o_host(), s.lse_host(), units=units)


@KERNELS
def test_config3_small_split_and_merge(kernel):
    w = syn.config(3, num_seqs=4, len_range=(6000, 500))
    s, _ = check(w, kernel=kernel)
    assert s.plan.n_splits[0] > 1  # the long sequence is split and merged


@KERNELS
def test_config3_full_sampled(kernel):
    w = syn.config(3)
    s = run(w, kernel=kernel)
    assert s.plan.n_splits[0] > 1
    compare(w, s.o_host(), s.lse_host(), units=[(0, 0), (3, 0), (7, 0)])


@KERNELS
@pytest.mark.parametrize("variant", [None, "noncausal"])
def test_config4_small(variant, kernel):
    w = syn.config(4, variant=variant, num_seqs=5, len_range=(200, 1300))
    check(w, kernel=kernel)


@KERNELS
def test_config4_full_sampled(kernel):
    w = syn.config(4)
    s = run(w, kernel=kernel)
    units = sample_units(w, 12, seed=4, include=[(int(np.argmax(w.seq_lens)), 7)])
    compare(w, s.o_host(), s.lse_host(), units=units)


@KERNELS
@pytest.mark.parametrize("h_r,q_len", syn.SWEEP_POINTS)
def test_config5_small(h_r, q_len, kernel):
    w = syn.config(5, h_r=h_r, q_len=q_len, num_seqs=3, len_range=(0, 700))
    check(w, kernel=kernel)


@KERNELS
@pytest.mark.parametrize("h_r,q_len", [(16, 1), (32, 16)])
def test_config5_full_sampled(h_r, q_len, kernel):
    w = syn.config(5, h_r=h_r, q_len=q_len)
    s = run(w, kernel=kernel)
    compare(w, s.o_host(), s.lse_host(), units=[(0, 0), (77, 0), (127, 0)])


# --------------------------------------------------------------- edge cases


@KERNELS
@pytest.mark.parametrize("q_len,causal", [(1, True), (4, True), (3, False)])
def test_empty_short_and_aligned_lengths(q_len, causal, kernel):
    lens = [0, 1, 2, 3, 16, 127, 128, 129, 256, 300]
    w = syn.make_workload("edge", lens, q_len, 2, 4, 16, seed=51, causal=causal, max_splits=4)
    s, _ = check(w, force_splits=2, kernel=kernel)
    lse = s.lse_host()
    assert np.all(np.isneginf(lse[0]))  # L = 0
    assert np.all(s.o_host()[0] == 0.0)


@KERNELS
def test_padded_work_list_changes_nothing(kernel):
    w = syn.config(2, num_seqs=5, len_range=(200, 900))
    a = run(w, kernel=kernel)
    b = run(w, pad_to=a.plan.num_work + 37, kernel=kernel)
    assert b.plan.num_work == a.plan.num_work + 37
    assert torch.equal(a.o_packed, b.o_packed) and torch.equal(a.lse, b.lse)


@pytest.mark.parametrize("cfg", [3, 5])
def test_merge_hint_unknown_gives_same_bytes(cfg):
    w = syn.config(cfg, num_seqs=3, len_range=(3000, 400) if cfg == 3 else (0, 3000))
    a = run(w)
    assert a.plan.max_n_splits > 1
    b = DecodeSession(w)
    from paged_fp8_kv_gb300 import decode_attn

    decode_attn(
        b.params, q=b.q_packed, k_cache=b.k_cache, v_cache=b.v_cache, block_table=b.block_table,
        seq_lens=b.seq_lens, work=b.work, n_splits=b.n_splits, q_descale=b.q_descale, k_descale=b.k_descale,
        v_descale=b.v_descale, o=b.o_packed, lse=b.lse, workspace=b.workspace, softmax_scale=w.softmax_scale,
        scale_o=w.scale_o, max_n_splits=0,
    )
    torch.cuda.synchronize()
    # the hint sizes the merge (warps per row), which may change the
    # summation order of merged rows: equal up to fp32 rounding
    torch.testing.assert_close(a.o_packed.float(), b.o_packed.float(), rtol=1e-2, atol=1e-6)
    torch.testing.assert_close(a.lse, b.lse, rtol=1e-6, atol=1e-6)


@KERNELS
def test_workspace_contents_do_not_matter(kernel):
    w = syn.config(3, num_seqs=3, len_range=(3000, 400))
    a = run(w, nan_workspace=True, kernel=kernel)
    b = run(w, nan_workspace=False, kernel=kernel)
    b.fill_workspace(1e30)
    b.step()
    torch.cuda.synchronize()
    assert torch.equal(a.o_packed, b.o_packed) and torch.equal(a.lse, b.lse)


@KERNELS
def test_unused_pages_and_table_padding_are_never_read(kernel):
    w = syn.config(4, num_seqs=3, len_range=(100, 700))
    a = run(w, kernel=kernel)
    w2 = copy.deepcopy(w)
    owned = set()
    for bi, L in enumerate(w.seq_lens):
        owned |= set(w.block_table[bi, : -(-int(L) // w.page_size)].tolist())
    free = [p for p in range(w.num_pages) if p not in owned]
    w2.k_cache[free] = 0x3F
    w2.v_cache[free] = 0x40
    b = run(w2, kernel=kernel)
    assert torch.equal(a.o_packed, b.o_packed) and torch.equal(a.lse, b.lse)


@KERNELS
def test_page_permutation_gives_identical_bytes(kernel):
    w = syn.config(2, num_seqs=4, len_range=(300, 800))
    a = run(w, kernel=kernel)
    w2 = copy.deepcopy(w)
    perm = np.random.default_rng(9).permutation(w.num_pages)
    inv = np.argsort(perm)
    w2.k_cache = np.ascontiguousarray(w.k_cache[perm])
    w2.v_cache = np.ascontiguousarray(w.v_cache[perm])
    for bi, L in enumerate(w.seq_lens):
        n = -(-int(L) // w.page_size)
        w2.block_table[bi, :n] = inv[w.block_table[bi, :n]]
    b = run(w2, kernel=kernel)
    assert torch.equal(a.o_packed, b.o_packed) and torch.equal(a.lse, b.lse)


@KERNELS
def test_determinism_and_graph_replay(kernel):
    w = syn.config(4, num_seqs=4, len_range=(500, 2000))
    s = run(w, kernel=kernel)
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


@KERNELS
@pytest.mark.parametrize("layout", ["hnd", "interleaved", "flashinfer"])
def test_kv_layouts_match_nhd(layout, kernel):
    w = syn.config(4, num_seqs=3, len_range=(200, 900))
    a = run(w, kernel=kernel)
    b = run(w, kv_layout=layout, kernel=kernel)
    assert torch.equal(a.o_packed, b.o_packed) and torch.equal(a.lse, b.lse)


@KERNELS
@pytest.mark.parametrize("kind", ["per_tensor", "per_head"])
def test_descale_broadcasts(kind, kernel):
    w = syn.config(2, num_seqs=3, len_range=(200, 700))
    if kind == "per_tensor":
        w.k_descale = np.array([1.375], dtype=np.float32)
        w.v_descale = np.array([0.625], dtype=np.float32)
    else:
        w.k_descale = np.linspace(0.5, 2.0, w.h_k).astype(np.float32)
        w.v_descale = np.linspace(2.0, 0.5, w.h_k).astype(np.float32)
    check(w, kernel=kernel)


@pytest.mark.parametrize("q_is_e4m3", [False, True])
def test_pack_unpack_bit_exact(q_is_e4m3):
    w = syn.make_workload("pack", [50, 60, 70], 5, 3, 4, 16, seed=61, q_is_e4m3=q_is_e4m3)
    s = DecodeSession(w)
    from paged_fp8_kv_gb300 import pack_q, unpack_o

    pack_q(s.q_vllm, s.q_packed, 3, 5, 3, 4)
    torch.cuda.synchronize()
    ref = pack_q_ref(w.q.view(np.int16) if w.q.dtype == np.uint16 else w.q, 3, 5, 3, 4)
    np.testing.assert_array_equal(s.q_packed.cpu().numpy(), ref)
    src = torch.randn(3, 3, 20, 128, device="cuda").to(torch.bfloat16)
    dst = torch.empty(15, 12, 128, dtype=torch.bfloat16, device="cuda")
    unpack_o(src, dst, 3, 5, 3, 4)
    torch.cuda.synchronize()
    ref_o = unpack_o_ref(src.view(torch.int16).cpu().numpy(), 3, 5, 3, 4)
    np.testing.assert_array_equal(dst.view(torch.int16).cpu().numpy(), ref_o)


def test_unpacked_output_matches_oracle_layout():
    w = syn.config(4, num_seqs=2, len_range=(300, 600))
    s = run(w)
    ref_o, _ = oracle.attention(w)
    got = s.o_vllm.float().cpu().numpy()
    ref_v = unpack_o_ref(ref_o, w.num_seqs, w.q_len, w.h_k, w.h_r)
    assert np.all(np.abs(got - ref_v) <= 2e-2 + 2e-2 * np.abs(ref_v))


@pytest.mark.parametrize(
    "cfg,kw,kernel",
    [
        (2, dict(num_seqs=4, len_range=(300, 2000)), 2),  # swap-AB
        (2, dict(num_seqs=4, len_range=(300, 2000)), 3),  # head-grouped
        (4, dict(num_seqs=3, len_range=(500, 1500)), 4),  # query rows
        (3, dict(num_seqs=3, len_range=(3000, 300), max_splits=16), 2),  # fully-fp8, split
    ],
    ids=["swap_ab", "grouped", "query_rows", "fp8_split"],
)
def test_kv_evict_first_leaves_results_unchanged(cfg, kw, kernel):
    # an L2 cache policy on the K/V loads changes no byte of the output
    w = syn.config(cfg, **kw)
    a = run(w, kernel=kernel, kv_evict_first=-1)
    b = run(w, kernel=kernel, kv_evict_first=1)
    assert torch.equal(a.o_packed, b.o_packed) and torch.equal(a.lse, b.lse)
    compare(w, b.o_host(), b.lse_host())


@pytest.mark.parametrize("splits,lo,hi", [(3, 2, 4), (6, 5, 8), (12, 9, 16), (40, 17, 64), (100, 65, 128)])
def test_merge_instances_by_split_count(splits, lo, hi):
    # the merge stages 4, 8 or 16 splits a warp and spreads a row over 1, 4
    # or 16 warps by the largest split count: each instance against the oracle
    w = syn.config(2, num_seqs=3, len_range=(25600, 26000), max_splits=128)
    s, _ = check(w, force_splits=splits)
    assert lo <= s.plan.max_n_splits <= hi


def test_merge_refuses_a_hint_below_the_split_count():
    # a max_n_splits hint of 2 sizes the merge for 4 splits a row; a plan
    # with 6 splits must be refused (status word), not merged in part; with
    # the right hint the same call merges and matches the oracle
    import paged_fp8_kv_gb300 as mj

    w = syn.config(2, num_seqs=3, len_range=(25600, 26000), max_splits=16)
    s = DecodeSession(w, force_splits=6)
    assert s.plan.max_n_splits == 6
    s.fill_workspace(float("nan"))

    def call(hint, status):
        mj.decode_attn(
            s.params, q=s.q_packed, k_cache=s.k_cache, v_cache=s.v_cache, block_table=s.block_table,
            seq_lens=s.seq_lens, work=s.work, n_splits=s.n_splits, q_descale=s.q_descale,
            k_descale=s.k_descale, v_descale=s.v_descale, o=s.o_packed, lse=s.lse, workspace=s.workspace,
            softmax_scale=w.softmax_scale, scale_o=w.scale_o, status=status, max_n_splits=hint,
        )
        torch.cuda.synchronize()

    s.o_packed.fill_(7.0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    call(2, status)
    assert int(status.item()) == 1  # MJ_ERR_INVALID_ARG
    # every sequence had 6 splits: none was merged, O kept its old bytes
    assert torch.all(s.o_packed.float() == 7.0)
    status.zero_()
    call(6, status)
    assert int(status.item()) == 0
    compare(w, s.o_host(), s.lse_host())


@pytest.mark.parametrize("cfg,kw", [(4, dict(num_seqs=3, len_range=(500, 1500))), (3, dict(num_seqs=3, len_range=(3000, 300)))],
                         ids=["spec_verify_qlen4", "skewed_fp8_split"])
def test_staged_serving_step_matches_the_step(cfg, kw):
    # the host-to-host serving step (one pinned input copy, the step as a
    # CUDA graph, one output copy) gives the plain step's bytes, and is
    # captured again when the plan's shape changes
    import paged_fp8_kv_gb300 as mj

    w = syn.config(cfg, **kw)
    s = run(w)
    ref_o, ref_lse = s.o_vllm.cpu(), s.lse.cpu()
    e = DecodeSession(w)
    e.stage()
    for force in (0, 3, 0):
        plan = mj.decode_plan(e.params, w.seq_lens, sm_count=e.sm_count, force_splits=force)
        out = e.staged_step(plan)
        torch.cuda.synchronize()
        o = out["o"].clone()
        lse = out["lse"].view(w.num_seqs, w.h_k, w.n_q).clone()
        if force == 0:
            assert torch.equal(o.view(torch.int16), ref_o.view(torch.int16))
            assert torch.equal(lse, ref_lse)
        else:
            packed = torch.from_numpy(pack_q_ref(o.float().numpy(), w.num_seqs, w.q_len, w.h_k, w.h_r))
            compare(w, packed.numpy(), lse.numpy())


@pytest.mark.parametrize("cfg,kw", [(4, dict(num_seqs=3, len_range=(500, 1500))), (3, dict(num_seqs=3, len_range=(3000, 300)))],
                         ids=["spec_verify_qlen4", "skewed_fp8_split"])
def test_pipelined_serving_steps_match_the_synchronous_step(cfg, kw):
    # two slots over one KV pool, steps queued back to back with a different
    # Q each: every step's O and LSE equal the synchronous staged step's on
    # the same inputs (same kernels, same plan: the same bytes), and step 0
    # matches the oracle
    import paged_fp8_kv_gb300 as mj
    from paged_fp8_kv_gb300.session import StagedPipeline

    w = syn.config(cfg, **kw)
    pipe = StagedPipeline(w, depth=2)
    assert pipe.slots[1].k_cache.data_ptr() == pipe.slots[0].k_cache.data_ptr()  # one pool
    e = DecodeSession(w)
    e.stage()
    p0 = pipe.slots[0]
    base = torch.from_numpy(w.q.view(np.int16) if w.q.dtype == np.uint16 else w.q)

    def q_of(i):
        if base.dtype == torch.int16:  # bf16 bits: a different Q per step
            return (base.view(torch.bfloat16).float() * (1.0 + 0.25 * i)).to(torch.bfloat16).view(torch.int16)
        return torch.roll(base, shifts=i, dims=0)  # e4m3 codes: rows rotated

    steps, got = 5, {}
    for i in range(steps):
        plan = mj.decode_plan(p0.params, w.seq_lens, sm_count=p0.sm_count, force_splits=3 if i == 3 else 0)
        pipe.inputs(i)["q"].copy_(q_of(i))
        pipe.submit(i, plan)
        if i >= 1:
            out = pipe.outputs(i - 1)
            got[i - 1] = (out["o"].clone(), out["lse"].clone())
    out = pipe.outputs(steps - 1)
    got[steps - 1] = (out["o"].clone(), out["lse"].clone())
    for i in range(steps):
        plan = mj.decode_plan(e.params, w.seq_lens, sm_count=e.sm_count, force_splits=3 if i == 3 else 0)
        e._host_in["q"].copy_(q_of(i))
        ref = e.staged_step(plan)
        torch.cuda.synchronize()
        assert torch.equal(got[i][0].view(torch.int16), ref["o"].view(torch.int16)), f"step {i}"
        assert torch.equal(got[i][1], ref["lse"]), f"step {i}"
    o0 = got[0][0].float().numpy()
    compare(w, pack_q_ref(o0, w.num_seqs, w.q_len, w.h_k, w.h_r), got[0][1].view(w.num_seqs, w.h_k, w.n_q).numpy())
