"""The C ABI without a GPU: the library loads and exports every symbol the
header declares; the host plan matches the plan oracle bit for bit; argument
validation rejects bad calls before anything is launched."""

import ctypes
import json
import os
import re

import numpy as np
import pytest

import paged_fp8_kv_gb300 as mj
from oracle.plan_ref import plan_ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mj.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    from paged_fp8_kv_gb300.build import build

    build()


def test_every_declared_symbol_is_exported():
    text = open(HEADER).read()
    names = sorted(set(re.findall(r"\b(mj_[a-z_0-9]+)\s*\(", text)))
    assert len(names) >= 7
    L = mj.lib()
    for n in names:
        assert hasattr(L, n), f"{n} declared in mj.h but not exported"


def _params(b, h_k=1, q_len=1, h_r=4, ps=16, max_blocks=1 << 16, max_splits=16, q_dtype=0, kernel=0):
    return mj.make_params(b, q_len, h_k, h_r, ps, max_blocks, 100000, True, q_dtype, max_splits, 128, kernel)


@pytest.mark.parametrize("case", json.load(open(os.path.join(ROOT, "tests", "golden", "plan_examples.json")))["cases"])
def test_plan_golden(case):
    a = case["args"]
    p = _params(len(a["seq_lens"]), h_k=a["h_k"], max_splits=a["max_splits"])
    plan = mj.decode_plan(
        p,
        a["seq_lens"],
        sm_count=a["sm_count"],
        ctas_per_sm=a["ctas_per_sm"],
        n_q_tiles=a["n_q_tiles"],
        force_splits=a.get("force_splits", 0),
        pad_to=a.get("pad_to", 0),
    )
    assert plan.chunk_tiles == case["chunk_tiles"]
    assert plan.n_splits.tolist() == case["n_splits"]
    if "work" in case:
        assert plan.work.tolist() == case["work"]
    else:
        assert plan.num_work == case["work_len"]


def test_plan_matches_oracle_bit_exact():
    rng = np.random.default_rng(41)
    for _ in range(500):
        b = int(rng.integers(1, 64))
        seq_lens = rng.integers(0, 40000, size=b)
        if rng.random() < 0.3:
            seq_lens[0] = int(rng.integers(100000, 300000))
        h_k = int(rng.choice([1, 2, 4, 8]))
        sm = int(rng.choice([20, 132, 148, 152]))
        cps = int(rng.integers(1, 9))
        ntiles = int(rng.choice([1, 2, 3]))
        max_splits = int(rng.choice([1, 2, 16, 64, 256]))
        force = int(rng.choice([0, 0, 0, 2, 7]))
        min_chunk = int(rng.choice([1, 1, 3]))
        ref = plan_ref(seq_lens.tolist(), h_k, ntiles, sm, cps, max_splits, force, min_chunk, 0)
        pad = 0 if rng.random() < 0.5 else len(ref.work) + int(rng.integers(0, 9))
        if pad:
            ref = plan_ref(seq_lens.tolist(), h_k, ntiles, sm, cps, max_splits, force, min_chunk, pad)
        p = _params(b, h_k=h_k, max_splits=max_splits, max_blocks=300000 // 16 + 1)
        got = mj.decode_plan(p, seq_lens, sm, cps, ntiles, force, min_chunk, pad)
        assert got.work.tolist() == [list(w) for w in ref.work]
        assert got.n_splits.tolist() == ref.n_splits
        assert got.chunk_tiles == ref.chunk_tiles


def test_plan_reports_library_defaults():
    p = _params(4, h_k=8, h_r=4)
    plan = mj.decode_plan(p, [1000, 2000, 3000, 4000])
    assert plan.opts.sm_count == 152 and plan.opts.ctas_per_sm >= 1 and plan.opts.n_q_tiles >= 1
    ref = plan_ref([1000, 2000, 3000, 4000], 8, plan.opts.n_q_tiles, 152, plan.opts.ctas_per_sm, 16)
    assert plan.work.tolist() == [list(w) for w in ref.work]


def _plan_status(params, seq_lens, cap=None, **opts):
    L = mj.lib()
    o = mj.PlanOpts(opts.get("sm", 0), 0, 0, 0, 0, opts.get("pad_to", 0))
    sl = np.asarray(seq_lens, dtype=np.int32)
    cap = cap if cap is not None else 4096
    work = np.zeros((max(cap, 1), 4), dtype=np.int32)
    ns = np.zeros(max(params.num_seqs, 1), dtype=np.int32)
    nw = ctypes.c_int32()
    return L.mj_decode_plan(
        ctypes.byref(params), ctypes.byref(o), sl.ctypes.data, work.ctypes.data, cap, ctypes.addressof(nw), ns.ctypes.data, None
    )


def test_plan_rejects_bad_input():
    p = _params(2, max_blocks=4, ps=16)  # at most 64 rows
    assert _plan_status(p, [64, 10]) == mj.MJ_OK
    assert _plan_status(p, [65, 10]) == mj.MJ_ERR_INVALID_ARG
    assert _plan_status(p, [-1, 10]) == mj.MJ_ERR_INVALID_ARG
    assert _plan_status(p, [64, 10], cap=1) == mj.MJ_ERR_CAPACITY
    assert _plan_status(p, [64, 10], pad_to=1) == mj.MJ_ERR_INVALID_ARG
    bad = _params(2)
    bad.head_dim = 64
    assert _plan_status(bad, [10, 10]) == mj.MJ_ERR_UNSUPPORTED
    bad = _params(2)
    bad.page_size = 8
    assert _plan_status(bad, [10, 10]) == mj.MJ_ERR_UNSUPPORTED
    bad = _params(2, max_splits=257)
    assert _plan_status(bad, [10, 10]) == mj.MJ_ERR_INVALID_ARG


def test_workspace_bytes():
    p = _params(3, h_k=2, q_len=2, h_r=4, max_splits=16)
    rows = 3 * 2 * 16 * 8
    ru = lambda x: (x + 255) // 256 * 256
    assert mj.workspace_bytes(p) == ru(rows * 128 * 4) + 2 * ru(rows * 4)
    assert mj.workspace_bytes(_params(3, max_splits=1)) == 0


def _good_args():
    a = mj.DecodeArgs()
    fake = 1 << 20  # aligned, never dereferenced: validation fails first
    for f in ("q", "k", "v", "block_table", "seq_lens", "work", "n_splits", "q_descale", "k_descale", "v_descale", "o", "lse"):
        setattr(a, f, fake)
    a.q_seq_stride = 4 * 128
    a.k_page, a.k_row, a.k_head = 16 * 128, 128, 128
    a.v_page, a.v_row, a.v_head = 16 * 128, 128, 128
    a.num_work = 1
    a.softmax_scale = 0.088
    a.scale_o = 1.0
    a.o_seq_stride = 4 * 128
    return a


def _attn_status(params, args):
    return mj.lib().mj_decode_attn(ctypes.byref(params), ctypes.byref(args), None)


def test_decode_attn_validation_rejects_before_launch():
    p = _params(1, h_r=4, max_splits=16)
    for field, val, want in [
        ("q", None, mj.MJ_ERR_INVALID_ARG),
        ("k", (1 << 20) + 8, mj.MJ_ERR_INVALID_ARG),  # misaligned
        ("k_row", 100, mj.MJ_ERR_INVALID_ARG),  # not a 16-byte multiple
        ("v_head", -16, mj.MJ_ERR_INVALID_ARG),
        ("num_work", 0, mj.MJ_ERR_INVALID_ARG),
        ("q_seq_stride", 3, mj.MJ_ERR_INVALID_ARG),
        ("softmax_scale", 0.0, mj.MJ_ERR_INVALID_ARG),
        ("workspace", None, mj.MJ_ERR_INVALID_ARG),  # max_splits > 1 needs one
    ]:
        a = _good_args()
        a.workspace = 1 << 20
        a.workspace_bytes = mj.workspace_bytes(p)
        setattr(a, field, val)
        assert _attn_status(p, a) == want, field
    a = _good_args()
    a.workspace = 1 << 20
    a.workspace_bytes = mj.workspace_bytes(p) - 1
    assert _attn_status(p, a) == mj.MJ_ERR_CAPACITY
    bad = _params(1, h_r=4)
    bad.head_dim = 256
    assert _attn_status(bad, _good_args()) == mj.MJ_ERR_UNSUPPORTED
    # two sequences: a sequence stride below one sequence's h_k * n_q rows of
    # d would make sequences overlap
    p2 = _params(2, h_k=2, h_r=4, max_splits=1)
    for field in ("q_seq_stride", "o_seq_stride"):
        a = _good_args()
        a.q_seq_stride = a.o_seq_stride = 2 * 4 * 128
        setattr(a, field, 2 * 4 * 128 - 8)
        assert _attn_status(p2, a) == mj.MJ_ERR_INVALID_ARG, field


def test_pack_validation():
    L = mj.lib()
    fake = 1 << 20
    assert L.mj_pack_q(fake, fake + (1 << 24), 3, 1, 1, 1, 1, 128, None) == mj.MJ_ERR_INVALID_ARG
    assert L.mj_pack_q(fake, fake + 8, 2, 1, 2, 1, 2, 128, None) == mj.MJ_ERR_INVALID_ARG  # misaligned dst
    assert L.mj_pack_q(fake, fake, 2, 1, 2, 1, 2, 128, None) == mj.MJ_ERR_INVALID_ARG  # overlap
    assert L.mj_unpack_o(None, fake, 1, 2, 1, 2, 128, None) == mj.MJ_ERR_INVALID_ARG


def test_plan_device_validation():
    # refusals on the host, before any launch
    L = mj.lib()
    p = _params(4, h_r=4)
    sl, work, ns = 1 << 20, 1 << 22, 1 << 24
    f = L.mj_decode_plan_device
    opts = lambda pad_to: mj.PlanOpts(152, 0, 0, 0, 0, pad_to)
    assert f(ctypes.byref(p), None, sl, work, ns, None, None, None) == mj.MJ_ERR_INVALID_ARG
    assert f(ctypes.byref(p), ctypes.byref(opts(0)), sl, work, ns, None, None, None) == mj.MJ_ERR_INVALID_ARG
    assert f(ctypes.byref(p), ctypes.byref(opts(8)), None, work, ns, None, None, None) == mj.MJ_ERR_INVALID_ARG
    assert f(ctypes.byref(p), ctypes.byref(opts(8)), sl, work + 4, ns, None, None, None) == mj.MJ_ERR_INVALID_ARG
    big = _params(16385, h_r=4)
    assert f(ctypes.byref(big), ctypes.byref(opts(8)), sl, work, ns, None, None, None) == mj.MJ_ERR_UNSUPPORTED


def test_plan_max_items_bounds_every_plan():
    # the bound on the work list holds for the rule's plans, whatever the
    # lengths; it is the tightest for an even batch that fills one wave
    rng = np.random.default_rng(17)
    for _ in range(300):
        b = int(rng.integers(1, 400))
        h_k = int(rng.choice([1, 2, 8]))
        ms = int(rng.choice([1, 16, 256]))
        p = _params(b, h_k=h_k, h_r=int(rng.choice([4, 16, 32])), max_splits=ms, max_blocks=4096)
        cps = int(rng.choice([1, 3, 5, 24]))
        force = int(rng.choice([0, 0, 3])) if ms > 1 else 0
        lens = rng.integers(0, 4096 * 16 + 1, size=b).tolist()
        if rng.random() < 0.3:
            lens = [4096 * 16] * b
        bound = mj.decode_plan_max_items(p, sm_count=152, ctas_per_sm=cps, force_splits=force)
        plan = mj.decode_plan(p, lens, sm_count=152, ctas_per_sm=cps, force_splits=force)
        assert plan.num_work <= bound
    assert mj.lib().mj_decode_plan_max_items(None, None) == -1


def test_check_hooks_validation():
    # the verification hooks refuse bad arguments on the host, before any launch
    L = mj.lib()
    p = _params(2, h_r=4)
    a = mj.DecodeArgs()
    assert L.mj_check_gather_kv(ctypes.byref(p), None, 0, 1 << 20, 128, None) == mj.MJ_ERR_INVALID_ARG
    assert L.mj_check_gather_kv(ctypes.byref(p), ctypes.byref(a), 0, 1 << 20, 128, None) == mj.MJ_ERR_INVALID_ARG
    a.k, a.v, a.block_table, a.seq_lens = 1 << 20, 1 << 21, 1 << 22, 1 << 23
    a.k_page = a.v_page = 16 * 128
    a.k_row = a.v_row = 128
    a.k_head = a.v_head = 128
    assert L.mj_check_gather_kv(ctypes.byref(p), ctypes.byref(a), 2, 1 << 24, 128, None) == mj.MJ_ERR_INVALID_ARG
    assert L.mj_check_gather_kv(ctypes.byref(p), ctypes.byref(a), 0, (1 << 24) + 8, 128, None) == mj.MJ_ERR_INVALID_ARG
    assert L.mj_check_gather_kv(ctypes.byref(p), ctypes.byref(a), 0, 1 << 24, 0, None) == mj.MJ_ERR_INVALID_ARG
    a.k_row = 100  # not a 16-byte multiple
    assert L.mj_check_gather_kv(ctypes.byref(p), ctypes.byref(a), 0, 1 << 24, 128, None) == mj.MJ_ERR_INVALID_ARG
    assert L.mj_check_dequant_e4m3(None, None) == mj.MJ_ERR_INVALID_ARG
    assert L.mj_check_dequant_e4m3((1 << 20) + 4, None) == mj.MJ_ERR_INVALID_ARG


def test_quantize_pack_validation():
    # every refusal happens on the host, before any launch
    L = mj.lib()
    src, dst, ds = 1 << 20, 1 << 26, 1 << 28
    q = L.mj_quantize_pack_q
    assert q(None, dst, ds, 1, 1, 1, 16, 128, None) == mj.MJ_ERR_INVALID_ARG
    assert q(src, dst, None, 1, 1, 1, 16, 128, None) == mj.MJ_ERR_INVALID_ARG
    assert q(src + 8, dst, ds, 1, 1, 1, 16, 128, None) == mj.MJ_ERR_INVALID_ARG  # misaligned Q
    assert q(src, dst + 4, ds, 1, 1, 1, 16, 128, None) == mj.MJ_ERR_INVALID_ARG  # misaligned codes
    assert q(src, dst, ds + 2, 1, 1, 1, 16, 128, None) == mj.MJ_ERR_INVALID_ARG  # misaligned descales
    assert q(src, dst, ds, 0, 1, 1, 16, 128, None) == mj.MJ_ERR_INVALID_ARG
    assert q(src, dst, ds, 1, 1, 1, 16, 120, None) == mj.MJ_ERR_UNSUPPORTED  # head_dim % 16
    assert q(src, src + 2048, ds, 1, 1, 1, 16, 128, None) == mj.MJ_ERR_INVALID_ARG  # codes inside Q
    assert q(src, dst, dst + 16, 1, 1, 1, 16, 128, None) == mj.MJ_ERR_INVALID_ARG  # descales inside codes


def test_status_strings_and_kernel_name():
    assert mj.status_string(mj.MJ_OK) == "ok"
    assert "timed out" in mj.status_string(mj.MJ_ERR_TIMEOUT)
    assert mj.kernel_name(_params(2, h_r=4)).startswith(("cc_", "tc_"))


def test_grouped_kernel_choice_and_plan():
    # the head-grouped kernel: 8 heads x 4 rows, 4 heads x 8 rows or 2 heads
    # x 32 rows per CTA
    grouped = mj.MJ_KERNEL_TENSOR_CORE_GROUPED
    assert mj.kernel_name(_params(2, h_k=8, h_r=4, kernel=grouped)) == "tcg_g8r4_bf16"
    assert mj.kernel_name(_params(2, h_k=8, h_r=8, kernel=grouped)) == "tcg_g4r8_bf16"
    assert mj.kernel_name(_params(2, h_k=12, h_r=2, kernel=grouped)) == "tcg_g4r8_bf16"
    assert mj.kernel_name(_params(2, h_k=8, h_r=16, kernel=grouped)) == "tcg_g2r32_bf16"
    assert mj.kernel_name(_params(2, h_k=6, h_r=4, kernel=grouped)) == "tcg_g2r32_bf16"
    assert mj.kernel_name(_params(2, h_k=8, q_len=4, h_r=8, kernel=grouped, q_dtype=1)) == "tcg_g2r32_e4m3"
    assert mj.kernel_name(_params(2, h_k=3, h_r=4, kernel=grouped)) == "tcg_g1r32_bf16"
    assert mj.kernel_name(_params(2, h_k=1, h_r=16, kernel=grouped)) == "tcg_g1r32_bf16"
    # more than 32 rows per head: refused
    for h_k, h_r in [(8, 40), (1, 33)]:
        p = _params(2, h_k=h_k, h_r=h_r, kernel=grouped)
        with pytest.raises(mj.MjError):
            mj.kernel_name(p)
        assert _plan_status(p, [10, 10]) == mj.MJ_ERR_UNSUPPORTED
    # its occupancy counts (CTA, kv head) pairs, so one wave covers every
    # head of sm_count * CTAs-per-SM * 8 / h_k work items
    p = _params(4, h_k=8, h_r=4, kernel=grouped)
    plan = mj.decode_plan(p, [1000, 2000, 3000, 4000])
    assert plan.opts.ctas_per_sm % 8 == 0 and plan.opts.n_q_tiles == 1
    ref = plan_ref([1000, 2000, 3000, 4000], 8, 1, 152, plan.opts.ctas_per_sm, 16)
    assert plan.work.tolist() == [list(w) for w in ref.work]


def test_query_rows_kernel_choice():
    # more than 16 packed rows: the query-rows kernel (32, 64 or 128 rows per q tile)
    assert mj.kernel_name(_params(2, h_k=1, q_len=2, h_r=32)) == "qm_r64_bf16"
    assert mj.kernel_name(_params(2, h_k=8, q_len=5, h_r=8)) == "qm_r64_bf16"
    assert mj.kernel_name(_params(2, h_k=1, q_len=4, h_r=32)) == "qm_bf16"
    # 17 to 32 rows: 32 rows per q tile (each held four times)
    assert mj.kernel_name(_params(2, h_k=1, q_len=1, h_r=32)) == "qm_r32_bf16"
    assert mj.kernel_name(_params(2, h_k=8, q_len=4, h_r=8)) == "qm_r32_bf16"
    assert mj.kernel_name(_params(2, h_k=3, q_len=3, h_r=6)) == "qm_r32_bf16"
    # up to 16 rows: the swap-AB kernel
    assert mj.kernel_name(_params(2, h_k=8, q_len=2, h_r=8)) == "tc_r16_bf16"
    assert mj.kernel_name(_params(2, h_k=1, q_len=1, h_r=16)) == "tc_r16_bf16"
    qr = mj.MJ_KERNEL_TENSOR_CORE_QROWS
    assert mj.kernel_name(_params(2, h_k=1, h_r=16, kernel=qr, q_dtype=1)) == "qm_r32_e4m3"
    assert mj.kernel_name(_params(2, h_k=1, q_len=8, h_r=16, kernel=qr, q_dtype=1)) == "qm_e4m3"
    # more than 128 rows: two q tiles of 128 rows per CTA
    assert mj.kernel_name(_params(2, h_k=1, q_len=16, h_r=16)) == "qm_pair_bf16"
    assert mj.kernel_name(_params(2, h_k=1, q_len=3, h_r=48)) == "qm_pair_bf16"
    assert mj.kernel_name(_params(2, h_k=1, q_len=16, h_r=32, kernel=qr, q_dtype=1)) == "qm_pair_e4m3"
    plan = mj.decode_plan(_params(4, h_k=1, q_len=16, h_r=32), [1000, 2000, 3000, 4000])
    assert plan.opts.n_q_tiles == 2  # 512 rows: two CTAs of two q tiles


def test_default_plan_splits_when_long_sequences_dominate():
    # 60 short sequences and 4 very long ones, 8 kv heads, 4 rows: one wave
    # of the occupancy-pinned plan would end on the 4 long sequences' CTAs,
    # and the library's default takes a finer plan, which the restated rule
    # reproduces from the reported options
    lens = [512] * 60 + [65536] * 4
    p = mj.make_params(64, 1, 8, 4, 16, 4096, 64 * 4096, True, mj.MJ_BF16, 16, 128, 0, 0)
    plan = mj.decode_plan(p, lens, sm_count=152)
    assert plan.max_n_splits > 1
    ref = plan_ref(lens, 8, plan.opts.n_q_tiles, 152, plan.opts.ctas_per_sm, 16)
    assert [tuple(x) for x in plan.work.tolist()] == [tuple(x) for x in ref.work]
    assert plan.n_splits.tolist() == ref.n_splits
    # the chosen slots are one of the model's candidates: 1, 5/3, 8/3 or 4
    # times the kernel's co-resident CTAs (what the device plan takes by
    # default)
    co = mj.PlanOpts(152, 0, 0, 0, 0, 0)
    assert mj.lib().mj_decode_plan_max_items(ctypes.byref(p), ctypes.byref(co)) > 0
    cands = {(co.ctas_per_sm * t + 2) // 3 for t in (3, 5, 8, 12)}
    assert plan.opts.ctas_per_sm in cands


def test_check_preconditions():
    from paged_fp8_kv_gb300 import synthetic as syn

    w = syn.make_workload("pre", [0, 1, 37, 100, 300], 1, 2, 4, 16, seed=7)
    p = mj.make_params(w.num_seqs, 1, 2, 4, 16, w.max_blocks, w.num_pages, True, mj.MJ_BF16, 16, 128, 0, 0)
    ok = (w.block_table, w.seq_lens, w.q_descale, w.k_descale, w.v_descale)
    # the generator leaves -1 / INT32_MAX garbage past each sequence's pages
    assert (w.block_table < 0).any()
    assert mj.check_preconditions(p, *ok) == (mj.MJ_OK, -1)
    bt = w.block_table.copy()
    bt[3, 2] = w.num_pages  # a page the sequence reads, out of the pool
    assert mj.check_preconditions(p, bt, *ok[1:]) == (mj.MJ_ERR_INVALID_ARG, 3)
    bt = w.block_table.copy()
    bt[2, 3] = -5  # page 3 of a 37-key sequence (3 pages): never read
    assert mj.check_preconditions(p, bt, *ok[1:]) == (mj.MJ_OK, -1)
    bt[2, 2] = -5  # its last page
    assert mj.check_preconditions(p, bt, *ok[1:]) == (mj.MJ_ERR_INVALID_ARG, 2)
    sl = w.seq_lens.copy()
    sl[4] = w.max_blocks * 16 + 1
    assert mj.check_preconditions(p, w.block_table, sl, *ok[2:]) == (mj.MJ_ERR_INVALID_ARG, 4)
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        kd = w.k_descale.copy()
        kd[1, 1] = bad
        assert mj.check_preconditions(p, w.block_table, w.seq_lens, w.q_descale, kd, w.v_descale) == (
            mj.MJ_ERR_INVALID_ARG,
            1,
        )
    # arrays of the wrong shape are refused before the checker reads them
    with pytest.raises(ValueError):
        mj.check_preconditions(p, w.block_table[:, :-1], *ok[1:])
    with pytest.raises(ValueError):
        mj.check_preconditions(p, w.block_table[:-1], *ok[1:])
    with pytest.raises(ValueError):
        mj.check_preconditions(p, w.block_table, w.seq_lens[:-1], *ok[2:])
    with pytest.raises(ValueError):
        mj.check_preconditions(p, w.block_table, w.seq_lens, w.q_descale, np.ones(3), w.v_descale)
    # per-tensor and per-head descales broadcast
    assert mj.check_preconditions(p, w.block_table, w.seq_lens, np.ones(1), np.ones(2), np.ones(2))[0] == mj.MJ_OK


def test_bounded_wait_hook_validation():
    L = mj.lib()
    fake = 1 << 20
    assert L.mj_check_bounded_wait(None, None, 1000, None) == mj.MJ_ERR_INVALID_ARG
    assert L.mj_check_bounded_wait(fake + 2, None, 1000, None) == mj.MJ_ERR_INVALID_ARG
    assert L.mj_check_bounded_wait(fake, fake + 4, 1000, None) == mj.MJ_ERR_INVALID_ARG
    for bad in (0, -5, 1000001):
        assert L.mj_check_bounded_wait(fake, None, bad, None) == mj.MJ_ERR_INVALID_ARG


def test_verbose_switch_prints_the_plan_and_nothing_without_it():
    import subprocess
    import sys

    code = (
        "import paged_fp8_kv_gb300 as mj\n"
        "p = mj.make_params(8, 1, 1, 16, 128, 1024, 2000, True, mj.MJ_E4M3, 256)\n"
        "mj.decode_plan(p, [131072] + [1024] * 7)\n"
    )
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, MJ_VERBOSE="1", PYTHONPATH=root)
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    line = [l for l in out.stderr.splitlines() if l.startswith("mj_decode_plan: SplitPlan(")]
    assert len(line) == 1, out.stderr
    for field in ("kernel=tc_r16_e4m3", "num_seqs=8", "chunk_tiles=4", "max_n_splits=256", "split_seqs=8"):
        assert field in line[0], line[0]
    env["MJ_VERBOSE"] = "0"
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    assert "SplitPlan" not in out.stderr


def test_narrow_kv_format_validation():
    p = _params(1, h_r=4, max_splits=16)
    p.kv_format = 5
    assert _attn_status(p, _good_args()) == mj.MJ_ERR_INVALID_ARG
    for kernel in (mj.MJ_KERNEL_CUDA_CORE, mj.MJ_KERNEL_TENSOR_CORE_GROUPED):
        q = _params(1, h_k=8, h_r=4, max_splits=16, kernel=kernel)
        q.kv_format = mj.MJ_KV_E2M1
        buf = ctypes.create_string_buffer(64)
        assert mj.lib().mj_kernel_name(ctypes.byref(q), buf, 64) == mj.MJ_ERR_UNSUPPORTED
    q = _params(1, h_r=4, max_splits=16)
    q.kv_format = mj.MJ_KV_E3M2
    buf = ctypes.create_string_buffer(64)
    assert mj.lib().mj_kernel_name(ctypes.byref(q), buf, 64) == mj.MJ_OK
    assert buf.value.decode().endswith("_kve3m2")
    # packed pools: 32-byte aligned bases and strides (16 is not enough)
    for field, val in (("k_row", 48), ("v_page", 16 * 96 + 16), ("k", (1 << 20) + 16)):
        a = _good_args()
        a.k_page, a.k_row, a.k_head = 16 * 64, 64, 64
        a.v_page, a.v_row, a.v_head = 16 * 64, 64, 64
        a.workspace = 1 << 20
        a.workspace_bytes = mj.workspace_bytes(q)
        setattr(a, field, val)
        assert _attn_status(q, a) == mj.MJ_ERR_INVALID_ARG, field


def test_nvfp4_validation():
    # e4m3 Q and at most 32 rows on the swap-AB kernel; scale planes needed
    buf = ctypes.create_string_buffer(64)
    for q_dtype, h_r, kernel, want in ((mj.MJ_BF16, 16, 0, mj.MJ_ERR_UNSUPPORTED), (mj.MJ_E4M3, 64, 0, mj.MJ_ERR_UNSUPPORTED),
                                       (mj.MJ_E4M3, 16, mj.MJ_KERNEL_TENSOR_CORE_QROWS, mj.MJ_ERR_UNSUPPORTED),
                                       (mj.MJ_E4M3, 16, 0, mj.MJ_OK), (mj.MJ_E4M3, 32, 0, mj.MJ_OK)):
        q = _params(1, h_r=h_r, max_splits=16, q_dtype=q_dtype, kernel=kernel)
        q.kv_format = mj.MJ_KV_NVFP4
        assert mj.lib().mj_kernel_name(ctypes.byref(q), buf, 64) == want, (q_dtype, h_r, kernel)
        if want == mj.MJ_OK:
            assert buf.value.decode().startswith("tc_") and buf.value.decode().endswith("_kvnvfp4")
    q = _params(1, h_r=16, max_splits=16, q_dtype=mj.MJ_E4M3)
    q.kv_format = mj.MJ_KV_NVFP4
    fake = 1 << 20
    for field, val in (("k_scales", None), ("v_scales", fake + 8), ("ks_head", 8), ("vs_page", 0)):
        a = _good_args()
        a.k_page, a.k_row, a.k_head = 16 * 64, 64, 64
        a.v_page, a.v_row, a.v_head = 16 * 64, 64, 64
        a.k_scales, a.v_scales = fake, fake
        a.ks_page, a.ks_head, a.vs_page, a.vs_head = 16 * 8, 16 * 8, 16 * 8, 16 * 8
        a.workspace = 1 << 20
        a.workspace_bytes = mj.workspace_bytes(q)
        setattr(a, field, val)
        assert _attn_status(q, a) == mj.MJ_ERR_INVALID_ARG, field
