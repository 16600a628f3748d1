"""CPU checks of the benchmark's bookkeeping: the algorithmic bytes and flops
of a step (worked by hand for the tiny reference workload) and the rule
that a recorded DRAM traffic figure is reported only for the kernel source
it was measured on."""

import hashlib
import json
import os

import pytest

import bench
import paged_fp8_kv_gb300 as mj
from paged_fp8_kv_gb300 import synthetic as syn


def tiny_plan(w):
    p = mj.make_params(
        w.num_seqs, w.q_len, w.h_k, w.h_r, w.page_size, w.max_blocks, w.num_pages, bool(w.causal),
        mj.MJ_BF16, w.max_splits, w.head_dim, 0, 0,
    )
    return mj.decode_plan(p, w.seq_lens, sm_count=152)


def test_algorithmic_bytes_by_hand():
    # tiny reference: 2 sequences of 37 and 100 keys, 1 kv head, 8 rows,
    # d = 128, pages of 16 rows, bf16 Q, nothing split
    w = syn.config(1)
    plan = tiny_plan(w)
    decode, merge, step = bench.algorithmic_bytes(w, plan)
    kv = (37 + 100) * 1 * 128 * 2  # K and V, one byte each
    q = o = 2 * 1 * 8 * 128 * 2  # bf16 Q in, bf16 O out
    lse = 2 * 1 * 8 * 4
    block_table = (3 + 7) * 4  # ceil(37 / 16) + ceil(100 / 16) entries
    meta = plan.num_work * 16 + 2 * 8 + 3 * 2 * 1 * 4  # work items, n_splits + seq_lens, 3 descales
    assert plan.num_work == 2
    assert decode == kv + q + o + lse + block_table + meta
    assert merge == 0
    assert step == decode


def test_narrow_kv_bytes_by_hand():
    # the same tiny problem with packed pools: fp4 rows of 64 bytes, fp6 rows
    # of 96, nvfp4 rows of 64 bytes of codes and 8 of scales
    for fmt, row in (("e2m1", 64), ("e3m2", 96), ("nvfp4", 72)):
        w = syn.make_workload("tiny_narrow", [37, 100], 1, 1, 8, 16, seed=1112, random_descales=False,
                              max_splits=1, num_pages=16, kv_format=fmt)
        plan = tiny_plan(w)
        decode, _, _ = bench.algorithmic_bytes(w, plan)
        fixed = 2 * (2 * 1 * 8 * 128 * 2) + 2 * 1 * 8 * 4 + (3 + 7) * 4 + plan.num_work * 16 + 2 * 8 + 3 * 2 * 1 * 4
        assert decode == (37 + 100) * 1 * row * 2 + fixed, fmt


def test_algorithmic_flops_by_hand():
    # every visible (key, row) pair costs 2 d for S and 2 d for O
    w = syn.config(1)
    assert bench.algorithmic_flops(w) == 4 * 128 * 8 * (37 + 100)
    # causal tail with 4 query tokens: token qi sees L - 4 + qi + 1 keys
    w4 = syn.config(4, num_seqs=2, len_range=(10, 20))
    vis = sum(sum(int(L) - 4 + qi + 1 for qi in range(4)) for L in w4.seq_lens)
    assert bench.algorithmic_flops(w4) == 4 * 128 * w4.h_k * w4.h_r * vis


def test_traffic_record_follows_the_source(tmp_path, monkeypatch):
    src = "pack.cu"
    path = os.path.join(bench.ROOT, "paged_fp8_kv_gb300", "csrc", src)
    sha = hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]
    rec = {
        "k_current": {"wl": {"source": src, "source_sha": sha, "dram_bytes_per_launch": 12345}},
        "k_stale": {"wl": {"source": src, "source_sha": "0" * 16, "dram_bytes_per_launch": 999}},
    }
    (tmp_path / "traffic.json").write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "PROFILES", str(tmp_path))
    assert bench.traffic_record("k_current", "wl") == 12345
    assert bench.traffic_record("k_stale", "wl") is None
    assert bench.traffic_record("k_current", "other") is None
    assert bench.traffic_record("unknown", "wl") is None


@pytest.mark.parametrize("name", ["tc_r8_bf16", "qm_pair_bf16", "qm_r32_bf16", "qm_r64_bf16", "tc_r16_e4m3"])
def test_committed_traffic_records_name_existing_sources(name):
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for wl, e in rec[name].items():
        assert os.path.exists(os.path.join(bench.ROOT, "paged_fp8_kv_gb300", "csrc", e["source"]))
        assert e["dram_bytes_per_launch"] > 0 and len(e["source_sha"]) == 16
        assert "ncu" in e["command"] and "--clock-control none" in e["command"]


def test_committed_traffic_records_point_at_their_kernels_source():
    """A record is invalidated by its source's hash: it must name the file
    that holds the kernel it was taken on (the library's kernel names start
    with the kernel family), and its capture must select that kernel."""
    rec = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    family = {"tcg": "decode_tcg.cu", "tc": "decode_tc.cu", "qm": "decode_qm.cu", "cc": "decode_cc.cu"}
    n = 0
    for kernel, per_wl in rec.items():
        if not isinstance(per_wl, dict):
            continue
        for wl, e in per_wl.items():
            if not (isinstance(e, dict) and "source" in e):
                continue
            src = family[kernel.split("_")[0]]
            assert e["source"] == src, (kernel, wl, e["source"])
            assert "regex:" + src[:-3] in e["command"], (kernel, wl)
            n += 1
    assert n >= 10


def test_cold_copies_put_twice_l2_between_reuses():
    """The timed loop's rotation: at least 2 x L2 of other inputs between two
    uses of one copy, else (over 16 copies) an L2 flush."""
    import bench

    l2 = 126 << 20
    for d in (1_343_200_000, 620_000_000, 260_000_000, 44_000_000, 35_000_000, 18_000_000):
        k = bench.cold_copies(d, l2)
        assert 2 <= k <= bench.COLD_MAX_COPIES
        assert (k - 1) * d >= 2 * l2
        assert (k - 2) * d < 2 * l2  # the fewest copies that do it
    assert bench.cold_copies(35_000, l2) == 1  # the tiny workload flushes
    assert bench.cold_copies(2 * l2 // 16, l2) == 1


def test_traffic_only_for_the_captured_configuration():
    """Shrunk batches or changed load options must not borrow the full
    workload's ncu traffic figure."""
    import bench

    sys_argv = ["bench.py"]
    import sys as _sys

    old = _sys.argv
    try:
        _sys.argv = sys_argv
        assert bench.traffic_applies(bench.parse())
        for extra in (["--num_seqs", "32"], ["--kv_layout", "hnd"], ["--ctas_per_sm", "2"], ["--max_splits", "8"]):
            _sys.argv = sys_argv + extra
            assert not bench.traffic_applies(bench.parse())
    finally:
        _sys.argv = old
