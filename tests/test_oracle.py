"""Pins of the fp64 oracle to facts the source pages and mathematics fix.

Each test checks the oracle against something other than itself:

* the e4m3 table against torch's float8_e4m3fn decoding (a library routine)
  and against the special codes the pages name (448, NaN = 0x7F);
* bf16 decoding against torch's bfloat16;
* closed forms: one visible key, identical keys, one-hot dominance;
* the causal tail by brute-force enumeration and by its equivalence with a
  truncated sequence;
* a Decimal (50-digit) log-sum-exp and output on tiny inputs;
* split-then-merge against the direct sum for random chunkings;
* invariances: page permutation, poison in unread memory, exact power-of-two
  rescaling of the descales;
* degenerate rows (no visible key) giving O = 0 and LSE = -inf;
* mutation checks: plausible mistakes planted in a COPY of the oracle source
  (dropped term, wrong index, swapped operand) each fail one of these pins.

Sources: the "mjolnir/t5_decode.py" page (module docstring on causal tail and
LSE; `emulate_decode`; the kernel epilogue's empty-row rule; the harness'
poisoning of unused pages with 0x7F).
"""

import copy
import ctypes
import json
import math
import os
import shutil
import subprocess
import tempfile
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import oracle
from paged_fp8_kv_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------- helpers


def tiny(seq_lens, q_len=1, h_k=1, h_r=2, page_size=16, seed=5, causal=True, q_is_e4m3=False, **kw):
    return syn.make_workload(
        "tiny", seq_lens, q_len, h_k, h_r, page_size, seed=seed, causal=causal, q_is_e4m3=q_is_e4m3, **kw
    )


def kv_row(w, cache, b, j, g):
    page = w.block_table[b, j // w.page_size]
    return cache[page, j % w.page_size, g]


def set_kv_row(w, cache, b, j, g, codes):
    page = w.block_table[b, j // w.page_size]
    cache[page, j % w.page_size, g] = codes


def e4m3(x):
    """e4m3 code of one value."""
    return syn.e4m3_encode(np.array([x], dtype=np.float32))[0]


def bf16(x):
    """bf16 bits of one value."""
    return syn.bf16_encode(np.array([x], dtype=np.float32))[0]


# ------------------------------------------------------------ format pins


def test_e4m3_table_matches_torch():
    ours = oracle.e4m3_table()
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32).double().numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))
    assert set(np.flatnonzero(np.isnan(ours)).tolist()) == {0x7F, 0xFF}
    # signed zeros decode with their sign
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_e4m3_golden_codes():
    g = json.load(open(os.path.join(GOLDEN, "e4m3_codes.json")))
    for code_s, val in g["codes"].items():
        got = oracle.e4m3_value(int(code_s, 16))
        if val == "nan":
            assert math.isnan(got), code_s
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), code_s


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    ours = np.array([oracle.bf16_value(int(b)) for b in bits])
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))


# --------------------------------------------------------- closed forms


def test_single_key_gives_v_and_logit():
    w = tiny([1], h_r=1, seed=11)
    # q = e_5 (bf16 1.0), k[5] = 1.5, kd = 2, scale = 0.5  ->  z = 1.5
    q = np.zeros_like(w.q)
    q[0, 0, 5] = bf16(1.0)
    w.q = q
    k = np.zeros(128, dtype=np.uint8)
    k[5] = e4m3(1.5)
    set_kv_row(w, w.k_cache, 0, 0, 0, k)
    w.k_descale[:] = 2.0
    w.v_descale[:] = 0.75
    w.softmax_scale = 0.5
    w.scale_o = 3.0
    o, lse = oracle.attention(w)
    v0 = oracle.e4m3_table()[kv_row(w, w.v_cache, 0, 0, 0)]
    np.testing.assert_array_equal(o[0, 0, 0], 3.0 * 0.75 * v0)
    assert lse[0, 0, 0] == 1.5


def test_identical_keys_give_mean_v():
    L = 37
    w = tiny([L], h_r=2, seed=12)
    k0 = kv_row(w, w.k_cache, 0, 0, 0).copy()
    for j in range(L):
        set_kv_row(w, w.k_cache, 0, j, 0, k0)
    o, lse = oracle.attention(w)
    tab = oracle.e4m3_table()
    V = np.stack([tab[kv_row(w, w.v_cache, 0, j, 0)] for j in range(L)])
    vd = float(w.v_descale[0, 0])
    # causal with q_len = 1: every row sees all L keys
    for n in range(2):
        np.testing.assert_allclose(o[0, 0, n], vd * V.mean(axis=0), rtol=1e-13, atol=1e-13)
        # single key LSE + ln L
        o1, lse1 = oracle.attention(_truncated(w, 1))
        assert abs(lse[0, 0, n] - (lse1[0, 0, n] + math.log(L))) < 1e-12


def _truncated(w, L):
    w2 = copy.deepcopy(w)
    w2.seq_lens = np.array([L] + list(w.seq_lens[1:]), dtype=np.int32)
    return w2


def test_one_hot_dominance_returns_that_value_row():
    L = 50
    w = tiny([L], h_r=1, seed=13)
    target = 17
    q = np.zeros_like(w.q)
    q[0, 0, 0] = bf16(64.0)
    w.q = q
    for j in range(L):
        k = np.zeros(128, dtype=np.uint8)
        k[0] = e4m3(448.0 if j == target else 1.0)
        set_kv_row(w, w.k_cache, 0, j, 0, k)
    w.k_descale[:] = 1.0
    w.softmax_scale = 1.0
    o, lse = oracle.attention(w)
    tab = oracle.e4m3_table()
    v_t = tab[kv_row(w, w.v_cache, 0, target, 0)] * w.v_descale[0, 0]
    # other keys are suppressed by exp(-64 * 447)
    np.testing.assert_array_equal(o[0, 0, 0], v_t)
    assert lse[0, 0, 0] == 64.0 * 448.0


# ------------------------------------------------------------ causal tail


def test_causal_tail_brute_force():
    # q_len = 4: token qi sees keys 0 .. L - 4 + qi
    L, q_len, h_r = 23, 4, 2
    w = tiny([L], q_len=q_len, h_r=h_r, seed=14)
    base_o, base_lse = oracle.attention(w)
    for j in range(L):
        w2 = copy.deepcopy(w)
        row = kv_row(w2, w2.k_cache, 0, j, 0).copy()
        row[:] = e4m3(3.0)
        set_kv_row(w2, w2.k_cache, 0, j, 0, row)
        o2, lse2 = oracle.attention(w2)
        for n in range(q_len * h_r):
            qi = n // h_r
            sees = j <= L - q_len + qi
            changed = lse2[0, 0, n] != base_lse[0, 0, n]
            assert changed == sees, (j, n)


def test_causal_tail_equals_truncated_sequence():
    L, q_len, h_r = 40, 3, 2
    w = tiny([L], q_len=q_len, h_r=h_r, seed=15)
    o, lse = oracle.attention(w)
    for qi in range(q_len):
        # a q_len = 1 problem over the first L - q_len + qi + 1 keys, with
        # token qi's queries
        w1 = copy.deepcopy(w)
        w1.q_len = 1
        w1.q = np.ascontiguousarray(w.q[qi : qi + 1])
        w1.seq_lens = np.array([L - q_len + qi + 1], dtype=np.int32)
        o1, lse1 = oracle.attention(w1)
        for hr in range(h_r):
            n = qi * h_r + hr
            np.testing.assert_array_equal(o[0, 0, n], o1[0, 0, hr])
            assert lse[0, 0, n] == lse1[0, 0, hr]


def test_noncausal_rows_see_everything():
    L, q_len, h_r = 33, 5, 2
    w = tiny([L], q_len=q_len, h_r=h_r, seed=16, causal=False)
    o, lse = oracle.attention(w)
    wc = copy.deepcopy(w)
    wc.causal = True
    oc, lsec = oracle.attention(wc)
    last = slice((q_len - 1) * h_r, q_len * h_r)  # the last token is unaffected by causality
    np.testing.assert_array_equal(o[0, 0, last], oc[0, 0, last])
    assert not np.array_equal(o[0, 0, :h_r], oc[0, 0, :h_r])


def test_rows_without_keys_are_zero_and_minus_inf():
    # L = 0 and L < q_len (causal): no visible key
    w = tiny([0, 2], q_len=4, h_r=2, seed=17)
    o, lse = oracle.attention(w)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(lse[0]))
    # seq 1 (L = 2): token qi sees keys 0 .. qi - 2 -> tokens 0 and 1 see nothing
    assert np.all(o[1, 0, :4] == 0.0) and np.all(np.isneginf(lse[1, 0, :4]))
    assert np.all(np.isfinite(lse[1, 0, 4:]))


# ------------------------------------------------------- exact arithmetic


def _decimal_row(w, b, g, n):
    getcontext().prec = 50
    tab = oracle.e4m3_table()
    d = w.head_dim
    qi, hr = divmod(n, w.h_r)
    h = g * w.h_r + hr
    if w.q_is_e4m3:
        qv = [Decimal(float(tab[c])) for c in w.q[b * w.q_len + qi, h]]
    else:
        qv = [Decimal(float(x)) for x in syn.bf16_bits_to_float(w.q[b * w.q_len + qi, h])]
    L = int(w.seq_lens[b])
    lim = min(L - 1, L - w.q_len + qi) if w.causal else L - 1
    scale = Decimal(w.softmax_scale) * Decimal(float(w.q_descale[b, g])) * Decimal(float(w.k_descale[b, g]))
    zs, vs = [], []
    for j in range(lim + 1):
        kr = kv_row(w, w.k_cache, b, j, g)
        dot = sum(qv[i] * Decimal(float(tab[kr[i]])) for i in range(d))
        zs.append(scale * dot)
        vs.append([Decimal(float(tab[c])) for c in kv_row(w, w.v_cache, b, j, g)])
    ez = [z.exp() for z in zs]
    tot = sum(ez)
    lse = tot.ln()
    out = Decimal(w.scale_o) * Decimal(float(w.v_descale[b, g]))
    o = [out * sum(e * v[i] for e, v in zip(ez, vs)) / tot for i in range(d)]
    return [float(x) for x in o], float(lse)


@pytest.mark.parametrize("q_is_e4m3", [False, True])
def test_decimal_logsumexp_tiny(q_is_e4m3):
    w = tiny([13, 40], q_len=2, h_k=2, h_r=2, seed=18, q_is_e4m3=q_is_e4m3)
    o, lse = oracle.attention(w)
    for b, g, n in [(0, 0, 0), (0, 1, 3), (1, 0, 2), (1, 1, 1)]:
        od, lsed = _decimal_row(w, b, g, n)
        assert abs(lse[b, g, n] - lsed) <= 1e-12 * max(1.0, abs(lsed))
        np.testing.assert_allclose(o[b, g, n], od, rtol=1e-11, atol=1e-12)


# ------------------------------------------------------------ split/merge


def test_split_then_merge_equals_direct():
    rng = np.random.default_rng(19)
    w = tiny([700], q_len=2, h_r=2, seed=19)
    o, lse = oracle.attention(w)
    out_scale = w.scale_o * float(w.v_descale[0, 0])
    for trial in range(5):
        cuts = sorted(set(rng.integers(1, 700, size=rng.integers(1, 8)).tolist()))
        bounds = [0] + cuts + [700]
        for n in range(4):
            parts = [oracle.partial(w, 0, 0, n, a, c) for a, c in zip(bounds[:-1], bounds[1:])]
            om, lm = oracle.merge([p[0] for p in parts], [p[1] for p in parts], np.stack([p[2] for p in parts]), out_scale)
            np.testing.assert_allclose(om, o[0, 0, n], rtol=1e-12, atol=1e-14)
            assert abs(lm - lse[0, 0, n]) <= 1e-12 * max(1, abs(lse[0, 0, n]))


def test_merge_of_empty_parts():
    o, lse = oracle.merge([-math.inf, -math.inf], [0.0, 0.0], np.zeros((2, 4)), 1.0)
    assert np.all(o == 0) and lse == -math.inf


# ------------------------------------------------------------ invariances


def test_page_permutation_invariance():
    w = tiny([100, 61], h_k=2, h_r=2, seed=20)
    o, lse = oracle.attention(w)
    perm = np.random.default_rng(20).permutation(w.num_pages)
    inv = np.argsort(perm)
    w2 = copy.deepcopy(w)
    w2.k_cache = np.ascontiguousarray(w.k_cache[perm])  # new page p holds old page perm[p]
    w2.v_cache = np.ascontiguousarray(w.v_cache[perm])
    used = w.block_table.copy()
    for b, L in enumerate(w.seq_lens):
        npg = -(-int(L) // w.page_size)
        w2.block_table[b, :npg] = inv[used[b, :npg]]
    o2, lse2 = oracle.attention(w2)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_poison_is_never_read():
    w = tiny([70, 33], h_r=2, seed=21)
    o, lse = oracle.attention(w)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    w2 = copy.deepcopy(w)
    owned = set()
    for b, L in enumerate(w.seq_lens):
        owned |= set(w.block_table[b, : -(-int(L) // w.page_size)].tolist())
    for p in range(w.num_pages):
        if p not in owned:
            w2.k_cache[p] = 0x42
            w2.v_cache[p] = 0x11
    o2, lse2 = oracle.attention(w2)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_power_of_two_descale_rescaling_is_exact():
    w = tiny([90], h_k=1, h_r=4, seed=22)
    o, lse = oracle.attention(w)
    w2 = copy.deepcopy(w)
    w2.k_descale = w.k_descale * 2.0
    w2.softmax_scale = w.softmax_scale / 2.0
    w2.v_descale = w.v_descale * 4.0
    w2.scale_o = w.scale_o / 4.0
    o2, lse2 = oracle.attention(w2)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_units_subset_matches_full():
    w = tiny([90, 20, 55], h_k=2, h_r=2, seed=23)
    o, lse = oracle.attention(w)
    units = [(2, 1), (0, 0), (1, 1)]
    ou, lu = oracle.attention(w, units=units, threads=2)
    for i, (b, g) in enumerate(units):
        np.testing.assert_array_equal(ou[i], o[b, g])
        np.testing.assert_array_equal(lu[i], lse[b, g])


# ---------------------------------------------------- planted mistakes


MUTATIONS = [
    ("row within page", "j % p->page_size", "(j + 1) % p->page_size"),
    ("page of a key", "j / p->page_size]", "(j / p->page_size) / 2]"),
    ("max shift dropped from weights", "std::exp(z[j - j0] - m)", "std::exp(z[j - j0] - m * 0.5)"),
    ("k descale dropped", "qd_at(b, g) * kd_at(b, g) * dot", "qd_at(b, g) * dot"),
    ("v read as k", "return kE4M3.v[v[row_off(b, j, g, p->v_page", "return kE4M3.v[k[row_off(b, j, g, p->v_page"),
    ("causal off by one", "L - p->q_len + qi;", "L - p->q_len + qi + 1;"),
    ("e4m3 exponent bias", "e - 7);", "e - 8);"),
    ("log of l dropped", "*lse = m + std::log(l);", "*lse = m;"),
    ("query token index", "const int qi = n / p->h_r;\n    const int h", "const int qi = n % p->q_len;\n    const int h"),
]


def _pins_hold(lib_path):
    """Run a subset of pins against a library built from mutated source."""
    saved = oracle._lib
    try:
        oracle._lib = None
        real_build = oracle.build
        oracle.build = lambda force=False: lib_path
        ok = True
        for fn in (
            test_e4m3_table_matches_torch,
            test_single_key_gives_v_and_logit,
            test_identical_keys_give_mean_v,
            test_causal_tail_brute_force,
            test_causal_tail_equals_truncated_sequence,
            lambda: test_decimal_logsumexp_tiny(False),
            test_split_then_merge_equals_direct,
        ):
            try:
                fn()
            except AssertionError:
                ok = False
                break
        return ok
    finally:
        oracle.build = real_build
        oracle._lib = saved


@pytest.mark.parametrize("label,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(label, old, new, tmp_path):
    src = open(oracle._SRC).read()
    assert old in src, f"mutation anchor missing: {label}"
    mutated = src.replace(old, new, 1)
    cpp = tmp_path / "mut.cpp"
    cpp.write_text(mutated)
    so = str(tmp_path / "libmut.so")
    subprocess.check_call(["g++", "-O1", "-std=c++17", "-shared", "-fPIC", "-pthread", str(cpp), "-o", so])
    assert not _pins_hold(so), f"no pin caught the planted mistake: {label}"
