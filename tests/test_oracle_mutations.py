"""Planted mistakes in copies of the oracle's Q quantisation and narrow-format
modules: each plausible slip (a tie rule, a saturation bound, a bias, a
subnormal step, a sign bit, a packing shift, an index order, a reduction
axis) must make one of the pins of tests/test_quant_ref.py or
tests/test_narrow_ref.py fail; the shipped modules pass them.  CPU only;
the mutated copies live in a temporary directory."""

import importlib.util
import os
import sys

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE_DIR = os.path.dirname(os.path.abspath(oracle.__file__))


def load(path, name, tmp_path, old=None, new=None):
    src = open(path).read()
    if old is not None:
        assert old in src, f"mutation anchor missing: {old!r}"
        src = src.replace(old, new, 1)
    src = src.replace("from .layout_ref import", "from oracle.layout_ref import")
    src = src.replace("from .quant_ref import", "from oracle.quant_ref import")
    src = src.replace("from . import", "from oracle import")
    f = tmp_path / f"{name}.py"
    f.write_text(src)
    spec = importlib.util.spec_from_file_location(name, str(f))
    mod = importlib.util.module_from_spec(spec)
    sys.modules[name] = mod  # dataclasses look their module up there
    try:
        spec.loader.exec_module(mod)
    finally:
        del sys.modules[name]
    return mod


# ------------------------------------------------------- Q quantisation


def pins_hold(all_pins, m) -> bool:
    """The pin files' own checks, run against module m (a mutant may divide
    by zero or overflow: numpy's warnings about that are expected here)."""
    try:
        with np.errstate(all="ignore"):
            all_pins(m)
        return True
    except Exception:
        return False


def quant_pins_hold(m) -> bool:
    from tests.test_quant_ref import all_pins

    return pins_hold(all_pins, m)


QUANT_MUTATIONS = [
    ("ties away from zero", "(frac > 0.5 or (frac == 0.5 and int(lo) % 2 == 1))", "(frac >= 0.5)"),
    ("saturates to NaN", "res[i] = sign | 0x7E  # saturate", "res[i] = sign | 0x7F  # saturate"),
    ("wrong largest value", "E4M3_MAX = 448.0", "E4M3_MAX = 240.0"),
    ("subnormal step", "step = 2.0**-9", "step = 2.0**-10"),
    ("sign bit dropped", "res[i] = sign | _code_of_magnitude(mag)", "res[i] = _code_of_magnitude(mag)"),
    ("amax over tokens only", "axis=(1, 3, 4)", "axis=(1, 4)"),
    ("no amax floor", "amax = np.maximum(amax, AMAX_FLOOR)", "amax = amax"),
    ("pack order", "return pack_q_ref(codes, num_seqs, q_len, h_k, h_r), descale", "return pack_q_ref(codes, num_seqs, q_len, h_r, h_k), descale"),
    ("exponent off by one", "step = 2.0 ** (e - 3)", "step = 2.0 ** (e - 2)"),
]


def test_quant_module_passes_its_pins(tmp_path):
    assert quant_pins_hold(load(os.path.join(ORACLE_DIR, "quant_ref.py"), "quant_ok", tmp_path))


@pytest.mark.parametrize("label,old,new", QUANT_MUTATIONS, ids=[m[0] for m in QUANT_MUTATIONS])
def test_quant_planted_mistake_is_caught(label, old, new, tmp_path):
    m = load(os.path.join(ORACLE_DIR, "quant_ref.py"), "quant_mut", tmp_path, old, new)
    assert not quant_pins_hold(m), f"no pin caught: {label}"


# ---------------------------------------------------------- narrow formats


def narrow_pins_hold(m) -> bool:
    from tests.test_narrow_ref import all_pins

    return pins_hold(all_pins, m)


NARROW_MUTATIONS = [
    ("e2m3 bias", '"e2m3": (2, 3, 1)', '"e2m3": (2, 3, 2)'),
    ("subnormal binade", "mag = (m / (1 << mb)) * 2.0 ** (1 - bias)", "mag = (m / (1 << mb)) * 2.0 ** (-bias)"),
    ("tie to the larger", "if best_dist is None or dist < best_dist:", "if best_dist is None or dist <= best_dist:"),
    ("negative zero", "(half if (v < 0 and table[best] != 0) else 0)", "(half if v < 0 else 0)"),
    ("bit order within a byte", "out[:, j // 8] |= ((flat[:, i] >> k) & 1) << (j % 8)", "out[:, j // 8] |= ((flat[:, i] >> k) & 1) << (7 - j % 8)"),
    ("bit order within a code", "out[:, j // 8] |= ((flat[:, i] >> k) & 1) << (j % 8)", "out[:, j // 8] |= ((flat[:, i] >> (bits - 1 - k)) & 1) << (j % 8)"),
    ("unpack reads the wrong byte", "out[:, i] |= ((flat[:, j // 8] >> (j % 8)) & 1) << k", "out[:, i] |= ((flat[:, (j // 8) ^ 1] >> (j % 8)) & 1) << k"),
    ("mantissa width", '"e3m2": (3, 2, 3)', '"e3m2": (2, 3, 3)'),
    ("sign of the search", "dist = abs(abs(v) - table[c])", "dist = abs(v - table[c])"),
    ("nvfp4 shift", "NVFP4_SHIFT = 2.0**-3", "NVFP4_SHIFT = 2.0**-2"),
    ("nvfp4 group of 8", "NVFP4_GROUP = 16  #", "NVFP4_GROUP = 8  #"),
    ("nvfp4 scale code as value", "e2m1[c] * e4[sc] * NVFP4_SHIFT", "e2m1[c] * sc * NVFP4_SHIFT"),
]


def test_narrow_module_passes_its_pins(tmp_path):
    assert narrow_pins_hold(load(os.path.join(ORACLE_DIR, "narrow_ref.py"), "narrow_ok", tmp_path))


@pytest.mark.parametrize("label,old,new", NARROW_MUTATIONS, ids=[m[0] for m in NARROW_MUTATIONS])
def test_narrow_planted_mistake_is_caught(label, old, new, tmp_path):
    m = load(os.path.join(ORACLE_DIR, "narrow_ref.py"), "narrow_mut", tmp_path, old, new)
    assert not narrow_pins_hold(m), f"no pin caught: {label}"


# ------------------------------------------------------------- row layout


def layout_pins_hold(m) -> bool:
    from tests.test_layout_ref import all_pins

    return pins_hold(all_pins, m)


LAYOUT_MUTATIONS = [
    ("unpack: token and head axes kept", "o_packed.reshape(num_seqs, h_k, q_len, h_r, d).transpose(0, 2, 1, 3, 4)", "o_packed.reshape(num_seqs, h_k, q_len, h_r, d).transpose(0, 1, 2, 3, 4)"),
    ("unpack: rows read head-major", "o_packed.reshape(num_seqs, h_k, q_len, h_r, d)", "o_packed.reshape(num_seqs, h_k, h_r, q_len, d)"),
    ("unpack: kv and query heads swapped", ".reshape(num_seqs * q_len, h_k * h_r, d)", ".transpose(0, 1, 3, 2, 4).reshape(num_seqs * q_len, h_k * h_r, d)"),
    ("pack: rows written head-major", "q_vllm.reshape(num_seqs, q_len, h_k, h_r, d).transpose(0, 2, 1, 3, 4)", "q_vllm.reshape(num_seqs, q_len, h_k, h_r, d).transpose(0, 2, 3, 1, 4)"),
]


def test_layout_module_passes_its_pins(tmp_path):
    assert layout_pins_hold(load(os.path.join(ORACLE_DIR, "layout_ref.py"), "layout_ok", tmp_path))


@pytest.mark.parametrize("label,old,new", LAYOUT_MUTATIONS, ids=[m[0] for m in LAYOUT_MUTATIONS])
def test_layout_planted_mistake_is_caught(label, old, new, tmp_path):
    m = load(os.path.join(ORACLE_DIR, "layout_ref.py"), "layout_mut", tmp_path, old, new)
    assert not layout_pins_hold(m), f"no pin caught: {label}"


# ------------------------------------------------------------------- plan


def plan_pins_hold(m) -> bool:
    from tests.test_plan_ref import all_pins

    return pins_hold(all_pins, m)


PLAN_MUTATIONS = [
    ("tile of 64 rows", "TILE_ROWS = 128", "TILE_ROWS = 64"),
    ("empty sequence owns no tile", "return max(1, whole + (1 if rest else 0))", "return whole + (1 if rest else 0)"),
    ("slots ignore the q tiles", "slots = max(1, (sm_count * ctas_per_sm) // (h_k * n_q_tiles))", "slots = max(1, (sm_count * ctas_per_sm) // h_k)"),
    ("no max_splits floor", "while _pieces(longest, floor_chunk) > max_splits:", "while False:"),
    ("a full wave does not fit", "while chunk < longest and sum(_pieces(t, chunk) for t in tiles) > slots:", "while chunk < longest and sum(_pieces(t, chunk) for t in tiles) >= slots:"),
    ("largest fitting chunk", "while chunk < longest and sum(_pieces(t, chunk) for t in tiles) > slots:", "while chunk < longest and sum(_pieces(t, chunk + 1) for t in tiles) <= slots:"),
    ("shortest first", "items.sort(key=lambda it: (-(it[2] - it[1]), it[0], it[3]))", "items.sort(key=lambda it: (it[2] - it[1], it[0], it[3]))"),
    ("ties by last sequence", "items.sort(key=lambda it: (-(it[2] - it[1]), it[0], it[3]))", "items.sort(key=lambda it: (-(it[2] - it[1]), -it[0], it[3]))"),
    ("force ignores the floor", "        chunk = floor_chunk\n        while _pieces(longest, chunk) > force_splits:", "        chunk = 1\n        while _pieces(longest, chunk) > force_splits:"),
]


def test_plan_module_passes_its_pins(tmp_path):
    assert plan_pins_hold(load(os.path.join(ORACLE_DIR, "plan_ref.py"), "plan_ok", tmp_path))


@pytest.mark.parametrize("label,old,new", PLAN_MUTATIONS, ids=[m[0] for m in PLAN_MUTATIONS])
def test_plan_planted_mistake_is_caught(label, old, new, tmp_path):
    m = load(os.path.join(ORACLE_DIR, "plan_ref.py"), "plan_mut", tmp_path, old, new)
    assert not plan_pins_hold(m), f"no pin caught: {label}"
