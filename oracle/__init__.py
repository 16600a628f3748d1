"""fp64 CPU oracle for paged fp8-KV split-KV decode attention.

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this package.  The
CUDA library (``paged_fp8_kv_gb300``) never imports it and shares no code
with it; the only code both sides use is the seeded input generator
``paged_fp8_kv_gb300.synthetic``, which holds none of the method's
arithmetic.

* ``decode_ref.cpp`` - the plain attention definition over a paged cache,
  in fp64, threaded over (sequence, kv head) units (built into
  ``liboracle.so`` by :func:`build`).
* ``plan_ref.py`` - a plain restatement of the occupancy-pinned plan.
* ``layout_ref.py`` - the query / output row permutation.
* ``quant_ref.py`` - the per-(sequence, kv head) fp8 query quantisation
  fused with the pack, with its own e4m3 encoder.
* ``narrow_ref.py`` - the narrow KV formats (fp6 e3m2 / e2m3, fp4 e2m1):
  value tables, the page's quantiser and bit packing, and their exact e4m3
  view for the attention oracle.

Every function here is pinned by ``tests/test_oracle.py`` against facts the
source pages and mathematics fix (see that file's docstring).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

from .plan_ref import PlanRef, plan_ref  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "liboracle.so")
_SRC = os.path.join(_HERE, "decode_ref.cpp")


def build(force: bool = False) -> str:
    """Compile decode_ref.cpp into liboracle.so (plain g++, no CUDA)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", _SRC, "-o", tmp]
        )
        os.replace(tmp, _SO)
    return _SO


class OracleProblem(ctypes.Structure):
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("q_len", ctypes.c_int32),
        ("h_k", ctypes.c_int32),
        ("h_r", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32),
        ("max_blocks", ctypes.c_int32),
        ("causal", ctypes.c_int32),
        ("q_is_e4m3", ctypes.c_int32),
        ("softmax_scale", ctypes.c_double),
        ("scale_o", ctypes.c_double),
        ("q_seq", ctypes.c_int64),
        ("q_tok", ctypes.c_int64),
        ("q_head", ctypes.c_int64),
        ("k_page", ctypes.c_int64),
        ("k_row", ctypes.c_int64),
        ("k_head", ctypes.c_int64),
        ("v_page", ctypes.c_int64),
        ("v_row", ctypes.c_int64),
        ("v_head", ctypes.c_int64),
        ("qd_seq", ctypes.c_int64),
        ("qd_head", ctypes.c_int64),
        ("kd_seq", ctypes.c_int64),
        ("kd_head", ctypes.c_int64),
        ("vd_seq", ctypes.c_int64),
        ("vd_head", ctypes.c_int64),
    ]


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        vp = ctypes.c_void_p
        _lib.oracle_e4m3_value.restype = ctypes.c_double
        _lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        _lib.oracle_bf16_value.restype = ctypes.c_double
        _lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        _lib.oracle_attention.restype = ctypes.c_int
        _lib.oracle_attention.argtypes = [P(OracleProblem)] + [vp] * 8 + [
            vp,
            ctypes.c_int32,
            vp,
            vp,
            ctypes.c_int32,
        ]
        _lib.oracle_partial.restype = ctypes.c_int
        _lib.oracle_partial.argtypes = [P(OracleProblem)] + [vp] * 8 + [
            ctypes.c_int32,
            ctypes.c_int32,
            ctypes.c_int32,
            ctypes.c_int64,
            ctypes.c_int64,
            vp,
            vp,
            vp,
        ]
        _lib.oracle_merge.restype = ctypes.c_int
        _lib.oracle_merge.argtypes = [ctypes.c_int32, ctypes.c_int32, vp, vp, vp, ctypes.c_double, vp, vp]
    return _lib


def e4m3_value(code: int) -> float:
    return lib().oracle_e4m3_value(int(code))


def e4m3_table() -> np.ndarray:
    return np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)


def bf16_value(bits: int) -> float:
    return lib().oracle_bf16_value(int(bits))


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def problem_from(w) -> OracleProblem:
    """OracleProblem for a :class:`paged_fp8_kv_gb300.synthetic.Workload`."""
    p = OracleProblem()
    p.num_seqs, p.q_len, p.h_k, p.h_r = w.num_seqs, w.q_len, w.h_k, w.h_r
    p.head_dim, p.page_size, p.max_blocks = w.head_dim, w.page_size, w.max_blocks
    p.causal, p.q_is_e4m3 = int(w.causal), int(w.q_is_e4m3)
    p.softmax_scale, p.scale_o = float(w.softmax_scale), float(w.scale_o)
    p.q_seq, p.q_tok, p.q_head = w.q_strides
    p.k_page, p.k_row, p.k_head = w.k_strides
    p.v_page, p.v_row, p.v_head = w.v_strides
    p.qd_seq, p.qd_head = w.qd_strides
    p.kd_seq, p.kd_head = w.kd_strides
    p.vd_seq, p.vd_head = w.vd_strides
    return p


def _arrays(w):
    return (w.q, w.k_cache, w.v_cache, w.block_table, w.seq_lens, w.q_descale, w.k_descale, w.v_descale)


def attention(w, units: Optional[Sequence[Sequence[int]]] = None, threads: int = 0):
    """fp64 O (units, n_q, d) and LSE (units, n_q) for a workload.

    ``units`` lists (b, g) pairs; None means every (b, g), b-major, in which
    case the result is shaped (b, h_k, n_q, d) / (b, h_k, n_q)."""
    p = problem_from(w)
    arrs = [np.ascontiguousarray(a) if a.ndim == 0 else a for a in _arrays(w)]
    n_q = w.q_len * w.h_r
    if units is None:
        n_u = w.num_seqs * w.h_k
        u_arr = None
    else:
        u_arr = np.ascontiguousarray(np.asarray(units, dtype=np.int32).reshape(-1, 2))
        n_u = u_arr.shape[0]
    o = np.zeros((n_u, n_q, w.head_dim), dtype=np.float64)
    lse = np.zeros((n_u, n_q), dtype=np.float64)
    rc = lib().oracle_attention(
        ctypes.byref(p),
        *[_ptr(a) for a in arrs],
        None if u_arr is None else _ptr(u_arr),
        n_u,
        _ptr(o),
        _ptr(lse),
        int(threads),
    )
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    if units is None:
        return o.reshape(w.num_seqs, w.h_k, n_q, w.head_dim), lse.reshape(w.num_seqs, w.h_k, n_q)
    return o, lse


def partial(w, b: int, g: int, n: int, j0: int, j1: int):
    """(m, l, acc[d]) of one row over keys [j0, j1), unnormalised."""
    p = problem_from(w)
    m = np.zeros(1)
    l = np.zeros(1)
    acc = np.zeros(w.head_dim)
    rc = lib().oracle_partial(
        ctypes.byref(p), *[_ptr(a) for a in _arrays(w)], b, g, n, j0, j1, _ptr(m), _ptr(l), _ptr(acc)
    )
    if rc != 0:
        raise ValueError("oracle_partial rejected its arguments")
    return float(m[0]), float(l[0]), acc


def merge(ms, ls, accs, out_scale: float):
    """Combine partial statistics into (O[d], LSE)."""
    ms = np.ascontiguousarray(ms, dtype=np.float64)
    ls = np.ascontiguousarray(ls, dtype=np.float64)
    accs = np.ascontiguousarray(accs, dtype=np.float64)
    d = accs.shape[-1]
    o = np.zeros(d)
    lse = np.zeros(1)
    rc = lib().oracle_merge(len(ms), d, _ptr(ms), _ptr(ls), _ptr(accs), float(out_scale), _ptr(o), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_merge rejected its arguments")
    return o, float(lse[0])
