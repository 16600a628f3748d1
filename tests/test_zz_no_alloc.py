"""The allocation-free entry point, mj_decode_attn_static_ws.

Some callers may not allocate device memory when they call into the library
(their runtime reserved the whole device for its own arena, or they live
inside a framework that owns the allocator).  For them the library keeps the
split-KV scratch in a fixed device array and this entry point uses it instead
of a caller workspace.  This test calls it through the C ABI, twice in a row
(the second call finds the array holding the first call's partials and, for
the head-grouped kernel, its unit counter), and checks that both give the
regular entry point's bytes exactly: the same kernels run the same plan, and
the library's results are deterministic.  It also checks that a problem too
large for the array is refused before anything runs.

The file name sorts last so that a run stopping at the first failure has
already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import paged_fp8_kv_gb300 as mj
from paged_fp8_kv_gb300 import synthetic as syn
from paged_fp8_kv_gb300.session import DecodeSession

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_fp8_kv_gb300.build import build

    build()


def _args(s, o, lse):
    """mj_decode_args for a session's buffers, with no workspace."""
    a = mj.DecodeArgs()
    a.q = s.q_packed.data_ptr()
    a.q_seq_stride = int(s.q_packed.stride(0))
    a.k, a.v = s.k_cache.data_ptr(), s.v_cache.data_ptr()
    a.k_page, a.k_row, a.k_head = mj.kv_strides(s.k_cache)
    a.v_page, a.v_row, a.v_head = mj.kv_strides(s.v_cache)
    a.block_table, a.seq_lens = s.block_table.data_ptr(), s.seq_lens.data_ptr()
    a.work, a.n_splits = s.work.data_ptr(), s.n_splits.data_ptr()
    a.num_work = int(s.work.shape[0])
    a.q_descale, a.k_descale, a.v_descale = s.q_descale.data_ptr(), s.k_descale.data_ptr(), s.v_descale.data_ptr()
    a.qd_seq, a.qd_head = mj.descale_strides(s.q_descale, s.num_seqs, s.h_k)
    a.kd_seq, a.kd_head = mj.descale_strides(s.k_descale, s.num_seqs, s.h_k)
    a.vd_seq, a.vd_head = mj.descale_strides(s.v_descale, s.num_seqs, s.h_k)
    a.softmax_scale, a.scale_o = float(s.w.softmax_scale), float(s.w.scale_o)
    a.o = o.data_ptr()
    a.o_seq_stride = int(o.stride(0))
    a.lse = lse.data_ptr()
    a.workspace = None
    a.workspace_bytes = 0
    a.status = None
    a.max_n_splits = s.plan.max_n_splits
    a.timing_events = None
    return a


def _static_call(s, o, lse):
    L = mj.lib()
    fn = L.mj_decode_attn_static_ws
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(mj.DecodeParams), ctypes.POINTER(mj.DecodeArgs), ctypes.c_void_p]
    a = _args(s, o, lse)
    return fn(ctypes.byref(s.params), ctypes.byref(a), torch.cuda.current_stream().cuda_stream)


CASES = [
    # a skewed fully-fp8 batch whose long sequence is split, so the merge
    # reads the static scratch
    (1, lambda: syn.config(3, num_seqs=4, len_range=(9000, 700))),
    (2, lambda: syn.config(3, num_seqs=4, len_range=(9000, 700))),
    # the head-grouped kernel keeps its unit counter in the scratch as well
    (3, lambda: syn.config(2, num_seqs=8, len_range=(3000, 6000))),
]


@pytest.mark.parametrize("kernel,make", CASES, ids=["cuda_core", "tensor_core", "grouped"])
def test_static_workspace_matches_regular_entry(kernel, make):
    w = make()
    s = DecodeSession(w, kernel=kernel)
    assert s.plan.max_n_splits > 1
    assert 0 < mj.workspace_bytes(s.params) <= (32 << 20)
    s.fill_workspace(float("nan"))
    s.decode()
    torch.cuda.synchronize()
    ref_o = s.o_packed.clone()
    ref_lse = s.lse.clone()
    for call in range(2):
        o = torch.full_like(s.o_packed, float("nan"))
        lse = torch.full_like(s.lse, float("nan"))
        assert _static_call(s, o, lse) == mj.MJ_OK
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o), f"O differs on call {call}"
        assert torch.equal(lse, ref_lse), f"LSE differs on call {call}"


def test_static_workspace_refuses_oversized_problems():
    w = syn.config(3, num_seqs=4, len_range=(9000, 700))
    s = DecodeSession(w)
    big = mj.make_params(4096, 1, 8, 16, 128, s.params.max_blocks, s.params.num_pages, True, mj.MJ_E4M3, 256)
    assert mj.workspace_bytes(big) > (32 << 20)
    L = mj.lib()
    fn = L.mj_decode_attn_static_ws
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(mj.DecodeParams), ctypes.POINTER(mj.DecodeArgs), ctypes.c_void_p]
    a = _args(s, s.o_packed, s.lse)
    assert fn(ctypes.byref(big), ctypes.byref(a), None) == mj.MJ_ERR_CAPACITY
