"""Paged fp8-KV split-KV decode attention for GB300 (sm_103a).

A thin ctypes binding over the C ABI of ``libmj.so`` (declared in
``include/mj.h``): argument marshalling only.  Every step of the decode path
runs in the library's CUDA kernels; there is no Python or CPU fallback, and
loading fails loudly when the library has not been built
(``python -m paged_fp8_kv_gb300.build``).

PyTorch is used only for device memory, streams and events.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmj.so")

MJ_OK = 0
MJ_ERR_INVALID_ARG = 1
MJ_ERR_UNSUPPORTED = 2
MJ_ERR_CAPACITY = 3
MJ_ERR_CUDA = 4
MJ_ERR_TIMEOUT = 5

MJ_BF16 = 0
MJ_E4M3 = 1

MJ_KV_E4M3 = 0
MJ_KV_E3M2 = 1
MJ_KV_E2M3 = 2
MJ_KV_E2M1 = 3
MJ_KV_NVFP4 = 4
KV_FORMATS = {"e4m3": MJ_KV_E4M3, "e3m2": MJ_KV_E3M2, "e2m3": MJ_KV_E2M3, "e2m1": MJ_KV_E2M1, "nvfp4": MJ_KV_NVFP4}

MJ_KERNEL_AUTO = 0
MJ_KERNEL_CUDA_CORE = 1
MJ_KERNEL_TENSOR_CORE = 2
MJ_KERNEL_TENSOR_CORE_GROUPED = 3
MJ_KERNEL_TENSOR_CORE_QROWS = 4


class MjError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


class DecodeParams(ctypes.Structure):
    _fields_ = [
        (name, ctypes.c_int32)
        for name in (
            "num_seqs",
            "q_len",
            "h_k",
            "h_r",
            "head_dim",
            "page_size",
            "max_blocks",
            "num_pages",
            "causal",
            "q_dtype",
            "max_splits",
            "kernel",
            "l2_prefetch",
            "kv_evict_first",
            "kv_format",
        )
    ]


class PlanOpts(ctypes.Structure):
    _fields_ = [
        (name, ctypes.c_int32)
        for name in ("sm_count", "ctas_per_sm", "n_q_tiles", "force_splits", "min_chunk_tiles", "pad_to")
    ]


_vp = ctypes.c_void_p
_i64 = ctypes.c_int64


class DecodeArgs(ctypes.Structure):
    _fields_ = [
        ("q", _vp),
        ("q_seq_stride", _i64),
        ("k", _vp),
        ("v", _vp),
        ("k_page", _i64),
        ("k_row", _i64),
        ("k_head", _i64),
        ("v_page", _i64),
        ("v_row", _i64),
        ("v_head", _i64),
        ("block_table", _vp),
        ("seq_lens", _vp),
        ("work", _vp),
        ("n_splits", _vp),
        ("num_work", ctypes.c_int32),
        ("q_descale", _vp),
        ("k_descale", _vp),
        ("v_descale", _vp),
        ("qd_seq", _i64),
        ("qd_head", _i64),
        ("kd_seq", _i64),
        ("kd_head", _i64),
        ("vd_seq", _i64),
        ("vd_head", _i64),
        ("softmax_scale", ctypes.c_float),
        ("scale_o", ctypes.c_float),
        ("o", _vp),
        ("o_seq_stride", _i64),
        ("lse", _vp),
        ("workspace", _vp),
        ("workspace_bytes", ctypes.c_size_t),
        ("status", _vp),
        ("max_n_splits", ctypes.c_int32),
        ("timing_events", _vp),
        ("k_scales", _vp),
        ("v_scales", _vp),
        ("ks_page", _i64),
        ("ks_head", _i64),
        ("vs_page", _i64),
        ("vs_head", _i64),
    ]


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libmj.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -m paged_fp8_kv_gb300.build` "
                "(there is no fallback implementation)"
            )
        L = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER
        L.mj_decode_plan.restype = ctypes.c_int
        L.mj_decode_plan.argtypes = [P(DecodeParams), P(PlanOpts), _vp, _vp, ctypes.c_int32, _vp, _vp, _vp]
        L.mj_decode_workspace_bytes.restype = ctypes.c_size_t
        L.mj_decode_workspace_bytes.argtypes = [P(DecodeParams)]
        L.mj_decode_attn.restype = ctypes.c_int
        L.mj_decode_attn.argtypes = [P(DecodeParams), P(DecodeArgs), _vp]
        L.mj_pack_q.restype = ctypes.c_int
        L.mj_pack_q.argtypes = [_vp, _vp] + [ctypes.c_int32] * 6 + [_vp]
        L.mj_decode_plan_max_items.restype = ctypes.c_int32
        L.mj_decode_plan_max_items.argtypes = [_vp, _vp]
        L.mj_decode_plan_device.restype = ctypes.c_int
        L.mj_decode_plan_device.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
        L.mj_check_preconditions.restype = ctypes.c_int
        L.mj_check_preconditions.argtypes = [P(DecodeParams), _vp, _vp, _vp, _vp, _vp] + [_i64] * 6 + [_vp]
        L.mj_check_gather_kv.restype = ctypes.c_int
        L.mj_check_gather_kv.argtypes = [P(DecodeParams), P(DecodeArgs), ctypes.c_int32, _vp, ctypes.c_int32, _vp]
        L.mj_check_dequant_e4m3.restype = ctypes.c_int
        L.mj_check_dequant_e4m3.argtypes = [_vp, _vp]
        L.mj_check_bounded_wait.restype = ctypes.c_int
        L.mj_check_bounded_wait.argtypes = [_vp, _vp, ctypes.c_int32, _vp]
        L.mj_quantize_pack_q.restype = ctypes.c_int
        L.mj_quantize_pack_q.argtypes = [_vp, _vp, _vp] + [ctypes.c_int32] * 5 + [_vp]
        L.mj_unpack_o.restype = ctypes.c_int
        L.mj_unpack_o.argtypes = [_vp, _vp] + [ctypes.c_int32] * 5 + [_vp]
        L.mj_status_string.restype = ctypes.c_char_p
        L.mj_status_string.argtypes = [ctypes.c_int]
        L.mj_kernel_name.restype = ctypes.c_int
        L.mj_kernel_name.argtypes = [P(DecodeParams), ctypes.c_char_p, ctypes.c_int32]
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().mj_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != MJ_OK:
        raise MjError(status, what)


def make_params(
    num_seqs: int,
    q_len: int,
    h_k: int,
    h_r: int,
    page_size: int,
    max_blocks: int,
    num_pages: int,
    causal: bool = True,
    q_dtype: int = MJ_BF16,
    max_splits: int = 16,
    head_dim: int = 128,
    kernel: int = MJ_KERNEL_AUTO,
    l2_prefetch: int = 0,
    kv_evict_first: int = 0,
    kv_format: int = MJ_KV_E4M3,
) -> DecodeParams:
    return DecodeParams(
        num_seqs,
        q_len,
        h_k,
        h_r,
        head_dim,
        page_size,
        max_blocks,
        num_pages,
        int(causal),
        q_dtype,
        max_splits,
        kernel,
        l2_prefetch,
        kv_evict_first,
        kv_format,
    )


@dataclass
class Plan:
    work: np.ndarray  # int32 (num_work, 4)
    n_splits: np.ndarray  # int32 (num_seqs,)
    chunk_tiles: int
    opts: PlanOpts

    @property
    def num_work(self) -> int:
        return int(self.work.shape[0])

    @property
    def max_n_splits(self) -> int:
        return int(self.n_splits.max())


def decode_plan(
    params: DecodeParams,
    seq_lens: Sequence[int],
    sm_count: int = 0,
    ctas_per_sm: int = 0,
    n_q_tiles: int = 0,
    force_splits: int = 0,
    min_chunk_tiles: int = 0,
    pad_to: int = 0,
) -> Plan:
    """mj_decode_plan on host seq_lens."""
    sl = np.ascontiguousarray(np.asarray(seq_lens, dtype=np.int32))
    opts = PlanOpts(sm_count, ctas_per_sm, n_q_tiles, force_splits, min_chunk_tiles, pad_to)
    cap = max(pad_to, int(params.num_seqs) * int(params.max_splits), 1)
    work = np.zeros((cap, 4), dtype=np.int32)
    n_splits = np.zeros(int(params.num_seqs), dtype=np.int32)
    num_work = ctypes.c_int32(0)
    chunk = ctypes.c_int32(0)
    st = lib().mj_decode_plan(
        ctypes.byref(params),
        ctypes.byref(opts),
        sl.ctypes.data,
        work.ctypes.data,
        cap,
        ctypes.addressof(num_work),
        n_splits.ctypes.data,
        ctypes.addressof(chunk),
    )
    _check(st, "mj_decode_plan")
    return Plan(work[: num_work.value].copy(), n_splits, chunk.value, opts)


def workspace_bytes(params: DecodeParams) -> int:
    return int(lib().mj_decode_workspace_bytes(ctypes.byref(params)))


def kernel_name(params: DecodeParams) -> str:
    buf = ctypes.create_string_buffer(64)
    _check(lib().mj_kernel_name(ctypes.byref(params), buf, 64), "mj_kernel_name")
    return buf.value.decode()


# ------------------------------------------------------------ torch glue


def _ptr(t) -> Optional[int]:
    return None if t is None else int(t.data_ptr())


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch

        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def descale_strides(t, num_seqs: int, h_k: int) -> Tuple[int, int]:
    """(seq, head) element strides of a descale tensor: one element is a
    per-tensor scale, (h_k,) per head, (b, h_k) per sequence and head."""
    if t.numel() == 1:
        return (0, 0)
    if t.dim() == 1:
        if t.shape[0] != h_k:
            raise ValueError(f"descale shape {tuple(t.shape)}")
        return (0, int(t.stride(0)))
    if t.dim() != 2 or t.shape[1] != h_k or t.shape[0] != num_seqs:
        raise ValueError(f"descale shape {tuple(t.shape)}")
    return (int(t.stride(0)), int(t.stride(1)))


def kv_strides(t) -> Tuple[int, int, int]:
    """(page, row, head) strides of a (num_pages, PS, h_k, d) byte view."""
    if t.element_size() != 1 or t.stride(3) != 1:
        raise ValueError("KV cache must be a 1-byte view with d contiguous")
    return (int(t.stride(0)), int(t.stride(1)), int(t.stride(2)))


def decode_attn(
    params: DecodeParams,
    *,
    q,
    k_cache,
    v_cache,
    block_table,
    seq_lens,
    work,
    n_splits,
    q_descale,
    k_descale,
    v_descale,
    o,
    lse,
    workspace=None,
    softmax_scale: float,
    scale_o: float = 1.0,
    status=None,
    max_n_splits: int = 0,
    timing_events=None,
    stream=None,
    k_scales=None,
    v_scales=None,
) -> None:
    """mj_decode_attn on device tensors.

    q / o are packed (b, h_k, n_q, d) views (rows contiguous, sequence stride
    free); k_cache / v_cache are (num_pages, PS, h_k, d) 1-byte views of any
    physical layout with d contiguous."""
    a = DecodeArgs()
    a.q = _ptr(q)
    a.q_seq_stride = int(q.stride(0))
    a.k, a.v = _ptr(k_cache), _ptr(v_cache)
    a.k_page, a.k_row, a.k_head = kv_strides(k_cache)
    a.v_page, a.v_row, a.v_head = kv_strides(v_cache)
    a.block_table, a.seq_lens = _ptr(block_table), _ptr(seq_lens)
    a.work, a.n_splits = _ptr(work), _ptr(n_splits)
    a.num_work = int(work.shape[0])
    nb, hk = int(params.num_seqs), int(params.h_k)
    a.q_descale, a.k_descale, a.v_descale = _ptr(q_descale), _ptr(k_descale), _ptr(v_descale)
    a.qd_seq, a.qd_head = descale_strides(q_descale, nb, hk)
    a.kd_seq, a.kd_head = descale_strides(k_descale, nb, hk)
    a.vd_seq, a.vd_head = descale_strides(v_descale, nb, hk)
    a.softmax_scale, a.scale_o = float(softmax_scale), float(scale_o)
    a.o = _ptr(o)
    a.o_seq_stride = int(o.stride(0))
    a.lse = _ptr(lse)
    a.workspace = _ptr(workspace)
    a.workspace_bytes = 0 if workspace is None else int(workspace.numel() * workspace.element_size())
    a.status = _ptr(status)
    a.max_n_splits = int(max_n_splits)
    ev_arr = None
    if timing_events is not None:
        handles = [int(e.cuda_event) for e in timing_events]
        if len(handles) != 3 or not all(handles):
            raise ValueError("timing_events: three created CUDA events (record each once first)")
        ev_arr = (ctypes.c_void_p * 3)(*handles)
        a.timing_events = ctypes.cast(ev_arr, ctypes.c_void_p)
    _set_scales(a, k_scales, v_scales)
    st = lib().mj_decode_attn(ctypes.byref(params), ctypes.byref(a), _stream_handle(stream))
    _check(st, "mj_decode_attn")


def scale_strides(t) -> Tuple[int, int]:
    """(page, head) byte strides of an nvfp4 scale plane viewed as
    (num_pages, h_k, page_size, d / 16) uint8 (rows 8 bytes apart)."""
    if t.dim() != 4 or t.element_size() != 1 or t.stride(3) != 1 or t.stride(2) != t.shape[3]:
        raise ValueError("scale plane: (pages, h_k, page_size, d/16) bytes with contiguous rows")
    return int(t.stride(0)), int(t.stride(1))


def _set_scales(a, k_scales, v_scales) -> None:
    if k_scales is None or v_scales is None:
        return
    a.k_scales, a.v_scales = _ptr(k_scales), _ptr(v_scales)
    a.ks_page, a.ks_head = scale_strides(k_scales)
    a.vs_page, a.vs_head = scale_strides(v_scales)


def pack_q(q_vllm, q_packed, num_seqs: int, q_len: int, h_k: int, h_r: int, stream=None) -> None:
    """mj_pack_q: (b*q_len, h_k*h_r, d) -> (b, h_k, q_len*h_r, d)."""
    st = lib().mj_pack_q(
        _ptr(q_vllm),
        _ptr(q_packed),
        int(q_vllm.element_size()),
        num_seqs,
        q_len,
        h_k,
        h_r,
        int(q_vllm.shape[-1]),
        _stream_handle(stream),
    )
    _check(st, "mj_pack_q")


def check_preconditions(params: DecodeParams, block_table, seq_lens, q_descale, k_descale, v_descale):
    """mj_check_preconditions on host (numpy) copies; returns (status, first
    offending sequence or -1)."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    nb, hk = int(params.num_seqs), int(params.h_k)
    # the C checker reads num_seqs rows of max_blocks entries and num_seqs
    # lengths: refuse arrays of another shape instead of reading past them
    if bt.shape != (nb, int(params.max_blocks)):
        raise ValueError(f"block_table shape {bt.shape}, expected {(nb, int(params.max_blocks))}")
    if sl.shape != (nb,):
        raise ValueError(f"seq_lens shape {sl.shape}, expected {(nb,)}")
    ds = [np.ascontiguousarray(d, dtype=np.float32) for d in (q_descale, k_descale, v_descale)]

    def strides(d):  # the element strides descale_strides gives a tensor
        if d.size == 1:
            return (0, 0)
        if d.ndim == 1 and d.shape[0] == hk:
            return (0, 1)
        if d.ndim == 2 and d.shape == (nb, hk):
            return (hk, 1)
        raise ValueError(f"descale shape {d.shape}")

    st_ = [strides(d) for d in ds]
    bad = ctypes.c_int32(0)
    st = lib().mj_check_preconditions(
        ctypes.byref(params),
        bt.ctypes.data,
        sl.ctypes.data,
        ds[0].ctypes.data,
        ds[1].ctypes.data,
        ds[2].ctypes.data,
        *st_[0],
        *st_[1],
        *st_[2],
        ctypes.addressof(bad),
    )
    return int(st), int(bad.value)


def check_gather_kv(params: DecodeParams, k_cache, v_cache, block_table, seq_lens, values: bool, out,
                    stream=None, k_scales=None, v_scales=None) -> None:
    """mj_check_gather_kv: the decode path's K (values False) or V rows of
    every (sequence, kv head) into out (b, h_k, out_rows, 128) uint8 (for an
    nvfp4 pool, the e4m3 rows its conversion gives)."""
    a = DecodeArgs()
    a.k, a.v = _ptr(k_cache), _ptr(v_cache)
    a.k_page, a.k_row, a.k_head = kv_strides(k_cache)
    a.v_page, a.v_row, a.v_head = kv_strides(v_cache)
    a.block_table, a.seq_lens = _ptr(block_table), _ptr(seq_lens)
    _set_scales(a, k_scales, v_scales)
    st = lib().mj_check_gather_kv(
        ctypes.byref(params), ctypes.byref(a), int(bool(values)), _ptr(out), int(out.shape[2]), _stream_handle(stream)
    )
    _check(st, "mj_check_gather_kv")


def check_dequant_e4m3(out, stream=None) -> None:
    """mj_check_dequant_e4m3: out (256,) float32 = the CUDA-core kernel's
    value of every e4m3 code."""
    _check(lib().mj_check_dequant_e4m3(_ptr(out), _stream_handle(stream)), "mj_check_dequant_e4m3")


def check_bounded_wait(status, waited_ns=None, limit_us: int = 1000, stream=None) -> None:
    """mj_check_bounded_wait: one warp waits limit_us on an mbarrier that
    never completes, then writes MJ_ERR_TIMEOUT to status (device int32) and
    the time waited to waited_ns (device int64, optional)."""
    _check(
        lib().mj_check_bounded_wait(_ptr(status), _ptr(waited_ns), int(limit_us), _stream_handle(stream)),
        "mj_check_bounded_wait",
    )


def decode_plan_max_items(
    params: DecodeParams,
    sm_count: int = 0,
    ctas_per_sm: int = 0,
    n_q_tiles: int = 0,
    force_splits: int = 0,
    min_chunk_tiles: int = 0,
) -> int:
    """mj_decode_plan_max_items: the tightest pad_to for the device plan."""
    opts = PlanOpts(sm_count, ctas_per_sm, n_q_tiles, force_splits, min_chunk_tiles, 0)
    n = int(lib().mj_decode_plan_max_items(ctypes.byref(params), ctypes.byref(opts)))
    if n < 0:
        raise MjError(MJ_ERR_INVALID_ARG, "mj_decode_plan_max_items")
    return n


def decode_plan_device(
    params: DecodeParams,
    seq_lens,
    work,
    n_splits,
    pad_to: int,
    sm_count: int = 0,
    ctas_per_sm: int = 0,
    n_q_tiles: int = 0,
    force_splits: int = 0,
    min_chunk_tiles: int = 0,
    chunk_tiles=None,
    status=None,
    stream=None,
) -> PlanOpts:
    """mj_decode_plan_device on device seq_lens (int32 (b,)) into device work
    (int32 (pad_to, 4)) and n_splits (int32 (b,)); returns the options used."""
    opts = PlanOpts(sm_count, ctas_per_sm, n_q_tiles, force_splits, min_chunk_tiles, pad_to)
    st = lib().mj_decode_plan_device(
        ctypes.byref(params),
        ctypes.byref(opts),
        _ptr(seq_lens),
        _ptr(work),
        _ptr(n_splits),
        _ptr(chunk_tiles),
        _ptr(status),
        _stream_handle(stream),
    )
    _check(st, "mj_decode_plan_device")
    return opts


def quantize_pack_q(q_vllm, q_packed, q_descale, num_seqs: int, q_len: int, h_k: int, h_r: int, stream=None) -> None:
    """mj_quantize_pack_q: bf16 (b*q_len, h_k*h_r, d) -> e4m3 codes
    (b, h_k, q_len*h_r, d) and fp32 descales (b, h_k)."""
    st = lib().mj_quantize_pack_q(
        _ptr(q_vllm),
        _ptr(q_packed),
        _ptr(q_descale),
        num_seqs,
        q_len,
        h_k,
        h_r,
        int(q_vllm.shape[-1]),
        _stream_handle(stream),
    )
    _check(st, "mj_quantize_pack_q")


def unpack_o(o_packed, o_vllm, num_seqs: int, q_len: int, h_k: int, h_r: int, stream=None) -> None:
    """mj_unpack_o: (b, h_k, q_len*h_r, d) -> (b*q_len, h_k*h_r, d), bf16."""
    st = lib().mj_unpack_o(
        _ptr(o_packed), _ptr(o_vllm), num_seqs, q_len, h_k, h_r, int(o_packed.shape[-1]), _stream_handle(stream)
    )
    _check(st, "mj_unpack_o")
