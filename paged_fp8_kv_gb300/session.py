"""Device-resident decode step for one batch: the buffers a caller keeps
between steps, and the calls of one step (plan, pack, decode + merge,
unpack), all through the C ABI.  Marshalling only.
"""

from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import (
    MJ_BF16,
    MJ_E4M3,
    decode_attn,
    decode_plan,
    kernel_name,
    KV_FORMATS,
    make_params,
    pack_q,
    unpack_o,
    workspace_bytes,
)


class DecodeSession:
    """Holds a workload's cache, tables and outputs on the GPU.

    ``w`` is any object with the fields of
    :class:`paged_fp8_kv_gb300.synthetic.Workload` (host numpy arrays)."""

    def __init__(
        self,
        w,
        device: str = "cuda",
        max_splits: Optional[int] = None,
        sm_count: Optional[int] = None,
        force_splits: int = 0,
        pad_to: int = 0,
        kv_layout: str = "nhd",
        kernel: int = 0,
        l2_prefetch: int = 0,
        kv_evict_first: int = 0,
        ctas_per_sm: int = 0,
        share_pool_with: Optional["DecodeSession"] = None,
    ):
        """``share_pool_with``: another session of the same workload whose
        device KV pool (pages, scale planes, descales) this one reads instead
        of holding its own copy."""
        self.w = w
        self.ctas_per_sm = int(ctas_per_sm)
        self.device = torch.device(device)
        dev = self.device
        self.num_seqs, self.q_len, self.h_k, self.h_r = w.num_seqs, w.q_len, w.h_k, w.h_r
        self.n_q = w.q_len * w.h_r
        self.d = w.head_dim
        self.q_dtype = MJ_E4M3 if w.q_is_e4m3 else MJ_BF16
        self.max_splits = int(max_splits if max_splits is not None else w.max_splits)
        self.params = make_params(
            w.num_seqs,
            w.q_len,
            w.h_k,
            w.h_r,
            w.page_size,
            w.max_blocks,
            w.num_pages,
            bool(w.causal),
            self.q_dtype,
            self.max_splits,
            w.head_dim,
            kernel,
            l2_prefetch,
            kv_evict_first,
            KV_FORMATS[getattr(w, "kv_format", "e4m3")],
        )
        self.kernel = kernel_name(self.params)
        if sm_count is None:
            sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
        self.sm_count = int(sm_count)

        # KV cache in the requested physical layout, exposed as logical
        # (num_pages, PS, h_k, row bytes) byte views (row bytes = d for e4m3,
        # d * bits / 8 for the packed narrow formats).
        k = torch.from_numpy(w.k_cache)
        v = torch.from_numpy(w.v_cache)
        if share_pool_with is not None:
            o = share_pool_with
            self.k_cache, self.v_cache = o.k_cache, o.v_cache
            if hasattr(o, "_kv_buf"):
                self._kv_buf = o._kv_buf
        elif kv_layout == "nhd":
            self.k_cache = k.to(dev)
            self.v_cache = v.to(dev)
        elif kv_layout == "hnd":  # (pages, 2, h_k, PS, d)
            buf = torch.stack([k.permute(0, 2, 1, 3), v.permute(0, 2, 1, 3)], dim=1).contiguous().to(dev)
            self.k_cache = buf[:, 0].transpose(1, 2)
            self.v_cache = buf[:, 1].transpose(1, 2)
            self._kv_buf = buf
        elif kv_layout == "interleaved":  # (pages, h_k, PS, 2d)
            buf = torch.cat([k.permute(0, 2, 1, 3), v.permute(0, 2, 1, 3)], dim=-1).contiguous().to(dev)
            kv = buf.transpose(1, 2)
            rb = k.shape[-1]
            self.k_cache = kv[..., :rb]
            self.v_cache = kv[..., rb:]
            self._kv_buf = buf
        elif kv_layout == "flashinfer":  # (pages, 2, PS, h_k, d)
            buf = torch.stack([k, v], dim=1).contiguous().to(dev)
            self.k_cache = buf[:, 0]
            self.v_cache = buf[:, 1]
            self._kv_buf = buf
        else:
            raise ValueError(kv_layout)

        # nvfp4: the scale planes, (num_pages, h_k, PS, d / 16) e4m3 codes
        ks, vs = getattr(w, "k_scales", None), getattr(w, "v_scales", None)
        if share_pool_with is not None:
            self.k_scales, self.v_scales = share_pool_with.k_scales, share_pool_with.v_scales
        else:
            self.k_scales = torch.from_numpy(ks).to(dev) if ks is not None else None
            self.v_scales = torch.from_numpy(vs).to(dev) if vs is not None else None
        self.block_table = torch.from_numpy(w.block_table).to(dev)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(dev)
        self.q_descale = torch.from_numpy(np.ascontiguousarray(w.q_descale)).to(dev)
        self.k_descale = torch.from_numpy(np.ascontiguousarray(w.k_descale)).to(dev)
        self.v_descale = torch.from_numpy(np.ascontiguousarray(w.v_descale)).to(dev)

        q_host = torch.from_numpy(w.q.view(np.int16) if w.q.dtype == np.uint16 else w.q)
        self.q_vllm = q_host.to(dev)  # (b*q_len, h_q, d), int16 (bf16 bits) or uint8
        self.q_packed = (
            self.q_vllm.view(self.num_seqs, self.h_k, self.n_q, self.d)
            if self.q_len == 1
            else torch.empty(self.num_seqs, self.h_k, self.n_q, self.d, dtype=self.q_vllm.dtype, device=dev)
        )
        self.o_packed = torch.empty(self.num_seqs, self.h_k, self.n_q, self.d, dtype=torch.bfloat16, device=dev)
        self.o_vllm = (
            self.o_packed.view(self.num_seqs * self.q_len, self.h_k * self.h_r, self.d)
            if self.q_len == 1
            else torch.empty(self.num_seqs * self.q_len, self.h_k * self.h_r, self.d, dtype=torch.bfloat16, device=dev)
        )
        self.lse = torch.empty(self.num_seqs, self.h_k, self.n_q, dtype=torch.float32, device=dev)
        ws = workspace_bytes(self.params)
        self.workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev) if ws else None
        self.replan(w.seq_lens, force_splits=force_splits, pad_to=pad_to)

    def replan(self, seq_lens_host, force_splits: int = 0, pad_to: int = 0) -> None:
        self.plan = decode_plan(
            self.params,
            seq_lens_host,
            sm_count=self.sm_count,
            ctas_per_sm=self.ctas_per_sm,
            force_splits=force_splits,
            pad_to=pad_to,
        )
        self.work = torch.from_numpy(self.plan.work).to(self.device)
        self.n_splits = torch.from_numpy(self.plan.n_splits).to(self.device)

    def fill_workspace(self, value: float) -> None:
        if self.workspace is not None:
            self.workspace.view(torch.float32)[: self.workspace.numel() // 4].fill_(value)

    def decode(self, stream=None, status=None, timing_events=None) -> None:
        decode_attn(
            self.params,
            q=self.q_packed,
            k_cache=self.k_cache,
            v_cache=self.v_cache,
            block_table=self.block_table,
            seq_lens=self.seq_lens,
            work=self.work,
            n_splits=self.n_splits,
            q_descale=self.q_descale,
            k_descale=self.k_descale,
            v_descale=self.v_descale,
            o=self.o_packed,
            lse=self.lse,
            workspace=self.workspace,
            softmax_scale=self.w.softmax_scale,
            scale_o=self.w.scale_o,
            status=status,
            max_n_splits=self.plan.max_n_splits,
            timing_events=timing_events,
            stream=stream,
            k_scales=self.k_scales,
            v_scales=self.v_scales,
        )

    def step(self, stream=None, status=None, timing_events=None) -> None:
        """pack (q_len > 1) -> decode + merge -> unpack (q_len > 1)."""
        if self.q_len > 1:
            pack_q(self.q_vllm, self.q_packed, self.num_seqs, self.q_len, self.h_k, self.h_r, stream=stream)
        self.decode(stream=stream, status=status, timing_events=timing_events)
        if self.q_len > 1:
            unpack_o(self.o_packed, self.o_vllm, self.num_seqs, self.q_len, self.h_k, self.h_r, stream=stream)

    def launches_per_step(self) -> int:
        n = 1 + (1 if self.plan.max_n_splits > 1 else 0)
        return n + (2 if self.q_len > 1 else 0)

    # host copies of the outputs, packed (b, h_k, n_q, d) / (b, h_k, n_q)
    def o_host(self) -> np.ndarray:
        return self.o_packed.float().cpu().numpy()

    def lse_host(self) -> np.ndarray:
        return self.lse.cpu().numpy()

    # ------------------------------------------------ host-to-host serving step

    def stage(self, work_cap: Optional[int] = None):
        """Prepare a serving loop's step from host memory: the step's inputs
        (Q in vLLM's layout, seq_lens, block table, work list, n_splits) become
        views of ONE device buffer with a pinned host twin, and the outputs (O
        in vLLM's layout, LSE) views of one more, so that a step is one
        host-to-device copy, the decode step (replayed as a CUDA graph), and one
        device-to-host copy.  Returns the pinned host views, keyed by name; the
        caller fills q / seq_lens / block_table and calls staged_step()."""
        dev = self.device
        cap = int(work_cap or max(1, self.num_seqs * self.max_splits))

        def layout(items):
            off, out = 0, {}
            for name, shape, dtype in items:
                off = (off + 255) // 256 * 256
                nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
                out[name] = (off, shape, dtype, nbytes)
                off += nbytes
            return out, (off + 255) // 256 * 256

        ins, in_bytes = layout([
            ("q", tuple(self.q_vllm.shape), self.q_vllm.dtype),
            ("seq_lens", tuple(self.seq_lens.shape), torch.int32),
            ("block_table", tuple(self.block_table.shape), torch.int32),
            ("work", (cap, 4), torch.int32),
            ("n_splits", (self.num_seqs,), torch.int32),
        ])
        outs, out_bytes = layout([
            ("o", (self.num_seqs * self.q_len, self.h_k * self.h_r, self.d), torch.bfloat16),
            ("lse", tuple(self.lse.shape), torch.float32),
        ])
        self._in_dev = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
        self._in_host = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
        self._out_dev = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
        self._out_host = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()

        def view(buf, spec):
            off, shape, dtype, nbytes = spec
            return buf[off : off + nbytes].view(dtype).view(shape)

        dv = {k: view(self._in_dev, v) for k, v in ins.items()}
        hv = {k: view(self._in_host, v) for k, v in ins.items()}
        hv["q"].copy_(self.q_vllm)
        hv["seq_lens"].copy_(self.seq_lens)
        hv["block_table"].copy_(self.block_table)
        self.q_vllm, self.seq_lens, self.block_table = dv["q"], dv["seq_lens"], dv["block_table"]
        if self.q_len == 1:
            self.q_packed = self.q_vllm.view(self.num_seqs, self.h_k, self.n_q, self.d)
        self._work_dev, self.n_splits = dv["work"], dv["n_splits"]
        o = view(self._out_dev, outs["o"])
        self.lse = view(self._out_dev, outs["lse"]).view(self.num_seqs, self.h_k, self.n_q)
        if self.q_len == 1:
            self.o_packed = o.view(self.num_seqs, self.h_k, self.n_q, self.d)
        self.o_vllm = o
        self._host_out = {k: view(self._out_host, v) for k, v in outs.items()}
        self._host_in = hv
        self._graph, self._graph_key = None, None
        return hv

    def staged_step(self, plan) -> dict:
        """One serving step from the pinned host views stage() returned: the
        plan's work list and split counts join the inputs there, one
        host-to-device copy, the step as a CUDA graph (captured again only when
        the plan's item count or largest split count changes), one
        device-to-host copy of O and LSE.  Returns the pinned output views
        (valid once the stream is synchronised)."""
        self._stage_plan(plan)
        self._in_dev.copy_(self._in_host, non_blocking=True)
        self._graph_for(plan).replay()
        self._out_host.copy_(self._out_dev, non_blocking=True)
        return self._host_out

    def _stage_plan(self, plan) -> None:
        n = plan.num_work
        self._host_in["work"].numpy()[:n] = plan.work
        self._host_in["n_splits"].numpy()[:] = plan.n_splits
        self.plan = plan
        self.work = self._work_dev[:n]

    def _graph_for(self, plan):
        """The step's CUDA graph for this plan shape (captured on a side
        stream after the current stream's work, the first time a shape is
        seen)."""
        key = (plan.num_work, plan.max_n_splits)
        if self._graph is None or self._graph_key != key:
            stream = torch.cuda.current_stream(self.device)
            side = torch.cuda.Stream(self.device)
            side.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                self.step(stream=side)
            stream.wait_stream(side)
            self._graph, self._graph_key = g, key
        return self._graph

    def staged_bytes(self):
        """(host-to-device, device-to-host) bytes a staged step copies."""
        return int(self._in_host.numel()), int(self._out_host.numel())


class StagedPipeline:
    """Serving steps from host memory with the copies off the critical path:
    ``depth`` staged sessions over ONE device KV pool take the steps in turn.
    Step i (slot i % depth) queues its input copy on an input-copy stream, its
    graph replay on a compute stream once that copy is in, and the copy of its
    O and LSE back on an output-copy stream once the replay is done (two copy
    streams: the next step's input copy does not queue behind this step's
    output copy, which waits for the replay); the host then
    returns at once, plans step i + 1 and queues it, so that the copies and
    the host's work of one step overlap the device work of its neighbours.

    inputs(i) returns slot i's pinned host inputs (q, seq_lens, block_table),
    free to fill once step i - depth's input copy has completed; submit(i,
    plan) queues the step; outputs(i) waits for step i's output copy and
    returns its pinned O / LSE views, valid until submit(i + depth)."""

    def __init__(self, w, depth: int = 2, device: str = "cuda", **session_kw):
        if depth < 1:
            raise ValueError("depth >= 1")
        first = DecodeSession(w, device=device, **session_kw)
        self.slots = [first] + [DecodeSession(w, device=device, share_pool_with=first, **session_kw) for _ in range(depth - 1)]
        self.host_in = [s.stage() for s in self.slots]
        self.device = first.device
        self.depth = depth
        self.h2d_stream = torch.cuda.Stream(self.device)
        self.d2h_stream = torch.cuda.Stream(self.device)
        self.compute_stream = torch.cuda.Stream(self.device)
        mk = lambda: [torch.cuda.Event() for _ in range(depth)]
        self.ev_in, self.ev_done, self.ev_out = mk(), mk(), mk()
        self.used = [False] * depth

    def inputs(self, i: int) -> dict:
        k = i % self.depth
        if self.used[k]:
            self.ev_in[k].synchronize()  # step i - depth has read the pinned inputs
        return self.host_in[k]

    def submit(self, i: int, plan) -> None:
        k = i % self.depth
        s = self.slots[k]
        if self.used[k]:
            self.ev_out[k].synchronize()  # step i - depth's outputs are out (and read by now)
        s._stage_plan(plan)
        g = s._graph_for(plan)
        with torch.cuda.stream(self.h2d_stream):
            if self.used[k]:
                self.h2d_stream.wait_event(self.ev_done[k])  # its replay has read the device inputs
            s._in_dev.copy_(s._in_host, non_blocking=True)
            self.ev_in[k].record(self.h2d_stream)
        with torch.cuda.stream(self.compute_stream):
            self.compute_stream.wait_event(self.ev_in[k])
            g.replay()
            self.ev_done[k].record(self.compute_stream)
        with torch.cuda.stream(self.d2h_stream):
            self.d2h_stream.wait_event(self.ev_done[k])
            s._out_host.copy_(s._out_dev, non_blocking=True)
            self.ev_out[k].record(self.d2h_stream)
        self.used[k] = True

    def outputs(self, i: int) -> dict:
        k = i % self.depth
        self.ev_out[k].synchronize()
        return self.slots[k]._host_out

    def bytes_per_step(self):
        return self.slots[0].staged_bytes()
