"""Benchmark: paged fp8-KV split-KV decode attention on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mj|reference]
                    [--config 4] [--variant ...] [--h_r ..] [--q_len ..] [--suite 0|1]

One step = one pass of the decode hot path over one batch: pack Q (q_len >
1), the decode kernel over every work item, the merge of split sequences,
unpack O (q_len > 1).  The plan is host work done once per batch shape and
reported separately (`plan_us`).  Inputs are synthetic (seeded, see
paged_fp8_kv_gb300/synthetic.py) and already resident in HBM.

`value` is algorithmic bytes per step (KV rows < L, Q, O, LSE, block table,
work list, descales, split partials written and read) / device time, in
GB/s, summed over ranks.  Every timed step finds its inputs cold: the loop
turns through enough device copies of the workload's inputs that at least
twice the L2 of other inputs is read between two uses of one copy (a GPU
sleep between steps, outside the step's events, keeps the host ahead);
workloads too small for that (over 16 copies) flush L2 with a 512 MiB write
before every step instead.  The page's own harness flushes with that write
before every call; the headline's `l2_write_flush` record times the step
that way too (the decode then also writes back the flush's dirty lines).

`--impl reference` times the fp64 CPU oracle, the only reference this
method has, on a bounded sample of the same workload.

The headline workload is config 4 (speculative verify, the largest).  With
no workload flag the line also carries `suite`: every workload of the five
configurations (the ten sweep points included) timed the same way in the
same run, with decode time, step time and roofline fraction each.

With N > 1 (torchrun) every rank runs an independent replica: there is no
data-path collective; barriers only bracket the timed region.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/step and KV GB/s vs GB300 HBM roofline, at 1 GPU"
PROFILES = os.path.join(ROOT, "profiles")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="mj", choices=["mj", "reference"])
    ap.add_argument("--config", type=int, default=4, help="headline workload: 4 = speculative verify (the largest config)")
    ap.add_argument("--variant", default=None)
    ap.add_argument("--h_r", type=int, default=None)
    ap.add_argument("--q_len", type=int, default=None)
    ap.add_argument("--max_splits", type=int, default=None)
    ap.add_argument("--num_seqs", type=int, default=None, help="smaller batch of the same config (profiling)")
    ap.add_argument("--kv_layout", default="nhd", choices=["nhd", "hnd", "interleaved", "flashinfer"])
    ap.add_argument("--kv_format", default="e4m3", choices=["e4m3", "e3m2", "e2m3", "e2m1", "nvfp4"], help="K/V pool element format")
    ap.add_argument("--kernel", type=int, default=0, help="0 auto, 1 CUDA-core, 2 tensor-core (swap-AB), 3 head-grouped tensor-core, 4 query-rows tensor-core")
    ap.add_argument("--l2_prefetch", type=int, default=0, help="0 default, -1 off, 1..8 tiles ahead")
    ap.add_argument("--kv_evict_first", type=int, default=0, help="K/V loads with L2 EVICT_FIRST: 0 default, -1 off, 1 on")
    ap.add_argument("--ctas_per_sm", type=int, default=0, help="plan slots per SM (0: the library's choice)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time steps as plain launches, not CUDA-graph replays")
    ap.add_argument(
        "--l2",
        default="rotate",
        choices=["rotate", "flush"],
        help="cold KV at every timed step: rotate device copies of the inputs (no flush), or flush L2 with a 512 MiB write",
    )
    ap.add_argument("--q_quant", action="store_true", help="also time the fused fp8 Q quantisation + pack for this shape")
    ap.add_argument("--suite", type=int, default=-1, help="1: also time every workload of the five configs (default: on when no workload flag is given)")
    ap.add_argument("--suite_steps", type=int, default=60, help="timed steps per suite workload")
    return ap.parse_args()


# --------------------------------------------------------------- workload


def workload(args):
    from paged_fp8_kv_gb300 import synthetic as syn

    return syn.config(
        args.config,
        variant=args.variant,
        h_r=args.h_r,
        q_len=args.q_len,
        max_splits=args.max_splits,
        num_seqs=args.num_seqs,
        kv_format=args.kv_format,
    )


def describe(w) -> str:
    lens = w.seq_lens
    return (
        f"{w.name}: b={w.num_seqs}, q_len={w.q_len}, h_k={w.h_k}, h_r={w.h_r}, d={w.head_dim}, "
        f"PS={w.page_size}, L in [{int(lens.min())},{int(lens.max())}] (sum {int(lens.sum())}), "
        f"{'causal' if w.causal else 'non-causal'}, Q {'e4m3' if w.q_is_e4m3 else 'bf16'}, KV {w.kv_format}"
    )


def algorithmic_bytes(w, plan):
    """(decode kernel bytes, merge kernel bytes, step bytes): what the method
    must move, not what a kernel happens to touch."""
    b, h_k, n_q, d = w.num_seqs, w.h_k, w.n_q, w.head_dim
    lens = w.seq_lens.astype(np.int64)
    qb = 1 if w.q_is_e4m3 else 2
    kv = w.kv_bytes()  # K + V rows below L in the pool's format (nvfp4: codes and scales)
    q = b * h_k * n_q * d * qb
    o = b * h_k * n_q * d * 2
    lse = b * h_k * n_q * 4
    bt = int(np.sum(-(-lens // w.page_size))) * 4
    meta = plan.num_work * 16 + b * 8 + 3 * b * h_k * 4
    split = plan.n_splits > 1
    part_rows = int(plan.n_splits[split].sum()) * h_k * n_q
    part = part_rows * (4 * d + 8)
    split_out = int(split.sum()) * h_k * n_q * (2 * d + 4)
    decode = kv + q + (o + lse - split_out) + bt + meta + part
    merge = part + split_out + b * 4 if split.any() else 0
    step = kv + q + o + lse + bt + meta + 2 * part
    if w.q_len > 1:  # pack reads + writes Q, unpack reads + writes O
        step += 2 * q + 2 * o
    return decode, merge, step


# ------------------------------------------------------------------ clocks


class ClockSampler:
    FIELDS = (
        "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
        "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
        "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"
    )

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"mj_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f,
                stderr=subprocess.DEVNULL,
            )
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons), "samples": len(sm)}


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return float(p["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def algorithmic_flops(w) -> int:
    """QK^T and PV multiply-adds of one decode launch (2 flops each): every
    visible (key, packed row) pair costs 2 d for S and 2 d for O."""
    L = np.asarray(w.seq_lens, dtype=np.int64)[:, None]
    qi = np.arange(w.q_len, dtype=np.int64)[None, :]
    vis = np.clip(L - w.q_len + qi + 1, 0, L) if w.causal else np.repeat(L, w.q_len, axis=1)
    return 4 * w.head_dim * w.h_k * w.h_r * int(vis.sum())


def tensor_peak():
    """e4m3 dense peak for a kernel timed alone: the measured burst bf16 GEMM
    rate x 2 (the nominal fp8 : bf16 ratio of the tensor cores)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return 2.0 * float(p["bf16_tflops"]), "measured bf16 burst x 2 (e4m3 : bf16 nominal)"
    return 2.0 * 1900.0, "fallback bf16 burst x 2"


def clocks_now(index: int):
    """One read-only nvidia-smi query of the SM clock and throttle reasons."""
    try:
        out = subprocess.run(
            ["nvidia-smi", "-i", str(index), f"--query-gpu={ClockSampler.FIELDS}", "--format=csv,noheader,nounits"],
            capture_output=True, text=True, timeout=10,
        ).stdout.strip().splitlines()
        parts = [p.strip() for p in out[0].split(",")]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        return {
            "sm_mhz": float(parts[0]),
            "sm_max_mhz": float(parts[1]),
            "reasons": sorted(nm for nm, v in zip(names, parts[4:8]) if v.lower().startswith("active")),
        }
    except Exception:
        return None


def traffic_applies(args) -> bool:
    """The committed traffic figures were taken on the full workloads with
    the default pool layout, plan and load options; a run that changes any
    of them reports none."""
    return (
        args.num_seqs is None
        and args.max_splits is None
        and args.kv_layout == "nhd"
        and args.l2_prefetch == 0
        and args.kv_evict_first == 0
        and args.ctas_per_sm == 0
    )


def traffic_record(kernel: str, workload_name: str):
    """dram bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(PROFILES, "traffic.json")
    if not os.path.exists(path):
        return None
    rec = json.load(open(path))
    entry = rec.get(kernel, {}).get(workload_name)
    if not entry:
        return None
    src = os.path.join(ROOT, "paged_fp8_kv_gb300", "csrc", entry["source"])
    if not os.path.exists(src):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return entry["dram_bytes_per_launch"] if sha == entry["source_sha"] else None


# --------------------------------------------------------------- GPU arm


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest of the ranks' values: the step time reported for N
    replicas is the slowest one's (every rank calls this)."""
    if world <= 1:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(world: int, step_bytes: int, step_ms: float) -> float:
    """Whole-job throughput: every replica moves step_bytes per step."""
    return world * step_bytes / (step_ms * 1e-3) / 1e9


COLD_MAX_COPIES = 16
SPACER_CYCLES = 150_000  # GPU sleep between rotated steps (about 75 us)


def l2_bytes(dev) -> int:
    import torch

    return int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (126 << 20))


def cold_copies(d_bytes: int, l2: int) -> int:
    """Device copies of a workload's inputs the timed loop turns through so
    that every step finds its KV cold: at least twice the L2 (l2 bytes) of
    other inputs is read between two uses of one copy of d_bytes.  1: too
    small to rotate (more than COLD_MAX_COPIES copies), the loop flushes L2
    instead."""
    k = 1 + -(-2 * int(l2) // max(int(d_bytes), 1))
    return k if k <= COLD_MAX_COPIES else 1


def l2_note(copies: int, d_bytes: int) -> str:
    if copies > 1:
        return (
            f"KV cold: {copies} device copies of the inputs used in turn ({(copies - 1) * d_bytes / 1e6:.0f} MB "
            "read between two uses of one, >= 2x L2), no flush in the loop; a GPU sleep between steps "
            "(outside the step events) keeps the host ahead"
        )
    return "flushed before every step (512 MiB write outside the step events)"


def time_steps(sessions, dev, flush, steps: int, warmup: int, eager: bool = False, world: int = 1):
    """Times `steps` decode steps, turning through `sessions` (device copies
    of one workload's inputs: cold KV at every step, a GPU sleep before each);
    with one session L2 is flushed (a 512 MiB write) before each step instead,
    outside the step's events.  The step time comes from CUDA-graph replays
    (pack, decode, merge, unpack), decode and merge times from eager steps
    with events between the kernels.  Returns (step_ms, decode_ms, merge_ms)."""
    import torch

    k = len(sessions)

    def gap(i):
        if k > 1:
            torch.cuda._sleep(SPACER_CYCLES)
        else:
            flush.fill_(i & 0xFF)  # L2 flush, outside the step's events

    stream = torch.cuda.current_stream(dev)
    for j in range(warmup * k):
        gap(j)
        sessions[j % k].step()
    torch.cuda.synchronize()
    # A step is timed as one replay of a CUDA graph holding (pack, decode,
    # merge, unpack); the library makes no host sync, so it captures as is.
    graphs = None
    if not eager:
        graphs = []
        for s in sessions:
            cs = torch.cuda.Stream(dev)
            cs.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cs):
                s.step(stream=cs)
            graphs.append(g)
        torch.cuda.synchronize()
        for j in range(warmup * k):
            gap(j)
            graphs[j % k].replay()
        torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    for e in [x for row in evs for x in row]:
        e.record()  # torch creates the CUDA event lazily, at its first record
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # Even steps carry events between the decode and the merge launch (the
    # per-kernel times of the roofline); an event there also serialises the
    # merge behind the decode grid, so the step time comes from the odd
    # steps, which run exactly as a caller's would (graph replays, the merge
    # a programmatic dependent of the decode grid).
    for i in range(steps):
        gap(i)
        sev[i][0].record()
        if i % 2 == 0 or steps == 1:
            sessions[i % k].step(timing_events=evs[i])
        elif graphs is not None:
            graphs[i % k].replay()
        else:
            sessions[i % k].step()
        sev[i][1].record()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    inner = range(0, steps, 2)
    plain = range(1, steps, 2) if steps > 1 else range(1)
    decode_ms = float(np.mean([evs[i][0].elapsed_time(evs[i][1]) for i in inner]))
    merge_ms = float(np.mean([evs[i][1].elapsed_time(evs[i][2]) for i in inner]))
    step_ms = float(np.mean([sev[i][0].elapsed_time(sev[i][1]) for i in plain]))
    return step_ms, decode_ms, merge_ms


def run_mj(args, rank, world, local_rank):
    import torch

    from paged_fp8_kv_gb300.build import build
    from paged_fp8_kv_gb300.session import DecodeSession
    from paged_fp8_kv_gb300 import decode_plan

    if rank == 0:
        build()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = workload(args)
    s = DecodeSession(w, device=str(dev), kv_layout=args.kv_layout, kernel=args.kernel, l2_prefetch=args.l2_prefetch,
        kv_evict_first=args.kv_evict_first, ctas_per_sm=args.ctas_per_sm,
    )
    d_bytes, m_bytes, step_bytes = algorithmic_bytes(w, s.plan)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)

    # host plan cost (the plan runs once per batch shape, on the host)
    t = time.perf_counter()
    for _ in range(20):
        decode_plan(s.params, w.seq_lens, sm_count=s.sm_count, ctas_per_sm=s.ctas_per_sm)
    plan_us = (time.perf_counter() - t) / 20 * 1e6

    # device copies of the inputs the timed loop turns through (cold KV at
    # every step without an L2 flush); 1: the loop flushes L2 instead
    copies = cold_copies(d_bytes, l2_bytes(dev)) if args.l2 == "rotate" else 1
    sessions = [s] + [
        DecodeSession(w, device=str(dev), kv_layout=args.kv_layout, kernel=args.kernel, l2_prefetch=args.l2_prefetch,
            kv_evict_first=args.kv_evict_first, ctas_per_sm=args.ctas_per_sm,
        )
        for _ in range(copies - 1)
    ]
    clk_before = clocks_now(local_rank)
    with ClockSampler(local_rank) as clk:
        step_ms, t_dec, merge_ms = time_steps(sessions, dev, flush, args.steps, args.warmup, args.eager, world)
        # the page's harness: a 512 MiB write before every step
        fl_steps = min(args.steps, 200)
        f_step, f_dec, f_mer = time_steps([s], dev, flush, fl_steps, args.warmup, args.eager, world)
    clk_after = clocks_now(local_rank)
    step_ms = max_over_ranks(step_ms, world, dev)
    f_step = max_over_ranks(f_step, world, dev)
    del sessions[1:]
    torch.cuda.empty_cache()
    write_flush = {
        "us_per_step": round(f_step * 1e3, 2),
        "decode_us": round(f_dec * 1e3, 2),
        "merge_us": round(f_mer * 1e3, 2),
        "steps": fl_steps,
        "note": "L2 flushed by a 512 MiB write before every step (the page's harness); the decode also "
        "writes back the flush's dirty lines",
    }

    launches = s.launches_per_step() * args.steps
    q_quant = q_quant_measure(w, dev, flush) if (w.q_is_e4m3 or args.q_quant) and rank == 0 else None
    plan_dev = plan_device_measure(s, w, dev, flush) if rank == 0 else None
    e2e = None if args.no_e2e else e2e_measure(args, s, w, step_bytes, dev)
    clocks = clk.summary()
    suite = None
    suite_clocks = None
    if rank == 0 and args.suite == 1:
        main_key = (args.config, args.variant, args.h_r, args.q_len, args.kv_format)
        with ClockSampler(local_rank) as sclk:
            suite = run_suite(args, dev, flush, reuse={main_key: w})
        suite_clocks = sclk.summary()
    return dict(
        w=w,
        s=s,
        step_ms=step_ms,
        decode_ms=t_dec,
        merge_ms=merge_ms,
        copies=copies,
        write_flush=write_flush,
        d_bytes=d_bytes,
        m_bytes=m_bytes,
        step_bytes=step_bytes,
        plan_us=plan_us,
        launches=launches,
        e2e=e2e,
        clocks=clock_record(clocks, clk_before, clk_after, suite_clocks),
        q_quant=q_quant,
        plan_dev=plan_dev,
        suite=suite,
    )


def clock_record(timed, before, after, suite):
    """The clocks line: samples taken during the timed region (often none:
    the region can be a few milliseconds), one query right before and right
    after it, and the samples taken while the suite ran (seconds of load)."""
    rec = {"during_timed": timed, "before": before, "after": after, "during_suite": suite}
    under = [c for c in (timed, suite) if c]
    pts = [c for c in (before, after) if c]
    src = under[0] if under else (pts[0] if pts else None)
    if src is None:
        return None
    reasons = sorted(set(r for c in under + pts for r in c.get("reasons", [])))
    mhz = [c["sm_mhz"] for c in under] or [c["sm_mhz"] for c in pts]
    return {
        "sm_mhz": float(np.median(mhz)),
        "sm_max_mhz": max(c["sm_max_mhz"] for c in under + pts),
        "reasons": reasons,
        "detail": rec,
    }


SUITE = (
    [(1, {}), (2, {}), (3, {}), (4, {}), (4, {"variant": "noncausal"})]
    + [(5, {"h_r": hr, "q_len": ql}) for hr in (16, 32) for ql in (1, 2, 4, 8, 16)]
    # narrow KV pools (fp4 / fp6 codes read by the MMA as they are)
    + [(2, {"kv_format": "e2m1"}), (3, {"kv_format": "e2m3"}), (4, {"kv_format": "e2m1"}), (4, {"kv_format": "e3m2"})]
    # nvfp4 (converted to e4m3 in the kernel; the fp8-Q configuration)
    + [(3, {"kv_format": "nvfp4"})]
)


def run_suite(args, dev, flush, reuse=None):
    """Every workload of the five configurations at full size, each timed like
    the headline (graph-replayed steps, cold KV at every step by rotated
    input copies or an L2 flush, decode and merge from event-split steps),
    with the automatic kernel and plan; each also timed with the page's
    512 MiB write flush before every step."""
    import torch

    from paged_fp8_kv_gb300 import synthetic as syn
    from paged_fp8_kv_gb300.session import DecodeSession

    peak, _ = measured_peaks()
    tpk, _ = tensor_peak()
    out = []
    for cfg, opts in SUITE:
        key = (cfg, opts.get("variant"), opts.get("h_r"), opts.get("q_len"), opts.get("kv_format", "e4m3"))
        w = (reuse or {}).get(key) or syn.config(cfg, **opts)
        s = DecodeSession(w, device=str(dev))
        d_bytes, _, step_bytes = algorithmic_bytes(w, s.plan)
        copies = cold_copies(d_bytes, l2_bytes(dev)) if args.l2 == "rotate" else 1
        sessions = [s] + [DecodeSession(w, device=str(dev)) for _ in range(copies - 1)]
        step_ms, dec_ms, mer_ms = time_steps(sessions, dev, flush, args.suite_steps, 5)
        f_step, f_dec, _ = time_steps([s], dev, flush, args.suite_steps, 5)
        rec = {
            "workload": w.name,
            "kernel": s.kernel,
            "n_q": w.n_q,
            "plan": {"work_items": s.plan.num_work, "max_n_splits": s.plan.max_n_splits, "ctas_per_sm": s.plan.opts.ctas_per_sm},
            "l2": f"rotate x{copies}" if copies > 1 else "flush",
            "us_per_step": round(step_ms * 1e3, 2),
            "decode_us": round(dec_ms * 1e3, 2),
            "merge_us": round(mer_ms * 1e3, 2) if s.plan.max_n_splits > 1 else 0.0,
            "step_gbs": round(step_bytes / (step_ms * 1e-3) / 1e9, 1),
            "frac": round(d_bytes / (dec_ms * 1e-3) / 1e9 / peak, 4),
            "frac_of_8000_gbs": round(d_bytes / (dec_ms * 1e-3) / 1e9 / 8000.0, 4),
            "write_flush": {
                "us_per_step": round(f_step * 1e3, 2),
                "decode_us": round(f_dec * 1e3, 2),
                "frac": round(d_bytes / (f_dec * 1e-3) / 1e9 / peak, 4),
            },
        }
        if w.n_q >= 128:
            rec["tensor_frac"] = round(algorithmic_flops(w) / (dec_ms * 1e-3) / 1e12 / tpk, 4)
        out.append(rec)
        del s, sessions
        torch.cuda.empty_cache()
    return out


def plan_device_measure(s, w, dev, flush, launches: int = 200):
    """The same plan built on the device (mj_decode_plan_device, the form a
    captured graph replays): checked equal to the host plan the steps used,
    timed alone with CUDA events after an L2 flush, and as the extra cost
    in a graph step: replays of (device plan, decode, merge) against
    (decode, merge) on the host plan's work list."""
    import torch

    import paged_fp8_kv_gb300 as mj

    o = s.plan.opts
    kw = dict(sm_count=o.sm_count, ctas_per_sm=o.ctas_per_sm, n_q_tiles=o.n_q_tiles, min_chunk_tiles=o.min_chunk_tiles)
    pad_to = mj.decode_plan_max_items(s.params, **kw)  # the tightest fixed length
    work = torch.empty((pad_to, 4), dtype=torch.int32, device=dev)
    ns = torch.empty((w.num_seqs,), dtype=torch.int32, device=dev)
    mj.decode_plan_device(s.params, s.seq_lens, work, ns, pad_to, **kw)
    torch.cuda.synchronize()
    same = bool(
        np.array_equal(work[: s.plan.num_work].cpu().numpy(), s.plan.work)
        and not work[s.plan.num_work :].any().item()
        and np.array_equal(ns.cpu().numpy(), s.plan.n_splits)
    )

    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for e0, e1 in evs:
            flush.fill_(3)
            e0.record()
            fn()
            e1.record()
        torch.cuda.synchronize()
        return float(np.mean([e0.elapsed_time(e1) for e0, e1 in evs])) * 1e3

    us = timed(lambda: mj.decode_plan_device(s.params, s.seq_lens, work, ns, pad_to, **kw), launches)

    def decode(work_t, max_n, stream):
        mj.decode_attn(
            s.params,
            q=s.q_packed,
            k_cache=s.k_cache,
            v_cache=s.v_cache,
            block_table=s.block_table,
            seq_lens=s.seq_lens,
            work=work_t,
            n_splits=ns,
            q_descale=s.q_descale,
            k_descale=s.k_descale,
            v_descale=s.v_descale,
            o=s.o_packed,
            lse=s.lse,
            workspace=s.workspace,
            softmax_scale=w.softmax_scale,
            scale_o=w.scale_o,
            max_n_splits=max_n,
            stream=stream,
            k_scales=s.k_scales,
            v_scales=s.v_scales,
        )

    cs = torch.cuda.Stream(dev)
    cs.wait_stream(torch.cuda.current_stream(dev))
    g_host, g_dev = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_host, stream=cs):
        decode(s.work, s.plan.max_n_splits, cs)
    with torch.cuda.graph(g_dev, stream=cs):
        mj.decode_plan_device(s.params, s.seq_lens, work, ns, pad_to, stream=cs, **kw)
        decode(work, s.max_splits, cs)
    torch.cuda.synchronize()
    for g in (g_host, g_dev):
        for _ in range(3):
            g.replay()
    t_host = timed(g_host.replay, 100)
    t_dev = timed(g_dev.replay, 100)
    return {
        "us_per_launch": round(us, 2),
        "pad_to": pad_to,
        "equals_host_plan": same,
        "graph_step_us_host_plan": round(t_host, 2),
        "graph_step_us_device_plan": round(t_dev, 2),
    }


def q_quant_measure(w, dev, flush, launches: int = 200):
    """The upstream fp8 step for this workload's query shape: bf16 Q in
    vLLM's layout -> e4m3 packed rows and per-(sequence, kv head)
    descales, one fused launch (mj_quantize_pack_q), timed alone with CUDA
    events after an L2 flush.  Bytes: bf16 Q read once, codes and descales
    written."""
    import torch

    from paged_fp8_kv_gb300 import quantize_pack_q

    gen = torch.Generator(device=dev)
    gen.manual_seed(1234)
    q = torch.randn((w.num_seqs * w.q_len, w.h_q, w.head_dim), generator=gen, device=dev).to(torch.bfloat16)
    q8 = torch.empty((w.num_seqs, w.h_k, w.n_q, w.head_dim), dtype=torch.uint8, device=dev)
    ds = torch.empty((w.num_seqs, w.h_k), dtype=torch.float32, device=dev)
    for _ in range(3):
        quantize_pack_q(q, q8, ds, w.num_seqs, w.q_len, w.h_k, w.h_r)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(launches)]
    torch.cuda.synchronize()
    for e0, e1 in evs:
        flush.fill_(7)
        e0.record()
        quantize_pack_q(q, q8, ds, w.num_seqs, w.q_len, w.h_k, w.h_r)
        e1.record()
    torch.cuda.synchronize()
    us = float(np.mean([e0.elapsed_time(e1) for e0, e1 in evs])) * 1e3
    nbytes = q.numel() * 2 + q8.numel() + ds.numel() * 4
    peak, _ = measured_peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    return {
        "kernel": "quantize_pack_q",
        "shape": f"({w.num_seqs * w.q_len}, {w.h_q}, {w.head_dim}) bf16 -> ({w.num_seqs}, {w.h_k}, {w.n_q}, {w.head_dim}) e4m3",
        "us_per_launch": round(us, 2),
        "bytes_per_launch": int(nbytes),
        "achieved_gbs": round(gbs, 1),
        "frac_of_hbm": round(gbs / peak, 4),
    }


def e2e_measure(args, s, w, step_bytes, dev):
    """Same step through the public API from HOST buffers, as a serving loop
    runs it.  Every step: the host plan, one host-to-device copy of the
    step's inputs (Q, seq_lens, block table, work list, n_splits, staged in
    one pinned buffer), the step as a CUDA graph replay, one device-to-host
    copy of O and LSE.  Two loops, host wall clock per step:
    - pipelined (StagedPipeline, two slots over one KV pool): a step's copies
      run on a copy stream and the host plans the next step while the device
      works, the steady state of a serving loop (the line's `value`);
    - synchronous (DecodeSession.stage / staged_step, a synchronisation after
      every step): one step's latency alone."""
    import torch

    from paged_fp8_kv_gb300 import decode_plan
    from paged_fp8_kv_gb300.session import DecodeSession, StagedPipeline

    kw = dict(kv_layout=args.kv_layout, kernel=args.kernel, l2_prefetch=args.l2_prefetch,
              kv_evict_first=args.kv_evict_first, ctas_per_sm=args.ctas_per_sm)
    seq_host = w.seq_lens

    e = DecodeSession(w, device=str(dev), **kw)
    e.stage()
    times = []
    for i in range(args.warmup + args.steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        plan = decode_plan(e.params, seq_host, sm_count=e.sm_count, ctas_per_sm=e.ctas_per_sm)
        e.staged_step(plan)
        torch.cuda.synchronize()
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    h2d, d2h = e.staged_bytes()
    t_sync = float(np.mean(times))
    del e
    torch.cuda.empty_cache()

    pipe = StagedPipeline(w, depth=2, device=str(dev), **kw)
    p0 = pipe.slots[0]

    def one(i):
        plan = decode_plan(p0.params, seq_host, sm_count=p0.sm_count, ctas_per_sm=p0.ctas_per_sm)
        pipe.inputs(i)  # (the synthetic inputs stay as staged)
        pipe.submit(i, plan)

    for i in range(args.warmup):
        one(i)
    if args.warmup > 0:
        pipe.outputs(args.warmup - 1)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.warmup, args.warmup + args.steps):
        one(i)
    pipe.outputs(args.warmup + args.steps - 1)
    t_pipe = (time.perf_counter() - t0) / args.steps
    del pipe, p0
    torch.cuda.empty_cache()
    return {
        "value": round(step_bytes / t_pipe / 1e9, 2),
        "unit": "GB/s",
        "us_per_step": round(t_pipe * 1e6, 2),
        "h2d_bytes_per_step": int(h2d),
        "d2h_bytes_per_step": int(d2h),
        "how": "host plan, one pinned H2D copy of the inputs, the step as a CUDA graph replay, one D2H copy of O "
        "and LSE, every step; pipelined two deep (input and output copies on two copy streams, the next step planned and queued while "
        "the device works), host wall clock from the first step queued to the last step's outputs in host memory",
        "synchronous": {
            "value": round(step_bytes / t_sync / 1e9, 2),
            "us_per_step": round(t_sync * 1e6, 2),
            "how": "the same step with a synchronisation after each: one step's latency",
        },
    }


# ------------------------------------------------------------ CPU oracle


def oracle_sample(w, budget_s: float, threads: int = 0, seed: int = 0):
    """Time the fp64 oracle on random (seq, kv head) units until about
    budget_s of work; returns (GB/s of algorithmic KV bytes, units, threads)."""
    import oracle

    rng = np.random.default_rng(seed)
    order = [(int(b), int(g)) for b in rng.permutation(w.num_seqs) for g in range(w.h_k)]
    nthreads = threads or (os.cpu_count() or 1)
    done_bytes, done_t, units_done = 0, 0.0, 0
    batch = max(1, nthreads)
    i = 0
    # cycle over the workload's units (the whole workload may take less
    # than the budget on many cores)
    while done_t < budget_s:
        units = [order[(i + k) % len(order)] for k in range(min(batch, len(order)))]
        i += len(units)
        t = time.perf_counter()
        oracle.attention(w, units=units, threads=nthreads)
        done_t += time.perf_counter() - t
        done_bytes += sum(int(w.seq_lens[b]) for b, _ in units) * w.head_dim * 2
        units_done += len(units)
        batch = min(batch * 2, 4096)
    return done_bytes / done_t / 1e9, units_done, nthreads, done_t


# ------------------------------------------------------------------ main


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.suite == -1:
        # the whole table by default; off when a single workload was asked for
        flags = (args.variant, args.h_r, args.q_len, args.num_seqs, args.max_splits)
        explicit = (
            any(f is not None for f in flags)
            or args.kernel != 0
            or "--config" in sys.argv
            or args.kv_format != "e4m3"
            or args.ctas_per_sm != 0
        )
        args.suite = 0 if explicit else 1
    if args.impl == "reference":
        if rank != 0:
            return
        w = workload(args)
        vals, units, nthreads = [], 0, os.cpu_count() or 1
        # each step a bounded sample: the whole run stays near two minutes
        step_budget = max(0.05, min(2.0, 120.0 / (args.warmup + args.steps)))
        for i in range(args.warmup + args.steps):
            gbs, u, nthreads, _ = oracle_sample(w, budget_s=step_budget, seed=i)
            if i >= args.warmup:
                vals.append(gbs)
                units = u
        v = float(np.mean(vals))
        line = {
            "impl": "reference",
            "metric": METRIC,
            "value": round(v, 4),
            "unit": "GB/s",
            "n_gpus": args.gpus,
            "steps": args.steps,
            "warmup": args.warmup,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": describe(w)},
            "cpu_baseline": {
                "value": round(v, 4),
                "unit": "GB/s",
                "cores": nthreads,
                "kind": "oracle",
                "sample": f"{units} random (seq, kv-head) units per step, ~{step_budget:.2f} s of fp64 oracle work; GB/s of KV rows read",
            },
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line))
        return

    import torch

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    r = run_mj(args, rank, world, local_rank)
    w, s = r["w"], r["s"]
    peak, peak_src = measured_peaks()
    achieved = r["d_bytes"] / (r["decode_ms"] * 1e-3) / 1e9
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        gbs, units, nthreads, secs = oracle_sample(w, budget_s=15.0)
        cpu = {
            "value": round(gbs, 4),
            "unit": "GB/s",
            "cores": nthreads,
            "kind": "oracle",
            "sample": f"{units} (seq, kv-head) units of the same workload ({units / (w.num_seqs * w.h_k):.1f} passes over its {w.num_seqs * w.h_k} units, random order), {secs:.1f} s of fp64 oracle work; GB/s of KV rows read",
        }
    value = whole_job_gbs(world, r["step_bytes"], r["step_ms"])
    if rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(r["step_ms"], 5),
            "us_per_step": round(r["step_ms"] * 1e3, 2),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": {
                "workload": describe(w),
                "kernel": s.kernel,
                "kv_layout": args.kv_layout,
                "l2_prefetch": args.l2_prefetch,
                "kv_evict_first": args.kv_evict_first,
                "max_splits": s.max_splits,
                "plan": {
                    "work_items": s.plan.num_work,
                    "chunk_tiles": s.plan.chunk_tiles,
                    "max_n_splits": s.plan.max_n_splits,
                    "ctas_per_sm": s.plan.opts.ctas_per_sm,
                    "sm_count": s.plan.opts.sm_count,
                },
                "l2": l2_note(r["copies"], r["d_bytes"]),
                "step_timing": "eager launches" if args.eager else "CUDA-graph replay of the step (pack, decode, merge, unpack)",
                "parallelism": f"replicas x{world}",
                "bytes_per_step": r["step_bytes"],
                "plan_us": round(r["plan_us"], 2),
            },
            "frac_of_8000_gbs": round(value / world / 8000.0, 4),
            "roofline": {
                "bound": "hbm",
                "kernel": s.kernel,
                "achieved": round(achieved, 2),
                "peak": peak,
                "peak_source": peak_src,
                "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": traffic_record(s.kernel, w.name) if traffic_applies(args) else None,
                "algorithmic_bytes_per_launch": r["d_bytes"],
                "decode_us": round(r["decode_ms"] * 1e3, 2),
                "merge_us": round(r["merge_ms"] * 1e3, 2),
            },
            "l2_write_flush": {
                **r["write_flush"],
                "frac": round(r["d_bytes"] / (r["write_flush"]["decode_us"] * 1e-6) / 1e9 / peak, 4),
            },
            "cpu_baseline": cpu,
            "e2e": r["e2e"],
            "gpu_launches": r["launches"],
            **({"q_quant": r["q_quant"]} if r["q_quant"] else {}),
            **({"plan_device": r["plan_dev"]} if r["plan_dev"] else {}),
            "clocks": r["clocks"],
            **({"suite": r["suite"]} if r["suite"] else {}),
        }
        if w.q_len * w.h_r >= 128:
            # at 128 or more packed rows the contraction nears the tensor
            # ridge: its roof beside the HBM one (the kernels issue e4m3
            # MMAs, timed alone: the burst peak; with bf16 Q the hi and lo
            # parts of Q and P double the executed MMA work over these
            # algorithmic flops)
            tpk, tsrc = tensor_peak()
            tfl = algorithmic_flops(w) / (r["decode_ms"] * 1e-3) / 1e12
            line["roofline_tensor"] = {
                "bound": "tensor",
                "achieved": round(tfl, 2),
                "peak": tpk,
                "peak_source": tsrc,
                "unit": "TFLOP/s",
                "frac": round(tfl / tpk, 4),
                "flops_per_launch": algorithmic_flops(w),
            }
        print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
