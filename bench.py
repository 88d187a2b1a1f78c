#!/usr/bin/env python
"""Benchmark: multi-tenant LoRA adapted-layer decode on one GB300 (or N replicas).

Workload: the pages' 70B attention layer at decode -- q/o 8192->8192, k/v 8192->1024, 128
rows each carrying its own adapter (128 distinct rank-8 adapters on all four projections),
scale 1 ("m07 -- Multi-Adapter (LoRA) Serving", section 2 "Scale Numbers", the batch-128
distinct-adapter case).  One step = the whole hot path for one batch: q/k/v in one call
(they read the same x), then o.  The batch's rows are grouped once per step for every projection
(lora_plan_rows), then each call is shrink + tcgen05 base/expand (lora_layer_forward_planned).

Printed (rank 0, one JSON line): tokens/s (rows/s) over all GPUs, ms per step, HBM GB/s of
algorithmic bytes, the dominant kernel's roofline fraction (CUDA events on the launch
stream), the end-to-end number through the C ABI with host buffers, the CPU oracle as a
reported baseline, and SM clocks sampled during the timed region.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference]
Multi-GPU: one process per GPU (torchrun); every rank runs its own replica (the path has no
exchange step), value = rows of all ranks / max step time over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "adapted-layer decode tokens/s & HBM GB/s at batch 128, distinct adapters, 1 GB300"
UNIT = "tokens/s"
FLUSH_BYTES = 256 << 20  # > 129 MB L2
L2_BYTES = 129e6  # the L2 of this part (bytes)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="timed loop only (for profiler launch lists)")
    ap.add_argument("--workload", default="attn70b", choices=sorted(WORKLOADS) + ["layers8"],
                    help="attn70b (the headline) or another of the pages' configurations")
    return ap.parse_args()


# name -> (constructor, kind); the headline is attn70b
WORKLOADS = {"attn70b": (wl.attn70b_decode, "decode"), "all70b": (wl.all70b_decode, "decode"),
             "zipf": (wl.zipf_pool, "decode"), "prefill": (wl.prefill_segments, "prefill"),
             # the prefill path at a size a profiler capture can replay (8 requests, ~8.7k tokens)
             "prefill_small": (lambda: wl.prefill_segments(n_req=8), "prefill"),
             # the same decode batches with int8 adapter factors (codes + per-rank-row scales)
             "attn70b_i8": (wl.attn70b_decode, "decode"), "all70b_i8": (wl.all70b_decode, "decode"),
             # the same decode batches with an int4 base (codes + one fp32 scale per output row)
             "attn70b_w4": (wl.attn70b_decode, "decode"), "all70b_w4": (wl.all70b_decode, "decode")}
INT8 = {"attn70b_i8", "all70b_i8"}
W4 = {"attn70b_w4", "all70b_w4"}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def replica_rate(ms_local, rows_per_rank, world, device=None):
    """Whole-job rate of `world` independent replicas: every rank processed rows_per_rank rows in
    its own ms_local per step; the job's step is the slowest rank's (max over ranks, one
    all-reduce), and the rate is all ranks' rows over it.  Returns (rows/s, the job's ms)."""
    ms = float(ms_local)
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return world * rows_per_rank / (ms / 1e3), ms


def algorithmic_bytes(w, int8=False, w4=False):
    """Algorithmic bytes of one step: W once (int4 base: half a byte per weight plus one fp32
    scale per output row), each distinct adapter's factors once (int8: one byte per code plus the
    fp32 scale of each rank row, counted with A), x once per stage, y written once (fp32)."""
    ids = w.row_adapters()
    distinct = sorted(set(int(a) for a in ids if a >= 0))
    mods = w.module_names()
    e = 1 if int8 else 2
    if w4:
        W = sum(w.modules[m][0] * w.modules[m][1] // 2 + 4 * w.modules[m][1] for m in mods)
    else:
        W = sum(w.modules[m][0] * w.modules[m][1] * 2 for m in mods)
    A = sum(int(w.ranks[a]) * (w.modules[m][0] * e + (4 if int8 else 0)) for a in distinct for m in mods)
    B = sum(int(w.ranks[a]) * w.modules[m][1] * e for a in distinct for m in mods)
    X = sum(w.n_rows * w.modules[st[0]][0] * 2 for st in w.stages)
    Y = sum(w.n_rows * w.modules[m][1] * 4 for m in mods)
    # bf16 factors: the shrink runs inside the gemm (A tiles); int8 factors: a CUDA-core shrink
    gemm = W + X + (0 if int8 else A)
    return {"W": W, "A": A, "B": B, "x": X, "y": Y, "total": W + A + B + X + Y,
            "gemm": gemm, "shrink": A + X if int8 else 0, "finalize": B + Y, "distinct": len(distinct)}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def tensor_peak():
    """Dense bf16 TFLOP/s for a kernel inside a long step (the sustained figure)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 1700.0, "fallback"


def step_flops(w):
    """Dense flops of one step: base 2 n d_in d_out per projection plus the LoRA shrink and
    expand, 2 n r (d_in + d_out), each row with its own adapter's rank."""
    ranks = np.array([int(w.ranks[a]) if a >= 0 else 0 for a in w.row_adapters()], np.int64)
    base = sum(2 * w.n_rows * w.modules[m][0] * w.modules[m][1] for m in w.module_names())
    lora = sum(int(2 * ranks.sum() * (w.modules[m][0] + w.modules[m][1])) for m in w.module_names())
    return base, lora


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"lora_bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        mhz, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(mhz)}


# ---------------------------------------------------------------------------------------------
def cpu_baseline(w, xs, Ws, factors, budget_s=10.0, single_core_s=3.0):
    """The oracle as it stands, on this host's cores: whole steps (every row, every projection)
    repeated until ~budget_s of work; returns rows/s.  The same oracle on one core is timed too,
    on the first 8 rows of the step, for ~single_core_s."""
    import oracle

    def timed_rows(rows, threads, budget):
        t0 = time.perf_counter()
        done = 0
        while True:
            for st, mods in enumerate(w.stages):
                for m in mods:
                    oracle.workload_module(w, m, rows=rows, threads=threads, stage_x=xs[st], W=Ws[m], factors=factors)
            done += len(rows)
            if time.perf_counter() - t0 >= budget:
                return done, time.perf_counter() - t0

    done, dt = timed_rows(np.arange(w.n_rows), 0, budget_s)
    n_proj = sum(len(mods) for mods in w.stages)
    out = {"value": done / dt, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
           "sample": f"{done // w.n_rows} full step(s) of the workload ({done} rows x {n_proj} projections), fp64",
           "seconds": round(dt, 2)}
    done1, dt1 = timed_rows(np.arange(min(8, w.n_rows)), 1, single_core_s)
    out["single_core"] = {"value": done1 / dt1, "unit": UNIT, "cores": 1,
                          "sample": f"{done1} rows (the step's first 8, repeated) x {n_proj} projections, fp64",
                          "seconds": round(dt1, 2)}
    return out


def make_inputs(w):
    xs = [w.x(i) for i in range(len(w.stages))]
    Ws = {m: w.W(m) for m in w.module_names()}
    factors = {(int(a), m): (w.A(int(a), m), w.B(int(a), m)) for a in w.used_adapters() for m in w.module_names()}
    return xs, Ws, factors


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    xs, Ws, factors = make_inputs(w)
    import oracle
    rows = np.arange(16)  # each step: a bounded 16-row sample of the batch, all four projections
    def step():
        for st, mods in enumerate(w.stages):
            for m in mods:
                oracle.workload_module(w, m, rows=rows, stage_x=xs[st], W=Ws[m], factors=factors)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    v = len(rows) * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "rows_per_step": int(len(rows)), "batch_rows": w.n_rows},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"{len(rows)} of {w.n_rows} rows per step, all four projections"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, w):
    import torch
    import torch.distributed as dist
    import adapter_serving_gb300 as L

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    names = w.module_names()
    xs, Ws, factors = make_inputs(w)

    # ---- pool with the batch's adapters resident
    adapters = w.used_adapters()
    pages = (sum(max(8, int(w.ranks[a])) for a in adapters) + 63) // 64 + 4
    int8 = args.workload in INT8
    pool = L.Pool([w.modules[m][0] for m in names], [w.modules[m][1] for m in names], w.n_adapters,
                  max_rank=64, pages=[pages] * len(names), max_rows=w.n_rows,
                  factor_dtype="int8" if int8 else "bf16")
    for a in adapters:
        for mi, m in enumerate(names):
            A, B = factors[(int(a), m)]
            if int8:  # the library's quantizer: one scale per rank row of A and of B transposed
                qA, sA = L.quantize_rows_int8(A)
                qBt, sB = L.quantize_rows_int8(np.ascontiguousarray(B.T))
                pool.load_i8(int(a), mi, qA, sA, np.ascontiguousarray(qBt.T), sB)
            else:
                pool.load(int(a), mi, torch.from_numpy(A).view(torch.bfloat16), torch.from_numpy(B).view(torch.bfloat16))
    bf = lambda b: torch.from_numpy(b).view(torch.bfloat16).to(dev)
    xd = [bf(x) for x in xs]
    w4 = args.workload in W4
    if w4:  # the library's quantizer: int4 codes, one fp32 scale per output row
        Wq = {m: L.quantize_w4(Ws[m]) for m in names}
        Wd = {m: (torch.from_numpy(Wq[m][0]).to(dev), torch.from_numpy(Wq[m][1]).to(dev)) for m in names}
        del Wq
    else:
        Wd = {m: bf(Ws[m]) for m in names}
    yd = {m: torch.empty(w.n_rows, w.modules[m][1], device=dev) for m in names}
    grouped = w.ids is None
    if grouped:  # prefill: contiguous request segments; the base-only run gives every segment -1
        ids = torch.from_numpy(w.seg_adapter).to(dev)
        ss_d = torch.from_numpy(w.seg_start).to(dev)
    else:
        ids = torch.from_numpy(w.ids).to(dev)
    ids_base = torch.full_like(ids, -1)
    def io_of(m, x, y):
        return (names.index(m), x, *Wd[m], y) if w4 else (names.index(m), x, Wd[m], y)

    stage_io = [[io_of(m, xd[st], yd[m]) for m in mods] for st, mods in enumerate(w.stages)]
    stream = torch.cuda.current_stream()
    forward_planned = pool.layer_forward_planned_w4 if w4 else pool.layer_forward_planned

    def step(id_t):
        if not grouped:  # decode: one row grouping per batch serves every call of the step
            pool.plan_rows(id_t, stream=stream)
        for io in stage_io:
            if grouped:
                pool.segment_forward(io, ss_d, id_t, w.n_rows, w.scale, stream=stream)
            else:
                forward_planned(io, w.scale, stream=stream)

    # L2 flush before every timed step: write a buffer larger than L2, then read another one, so the
    # step starts with a cold L2 that holds no dirty lines (a write-only flush leaves up to 129 MB of
    # its own dirty lines, whose write-back would land inside the timed step)
    flush = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_rd = torch.zeros(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_sink = torch.empty(1, dtype=torch.float32, device=dev)

    def flush_l2():
        flush.zero_()
        torch.sum(flush_rd, dim=0, keepdim=True, out=flush_sink)

    def timed(n, id_t, per_step=None):
        """Device time of n steps, L2 flushed before each (the flush is outside the events)."""
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            flush_l2()
            evs[i][0].record(stream)
            (per_step or step)(id_t)
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in evs)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(3, args.warmup)):
        step(ids)
    torch.cuda.synchronize()
    code, detail = pool.last_device_error()
    if code:
        raise RuntimeError(f"device error {L.DEVERR.get(code)} at {detail}")

    sampler = ClockSampler(local)
    if not args.no_clocks:
        sampler.start()
        time.sleep(0.3)
    barrier()
    total_ms = timed(args.steps, ids)
    barrier()
    clocks = None
    if not args.no_clocks:
        # keep the same load running so the 100 ms sampler sees the clocks under it
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 1.5:
            timed(20, ids)
        clocks = sampler.stop()
    value, ms = replica_rate(total_ms / args.steps, w.n_rows, world, dev)
    ab = algorithmic_bytes(w, int8, w4)
    ranks = sorted(set(int(w.ranks[a]) for a in w.used_adapters()))
    line = {"metric": METRIC if args.workload == "attn70b" else f"{args.workload}: tokens/s", "value": value,
            "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16, int8 adapter factors" if int8 else ("bf16, int4 base weights" if w4 else "bf16"),
            "data": "synthetic",
            "config": {"workload": w.name + ("_int8_factors" if int8 else "") + ("_int4_base" if w4 else ""),
                       "batch_rows": w.n_rows, "distinct_adapters": ab["distinct"],
                       "ranks": ranks,
                       "projections": ", ".join(f"{m} {w.modules[m][0]}->{w.modules[m][1]}" for m in names),
                       "calls_per_step": len(w.stages), "output": "fp32",
                       "l2": "flushed before every timed step (256 MiB written, then 256 MiB of another "
                             "buffer read: a cold L2 with no dirty lines)",
                       "parallelism": f"replicas x{world}"},
            "hbm_gbs": ab["total"] / (ms / 1e3) / 1e9,
            "algorithmic_bytes_per_step": ab["total"],
            "gpu_launches": (3 * len(w.stages) if grouped else
                             1 + (3 if int8 else 2) * len(w.stages)) * args.steps}
    if grouped:
        base_f, lora_f = step_flops(w)
        tp, tsrc = tensor_peak()
        line["tensor"] = {"tflops": (base_f + lora_f) / (ms / 1e3) / 1e12, "peak": tp, "peak_source": tsrc,
                          "frac": (base_f + lora_f) / (ms / 1e3) / 1e12 / tp, "flops_per_step": base_f + lora_f,
                          "lora_flops_per_step": lora_f}
    if clocks:
        line["clocks"] = clocks

    if not args.no_extras and not grouped:
        # ---- per-kernel device time on the launch stream (library event pairs)
        pool.profile(True)
        timed(args.steps, ids)
        kt = {k: pool.profile_read(k) for k in ("prep", "shrink", "gemm", "finalize")}
        pool.profile(False)
        hbm, src = peaks()
        g_launch, g_ms = kt["gemm"]
        achieved = ab["gemm"] * args.steps / (g_ms / 1e3) / 1e9
        line["roofline"] = {"kernel": "decode_gemm_kernel (tcgen05: W tiles" + (
                                "" if int8 else " and the shrink's gathered A tiles") + ", stream-K)",
                            "bound": "hbm",
                            "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                            "frac_of_8tbs": achieved / 8000.0,
                            "peak_source": src,
                            "traffic": GEMM_DRAM_BYTES_PER_LAUNCH.get(args.workload),
                            "algorithmic_bytes_per_step": ab["gemm"], "launches_per_step": g_launch / args.steps}
        line["kernel_ms_per_step"] = {k: v[1] / args.steps for k, v in kt.items()}
        f_ms = kt["finalize"][1] / args.steps
        line["finalize_roofline"] = {"achieved": ab["finalize"] / (f_ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                                     "frac": ab["finalize"] / (f_ms / 1e3) / 1e9 / hbm,
                                     "algorithmic_bytes_per_step": ab["finalize"]}
        if ab["shrink"]:
            s_ms = kt["shrink"][1] / args.steps
            line["shrink_roofline"] = {"achieved": ab["shrink"] / (s_ms / 1e3) / 1e9, "peak": hbm, "unit": "GB/s",
                                       "frac": ab["shrink"] / (s_ms / 1e3) / 1e9 / hbm}
        # ---- the base-only layer on the same W and x (every row id -1)
        base_ms = timed(args.steps, ids_base) / args.steps
        line["base_only_ms_per_step"] = base_ms
        line["overhead_vs_base"] = ms / base_ms - 1
        line["byte_ratio_adapters_vs_base"] = (ab["A"] + ab["B"]) / ab["W"]
        # ---- end to end through the C ABI with host buffers (pinned), copies inside the timing
        hx = [torch.from_numpy(x).view(torch.bfloat16).pin_memory() for x in xs]
        hid = torch.from_numpy(w.ids).pin_memory()
        hy = {m: torch.empty(w.n_rows, w.modules[m][1], dtype=torch.float32).pin_memory() for m in names}
        h2d = sum(x.numel() * 2 for x in hx) + hid.numel() * 4
        d2h = sum(y.numel() * 4 for y in hy.values())

        # One library call per step with host buffers (lora_layer_step_host, or its int4-base twin
        # lora_layer_step_host_w4): the ids and the stages' x go up, the step runs, every y comes
        # back (a stage's outputs while the next stage computes); the call's work ends when the
        # last output has landed.  Steps run back to back on one stream, so all bytes of both
        # directions are inside the timed region.  No L2 flush between steps (see "timing").
        step_host = pool.layer_step_host_w4 if w4 else pool.layer_step_host
        # A base that fits L2 (the int4 codes: 76 MB) could be found there by the next step; then
        # each buffer set reads its own copy of W, so a step's W was last read two steps before.
        w_fits_l2 = ab["W"] <= L2_BYTES
        w_sets = [Wd, {m: (tuple(t.clone() for t in Wd[m]) if w4 else Wd[m].clone()) for m in names}
                  if w_fits_l2 else Wd]

        def io_w(m, x, y, Wm):
            return (names.index(m), x, *Wm[m], y) if w4 else (names.index(m), x, Wm[m], y)

        sets = []
        for b in range(2):  # two device buffer sets, alternating: step k+1's inputs go up while step k computes
            xb = [torch.empty_like(x) for x in xd]
            yb = {m: torch.empty_like(yd[m]) for m in names}
            sets.append((torch.empty_like(ids), [[io_w(m, xb[st], yb[m], w_sets[b]) for m in mods]
                                                 for st, mods in enumerate(w.stages)]))
        hy_sets = [[torch.empty_like(hy[m]).pin_memory() for mods in w.stages for m in mods] for _ in range(2)]

        def e2e_run(k_steps):
            """k_steps steps, one call each; returns (device ms, host wall ms) per step."""
            start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            start.record(stream)
            for k in range(k_steps):
                ids_b, stages_b = sets[k % 2]
                step_host(stages_b, ids_b, hid, hx, hy_sets[k % 2], w.scale, stream=stream)
            pool.host_wait(stream=stream)  # every step's outputs are in host memory
            end.record(stream)
            torch.cuda.synchronize()
            return start.elapsed_time(end) / k_steps, (time.perf_counter() - t0) * 1e3 / k_steps
        how = ("one lora_layer_step_host" + ("_w4" if w4 else "") + " call per step (ids and x up, the step, "
               "every y down; pinned host buffers, two device buffer sets alternating, so a step's copies "
               "overlap its neighbours' compute)")

        e2e_run(4)  # warm-up
        barrier()
        runs = [e2e_run(args.steps) for _ in range(5)]
        dev_ms = sorted(r[0] for r in runs)
        wall_ms = sorted(r[1] for r in runs)
        e_value, e_ms = replica_rate(dev_ms[2], w.n_rows, world, dev)  # median of 5, max over ranks
        line["e2e"] = {"value": e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
                       "ms_per_step_runs": dev_ms, "host_wall_ms_per_step_runs": wall_ms,
                       "timing": f"{how}; median of 5 runs of {args.steps} steps (device time, first upload to "
                                 f"last download); no L2 flush ({ab['W'] / 1e6:.0f} MB of W per step"
                                 + (f" > {L2_BYTES / 1e6:.0f} MB L2)" if not w_fits_l2 else
                                    f", less than the {L2_BYTES / 1e6:.0f} MB L2, so the two buffer sets read two "
                                    f"copies of W: a step's W was last read two steps, {2 * ab['total'] / 1e6:.0f} MB "
                                    "of traffic, before)")}
        code, detail = pool.last_device_error()
        if code:
            raise RuntimeError(f"device error {L.DEVERR.get(code)} at {detail}")
        if rank == 0 and not args.no_cpu_baseline and args.workload == "attn70b":
            line["cpu_baseline"] = cpu_baseline(w, xs, Ws, factors)
    if rank == 0:
        print(json.dumps(line), flush=True)
    pool.close()
    if world > 1:
        dist.destroy_process_group()


def run_layers(args):
    """Adapter loads pipelined across layers ("12. Adapter Serving and Multi-Tenant Customization",
    section "Switching cost: I/O, not compute"): 8 layers of the 70B attention projections, one
    pool per layer, 128 decode rows on 128 distinct rank-16 adapters.  Every step 4 cold adapters
    arrive (and 4 leave): their factors for all 8 layers are loaded while the step runs.  Three
    timings of the same forwards: every adapter already resident; the loads on a copy stream, layer
    by layer, each layer's forward waiting for its own layer's loads only (lora_layer_gate); the
    loads queued on the compute stream before each layer (no overlap)."""
    import torch
    import adapter_serving_gb300 as L
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n_layers, n, rank, n_cold = 8, 128, 16, 4
    mods = {"q": (8192, 8192), "k": (8192, 1024), "v": (8192, 1024), "o": (8192, 8192)}
    stages = [["q", "k", "v"], ["o"]]
    names = list(mods)
    g = torch.Generator(device=dev)
    g.manual_seed(1234)

    def randn(*shape, std=1.0):
        return (torch.randn(*shape, generator=g, device=dev) * std).to(torch.bfloat16)

    Ws = [{m: randn(mods[m][1], mods[m][0], std=mods[m][0] ** -0.5) for m in names} for _ in range(n_layers)]
    xs = [[randn(n, 8192) for _ in stages] for _ in range(n_layers)]
    ys = [{m: torch.empty(n, mods[m][1], device=dev) for m in names} for _ in range(n_layers)]
    total = 2 * (max(3, args.warmup) + args.steps) + 2  # pipelined and serial steps, each brings n_cold adapters
    n_ad = 128 + n_cold * (total + 1)
    live0 = 128
    pages = [(live0 + 3 * n_cold) * rank // 64 + 2] * len(names)  # the batch's, the cold ones, those leaving
    pools = [L.Pool([mods[m][0] for m in names], [mods[m][1] for m in names], n_ad, max_rank=64, pages=pages,
                    max_rows=n) for _ in range(n_layers)]
    # host factors: 8 pinned sets per layer, adapter a uses set a % 8 (the values do not matter here)
    hf = [[{m: (randn(rank, mods[m][0], std=0.02).cpu().pin_memory(), randn(mods[m][1], rank, std=0.02).cpu().pin_memory())
            for m in names} for _ in range(8)] for _ in range(n_layers)]

    def items(l, adapters):
        return [(a, names.index(m), *hf[l][a % 8][m]) for a in adapters for m in names]

    for l in range(n_layers):
        pools[l].load_many(items(l, range(live0)))
    # a cold adapter's factors for a layer arrive as one packed pinned blob (what a loader reading
    # them from host storage would hand over): blob h of layer l holds factor sets 4h .. 4h + 3,
    # adapter a uses set a % 8, and the cold adapters of a step are 4 consecutive ids
    packs = [[L.pack_factors([(i, names.index(m), *hf[l][4 * h + i][m]) for i in range(n_cold) for m in names])
              for h in range(2)] for l in range(n_layers)]
    staging = [torch.empty(packs[l][0][1].numel(), dtype=torch.uint8, device=dev) for l in range(n_layers)]
    torch.cuda.synchronize()
    load_bytes = sum(packs[l][0][1].numel() for l in range(n_layers))
    compute = torch.cuda.current_stream()
    # the loads' small kernels (table writes, the scatter of a packed blob) take SM slots as soon as
    # any are free, ahead of the forwards' waiting blocks: a high-priority copy stream
    copy_s = torch.cuda.Stream(device=dev, priority=-1)
    gate = L.LayerGate(n_layers)
    group = 4  # layers per gate wait
    # the rows of step k with loads: the 128 adapters resident once its cold ones are in (all
    # precomputed, so no host copy sits inside a step)
    ids_k = torch.stack([torch.arange(n_cold * (k + 1), n_cold * (k + 1) + live0, dtype=torch.int32)
                         for k in range(total)]).to(dev)
    ids_res = torch.arange(live0, dtype=torch.int32, device=dev)
    nxt = [live0]  # next cold adapter id
    step_end = [None, None, None]  # compute done, per loads step (ring)

    def layer_io(l):
        return [[(names.index(m), xs[l][st], Ws[l][m], ys[l][m]) for m in mods_] for st, mods_ in enumerate(stages)]

    ios = [layer_io(l) for l in range(n_layers)]

    def step(mode):
        """One 8-layer step; mode: 'resident', 'pipelined' or 'serial'."""
        if mode == "resident":
            for l in range(n_layers):
                pools[l].layer_step(ios[l], ids_res, 1.0, stream=compute)
            return
        k = (nxt[0] - live0) // n_cold  # loads step k: live = [n_cold (k + 1), n_cold (k + 1) + 128)
        ids_d = ids_k[k]
        cold = list(range(nxt[0], nxt[0] + n_cold))
        nxt[0] += n_cold
        h = (cold[0] % 8) // n_cold

        def load_layer(l, s):
            if evict:
                pools[l].unload_many(evict, stream=s)
            its, blob = packs[l][h]
            pools[l].load_packed([(cold[i], m, r, ao, bo) for i, m, r, ao, bo in its], blob, staging[l], stream=s)

        if mode == "serial":
            evict = list(range(n_cold * k, n_cold * (k + 1)))  # last used by the step before
            for l in range(n_layers):
                load_layer(l, compute)
                pools[l].layer_step(ios[l], ids_d, 1.0, stream=compute)
            return
        # The adapters that left the batch a step ago were last read by step k - 2's forwards: their
        # pages go back once that step is done (an event), so this step's loads need not wait for
        # the step still computing and may run ahead of it (the pool keeps room for them).
        evict = list(range(n_cold * (k - 1), n_cold * k)) if k > 0 else []
        done_k2 = step_end[(k - 2) % 3] if k >= 2 else None
        if done_k2 is not None:
            copy_s.wait_event(done_k2)
        elif k == 1:
            copy_s.wait_stream(compute)

        def loads(l):
            load_layer(l, copy_s)
            gate.mark(l, copy_s)

        # the loads go up a group of layers ahead; the forwards wait once per group, before its first
        # layer, for that group's loads (each stream wait keeps one forward from launching early)
        for l in range(min(group, n_layers)):
            loads(l)
        for l in range(n_layers):
            if l % group == 0:
                for j in range(l + group, min(l + 2 * group, n_layers)):
                    loads(j)  # the next group's loads, queued before this group's forwards
                for j in range(l, min(l + group, n_layers)):
                    gate.wait(j, compute)
            pools[l].layer_step(ios[l], ids_d, 1.0, stream=compute)
        ev = torch.cuda.Event()
        ev.record(compute)
        step_end[k % 3] = ev

    def timed(mode, k):
        """Per-step device times (events on the compute stream) and the host's ms per step."""
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(k)]
        t0 = time.perf_counter()
        for i in range(k):
            ev[i][0].record(compute)
            step(mode)
            ev[i][1].record(compute)
        host_ms = (time.perf_counter() - t0) * 1e3 / k
        torch.cuda.synchronize()
        return sorted(a.elapsed_time(b) for a, b in ev), host_ms

    res, host = {}, {}
    for mode in ("resident", "pipelined", "serial"):
        for _ in range(max(3, args.warmup)):
            step(mode)
        torch.cuda.synchronize()
        res[mode], host[mode] = timed(mode, args.steps)
    for l in range(n_layers):
        code, detail = pools[l].last_device_error()
        if code:
            raise RuntimeError(f"device error {L.DEVERR.get(code)} at {detail} (layer {l})")
    med = {k: statistics.median(v) for k, v in res.items()}
    line = {"metric": "layers8: 8-layer decode step with cold-adapter loads in flight, tokens/s", "value": n / (med["pipelined"] / 1e3),
            "unit": UNIT, "n_gpus": 1, "steps": args.steps, "warmup": max(3, args.warmup),
            "ms_per_step": med["pipelined"], "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": "layers8_attn70b_decode_b128_r16_4cold", "layers": n_layers, "batch_rows": n,
                       "rank": rank, "cold_adapters_per_step": n_cold,
                       "projections": ", ".join(f"{m} {mods[m][0]}->{mods[m][1]}" for m in names),
                       "l2": "no flush: each layer reads 302 MB of W, more than the 129 MB L2"},
            "gpu_launches": n_layers * (1 + 2 * len(stages)) * args.steps,
            "loads": {"bytes_per_step": load_bytes,
                      "ms_per_step_resident": med["resident"],
                      "ms_per_step_pipelined": med["pipelined"],
                      "ms_per_step_serial": med["serial"],
                      "pipelined_over_resident": med["pipelined"] / med["resident"] - 1,
                      "serial_over_resident": med["serial"] / med["resident"] - 1,
                      "copy_gbs_if_hidden": load_bytes / (med["resident"] / 1e3) / 1e9,
                      "host_ms_per_step": host,
                      "timing": "per-step device time (events on the compute stream), median of the steps"}}
    print(json.dumps(line), flush=True)
    gate.close()
    for pool in pools:
        pool.close()


def _build():
    import importlib.util
    spec = importlib.util.spec_from_file_location("_lora_build", os.path.join(ROOT, "adapter_serving_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per decode_gemm_kernel launch, the
# mean of the q/k/v and o launches of the workload, from the ncu captures summarised in profiles/
# (decode_gemm_kernel_*); absent for a workload without a capture, and to be removed whenever the
# kernel changes.
GEMM_DRAM_BYTES_PER_LAUNCH = {"attn70b": 191158528, "zipf": 246900992, "attn70b_w4": 76028672}


def main():
    args = parse()
    if args.impl == "ours":
        _build()
    if args.workload == "layers8":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the oracle has no layer pipeline to time"}))
        else:
            run_layers(args)
        return
    w = WORKLOADS[args.workload][0]()
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
