"""Test helpers: put a ``workloads.Workload`` into a GPU pool, run it through the C ABI, and
compare with the oracle.  Used by the GPU parity tests only."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads as wl

MAX_ABS = 2e-2   # the stated parity bar for bf16 inputs with fp32 accumulation
REL_L2 = 1e-3


def to_dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16).cuda()


def to_host_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16)


def pages_for(ranks, adapters, slack=4):
    rows = sum(max(8, 1 << (int(ranks[a]) - 1).bit_length()) for a in adapters)
    return (rows + 63) // 64 + slack


def make_pool(w, adapters=None, max_rows=None, factors=None, pages=None):
    """Pool with one module per workload module; loads ``adapters`` (default: the used ones)."""
    import adapter_serving_gb300 as L
    names = w.module_names()
    adapters = w.used_adapters() if adapters is None else adapters
    if pages is None:
        pages = [pages_for(w.ranks, adapters)] * len(names)
    pool = L.Pool([w.modules[m][0] for m in names], [w.modules[m][1] for m in names], w.n_adapters,
                  max_rank=64, pages=pages, max_rows=max_rows or max(w.n_rows, 1))
    cache = {} if factors is None else factors
    for a in adapters:
        for mi, m in enumerate(names):
            if (int(a), m) not in cache:
                cache[(int(a), m)] = (w.A(int(a), m), w.B(int(a), m))
            A, B = cache[(int(a), m)]
            pool.load(int(a), mi, to_host_bf16(A), to_host_bf16(B))
    torch.cuda.synchronize()
    return pool, cache


def run_stage(pool, w, stage, x_bits=None, W_bits=None, y_dtype=torch.float32, ids=None, segments=False):
    """Forward one stage (modules sharing x) through the C ABI; returns {module: y (torch, cuda)}."""
    names = w.module_names()
    x = to_dev_bf16(w.x(stage) if x_bits is None else x_bits)
    ios, outs = [], {}
    for m in w.stages[stage]:
        Wd = to_dev_bf16(w.W(m) if W_bits is None else W_bits[m])
        y = torch.full((w.n_rows, w.modules[m][1]), float("nan"), dtype=y_dtype, device="cuda")
        ios.append((names.index(m), x, Wd, y))
        outs[m] = y
    if segments:
        ss = torch.from_numpy(w.seg_start).cuda()
        sa = torch.from_numpy(w.seg_adapter).cuda()
        pool.segment_forward(ios, ss, sa, w.n_rows, w.scale)
    else:
        idt = torch.from_numpy(w.row_adapters() if ids is None else ids).cuda()
        pool.layer_forward(ios, idt, w.scale)
    torch.cuda.synchronize()
    return outs


def check_close(y, ref, max_abs=MAX_ABS, rel_l2=REL_L2, what=""):
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert y.shape == ref.shape, (y.shape, ref.shape)
    assert np.all(np.isfinite(y)), f"{what}: non-finite outputs"
    err = y - ref
    ma = float(np.abs(err).max()) if err.size else 0.0
    rl = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-30))
    assert ma <= max_abs and rl <= rel_l2, f"{what}: max-abs {ma:.3e} (<= {max_abs}), rel-L2 {rl:.3e} (<= {rel_l2})"
    return ma, rl


def bf16_ulps(y_bits, ref):
    """Distance in bf16 ulps between device bf16 outputs and the oracle rounded to bf16 (RNE)."""
    ref_bits = wl.f32_to_bf16_bits(np.asarray(ref, np.float64).astype(np.float32))

    def key(b):
        b = b.astype(np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(key(np.asarray(y_bits, np.uint16)) - key(ref_bits))


BF16_FLOOR_MAG = 2.0 ** -6   # below this |oracle|, an fp32 sum's rounding may exceed a bf16 ulp
BF16_FLOOR_ABS = 2.0 ** -13  # one bf16 ulp at that magnitude


def bf16_gate(y_bits, ref):
    """Outputs where the bf16 gate fails (an empty array when it holds).  A bf16 output is one
    rounding of the fp32 result, so it lies within 1 bf16 ulp of the oracle rounded alike -- as long
    as the fp32 result's own error (about 1e-6 of the magnitude of the summed terms) stays below
    half an ulp.  Near zero, where terms cancel, that error can exceed the ulp of the tiny result:
    outputs with |oracle| < 2^-6 are held to 2^-13 absolute instead (one ulp at 2^-6, ten times
    the fp32 path's typical error)."""
    ref = np.asarray(ref, np.float64)
    y = wl.bf16_bits_to_f32(np.asarray(y_bits, np.uint16)).astype(np.float64)
    ok = bf16_ulps(y_bits, ref) <= 1
    ok |= (np.abs(ref) < BF16_FLOOR_MAG) & (np.abs(y - ref) <= BF16_FLOOR_ABS)
    return np.argwhere(~ok)


def oracle_rows(w, module, stage, rows=None, threads=0, x_bits=None, W_bits=None, factors=None):
    return oracle.workload_module(w, module, rows=rows, threads=threads, stage_x=x_bits, W=W_bits,
                                  factors=factors)
