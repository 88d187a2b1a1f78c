"""The oracle: TEST INFRASTRUCTURE ONLY.

A plain, slow, fp64 CPU reference of the multi-tenant LoRA adapted linear layer, plus
the pages' sizing formulas. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg may import it. It shares no code with the
GPU library (``adapter_serving_gb300``) and never imports it.

* ``adapted_linear`` -- ``y_i = W x_i + s * B_a (A_a x_i)`` per row in fp64, from the C
  file next to this one (pages: "m07 -- Multi-Adapter (LoRA) Serving", section 6 "Deep
  Dive A", the forward y = Wx + (B.A)x.(alpha/r); "12. Adapter Serving ...", section "What
  an adapter adds to a forward pass").
* ``segments`` -- stable grouping of rows by adapter id ("m07", section 6, the index
  vector sequence -> adapter slot; "LoRA, quotas and noisy neighbours", section "One weight
  read, many adapters", rows tagged with their adapter).
* sizing: ``lora_params`` (``r (d_in + d_out)``, "m07" section 2 "Scale Numbers"),
  ``step_adapter_bytes`` (adapters are read once per DISTINCT adapter per decode step,
  "m07" section 6 "The cost is bandwidth, not compute"), ``base_bytes`` (base weights read
  once per step), ``lora_flop_ratio`` (the same section's ratio ``r(d_in+d_out)/(d_in d_out)``)
  and ``lora_extra_flops`` ("12. Adapter Serving ...", 2 x 2 x d x r per token).
* quantized variants: ``quantize_rows_int8`` / ``adapted_linear_factors64`` (int8 adapter
  factors) and ``quantize_rows_int4`` / ``adapted_linear_w4`` (an int4 base with bf16 or int8
  adapters, "12. Adapter Serving ...", section "Quantization").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lora_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liblora_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, OpenMP); returns the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            lib.oracle_adapted_linear.argtypes = [ctypes.c_int, P, ctypes.c_int, ctypes.c_int, P, P, P,
                                                  ctypes.c_int, P, P, P, ctypes.c_double, P, P,
                                                  ctypes.c_int, ctypes.c_int]
            lib.oracle_adapted_linear.restype = ctypes.c_int
            lib.oracle_segments.argtypes = [ctypes.c_int, P, P, P, P, P]
            lib.oracle_segments.restype = ctypes.c_int
            lib.oracle_max_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def adapted_linear(x, W, ids, A, B, scale, rows=None, threads=0, return_t=False):
    """fp64 ``y[s, :]`` for each selected row ``rows[s]`` (all rows if None).

    x: uint16 bf16 bits [n, d_in]; W: [d_out, d_in]; ids: int32 [n] (-1 = base only);
    A / B: sequences indexed by adapter id giving bf16-bit arrays [r_a, d_in] / [d_out, r_a]
    (``None`` for an adapter that has no factors). Returns float64 [n_sel, d_out]
    (and the unscaled shrink ``t`` [n_sel, max_rank] if ``return_t``).
    """
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    W = np.ascontiguousarray(W, dtype=np.uint16)
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n, d_in = x.shape
    d_out = W.shape[0]
    if W.shape[1] != d_in or ids.shape[0] != n:
        raise ValueError("shape mismatch")
    rows = np.arange(n, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    n_ad = len(A)
    keep = []
    a_ptrs = (ctypes.c_void_p * max(1, n_ad))()
    b_ptrs = (ctypes.c_void_p * max(1, n_ad))()
    ranks = np.zeros(max(1, n_ad), np.int32)
    for a in range(n_ad):
        if A[a] is None:
            continue
        Aa = np.ascontiguousarray(A[a], dtype=np.uint16)
        Ba = np.ascontiguousarray(B[a], dtype=np.uint16)
        r = Aa.shape[0]
        if Aa.shape != (r, d_in) or Ba.shape != (d_out, r):
            raise ValueError(f"adapter {a}: bad factor shapes {Aa.shape} {Ba.shape}")
        keep += [Aa, Ba]
        a_ptrs[a] = Aa.ctypes.data
        b_ptrs[a] = Ba.ctypes.data
        ranks[a] = r
    max_rank = max(1, int(ranks.max()))
    y = np.empty((len(rows), d_out), np.float64)
    t = np.empty((len(rows), max_rank), np.float64)
    rc = lib.oracle_adapted_linear(len(rows), _ptr(rows), d_in, d_out, _ptr(x), _ptr(W), _ptr(ids),
                                   n_ad, _ptr(ranks), ctypes.cast(a_ptrs, ctypes.c_void_p),
                                   ctypes.cast(b_ptrs, ctypes.c_void_p), float(scale), _ptr(y), _ptr(t),
                                   max_rank, int(threads))
    if rc != 0:
        raise ValueError("oracle: invalid adapter id or rank")
    return (y, t) if return_t else y


def quantize_rows_int8(bits):
    """Symmetric int8 codes with one fp32 scale per row ("m07 -- Multi-Adapter (LoRA) Serving",
    section 9 "Bottlenecks and Evolution", item 3: quantize adapters to int8).  For each row:
    scale = max|v| / 127 and code = round-half-even(v / scale), clipped to [-127, 127], all in fp32
    (a zero row gets scale 0 and codes 0).  ``bits``: uint16 bf16 bits [rows, cols]; returns
    (int8 [rows, cols], float32 [rows]).  For an adapter the rows are A's rank rows and B's rank
    columns (the rows of B transposed), so both scales belong to one rank index."""
    v = (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    v = v.reshape(np.shape(bits))
    scale = (np.abs(v).max(axis=1) / np.float32(127.0)).astype(np.float32)
    codes = np.zeros(v.shape, np.int8)
    nz = scale > 0
    q = np.rint(v[nz] / scale[nz, None])  # float32 / float32: one IEEE rounding, then half-to-even
    codes[nz] = np.clip(q, -127, 127).astype(np.int8)
    return codes, scale


def dequantize_rows_int8(codes, scale):
    """The factor the int8 codes stand for, exactly: code * scale in fp64."""
    return np.asarray(codes, np.float64) * np.asarray(scale, np.float64)[:, None]


def quantize_rows_int4(bits):
    """Symmetric int4 base weights with one fp32 scale per output row ("12. Adapter Serving and
    Multi-Tenant Customization", section "Quantization": the base model in INT4, the adapters in
    BF16).  The pages fix neither the grouping nor the rounding; this follows the int8 rule with 7
    in place of 127: scale = max|v| / 7 and code = round-half-even(v / scale), clipped to [-7, 7],
    all in fp32 (a zero row gets scale 0 and codes 0).  ``bits``: uint16 bf16 bits [rows, cols];
    returns (int8 [rows, cols] holding the codes, float32 [rows])."""
    v = (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    v = v.reshape(np.shape(bits))
    scale = (np.abs(v).max(axis=1) / np.float32(7.0)).astype(np.float32)
    codes = np.zeros(v.shape, np.int8)
    nz = scale > 0
    q = np.rint(v[nz] / scale[nz, None])  # float32 / float32: one IEEE rounding, then half-to-even
    codes[nz] = np.clip(q, -7, 7).astype(np.int8)
    return codes, scale


def adapted_linear_w4(x, codes, wscale, ids, A64, B64, scale, rows=None):
    """fp64 ``y_i = W x_i + s * B_a (A_a x_i)`` with the base given as int4 codes and row scales:
    W = codes * scale[:, None], exact in fp64 (the dequantised base of section "Quantization"), and
    the factors as fp64 arrays (bf16 or int8 factors converted exactly; None where not used).
    The plain definition in numpy fp64, the base term as one matrix product."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    rows = np.arange(len(ids), dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    W64 = np.asarray(codes, np.float64) * np.asarray(wscale, np.float64)[:, None]
    xf = (np.ascontiguousarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xf = xf.reshape(np.shape(x))[rows]
    y = xf @ W64.T
    for k, i in enumerate(rows):
        a = int(ids[i])
        if a < 0:
            continue
        y[k] += scale * (B64[a] @ (A64[a] @ xf[k]))
    return y


def adapted_linear_factors64(x, W, ids, A64, B64, scale, rows=None, threads=0):
    """fp64 ``y_i = W x_i + s * B_a (A_a x_i)`` with the factors given as fp64 arrays (the int8
    codes times their scales).  The base term comes from ``adapted_linear`` with every row
    base-only; the adapter term is the plain definition in numpy fp64, row by row."""
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n = len(ids)
    rows = np.arange(n, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64)
    y = adapted_linear(x, W, np.full(n, -1, np.int32), [None] * max(1, len(A64)), [None] * max(1, len(A64)),
                       scale, rows=rows, threads=threads)
    xf = (np.ascontiguousarray(x, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xf = xf.reshape(np.shape(x))
    for k, i in enumerate(rows):
        a = int(ids[i])
        if a < 0:
            continue
        t = A64[a] @ xf[i]
        y[k] += scale * (B64[a] @ t)
    return y


def segments(ids):
    """(perm, seg_start, seg_adapter): rows stably grouped by ascending adapter id."""
    lib = _load()
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n = len(ids)
    perm = np.empty(max(1, n), np.int32)
    seg_start = np.empty(n + 1, np.int32)
    seg_adapter = np.empty(max(1, n), np.int32)
    ns = np.zeros(1, np.int32)
    lib.oracle_segments(n, _ptr(ids), _ptr(perm), _ptr(seg_start), _ptr(seg_adapter), _ptr(ns))
    k = int(ns[0])
    return perm[:n].copy(), seg_start[:k + 1].copy(), seg_adapter[:k].copy()


# ---- sizing formulas ------------------------------------------------------------------

def lora_params(r: int, d_in: int, d_out: int) -> int:
    """Parameters one rank-r adapter adds to one (d_out, d_in) projection: r (d_in + d_out)."""
    return r * (d_in + d_out)


def adapter_bytes(modules, r, layers=1, bytes_per_param=2) -> int:
    """Bytes of one adapter of rank r over ``modules`` (iterable of (d_in, d_out)) and ``layers``."""
    return layers * sum(lora_params(r, di, do) for di, do in modules) * bytes_per_param


def base_bytes(modules, bytes_per_param=2) -> int:
    """Base-weight bytes read once per decode step: sum of d_in * d_out."""
    return sum(di * do for di, do in modules) * bytes_per_param


def step_adapter_bytes(row_ids, ranks, modules, bytes_per_param=2) -> int:
    """Adapter bytes one decode step reads: each DISTINCT adapter's factors once."""
    distinct = sorted(set(int(a) for a in np.asarray(row_ids).ravel() if a >= 0))
    return sum(adapter_bytes(modules, int(ranks[a]), 1, bytes_per_param) for a in distinct)


def distinct_adapters(row_ids) -> int:
    return len(set(int(a) for a in np.asarray(row_ids).ravel() if a >= 0))


def lora_flop_ratio(r: int, d_in: int, d_out: int) -> float:
    """LoRA FLOPs over base FLOPs per token for one projection: r (d_in + d_out) / (d_in d_out)."""
    return r * (d_in + d_out) / (d_in * d_out)


def lora_extra_flops(r: int, d: int) -> int:
    """Extra FLOPs per token per square d x d projection: two rank-r products, 2 x 2 x d x r."""
    return 2 * 2 * d * r


# ---- whole workloads --------------------------------------------------------------------

def workload_module(wl, module, rows=None, threads=0, stage_x=None, W=None, factors=None, return_t=False):
    """Oracle output of one module of a ``workloads.Workload`` for the selected rows."""
    st = next(i for i, s in enumerate(wl.stages) if module in s)
    x = wl.x(st) if stage_x is None else stage_x
    W = wl.W(module) if W is None else W
    ids = wl.row_adapters()
    used = set(int(a) for a in (ids if rows is None else ids[np.asarray(rows)]) if a >= 0)
    A = [None] * wl.n_adapters
    B = [None] * wl.n_adapters
    for a in used:
        if factors is not None:
            A[a], B[a] = factors[(a, module)]
        else:
            A[a], B[a] = wl.A(a, module), wl.B(a, module)
    return adapted_linear(x, W, ids, A, B, wl.scale, rows=rows, threads=threads, return_t=return_t)
