"""GB300 (sm_103a) multi-tenant LoRA adapted linear layer.

``y_i = W x_i + s * B_a (A_a x_i)`` for a batch whose rows each carry their own adapter id,
with the base W read once per call and every distinct adapter's factors gathered once
through a paged pool ("m07 -- Multi-Adapter (LoRA) Serving", section 6 "Deep Dive A:
Batching Heterogeneous Adapters"; "LoRA, quotas and noisy neighbours", section "One weight
read, many adapters").

This module is the Python binding of the C ABI in ``include/lora_gb300.h``: it marshals
arguments (torch tensors -> device pointers, the current CUDA stream) and nothing else;
every step of the forward runs in the CUDA library ``_build/liblora_gb300.so``. Importing
the package loads that library and fails loudly if it is missing -- there is no CPU path.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

__all__ = ["Pool", "AdapterCache", "LoraError", "build_segments", "form_batch", "quantize_rows_int8", "quantize_w4", "lib", "LIB_PATH", "DTYPE_F32", "DTYPE_BF16"]

LIB_PATH = _build.LIB
if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"CUDA library not built: {LIB_PATH} is missing. Run `python adapter_serving_gb300/build.py` "
        "(or __graft_entry__.build()) first.")
lib = ctypes.CDLL(LIB_PATH)

OK, EINVAL, ENOTLOADED, ENOMEM, ECUDA, EUNSUPPORTED, EDEVICE, EPINNED = 0, -1, -2, -3, -5, -6, -7, -8
DTYPE_F32, DTYPE_BF16 = 0, 1
MAX_MODULES, MAX_RANK, PAGE_ROWS, MAX_DECODE_ROWS = 8, 64, 64, 256
DEVERR = {0: "none", 1: "bad adapter id", 2: "adapter not loaded", 3: "in-kernel wait timed out",
          4: "bad segment table"}

_P, _I32, _I64, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float


class lora_pool_desc(ctypes.Structure):
    _fields_ = [("n_modules", _I32), ("d_in", ctypes.POINTER(_I32)), ("d_out", ctypes.POINTER(_I32)),
                ("max_adapters", _I32), ("max_rank", _I32), ("pages", ctypes.POINTER(_I64)), ("max_rows", _I32),
                ("factor_dtype", _I32)]


class lora_module_io(ctypes.Structure):
    _fields_ = [("module", _I32), ("x", _P), ("W", _P), ("y", _P)]


class lora_module_io_w4(ctypes.Structure):
    _fields_ = [("module", _I32), ("x", _P), ("W_codes", _P), ("W_scale", _P), ("y", _P)]


class lora_load_item(ctypes.Structure):
    _fields_ = [("adapter", _I32), ("module", _I32), ("rank", _I32), ("A", _P), ("B", _P)]


class lora_packed_item(ctypes.Structure):
    _fields_ = [("adapter", _I32), ("module", _I32), ("rank", _I32), ("pad_", _I32), ("a_offset", _I64),
                ("b_offset", _I64)]


class lora_batch_policy(ctypes.Structure):
    _fields_ = [("max_batch", _I32), ("max_distinct", _I32), ("min_batch", _I32), ("tail_slots", _I32),
                ("max_queue_ms", ctypes.c_double)]


def _sig(name, res, *args):
    f = getattr(lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_sig("lora_pool_create", ctypes.c_int, ctypes.POINTER(lora_pool_desc), ctypes.POINTER(_P))
_sig("lora_pool_destroy", ctypes.c_int, _P)
_sig("lora_pool_load", ctypes.c_int, _P, _I32, _I32, _P, _P, _I32, _P)
_sig("lora_pool_load_many", ctypes.c_int, _P, _I32, ctypes.POINTER(lora_load_item), ctypes.POINTER(_I32), _P)
_sig("lora_pool_load_packed", ctypes.c_int, _P, _I32, ctypes.POINTER(lora_packed_item), _P, _P, _I64,
     ctypes.POINTER(_I32), _P)
_sig("lora_pool_unload_many", ctypes.c_int, _P, _I32, ctypes.POINTER(_I32), ctypes.POINTER(_I32), _P)
_sig("lora_layer_step", ctypes.c_int, _P, _P, _I32, _I32, ctypes.POINTER(_I32), ctypes.POINTER(lora_module_io), _F,
     _I32, _P)
_sig("lora_layer_step_host", ctypes.c_int, _P, _P, _P, _I32, _I32, ctypes.POINTER(_I32), ctypes.POINTER(lora_module_io),
     ctypes.POINTER(_P), ctypes.POINTER(_P), _F, _I32, _P)
_sig("lora_pool_host_wait", ctypes.c_int, _P, _P)
_sig("lora_layer_gate_create", ctypes.c_int, _I32, ctypes.POINTER(_P))
_sig("lora_layer_gate_destroy", ctypes.c_int, _P)
_sig("lora_layer_gate_mark", ctypes.c_int, _P, _I32, _P)
_sig("lora_layer_gate_wait", ctypes.c_int, _P, _I32, _P)
_sig("lora_pool_unload", ctypes.c_int, _P, _I32, _P)
_sig("lora_pool_load_i8", ctypes.c_int, _P, _I32, _I32, _P, _P, _P, _P, _I32, _P)
_sig("lora_quantize_rows_int8", ctypes.c_int, _P, _I64, _I64, _P, _P)
_sig("lora_quantize_w4", ctypes.c_int, _P, _I64, _I64, _P, _P)
_sig("lora_pool_query", ctypes.c_int, _P, _I32, _I32, ctypes.POINTER(_I32), ctypes.POINTER(_I64))
_sig("lora_pool_free_rows", ctypes.c_int, _P, _I32, ctypes.POINTER(_I64))
_sig("lora_build_segments", ctypes.c_int, _P, _I32, _P, _P, _P, ctypes.POINTER(_I32))
_sig("lora_cache_create", ctypes.c_int, _I64, ctypes.c_double, ctypes.c_double, ctypes.POINTER(_P))
_sig("lora_cache_destroy", ctypes.c_int, _P)
_sig("lora_cache_acquire", ctypes.c_int, _P, _I32, _I64, ctypes.c_double, _P, _I32, ctypes.POINTER(_I32),
     ctypes.POINTER(_I32))
_sig("lora_cache_release", ctypes.c_int, _P, _I32)
_sig("lora_cache_stats", ctypes.c_int, _P, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I32))
_sig("lora_cache_resident", ctypes.c_int, _P, _I32, ctypes.POINTER(_I32), ctypes.POINTER(_I32))
_sig("lora_form_batch", ctypes.c_int, _P, _P, _I32, ctypes.POINTER(lora_batch_policy), _P, ctypes.POINTER(_I32),
     ctypes.POINTER(_I32))
_sig("lora_layer_forward", ctypes.c_int, _P, _I32, ctypes.POINTER(lora_module_io), _P, _I32, _F, _I32, _P)
_sig("lora_plan_rows", ctypes.c_int, _P, _P, _I32, _P)
_sig("lora_layer_forward_planned", ctypes.c_int, _P, _I32, ctypes.POINTER(lora_module_io), _F, _I32, _P)
_sig("lora_layer_forward_w4", ctypes.c_int, _P, _I32, ctypes.POINTER(lora_module_io_w4), _P, _I32, _F, _I32, _P)
_sig("lora_layer_forward_planned_w4", ctypes.c_int, _P, _I32, ctypes.POINTER(lora_module_io_w4), _F, _I32, _P)
_sig("lora_layer_step_host_w4", ctypes.c_int, _P, _P, _P, _I32, _I32, ctypes.POINTER(_I32),
     ctypes.POINTER(lora_module_io_w4), ctypes.POINTER(_P), ctypes.POINTER(_P), _F, _I32, _P)
_sig("lora_linear_forward", ctypes.c_int, _P, _I32, _P, _P, _P, _I32, _F, _P, _I32, _P)
_sig("lora_segment_forward", ctypes.c_int, _P, _I32, ctypes.POINTER(lora_module_io), _P, _P, _I32, _I32, _F,
     _I32, _P)
_sig("lora_linear_forward_static", ctypes.c_int, _P, _P, _I32, _I32, _P, _I32, _P, _P, _I32, _I32, _F, _P, _I32,
     _P)
_sig("lora_pool_last_segments", ctypes.c_int, _P, _P, _P, _P, ctypes.POINTER(_I32), ctypes.POINTER(_I32))
_sig("lora_last_device_error", ctypes.c_int, _P, ctypes.POINTER(_I32), ctypes.POINTER(_I32))
_sig("lora_profile_enable", ctypes.c_int, _P, _I32)
_sig("lora_pool_set_wait_budget", ctypes.c_int, _P, ctypes.c_uint64)
_sig("lora_profile_read", ctypes.c_int, _P, _I32, ctypes.POINTER(_I32), ctypes.POINTER(ctypes.c_double))
_sig("lora_last_cuda_error", ctypes.c_char_p)
_sig("lora_status_string", ctypes.c_char_p, ctypes.c_int)
_sig("lora_version", ctypes.c_int)


class LoraError(RuntimeError):
    def __init__(self, status, what):
        msg = f"{what}: {lib.lora_status_string(status).decode()} ({status})"
        if status == ECUDA:
            msg += f" [{lib.lora_last_cuda_error().decode()}]"
        super().__init__(msg)
        self.status = status


def _check(rc, what):
    if rc != OK:
        raise LoraError(rc, what)


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _dev_bf16(t, what):
    import torch
    if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
        raise ValueError(f"{what}: need a contiguous CUDA bf16 tensor")
    return t


def _dev_i32(t, what):
    import torch
    if not (t.is_cuda and t.dtype == torch.int32 and t.is_contiguous()):
        raise ValueError(f"{what}: need a contiguous CUDA int32 tensor")
    return t


def _y_dtype(y):
    import torch
    if not (y.is_cuda and y.is_contiguous()):
        raise ValueError("y: need a contiguous CUDA tensor")
    if y.dtype == torch.float32:
        return DTYPE_F32
    if y.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise ValueError("y: float32 or bfloat16")


def build_segments(ids):
    """Host-side stable grouping of rows by adapter id (lora_build_segments)."""
    import numpy as np
    ids = np.ascontiguousarray(ids, dtype=np.int32)
    n = len(ids)
    perm = np.empty(max(1, n), np.int32)
    seg_start = np.empty(n + 1, np.int32)
    seg_adapter = np.empty(max(1, n), np.int32)
    ns = _I32(0)
    _check(lib.lora_build_segments(ids.ctypes.data, n, perm.ctypes.data, seg_start.ctypes.data,
                                   seg_adapter.ctypes.data, ctypes.byref(ns)), "lora_build_segments")
    k = ns.value
    return perm[:n].copy(), seg_start[:k + 1].copy(), seg_adapter[:k].copy()


def quantize_rows_int8(bits):
    """Host int8 quantization, one fp32 scale per row (lora_quantize_rows_int8): ``bits`` are bf16
    values (uint16 numpy array or bf16 torch tensor) [rows, cols]; returns (int8 codes, fp32 scales)
    as numpy arrays."""
    import numpy as np
    if hasattr(bits, "view") and not isinstance(bits, np.ndarray):  # torch bf16 tensor
        import torch
        bits = bits.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    if b.ndim != 2:
        raise ValueError("need a 2-D array")
    codes = np.empty(b.shape, np.int8)
    scales = np.empty(b.shape[0], np.float32)
    _check(lib.lora_quantize_rows_int8(b.ctypes.data, b.shape[0], b.shape[1], codes.ctypes.data, scales.ctypes.data),
           "lora_quantize_rows_int8")
    return codes, scales


def quantize_w4(bits):
    """Host int4 quantization of base weights, one fp32 scale per row (lora_quantize_w4): ``bits``
    are bf16 values (uint16 numpy array or bf16 torch tensor) [rows, cols], cols a multiple of 8;
    returns (packed uint8 [rows, cols // 2] in the kernel's layout, fp32 scales [rows])."""
    import numpy as np
    if hasattr(bits, "view") and not isinstance(bits, np.ndarray):  # torch bf16 tensor
        import torch
        bits = bits.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    if b.ndim != 2:
        raise ValueError("need a 2-D array")
    packed = np.empty((b.shape[0], b.shape[1] // 2), np.uint8)
    scales = np.empty(b.shape[0], np.float32)
    _check(lib.lora_quantize_w4(b.ctypes.data, b.shape[0], b.shape[1], packed.ctypes.data, scales.ctypes.data),
           "lora_quantize_w4")
    return packed, scales


def form_batch(queue_adapter, queue_waited_ms, max_batch, max_distinct=32, min_batch=1, tail_slots=4,
               max_queue_ms=200.0):
    """Adapter-aware batch former (lora_form_batch): returns (queue indices of the next step's
    requests in batch order, distinct adapters among them).  Defaults are the pages' values: a cap
    of 32 adapters, 4 reserved tail slots, a 200 ms age deadline."""
    import numpy as np
    qa = np.ascontiguousarray(queue_adapter, dtype=np.int32)
    qw = np.ascontiguousarray(queue_waited_ms, dtype=np.float64)
    if qa.shape != qw.shape or qa.ndim != 1:
        raise ValueError("queue_adapter and queue_waited_ms: need two 1-D arrays of one length")
    pol = lora_batch_policy(int(max_batch), int(max_distinct), int(min_batch), int(tail_slots), float(max_queue_ms))
    out = np.empty(max(1, min(len(qa), int(max_batch))), np.int32)
    n, d = _I32(0), _I32(0)
    _check(lib.lora_form_batch(qa.ctypes.data, qw.ctypes.data, len(qa), ctypes.byref(pol), out.ctypes.data,
                               ctypes.byref(n), ctypes.byref(d)), "lora_form_batch")
    return out[:n.value].copy(), d.value


def pack_factors(entries, pin=True):
    """Pack bf16 factors for lora_pool_load_packed: entries = [(adapter_id, module, A, B)] with A
    [rank, d_in] and B [d_out, rank] bf16 (torch tensors or uint16 numpy arrays).  Returns (items,
    blob): the items for Pool.load_packed and one pinned uint8 tensor holding every A at a 16-byte
    aligned offset, each followed by its B (pin=False: ordinary host memory, for inspection)."""
    import numpy as np
    import torch
    items, parts, off = [], [], 0
    for a, m, A, B in entries:
        A = A.view(torch.uint16).numpy() if hasattr(A, "numpy") else np.asarray(A, np.uint16)
        B = B.view(torch.uint16).numpy() if hasattr(B, "numpy") else np.asarray(B, np.uint16)
        pad = (-off) % 16
        parts.append(np.zeros(pad, np.uint8))
        off += pad
        ao = off
        parts.append(np.ascontiguousarray(A).view(np.uint8).ravel())
        off += A.nbytes
        bo = off
        parts.append(np.ascontiguousarray(B).view(np.uint8).ravel())
        off += B.nbytes
        items.append((int(a), int(m), int(A.shape[0]), ao, bo))
    blob = torch.from_numpy(np.concatenate(parts) if parts else np.zeros(0, np.uint8))
    return items, (blob.pin_memory() if pin else blob)


class LayerGate:
    """One CUDA event per layer (lora_layer_gate_*): mark(l, copy_stream) after layer l's loads,
    wait(l, compute_stream) before layer l's forward."""

    def __init__(self, n_layers):
        h = _P()
        _check(lib.lora_layer_gate_create(int(n_layers), ctypes.byref(h)), "lora_layer_gate_create")
        self.handle = h
        self.n_layers = int(n_layers)

    def mark(self, layer, stream=None):
        _check(lib.lora_layer_gate_mark(self.handle, int(layer), _stream(stream)), "lora_layer_gate_mark")

    def wait(self, layer, stream=None):
        _check(lib.lora_layer_gate_wait(self.handle, int(layer), _stream(stream)), "lora_layer_gate_wait")

    def close(self):
        if self.handle:
            lib.lora_layer_gate_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class AdapterCache:
    """Residency decisions for a pool (lora_cache_*): value-per-byte eviction, reference counts,
    the pinning guard.  Host only; the caller applies the decisions to the pool."""

    def __init__(self, budget_bytes, guard_fraction=0.8, window_s=3600.0):
        h = _P()
        _check(lib.lora_cache_create(int(budget_bytes), float(guard_fraction), float(window_s), ctypes.byref(h)),
               "lora_cache_create")
        self.handle = h

    def acquire(self, adapter, nbytes, now_s):
        """Returns (adapters to unload first, whether `adapter` must be loaded); raises LoraError
        with status EPINNED (guard) or ENOMEM (no room)."""
        cap = 4096
        ev = (_I32 * cap)()
        n, load = _I32(0), _I32(0)
        _check(lib.lora_cache_acquire(self.handle, int(adapter), int(nbytes), float(now_s), ev, cap, ctypes.byref(n),
                                      ctypes.byref(load)), "lora_cache_acquire")
        return [ev[i] for i in range(n.value)], bool(load.value)

    def release(self, adapter):
        _check(lib.lora_cache_release(self.handle, int(adapter)), "lora_cache_release")

    def stats(self):
        """(resident bytes, pinned bytes, resident adapters)"""
        u, p, r = _I64(0), _I64(0), _I32(0)
        _check(lib.lora_cache_stats(self.handle, ctypes.byref(u), ctypes.byref(p), ctypes.byref(r)), "lora_cache_stats")
        return u.value, p.value, r.value

    def resident(self, adapter):
        """(resident, references)"""
        r, k = _I32(0), _I32(0)
        _check(lib.lora_cache_resident(self.handle, int(adapter), ctypes.byref(r), ctypes.byref(k)),
               "lora_cache_resident")
        return bool(r.value), k.value

    def close(self):
        if self.handle:
            lib.lora_cache_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Pool:
    """A paged adapter pool on the current CUDA device (lora_pool_create / _destroy)."""

    def __init__(self, d_in, d_out, max_adapters, max_rank=MAX_RANK, pages=None, max_rows=MAX_DECODE_ROWS,
                 factor_dtype="bf16"):
        """factor_dtype: "bf16" (load) or "int8" (load_i8: codes + per-rank-row scales; decode only)."""
        if factor_dtype not in ("bf16", "int8"):
            raise ValueError("factor_dtype: 'bf16' or 'int8'")
        n = len(d_in)
        self.d_in, self.d_out = list(map(int, d_in)), list(map(int, d_out))
        self._din = (_I32 * n)(*self.d_in)
        self._dout = (_I32 * n)(*self.d_out)
        self._pages = None if pages is None else (_I64 * n)(*map(int, pages))
        desc = lora_pool_desc(n, self._din, self._dout, int(max_adapters), int(max_rank),
                              self._pages, int(max_rows), 1 if factor_dtype == "int8" else 0)
        self.factor_dtype = factor_dtype
        h = _P()
        _check(lib.lora_pool_create(ctypes.byref(desc), ctypes.byref(h)), "lora_pool_create")
        self.handle = h
        self.max_adapters, self.max_rank, self.max_rows = int(max_adapters), int(max_rank), int(max_rows)

    def close(self):
        if self.handle:
            lib.lora_pool_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- residency
    def load(self, adapter_id, module, A, B, stream=None):
        """A: bf16 [rank, d_in], B: bf16 [d_out, rank]; host (pinned or pageable) or CUDA tensors."""
        import torch
        for t, nm in ((A, "A"), (B, "B")):
            if t.dtype != torch.bfloat16 or not t.is_contiguous():
                raise ValueError(f"{nm}: need a contiguous bf16 tensor")
        rank = A.shape[0]
        if B.shape != (self.d_out[module], rank) or A.shape != (rank, self.d_in[module]):
            raise ValueError(f"factor shapes {tuple(A.shape)} / {tuple(B.shape)} do not match module {module}")
        _check(lib.lora_pool_load(self.handle, int(adapter_id), int(module), _ptr(A), _ptr(B), int(rank),
                                  _stream(stream)), "lora_pool_load")

    def load_many(self, items, stream=None):
        """items: [(adapter_id, module, A, B)] as for load (host tensors should be pinned for the
        copies to run asynchronously); one call, one table-write launch per 64 items."""
        import torch
        arr = (lora_load_item * max(1, len(items)))()
        for i, (a, m, A, B) in enumerate(items):
            for t, nm in ((A, "A"), (B, "B")):
                if t.dtype != torch.bfloat16 or not t.is_contiguous():
                    raise ValueError(f"{nm}: need a contiguous bf16 tensor")
            rank = A.shape[0]
            if B.shape != (self.d_out[m], rank) or A.shape != (rank, self.d_in[m]):
                raise ValueError(f"factor shapes {tuple(A.shape)} / {tuple(B.shape)} do not match module {m}")
            arr[i] = lora_load_item(int(a), int(m), int(rank), A.data_ptr(), B.data_ptr())
        done = _I32(0)
        _check(lib.lora_pool_load_many(self.handle, len(items), arr, ctypes.byref(done), _stream(stream)),
               "lora_pool_load_many")
        return done.value

    def load_packed(self, items, host_blob, dev_staging, stream=None):
        """items: [(adapter_id, module, rank, a_offset, b_offset)], byte offsets of A [rank, d_in]
        and B [d_out, rank] (bf16) in host_blob (a pinned uint8 tensor); dev_staging: a CUDA uint8
        tensor at least as large.  One copy and one scatter launch (lora_pool_load_packed)."""
        arr = (lora_packed_item * max(1, len(items)))()
        for i, (a, m, r, ao, bo) in enumerate(items):
            arr[i] = lora_packed_item(int(a), int(m), int(r), 0, int(ao), int(bo))
        if dev_staging.numel() * dev_staging.element_size() < host_blob.numel() * host_blob.element_size():
            raise ValueError("dev_staging is smaller than host_blob")
        done = _I32(0)
        _check(lib.lora_pool_load_packed(self.handle, len(items), arr, _ptr(host_blob), _ptr(dev_staging),
                                         host_blob.numel() * host_blob.element_size(), ctypes.byref(done),
                                         _stream(stream)), "lora_pool_load_packed")
        return done.value

    def unload_many(self, adapter_ids, stream=None):
        ids = (_I32 * max(1, len(adapter_ids)))(*[int(a) for a in adapter_ids])
        done = _I32(0)
        _check(lib.lora_pool_unload_many(self.handle, len(adapter_ids), ids, ctypes.byref(done), _stream(stream)),
               "lora_pool_unload_many")
        return done.value

    def load_i8(self, adapter_id, module, qA, sA, qB, sB, stream=None):
        """int8 pool: qA int8 [rank, d_in], sA fp32 [rank], qB int8 [d_out, rank], sB fp32 [rank]
        (numpy arrays or host/CUDA tensors for the codes; the scales on the host)."""
        import numpy as np

        def _arr(a, dt):
            if hasattr(a, "data_ptr"):
                return a, a.data_ptr()
            a = np.ascontiguousarray(a, dtype=dt)
            return a, a.ctypes.data
        qA, pa = _arr(qA, np.int8)
        qB, pb = _arr(qB, np.int8)
        sA = np.ascontiguousarray(sA, dtype=np.float32)
        sB = np.ascontiguousarray(sB, dtype=np.float32)
        rank = int(qA.shape[0])
        if tuple(qA.shape) != (rank, self.d_in[module]) or tuple(qB.shape) != (self.d_out[module], rank) or \
                sA.shape != (rank,) or sB.shape != (rank,):
            raise ValueError(f"int8 factor shapes do not match module {module}")
        _check(lib.lora_pool_load_i8(self.handle, int(adapter_id), int(module), ctypes.c_void_p(pa), sA.ctypes.data,
                                     ctypes.c_void_p(pb), sB.ctypes.data, rank, _stream(stream)), "lora_pool_load_i8")

    def unload(self, adapter_id, stream=None):
        _check(lib.lora_pool_unload(self.handle, int(adapter_id), _stream(stream)), "lora_pool_unload")

    def query(self, adapter_id, module):
        r, off = _I32(0), _I64(0)
        _check(lib.lora_pool_query(self.handle, int(adapter_id), int(module), ctypes.byref(r), ctypes.byref(off)),
               "lora_pool_query")
        return r.value, off.value

    def free_rows(self, module):
        f = _I64(0)
        _check(lib.lora_pool_free_rows(self.handle, int(module), ctypes.byref(f)), "lora_pool_free_rows")
        return f.value

    # ---- forward
    @staticmethod
    def _ios(ios):
        arr = (lora_module_io * len(ios))()
        dt = None
        for i, (module, x, W, y) in enumerate(ios):
            _dev_bf16(x, "x"), _dev_bf16(W, "W")
            d = _y_dtype(y)
            if dt is not None and d != dt:
                raise ValueError("all outputs of one call share a dtype")
            dt = d
            arr[i] = lora_module_io(int(module), x.data_ptr(), W.data_ptr(), y.data_ptr())
        return arr, dt

    @staticmethod
    def _ios_w4(ios):
        import torch
        arr = (lora_module_io_w4 * len(ios))()
        dt = None
        for i, (module, x, codes, wscale, y) in enumerate(ios):
            _dev_bf16(x, "x")
            if not (codes.is_cuda and codes.dtype == torch.uint8 and codes.is_contiguous()):
                raise ValueError("W codes: need a contiguous CUDA uint8 tensor")
            if not (wscale.is_cuda and wscale.dtype == torch.float32 and wscale.is_contiguous()):
                raise ValueError("W scales: need a contiguous CUDA float32 tensor")
            d = _y_dtype(y)
            if dt is not None and d != dt:
                raise ValueError("all outputs of one call share a dtype")
            dt = d
            arr[i] = lora_module_io_w4(int(module), x.data_ptr(), codes.data_ptr(), wscale.data_ptr(), y.data_ptr())
        return arr, dt

    def layer_forward_w4(self, ios, row_adapter_ids, scale, stream=None):
        """int4 base: ios = [(module, x, W_codes, W_scale, y)] (quantize_w4's codes and scales on
        the device), row_adapter_ids: CUDA int32 [n] (-1 = base only)."""
        arr, dt = self._ios_w4(ios)
        ids = _dev_i32(row_adapter_ids, "row_adapter_ids")
        _check(lib.lora_layer_forward_w4(self.handle, len(ios), arr, _ptr(ids), ids.numel(), float(scale), dt,
                                         _stream(stream)), "lora_layer_forward_w4")

    def layer_forward_planned_w4(self, ios, scale, stream=None):
        """int4 base on the rows of the last plan_rows: ios = [(module, x, W_codes, W_scale, y)]."""
        arr, dt = self._ios_w4(ios)
        _check(lib.lora_layer_forward_planned_w4(self.handle, len(ios), arr, float(scale), dt, _stream(stream)),
               "lora_layer_forward_planned_w4")

    def layer_forward(self, ios, row_adapter_ids, scale, stream=None):
        """ios: [(module, x, W, y)], row_adapter_ids: CUDA int32 [n] (-1 = base only)."""
        arr, dt = self._ios(ios)
        ids = _dev_i32(row_adapter_ids, "row_adapter_ids")
        _check(lib.lora_layer_forward(self.handle, len(ios), arr, _ptr(ids), ids.numel(), float(scale), dt,
                                      _stream(stream)), "lora_layer_forward")

    def plan_rows(self, row_adapter_ids, stream=None):
        """Group a decode batch once for every module (lora_plan_rows); then layer_forward_planned."""
        ids = _dev_i32(row_adapter_ids, "row_adapter_ids")
        _check(lib.lora_plan_rows(self.handle, _ptr(ids), ids.numel(), _stream(stream)), "lora_plan_rows")

    def layer_forward_planned(self, ios, scale, stream=None):
        """ios: [(module, x, W, y)] on the rows of the last plan_rows."""
        arr, dt = self._ios(ios)
        _check(lib.lora_layer_forward_planned(self.handle, len(ios), arr, float(scale), dt, _stream(stream)),
               "lora_layer_forward_planned")

    def layer_step(self, stages, row_adapter_ids, scale, stream=None):
        """One decode layer in one call (lora_layer_step): plan the rows, then every stage in
        order.  stages: [[(module, x, W, y), ...], ...] (a stage's projections share x)."""
        flat = [io for st in stages for io in st]
        arr, dt = self._ios(flat)
        sn = (_I32 * max(1, len(stages)))(*[len(st) for st in stages])
        ids = _dev_i32(row_adapter_ids, "row_adapter_ids")
        _check(lib.lora_layer_step(self.handle, _ptr(ids), ids.numel(), len(stages), sn, arr, float(scale), dt,
                                   _stream(stream)), "lora_layer_step")

    def layer_step_host(self, stages, row_adapter_ids, host_ids, host_x, host_y, scale, stream=None):
        """lora_layer_step_host: stages as for layer_step (device x, W, y; row_adapter_ids the
        device ids buffer); host_ids: pinned int32 [n]; host_x[st]: pinned bf16 input of stage st;
        host_y: pinned outputs, one per projection in stage order.  One call moves the step's
        inputs in, runs it and moves its outputs out; the outputs are in host memory once `stream`
        has passed a later host_wait()."""
        import torch
        flat = [io for st in stages for io in st]
        arr, dt = self._ios(flat)
        sn = (_I32 * max(1, len(stages)))(*[len(st) for st in stages])
        ids = _dev_i32(row_adapter_ids, "row_adapter_ids")
        if host_ids.dtype != torch.int32 or host_ids.numel() != ids.numel():
            raise ValueError("host_ids: int32, one per row")
        hx = (_P * max(1, len(stages)))(*[t.data_ptr() for t in host_x])
        hy = (_P * max(1, len(flat)))(*[t.data_ptr() for t in host_y])
        _check(lib.lora_layer_step_host(self.handle, _ptr(host_ids), _ptr(ids), ids.numel(), len(stages), sn, arr, hx,
                                        hy, float(scale), dt, _stream(stream)), "lora_layer_step_host")

    def layer_step_host_w4(self, stages, row_adapter_ids, host_ids, host_x, host_y, scale, stream=None):
        """lora_layer_step_host_w4: as layer_step_host, each stage's entries (module, x, W_codes,
        W_scale, y) as for layer_forward_w4."""
        import torch
        flat = [io for st in stages for io in st]
        arr, dt = self._ios_w4(flat)
        sn = (_I32 * max(1, len(stages)))(*[len(st) for st in stages])
        ids = _dev_i32(row_adapter_ids, "row_adapter_ids")
        if host_ids.dtype != torch.int32 or host_ids.numel() != ids.numel():
            raise ValueError("host_ids: int32, one per row")
        hx = (_P * max(1, len(stages)))(*[t.data_ptr() for t in host_x])
        hy = (_P * max(1, len(flat)))(*[t.data_ptr() for t in host_y])
        _check(lib.lora_layer_step_host_w4(self.handle, _ptr(host_ids), _ptr(ids), ids.numel(), len(stages), sn, arr,
                                           hx, hy, float(scale), dt, _stream(stream)), "lora_layer_step_host_w4")

    def host_wait(self, stream=None):
        """Make `stream` wait for every download layer_step_host has queued (lora_pool_host_wait)."""
        _check(lib.lora_pool_host_wait(self.handle, _stream(stream)), "lora_pool_host_wait")

    def linear_forward(self, module, x, W, row_adapter_ids, scale, y, stream=None):
        _dev_bf16(x, "x"), _dev_bf16(W, "W")
        ids = _dev_i32(row_adapter_ids, "row_adapter_ids")
        _check(lib.lora_linear_forward(self.handle, int(module), _ptr(x), _ptr(W), _ptr(ids), ids.numel(),
                                       float(scale), _ptr(y), _y_dtype(y), _stream(stream)), "lora_linear_forward")

    def segment_forward(self, ios, seg_start, seg_adapter, n, scale, stream=None):
        """Grouped rows: seg_start CUDA int32 [n_seg+1], seg_adapter CUDA int32 [n_seg]."""
        arr, dt = self._ios(ios)
        ss, sa = _dev_i32(seg_start, "seg_start"), _dev_i32(seg_adapter, "seg_adapter")
        _check(lib.lora_segment_forward(self.handle, len(ios), arr, _ptr(ss), _ptr(sa), sa.numel(), int(n),
                                        float(scale), dt, _stream(stream)), "lora_segment_forward")

    def last_segments(self):
        """(perm or None, seg_start, seg_adapter) of the most recent forward, read back from the device."""
        import numpy as np
        n, ns = _I32(0), _I32(0)
        _check(lib.lora_pool_last_segments(self.handle, None, None, None, ctypes.byref(ns), ctypes.byref(n)),
               "lora_pool_last_segments")
        perm = np.full(max(1, n.value), -7, np.int32)
        ss = np.empty(ns.value + 1, np.int32)
        sa = np.empty(max(1, ns.value), np.int32)
        _check(lib.lora_pool_last_segments(self.handle, perm.ctypes.data, ss.ctypes.data, sa.ctypes.data,
                                           ctypes.byref(ns), ctypes.byref(n)), "lora_pool_last_segments")
        decoded = n.value <= MAX_DECODE_ROWS
        return (perm[:n.value].copy() if decoded else None), ss, sa[:ns.value].copy()

    KERNELS = {"prep": 0, "shrink": 1, "gemm": 2, "finalize": 3}

    def set_wait_budget(self, budget_ns):
        """Budget of each bounded in-kernel wait (lora_pool_set_wait_budget); 0 = the 2 s default."""
        _check(lib.lora_pool_set_wait_budget(self.handle, int(budget_ns)), "lora_pool_set_wait_budget")

    def profile(self, enable=True):
        _check(lib.lora_profile_enable(self.handle, 1 if enable else 0), "lora_profile_enable")

    def profile_read(self, kernel):
        """(launches, total device ms) of one kernel kind since the last read."""
        n, ms = _I32(0), ctypes.c_double(0)
        _check(lib.lora_profile_read(self.handle, self.KERNELS[kernel], ctypes.byref(n), ctypes.byref(ms)),
               "lora_profile_read")
        return n.value, ms.value

    def last_device_error(self):
        c, d = _I32(0), _I32(0)
        _check(lib.lora_last_device_error(self.handle, ctypes.byref(c), ctypes.byref(d)), "lora_last_device_error")
        return c.value, d.value
