"""CPU-only checks of the C-ABI library: it builds, loads, exports every function the header
declares, and its host-side logic (row grouping, status strings, argument checks) is right.
No kernel is launched here."""
import os
import re

import numpy as np
import pytest
import torch

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lora_gb300.h")


def _lib():
    import adapter_serving_gb300 as L
    return L


def header_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(lora_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_boundary():
    fns = header_functions()
    for f in ("lora_pool_create", "lora_pool_load", "lora_linear_forward", "lora_layer_forward",
              "lora_segment_forward", "lora_build_segments", "lora_pool_destroy", "lora_status_string"):
        assert f in fns


def test_library_exports_every_declared_symbol():
    L = _lib()
    missing = [f for f in header_functions() if not hasattr(L.lib, f)]
    assert not missing, missing
    assert L.lib.lora_version() >= 10000


def test_library_is_sm103a_only_build():
    from adapter_serving_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert os.path.exists(build.LIB)


def test_status_strings():
    L = _lib()
    for code in (0, -1, -2, -3, -5, -6, -7):
        s = L.lib.lora_status_string(code).decode()
        assert s and s != "unknown status"
    assert L.lib.lora_status_string(-99).decode() == "unknown status"


@pytest.mark.parametrize("seed", range(8))
def test_host_segments_bit_exact_vs_oracle(seed):
    L = _lib()
    g = np.random.default_rng(100 + seed)
    n = int(g.integers(0, 400))
    ids = g.integers(-1, int(g.integers(1, 60)), size=n).astype(np.int32)
    got = L.build_segments(ids)
    ref = oracle.segments(ids)
    for a, b in zip(got, ref):
        assert np.array_equal(a, b)


def test_host_argument_checks_without_gpu():
    L = _lib()
    import ctypes
    # null / malformed arguments are rejected before any CUDA call
    assert L.lib.lora_pool_create(None, None) == L.EINVAL
    assert L.lib.lora_build_segments(None, -1, None, None, None, None) == L.EINVAL
    assert L.lib.lora_layer_forward(None, 1, None, None, 4, ctypes.c_float(1.0), 0, None) == L.EINVAL
    assert L.lib.lora_layer_forward_w4(None, 1, None, None, 4, ctypes.c_float(1.0), 0, None) == L.EINVAL
    assert L.lib.lora_layer_forward_planned_w4(None, 1, None, ctypes.c_float(1.0), 0, None) == L.EINVAL
    assert L.lib.lora_layer_forward_planned(None, 0, None, ctypes.c_float(1.0), 0, None) == L.EINVAL
    assert L.lib.lora_quantize_w4(None, 1, 8, None, None) == L.EINVAL
    assert L.lib.lora_pool_destroy(None) == L.EINVAL
    d_in = (ctypes.c_int32 * 1)(1000)
    d_out = (ctypes.c_int32 * 1)(1001)  # not a multiple of 8
    desc = L.lora_pool_desc(1, d_in, d_out, 4, 8, None, 16)
    h = ctypes.c_void_p()
    assert L.lib.lora_pool_create(ctypes.byref(desc), ctypes.byref(h)) == L.EINVAL
    desc = L.lora_pool_desc(1, d_in, d_in, 4, 65, None, 16)  # rank above 64
    assert L.lib.lora_pool_create(ctypes.byref(desc), ctypes.byref(h)) == L.EINVAL


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure path")
def test_pool_create_fails_cleanly_without_gpu():
    L = _lib()
    with pytest.raises(L.LoraError) as e:
        L.Pool([1024], [1024], 4)
    assert e.value.status == L.ECUDA


def test_ring_slot_without_division():
    """The gemm's TMA ring finds fill k's slot and round as k - umulhi(k, ceil(2^32 / S)) * S and
    umulhi(k, ceil(2^32 / S)) for S <= 8 stages: exact for every k below 2^32 / 8 (checked here on
    a dense range and at the top of that range)."""
    for S in range(2, 9):
        m = 0xFFFFFFFF // S + 1
        k = np.arange(0, 1 << 20, dtype=np.uint64)
        q = (k * np.uint64(m)) >> np.uint64(32)
        assert np.array_equal(q, k // np.uint64(S))
        assert np.array_equal(k - q * np.uint64(S), k % np.uint64(S))
        top = np.arange((1 << 29) - (1 << 16), 1 << 29, dtype=np.uint64)
        assert np.array_equal((top * np.uint64(m)) >> np.uint64(32), top // np.uint64(S))


def test_pack_factors_layout():
    """pack_factors: every A at a 16-byte aligned offset, its B right after, bytes unchanged."""
    import torch
    L = pytest.importorskip("adapter_serving_gb300")
    g = np.random.default_rng(0)
    entries = []
    for a, (r, d_in, d_out) in enumerate([(5, 24, 40), (8, 64, 16), (3, 8, 8)]):
        A = g.integers(0, 2**16, (r, d_in), dtype=np.uint16)
        B = g.integers(0, 2**16, (d_out, r), dtype=np.uint16)
        entries.append((a, a % 2, A, B))
    items, blob = L.pack_factors(entries, pin=False)
    raw = blob.numpy()
    for (a, m, A, B), (ia, im, r, ao, bo) in zip(entries, items):
        assert (ia, im, r) == (a, m, A.shape[0]) and ao % 16 == 0 and bo == ao + A.nbytes
        assert np.array_equal(raw[ao:ao + A.nbytes].view(np.uint16).reshape(A.shape), A)
        assert np.array_equal(raw[bo:bo + B.nbytes].view(np.uint16).reshape(B.shape), B)
