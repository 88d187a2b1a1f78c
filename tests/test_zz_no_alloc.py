"""The allocation-free entry point, lora_linear_forward_static, called through the C ABI.

It exists for callers that cannot call cudaMalloc (a runtime that already owns all device
memory, or a framework that forbids raw allocations): they pass their adapters as stacked
buffers and the call keeps its scratch in a fixed device array inside the library.  Its
output must match the pooled entry point, lora_linear_forward, on the same inputs within the
parity tolerance, on two calls in a row (the second call runs on whatever the first left in
the shared scratch), and the fp64 oracle's.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import copy

import workloads as wl
from harness import check_close, make_pool, oracle_rows, to_dev_bf16

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _oracle(w, x_bits, ids):
    """The oracle's y for these rows: ids outside [-1, n_adapters) stand for base only."""
    v = copy.copy(w)
    v.ids = np.where(np.asarray(ids) >= w.n_adapters, -1, np.asarray(ids)).astype(np.int32)
    v.n_rows = len(ids)
    return oracle_rows(v, "p", 0, x_bits=x_bits)


def _static_forward(L, x, W, ids, A_stack, B_stack, n_adapters, rank, scale, y):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.lib.lora_linear_forward_static(x.data_ptr(), W.data_ptr(), x.shape[1], W.shape[0], ids.data_ptr(),
                                          ids.numel(), A_stack.data_ptr(), B_stack.data_ptr(), n_adapters, rank,
                                          ctypes.c_float(scale), y.data_ptr(), L.DTYPE_F32, stream)
    assert rc == L.OK, (rc, L.lib.lora_last_cuda_error())


@pytest.mark.parametrize("rank", [8, 64])
def test_static_entry_point_matches_pooled_entry_point(rank):
    import adapter_serving_gb300 as L
    n_ad, d_in, d_out = 24, 1024, 768
    names = ["p"]
    w = wl.custom("noalloc", {"p": (d_in, d_out)}, [names], 100, np.full(n_ad, rank, np.int32), 1.5, seed=40,
                  ids=wl.random_ids(100, n_ad, 40, p_base=0.1))
    pool, factors = make_pool(w, adapters=range(n_ad))
    A_stack = to_dev_bf16(np.stack([factors[(a, "p")][0] for a in range(n_ad)]))
    B_stack = to_dev_bf16(np.stack([factors[(a, "p")][1] for a in range(n_ad)]))
    W = to_dev_bf16(w.W("p"))
    for call in range(2):
        n = 100 if call == 0 else 37  # the second call reuses the scratch the first one left
        x_bits = wl.normal_bf16([41, call], n * d_in, 1.0).reshape(n, d_in)
        x = to_dev_bf16(x_bits)
        ids_h = wl.random_ids(n, n_ad, 50 + call, p_base=0.1)
        ids = torch.from_numpy(ids_h).cuda()
        y_ref = torch.full((n, d_out), float("nan"), device="cuda")
        y_st = torch.full((n, d_out), float("nan"), device="cuda")
        pool.linear_forward(0, x, W, ids, w.scale, y_ref)
        _static_forward(L, x, W, ids, A_stack, B_stack, n_ad, rank, w.scale, y_st)
        torch.cuda.synchronize()
        check_close(y_st.cpu().numpy(), y_ref.cpu().numpy(), what=f"static call {call}")
        check_close(y_st.cpu().numpy(), _oracle(w, x_bits, ids_h), what=f"static call {call} vs oracle")


def test_static_entry_point_matches_the_oracle_on_ragged_shapes():
    """Rank 16, d_in not a multiple of 64, d_out = 776 (six full 128-row tiles and a ragged one),
    61 rows with base-only rows and two ids at or above n_adapters (served base only), two calls."""
    import adapter_serving_gb300 as L
    n_ad, d_in, d_out, n = 20, 1000, 776, 61
    ids = wl.random_ids(n, n_ad, 61, p_base=0.15).copy()
    ids[5], ids[40] = n_ad, n_ad + 7
    w = wl.custom("noalloc_ragged", {"p": (d_in, d_out)}, [["p"]], n, np.full(n_ad, 16, np.int32), 1.25, seed=61,
                  ids=np.where(ids >= n_ad, -1, ids).astype(np.int32))
    A_stack = to_dev_bf16(np.stack([w.A(a, "p") for a in range(n_ad)]))
    B_stack = to_dev_bf16(np.stack([w.B(a, "p") for a in range(n_ad)]))
    x = to_dev_bf16(w.x(0))
    W = to_dev_bf16(w.W("p"))
    ref = _oracle(w, w.x(0), ids)
    for call in range(2):
        y = torch.full((n, d_out), float("nan"), device="cuda")
        _static_forward(L, x, W, torch.from_numpy(ids).cuda(), A_stack, B_stack, n_ad, 16, w.scale, y)
        torch.cuda.synchronize()
        check_close(y.cpu().numpy(), ref, what=f"static ragged call {call}")


def test_static_entry_point_rejects_sizes_beyond_its_scratch():
    import adapter_serving_gb300 as L
    x = torch.zeros((129, 64), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(129, dtype=torch.int32, device="cuda")
    A = torch.zeros((1, 8, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((1, 64, 8), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((129, 64), device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.lib.lora_linear_forward_static(x.data_ptr(), W.data_ptr(), 64, 64, ids.data_ptr(), 129, A.data_ptr(),
                                          B.data_ptr(), 1, 8, ctypes.c_float(1.0), y.data_ptr(), L.DTYPE_F32, stream)
    assert rc == L.EUNSUPPORTED
    assert b"static scratch" in L.lib.lora_last_cuda_error()
