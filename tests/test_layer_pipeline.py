"""Adapter loads pipelined across the layers of a forward pass ("12. Adapter Serving and
Multi-Tenant Customization", section "Switching cost: I/O, not compute": a cold adapter's factors
are a copy, so those a later layer needs can arrive while the earlier layers run).

Every layer has its own pool.  At the start of a step the cold adapters' factors are queued layer
by layer on a copy stream (lora_pool_load_many), each layer's loads followed by a gate mark; each
layer's forward (lora_layer_step) waits on its own mark only.  Every layer's output is checked
against the fp64 oracle, step after step, while adapters are evicted and loaded."""
import copy

import numpy as np
import pytest
import torch

import workloads as wl
from harness import check_close, oracle_rows, to_dev_bf16, to_host_bf16

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

N_LAYERS = 8
D, KV = 1024, 256
MODS = {"q": (D, D), "k": (D, KV), "v": (D, KV), "o": (D, D)}
STAGES = [["q", "k", "v"], ["o"]]


def _layers(n_ad, ranks, n_rows):
    return [wl.custom(f"layer{l}", dict(MODS), STAGES, n_rows, ranks, 1.0, seed=100 + l,
                      ids=np.full(n_rows, -1, np.int32)) for l in range(N_LAYERS)]


def _pool(L, w, n_ad):
    names = w.module_names()
    pages = [(16 * int(w.ranks.max()) + 63) // 64 + 2] * len(names)  # room for 16 resident adapters
    return L.Pool([w.modules[m][0] for m in names], [w.modules[m][1] for m in names], n_ad, max_rank=64,
                  pages=pages, max_rows=w.n_rows)


def _factors(w, adapters):
    """Pinned host copies of the factors (the copies are then asynchronous)."""
    return {(a, m): (to_host_bf16(w.A(a, m)).pin_memory(), to_host_bf16(w.B(a, m)).pin_memory())
            for a in adapters for m in w.module_names()}


def test_layer_pipelined_loads_every_layer_matches_the_oracle():
    import adapter_serving_gb300 as L
    n_ad, n_rows = 24, 48
    ranks = np.random.default_rng(7).choice(np.array([8, 16], np.int32), n_ad)
    layers = _layers(n_ad, ranks, n_rows)
    names = layers[0].module_names()
    pools = [_pool(L, w, n_ad) for w in layers]
    fac = [_factors(w, range(20)) for w in layers]
    gate = L.LayerGate(N_LAYERS)
    compute = torch.cuda.current_stream()
    copy_s = torch.cuda.Stream()
    # every layer's inputs and weights on the device before the steps: inside a step only the
    # gate orders the forwards against the loads
    xs = [[to_dev_bf16(w.x(st)) for st in range(len(STAGES))] for w in layers]
    Ws = [{m: to_dev_bf16(w.W(m)) for m in names} for w in layers]
    # adapters 0..7 resident before the first step; each step then evicts four and needs four cold
    # ones, whose factors for a layer come as one packed blob (one copy and one scatter launch)
    for l, pool in enumerate(pools):
        pool.load_many([(a, names.index(m), *fac[l][(a, m)]) for a in range(8) for m in names])
    packs = {(l, step): L.pack_factors([(a, names.index(m), *fac[l][(a, m)])
                                        for a in range(8 + 4 * step, 12 + 4 * step) for m in names])
             for l in range(N_LAYERS) for step in range(3)}
    staging = [torch.empty(max(packs[(l, st)][1].numel() for st in range(3)), dtype=torch.uint8, device="cuda")
               for l in range(N_LAYERS)]
    torch.cuda.synchronize()
    g = np.random.default_rng(9)
    for step in range(3):
        evict = list(range(4 * step - 4, 4 * step)) if step > 0 else []
        cold = list(range(8 + 4 * step, 12 + 4 * step))
        live = np.arange(4 * step, 12 + 4 * step)
        ids = np.where(g.random(n_rows) < 0.1, -1, g.choice(live, n_rows)).astype(np.int32)
        ids[:len(cold)] = cold  # every cold adapter is used
        copy_s.wait_stream(compute)  # evicted pages are reused only after the forwards that read them
        for l, pool in enumerate(pools):
            if evict:
                assert pool.unload_many(evict, stream=copy_s) == len(evict)
            items, blob = packs[(l, step)]
            assert pool.load_packed(items, blob, staging[l], stream=copy_s) == len(cold) * len(names)
            gate.mark(l, copy_s)
        ids_d = torch.from_numpy(ids).cuda()
        outs = []
        for l, (w, pool) in enumerate(zip(layers, pools)):
            ys = {m: torch.full((n_rows, w.modules[m][1]), float("nan"), device="cuda") for m in names}
            stages = [[(names.index(m), xs[l][st], Ws[l][m], ys[m]) for m in STAGES[st]] for st in range(len(STAGES))]
            gate.wait(l, compute)
            pool.layer_step(stages, ids_d, w.scale, stream=compute)
            outs.append(ys)
        torch.cuda.synchronize()
        for l, w in enumerate(layers):
            v = copy.copy(w)
            v.ids = ids
            for m in names:
                check_close(outs[l][m].cpu().double().numpy(), oracle_rows(v, m, 0 if m != "o" else 1),
                            what=f"step {step} layer {l} {m}")
            code, _ = pools[l].last_device_error()
            assert code == 0
    gate.close()
    for pool in pools:
        pool.close()


def test_load_many_equals_single_loads_and_stops_at_a_bad_item():
    import adapter_serving_gb300 as L
    n_ad, n_rows = 70, 64
    ranks = np.random.default_rng(3).choice(np.array([4, 8, 16, 32, 64], np.int32), n_ad)
    w = wl.custom("load_many", {"p": (512, 384)}, [["p"]], n_rows, ranks, 1.5, seed=21,
                  ids=wl.random_ids(n_rows, n_ad, 21, p_base=0.1))
    pages = [(int(ranks.sum()) + 63) // 64 + 70]
    one = L.Pool([512], [384], n_ad, max_rank=64, pages=pages, max_rows=n_rows)
    many = L.Pool([512], [384], n_ad, max_rank=64, pages=pages, max_rows=n_rows)
    f = _factors(w, range(n_ad))
    for a in range(n_ad):
        one.load(a, 0, *f[(a, "p")])
    assert many.load_many([(a, 0, *f[(a, "p")]) for a in range(n_ad)]) == n_ad  # more than one table launch
    x, W = to_dev_bf16(w.x(0)), to_dev_bf16(w.W("p"))
    ids = torch.from_numpy(w.ids).cuda()
    y1 = torch.empty(n_rows, 384, device="cuda")
    y2 = torch.empty(n_rows, 384, device="cuda")
    one.linear_forward(0, x, W, ids, w.scale, y1)
    many.linear_forward(0, x, W, ids, w.scale, y2)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    check_close(y2.cpu().double().numpy(), oracle_rows(w, "p", 0), what="load_many")
    # a bad item (rank 65 > max_rank) stops the call: the items before it are loaded, it and the
    # items after it are not, and the adapter it named keeps its entry
    bad_A = torch.zeros(65, 512, dtype=torch.bfloat16).pin_memory()
    bad_B = torch.zeros(384, 65, dtype=torch.bfloat16).pin_memory()
    items = [(0, 0, *f[(0, "p")]), (1, 0, bad_A, bad_B), (2, 0, *f[(2, "p")])]
    arr = (L.lora_load_item * 3)()
    for i, (a, m, A, B) in enumerate(items):
        arr[i] = L.lora_load_item(a, m, int(A.shape[0]), A.data_ptr(), B.data_ptr())
    done = L.ctypes.c_int32(-1)
    rc = L.lib.lora_pool_load_many(many.handle, 3, arr, L.ctypes.byref(done), L._stream(None))
    assert rc == L.EINVAL and done.value == 1
    many.linear_forward(0, x, W, ids, w.scale, y2)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    one.close()
    many.close()


def test_layer_step_equals_plan_and_planned_calls_bit_for_bit():
    import adapter_serving_gb300 as L
    n_ad, n_rows = 20, 96
    ranks = np.full(n_ad, 16, np.int32)
    w = wl.custom("layer_step", dict(MODS), STAGES, n_rows, ranks, 1.0, seed=5,
                  ids=wl.random_ids(n_rows, n_ad, 5, p_base=0.1))
    names = w.module_names()
    pool = _pool(L, w, n_ad)
    f = _factors(w, w.used_adapters().tolist())
    pool.load_many([(a, names.index(m), *f[(a, m)]) for (a, m) in f])
    x = [to_dev_bf16(w.x(st)) for st in range(len(STAGES))]
    Wd = {m: to_dev_bf16(w.W(m)) for m in names}
    ids = torch.from_numpy(w.ids).cuda()
    a = {m: torch.empty(n_rows, w.modules[m][1], device="cuda") for m in names}
    b = {m: torch.empty(n_rows, w.modules[m][1], device="cuda") for m in names}
    pool.plan_rows(ids)
    for st in range(len(STAGES)):
        pool.layer_forward_planned([(names.index(m), x[st], Wd[m], a[m]) for m in STAGES[st]], w.scale)
    pool.layer_step([[(names.index(m), x[st], Wd[m], b[m]) for m in STAGES[st]] for st in range(len(STAGES))],
                    ids, w.scale)
    torch.cuda.synchronize()
    for m in names:
        assert torch.equal(a[m], b[m]), m
    pool.close()


def test_layer_step_host_moves_inputs_and_outputs_in_one_call():
    """The host-buffer step gives, in pinned host memory, the bits the device step leaves in y."""
    import adapter_serving_gb300 as L
    n_ad, n_rows = 20, 80
    ranks = np.random.default_rng(4).choice(np.array([8, 16, 32], np.int32), n_ad)
    w = wl.custom("layer_step_host", dict(MODS), STAGES, n_rows, ranks, 1.0, seed=8,
                  ids=wl.random_ids(n_rows, n_ad, 8, p_base=0.1))
    names = w.module_names()
    pool = _pool(L, w, n_ad)
    f = _factors(w, w.used_adapters().tolist())
    pool.load_many([(a, names.index(m), *f[(a, m)]) for (a, m) in f])
    Wd = {m: to_dev_bf16(w.W(m)) for m in names}
    for y_dtype in (torch.float32, torch.bfloat16):
        # device reference
        xd = [to_dev_bf16(w.x(st)) for st in range(len(STAGES))]
        ref = {m: torch.empty(n_rows, w.modules[m][1], dtype=y_dtype, device="cuda") for m in names}
        pool.layer_step([[(names.index(m), xd[st], Wd[m], ref[m]) for m in STAGES[st]] for st in range(len(STAGES))],
                        torch.from_numpy(w.ids).cuda(), w.scale)
        # host in, host out: the device buffers start as garbage
        ids_d = torch.full((n_rows,), 12345, dtype=torch.int32, device="cuda")
        xb = [torch.zeros_like(x) for x in xd]
        yb = {m: torch.full_like(ref[m], float("nan")) for m in names}
        hid = torch.from_numpy(w.ids).pin_memory()
        hx = [to_host_bf16(w.x(st)).pin_memory() for st in range(len(STAGES))]
        hy = {m: torch.full(ref[m].shape, float("nan"), dtype=y_dtype).pin_memory() for m in names}
        order = [m for st in STAGES for m in st]
        pool.layer_step_host([[(names.index(m), xb[st], Wd[m], yb[m]) for m in STAGES[st]] for st in range(len(STAGES))],
                             ids_d, hid, hx, [hy[m] for m in order], w.scale)
        pool.host_wait()
        torch.cuda.current_stream().synchronize()
        for m in names:
            assert torch.equal(hy[m], ref[m].cpu()), (m, y_dtype)
    pool.close()


def test_packed_loads_equal_single_loads_and_refuse_bad_items():
    """Ranks that need padding (5, 12, 33) and exact ones (8, 64): one packed blob, one copy, one
    scatter launch, the same bits as single loads; a bad item queues nothing; running out of rows
    stops at that item; unload_many clears every module."""
    import adapter_serving_gb300 as L
    n_ad, n_rows = 30, 64
    ranks = np.random.default_rng(5).choice(np.array([5, 8, 12, 33, 64], np.int32), n_ad)
    w = wl.custom("packed", {"p": (512, 384), "r": (256, 1024)}, [["p"], ["r"]], n_rows, ranks, 1.5, seed=31,
                  ids=wl.random_ids(n_rows, n_ad, 31, p_base=0.1))
    names = w.module_names()
    pages = [(n_ad * 64) // 64 + 2] * 2
    one = L.Pool([512, 256], [384, 1024], n_ad, max_rank=64, pages=pages, max_rows=n_rows)
    packed = L.Pool([512, 256], [384, 1024], n_ad, max_rank=64, pages=pages, max_rows=n_rows)
    f = _factors(w, range(n_ad))
    for (a, m), (A, B) in f.items():
        one.load(a, names.index(m), A, B)
    items, blob = L.pack_factors([(a, names.index(m), A, B) for (a, m), (A, B) in f.items()])
    staging = torch.empty(blob.numel(), dtype=torch.uint8, device="cuda")
    assert packed.load_packed(items, blob, staging) == len(items)  # more than one scatter launch
    ids = torch.from_numpy(w.ids).cuda()
    for st, m in enumerate(names):
        x, W = to_dev_bf16(w.x(st)), to_dev_bf16(w.W(m))
        y1 = torch.empty(n_rows, w.modules[m][1], device="cuda")
        y2 = torch.empty_like(y1)
        one.linear_forward(st, x, W, ids, w.scale, y1)
        packed.linear_forward(st, x, W, ids, w.scale, y2)
        torch.cuda.synchronize()
        assert torch.equal(y1, y2), m
        check_close(y2.cpu().double().numpy(), oracle_rows(w, m, st), what=f"packed/{m}")
    # an offset past the blob: EINVAL and nothing loaded (adapter 0 keeps its factors)
    bad = [(0, 0, int(ranks[0]), 0, blob.numel())]
    with pytest.raises(L.LoraError):
        packed.load_packed(bad, blob, staging)
    assert packed.query(0, 0)[0] == int(ranks[0])
    # unload_many, then a pool too small: the load stops at the first item that finds no rows
    assert packed.unload_many(list(range(n_ad))) == n_ad
    small = L.Pool([512, 256], [384, 1024], n_ad, max_rank=64, pages=[1, 1], max_rows=n_rows)
    items64 = [(a, 0, 64, 0, 0) for a in range(3)]
    blob64 = torch.zeros(64 * 512 * 2 + 384 * 64 * 2, dtype=torch.uint8).pin_memory()
    done = L.ctypes.c_int32(-1)
    arr = (L.lora_packed_item * 3)(*[L.lora_packed_item(a, m, r, 0, ao, 64 * 512 * 2) for a, m, r, ao, _ in items64])
    st64 = torch.empty(blob64.numel(), dtype=torch.uint8, device="cuda")
    rc = L.lib.lora_pool_load_packed(small.handle, 3, arr, blob64.data_ptr(), st64.data_ptr(), blob64.numel(),
                                     L.ctypes.byref(done), L._stream(None))
    assert rc == L.ENOMEM and done.value == 1
    torch.cuda.synchronize()
    one.close()
    packed.close()
    small.close()
