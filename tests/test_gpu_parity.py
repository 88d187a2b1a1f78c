"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded
inputs.  Bar: max-abs <= 2e-2 and rel-L2 <= 1e-3 on fp32 outputs (bf16 inputs, fp32
accumulate); bf16 outputs within 1 bf16 ulp of the oracle rounded to bf16; the row grouping
(gather / segment indices) bit-exact.  Small cases are checked on every output; the
full-size workloads on sampled rows the oracle computes one by one."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from harness import (bf16_gate, check_close, make_pool, oracle_rows, run_stage, to_dev_bf16, to_host_bf16)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _check_all(w, pool, factors, stages=None, rows=None, y_dtype=torch.float32, segments=False, ids=None):
    """Run every stage and compare each module with the oracle on ``rows`` (all rows if None)."""
    for st in (range(len(w.stages)) if stages is None else stages):
        x_bits = w.x(st)
        W_bits = {m: w.W(m) for m in w.stages[st]}
        outs = run_stage(pool, w, st, x_bits=x_bits, W_bits=W_bits, y_dtype=y_dtype, ids=ids, segments=segments)
        for m in w.stages[st]:
            wv = w if ids is None else _with_ids(w, ids)
            ref = oracle_rows(wv, m, st, rows=rows, x_bits=x_bits, W_bits=W_bits[m], factors=factors)
            y = outs[m].float().cpu().numpy().astype(np.float64)
            # every output is written (y starts as NaN), whichever rows the oracle checks
            assert np.all(np.isfinite(y)), f"{w.name}/{m}: outputs left unwritten"
            if rows is not None:
                y = y[np.asarray(rows)]
            if y_dtype == torch.float32:
                check_close(y, ref, what=f"{w.name}/{m}")
            else:
                yb = outs[m].view(torch.int16).cpu().numpy().view(np.uint16)
                if rows is not None:
                    yb = yb[np.asarray(rows)]
                bad = bf16_gate(yb, ref)
                assert len(bad) == 0, f"{w.name}/{m}: bf16 outputs off at {bad[:4].tolist()}"


def _with_ids(w, ids):
    import copy
    v = copy.copy(w)
    v.ids = np.asarray(ids, np.int32)
    return v


# ------------------------------------------------------------------ small, every output ---

def test_tiny_workload_all_outputs():
    w = wl.tiny()
    pool, f = make_pool(w)
    _check_all(w, pool, f)
    _check_all(w, pool, f, y_dtype=torch.bfloat16)
    assert pool.last_device_error() == (0, 0)


def _reduced_attn(n=100, n_ad=64, ranks=8, d=1024, kv=256, seed=3, p_base=0.1):
    ids = wl.random_ids(n, n_ad, seed, p_base=p_base)
    r = np.full(n_ad, ranks, np.int32) if np.isscalar(ranks) else np.asarray(ranks, np.int32)
    return wl.custom("reduced_attn", {"q": (d, d), "k": (d, kv), "v": (d, kv), "o": (d, d)},
                     [["q", "k", "v"], ["o"]], n, r, 1.0, seed=seed, ids=ids)


def test_bounded_waits_run_out_cleanly_and_the_next_call_is_correct():
    """A wait budget of 100 ns is far below one TMA round trip, so the first wait of every gemm CTA
    gives up: it records LORA_DEVERR_TIMEOUT, the CTA stops issuing, waits for the copies and MMAs
    it already issued, frees its tensor memory and returns.  Nothing hangs or faults.  With the
    default budget back, the next calls (which allocate tensor memory again) match the oracle."""
    w = _reduced_attn(n=48, n_ad=12, seed=41)
    pool, f = make_pool(w)
    pool.set_wait_budget(100)
    for st in range(len(w.stages)):
        run_stage(pool, w, st)  # outputs undefined
    code, _ = pool.last_device_error()
    assert code == 3, f"expected an in-kernel wait timeout, got device error {code}"
    pool.set_wait_budget(0)
    for _ in range(2):
        _check_all(w, pool, f)
    code, _ = pool.last_device_error()
    assert code == 0
    pool.close()


def test_reduced_attention_layer_ragged_batch():
    w = _reduced_attn()
    pool, f = make_pool(w)
    _check_all(w, pool, f)


@pytest.mark.parametrize("n", [1, 15, 16, 17, 128, 255, 256])
def test_batch_sizes(n):
    w = _reduced_attn(n=n, n_ad=12, seed=n)
    pool, f = make_pool(w)
    _check_all(w, pool, f, stages=[0])


def test_ragged_dims_mixed_ranks():
    """d_in, d_out not multiples of the tile sizes; ranks 3, 8, 13, 40, 64 (storage 8..64)."""
    ranks = np.array([3, 8, 13, 40, 64, 1], np.int32)
    ids = wl.random_ids(37, len(ranks), 11, p_base=0.15)
    w = wl.custom("ragged", {"a": (1000, 328), "b": (1000, 136)}, [["a", "b"]], 37, ranks, -0.7, seed=5, ids=ids)
    pool, f = make_pool(w)
    _check_all(w, pool, f)
    _check_all(w, pool, f, y_dtype=torch.bfloat16)


def test_shared_adapters_segments_bit_exact():
    """Few adapters, many rows each: the device grouping must equal the oracle's exactly."""
    ids = wl.random_ids(200, 5, 21, p_base=0.2)
    w = wl.custom("shared", {"p": (512, 384)}, [["p"]], 200, [16, 8, 64, 32, 8], 1.25, seed=8, ids=ids)
    pool, f = make_pool(w)
    _check_all(w, pool, f)
    perm, ss, sa = pool.last_segments()
    rperm, rss, rsa = oracle.segments(ids)
    assert np.array_equal(perm, rperm) and np.array_equal(ss, rss) and np.array_equal(sa, rsa)


def test_grouped_rows_prefill_path():
    """n > 256: contiguous segments (chunked tcgen05 path), several segments per chunk."""
    lens = np.array([300, 17, 129, 1, 64, 500, 90])
    ss = np.zeros(len(lens) + 1, np.int32)
    ss[1:] = np.cumsum(lens)
    sa = np.array([4, -1, 0, 2, 2, 1, 3], np.int32)
    w = wl.custom("grouped", {"q": (768, 512), "g": (768, 640)}, [["q", "g"]], int(ss[-1]),
                  [16, 16, 8, 32, 16], 1.0, seed=9, seg_start=ss, seg_adapter=sa)
    pool, f = make_pool(w)
    _check_all(w, pool, f, segments=True)
    _, gss, gsa = pool.last_segments()
    assert np.array_equal(gss, ss) and np.array_equal(gsa, sa)


def test_segment_api_small_batch_uses_decode_path():
    ss = np.array([0, 5, 9, 40], np.int32)
    sa = np.array([1, 0, -1], np.int32)
    w = wl.custom("segsmall", {"q": (256, 256)}, [["q"]], 40, [8, 16], 0.5, seed=4, seg_start=ss, seg_adapter=sa)
    pool, f = make_pool(w)
    _check_all(w, pool, f, segments=True)


# -------------------------------------------------------------------------- invariants -----

def test_b_zero_is_bit_identical_to_base_only():
    """B = 0 adds exact zeros, and the split of W's k-range over the CTAs does not depend on the
    adapters of the batch, so the output equals the base-only output bit for bit."""
    w = _reduced_attn(n=64, n_ad=8, seed=30, p_base=0.0)
    pool, f = make_pool(w, factors={(a, m): (w.A(a, m), np.zeros_like(w.B(a, m)))
                                    for a in range(8) for m in w.module_names()})
    y_lora = run_stage(pool, w, 0)
    y_base = run_stage(pool, w, 0, ids=np.full(w.n_rows, -1, np.int32))
    for m in w.stages[0]:
        assert torch.equal(y_lora[m], y_base[m]), m


def test_deterministic_and_row_permutation():
    w = _reduced_attn(n=96, n_ad=20, seed=31)
    pool, f = make_pool(w)
    x = w.x(0)
    a = run_stage(pool, w, 0, x_bits=x)
    b = run_stage(pool, w, 0, x_bits=x)
    for m in a:
        assert torch.equal(a[m], b[m])
    p = np.random.default_rng(0).permutation(w.n_rows)
    c = run_stage(pool, w, 0, x_bits=x[p], ids=w.ids[p])
    for m in a:
        assert torch.equal(c[m], a[m][torch.from_numpy(p).cuda()]), m


def test_graph_replay_sees_reloaded_adapter():
    """Factor addresses come from the device table, so a captured graph follows a reload."""
    w = _reduced_attn(n=32, n_ad=4, seed=32, p_base=0.0)
    pool, f = make_pool(w)
    names = w.module_names()
    x = to_dev_bf16(w.x(1))
    Wd = to_dev_bf16(w.W("o"))
    y = torch.zeros(w.n_rows, w.modules["o"][1], device="cuda")
    ids = torch.from_numpy(w.ids).cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pool.layer_forward([(names.index("o"), x, Wd, y)], ids, w.scale)  # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pool.layer_forward([(names.index("o"), x, Wd, y)], ids, w.scale)
    g.replay()
    torch.cuda.synchronize()
    ref = oracle_rows(w, "o", 1, factors=f)
    check_close(y.cpu().numpy(), ref, what="graph")
    # reload adapter ids[0] with new factors, replay the same graph
    a0 = int(w.ids[0])
    g2 = np.random.default_rng(5)
    A_new = wl.f32_to_bf16_bits(g2.standard_normal((8, 1024)).astype(np.float32) / 32)
    B_new = wl.f32_to_bf16_bits(g2.standard_normal((1024, 8)).astype(np.float32) / 3)
    pool.load(a0, names.index("o"), to_host_bf16(A_new), to_host_bf16(B_new))
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    f2 = dict(f)
    f2[(a0, "o")] = (A_new, B_new)
    ref2 = oracle_rows(w, "o", 1, factors=f2)
    check_close(y.cpu().numpy(), ref2, what="graph after reload")
    assert np.abs(ref2 - ref).max() > 1e-2  # the reload really changed the answer


# ----------------------------------------------------------------------- error paths -----

def test_bad_and_unloaded_ids_are_reported_and_served_base_only():
    w = _reduced_attn(n=24, n_ad=6, seed=33, p_base=0.0)
    pool, f = make_pool(w, adapters=[0, 1, 2, 3])  # 4 and 5 are not resident
    ids = w.ids.copy()
    ids[3] = 4            # not loaded
    ids[7] = 99           # out of range
    ids[8] = -5           # out of range
    out = run_stage(pool, w, 0, ids=ids)
    code, detail = pool.last_device_error()
    assert code in (1, 2)
    fixed = ids.copy()
    fixed[[3, 7, 8]] = -1
    fixed[fixed >= 4] = -1
    ref = oracle_rows(_with_ids(w, fixed), "q", 0, factors=f)
    check_close(out["q"].cpu().numpy(), ref, what="bad ids")
    assert pool.last_device_error() == (0, 0)  # reading clears it


def test_pool_capacity_rank_and_reload_accounting():
    import adapter_serving_gb300 as L
    pool = L.Pool([256], [128], 10, max_rank=32, pages=[1], max_rows=16)
    assert pool.free_rows(0) == 64
    A = lambda r: to_host_bf16(np.zeros((r, 256), np.uint16))
    B = lambda r: to_host_bf16(np.zeros((128, r), np.uint16))
    pool.load(0, 0, A(32), B(32))
    pool.load(1, 0, A(8), B(8))
    pool.load(2, 0, A(16), B(16))
    assert pool.free_rows(0) == 8
    with pytest.raises(L.LoraError) as e:
        pool.load(3, 0, A(16), B(16))
    assert e.value.status == L.ENOMEM
    with pytest.raises(L.LoraError) as e:
        pool.load(3, 0, A(33), B(33))  # above max_rank
    assert e.value.status == L.EINVAL
    pool.load(3, 0, A(5), B(5))        # rank 5 -> 8 storage rows
    assert pool.free_rows(0) == 0
    assert pool.query(3, 0)[0] == 5
    pool.unload(0)
    pool.unload(2)
    assert pool.free_rows(0) == 48
    with pytest.raises(L.LoraError) as e:
        pool.unload(2)
    assert e.value.status == L.ENOTLOADED
    pool.load(0, 0, A(32), B(32))      # buddies merged back: a 32-row run is free again
    assert pool.free_rows(0) == 16
    torch.cuda.synchronize()


def test_empty_batch_is_a_no_op():
    w = _reduced_attn(n=4, n_ad=2, seed=34)
    pool, f = make_pool(w)
    y = torch.full((0, 1024), 1.0, device="cuda")
    x = torch.zeros((0, 1024), dtype=torch.bfloat16, device="cuda")
    Wd = to_dev_bf16(w.W("q"))
    pool.layer_forward([(0, x, Wd, y)], torch.zeros(0, dtype=torch.int32, device="cuda"), 1.0)
    torch.cuda.synchronize()


# ------------------------------------------------------------- full-size workloads -----

def _sample_rows(n, k, seed):
    g = np.random.default_rng(seed)
    return np.sort(g.choice(n, size=min(k, n), replace=False))


def _rows_by_rank(w, k, seed):
    """About k rows, spread over every rank class the batch uses (base-only rows count as one
    class) and over the batch: each class gives its first and last row and evenly spaced ones."""
    ids = w.row_adapters()
    rk = np.where(ids >= 0, w.ranks[np.maximum(ids, 0)], 0)
    classes = np.unique(rk)
    per = max(2, k // len(classes))
    out = []
    for c in classes:
        idx = np.flatnonzero(rk == c)
        out.extend(idx[np.linspace(0, len(idx) - 1, min(per, len(idx))).round().astype(int)])
    return np.unique(np.concatenate([np.array(out, np.int64), _sample_rows(w.n_rows, 4, seed)]))


def test_attn70b_decode_full_size_all_rows():
    w = wl.attn70b_decode()
    pool, f = make_pool(w)
    _check_all(w, pool, f)  # every row and every output
    perm, ss, sa = pool.last_segments()
    rp, rss, rsa = oracle.segments(w.ids)
    assert np.array_equal(perm, rp) and np.array_equal(ss, rss) and np.array_equal(sa, rsa)


def test_all70b_decode_full_size_sampled():
    w = wl.all70b_decode()
    pool, f = make_pool(w)
    _check_all(w, pool, f, rows=np.arange(0, w.n_rows, 4) + (np.arange(0, w.n_rows, 4) // 4) % 4)


def test_zipf_pool_5000_adapters_sampled():
    w = wl.zipf_pool()
    adapters = np.arange(w.n_adapters)
    names = w.module_names()
    pages = [(sum(int(r) for r in w.ranks) + 63) // 64 + 8] * len(names)
    used = set(w.used_adapters().tolist())
    f = {}
    import adapter_serving_gb300 as L
    pool = L.Pool([w.modules[m][0] for m in names], [w.modules[m][1] for m in names], w.n_adapters,
                  max_rank=64, pages=pages, max_rows=w.n_rows)
    for a in adapters:
        for mi, m in enumerate(names):
            A, B = w.A(int(a), m), w.B(int(a), m)
            if int(a) in used:
                f[(int(a), m)] = (A, B)
            pool.load(int(a), mi, to_host_bf16(A), to_host_bf16(B))
    torch.cuda.synchronize()
    # every rank class, and the first and last row of every 16-row block of the adapter-sorted
    # batch (the finalize's blocks, launched in the prep's order)
    perm_ref, _, _ = oracle.segments(w.ids)
    ends = np.concatenate([np.arange(0, w.n_rows, 16), np.minimum(np.arange(15, w.n_rows + 15, 16), w.n_rows - 1)])
    rows = np.unique(np.concatenate([_rows_by_rank(w, 32, 3), np.asarray(perm_ref)[ends]]))
    assert len(rows) >= 32
    _check_all(w, pool, f, rows=rows)
    perm, ss, sa = pool.last_segments()
    rp, rss, rsa = oracle.segments(w.ids)
    assert np.array_equal(perm, rp) and np.array_equal(ss, rss) and np.array_equal(sa, rsa)


def test_prefill_segments_full_size_sampled():
    w = wl.prefill_segments()
    pool, f = make_pool(w, max_rows=w.n_rows)
    ss = w.seg_start
    rows = np.unique(np.concatenate([ss[:-1], ss[1:] - 1, _sample_rows(w.n_rows, 24, 4)]))
    rows = rows[:: max(1, len(rows) // 48)]
    _check_all(w, pool, f, rows=rows, segments=True)


def test_planned_forward_equals_own_grouping_bit_for_bit():
    """One plan per batch (lora_plan_rows) serves both calls of the layer; the kernels then see the
    same grouping and packs as a call that groups its own rows, so the outputs are identical."""
    import adapter_serving_gb300 as L
    w = _reduced_attn(n=96, n_ad=20, seed=33, p_base=0.15)
    pool, f = make_pool(w)
    own = {}
    for st in range(len(w.stages)):
        own.update(run_stage(pool, w, st))
    names = w.module_names()
    ids = torch.from_numpy(w.ids).cuda()
    pool.plan_rows(ids)
    planned = {}
    for st in range(len(w.stages)):
        x = to_dev_bf16(w.x(st))
        ios = []
        for m in w.stages[st]:
            y = torch.full((w.n_rows, w.modules[m][1]), float("nan"), device="cuda")
            ios.append((names.index(m), x, to_dev_bf16(w.W(m)), y))
            planned[m] = y
        pool.layer_forward_planned(ios, w.scale)
    torch.cuda.synchronize()
    for m in names:
        assert torch.equal(planned[m], own[m]), m
    # the plan ends with a load, and with a call that groups its own rows
    st0 = [(names.index(m), to_dev_bf16(w.x(0)), to_dev_bf16(w.W(m)), planned[m]) for m in w.stages[0]]
    a0 = int(w.used_adapters()[0])
    pool.load(a0, 0, to_host_bf16(f[(a0, names[0])][0]), to_host_bf16(f[(a0, names[0])][1]))
    with pytest.raises(L.LoraError):
        pool.layer_forward_planned(st0, w.scale)
    pool.plan_rows(ids)
    run_stage(pool, w, 0)
    with pytest.raises(L.LoraError):
        pool.layer_forward_planned(st0, w.scale)
    pool.close()
