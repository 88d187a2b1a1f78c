"""Pins for the oracle: each test ties it to something other than itself.

* the pages' printed sizing numbers (tests/golden/sizing_pins.json, cited per value);
* a hand-worked forward with exact small integers (tests/golden/tiny_forward.json);
* exact rational arithmetic (``fractions``) on tiny integer inputs -- brute force;
* special cases that reduce to a plain library matmul: B = 0 is the base layer, one
  adapter for every row equals the merged weight W + s B A ("m07 -- Multi-Adapter (LoRA)
  Serving", section 1, adapters can be merged into the base; section 5, promotion to a
  merged deployment);
* invariants: base-only rows, zero-padding the rank, row permutation, an adapter equals
  the sum of its rank-1 pieces, linearity in the scale;
* the row grouping against Python's stable ``sorted``.
Every test here runs on the CPU only.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads as wl

GOLD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
ATTN = [(8192, 8192), (8192, 1024), (8192, 1024), (8192, 8192)]
MLP = [(8192, 28672), (8192, 28672), (28672, 8192)]


def bits(a):
    """Exact bf16 bits of small floats (the tests only use values bf16 represents exactly)."""
    a32 = np.asarray(a, dtype=np.float32)
    b = wl.f32_to_bf16_bits(a32)
    assert np.array_equal(wl.bf16_bits_to_f32(b), a32), "test value not exact in bf16"
    return b


def f64(b):
    return wl.bf16_bits_to_f32(b).astype(np.float64)


# ---------------------------------------------------------------- the pages' numbers ---

def _pin_value(pid):
    a8 = oracle.adapter_bytes(ATTN, 8, 80)
    a16 = oracle.adapter_bytes(ATTN, 16, 80)
    a64 = oracle.adapter_bytes(ATTN + MLP, 64, 80)
    G = 2 ** 30
    table = {
        "attn_r8_adapter_MB": math.floor(a8 / 1e6),
        "all_r64_adapter_GB_1dp": round(a64 / 1e9, 1),
        "all_r64_adapter_GB_2dp": round(a64 / 1e9, 2),
        "cost_spread_x": math.floor(a64 / a8),
        "attn_r8_pct_of_140GB": round(100 * a8 / 140e9, 2),
        "all_r64_pct_of_140GB": round(100 * a64 / 140e9, 1),
        "extra_decode_pct_b128_attn_r8": round(100 * 128 * a8 / 140e9),
        "extra_decode_pct_b128_all_r64": math.floor(100 * 128 * a64 / 140e9),
        "extra_decode_pct_b64_all_r64": round(100 * 64 * a64 / 140e9, 1),
        "extra_decode_pct_cap32_all_r64": round(100 * 32 * a64 / 140e9),
        "hbm_100_attn_r8_pct_kv": round(100 * 100 * a8 / G / 172.5, 1),
        "hbm_100_attn_r16_pct_kv": round(100 * 100 * a16 / G / 172.5, 1),
        "hbm_100_all_r64_GiB": round(100 * a64 / G),
        "hbm_100_all_r64_pct_kv": 100 * 100 * a64 / G / 172.5,
        "mlp_plus_attn_over_attn_params": round(
            sum(oracle.lora_params(1, i, o) for i, o in ATTN + MLP) / sum(oracle.lora_params(1, i, o) for i, o in ATTN), 1),
        "lora_flop_ratio_pct_r16_8192": round(100 * oracle.lora_flop_ratio(16, 8192, 8192), 2),
        "lora_extra_flops_r16_8192": oracle.lora_extra_flops(16, 8192),
        "base_flops_8192_millions": math.floor(2 * 8192 * 8192 / 1e6),
        "pair_r16_8192_KiB": oracle.adapter_bytes([(8192, 8192)], 16) / 1024,
        "attn_r16_nongqa_80_layers_MiB": oracle.adapter_bytes([(8192, 8192)] * 4, 16, 80) / 2 ** 20,
    }
    return table[pid]


_PINS = json.load(open(os.path.join(GOLD, "sizing_pins.json")))["pins"]


@pytest.mark.parametrize("pin", _PINS, ids=[p["id"] for p in _PINS])
def test_pages_sizing_numbers(pin):
    got = _pin_value(pin["id"])
    if pin["compare"].startswith("abs("):
        assert abs(got - pin["value"]) <= 0.06, (pin["id"], got)
    else:
        assert got == pin["value"], (pin["id"], got, pin["cite"])


def test_config_step_bytes():
    """Per-layer decode-step bytes of the benchmark shapes, from the same formula."""
    attn = wl.attn70b_decode()
    ids = attn.ids
    mods = [attn.modules[m] for m in attn.module_names()]
    assert oracle.base_bytes(mods) == 301_989_888
    assert oracle.step_adapter_bytes(ids, attn.ranks, mods) == 104_857_600
    assert oracle.distinct_adapters(ids) == 128
    full = wl.all70b_decode()
    mods = [full.modules[m] for m in full.module_names()]
    assert oracle.base_bytes(mods) == 1_711_276_032
    assert oracle.step_adapter_bytes(full.ids, full.ranks, mods) == 2_650_800_128
    # shared adapters are read once: a batch where every row uses adapter 3
    assert oracle.step_adapter_bytes(np.full(128, 3), attn.ranks, mods[:4]) == oracle.adapter_bytes(mods[:4], 8)


# ------------------------------------------------------------------ worked example ---

def test_hand_worked_example():
    g = json.load(open(os.path.join(GOLD, "tiny_forward.json")))
    A = [bits(a) for a in g["A"]]
    B = [bits(b) for b in g["B"]]
    y = oracle.adapted_linear(bits(g["x"]), bits(g["W"]), np.array(g["ids"], np.int32), A, B, g["scale"])
    assert np.array_equal(y, np.array(g["y"], np.float64))


def test_bruteforce_exact_rationals():
    """Tiny integer/half-integer inputs: the fp64 oracle must equal exact rational arithmetic."""
    rng = np.random.default_rng(7)
    n, d_in, d_out, n_ad = 5, 6, 4, 3
    ranks = [1, 2, 3]
    vals = lambda *s: rng.integers(-8, 9, size=s) / 2.0
    x, W = vals(n, d_in), vals(d_out, d_in)
    A = [vals(r, d_in) for r in ranks]
    B = [vals(d_out, r) for r in ranks]
    ids = np.array([0, 2, -1, 1, 2], np.int32)
    s = Fraction(3, 2)
    y = oracle.adapted_linear(bits(x), bits(W), ids, [bits(a) for a in A], [bits(b) for b in B], float(s))
    F = lambda v: Fraction(float(v))
    for i in range(n):
        a = ids[i]
        for o in range(d_out):
            exact = sum(F(W[o, k]) * F(x[i, k]) for k in range(d_in))
            if a >= 0:
                t = [sum(F(A[a][j, k]) * F(x[i, k]) for k in range(d_in)) for j in range(ranks[a])]
                exact += s * sum(F(B[a][o, j]) * t[j] for j in range(ranks[a]))
            assert Fraction(y[i, o]) == exact, (i, o)


# ------------------------------------------------------ library special cases -------

def _rand_case(seed, n=24, d_in=96, d_out=80, ranks=(4, 8, 3), p_base=0.2):
    g = np.random.default_rng(seed)
    x = wl.f32_to_bf16_bits(g.standard_normal((n, d_in), dtype=np.float32))
    W = wl.f32_to_bf16_bits(g.standard_normal((d_out, d_in), dtype=np.float32) / np.sqrt(d_in))
    A = [wl.f32_to_bf16_bits(g.standard_normal((r, d_in), dtype=np.float32) / np.sqrt(d_in)) for r in ranks]
    B = [wl.f32_to_bf16_bits(g.standard_normal((d_out, r), dtype=np.float32) / np.sqrt(r)) for r in ranks]
    ids = g.integers(0, len(ranks), size=n).astype(np.int32)
    ids[g.random(n) < p_base] = -1
    return x, W, ids, A, B


def test_b_zero_is_base_layer():
    x, W, ids, A, B = _rand_case(1)
    Bz = [np.zeros_like(b) for b in B]
    y = oracle.adapted_linear(x, W, ids, A, Bz, 2.0)
    ref = f64(x) @ f64(W).T
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_one_adapter_equals_merged_weight():
    x, W, _, A, B = _rand_case(2, p_base=0)
    s = 0.75
    ids = np.full(x.shape[0], 1, np.int32)
    y = oracle.adapted_linear(x, W, ids, A, B, s)
    merged = f64(W) + s * (f64(B[1]) @ f64(A[1]))
    np.testing.assert_allclose(y, f64(x) @ merged.T, rtol=1e-11, atol=1e-12)


def test_mixed_rows_match_their_merged_weight():
    x, W, ids, A, B = _rand_case(3)
    s = -1.25
    y = oracle.adapted_linear(x, W, ids, A, B, s)
    for i, a in enumerate(ids):
        Wa = f64(W) if a < 0 else f64(W) + s * (f64(B[a]) @ f64(A[a]))
        np.testing.assert_allclose(y[i], Wa @ f64(x[i]), rtol=1e-11, atol=1e-12)


def test_shrink_matches_matmul():
    x, W, ids, A, B = _rand_case(4, p_base=0)
    y, t = oracle.adapted_linear(x, W, ids, A, B, 1.0, return_t=True)
    for i, a in enumerate(ids):
        r = A[a].shape[0]
        np.testing.assert_allclose(t[i, :r], f64(A[a]) @ f64(x[i]), rtol=1e-12, atol=1e-13)
        assert np.all(t[i, r:] == 0)


# ---------------------------------------------------------------- invariants --------

def test_base_only_rows():
    x, W, ids, A, B = _rand_case(5)
    ids[:] = -1
    y = oracle.adapted_linear(x, W, ids, A, B, 3.0)
    assert np.array_equal(y, oracle.adapted_linear(x, W, ids, A, [np.zeros_like(b) for b in B], 3.0))
    np.testing.assert_allclose(y, f64(x) @ f64(W).T, rtol=1e-12)


def test_zero_padding_rank_changes_nothing():
    x, W, ids, A, B = _rand_case(6)
    y = oracle.adapted_linear(x, W, ids, A, B, 1.5)
    Ap = [np.concatenate([a, np.zeros((64 - a.shape[0], a.shape[1]), np.uint16)]) for a in A]
    Bp = [np.concatenate([b, np.zeros((b.shape[0], 64 - b.shape[1]), np.uint16)], axis=1) for b in B]
    assert np.array_equal(y, oracle.adapted_linear(x, W, ids, Ap, Bp, 1.5))


def test_row_permutation():
    x, W, ids, A, B = _rand_case(7)
    p = np.random.default_rng(0).permutation(len(ids))
    y = oracle.adapted_linear(x, W, ids, A, B, 1.0)
    yp = oracle.adapted_linear(x[p], W, ids[p], A, B, 1.0)
    assert np.array_equal(yp, y[p])
    # selecting rows computes exactly those rows
    sel = np.array([3, 0, 17])
    assert np.array_equal(oracle.adapted_linear(x, W, ids, A, B, 1.0, rows=sel), y[sel])


def test_adapter_is_sum_of_rank_one_pieces():
    x, W, ids, A, B = _rand_case(8, p_base=0)
    s = 2.0
    base = oracle.adapted_linear(x, W, np.full_like(ids, -1), A, B, s)
    y = oracle.adapted_linear(x, W, ids, A, B, s)
    acc = np.zeros_like(y)
    for j in range(max(a.shape[0] for a in A)):
        A1 = [a[j:j + 1] if j < a.shape[0] else np.zeros((1, a.shape[1]), np.uint16) for a in A]
        B1 = [b[:, j:j + 1] if j < b.shape[1] else np.zeros((b.shape[0], 1), np.uint16) for b in B]
        acc += oracle.adapted_linear(x, W, ids, A1, B1, s) - base
    np.testing.assert_allclose(y - base, acc, rtol=1e-9, atol=1e-11)


def test_linear_in_scale():
    x, W, ids, A, B = _rand_case(9)
    base = oracle.adapted_linear(x, W, ids, A, B, 0.0)
    d1 = oracle.adapted_linear(x, W, ids, A, B, 1.0) - base
    d3 = oracle.adapted_linear(x, W, ids, A, B, -3.0) - base
    np.testing.assert_allclose(d3, -3.0 * d1, rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(base, f64(x) @ f64(W).T, rtol=1e-12)


def test_invalid_ids_rejected():
    x, W, ids, A, B = _rand_case(10)
    ids[0] = len(A)
    with pytest.raises(ValueError):
        oracle.adapted_linear(x, W, ids, A, B, 1.0)
    ids[0] = -2
    with pytest.raises(ValueError):
        oracle.adapted_linear(x, W, ids, A, B, 1.0)


# ---------------------------------------------------------------- row grouping ------

@pytest.mark.parametrize("seed", range(6))
def test_segments_stable_sort(seed):
    g = np.random.default_rng(seed)
    n = int(g.integers(1, 300))
    ids = g.integers(-1, int(g.integers(1, 40)), size=n).astype(np.int32)
    perm, seg_start, seg_adapter = oracle.segments(ids)
    ref = sorted(range(n), key=lambda i: int(ids[i]))  # Python's sort is stable
    assert perm.tolist() == ref
    uniq = sorted(set(ids.tolist()))
    assert seg_adapter.tolist() == uniq
    assert seg_start[0] == 0 and seg_start[-1] == n
    for s, a in enumerate(seg_adapter):
        assert np.all(ids[perm[seg_start[s]:seg_start[s + 1]]] == a)


def test_segments_edge_cases():
    for ids in ([], [5], [-1, -1], [3, 3, 3], [2, 1, 0]):
        ids = np.array(ids, np.int32)
        perm, ss, sa = oracle.segments(ids)
        assert perm.tolist() == sorted(range(len(ids)), key=lambda i: int(ids[i]))
        assert ss[-1] == len(ids) and len(sa) == len(set(ids.tolist()))


# ---------------------------------------------------------- input generation --------

def test_bf16_rounding_matches_torch():
    g = np.random.default_rng(0)
    a = np.concatenate([g.standard_normal(100_000).astype(np.float32) * 10,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 3.0e38, -1e-40, 65504.0], np.float32)])
    ours = wl.f32_to_bf16_bits(a)
    ref = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_generators_are_reproducible():
    w = wl.tiny()
    assert np.array_equal(w.W("proj"), wl.tiny().W("proj"))
    assert w.W("proj").shape == (1024, 1024) and w.A(1, "proj").shape == (8, 1024) and w.B(1, "proj").shape == (1024, 8)
    big = wl.normal_bf16([0, 9], (1 << 22) * 2 + 5, 1.0)
    assert np.array_equal(big, wl.normal_bf16([0, 9], (1 << 22) * 2 + 5, 1.0))
    v = wl.bf16_bits_to_f32(big).astype(np.float64)
    assert abs(v.mean()) < 2e-3 and abs(v.std() - 1) < 2e-3
    z = wl.zipf_pool()
    assert z.ids.min() >= 0 and z.ids.max() < 5000 and len(z.ids) == 256
    assert set(np.unique(z.ranks).tolist()) <= {8, 16, 32, 64}
    p = wl.prefill_segments()
    lens = np.diff(p.seg_start)
    assert len(lens) == 64 and lens.min() >= 128 and lens.max() <= 2048


def test_bf16_output_gate():
    """The bf16 output gate: 1 ulp of the oracle rounded to bf16, or 2^-13 absolute where the
    oracle is below 2^-6 in magnitude."""
    from harness import bf16_gate
    ref = np.array([1.0, -3.0, 0.25, 1e-4, -2e-3, 0.5])
    bits = wl.f32_to_bf16_bits(ref.astype(np.float32))
    assert len(bf16_gate(bits, ref)) == 0
    one_up = bits.copy()
    one_up[0] += 1                      # 1 ulp above 1.0: allowed
    assert len(bf16_gate(one_up, ref)) == 0
    two_up = bits.copy()
    two_up[1] += 2                      # 2 ulps off at -3.0: refused
    assert bf16_gate(two_up, ref).ravel().tolist() == [1]
    tiny = bits.copy()
    tiny[3] += 3                        # 3 ulps off at 1e-4, but 3 * 2^-21 < 2^-13: allowed
    assert len(bf16_gate(tiny, ref)) == 0
    far = wl.f32_to_bf16_bits(np.array([1e-4 + 2 ** -12], np.float32))
    assert bf16_gate(far, ref[3:4]).ravel().tolist() == [0]   # 2^-12 off near zero: refused
