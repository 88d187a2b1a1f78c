"""int8 adapter factors ("m07 -- Multi-Adapter (LoRA) Serving", section 9 "Bottlenecks and
Evolution", item 3: adapters tolerate int8 better than base weights; half the bytes).

Codes are symmetric with one fp32 scale per rank row of A and per rank row of B transposed, so
both of a rank index's scales fold into t_j and the expand only converts codes.

* the oracle's quantizer against what rounding to the nearest code means (exact rationals), its
  error bound and its special cases; the library's quantizer against the oracle bit for bit;
* the oracle's forward on fp64 factors against the pinned C oracle on bf16 factors;
* (GPU) int8 pools through the same decode path, against the fp64 forward on the dequantised
  factors; a zero B is bit-identical to the base-only layer; the calls an int8 pool refuses.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wl

ATTN = [(8192, 8192), (8192, 1024), (8192, 1024), (8192, 8192)]


def _rows(seed, rows, cols):
    g = np.random.default_rng(seed)
    v = g.standard_normal((rows, cols)).astype(np.float32)
    v *= g.choice(np.array([1e-3, 0.07, 1.0, 300.0], np.float32), (rows, 1))
    return wl.f32_to_bf16_bits(v)


def _f32(bits):
    return wl.bf16_bits_to_f32(bits)


@pytest.mark.parametrize("seed", range(3))
def test_oracle_quantizer_rounds_to_the_nearest_code(seed):
    bits = _rows(seed, 6, 257)
    bits[1] = 0
    codes, scale = oracle.quantize_rows_int8(bits)
    v = _f32(bits)
    assert codes.dtype == np.int8 and scale.dtype == np.float32
    assert np.all(codes[1] == 0) and scale[1] == 0
    for r in range(len(bits)):
        if scale[r] == 0:
            continue
        m = np.abs(v[r]).max()
        # the scale is max/127 rounded once to fp32
        assert abs(Fraction(float(scale[r])) - Fraction(float(m)) / 127) <= Fraction(float(scale[r])) * Fraction(1, 2**23)
        assert np.abs(codes[r]).max() == 127 and np.all(np.abs(codes[r]) <= 127)
        s = Fraction(float(scale[r]))
        for c in range(v.shape[1]):
            e = Fraction(float(v[r, c])) / s        # the exact quotient
            k = int(codes[r, c])
            # nearest code; at an exact-quotient distance below 2^-18 from a half-integer the single
            # fp32 rounding of the quotient may go either way
            assert abs(e - k) <= Fraction(1, 2) + Fraction(1, 2**18)
            if abs(abs(e - int(e)) - Fraction(1, 2)) > Fraction(1, 2**18) and abs(e) < 127:
                assert k == round(e)
        # dequantised error bound: half a step (plus the quotient's rounding)
        assert np.all(np.abs(codes[r].astype(np.float64) * float(scale[r]) - v[r]) <= float(scale[r]) * (0.5 + 2**-17))


def test_oracle_quantizer_signs_and_exact_multiples():
    """Values that are exact multiples of the step come back exactly; signs are kept."""
    v = np.array([[127.0, -64.0, 32.0, 1.0, -1.0, 0.0, 96.0, -127.0]], np.float32)
    codes, scale = oracle.quantize_rows_int8(wl.f32_to_bf16_bits(v))
    assert scale[0] == 1.0
    assert codes[0].tolist() == [127, -64, 32, 1, -1, 0, 96, -127]


def test_oracle_dequantize_rows_int8_hand_worked():
    """Each code times its own row's scale, exactly in fp64.  Three rows with distinct scales on a
    square matrix: a scale taken along the columns gives other values here."""
    codes = np.array([[1, -2, 127], [0, 5, -127], [3, 3, 3]], np.int8)
    scale = np.array([0.5, 0.25, 2.0], np.float32)
    got = oracle.dequantize_rows_int8(codes, scale)
    want = np.array([[0.5, -1.0, 63.5], [0.0, 1.25, -31.75], [6.0, 6.0, 6.0]])
    assert got.dtype == np.float64 and got.shape == (3, 3)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("seed", range(2))
def test_oracle_dequantize_round_trip(seed):
    """Quantize then dequantize: every value is code x scale exactly (an int8 times an fp32 fits the
    53-bit fp64 significand), and lies within half a step of the value it stands for."""
    bits = _rows(seed, 5, 129)
    v = _f32(bits).astype(np.float64)
    codes, scale = oracle.quantize_rows_int8(bits)
    deq = oracle.dequantize_rows_int8(codes, scale)
    assert deq.shape == v.shape
    for r in range(v.shape[0]):
        s = Fraction(float(scale[r]))
        for c in range(0, v.shape[1], 7):
            assert Fraction(float(deq[r, c])) == int(codes[r, c]) * s
        assert np.all(np.abs(deq[r] - v[r]) <= float(scale[r]) * (0.5 + 2**-17))


def test_int8_halves_the_adapter_bytes():
    """Per adapter: r (d_in + d_out) one-byte codes plus two fp32 scales per rank index and
    projection, against 2 bytes per parameter in bf16."""
    bf16 = oracle.adapter_bytes(ATTN, 8, 1)
    i8 = oracle.adapter_bytes(ATTN, 8, 1, bytes_per_param=1) + 4 * 8 * 4 * 2
    assert bf16 == 2 * oracle.adapter_bytes(ATTN, 8, 1, bytes_per_param=1)
    assert 0.5 < i8 / bf16 < 0.501


@pytest.mark.parametrize("seed", range(2))
def test_oracle_fp64_factor_forward_matches_the_c_oracle(seed):
    """With factors that are bf16 values, the fp64-factor forward is the pinned C oracle."""
    w = wl.custom("f64fac", {"p": (256, 192)}, [["p"]], 12, [8, 16, 4], 1.5, seed=seed,
                  ids=wl.random_ids(12, 3, seed, p_base=0.2))
    A = [w.A(a, "p") for a in range(3)]
    B = [w.B(a, "p") for a in range(3)]
    ref = oracle.adapted_linear(w.x(0), w.W("p"), w.ids, A, B, w.scale)
    got = oracle.adapted_linear_factors64(w.x(0), w.W("p"), w.ids, [_f32(a).astype(np.float64) for a in A],
                                          [_f32(b).astype(np.float64) for b in B], w.scale)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_library_quantizer_is_the_oracle_bit_for_bit(seed):
    import adapter_serving_gb300 as L
    for rows, cols in ((1, 8), (7, 1024), (64, 8192)):
        bits = _rows(100 * seed + rows, rows, cols)
        bits[0, : cols // 2] = 0
        q1, s1 = L.quantize_rows_int8(bits)
        q2, s2 = oracle.quantize_rows_int8(bits)
        assert np.array_equal(q1, q2) and np.array_equal(s1.view(np.uint32), s2.view(np.uint32))


# ------------------------------------------------------------------------------- GPU ---

def _quantized(w, used):
    """codes and scales of every used adapter, and the factors they stand for (fp64)."""
    q = {}
    for a in used:
        for m in w.module_names():
            qA, sA = oracle.quantize_rows_int8(w.A(a, m))
            qBt, sB = oracle.quantize_rows_int8(np.ascontiguousarray(w.B(a, m).T))
            q[(a, m)] = (qA, sA, np.ascontiguousarray(qBt.T), sB,
                         oracle.dequantize_rows_int8(qA, sA), oracle.dequantize_rows_int8(qBt, sB).T)
    return q


def _i8_pool(w, q, pages=None):
    import adapter_serving_gb300 as L
    from harness import pages_for
    names = w.module_names()
    used = sorted({a for a, _ in q})
    pages = pages or [pages_for(w.ranks, used)] * len(names)
    pool = L.Pool([w.modules[m][0] for m in names], [w.modules[m][1] for m in names], w.n_adapters,
                  max_rank=64, pages=pages, max_rows=max(w.n_rows, 1), factor_dtype="int8")
    for (a, m), (qA, sA, qB, sB, _, _) in q.items():
        pool.load_i8(a, names.index(m), qA, sA, qB, sB)
    return pool


def _ref(w, q, m, st, rows=None):
    A64 = [None] * w.n_adapters
    B64 = [None] * w.n_adapters
    for (a, mm), v in q.items():
        if mm == m:
            A64[a], B64[a] = v[4], v[5]
    return oracle.adapted_linear_factors64(w.x(st), w.W(m), w.row_adapters(), A64, B64, w.scale, rows=rows)


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["tiny", "mixed", "qkv_like"])
def test_int8_decode_parity(case):
    from harness import check_close, run_stage
    if case == "tiny":
        w = wl.tiny()
    elif case == "mixed":
        ranks = np.random.default_rng(3).choice(np.array([4, 8, 16, 24, 32, 64], np.int32), 40)
        w = wl.custom("i8_mixed", {"p": (2048, 1536)}, [["p"]], 200, ranks, 1.0, seed=4,
                      ids=wl.random_ids(200, 40, 4, p_base=0.1))
    else:
        w = wl.custom("i8_qkv", {"q": (4096, 4096), "k": (4096, 512), "v": (4096, 512)}, [["q", "k", "v"]], 128,
                      np.full(128, 8, np.int32), 1.0, seed=5, ids=wl._perm_ids(128, 6))
    import torch
    from harness import bf16_gate
    q = _quantized(w, [int(a) for a in w.used_adapters()])
    pool = _i8_pool(w, q)
    outs = run_stage(pool, w, 0)
    outs16 = run_stage(pool, w, 0, y_dtype=torch.bfloat16)
    for m in w.stages[0]:
        ref = _ref(w, q, m, 0)
        check_close(outs[m].cpu().double().numpy(), ref, what=f"{case}/{m}")
        # bf16 output: one rounding of the fp32 result, within 1 bf16 ulp of the oracle rounded alike
        yb = outs16[m].view(torch.int16).cpu().numpy().view(np.uint16)
        bad = bf16_gate(yb, ref)
        assert len(bad) == 0, f"{case}/{m}: bf16 outputs off at {bad[:4].tolist()}"
    code, _ = pool.last_device_error()
    assert code == 0
    pool.close()


@pytest.mark.gpu
def test_int8_zero_b_is_bit_identical_to_base_only():
    import torch
    from harness import run_stage
    w = wl.custom("i8_zero_b", {"p": (1024, 2048)}, [["p"]], 64, np.full(16, 16, np.int32), 1.0, seed=7,
                  ids=wl.random_ids(64, 16, 7))
    q = _quantized(w, [int(a) for a in w.used_adapters()])
    for k in q:
        qA, sA, qB, sB, A64, B64 = q[k]
        q[k] = (qA, sA, np.zeros_like(qB), np.zeros_like(sB), A64, B64 * 0)
    pool = _i8_pool(w, q)
    y = run_stage(pool, w, 0)["p"]
    y0 = run_stage(pool, w, 0, ids=np.full(w.n_rows, -1, np.int32))["p"]
    assert torch.equal(y, y0)
    pool.close()


@pytest.mark.gpu
def test_int8_pool_refuses_what_it_does_not_serve():
    import torch
    import adapter_serving_gb300 as L
    from harness import to_host_bf16
    pool = L.Pool([1024], [1024], 4, max_rank=64, pages=[4], max_rows=512, factor_dtype="int8")
    A = to_host_bf16(np.zeros((8, 1024), np.uint16))
    B = to_host_bf16(np.zeros((1024, 8), np.uint16))
    with pytest.raises(L.LoraError):
        pool.load(0, 0, A, B)  # bf16 factors into an int8 pool
    pool.load_i8(0, 0, np.zeros((8, 1024), np.int8), np.zeros(8, np.float32), np.zeros((1024, 8), np.int8),
                 np.zeros(8, np.float32))
    x = torch.zeros(300, 1024, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(1024, 1024, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(300, 1024, device="cuda")
    ss = torch.tensor([0, 300], dtype=torch.int32, device="cuda")
    sa = torch.tensor([0], dtype=torch.int32, device="cuda")
    with pytest.raises(L.LoraError) as e:
        pool.segment_forward([(0, x, W, y)], ss, sa, 300, 1.0)  # grouped rows: bf16 pools only
    assert e.value.status == L.EUNSUPPORTED
    pool.close()


@pytest.mark.gpu
def test_int8_planned_forward_equals_own_grouping():
    """int8 packs (128 ranks per stage) through the row plan give the same bits as a call that
    groups its own rows, for fp32 and bf16 outputs."""
    import torch
    from harness import run_stage, to_dev_bf16
    ranks = np.random.default_rng(8).choice(np.array([8, 16, 32, 64], np.int32), 24)
    w = wl.custom("i8_plan", {"q": (2048, 2048), "o": (2048, 1024)}, [["q"], ["o"]], 77, ranks, 1.0, seed=9,
                  ids=wl.random_ids(77, 24, 9, p_base=0.1))
    q = _quantized(w, [int(a) for a in w.used_adapters()])
    pool = _i8_pool(w, q)
    names = w.module_names()
    for y_dtype in (torch.float32, torch.bfloat16):
        own = {}
        for st in range(len(w.stages)):
            own.update(run_stage(pool, w, st, y_dtype=y_dtype))
        pool.plan_rows(torch.from_numpy(w.ids).cuda())
        for st in range(len(w.stages)):
            x = to_dev_bf16(w.x(st))
            ios = []
            for m in w.stages[st]:
                y = torch.full((w.n_rows, w.modules[m][1]), float("nan"), dtype=y_dtype, device="cuda")
                ios.append((names.index(m), x, to_dev_bf16(w.W(m)), y))
            pool.layer_forward_planned(ios, w.scale)
            for (mi, _, _, y), m in zip(ios, w.stages[st]):
                torch.cuda.synchronize()
                assert torch.equal(y, own[m]), (m, y_dtype)
    pool.close()


@pytest.mark.gpu
def test_int8_full_size_attention_sampled_rows():
    """The 70B attention decode batch (q/k/v/o, 128 rows, 128 distinct rank-8 adapters) with int8
    factors, planned as the benchmark runs it, on rows the oracle computes one by one."""
    import torch
    from harness import check_close, to_dev_bf16
    w = wl.attn70b_decode()
    q = _quantized(w, [int(a) for a in w.used_adapters()])
    pool = _i8_pool(w, q)
    names = w.module_names()
    rows = np.arange(0, w.n_rows, 4) + (np.arange(0, w.n_rows, 4) // 4) % 4  # 32 rows, every residue mod 4
    pool.plan_rows(torch.from_numpy(w.ids).cuda())
    for st in range(len(w.stages)):
        x = to_dev_bf16(w.x(st))
        ios = []
        for m in w.stages[st]:
            y = torch.full((w.n_rows, w.modules[m][1]), float("nan"), dtype=torch.float32, device="cuda")
            ios.append((names.index(m), x, to_dev_bf16(w.W(m)), y))
        pool.layer_forward_planned(ios, w.scale)
        torch.cuda.synchronize()
        for (_, _, _, y), m in zip(ios, w.stages[st]):
            check_close(y.cpu().double().numpy()[rows], _ref(w, q, m, st, rows=rows), what=f"attn70b int8/{m}")
    code, _ = pool.last_device_error()
    assert code == 0
    pool.close()
