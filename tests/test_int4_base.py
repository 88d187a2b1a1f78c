"""int4 base weights with bf16 (or int8) adapters ("12. Adapter Serving and Multi-Tenant
Customization", section "Quantization": the base in INT4, the adapters in BF16; the kernel
dequantizes the base, adds the adapter term and accumulates wide; one batch mixes adapted and
base-only rows).

W = scale[o] * code[o, k] with code in [-7, 7] and one fp32 scale per output row.

* the oracle's quantizer against what rounding to the nearest code means (exact rationals), its
  error bound and special cases; the packed layout against a hand-worked word; the library's
  quantizer against the oracle bit for bit;
* the oracle's int4 forward against the pinned C oracle on a base whose dequantised values are
  bf16 numbers (power-of-two row scales), where the two must agree to rounding;
* (GPU) the int4 path against the oracle (own grouping and planned, fp32 and bf16 outputs, ragged
  d_in and d_out, mixed ranks, base-only rows, int8 factors); with power-of-two row scales the
  int4 path gives the bf16 path's bits; the calls it refuses.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wl


def _rows(seed, rows, cols):
    g = np.random.default_rng(seed)
    v = g.standard_normal((rows, cols)).astype(np.float32)
    v *= g.choice(np.array([1e-3, 0.07, 1.0, 300.0], np.float32), (rows, 1))
    return wl.f32_to_bf16_bits(v)


def _f32(bits):
    return wl.bf16_bits_to_f32(bits)


def _pack_w4(codes):
    """The packed layout the C header documents: every 8 consecutive elements of a row form one
    little-endian 32-bit word, element 2s at bits [4s, 4s + 4) and element 2s + 1 at bits
    [16 + 4s, 20 + 4s), each as code + 8."""
    c = np.asarray(codes, np.int64) + 8
    r, k = c.shape
    g = c.reshape(r, k // 8, 8)
    word = np.zeros((r, k // 8), np.uint32)
    for e in range(8):
        word |= (g[:, :, e].astype(np.uint32) << np.uint32((e & 1) * 16 + (e >> 1) * 4))
    return word.astype("<u4").view(np.uint8).reshape(r, k // 2)


def _pow2_base(seed, d_out, d_in):
    """A base whose int4 form is exact: codes in [-7, 7] with a +-7 in every row and row scales
    2^e, so W = code * 2^e is a bf16 number and quantizing it gives back (codes, 2^e)."""
    g = np.random.default_rng([seed, 44])
    codes = g.integers(-7, 8, (d_out, d_in)).astype(np.int8)
    codes[np.arange(d_out), g.integers(0, d_in, d_out)] = g.choice(np.array([-7, 7], np.int8), d_out)
    sc = np.ldexp(np.float32(1.0), g.integers(-9, -3, d_out)).astype(np.float32)
    W = wl.f32_to_bf16_bits(codes.astype(np.float32) * sc[:, None])
    return W, codes, sc


# ------------------------------------------------------------------------------ oracle pins ---

@pytest.mark.parametrize("seed", range(3))
def test_oracle_quantizer_rounds_to_the_nearest_code(seed):
    bits = _rows(seed, 6, 264)
    bits[2] = 0
    codes, scale = oracle.quantize_rows_int4(bits)
    v = _f32(bits)
    assert codes.dtype == np.int8 and scale.dtype == np.float32
    assert np.all(codes[2] == 0) and scale[2] == 0
    for r in range(len(bits)):
        if scale[r] == 0:
            continue
        m = np.abs(v[r]).max()
        # the scale is max/7 rounded once to fp32
        assert abs(Fraction(float(scale[r])) - Fraction(float(m)) / 7) <= Fraction(float(scale[r])) * Fraction(1, 2**23)
        assert np.abs(codes[r]).max() == 7 and np.all(np.abs(codes[r]) <= 7)
        s = Fraction(float(scale[r]))
        for c in range(v.shape[1]):
            e = Fraction(float(v[r, c])) / s  # the exact quotient
            k = int(codes[r, c])
            # nearest code; within 2^-20 of a half-integer the one fp32 rounding of the quotient may go either way
            assert abs(e - k) <= Fraction(1, 2) + Fraction(1, 2**20)
            if abs(abs(e - int(e)) - Fraction(1, 2)) > Fraction(1, 2**20) and abs(e) < 7:
                assert k == round(e)
        # dequantised error bound: half a step (plus the quotient's rounding)
        assert np.all(np.abs(codes[r].astype(np.float64) * float(scale[r]) - v[r]) <= float(scale[r]) * (0.5 + 2**-19))


def test_oracle_quantizer_half_even_and_signs():
    """With scale 1 (the row's max is 7) halves go to the even code; signs are kept."""
    v = np.array([[7.0, -7.0, 3.5, 2.5, -2.5, 0.5, -0.5, 1.5, 6.5, 0.0, -1.0, 4.0, -6.0, 5.5, -5.5, 0.25]], np.float32)
    codes, scale = oracle.quantize_rows_int4(wl.f32_to_bf16_bits(v))
    assert scale[0] == 1.0
    assert codes[0].tolist() == [7, -7, 4, 2, -2, 0, 0, 2, 6, 0, -1, 4, -6, 6, -6, 0]


def test_packed_layout_hand_worked_word():
    """Elements (1, -1, 7, 0, 2, -7, 3, 0): low half holds elements 0, 2, 4, 6 as 9, 15, 10, 11
    (0xBAF9), high half elements 1, 3, 5, 7 as 7, 8, 1, 8 (0x8187): bytes F9 BA 87 81."""
    codes = np.array([[1, -1, 7, 0, 2, -7, 3, 0]], np.int8)
    assert _pack_w4(codes).tolist() == [[0xF9, 0xBA, 0x87, 0x81]]


@pytest.mark.parametrize("seed", range(3))
def test_library_quantizer_is_the_oracle_bit_for_bit(seed):
    import adapter_serving_gb300 as L
    for rows, cols in ((1, 8), (7, 96), (64, 8192)):
        bits = _rows(100 * seed + rows, rows, cols)
        bits[0, : cols // 2] = 0
        if rows > 2:
            bits[2] = 0
        p1, s1 = L.quantize_w4(bits)
        c2, s2 = oracle.quantize_rows_int4(bits)
        assert np.array_equal(s1.view(np.uint32), s2.view(np.uint32))
        assert np.array_equal(p1, _pack_w4(c2))


def test_library_quantizer_argument_checks():
    import adapter_serving_gb300 as L
    with pytest.raises(L.LoraError):
        L.quantize_w4(np.zeros((2, 12), np.uint16))  # cols not a multiple of 8


def test_power_of_two_base_round_trips():
    W, codes, sc = _pow2_base(1, 40, 64)
    c2, s2 = oracle.quantize_rows_int4(W)
    assert np.array_equal(c2, codes) and np.array_equal(s2, sc)


@pytest.mark.parametrize("seed", range(2))
def test_oracle_w4_forward_matches_the_c_oracle(seed):
    """With an exactly representable base, the int4 forward is the pinned C oracle's forward."""
    W, codes, sc = _pow2_base(seed, 192, 256)
    w = wl.custom("w4pin", {"p": (256, 192)}, [["p"]], 12, [8, 16, 4], 1.5, seed=seed,
                  ids=wl.random_ids(12, 3, seed, p_base=0.2))
    A = [w.A(a, "p") for a in range(3)]
    B = [w.B(a, "p") for a in range(3)]
    ref = oracle.adapted_linear(w.x(0), W, w.ids, A, B, w.scale)
    got = oracle.adapted_linear_w4(w.x(0), codes, sc, w.ids, [_f32(a).astype(np.float64) for a in A],
                                   [_f32(b).astype(np.float64) for b in B], w.scale)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12)
    rows = np.array([0, 5, 11])
    sub = oracle.adapted_linear_w4(w.x(0), codes, sc, w.ids, [_f32(a).astype(np.float64) for a in A],
                                   [_f32(b).astype(np.float64) for b in B], w.scale, rows=rows)
    assert np.array_equal(sub, got[rows])


# ------------------------------------------------------------------------------------ GPU ---

def _quantize_base(w):
    return {m: oracle.quantize_rows_int4(w.W(m)) for m in w.module_names()}


def _factors64(w, m):
    A64 = [None] * w.n_adapters
    B64 = [None] * w.n_adapters
    for a in w.used_adapters():
        A64[int(a)] = _f32(w.A(int(a), m)).astype(np.float64)
        B64[int(a)] = _f32(w.B(int(a), m)).astype(np.float64)
    return A64, B64


def _run_w4(pool, w, st, qw, y_dtype=None, planned=False, ids=None):
    """One stage through lora_layer_forward_w4 (or plan + lora_layer_forward_planned_w4)."""
    import torch
    from harness import to_dev_bf16
    y_dtype = torch.float32 if y_dtype is None else y_dtype
    names = w.module_names()
    x = to_dev_bf16(w.x(st))
    ios, outs = [], {}
    for m in w.stages[st]:
        codes, sc = qw[m]
        y = torch.full((w.n_rows, w.modules[m][1]), float("nan"), dtype=y_dtype, device="cuda")
        ios.append((names.index(m), x, torch.from_numpy(_pack_w4(codes)).cuda(), torch.from_numpy(sc).cuda(), y))
        outs[m] = y
    idt = torch.from_numpy(w.row_adapters() if ids is None else ids).cuda()
    if planned:
        pool.plan_rows(idt)
        pool.layer_forward_planned_w4(ios, w.scale)
    else:
        pool.layer_forward_w4(ios, idt, w.scale)
    torch.cuda.synchronize()
    return outs


def _case(name):
    if name == "ragged":  # d_in 96: a half-empty last k-block; d_out 200: a ragged tile
        return wl.custom("w4_ragged", {"p": (96, 200)}, [["p"]], 20, [8, 16, 4, 32, 8, 64], 1.0, seed=3,
                         ids=wl.random_ids(20, 6, 3, p_base=0.2))
    if name == "mixed":
        ranks = np.random.default_rng(3).choice(np.array([4, 8, 16, 24, 32, 64], np.int32), 40)
        return wl.custom("w4_mixed", {"p": (2048, 1536)}, [["p"]], 200, ranks, 1.0, seed=4,
                         ids=wl.random_ids(200, 40, 4, p_base=0.1))
    return wl.custom("w4_qkv", {"q": (4096, 4096), "k": (4096, 512), "v": (4096, 512), "o": (4096, 4096)},
                     [["q", "k", "v"], ["o"]], 128, np.full(128, 8, np.int32), 1.0, seed=5, ids=wl._perm_ids(128, 6))


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["ragged", "mixed", "qkv_like"])
def test_w4_decode_parity(case):
    import torch
    from harness import bf16_gate, check_close, make_pool
    w = _case(case)
    qw = _quantize_base(w)
    pool, _ = make_pool(w)
    for st in range(len(w.stages)):
        for planned, y_dtype in ((False, torch.float32), (True, torch.float32), (True, torch.bfloat16)):
            outs = _run_w4(pool, w, st, qw, y_dtype=y_dtype, planned=planned)
            for m in w.stages[st]:
                A64, B64 = _factors64(w, m)
                ref = oracle.adapted_linear_w4(w.x(st), *qw[m], w.row_adapters(), A64, B64, w.scale)
                y = outs[m].float().cpu().double().numpy()
                if y_dtype == torch.bfloat16:  # one rounding of the fp32 result: within 1 ulp
                    yb = outs[m].view(torch.int16).cpu().numpy().view(np.uint16)
                    bad = bf16_gate(yb, ref)
                    assert len(bad) == 0, f"{case}/{m}: bf16 outputs off at {bad[:4].tolist()}"
                else:
                    check_close(y, ref, what=f"{case}/{m}/planned={planned}")
    code, _ = pool.last_device_error()
    assert code == 0
    pool.close()


@pytest.mark.gpu
def test_w4_with_power_of_two_scales_is_the_bf16_path_bit_for_bit():
    """(code x) * 2^e and (code * 2^e) x round alike, so the int4 path must give the bf16 path's
    bits when every row scale is a power of two (same tiles, same k order, same expand)."""
    from harness import make_pool, run_stage
    ranks = np.random.default_rng(2).choice(np.array([8, 16, 32, 64], np.int32), 24)
    w = wl.custom("w4_pow2", {"q": (2048, 2048), "k": (2048, 512)}, [["q", "k"]], 96, ranks, 1.0, seed=12,
                  ids=wl.random_ids(96, 24, 12, p_base=0.15))
    Wb, qw = {}, {}
    for i, m in enumerate(w.module_names()):
        d_in, d_out = w.modules[m]
        W, codes, sc = _pow2_base(20 + i, d_out, d_in)
        Wb[m], qw[m] = W, (codes, sc)
    pool, _ = make_pool(w)
    ref = run_stage(pool, w, 0, W_bits=Wb)
    got = _run_w4(pool, w, 0, qw)
    got_planned = _run_w4(pool, w, 0, qw, planned=True)
    for m in w.stages[0]:
        assert np.array_equal(got[m].cpu().numpy().view(np.uint32), ref[m].cpu().numpy().view(np.uint32)), m
        assert np.array_equal(got_planned[m].cpu().numpy().view(np.uint32), ref[m].cpu().numpy().view(np.uint32)), m
    pool.close()


@pytest.mark.gpu
def test_w4_host_step_gives_the_device_step_bits():
    """lora_layer_step_host_w4: ids and x from pinned host memory, y back to it, one call per step
    on two alternating device buffer sets; the host outputs equal the planned device calls'."""
    import torch
    from harness import make_pool, to_dev_bf16, to_host_bf16
    w = _case("qkv_like")
    qw = _quantize_base(w)
    pool, _ = make_pool(w)
    names = w.module_names()
    packed = {m: (torch.from_numpy(_pack_w4(qw[m][0])).cuda(), torch.from_numpy(qw[m][1]).cuda()) for m in names}
    ref = {}
    for st in range(len(w.stages)):
        ref.update(_run_w4(pool, w, st, qw, planned=True))
    order = [m for st in w.stages for m in st]
    hid = torch.from_numpy(w.row_adapters()).pin_memory()
    hx = [to_host_bf16(w.x(st)).pin_memory() for st in range(len(w.stages))]
    sets = []
    for b in range(2):
        ids_d = torch.full((w.n_rows,), 12345, dtype=torch.int32, device="cuda")  # garbage until uploaded
        xb = [torch.zeros_like(to_dev_bf16(w.x(st))) for st in range(len(w.stages))]
        yb = {m: torch.full((w.n_rows, w.modules[m][1]), float("nan"), device="cuda") for m in names}
        stages = [[(names.index(m), xb[st], *packed[m], yb[m]) for m in w.stages[st]] for st in range(len(w.stages))]
        hy = [torch.full((w.n_rows, w.modules[m][1]), float("nan")).pin_memory() for m in order]
        sets.append((ids_d, stages, hy))
    for k in range(4):
        ids_d, stages, hy = sets[k % 2]
        pool.layer_step_host_w4(stages, ids_d, hid, hx, hy, w.scale)
    pool.host_wait()
    torch.cuda.current_stream().synchronize()
    for _, _, hy in sets:
        for m, y in zip(order, hy):
            assert torch.equal(y, ref[m].cpu()), m
    pool.close()


@pytest.mark.gpu
def test_w4_with_int8_factors():
    """The int4 base under int8 adapter factors (both quantized variants in one call)."""
    from harness import check_close
    from test_int8_factors import _i8_pool, _quantized
    ranks = np.random.default_rng(8).choice(np.array([8, 16, 32, 64], np.int32), 24)
    w = wl.custom("w4_i8", {"q": (2048, 2048), "o": (2048, 1024)}, [["q"], ["o"]], 77, ranks, 1.0, seed=9,
                  ids=wl.random_ids(77, 24, 9, p_base=0.1))
    q = _quantized(w, [int(a) for a in w.used_adapters()])
    pool = _i8_pool(w, q)
    qw = _quantize_base(w)
    for st in range(len(w.stages)):
        outs = _run_w4(pool, w, st, qw, planned=(st == 1))
        for m in w.stages[st]:
            A64 = [None] * w.n_adapters
            B64 = [None] * w.n_adapters
            for (a, mm), v in q.items():
                if mm == m:
                    A64[a], B64[a] = v[4], v[5]
            ref = oracle.adapted_linear_w4(w.x(st), *qw[m], w.row_adapters(), A64, B64, w.scale)
            check_close(outs[m].cpu().double().numpy(), ref, what=f"w4+i8/{m}")
    code, _ = pool.last_device_error()
    assert code == 0
    pool.close()


@pytest.mark.gpu
def test_w4_full_size_attention_sampled_rows():
    """The 70B attention decode batch (q/k/v/o 8192 -> 8192/1024/1024/8192, 128 rows, 128 distinct
    rank-8 adapters) with an int4 base, on rows the oracle computes one by one."""
    from harness import check_close, make_pool
    w = wl.attn70b_decode()
    qw = _quantize_base(w)
    pool, _ = make_pool(w)
    rows = np.arange(0, w.n_rows, 4) + (np.arange(0, w.n_rows, 4) // 4) % 4  # 32 rows, every residue mod 4
    for st in range(len(w.stages)):
        outs = _run_w4(pool, w, st, qw, planned=True)
        for m in w.stages[st]:
            A64, B64 = _factors64(w, m)
            ref = oracle.adapted_linear_w4(w.x(st), *qw[m], w.row_adapters(), A64, B64, w.scale, rows=rows)
            check_close(outs[m].cpu().double().numpy()[rows], ref, what=f"attn70b w4/{m}")
    pool.close()


@pytest.mark.gpu
def test_w4_refusals_and_empty_batch():
    import torch
    import adapter_serving_gb300 as L
    pool = L.Pool([48, 1024], [256, 256], 4, max_rank=64, pages=[2, 2], max_rows=512)
    x48 = torch.zeros(4, 48, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(300, 1024, dtype=torch.bfloat16, device="cuda")
    codes48 = torch.zeros(256, 24, dtype=torch.uint8, device="cuda")
    codes = torch.zeros(256, 512, dtype=torch.uint8, device="cuda")
    sc = torch.ones(256, dtype=torch.float32, device="cuda")
    y = torch.zeros(300, 256, device="cuda")
    ids = torch.zeros(300, dtype=torch.int32, device="cuda")
    with pytest.raises(L.LoraError) as e:  # d_in % 32 != 0
        pool.layer_forward_w4([(0, x48, codes48, sc, y[:4])], ids[:4], 1.0)
    assert e.value.status == L.EUNSUPPORTED
    with pytest.raises(L.LoraError) as e:  # more rows than a decode batch
        pool.layer_forward_w4([(1, x, codes, sc, y)], ids, 1.0)
    assert e.value.status == L.EUNSUPPORTED
    pool.layer_forward_w4([(1, x[:0], codes, sc, y[:0])], ids[:0], 1.0)  # empty batch: nothing happens
    torch.cuda.synchronize()
    code, _ = pool.last_device_error()
    assert code == 0
    pool.close()
