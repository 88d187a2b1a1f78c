"""The bench's byte and FLOP accounting, the numerator of every roofline fraction it prints.

Each figure is worked out by hand from the projection shapes the pages give for a 70B model
("m07 — Multi-Adapter (LoRA) Serving", section 2: q/o 8192 x 8192, k/v 8192 x 1024 under GQA,
gate/up 8192 x 28672, down 28672 x 8192) and the cost statement of its section 6 (the base read
once per step, each distinct adapter's factors once, activations in and out once).  Nothing here
calls the library or the oracle."""
import pytest

import bench
import workloads as wl

# elements of the four attention projections: 2 x 8192^2 + 2 x 8192 x 1024
ATTN_W_ELEMS = 2 * 67_108_864 + 2 * 8_388_608
ATTN_D_IN = 4 * 8192                     # q, k, v, o all read 8192-wide inputs
ATTN_D_OUT = 8192 + 1024 + 1024 + 8192   # 18,432


def test_headline_step_bytes_by_hand():
    b = bench.algorithmic_bytes(wl.attn70b_decode())
    assert b["W"] == ATTN_W_ELEMS * 2 == 301_989_888
    assert b["A"] == 128 * 8 * ATTN_D_IN * 2 == 67_108_864      # 128 distinct rank-8 adapters
    assert b["B"] == 128 * 8 * ATTN_D_OUT * 2 == 37_748_736
    assert b["x"] == 2 * 128 * 8192 * 2 == 4_194_304             # two calls: q/k/v share x, o
    assert b["y"] == 128 * ATTN_D_OUT * 4 == 9_437_184           # fp32 outputs
    assert b["total"] == 420_478_976
    assert b["gemm"] == 301_989_888 + 67_108_864 + 4_194_304     # W, A tiles and x in the gemm
    assert b["finalize"] == 37_748_736 + 9_437_184
    assert b["distinct"] == 128


def test_all_projection_step_bytes_by_hand():
    b = bench.algorithmic_bytes(wl.all70b_decode())
    w_elems = ATTN_W_ELEMS + 3 * 8192 * 28672
    d_in = ATTN_D_IN + 8192 + 8192 + 28672     # gate, up read 8192; down reads 28672
    d_out = ATTN_D_OUT + 28672 + 28672 + 8192  # 83,968
    assert b["W"] == w_elems * 2 == 1_711_276_032
    assert b["A"] == 128 * 64 * d_in * 2 == 1_275_068_416
    assert b["B"] == 128 * 64 * d_out * 2 == 1_375_731_712
    assert b["x"] == 128 * (8192 + 8192 + 8192 + 28672) * 2       # four calls
    assert b["y"] == 128 * d_out * 4
    assert b["total"] == 4_418_699_264


def test_int8_factors_count_one_byte_per_code_and_a_scale_per_rank_row():
    b = bench.algorithmic_bytes(wl.attn70b_decode(), int8=True)
    assert b["A"] == 128 * 8 * 4 * (8192 + 4)   # codes + one fp32 scale per rank row, per projection
    assert b["B"] == 128 * 8 * ATTN_D_OUT
    assert b["gemm"] == b["W"] + b["x"]          # the CUDA-core shrink reads A beside the gemm
    assert b["shrink"] == b["A"] + b["x"]


def test_int4_base_counts_half_a_byte_per_weight_and_a_scale_per_output_row():
    b = bench.algorithmic_bytes(wl.attn70b_decode(), w4=True)
    assert b["W"] == ATTN_W_ELEMS // 2 + 4 * ATTN_D_OUT == 75_571_200
    assert b["A"] == 67_108_864 and b["B"] == 37_748_736


def test_zipf_step_counts_each_distinct_adapter_once():
    w = wl.zipf_pool()
    ids = w.row_adapters()
    seen, rank_rows = set(), 0
    for a in ids:                       # rows of one adapter cost its factors once
        if a >= 0 and a not in seen:
            seen.add(int(a))
            rank_rows += int(w.ranks[a])
    assert len(seen) == 127 and rank_rows == 2544
    b = bench.algorithmic_bytes(w)
    assert b["distinct"] == 127
    assert b["A"] == rank_rows * ATTN_D_IN * 2 == 166_723_584
    assert b["B"] == rank_rows * ATTN_D_OUT * 2 == 93_782_016
    assert b["gemm"] == 301_989_888 + 166_723_584 + 2 * 256 * 8192 * 2 == 477_102_080
    assert b["total"] == 589_758_464


def test_prefill_flops_by_hand():
    w = wl.prefill_segments()
    T = int(w.seg_start[-1])
    assert T == 76_183
    base, lora = bench.step_flops(w)
    assert base == 2 * T * (2 * 8192 * 8192 + 8192 * 28672)
    # every token's adapter has rank 16: shrink + expand, 2 r (d_in + d_out) per projection
    assert lora == 2 * T * 16 * ((8192 + 8192) + (8192 + 8192) + (8192 + 28672))
    assert (base + lora) == pytest.approx(5.64e13, rel=1e-3)
