"""Planted mistakes: the oracle's pins must catch a plausible error anywhere in it.

Each mutant is a plain fp64 restatement of an oracle function with one mistake planted in it (a
dropped term, a wrong sign, a wrong index, a transposed operand, a wrong rounding or scale).  The
test swaps it in for the oracle function, runs that function's pins, and requires at least one
pin to fail.  The same restatement with no mistake passes every pin, so a failure comes from the
planted mistake alone.  Everything here runs on the CPU; the GPU library is never involved.
"""
import numpy as np
import pytest

import oracle
import test_int4_base as Q
import test_oracle_pins as P
import workloads as wl


def _f64(b):
    return wl.bf16_bits_to_f32(np.asarray(b, np.uint16)).astype(np.float64)


def _forward(x, W, ids, A, B, scale, rows=None, threads=0, return_t=False, bug=None):
    """y_i = W x_i + s B_a (A_a x_i), row by row in fp64, with an optional planted mistake."""
    xf, Wf = _f64(x), _f64(W)
    if bug == "W_transposed_read":
        Wf = Wf.reshape(Wf.shape[1], Wf.shape[0]).T
    ids = np.asarray(ids, np.int32)
    n_ad = len(A)
    if np.any(ids < -1) or np.any(ids >= n_ad):
        raise ValueError("adapter id out of range")
    rows = np.arange(len(ids)) if rows is None else np.asarray(rows)
    rmax = max([a.shape[0] for a in A if a is not None] + [1])
    y = np.zeros((len(rows), Wf.shape[0]))
    t_all = np.zeros((len(rows), rmax))
    for k, i in enumerate(rows):
        a = int(ids[i])
        if bug == "base_skipped_for_adapted_rows" and a >= 0:
            base = np.zeros(Wf.shape[0])
        else:
            base = Wf @ xf[i]
        y[k] = base
        if a < 0:
            continue
        if bug == "wrong_adapter":
            a = (a + 1) % n_ad
        Af, Bf = _f64(A[a]), _f64(B[a])
        if bug == "B_transposed_read":
            Bf = Bf.reshape(Bf.shape[1], Bf.shape[0]).T
        if bug == "rank_truncated" and Af.shape[0] > 1:
            Af, Bf = Af[:-1], Bf[:, :-1]
        xi = xf[(i + 1) % len(ids)] if bug == "x_of_next_row_in_shrink" else xf[i]
        t = Af @ xi
        t_all[k, :len(t)] = t
        if bug == "adapter_dropped":
            continue
        s = {"no_scale": 1.0, "minus_adapter": -scale}.get(bug, scale)
        y[k] += s * (Bf @ t)
    return (y, t_all) if return_t else y


FORWARD_PINS = [P.test_hand_worked_example, P.test_bruteforce_exact_rationals, P.test_b_zero_is_base_layer,
                P.test_one_adapter_equals_merged_weight, P.test_mixed_rows_match_their_merged_weight,
                P.test_shrink_matches_matmul, P.test_base_only_rows, P.test_zero_padding_rank_changes_nothing,
                P.test_row_permutation, P.test_adapter_is_sum_of_rank_one_pieces, P.test_linear_in_scale,
                P.test_invalid_ids_rejected]
FORWARD_BUGS = ["adapter_dropped", "minus_adapter", "no_scale", "wrong_adapter", "B_transposed_read",
                "W_transposed_read", "rank_truncated", "x_of_next_row_in_shrink", "base_skipped_for_adapted_rows"]


def _failing_pins(pins):
    failed = []
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            failed.append(pin.__name__)
    return failed


def test_forward_restatement_passes_every_pin(monkeypatch):
    monkeypatch.setattr(oracle, "adapted_linear", lambda *a, **k: _forward(*a, **k))
    assert _failing_pins(FORWARD_PINS) == []


@pytest.mark.parametrize("bug", FORWARD_BUGS)
def test_forward_pins_catch_planted_mistake(monkeypatch, bug):
    monkeypatch.setattr(oracle, "adapted_linear", lambda *a, **k: _forward(*a, bug=bug, **k))
    assert _failing_pins(FORWARD_PINS), f"no pin caught {bug}"


# ---------------------------------------------------------------------------- int4 base ---

def _quantize4(bits, bug=None):
    v = wl.bf16_bits_to_f32(np.asarray(bits, np.uint16))
    levels = 8.0 if bug == "scale_over_8" else 7.0
    scale = (np.abs(v).max(axis=1) / np.float32(levels)).astype(np.float32)
    codes = np.zeros(v.shape, np.int8)
    nz = scale > 0
    q = v[nz] / scale[nz, None]
    if bug == "truncate":
        q = np.trunc(q)
    elif bug == "half_away_from_zero":
        q = np.sign(q) * np.floor(np.abs(q) + np.float32(0.5))
    else:
        q = np.rint(q)
    codes[nz] = np.clip(q, -7, 7).astype(np.int8)
    return codes, scale


def _nearest_code_seed0():
    Q.test_oracle_quantizer_rounds_to_the_nearest_code(0)


def _nearest_code_seed1():
    Q.test_oracle_quantizer_rounds_to_the_nearest_code(1)


QUANT_PINS = [_nearest_code_seed0, _nearest_code_seed1, Q.test_oracle_quantizer_half_even_and_signs,
              Q.test_power_of_two_base_round_trips]


def test_int4_quantizer_restatement_passes_every_pin(monkeypatch):
    monkeypatch.setattr(oracle, "quantize_rows_int4", lambda b: _quantize4(b))
    assert _failing_pins(QUANT_PINS) == []


@pytest.mark.parametrize("bug", ["scale_over_8", "truncate", "half_away_from_zero"])
def test_int4_quantizer_pins_catch_planted_mistake(monkeypatch, bug):
    monkeypatch.setattr(oracle, "quantize_rows_int4", lambda b: _quantize4(b, bug))
    assert _failing_pins(QUANT_PINS), f"no pin caught {bug}"


def _forward_w4(x, codes, wscale, ids, A64, B64, scale, rows=None, bug=None):
    xf = _f64(x)
    c = np.asarray(codes, np.float64)
    sc = np.asarray(wscale, np.float64)
    if bug == "row_scale_skipped":
        W = c
    elif bug == "scale_by_column":  # the row scales read along k (cycled when d_in > d_out)
        W = c * np.resize(sc, c.shape[1])[None, :]
    elif bug == "codes_left_offset":
        W = (c + 8) * sc[:, None]
    else:
        W = c * sc[:, None]
    ids = np.asarray(ids, np.int32)
    rows = np.arange(len(ids)) if rows is None else np.asarray(rows)
    y = np.zeros((len(rows), W.shape[0]))
    for k, i in enumerate(rows):
        y[k] = W @ xf[i]
        a = int(ids[i])
        if a >= 0 and bug != "adapter_dropped":
            y[k] += scale * (B64[a] @ (A64[a] @ xf[i]))
    return y


def _w4_forward_seed0():
    Q.test_oracle_w4_forward_matches_the_c_oracle(0)


def _w4_forward_seed1():
    Q.test_oracle_w4_forward_matches_the_c_oracle(1)


W4_PINS = [_w4_forward_seed0, _w4_forward_seed1]


def test_int4_forward_restatement_passes_every_pin(monkeypatch):
    monkeypatch.setattr(oracle, "adapted_linear_w4", lambda *a, **k: _forward_w4(*a, **k))
    assert _failing_pins(W4_PINS) == []


@pytest.mark.parametrize("bug", ["row_scale_skipped", "scale_by_column", "codes_left_offset", "adapter_dropped"])
def test_int4_forward_pins_catch_planted_mistake(monkeypatch, bug):
    monkeypatch.setattr(oracle, "adapted_linear_w4", lambda *a, **k: _forward_w4(*a, bug=bug, **k))
    assert _failing_pins(W4_PINS), f"no pin caught {bug}"


# ------------------------------------------------------------------------- batch former ---

import test_batch_former as TB  # noqa: E402
from oracle import batch_former as OB  # noqa: E402

_form_batch = OB.form_batch


def _hand_worked_cases():
    for case in TB._cases():
        TB.test_oracle_hand_worked_cases(case)


def _plain_grouping_properties():
    for seed in range(4):
        TB.test_oracle_properties_plain_grouping(seed)


def _fairness_properties():
    for seed in range(4):
        TB.test_oracle_properties_fairness(seed)


FORMER_PINS = [_hand_worked_cases, _plain_grouping_properties, _fairness_properties]


def _former_mutant(bug):
    def f(queue_adapter, queue_waited_ms, max_batch, max_distinct, min_batch=1, tail_slots=0, max_queue_ms=0.0):
        if bug == "cap_ignored":
            max_distinct = 10 ** 9
        elif bug == "tail_slots_ignored":
            tail_slots = 0
        elif bug == "age_override_ignored":
            max_queue_ms = 0.0
        elif bug == "min_batch_ignored":
            min_batch = 1
        elif bug == "newest_first":  # the queue walked from its tail
            n = len(queue_adapter)
            batch, d = _form_batch(list(queue_adapter)[::-1], list(queue_waited_ms)[::-1], max_batch, max_distinct,
                                   min_batch, tail_slots, max_queue_ms)
            return [n - 1 - i for i in batch], d
        return _form_batch(queue_adapter, queue_waited_ms, max_batch, max_distinct, min_batch, tail_slots,
                           max_queue_ms)
    return f


def test_batch_former_wrapper_without_mistake_passes_every_pin(monkeypatch):
    monkeypatch.setattr(OB, "form_batch", _former_mutant(None))
    assert _failing_pins(FORMER_PINS) == []


@pytest.mark.parametrize("bug", ["cap_ignored", "tail_slots_ignored", "age_override_ignored", "min_batch_ignored",
                                 "newest_first"])
def test_batch_former_pins_catch_planted_mistake(monkeypatch, bug):
    monkeypatch.setattr(OB, "form_batch", _former_mutant(bug))
    assert _failing_pins(FORMER_PINS), f"no pin caught {bug}"


# ------------------------------------------------------------------------ adapter cache ---

from fractions import Fraction  # noqa: E402

import test_adapter_cache as TC  # noqa: E402
from oracle import adapter_cache as OC  # noqa: E402


def _cache_properties():
    for seed in range(3):
        TC.test_oracle_properties_on_zipf_traffic(seed)


CACHE_PINS = [TC.test_value_per_byte_keeps_the_hot_adapter_that_lru_would_evict, TC.test_value_is_per_byte_not_per_adapter,
              TC.test_referenced_adapter_is_never_evicted,
              TC.test_pinning_guard_refuses_new_adapters_but_not_resident_ones, TC.test_value_counts_only_the_window,
              TC.test_no_room_changes_nothing, TC.test_ties_go_to_the_older_latest_request_then_the_smaller_id,
              TC.test_evicts_the_fewest_adapters_in_value_order, _cache_properties]

CACHE_BUGS = {
    # recency instead of value per byte
    "lru": ("_value", lambda self, a, now: max(self.requests.get(a, [float("-inf")]))),
    # requests counted, bytes ignored
    "count_only": ("_value", lambda self, a, now: Fraction(
        len([t for t in self.requests.get(a, []) if t > now - self.window]), 1)),
    # every request counts, however old
    "window_ignored": ("_value", lambda self, a, now: Fraction(len(self.requests.get(a, [])), self.bytes[a])),
    # the guard never sees pinned bytes
    "guard_blind": ("pinned_bytes", lambda self: 0),
}


def test_cache_pins_pass_unchanged():
    assert _failing_pins(CACHE_PINS) == []


@pytest.mark.parametrize("bug", sorted(CACHE_BUGS))
def test_cache_pins_catch_planted_mistake(monkeypatch, bug):
    name, fn = CACHE_BUGS[bug]
    monkeypatch.setattr(OC.AdapterCache, name, fn)
    assert _failing_pins(CACHE_PINS), f"no pin caught {bug}"


# ------------------------------------------------------------------ int8 adapter factors ---

import test_int8_factors as T8  # noqa: E402


def _quantize8(bits, bug=None):
    v = wl.bf16_bits_to_f32(np.asarray(bits, np.uint16))
    levels = 128.0 if bug == "scale_over_128" else 127.0
    scale = (np.abs(v).max(axis=1) / np.float32(levels)).astype(np.float32)
    codes = np.zeros(v.shape, np.int8)
    nz = scale > 0
    q = v[nz] / scale[nz, None]
    q = np.trunc(q) if bug == "truncate" else np.rint(q)
    if bug == "sign_lost":
        q = np.abs(q)
    codes[nz] = np.clip(q, -127, 127).astype(np.int8)
    return codes, scale


def _i8_nearest_seed0():
    T8.test_oracle_quantizer_rounds_to_the_nearest_code(0)


def _i8_nearest_seed1():
    T8.test_oracle_quantizer_rounds_to_the_nearest_code(1)


I8_QUANT_PINS = [_i8_nearest_seed0, _i8_nearest_seed1, T8.test_oracle_quantizer_signs_and_exact_multiples]


def test_int8_quantizer_restatement_passes_every_pin(monkeypatch):
    monkeypatch.setattr(oracle, "quantize_rows_int8", lambda b: _quantize8(b))
    assert _failing_pins(I8_QUANT_PINS) == []


@pytest.mark.parametrize("bug", ["scale_over_128", "truncate", "sign_lost"])
def test_int8_quantizer_pins_catch_planted_mistake(monkeypatch, bug):
    monkeypatch.setattr(oracle, "quantize_rows_int8", lambda b: _quantize8(b, bug))
    assert _failing_pins(I8_QUANT_PINS), f"no pin caught {bug}"


def _dequant8(codes, scale, bug=None):
    c = np.asarray(codes, np.float64)
    s = np.asarray(scale, np.float64)
    if bug == "codes_as_unsigned":
        c = np.asarray(codes, np.int8).view(np.uint8).astype(np.float64)
    if bug == "scale_rounded_to_bf16":
        s = wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(np.asarray(scale, np.float32))).astype(np.float64)
    if bug == "scale_along_columns":
        return c * s[None, :]
    return c * s[:, None]


def _deq_round_trip_seed0():
    T8.test_oracle_dequantize_round_trip(0)


DEQ8_PINS = [T8.test_oracle_dequantize_rows_int8_hand_worked, _deq_round_trip_seed0]


def test_int8_dequantizer_restatement_passes_every_pin(monkeypatch):
    monkeypatch.setattr(oracle, "dequantize_rows_int8", lambda c, s: _dequant8(c, s))
    assert _failing_pins(DEQ8_PINS) == []


@pytest.mark.parametrize("bug", ["scale_along_columns", "codes_as_unsigned", "scale_rounded_to_bf16"])
def test_int8_dequantizer_pins_catch_planted_mistake(monkeypatch, bug):
    monkeypatch.setattr(oracle, "dequantize_rows_int8", lambda c, s: _dequant8(c, s, bug))
    assert _failing_pins(DEQ8_PINS), f"no pin caught {bug}"


def _factors64(x, W, ids, A64, B64, scale, rows=None, threads=0, bug=None):
    xf, Wf = _f64(x), _f64(W)
    ids = np.asarray(ids, np.int32)
    rows = np.arange(len(ids)) if rows is None else np.asarray(rows)
    y = np.zeros((len(rows), Wf.shape[0]))
    for k, i in enumerate(rows):
        y[k] = Wf @ xf[i]
        a = int(ids[i])
        if a < 0:
            continue
        Bm = B64[a]
        if bug == "B_transposed_read":
            Bm = Bm.reshape(Bm.shape[1], Bm.shape[0]).T
        t = A64[a] @ xf[i]
        y[k] += (1.0 if bug == "t_not_scaled" else scale) * (Bm @ t)
    return y


def _f64_forward_seed0():
    T8.test_oracle_fp64_factor_forward_matches_the_c_oracle(0)


def _f64_forward_seed1():
    T8.test_oracle_fp64_factor_forward_matches_the_c_oracle(1)


F64_PINS = [_f64_forward_seed0, _f64_forward_seed1]


def test_factor_forward_restatement_passes_every_pin(monkeypatch):
    monkeypatch.setattr(oracle, "adapted_linear_factors64", lambda *a, **k: _factors64(*a, **k))
    assert _failing_pins(F64_PINS) == []


@pytest.mark.parametrize("bug", ["t_not_scaled", "B_transposed_read"])
def test_factor_forward_pins_catch_planted_mistake(monkeypatch, bug):
    monkeypatch.setattr(oracle, "adapted_linear_factors64", lambda *a, **k: _factors64(*a, bug=bug, **k))
    assert _failing_pins(F64_PINS), f"no pin caught {bug}"


# ------------------------------------------------------------------------- row grouping ---

def _segments(ids, bug=None):
    ids = np.asarray(ids, np.int32)
    n = len(ids)
    if bug == "unstable":  # ties in reverse arrival order
        perm = sorted(range(n), key=lambda i: (int(ids[i]), -i))
    elif bug == "base_rows_last":
        perm = sorted(range(n), key=lambda i: (int(ids[i]) < 0, int(ids[i])))
    elif bug == "descending":
        perm = sorted(range(n), key=lambda i: -int(ids[i]))
    else:
        perm = sorted(range(n), key=lambda i: int(ids[i]))
    seg_start, seg_adapter = [0], []
    for k, i in enumerate(perm):
        if k == 0 or ids[i] != ids[perm[k - 1]]:
            if k > 0:
                seg_start.append(k)
            seg_adapter.append(int(ids[i]))
    if n:
        seg_start.append(n)
    if bug == "last_segment_dropped" and seg_adapter:
        seg_adapter, seg_start = seg_adapter[:-1], seg_start[:-1]
    return np.array(perm, np.int32), np.array(seg_start, np.int32), np.array(seg_adapter, np.int32)


def _stable_sort_seeds():
    for seed in range(6):
        P.test_segments_stable_sort(seed)


SEGMENT_PINS = [_stable_sort_seeds, P.test_segments_edge_cases]


def test_segments_restatement_passes_every_pin(monkeypatch):
    monkeypatch.setattr(oracle, "segments", lambda ids: _segments(ids))
    assert _failing_pins(SEGMENT_PINS) == []


@pytest.mark.parametrize("bug", ["unstable", "base_rows_last", "descending", "last_segment_dropped"])
def test_segments_pins_catch_planted_mistake(monkeypatch, bug):
    monkeypatch.setattr(oracle, "segments", lambda ids: _segments(ids, bug))
    assert _failing_pins(SEGMENT_PINS), f"no pin caught {bug}"
