"""Seeded synthetic inputs for the multi-tenant LoRA adapted linear layer.

This module only draws numbers: activations, base weights, adapter factors, per-row
adapter ids and prefill segment lengths, all as bf16 bit patterns (``np.uint16``).
It holds none of the layer's arithmetic, so both the fp64 oracle and the GPU path can
consume exactly the same bytes.

Recipe (shapes and distributions follow the pages' 70B example, "m07 — Multi-Adapter
(LoRA) Serving", section 2 "Scale Numbers": 80 layers, d=8192, GQA kv-dim 1024,
FFN 28672; init distributions and ids as stated for each workload below):

* every float is drawn as float32 from numpy's PCG64, multiplied by its standard
  deviation in float32, then rounded to bf16 with round-to-nearest-even;
* x ~ N(0, 1), W ~ N(0, 1/d_in), A ~ N(0, 1/d_in), B ~ N(0, 1/r);
* each array has its own seed key, so arrays can be generated independently and in any
  order; large arrays are filled in fixed 4 Mi-element chunks, chunk c drawing from
  ``SeedSequence(key + [c])``, so the bytes never depend on the thread count.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_CHUNK = 1 << 22

# seed-key tags, one per kind of array
_TAG_W, _TAG_X, _TAG_A, _TAG_B, _TAG_IDS, _TAG_RANKS, _TAG_LENS, _TAG_QUEUE = 1, 2, 3, 4, 5, 6, 7, 8


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even), returned as uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).copy()
    u += ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _pool_workers() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal_bf16(key, n: int, std: float) -> np.ndarray:
    """n values ~ N(0, std^2) as bf16 bits, reproducible from ``key`` alone."""
    key = [int(k) for k in key]
    out = np.empty(n, dtype=np.uint16)
    n_chunks = (n + _CHUNK - 1) // _CHUNK
    stdf = np.float32(std)

    def fill(c):
        s, e = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(key + [c])))
        a = g.standard_normal(e - s, dtype=np.float32)
        a *= stdf
        out[s:e] = f32_to_bf16_bits(a)

    if n_chunks <= 1:
        for c in range(n_chunks):
            fill(c)
    else:
        with ThreadPoolExecutor(_pool_workers()) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out


@dataclasses.dataclass
class Workload:
    """One synthetic adapted-layer workload.

    ``stages`` lists groups of modules that read the same input activation x (q/k/v read
    the layer's hidden state; o, the MLP and down each read their own input). Rows carry
    their adapter id in ``ids`` (decode; -1 = base only), or come as contiguous request
    segments ``seg_start``/``seg_adapter`` (prefill).
    """
    name: str
    modules: dict                      # name -> (d_in, d_out)
    stages: list                       # list of lists of module names
    n_rows: int
    n_adapters: int
    ranks: np.ndarray                  # int32 [n_adapters]
    scale: float
    seed: int = 0
    ids: np.ndarray | None = None      # int32 [n_rows] (decode)
    seg_start: np.ndarray | None = None   # int32 [n_seg + 1] (prefill)
    seg_adapter: np.ndarray | None = None  # int32 [n_seg]
    description: str = ""

    # ---- arrays (bf16 bits) -------------------------------------------------------
    def module_names(self):
        return [m for st in self.stages for m in st]

    def module_index(self, name):
        return self.module_names().index(name)

    def W(self, module: str) -> np.ndarray:
        d_in, d_out = self.modules[module]
        mi = self.module_index(module)
        return normal_bf16([self.seed, _TAG_W, mi], d_in * d_out, 1.0 / np.sqrt(d_in)).reshape(d_out, d_in)

    def x(self, stage: int) -> np.ndarray:
        d_in = self.modules[self.stages[stage][0]][0]
        return normal_bf16([self.seed, _TAG_X, stage], self.n_rows * d_in, 1.0).reshape(self.n_rows, d_in)

    def A(self, adapter: int, module: str) -> np.ndarray:
        d_in, _ = self.modules[module]
        r = int(self.ranks[adapter])
        mi = self.module_index(module)
        return normal_bf16([self.seed, _TAG_A, adapter, mi], r * d_in, 1.0 / np.sqrt(d_in)).reshape(r, d_in)

    def B(self, adapter: int, module: str) -> np.ndarray:
        _, d_out = self.modules[module]
        r = int(self.ranks[adapter])
        mi = self.module_index(module)
        return normal_bf16([self.seed, _TAG_B, adapter, mi], d_out * r, 1.0 / np.sqrt(r)).reshape(d_out, r)

    def row_adapters(self) -> np.ndarray:
        """Adapter id of every row (expands prefill segments)."""
        if self.ids is not None:
            return self.ids
        out = np.empty(self.n_rows, dtype=np.int32)
        for s in range(len(self.seg_adapter)):
            out[self.seg_start[s]:self.seg_start[s + 1]] = self.seg_adapter[s]
        return out

    def used_adapters(self) -> np.ndarray:
        a = self.row_adapters()
        return np.unique(a[a >= 0])


# ---- the pages' 70B shapes ---------------------------------------------------------
D70 = 8192
KV70 = 1024
FFN70 = 28672
ATTN70 = {"q": (D70, D70), "k": (D70, KV70), "v": (D70, KV70), "o": (D70, D70)}
MLP70 = {"gate": (D70, FFN70), "up": (D70, FFN70), "down": (FFN70, D70)}


def _perm_ids(n, seed):
    return np.random.default_rng([seed, _TAG_IDS]).permutation(n).astype(np.int32)


def tiny(seed=0):
    """d_in = d_out = 1024, 16 decode rows, 4 adapters of rank 8, ids uniform over {0..3}, scale 2."""
    ids = np.random.default_rng([seed, _TAG_IDS]).integers(0, 4, size=16).astype(np.int32)
    return Workload("tiny_1024_n16_r8", {"proj": (1024, 1024)}, [["proj"]], 16, 4,
                    np.full(4, 8, np.int32), 2.0, seed, ids=ids,
                    description="single adapted linear 1024x1024, 16 rows, 4 adapters r=8, s=2")


def attn70b_decode(seed=0, perm_seed=1):
    """70B attention projections (q/o 8192->8192, k/v 8192->1024), 128 rows, 128 distinct rank-8 adapters."""
    return Workload("attn70b_decode_b128_r8", dict(ATTN70), [["q", "k", "v"], ["o"]], 128, 128,
                    np.full(128, 8, np.int32), 1.0, seed, ids=_perm_ids(128, perm_seed),
                    description="70B attention layer decode, batch 128, 128 distinct adapters r=8")


def all70b_decode(seed=0, perm_seed=1):
    """All seven 70B projections, 128 rows, 128 distinct rank-64 adapters."""
    mods = dict(ATTN70)
    mods.update(MLP70)
    return Workload("all70b_decode_b128_r64", mods, [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]],
                    128, 128, np.full(128, 64, np.int32), 1.0, seed, ids=_perm_ids(128, perm_seed),
                    description="70B attention+MLP layer decode, batch 128, 128 distinct adapters r=64")


def zipf_pool(seed=0, n_adapters=5000, n_rows=256, zipf_s=1.1):
    """5000 resident attention adapters with ranks from {8,16,32,64} (p=.4,.3,.2,.1);
    256 rows whose ids follow a bounded Zipf(1.1) over the 5000 adapters."""
    g = np.random.default_rng([seed, _TAG_RANKS])
    ranks = g.choice(np.array([8, 16, 32, 64], np.int32), size=n_adapters, p=[0.4, 0.3, 0.2, 0.1]).astype(np.int32)
    k = np.arange(1, n_adapters + 1, dtype=np.float64)
    p = k ** (-zipf_s)
    cdf = np.cumsum(p / p.sum())
    u = np.random.default_rng([seed, _TAG_IDS]).random(n_rows)
    ids = np.minimum(np.searchsorted(cdf, u, side="right"), n_adapters - 1).astype(np.int32)
    return Workload("zipf_pool_5000_b256", dict(ATTN70), [["q", "k", "v"], ["o"]], n_rows, n_adapters,
                    ranks, 1.0, seed, ids=ids,
                    description="paged pool, 5000 resident attention adapters, mixed ranks, 256 Zipf(1.1) rows")


def prefill_segments(seed=0, n_req=64, lo=128, hi=2048, rank=16):
    """64 prompts with lengths uniform in [128, 2048], request j uses adapter j (rank 16);
    projections q, o (8192->8192) and gate (8192->28672)."""
    lens = np.random.default_rng([seed, _TAG_LENS]).integers(lo, hi + 1, size=n_req)
    seg_start = np.zeros(n_req + 1, np.int32)
    seg_start[1:] = np.cumsum(lens)
    mods = {"q": (D70, D70), "o": (D70, D70), "gate": (D70, FFN70)}
    return Workload("prefill_64seg_r16", mods, [["q"], ["o"], ["gate"]], int(seg_start[-1]), n_req,
                    np.full(n_req, rank, np.int32), 1.0, seed,
                    seg_start=seg_start, seg_adapter=np.arange(n_req, dtype=np.int32),
                    description="prefill segment path, 64 requests, lengths U[128,2048], 64 adapters r=16")


def custom(name, modules, stages, n_rows, ranks, scale, seed=0, ids=None, seg_start=None, seg_adapter=None):
    """A reduced workload with the same distributions (for parity tests the oracle finishes quickly)."""
    ranks = np.asarray(ranks, np.int32)
    return Workload(name, dict(modules), [list(s) for s in stages], int(n_rows), len(ranks), ranks, float(scale),
                    seed, ids=None if ids is None else np.asarray(ids, np.int32),
                    seg_start=None if seg_start is None else np.asarray(seg_start, np.int32),
                    seg_adapter=None if seg_adapter is None else np.asarray(seg_adapter, np.int32))


def random_ids(n, n_adapters, seed, p_base=0.0):
    """Uniform ids over the adapters; a fraction ``p_base`` of rows is base-only (-1)."""
    g = np.random.default_rng([seed, _TAG_IDS, 99])
    ids = g.integers(0, n_adapters, size=n).astype(np.int32)
    if p_base > 0:
        ids[g.random(n) < p_base] = -1
    return ids


def request_queue(n, seed=0, n_adapters=5000, zipf_s=1.1, max_wait_ms=400.0, p_base=0.0):
    """A waiting queue for the batch former: n requests in arrival order whose adapters follow the
    bounded Zipf(1.1) over n_adapters of ``zipf_pool`` (a fraction ``p_base`` base-only, -1), and
    how long each has waited: arrival times uniform over the last ``max_wait_ms``, so the queue's
    first request has waited longest.  Returns (adapter ids int32 [n], waited ms float64 [n])."""
    g = np.random.default_rng([seed, _TAG_QUEUE])
    k = np.arange(1, n_adapters + 1, dtype=np.float64)
    p = k ** (-zipf_s)
    cdf = np.cumsum(p / p.sum())
    ids = np.minimum(np.searchsorted(cdf, g.random(n), side="right"), n_adapters - 1).astype(np.int32)
    if p_base > 0:
        ids[g.random(n) < p_base] = -1
    waited = np.sort(g.random(n) * max_wait_ms)[::-1].copy()
    return ids, waited


ALL = {"tiny": tiny, "attn70b": attn70b_decode, "all70b": all70b_decode, "zipf": zipf_pool,
       "prefill": prefill_segments}
