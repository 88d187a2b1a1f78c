// lora_kernels.cu -- the device side of the adapted linear layer y_i = W x_i + s B_a (A_a x_i).
//
//   prep_decode_kernel    row grouping: stable sort of the rows by adapter id, plus id checks
//   prep_segments_kernel  checks a given contiguous segment table (prefill)
//   shrink_kernel         t_i = s * A_a x_i for every row (CUDA cores; bandwidth-bound)
//   gemm_kernel           base W x_i on tcgen05 tensor cores, with the expand s B_a t_i written
//                         into the TMEM accumulator before the base MMAs accumulate on top
//
// The forward is the one on "m07 -- Multi-Adapter (LoRA) Serving", section 6 "Deep Dive A:
// Batching Heterogeneous Adapters" (one batched base GEMM shared by the batch, plus a gathered
// per-row adapter product) and "LoRA, quotas and noisy neighbours", section "One weight read,
// many adapters" (rows tagged with their adapter, grouped, one kernel per layer).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "lora_internal.h"
#include "ptx.cuh"

namespace lora {

__device__ __forceinline__ void report(int32_t *err, int32_t code, int32_t detail) {
    if (err && atomicCAS(err, 0, code) == 0) err[1] = detail;
}

// ============================================================================ prep ==========

// Largest s in [0, n_seg) with seg_start[s] <= q (seg_start non-decreasing, seg_start[0] = 0).
__device__ __forceinline__ int seg_of(const int32_t *seg_start, int n_seg, int q) {
    int lo = 0, hi = n_seg - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(seg_start + mid) <= q) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ bool segments_valid(const PrepParams &p) {
    __shared__ int s_bad;
    if (threadIdx.x == 0) s_bad = 0;
    __syncthreads();
    if (p.n_seg_in < 1) {
        if (threadIdx.x == 0) s_bad = 1;
    } else {
        for (int s = threadIdx.x; s <= p.n_seg_in; s += blockDim.x) {
            int v = p.seg_start_in[s];
            bool bad = (s == 0 && v != 0) || (s == p.n_seg_in && v != p.n) || v < 0 || v > p.n ||
                       (s > 0 && v < p.seg_start_in[s - 1]);
            if (bad) s_bad = 1;
        }
    }
    __syncthreads();
    bool ok = s_bad == 0;
    __syncthreads();
    return ok;
}

__device__ int checked_id(const PrepParams &p, int id, int where) {
    if (id < -1 || id >= p.max_adapters) {
        report(p.err, LORA_DEVERR_BAD_ADAPTER, where);
        return -1;
    }
    if (id >= 0) {
        for (int m = 0; m < p.n_mod; ++m) {
            if (p.table[m][id].rank <= 0) {
                report(p.err, LORA_DEVERR_NOT_LOADED, where);
                return -1;
            }
        }
    }
    return id;
}

// One block of 256 threads, n <= 256 rows.  Position of row i in the stable order:
// #{j : id_j < id_i} + #{j < i : id_j == id_i}.
__global__ void __launch_bounds__(256) prep_decode_kernel(const PrepParams p) {
    __shared__ int s_id[256];
    __shared__ int s_sorted[256];
    __shared__ int s_scan[256];
    const int tid = threadIdx.x;
    const int n = p.n;
    bool seg_ok = true;
    if (p.ids == nullptr) {
        seg_ok = segments_valid(p);
        if (!seg_ok && tid == 0) report(p.err, LORA_DEVERR_BAD_SEGMENTS, 0);
    }
    int id = -1;
    if (tid < n) {
        if (p.ids) {
            id = checked_id(p, p.ids[tid], tid);
        } else if (seg_ok) {
            int s = seg_of(p.seg_start_in, p.n_seg_in, tid);
            id = checked_id(p, p.seg_adapter_in[s], s);
        }
        s_id[tid] = id;
    }
    __syncthreads();
    if (tid < n) {
        int pos = 0;
        for (int j = 0; j < n; ++j) {
            int v = s_id[j];
            pos += (v < id) || (v == id && j < tid);
        }
        p.perm[pos] = tid;
        s_sorted[pos] = id;
    }
    __syncthreads();
    int flag = (tid < n) && (tid == 0 || s_sorted[tid] != s_sorted[tid - 1]);
    s_scan[tid] = flag;
    __syncthreads();
    for (int off = 1; off < 256; off <<= 1) {
        int v = tid >= off ? s_scan[tid - off] : 0;
        __syncthreads();
        s_scan[tid] += v;
        __syncthreads();
    }
    if (flag) {
        int seg = s_scan[tid] - 1;
        p.seg_start[seg] = tid;
        p.seg_adapter[seg] = s_sorted[tid];
    }
    if (tid == 0) {
        int ns = n > 0 ? s_scan[n - 1] : 0;
        *p.n_seg = ns;
        p.seg_start[ns] = n;
    }
}

// Grouped rows (prefill): validate the table, copy it into the workspace with unusable
// adapters replaced by -1 (base only).  A malformed table becomes one base-only segment.
__global__ void __launch_bounds__(1024) prep_segments_kernel(const PrepParams p) {
    const bool ok = segments_valid(p);
    if (!ok) {
        if (threadIdx.x == 0) {
            report(p.err, LORA_DEVERR_BAD_SEGMENTS, 0);
            p.seg_start[0] = 0;
            p.seg_start[1] = p.n;
            p.seg_adapter[0] = -1;
            *p.n_seg = 1;
        }
        return;
    }
    for (int s = threadIdx.x; s <= p.n_seg_in; s += blockDim.x) {
        p.seg_start[s] = p.seg_start_in[s];
        if (s < p.n_seg_in) p.seg_adapter[s] = checked_id(p, p.seg_adapter_in[s], s);
    }
    if (threadIdx.x == 0) *p.n_seg = p.n_seg_in;
}

__global__ void table_write_kernel(PoolEntry *dst, PoolEntry v) { *dst = v; }

// ========================================================================== shrink ==========
//
// t_q[j] = s * sum_k A_a[j, k] x_row(q)[k] for every sorted position q, j < rp (zero for
// j >= rank).  Block (unit, split): a unit is one segment (decode) or 64 consecutive
// positions (grouped rows); a split is a K range.  With several splits the partial sums go
// to the workspace and the last block to finish (atomic counter) adds them in split order,
// so the result does not depend on block timing.

__device__ __forceinline__ float dot8_bf16(uint4 a, uint4 b) {
    float r = bf16lo(a.x) * bf16lo(b.x);
    r = fmaf(bf16hi(a.x), bf16hi(b.x), r);
    r = fmaf(bf16lo(a.y), bf16lo(b.y), r);
    r = fmaf(bf16hi(a.y), bf16hi(b.y), r);
    r = fmaf(bf16lo(a.z), bf16lo(b.z), r);
    r = fmaf(bf16hi(a.z), bf16hi(b.z), r);
    r = fmaf(bf16lo(a.w), bf16lo(b.w), r);
    r = fmaf(bf16hi(a.w), bf16hi(b.w), r);
    return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__global__ void __launch_bounds__(kShrinkThreads) shrink_kernel(const __grid_constant__ ShrinkParams p) {
    __shared__ __align__(16) uint16_t xs[kShrinkRows * kShrinkKSub];
    __shared__ int s_last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int m = 0;
    while (m + 1 < p.n_mod && p.split_begin[m + 1] <= (int)blockIdx.y) ++m;
    const int kc = blockIdx.y - p.split_begin[m];
    const int ks = p.ksplit[m];
    if (kc >= ks) return;
    const int n_seg = *p.n_seg;
    const int u = blockIdx.x;
    int qlo, qhi, s;
    if (p.by_segment) {
        if (u >= n_seg) return;
        s = u;
        qlo = p.seg_start[s];
        qhi = p.seg_start[s + 1];
    } else {
        qlo = u * kShrinkGroupRows;
        if (qlo >= p.n) return;
        qhi = min(p.n, qlo + kShrinkGroupRows);
        s = seg_of(p.seg_start, n_seg, qlo);
    }
    const int d_in = p.d_in[m];
    const int kbeg = kc * p.kc[m];
    const int kend = min(d_in, kbeg + p.kc[m]);
    const uint16_t *x = p.x[m];
    float *T = p.T[m];
    const int rpmax = p.rpmax;

    for (int q = qlo; q < qhi;) {
        while (s + 1 < n_seg && p.seg_start[s + 1] <= q) ++s;
        int qe = min(qhi, p.seg_start[s + 1]);
        if (qe <= q) qe = q + 1;  // inconsistent table: still make progress, stay in bounds
        const int a = p.seg_adapter[s];
        int r = 0, rp = 0;
        const uint16_t *A = nullptr;
        if (a >= 0) {
            const PoolEntry *e = p.table[m] + a;
            r = e->rank;
            rp = e->rp;
            A = e->A;
        }
        for (int qb = q; qb < qe; qb += kShrinkRows) {
            const int nr = min(kShrinkRows, qe - qb);
            float acc[8][kShrinkRows];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
#pragma unroll
                for (int rr = 0; rr < kShrinkRows; ++rr) acc[jj][rr] = 0.f;
            if (r > 0) {
                for (int k0 = kbeg; k0 < kend; k0 += kShrinkKSub) {
                    const int kl = min(kShrinkKSub, kend - k0);
                    __syncthreads();
                    for (int idx = tid; idx < nr * (kShrinkKSub / 8); idx += kShrinkThreads) {
                        const int rr = idx / (kShrinkKSub / 8);
                        const int k = (idx % (kShrinkKSub / 8)) * 8;
                        const int row = p.perm ? p.perm[qb + rr] : qb + rr;
                        uint4 v = make_uint4(0, 0, 0, 0);
                        if (k < kl) v = __ldg(reinterpret_cast<const uint4 *>(x + (size_t)row * d_in + k0 + k));
                        *reinterpret_cast<uint4 *>(xs + rr * kShrinkKSub + k) = v;
                    }
                    __syncthreads();
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        const int j = warp + 8 * jj;
                        if (j < r) {
                            const uint16_t *Aj = A + (size_t)j * d_in + k0;
#pragma unroll 4
                            for (int kk = lane * 8; kk < kl; kk += 256) {
                                const uint4 av = __ldg(reinterpret_cast<const uint4 *>(Aj + kk));
#pragma unroll
                                for (int rr = 0; rr < kShrinkRows; ++rr) {
                                    if (rr < nr) {
                                        const uint4 xv = *reinterpret_cast<const uint4 *>(xs + rr * kShrinkKSub + kk);
                                        acc[jj][rr] += dot8_bf16(av, xv);
                                    }
                                }
                            }
                        }
                    }
                }
            }
            // reduce across the warp's lanes and write t (or the split's partial sum)
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = warp + 8 * jj;
                if (j < rp) {
#pragma unroll
                    for (int rr = 0; rr < kShrinkRows; ++rr) {
                        if (rr < nr) {
                            float v = (j < r) ? warp_sum(acc[jj][rr]) : 0.f;
                            if (lane == 0) {
                                if (ks == 1)
                                    T[(size_t)(qb + rr) * rpmax + j] = p.scale * v;
                                else
                                    p.partials[(((size_t)m * p.ks_max + kc) * p.n + (qb + rr)) * rpmax + j] = v;
                            }
                        }
                    }
                }
            }
        }
        q = qe;
    }
    if (ks == 1) return;

    // several K splits (decode, one segment per block): the last block adds them up in order
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        int old = atomicAdd(p.counters + m * p.max_units + u, 1);
        s_last = (old == ks - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int a = p.seg_adapter[s];
    const int rp = a >= 0 ? p.table[m][a].rp : 0;
    const int len = qhi - qlo;
    for (int idx = tid; idx < len * rp; idx += kShrinkThreads) {
        const int q = qlo + idx / rp, j = idx % rp;
        float v = 0.f;
        for (int c = 0; c < ks; ++c) v += __ldcg(p.partials + (((size_t)m * p.ks_max + c) * p.n + q) * rpmax + j);
        T[(size_t)q * rpmax + j] = p.scale * v;
    }
    if (tid == 0) p.counters[m * p.max_units + u] = 0;
}

// Decode shrink: one block per (segment, 2048-wide K split, module).  Each warp takes one rank
// row per pass and every lane issues its eight 16-byte loads of A up front (32 KiB of A in
// flight per block and pass), then reads the segment's x rows straight from L2.  Partial sums
// of the splits are combined by the last block of the segment, in split order.
__global__ void __launch_bounds__(kShrinkThreads, 2) shrink_decode_kernel(const __grid_constant__ ShrinkParams p) {
    __shared__ int s_last;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int m = 0;
    while (m + 1 < p.n_mod && p.split_begin[m + 1] <= (int)blockIdx.y) ++m;
    const int kc = blockIdx.y - p.split_begin[m];
    const int ks = p.ksplit[m];
    if (kc >= ks) return;
    const int u = blockIdx.x;
    if (u >= *p.n_seg) return;
    const int qlo = p.seg_start[u], qhi = p.seg_start[u + 1];
    const int a = p.seg_adapter[u];
    const int d_in = p.d_in[m];
    const int kbeg = kc * p.kc[m];
    const int kend = min(d_in, kbeg + p.kc[m]);
    const uint16_t *x = p.x[m];
    const int rpmax = p.rpmax;
    int r = 0, rp = 0;
    const uint16_t *A = nullptr;
    if (a >= 0) {
        const PoolEntry *e = p.table[m] + a;
        r = e->rank;
        rp = e->rp;
        A = e->A;
    }
    for (int j0 = 0; j0 < r; j0 += kShrinkThreads / 32) {
        const int j = j0 + warp;
        if (j >= r) break;  // warp-uniform
        uint4 av[kShrinkDecCh];
#pragma unroll
        for (int c = 0; c < kShrinkDecCh; ++c) {
            const int kk = kbeg + lane * 8 + 256 * c;
            av[c] = kk < kend ? __ldg(reinterpret_cast<const uint4 *>(A + (size_t)j * d_in + kk)) : make_uint4(0, 0, 0, 0);
        }
        for (int qb = qlo; qb < qhi; qb += kShrinkDecRows) {
            float acc[kShrinkDecRows];
#pragma unroll
            for (int rr = 0; rr < kShrinkDecRows; ++rr) {
                acc[rr] = 0.f;
                if (qb + rr < qhi) {
                    const uint16_t *xr = x + (size_t)p.perm[qb + rr] * d_in;
                    uint4 xv[kShrinkDecCh];
#pragma unroll
                    for (int c = 0; c < kShrinkDecCh; ++c) {
                        const int kk = kbeg + lane * 8 + 256 * c;
                        xv[c] = kk < kend ? __ldg(reinterpret_cast<const uint4 *>(xr + kk)) : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                    for (int c = 0; c < kShrinkDecCh; ++c) acc[rr] += dot8_bf16(av[c], xv[c]);
                }
            }
#pragma unroll
            for (int rr = 0; rr < kShrinkDecRows; ++rr) {
                if (qb + rr < qhi) {
                    const float v = warp_sum(acc[rr]);
                    if (lane == 0) {
                        if (ks == 1)
                            p.T[m][(size_t)(qb + rr) * rpmax + j] = p.scale * v;
                        else
                            p.partials[(((size_t)m * p.ks_max + kc) * p.n + (qb + rr)) * rpmax + j] = v;
                    }
                }
            }
        }
    }
    if (ks == 1) {
        for (int idx = tid; idx < (qhi - qlo) * (rp - r); idx += kShrinkThreads)
            p.T[m][(size_t)(qlo + idx / (rp - r)) * rpmax + r + idx % (rp - r)] = 0.f;
        return;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(p.counters + m * p.max_units + u, 1) == ks - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int idx = tid; idx < (qhi - qlo) * rp; idx += kShrinkThreads) {
        const int q = qlo + idx / rp, j = idx % rp;
        float v = 0.f;
        if (j < r)
            for (int c = 0; c < ks; ++c) v += __ldcg(p.partials + (((size_t)m * p.ks_max + c) * p.n + q) * rpmax + j);
        p.T[m][(size_t)q * rpmax + j] = p.scale * v;
    }
    if (tid == 0) p.counters[m * p.max_units + u] = 0;
}

// ============================================================================ gemm ==========

struct Item {
    int32_t m, w_tile, chunk, kb0, kb1, kbn, tile;
    int64_t it0;  // flattened index of the tile's first k-block
};

__device__ __forceinline__ void tile_coords(const GemmParams &p, int m, int lt, Item &it) {
    // grouped raster: raster_group W tiles x all row chunks, W-tile fastest
    const int C = p.n_chunks, MT = p.mod[m].m_tiles, G = p.raster_group;
    const int grp = lt / (G * C);
    const int rem = lt - grp * G * C;
    const int gw = min(G, MT - grp * G);
    it.chunk = rem / gw;
    it.w_tile = grp * G + rem % gw;
}

struct Sched {
    int64_t x, e;
    int32_t j, cta;
    __device__ void begin(const GemmParams &p, int c) {
        cta = c;
        j = 0;
        if (p.stream_k) {
            x = (int64_t)c * p.total_iters / p.n_cta;
            e = (int64_t)(c + 1) * p.total_iters / p.n_cta;
        }
    }
    __device__ bool next(const GemmParams &p, Item &it) {
        if (p.stream_k) {
            if (x >= e) return false;
            int m = 0;
            while (m + 1 < p.n_mod && p.mod[m + 1].iter_begin <= x) ++m;
            const int kbn = p.mod[m].k_blocks;
            const int64_t local = x - p.mod[m].iter_begin;
            const int lt = (int)(local / kbn);
            it.m = m;
            it.kbn = kbn;
            it.kb0 = (int)(local - (int64_t)lt * kbn);
            it.kb1 = (int)((e - x) < (int64_t)(kbn - it.kb0) ? it.kb0 + (e - x) : kbn);
            it.tile = p.mod[m].tile_begin + lt;
            it.it0 = p.mod[m].iter_begin + (int64_t)lt * kbn;
            tile_coords(p, m, lt, it);
            x += it.kb1 - it.kb0;
            return true;
        }
        const int t = cta + j * p.n_cta;
        if (t >= p.total_tiles) return false;
        ++j;
        int m = 0;
        while (m + 1 < p.n_mod && p.mod[m + 1].tile_begin <= t) ++m;
        const int lt = t - p.mod[m].tile_begin;
        it.m = m;
        it.kbn = p.mod[m].k_blocks;
        it.kb0 = 0;
        it.kb1 = it.kbn;
        it.tile = t;
        it.it0 = 0;
        tile_coords(p, m, lt, it);
        return true;
    }
};

// CTA whose stream-K range holds flattened iteration x.
__device__ __forceinline__ int cta_of(const GemmParams &p, int64_t x) {
    return (int)(((x + 1) * p.n_cta - 1) / p.total_iters);
}

// Expand metadata staged in shared memory by the epilogue warps (no global-latency chains in
// the per-unit loop): the row order (decode) and, for the segments the current tile touches,
// their first position, B factor address and storage rank.
struct EpiMeta {
    uint64_t wB[kMaxWin];      // B factor base of the window's segments (0 = base only)
    int32_t perm[kMaxWin];     // decode: sorted position -> row
    int32_t wss[kMaxWin + 4];  // window segment starts (clipped to the tile), wss[count] = qhi
    int32_t wrp[kMaxWin];      // storage rank (0 = base only)
    int32_t count;             // segments in the window
    int32_t module;            // module the window was built for (decode caching)
    int32_t qlo, qhi;
};

struct Unit {
    int32_t k, qa, qe;  // window segment, positions [qa, qe)
};

// Expand units of one tile: runs of at most unit_rows positions inside one window segment.
struct UnitCursor {
    int32_t k, q;
    __device__ void begin(const EpiMeta &w) {
        k = 0;
        q = w.qlo;
    }
    __device__ bool next(const GemmParams &p, const EpiMeta &w, Unit &u) {
        if (q >= w.qhi) return false;
        while (k + 1 < w.count && w.wss[k + 1] <= q) ++k;
        int qe = min(min(w.wss[k + 1], w.qhi), q + p.unit_rows);
        if (qe <= q) qe = q + 1;  // inconsistent table: still make progress, stay in bounds
        u.k = k;
        u.qa = q;
        u.qe = qe;
        q = qe;
        return true;
    }
};

struct EpiCtx {
    const GemmParams *p;
    uint8_t *ring;
    uint64_t *slot_bar;
    EpiMeta *meta;
    uint32_t tmem_base;
    uint32_t delta_col;  // first TMEM column of the expand (delta) region
    int etid;            // 0..127 among epilogue threads
    int o;               // TMEM lane = W row within the tile
    int lane_base;       // first TMEM lane of this warp
    int lane;
    uint32_t g_unit;     // expand units processed by this CTA so far (ring slot / parity)
};

// (Re)build the segment window for a tile: every segment overlapping its positions
// [qlo, qhi), with the factor addresses of module m.  Decode tiles of one module share the
// window, so it is rebuilt only when the module changes.
__device__ void build_window(EpiCtx &c, const Item &it) {
    const GemmParams &p = *c.p;
    EpiMeta &w = *c.meta;
    const int row0 = it.chunk * p.nt;
    if (p.decode && w.module == it.m) return;
    named_bar_sync(1, 128);  // nobody still reads the old window
    const int n_seg = *p.n_seg;
    int s0, cnt, qlo, qhi;
    if (p.decode) {
        qlo = 0;
        qhi = p.n;
        s0 = 0;
        cnt = min(n_seg, kMaxWin);
    } else {
        qlo = row0;
        qhi = min(p.n, row0 + p.nt);
        s0 = seg_of(p.seg_start, n_seg, qlo);
        const int s1 = seg_of(p.seg_start, n_seg, qhi - 1);
        cnt = min(s1 - s0 + 1, kMaxWin);
    }
    const PoolEntry *table = p.mod[it.m].table;
    for (int i = c.etid; i < cnt; i += 128) {
        const int s = s0 + i;
        const int a = __ldg(p.seg_adapter + s);
        w.wss[i] = max(__ldg(p.seg_start + s), qlo);
        uint64_t b = 0;
        int rp = 0;
        if (a >= 0) {
            b = reinterpret_cast<uint64_t>(table[a].B);
            rp = table[a].rp;
        }
        w.wB[i] = b;
        w.wrp[i] = rp;
    }
    if (c.etid == 0) {
        w.wss[cnt] = qhi;
        w.count = cnt;
        w.qlo = qlo;
        w.qhi = qhi;
        w.module = it.m;
    }
    named_bar_sync(1, 128);
}

// Stage one expand unit into a ring slot: the adapter's B rows [o0, o0 + 128) (cp.async,
// 16-byte chunks XOR-swizzled by row so each thread later reads its own row without bank
// conflicts) and the unit's t rows.  Every epilogue thread arrives on the slot barrier once
// its copies land.
__device__ void issue_unit(EpiCtx &c, const Item &it, const Unit &u, int slot) {
    const GemmParams &p = *c.p;
    const GemmModule &M = p.mod[it.m];
    const EpiMeta &w = *c.meta;
    const int rp = w.wrp[u.k];
    if (rp > 0) {
        const uint16_t *B = reinterpret_cast<const uint16_t *>(w.wB[u.k]);
        const uint32_t sbase = smem_u32(c.ring + (size_t)slot * p.slot_bytes);
        const int lg = __ffs(rp >> 3) - 1;  // log2(rp / 8)
        const int nch = 1 << lg;
        const int sh = 3 - lg;
        const int o0 = it.w_tile * kBM;
        for (int idx = c.etid; idx < (kBM << lg); idx += 128) {
            const int row = idx >> lg, ch = idx & (nch - 1);
            const int o = o0 + row;
            const bool v = o < M.d_out;
            const uint16_t *src = v ? B + (size_t)o * rp + ch * 8 : B;
            cp_async_16(sbase + (uint32_t)(((row << lg) + (ch ^ ((row >> sh) & (nch - 1)))) * 16), src,
                        v ? 16u : 0u);
        }
        const int tch = rp >> 2;
        const int rows = u.qe - u.qa;
        const float *Tsrc = M.T + (size_t)u.qa * p.rpmax;
        const uint32_t tbase = sbase + (uint32_t)(kBM * p.rpmax * 2);
        for (int idx = c.etid; idx < rows * tch; idx += 128) {
            const int r = idx / tch, ch = idx - r * tch;
            cp_async_16(tbase + (uint32_t)((r * rp + ch * 4) * 4), Tsrc + (size_t)r * p.rpmax + ch * 4, 16u);
        }
    }
    cp_async_arrive_noinc(c.slot_bar + slot);
}

template <int RP>
__device__ __forceinline__ void apply_unit(EpiCtx &c, const Unit &u, const uint8_t *sb, uint32_t tcol0, int row0) {
    constexpr int LG = (RP == 8) ? 0 : (RP == 16) ? 1 : (RP == 32) ? 2 : 3;
    constexpr int NCH = 1 << LG;
    constexpr int SH = 3 - LG;
    const GemmParams &p = *c.p;
    const EpiMeta &w = *c.meta;
    uint32_t b[RP / 2];
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
        const uint4 v = *reinterpret_cast<const uint4 *>(sb + ((c.o << LG) + (ch ^ ((c.o >> SH) & (NCH - 1)))) * 16);
        b[4 * ch + 0] = v.x;
        b[4 * ch + 1] = v.y;
        b[4 * ch + 2] = v.z;
        b[4 * ch + 3] = v.w;
    }
    const float *Ts = reinterpret_cast<const float *>(sb + kBM * p.rpmax * 2);
    for (int q = u.qa; q < u.qe; ++q) {
        const float4 *t4 = reinterpret_cast<const float4 *>(Ts + (q - u.qa) * RP);
        float acc = 0.f;
#pragma unroll
        for (int j4 = 0; j4 < RP / 4; ++j4) {
            const float4 tv = t4[j4];
            acc = fmaf(bf16lo(b[2 * j4]), tv.x, acc);
            acc = fmaf(bf16hi(b[2 * j4]), tv.y, acc);
            acc = fmaf(bf16lo(b[2 * j4 + 1]), tv.z, acc);
            acc = fmaf(bf16hi(b[2 * j4 + 1]), tv.w, acc);
        }
        const int col = p.decode ? w.perm[q] : q - row0;
        tmem_st1(tcol0 + (uint32_t)col, acc);
    }
}

// Expand for a tile this CTA heads: delta[o, col(q)] = sum_j B_a[o0 + o, j] * t_q[j] for every
// position q of the tile (0 for base-only rows), written into the TMEM delta region.  It runs
// while the MMA warp works on the same tile; the drain adds it to the accumulator.
__device__ bool init_expand(EpiCtx &c, const Item &it, volatile int *abort_flag) {
    const GemmParams &p = *c.p;
    build_window(c, it);
    const EpiMeta &w = *c.meta;
    const int row0 = it.chunk * p.nt;
    const uint32_t tcol0 = c.tmem_base + ((uint32_t)c.lane_base << 16) + c.delta_col;
    UnitCursor ic, cc;
    ic.begin(w);
    cc.begin(w);
    const uint32_t base = c.g_unit;
    uint32_t issued = 0, consumed = 0;
    Unit u;
    while (issued < (uint32_t)p.n_slots && ic.next(p, w, u)) {
        issue_unit(c, it, u, (base + issued) % p.n_slots);
        ++issued;
    }
    bool ok = true;
    while (cc.next(p, w, u)) {
        const uint32_t k = base + consumed;
        const int slot = k % p.n_slots;
        const bool landed = mbar_wait(c.slot_bar + slot, (k / p.n_slots) & 1, abort_flag, p.err);
        {
            // runs even if the wait gave up (the warp-wide TMEM stores need every lane); the
            // values are then meaningless but every access stays in bounds
            const uint8_t *sb = c.ring + (size_t)slot * p.slot_bytes;
            switch (w.wrp[u.k]) {
                case 8: apply_unit<8>(c, u, sb, tcol0, row0); break;
                case 16: apply_unit<16>(c, u, sb, tcol0, row0); break;
                case 32: apply_unit<32>(c, u, sb, tcol0, row0); break;
                case 64: apply_unit<64>(c, u, sb, tcol0, row0); break;
                default:
                    for (int q = u.qa; q < u.qe; ++q) {
                        const int col = p.decode ? w.perm[q] : q - row0;
                        tmem_st1(tcol0 + (uint32_t)col, 0.f);
                    }
            }
        }
        // every thread is done with the slot; leave together if any wait gave up
        const bool any_failed = named_bar_or(1, 128, !landed);
        ++consumed;
        if (any_failed) {
            ok = false;
            break;
        }
        if (ic.next(p, w, u)) {
            issue_unit(c, it, u, (base + issued) % p.n_slots);
            ++issued;
        }
    }
    // A timed-out wait can leave copies in flight: let them land before the slot is reused.
    while (consumed < issued) {
        const uint32_t k = base + consumed;
        mbar_wait(c.slot_bar + (k % p.n_slots), (k / p.n_slots) & 1, abort_flag, p.err);
        ++consumed;
    }
    c.g_unit = base + consumed;
    tmem_st_wait();
    return ok;
}

__device__ __forceinline__ void store_y(const GemmParams &p, const GemmModule &M, int row, int oo, float v) {
    if (p.y_bf16) {
        reinterpret_cast<uint16_t *>(M.y)[(size_t)row * M.d_out + oo] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    } else {
        reinterpret_cast<float *>(M.y)[(size_t)row * M.d_out + oo] = v;
    }
}

__device__ __forceinline__ void ld_cols16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    tmem_ld16(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// This CTA's share of a tile: accumulator (+ the expand delta when it heads the tile).
__device__ __forceinline__ void own_cols16(const EpiCtx &c, uint32_t tacc, bool head, int c0, float (&v)[16]) {
    ld_cols16(tacc + c0, v);
    if (head) {
        float d[16];
        ld_cols16(c.tmem_base + ((uint32_t)c.lane_base << 16) + c.delta_col + c0, d);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] += d[i];
    }
}

// Accumulator -> y.  A tile split over several CTAs (stream-K) is finished by the last CTA
// to get there (atomic counter); it adds the pieces in k order, so the sum never depends on
// timing.  No CTA ever waits for another.
__device__ void drain(EpiCtx &c, const Item &it, int buf, volatile int *misc_flag) {
    const GemmParams &p = *c.p;
    const GemmModule &M = p.mod[it.m];
    const int row0 = it.chunk * p.nt;
    const int ncols = p.decode ? p.n : min(p.nt, p.n - row0);
    const int ncols16 = (ncols + 15) & ~15;
    const int oo = it.w_tile * kBM + c.o;
    const bool o_ok = oo < M.d_out;
    const bool head = it.kb0 == 0;
    const uint32_t tacc = c.tmem_base + ((uint32_t)c.lane_base << 16) + (uint32_t)(buf * p.nt);
    const size_t slot_elems = (size_t)kBM * p.nt;

    if (head && it.kb1 == it.kbn) {
        for (int c0 = 0; c0 < ncols16; c0 += 16) {
            float v[16];
            own_cols16(c, tacc, true, c0, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int col = c0 + i;
                if (col < ncols && o_ok) store_y(p, M, p.decode ? col : row0 + col, oo, v[i]);
            }
        }
        return;
    }

    // ---- partial tile (stream-K) ----
    const int c_first = cta_of(p, it.it0);
    const int c_last = cta_of(p, it.it0 + it.kbn - 1);
    const int nc = c_last - c_first + 1;
    int32_t *counter = p.tile_counters + it.tile;
    bool finalize = false;
    if (head) {  // the head usually arrives last: finish directly if everyone else is in
        if (c.etid == 0) *misc_flag = (atomicAdd(counter, 0) == nc - 1);
        named_bar_sync(1, 128);
        finalize = *misc_flag != 0;
        named_bar_sync(1, 128);
    }
    if (!finalize) {
        const int64_t my_b = (int64_t)blockIdx.x * p.total_iters / p.n_cta;
        const int my_slot = (my_b >= it.it0) ? 0 : 1;
        float *dst = p.partials + ((size_t)blockIdx.x * 2 + my_slot) * slot_elems;
        for (int c0 = 0; c0 < ncols16; c0 += 16) {
            float v[16];
            own_cols16(c, tacc, head, c0, v);
#pragma unroll
            for (int i = 0; i < 16; ++i)
                if (c0 + i < ncols) dst[(size_t)(c0 + i) * kBM + c.o] = v[i];
        }
        __threadfence();
        named_bar_sync(1, 128);
        if (c.etid == 0) *misc_flag = (atomicAdd(counter, 1) == nc - 1);
        named_bar_sync(1, 128);
        finalize = *misc_flag != 0;
        named_bar_sync(1, 128);
    }
    if (!finalize) return;
    __threadfence();
    for (int c0 = 0; c0 < ncols16; c0 += 16) {
        float own[16], sum[16];
        own_cols16(c, tacc, head, c0, own);
        for (int jc = 0; jc < nc; ++jc) {
            const int cc = c_first + jc;
            float v[16];
            if (cc == (int)blockIdx.x) {
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = own[i];
            } else {
                const int64_t b_c = (int64_t)cc * p.total_iters / p.n_cta;
                const int sl = (b_c >= it.it0) ? 0 : 1;
                const float *src = p.partials + ((size_t)cc * 2 + sl) * slot_elems;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    v[i] = (c0 + i < ncols) ? __ldcg(src + (size_t)(c0 + i) * kBM + c.o) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) sum[i] = (jc == 0) ? v[i] : sum[i] + v[i];
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int col = c0 + i;
            if (col < ncols && o_ok) store_y(p, M, p.decode ? col : row0 + col, oo, sum[i]);
        }
    }
    if (c.etid == 0) *counter = 0;
}

__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.n_stages;
    const int NB = p.n_acc;
    const uint32_t a_bytes = kBM * kBK * 2;
    const uint32_t b_bytes = (uint32_t)p.nt * kBK * 2;
    const uint32_t stage_bytes = a_bytes + b_bytes;
    uint8_t *ring = smem + (size_t)S * stage_bytes;
    EpiMeta *meta = reinterpret_cast<EpiMeta *>(ring + (size_t)p.n_slots * p.slot_bytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(meta + 1);
    uint64_t *empty = full + S;
    uint64_t *acc_full = empty + S;
    uint64_t *acc_free = acc_full + 2;
    uint64_t *mma_done = acc_free + 2;
    uint64_t *slot_bar = mma_done + 1;
    uint32_t *misc = reinterpret_cast<uint32_t *>(slot_bar + p.n_slots);  // [0] tmem, [1] abort, [2] flag

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_free + b, kEpiWarps);
        }
        mbar_init(mma_done, 1);
        for (int s = 0; s < p.n_slots; ++s) mbar_init(slot_bar + s, 128);
        misc[1] = 0;
        misc[2] = 0;
        meta->module = -1;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int m = 0; m < p.n_mod; ++m) {
            tma_prefetch_desc(&p.mod[m].tmW);
            tma_prefetch_desc(&p.mod[m].tmX);
        }
    }
    if (warp == 1) tmem_alloc(misc, (uint32_t)p.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = misc[0];
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ TMA producer
            const uint64_t pol_w = p.decode ? l2_policy_evict_first() : l2_policy_evict_normal();
            const uint64_t pol_x = l2_policy_evict_last();
            Sched sc;
            sc.begin(p, blockIdx.x);
            Item it;
            uint32_t k = 0;  // stage fills issued
            bool ok = true;
            while (ok && sc.next(p, it)) {
                const GemmModule &M = p.mod[it.m];
                const int o0 = it.w_tile * kBM, row0 = it.chunk * p.nt;
                for (int kb = it.kb0; kb < it.kb1; ++kb, ++k) {
                    const int s = k % S;
                    if (!mbar_wait(empty + s, ((k / S) & 1) ^ 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    uint8_t *sa = smem + (size_t)s * stage_bytes;
                    mbar_arrive_expect_tx(full + s, stage_bytes);
                    tma_load_2d(sa, &M.tmW, full + s, kb * kBK, o0, pol_w);
                    tma_load_2d(sa + a_bytes, &M.tmX, full + s, kb * kBK, row0, pol_x);
                }
            }
            // never leave the block with copies still landing in its shared memory
            for (uint32_t q = (k > (uint32_t)S ? k - S : 0); q < k; ++q) {
                const uint32_t a = smem_u32(full + (q % S));
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(a, (q / S) & 1) && globaltimer() - t0 < kWaitBudgetNs) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            const uint32_t idesc = idesc_bf16_f32(kBM, (uint32_t)p.nt);
            Sched sc;
            sc.begin(p, blockIdx.x);
            Item it;
            uint32_t k = 0, li = 0;
            bool ok = true;
            while (ok && sc.next(p, it)) {
                const int buf = li % NB;
                const uint32_t use = li / NB;
                if (!mbar_wait(acc_free + buf, (use & 1) ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * p.nt);
                for (int kb = it.kb0; kb < it.kb1; ++kb, ++k) {
                    const int s = k % S;
                    if (!mbar_wait(full + s, (k / S) & 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)s * stage_bytes);
                    const uint64_t da = sdesc_kmajor_sw128(sa);
                    const uint64_t db = sdesc_kmajor_sw128(sa + a_bytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint32_t accum = (kb > it.kb0 || kk > 0) ? 1u : 0u;
                        umma_bf16(d, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2), idesc, accum);
                    }
                    umma_commit(empty + s);
                }
                if (!ok) break;
                umma_commit(acc_full + buf);
                ++li;
            }
            umma_commit(mma_done);
            const uint32_t a = smem_u32(mma_done);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(a, 0) && globaltimer() - t0 < kWaitBudgetNs) {
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        EpiCtx c;
        c.p = &p;
        c.ring = ring;
        c.slot_bar = slot_bar;
        c.meta = meta;
        c.tmem_base = tmem_base;
        c.delta_col = (uint32_t)(NB * p.nt);
        c.etid = threadIdx.x - 64;
        c.lane = lane;
        c.lane_base = (warp & 3) * 32;
        c.o = c.lane_base + lane;
        c.g_unit = 0;
        if (p.decode)
            for (int i = c.etid; i < p.n; i += 128) meta->perm[i] = __ldg(p.perm + i);
        volatile int *flag = reinterpret_cast<volatile int *>(misc + 2);
        Sched sc;
        sc.begin(p, blockIdx.x);
        Item it;
        uint32_t li = 0;
        while (sc.next(p, it)) {
            const int buf = li % NB;
            bool ok = true;
            if (it.kb0 == 0) ok = init_expand(c, it, abort_flag);
            const bool full_ok = mbar_wait(acc_full + buf, (li / NB) & 1, abort_flag, p.err);
            if (named_bar_or(1, 128, !(full_ok && ok))) break;
            tc_fence_after();
            drain(c, it, buf, flag);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free + buf);
            ++li;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
    }
}

// ====================================================================== launchers ==========

size_t gemm_smem_bytes(int nt, int n_stages, int n_slots, int slot_bytes) {
    const size_t stage = (size_t)kBM * kBK * 2 + (size_t)nt * kBK * 2;
    return 1024 + stage * n_stages + (size_t)n_slots * slot_bytes + sizeof(EpiMeta) +
           8 * (2 * (size_t)n_stages + 5 + n_slots) + 16;
}

cudaError_t launch_prep_decode(const PrepParams &p, cudaStream_t s) {
    prep_decode_kernel<<<1, 256, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_prep_segments(const PrepParams &p, cudaStream_t s) {
    prep_segments_kernel<<<1, 1024, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_shrink(const ShrinkParams &p, int grid_x, int grid_y, cudaStream_t s) {
    if (p.by_segment)
        shrink_decode_kernel<<<dim3(grid_x, grid_y), kShrinkThreads, 0, s>>>(p);
    else
        shrink_kernel<<<dim3(grid_x, grid_y), kShrinkThreads, 0, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_gemm(const GemmParams &p, size_t smem_bytes, cudaStream_t s) {
    static size_t configured = 0;
    if (smem_bytes > configured) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
        if (e != cudaSuccess) return e;
        configured = smem_bytes;
    }
    gemm_kernel<<<p.n_cta, kGemmThreads, smem_bytes, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_table_write(PoolEntry *dst, PoolEntry value, cudaStream_t s) {
    table_write_kernel<<<1, 1, 0, s>>>(dst, value);
    return cudaGetLastError();
}

}  // namespace lora
