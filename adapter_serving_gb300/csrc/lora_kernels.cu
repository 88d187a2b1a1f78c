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

// Decode shrink: one block per (segment, K split, module); a split covers the whole K for low
// ranks and is cut so one block reads about 128 KiB of A otherwise.  Each warp takes one rank
// row per pass and walks the split in 2048-wide steps: every lane issues its eight 16-byte
// loads of A up front, then reads the segment's x rows straight from L2.  Partial sums of the
// splits are combined by the last block of the segment, in split order.
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
    float *const T = p.T[m];
    const int32_t *const perm = p.perm;
    float *const partials = p.partials;
    const float scale = p.scale;
    const int ks_max = p.ks_max, n = p.n;
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
        for (int qb = qlo; qb < qhi; qb += kShrinkDecRows) {
            float acc[kShrinkDecRows];
#pragma unroll
            for (int rr = 0; rr < kShrinkDecRows; ++rr) acc[rr] = 0.f;
            int row[kShrinkDecRows];
#pragma unroll
            for (int rr = 0; rr < kShrinkDecRows; ++rr) row[rr] = qb + rr < qhi ? perm[qb + rr] : -1;
            // the block's K range in 2048-wide steps: 8 loads of A per lane, then x, then FMAs
            for (int k0 = kbeg; k0 < kend; k0 += kShrinkDecKC) {
                uint4 av[kShrinkDecCh];
#pragma unroll
                for (int c = 0; c < kShrinkDecCh; ++c) {
                    const int kk = k0 + lane * 8 + 256 * c;
                    av[c] = kk < kend ? __ldg(reinterpret_cast<const uint4 *>(A + (size_t)j * d_in + kk)) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int rr = 0; rr < kShrinkDecRows; ++rr) {
                    if (row[rr] >= 0) {
                        const uint16_t *xr = x + (size_t)row[rr] * d_in;
                        uint4 xv[kShrinkDecCh];
#pragma unroll
                        for (int c = 0; c < kShrinkDecCh; ++c) {
                            const int kk = k0 + lane * 8 + 256 * c;
                            xv[c] = kk < kend ? __ldg(reinterpret_cast<const uint4 *>(xr + kk)) : make_uint4(0, 0, 0, 0);
                        }
#pragma unroll
                        for (int c = 0; c < kShrinkDecCh; ++c) acc[rr] += dot8_bf16(av[c], xv[c]);
                    }
                }
            }
#pragma unroll
            for (int rr = 0; rr < kShrinkDecRows; ++rr) {
                if (qb + rr < qhi) {
                    const float v = warp_sum(acc[rr]);
                    if (lane == 0) {
                        if (ks == 1)
                            T[(size_t)row[rr] * rpmax + j] = scale * v;
                        else
                            partials[(((size_t)m * ks_max + kc) * n + (qb + rr)) * rpmax + j] = v;
                    }
                }
            }
        }
    }
    if (ks == 1) {
        for (int idx = tid; idx < (qhi - qlo) * (rp - r); idx += kShrinkThreads)
            T[(size_t)perm[qlo + idx / (rp - r)] * rpmax + r + idx % (rp - r)] = 0.f;
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
            for (int c = 0; c < ks; ++c) v += __ldcg(partials + (((size_t)m * ks_max + c) * n + q) * rpmax + j);
        T[(size_t)perm[q] * rpmax + j] = scale * v;
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

// Expand metadata staged in shared memory by the epilogue warps: for every TMEM column of the
// tile (a row of the batch), the B factor of its adapter and the storage rank (0 = base only).
struct EpiMeta {
    uint64_t colB[kMaxWin];  // B factor base ([d_out, rp]) of the column's adapter
    int32_t colrp[kMaxWin];  // storage rank of that adapter, 0 for base-only rows
    int32_t ncols;           // columns set up
    int32_t module;          // module the columns were set up for (decode caching)
    int32_t maxrp;           // largest storage rank among them (0: base-only tile)
    int32_t pad_;
};

// Everything the epilogue reads per call, copied out of the kernel parameters once.  Parameters
// reached through a runtime module index are generic loads that the compiler must repeat after
// every store (they might alias); locals never are.
struct EpiCtx {
    const GemmParams *p;
    uint8_t *ring;       // per-thread staging of B rows: chunk i of thread t at (i * 128 + t) * 16
    float *tstage;       // t rows of the current batch of columns, [16][rpmax]
    EpiMeta *meta;
    int decode, n, nt, y_bf16, n_cta, rpmax, ring_chunks;
    int64_t total_iters;
    float *partials;
    int32_t *tile_counters;
    const int32_t *perm, *seg_start, *seg_adapter, *n_seg;
    uint32_t tmem_base;
    uint32_t delta_col;  // first TMEM column of the expand (delta) buffers (one per accumulator)
    int etid;            // 0..127 among epilogue threads
    int o;               // TMEM lane = W row within the tile
    int lane_base;       // first TMEM lane of this warp
    int lane;
};

struct ModLocal {
    const CUtensorMap *tmY;
    void *y;
    const float *T;
    const PoolEntry *table;
    int d_out;
};
__device__ __forceinline__ ModLocal mod_local(const GemmParams &p, int m) {
    const GemmModule &M = p.mod[m];
    return ModLocal{&M.tmY, M.y, M.T, M.table, M.d_out};
}

// (Re)build the per-column metadata of a tile from the segment table: every row of the tile's
// positions gets its segment's adapter.  Decode tiles of one module share it, so it is rebuilt
// only when the module changes; for grouped rows it is built per tile.
__device__ void setup_columns(EpiCtx &c, const Item &it) {
    EpiMeta &w = *c.meta;
    if (c.decode && w.module == it.m) return;
    named_bar_sync(1, 128);  // nobody still reads the old columns
    if (c.etid == 0) w.maxrp = 0;
    named_bar_sync(1, 128);
    const int n_seg = *c.n_seg;
    const int row0 = it.chunk * c.nt;
    const int qlo = c.decode ? 0 : row0;
    const int qhi = c.decode ? c.n : min(c.n, row0 + c.nt);
    const int32_t *seg_start = c.seg_start, *seg_adapter = c.seg_adapter, *perm = c.perm;
    const int decode = c.decode;
    const int s0 = decode ? 0 : seg_of(seg_start, n_seg, qlo);
    const int s1 = decode ? n_seg - 1 : seg_of(seg_start, n_seg, qhi - 1);
    const PoolEntry *table = mod_local(*c.p, it.m).table;
    // one thread per position: find its segment (binary search in [s0, s1]), then its column
    for (int q = qlo + c.etid; q < qhi; q += 128) {
        int lo = s0, hi = s1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(seg_start + mid) <= q) lo = mid; else hi = mid - 1;
        }
        const int a = __ldg(seg_adapter + lo);
        uint64_t b = 0;
        int rp = 0;
        if (a >= 0) {
            b = reinterpret_cast<uint64_t>(table[a].B);
            rp = table[a].rp;
        }
        const int col = decode ? __ldg(perm + q) : q - row0;
        if (col >= 0 && col < kMaxWin) {
            w.colB[col] = b;
            w.colrp[col] = rp;
        }
        if (rp > 0) atomicMax(&w.maxrp, rp);
    }
    if (c.etid == 0) {
        w.ncols = qhi - qlo;
        w.module = it.m;
    }
    named_bar_sync(1, 128);
}

// Expand for a tile this CTA heads: delta[o, col] = sum_j B_a[o0 + o, j] * t_col[j] for every
// column (row of the batch) of the tile, 0 for base-only rows, written into the TMEM delta
// buffer paired with the tile's accumulator.  It runs while the MMA warp works (on this tile or
// the one before); the drain adds it to the accumulator.
//
// Columns go in blocks of 16 (one 16-column TMEM store per block), each block in batches of CB
// columns.  Column i of a batch owns NCH fixed 16-byte slots of the per-thread ring, so every
// address is known without a running counter and all loads and dot products of a batch are
// independent: each thread copies its own B row pieces with cp.async (it then waits only for
// its own copies), the 128 threads copy the batch's t rows together, one wait, one barrier,
// then the batch is computed.  NCH = storage rank / 8 of the largest rank among the columns.
template <int NCH>
__device__ void expand_blocks(EpiCtx &c, const Item &it, uint32_t tcol0) {
    constexpr int CB = (NCH <= 2) ? 16 / NCH : 32 / NCH;  // columns per batch (ring: CB * NCH slots)
    constexpr int NB16 = 16 / CB;                       // batches per 16-column block
    const EpiMeta &w = *c.meta;
    const ModLocal M = mod_local(*c.p, it.m);
    const int row0 = it.chunk * c.nt;
    const int ncols = w.ncols;
    const int rpmax = c.rpmax;
    const int oo = it.w_tile * kBM + c.o;
    const bool o_ok = oo < M.d_out;
    const uint32_t ring_me = smem_u32(c.ring) + (uint32_t)c.o * 16;
    const uint32_t tst = smem_u32(c.tstage);
    const float *Tg = M.T + (size_t)row0 * rpmax;  // t rows in row order
    for (int b0 = 0; b0 < ncols; b0 += 16) {
        float d[16];
#pragma unroll
        for (int k = 0; k < NB16; ++k) {
            const int cb = b0 + k * CB;
            int rp[CB];
#pragma unroll
            for (int i = 0; i < CB; ++i) rp[i] = cb + i < ncols ? w.colrp[cb + i] : 0;
#pragma unroll
            for (int i = 0; i < CB; ++i) {
                if (rp[i] > 0) {
                    const uint16_t *src =
                        reinterpret_cast<const uint16_t *>(w.colB[cb + i]) + (size_t)(o_ok ? oo : 0) * rp[i];
#pragma unroll
                    for (int ch = 0; ch < NCH; ++ch)
                        if (ch * 8 < rp[i])
                            cp_async_16(ring_me + (uint32_t)((i * NCH + ch) * 128 * 16), src + ch * 8, o_ok ? 16u : 0u);
                }
            }
            const int nrow = min(CB, ncols - cb);
            if (nrow > 0) {
                const int tchunks = nrow * (rpmax >> 2);
                for (int idx = c.etid; idx < tchunks; idx += 128)
                    cp_async_16(tst + (uint32_t)idx * 16, Tg + (size_t)cb * rpmax + idx * 4, 16u);
            }
            cp_async_commit();
            cp_async_wait_all();
            named_bar_sync(1, 128);  // everyone's t rows have landed
#pragma unroll
            for (int i = 0; i < CB; ++i) {
                const float *t = c.tstage + i * rpmax;
                float acc = 0.f;
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch) {
                    if (ch * 8 < rp[i]) {
                        const uint4 bv = *reinterpret_cast<const uint4 *>(c.ring + ((size_t)(i * NCH + ch) * 128 + c.o) * 16);
                        const float4 ta = *reinterpret_cast<const float4 *>(t + ch * 8);
                        const float4 tb = *reinterpret_cast<const float4 *>(t + ch * 8 + 4);
                        acc = fmaf(bf16lo(bv.x), ta.x, acc);
                        acc = fmaf(bf16hi(bv.x), ta.y, acc);
                        acc = fmaf(bf16lo(bv.y), ta.z, acc);
                        acc = fmaf(bf16hi(bv.y), ta.w, acc);
                        acc = fmaf(bf16lo(bv.z), tb.x, acc);
                        acc = fmaf(bf16hi(bv.z), tb.y, acc);
                        acc = fmaf(bf16lo(bv.w), tb.z, acc);
                        acc = fmaf(bf16hi(bv.w), tb.w, acc);
                    }
                }
                d[k * CB + i] = acc;
            }
            named_bar_sync(1, 128);  // the t rows may be overwritten by the next batch
        }
        tmem_st16(tcol0 + (uint32_t)b0, d);
    }
}

__device__ void init_expand(EpiCtx &c, const Item &it, int buf) {
    setup_columns(c, it);
    const uint32_t tcol0 = c.tmem_base + ((uint32_t)c.lane_base << 16) + c.delta_col + (uint32_t)(buf * c.nt);
    switch (c.meta->maxrp) {
        case 8: expand_blocks<1>(c, it, tcol0); break;
        case 16: expand_blocks<2>(c, it, tcol0); break;
        case 32: expand_blocks<4>(c, it, tcol0); break;
        case 64: expand_blocks<8>(c, it, tcol0); break;
        default: {  // base-only tile
            float z[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) z[i] = 0.f;
            for (int b0 = 0; b0 < c.meta->ncols; b0 += 16) tmem_st16(tcol0 + (uint32_t)b0, z);
        }
    }
    tmem_st_wait();
}


// This CTA's share of 16 columns of a tile: accumulator (+ the expand delta when it heads the
// tile), both TMEM loads in flight before the one wait.
__device__ __forceinline__ void own_cols16(const EpiCtx &c, uint32_t tacc, uint32_t tdel, bool head, int c0,
                                           float (&v)[16]) {
    uint32_t r[16], d[16];
    tmem_ld16(tacc + c0, r);
    if (head) tmem_ld16(tdel + c0, d);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]) + (head ? __uint_as_float(d[i]) : 0.f);
}


// Partial tiles (stream-K pieces) are kept in column quads: element (column c, lane o) at
// ((c / 4) * 128 + o) * 4 + c % 4.  A thread's 16 columns are four 16-byte vectors and a warp
// stores or loads 512 contiguous bytes per instruction.
__device__ __forceinline__ float4 *piece_quads(float *piece, int c0, int o) {
    return reinterpret_cast<float4 *>(piece) + (size_t)(c0 >> 2) * kBM + o;
}

// Drain: accumulator (+ expand delta when this CTA heads the tile) -> y.  y goes out through
// shared memory and TMA tensor stores of [16 columns][128 lanes] blocks: the blocks of a round
// are staged together (the round is as many blocks as the staging buffer holds), then one
// barrier and the round's stores back to back.
//
// A tile split over several CTAs (stream-K) is finished by one CTA that adds the pieces in k
// order, so the sum never depends on timing.  The piece holding k-block 0 is always the last
// item of its CTA and the other pieces are the first items of theirs, so that CTA waits
// (bounded) for the others and then finishes the tile without writing its own piece; if the
// wait runs out it falls back to "write your piece, last to arrive finishes".  Pieces go to
// global memory with plain vector stores; the finishing CTA pulls the other pieces into its idle
// stage buffers with bulk copies when it can, else reads them with vector loads.
struct DrainBufs {
    uint8_t *ybuf;       // y staging (the expand ring, idle during a drain)
    uint32_t ybuf_bytes;
    uint8_t *stage;      // the stage buffers, free once the CTA's last item has been multiplied
    uint32_t stage_bytes;
    uint64_t *ld_bar;    // completion of the bulk copies of other pieces
    uint32_t ld_phase;   // phases of ld_bar completed so far
};

constexpr uint64_t kHeadWaitNs = 50000;  // how long a finishing CTA waits for the other pieces

__device__ void drain(EpiCtx &c, const Item &it, int buf, bool last, volatile int *misc_flag,
                      volatile int *abort_flag, DrainBufs &db) {
    const ModLocal M = mod_local(*c.p, it.m);
    const int nt = c.nt, decode = c.decode, y_bf16 = c.y_bf16, n_cta = c.n_cta;
    const int64_t total_iters = c.total_iters;
    float *const partials = c.partials;
    const int row0 = it.chunk * nt;
    const int ncols = decode ? c.n : min(nt, c.n - row0);
    const int ncols16 = (ncols + 15) & ~15;
    const int o0 = it.w_tile * kBM;
    const bool head = it.kb0 == 0;
    const uint32_t lane_off = (uint32_t)c.lane_base << 16;
    const uint32_t tacc = c.tmem_base + lane_off + (uint32_t)(buf * nt);
    const uint32_t tdel = c.tmem_base + lane_off + c.delta_col + (uint32_t)(buf * nt);
    const size_t slot_elems = (size_t)kBM * nt;
    const bool leader = c.etid == 0;
    const uint32_t esz = y_bf16 ? 2u : 4u;
    const uint32_t piece_bytes = (uint32_t)ncols16 * kBM * 4;

    // y staging for a block of 16 columns at `dst` ([column][lane], fp32 or bf16)
    auto put16 = [&](uint8_t *dst, const float (&v)[16]) {
        if (!y_bf16) {
            float *f = reinterpret_cast<float *>(dst);
#pragma unroll
            for (int i = 0; i < 16; ++i) f[i * kBM + c.o] = v[i];
        } else {
            uint16_t *h = reinterpret_cast<uint16_t *>(dst);
#pragma unroll
            for (int i = 0; i < 16; ++i) h[i * kBM + c.o] = __bfloat16_as_ushort(__float2bfloat16_rn(v[i]));
        }
    };
    // block c0 of y: into its slot of the current round; the round's stores go out when it is full
    const uint32_t block_bytes = 16u * kBM * esz;
    const int round_blocks = (int)(db.ybuf_bytes / block_bytes);
    auto emit = [&](int c0, const float (&v)[16]) {
        const int slot = (c0 >> 4) % round_blocks;
        if (slot == 0) {  // the previous round's stores must have read the buffer
            if (leader) bulk_wait_read<0>();
            named_bar_sync(1, 128);
        }
        put16(db.ybuf + (size_t)slot * block_bytes, v);
        if (slot == round_blocks - 1 || c0 + 16 >= ncols16) {
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (leader) {
                for (int k = 0; k <= slot; ++k)
                    tma_store_2d(M.tmY, db.ybuf + (size_t)k * block_bytes, o0, row0 + c0 - 16 * (slot - k));
                bulk_commit();
            }
        }
    };

    if (head && it.kb1 == it.kbn) {
        for (int c0 = 0; c0 < ncols16; c0 += 16) {
            float v[16];
            own_cols16(c, tacc, tdel, true, c0, v);
            emit(c0, v);
        }
        return;
    }

    // ---- partial tile (stream-K) ----
    const int c_first = (int)(((it.it0 + 1) * n_cta - 1) / total_iters);  // CTA holding iteration it0
    const int c_last = (int)(((it.it0 + it.kbn) * n_cta - 1) / total_iters);
    const int nc = c_last - c_first + 1;
    const int self_idx = (int)blockIdx.x - c_first;
    int32_t *counter = c.tile_counters + it.tile;
    auto part_of = [&](int cta) -> float * {  // the piece of CTA `cta`
        const int64_t b_c = (int64_t)cta * total_iters / n_cta;
        return partials + ((size_t)cta * 2 + ((b_c >= it.it0) ? 0 : 1)) * slot_elems;
    };
    bool finalize = false;
    if (head) {
        if (leader) {
            const uint64_t t0 = globaltimer();
            int seen = ld_acquire_gpu(counter);
            while (seen != nc - 1 && globaltimer() - t0 < kHeadWaitNs) seen = ld_acquire_gpu(counter);
            *misc_flag = (seen == nc - 1);
        }
        named_bar_sync(1, 128);
        finalize = *misc_flag != 0;
        named_bar_sync(1, 128);
    }
    if (!finalize) {
        float *dst = part_of(blockIdx.x);
        for (int c0 = 0; c0 < ncols16; c0 += 16) {
            float v[16];
            own_cols16(c, tacc, tdel, head, c0, v);
            float4 *q = piece_quads(dst, c0, c.o);
#pragma unroll
            for (int k = 0; k < 4; ++k) __stcg(q + k * kBM, make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]));
        }
        __threadfence();  // this thread's share of the piece is visible device-wide
        named_bar_sync(1, 128);
        if (leader) *misc_flag = (atomicAdd(counter, 1) == nc - 1);
        named_bar_sync(1, 128);
        finalize = *misc_flag != 0;
        named_bar_sync(1, 128);
        if (!finalize) return;
    }
    __threadfence();

    // finish: the other pieces, staged in shared memory when the stage buffers are idle
    const uint32_t others_bytes = (uint32_t)(nc - 1) * piece_bytes;
    const bool staged = last && (uint64_t)others_bytes <= db.stage_bytes;
    if (staged) {
        fence_proxy_async_global();  // the pieces were written through the generic proxy
        if (leader) {
            mbar_arrive_expect_tx(db.ld_bar, others_bytes);
            for (int k = 0, j = 0; k < nc; ++k)
                if (k != self_idx) bulk_load(db.stage + (size_t)(j++) * piece_bytes, part_of(c_first + k), piece_bytes, db.ld_bar);
        }
        // bounded wait; a timeout has already raised the abort flag
        mbar_wait(db.ld_bar, db.ld_phase & 1, abort_flag, nullptr);
        ++db.ld_phase;
    }
    const uint32_t pbase = smem_u32(db.stage) + (uint32_t)c.o * 16;  // this lane's quad of piece 0, block 0
    for (int c0 = 0; c0 < ncols16; c0 += 16) {
        float own[16], sum[16];
        own_cols16(c, tacc, tdel, head, c0, own);
        for (int jc = 0, j = 0; jc < nc; ++jc) {
            float4 q[4];
            if (jc == self_idx) {
#pragma unroll
                for (int k = 0; k < 4; ++k) q[k] = make_float4(own[4 * k], own[4 * k + 1], own[4 * k + 2], own[4 * k + 3]);
            } else if (staged) {
                const uint32_t a = pbase + (uint32_t)(j++) * piece_bytes + (uint32_t)(c0 >> 2) * kBM * 16;
#pragma unroll
                for (int k = 0; k < 4; ++k) q[k] = lds128(a + (uint32_t)k * kBM * 16);
            } else {
                const float4 *src = piece_quads(part_of(c_first + jc), c0, c.o);
#pragma unroll
                for (int k = 0; k < 4; ++k) q[k] = __ldcg(src + k * kBM);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float a[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) sum[4 * k + e] = jc == 0 ? a[e] : sum[4 * k + e] + a[e];
            }
        }
        emit(c0, sum);
    }
    if (leader) *counter = 0;
}

__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.n_stages;
    const int NB = p.n_acc;
    const uint32_t a_bytes = kBM * kBK * 2;
    const uint32_t b_bytes = (uint32_t)p.nt * kBK * 2;
    const uint32_t stage_bytes = a_bytes + b_bytes;
    uint8_t *ring = smem + (size_t)S * stage_bytes;  // per-thread B staging, ring_chunks * 2 KiB
    float *tstage = reinterpret_cast<float *>(ring + (size_t)p.ring_chunks * 128 * 16);  // [16][rpmax]
    EpiMeta *meta = reinterpret_cast<EpiMeta *>(tstage + 16 * p.rpmax);
    uint64_t *full = reinterpret_cast<uint64_t *>(meta + 1);
    uint64_t *empty = full + S;
    uint64_t *acc_full = empty + S;
    uint64_t *acc_free = acc_full + 2;
    uint64_t *mma_done = acc_free + 2;
    uint64_t *ld_bar = mma_done + 1;  // drain: bulk copies of other pieces
    uint32_t *misc = reinterpret_cast<uint32_t *>(ld_bar + 2);  // [0] tmem, [1] abort, [2] flag

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
        mbar_init(ld_bar, 1);
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
        c.tstage = tstage;
        c.meta = meta;
        c.tmem_base = tmem_base;
        c.delta_col = (uint32_t)(NB * p.nt);
        c.etid = threadIdx.x - 64;
        c.lane = lane;
        c.lane_base = (warp & 3) * 32;
        c.o = c.lane_base + lane;
        c.decode = p.decode;
        c.n = p.n;
        c.nt = p.nt;
        c.y_bf16 = p.y_bf16;
        c.n_cta = p.n_cta;
        c.rpmax = p.rpmax;
        c.ring_chunks = p.ring_chunks;
        c.total_iters = p.total_iters;
        c.partials = p.partials;
        c.tile_counters = p.tile_counters;
        c.perm = p.perm;
        c.seg_start = p.seg_start;
        c.seg_adapter = p.seg_adapter;
        c.n_seg = p.n_seg;
        volatile int *flag = reinterpret_cast<volatile int *>(misc + 2);
        DrainBufs db;
        db.ybuf = ring;
        db.ybuf_bytes = (uint32_t)p.ring_chunks * 128 * 16;
        db.stage = smem;
        db.stage_bytes = (uint32_t)S * stage_bytes;
        db.ld_bar = ld_bar;
        db.ld_phase = 0;
        // The expand of a tile this CTA heads is prepared one item ahead when there are two
        // accumulator/delta buffer pairs, so it overlaps the MMAs of the item before it.
        Sched sc;
        sc.begin(p, blockIdx.x);
        Item cur, nxt;
        bool has_cur = sc.next(p, cur);
        uint32_t li = 0;
        if (has_cur && cur.kb0 == 0) init_expand(c, cur, 0);
        while (has_cur) {
            const int buf = li % NB;
            const bool has_nxt = sc.next(p, nxt);
            if (has_nxt && NB == 2 && nxt.kb0 == 0) init_expand(c, nxt, (li + 1) % 2);
            const bool full_ok = mbar_wait(acc_full + buf, (li / NB) & 1, abort_flag, p.err);
            if (named_bar_or(1, 128, !full_ok)) break;
            tc_fence_after();
            drain(c, cur, buf, !has_nxt, flag, abort_flag, db);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free + buf);
            // the staging buffers live in the ring, which the next expand reuses
            if (c.etid == 0) bulk_wait_read<0>();
            named_bar_sync(1, 128);
            if (has_nxt && NB == 1 && nxt.kb0 == 0) init_expand(c, nxt, 0);
            cur = nxt;
            has_cur = has_nxt;
            ++li;
        }
        if (c.etid == 0) bulk_wait<0>();  // every output store has been performed
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

size_t gemm_smem_bytes(int nt, int n_stages, int ring_chunks, int rpmax) {
    const size_t stage = (size_t)kBM * kBK * 2 + (size_t)nt * kBK * 2;
    return 1024 + stage * n_stages + (size_t)ring_chunks * 128 * 16 + (size_t)16 * rpmax * 4 + sizeof(EpiMeta) +
           8 * (2 * (size_t)n_stages + 7) + 16;
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
