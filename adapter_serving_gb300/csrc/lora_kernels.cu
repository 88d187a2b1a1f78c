// lora_kernels.cu -- the grouped-rows (prefill) side of the adapted linear layer
// y_i = W x_i + s B_a (A_a x_i), and the CUDA-core shrinks:
//
//   prep_segments_kernel  checks a given contiguous segment table (prefill), expand slots per
//                         row chunk
//   shrink_kernel         t_i = s * A_a x_i for every row of a segment table (grouped rows)
//   shrink_decode_kernel  the same for a decode batch with int8 factors (bf16 factors take the
//                         shrink on the tensor cores, decode_kernels.cu)
//   gemm_kernel           grouped rows: base W x_i on tcgen05 tensor cores into TMEM; the expand
//                         s B_a t_i from B stages in the same TMA ring, written into the tile's
//                         accumulator before its MMAs start
//
// The forward is the one on "m07 -- Multi-Adapter (LoRA) Serving", section 6 "Deep Dive A:
// Batching Heterogeneous Adapters" (one batched base GEMM shared by the batch, plus a gathered
// per-row adapter product; prefill rows arrive as contiguous per-request segments) and "LoRA,
// quotas and noisy neighbours", section "One weight read, many adapters" (rows tagged with their
// adapter, grouped, one kernel per layer).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>
#include <type_traits>
#include <utility>

#include "lora_internal.h"
#include "ptx.cuh"
#include "prep_common.cuh"

namespace lora {

__device__ int checked_id(const PrepParams &p, int id, int where) {
    if (id < -1 || id >= p.max_adapters) {
        report(p.err, LORA_DEVERR_BAD_ADAPTER, where);
        return -1;
    }
    if (id >= 0) {
        int rank[LORA_MAX_MODULES];  // all loads in flight before the first test
#pragma unroll
        for (int m = 0; m < LORA_MAX_MODULES; ++m) rank[m] = m < p.n_mod ? p.table[m][id].rank : 1;
        bool ok = true;
#pragma unroll
        for (int m = 0; m < LORA_MAX_MODULES; ++m) ok = ok && rank[m] > 0;
        if (!ok) {
            report(p.err, LORA_DEVERR_NOT_LOADED, where);
            return -1;
        }
    }
    return id;
}

// Grouped rows (prefill): validate the table, copy it into the workspace with unusable
// adapters replaced by -1 (base only).  A malformed table becomes one base-only segment.
__global__ void __launch_bounds__(1024) prep_segments_kernel(const PrepParams p) {
    grid_dep_wait();
    grid_dep_launch();
    const bool ok = segments_valid_block(p);
    if (!ok) {
        if (threadIdx.x == 0) {
            report(p.err, LORA_DEVERR_BAD_SEGMENTS, 0);
            p.seg_start[0] = 0;
            p.seg_start[1] = p.n;
            p.seg_adapter[0] = -1;
            *p.n_seg = 1;
        }
        if (p.chunk_nb != nullptr)
            for (int c = threadIdx.x; c < (p.n + p.nt - 1) / p.nt; c += blockDim.x) {
                p.chunk_seg0[c] = 0;
                p.chunk_nb[c] = 0;
            }
        return;
    }
    for (int s = threadIdx.x; s <= p.n_seg_in; s += blockDim.x) {
        p.seg_start[s] = p.seg_start_in[s];
        if (s < p.n_seg_in) p.seg_adapter[s] = checked_id(p, p.seg_adapter_in[s], s);
    }
    if (threadIdx.x == 0) *p.n_seg = p.n_seg_in;
    if (p.chunk_nb == nullptr) return;
    // expand slots of every row chunk: each segment's rows in the chunk, in runs of pf_ch
    __syncthreads();
    const int ns = p.n_seg_in, nt = p.nt, chunks = (p.n + nt - 1) / nt;
    for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
        const int row0 = c * nt, row1 = min(p.n, row0 + nt);
        int sg = seg_of(p.seg_start, ns, row0);
        p.chunk_seg0[c] = sg;
        int nb = 0;
        for (; sg < ns && p.seg_start[sg] < row1; ++sg) {
            if (p.seg_adapter[sg] < 0) continue;
            const int rows = min(p.seg_start[sg + 1], row1) - max(p.seg_start[sg], row0);
            nb += (rows + p.pf_ch - 1) / p.pf_ch;
        }
        p.chunk_nb[c] = nb;
    }
}

__global__ void table_write_kernel(PoolEntry *dst, PoolEntry v) { *dst = v; }
__global__ void table_write_many_kernel(const __grid_constant__ TableWrites w) {
    if ((int)threadIdx.x < w.n) *w.dst[threadIdx.x] = w.v[threadIdx.x];
}

// Block (item, part): a share of the item's A rows and B rows.  A ([rp, d_in] bf16, d_in a
// multiple of 8) moves in 16-byte chunks, the rows past the rank zeroed.  B ([d_out, rp]) moves in
// 16-byte chunks too when the rank is the storage rank (its rows are then contiguous in both
// places), else element by element with the columns past the rank zeroed.  Block (item, 0)
// publishes the entry; later kernels on the stream see it only after the whole grid has finished.
__global__ void __launch_bounds__(256) packed_load_kernel(const __grid_constant__ PackedJobs jobs) {
    const PackedJob &J = jobs.j[blockIdx.x];
    const int rank = J.val.rank, rp = J.val.rp, d_in = J.d_in, d_out = J.d_out;
    const int stride = gridDim.y * blockDim.x, t0 = blockIdx.y * blockDim.x + threadIdx.x;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const int cpr = d_in / 8;  // 16-byte chunks per A row
    const int a_live = rank * cpr, a_all = rp * cpr;
    uint4 *dA = reinterpret_cast<uint4 *>(const_cast<uint16_t *>(J.val.A));
    const uint4 *sA = reinterpret_cast<const uint4 *>(J.srcA);
    for (int c = t0; c < a_all; c += stride) dA[c] = c < a_live ? sA[c] : zero;
    uint16_t *dB = const_cast<uint16_t *>(J.val.B);
    const bool b_vec = rank == rp && (reinterpret_cast<uintptr_t>(J.srcB) & 15) == 0;
    if (b_vec) {
        const int b_chunks = d_out * rp / 8;
        uint4 *d4 = reinterpret_cast<uint4 *>(dB);
        const uint4 *s4 = reinterpret_cast<const uint4 *>(J.srcB);
        for (int c = t0; c < b_chunks; c += stride) d4[c] = s4[c];
    } else {
        const uint16_t *sB = reinterpret_cast<const uint16_t *>(J.srcB);
        const int b_elems = d_out * rp;
        for (int e = t0; e < b_elems; e += stride) {
            const int r = e / rp, c = e - r * rp;
            dB[e] = c < rank ? sB[r * rank + c] : (uint16_t)0;
        }
    }
    if (blockIdx.y == 0 && threadIdx.x == 0) *J.dst = J.val;
}

// ========================================================================== shrink ==========
//
// t_q[j] = s * sum_k A_a[j, k] x_row(q)[k] for every position q, j < rp (zero for j >= rank).
// With several K splits the partial sums go to the workspace and the last block to finish
// (atomic counter) adds them in split order, so the result does not depend on block timing.

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

// 8 int8 codes of A (a.x bytes 0..3, a.y bytes 0..3) against 8 bf16 values of x
__device__ __forceinline__ float dot8_i8_bf16(uint2 a, uint4 b) {
    const float4 lo = i8x4(a.x), hi = i8x4(a.y);
    float r = lo.x * bf16lo(b.x);
    r = fmaf(lo.y, bf16hi(b.x), r);
    r = fmaf(lo.z, bf16lo(b.y), r);
    r = fmaf(lo.w, bf16hi(b.y), r);
    r = fmaf(hi.x, bf16lo(b.z), r);
    r = fmaf(hi.y, bf16hi(b.z), r);
    r = fmaf(hi.z, bf16lo(b.w), r);
    r = fmaf(hi.w, bf16hi(b.w), r);
    return r;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Grouped rows: one block per 64 rows and K split; rows staged in shared memory, each warp takes
// eight rank rows.
__global__ void __launch_bounds__(kShrinkThreads) shrink_kernel(const __grid_constant__ ShrinkParams p) {
    __shared__ __align__(16) uint16_t xs[kShrinkRows * kShrinkKSub];
    grid_dep_wait();
    grid_dep_launch();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int m = 0;
    while (m + 1 < p.n_mod && p.split_begin[m + 1] <= (int)blockIdx.y) ++m;
    const int kc = blockIdx.y - p.split_begin[m];
    if (kc >= p.ksplit[m]) return;
    const int n_seg = *p.n_seg;
    const int u = blockIdx.x;
    const int qlo = u * kShrinkGroupRows;
    if (qlo >= p.n) return;
    const int qhi = min(p.n, qlo + kShrinkGroupRows);
    int s = seg_of(p.seg_start, n_seg, qlo);
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
                        const int row = qb + rr;
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
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = warp + 8 * jj;
                if (j < rp) {
#pragma unroll
                    for (int rr = 0; rr < kShrinkRows; ++rr) {
                        if (rr < nr) {
                            float v = (j < r) ? warp_sum(acc[jj][rr]) : 0.f;
                            if (lane == 0) T[(size_t)(qb + rr) * rpmax + j] = p.scale * v;
                        }
                    }
                }
            }
        }
        q = qe;
    }
}

// Decode shrink for int8 factors: one block per (sorted position, K split, module); each warp takes
// one rank row per pass and walks the split in 2048-wide steps: every lane issues its eight
// 8-byte loads of A codes up front, then reads the row's x from L2.  Partial sums of the splits are
// combined by the last block of the position, in split order.  t_j is scaled by s and by the rank
// row's fold scale (A scale x B scale) and written to row perm[q] of T.
__device__ __forceinline__ void shrink_decode_body(const ShrinkParams &p, int &s_last) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int m = 0;
    while (m + 1 < p.n_mod && p.split_begin[m + 1] <= (int)blockIdx.y) ++m;
    const int kc = blockIdx.y - p.split_begin[m];
    if (kc >= p.ksplit[m]) return;
    const int u = blockIdx.x;
    if (u >= p.n) return;
    const int a = p.qadapter[u];
    const int d_in = p.d_in[m];
    if (a < 0) return;  // base-only position: no t row (every split of it returns here)
    const PoolEntry *e = p.table[m] + a;
    const int rp_u = e->rp;
    // The split width was chosen for the largest storage rank in the pool; a lower-rank adapter
    // takes proportionally wider splits, so fewer of them (blocks past its count leave at once).
    int kcw = p.kc[m];
    for (int r2 = rp_u; r2 < p.rpmax && kcw < d_in; r2 <<= 1) kcw <<= 1;
    const int ks = (d_in + kcw - 1) / kcw;
    if (kc >= ks) return;
    const int kbeg = kc * kcw;
    const int kend = min(d_in, kbeg + kcw);
    const uint16_t *x = p.x[m];
    float *const trow = p.T[m] + (size_t)p.perm[u] * p.rpmax;
    float *const partials = p.partials;
    const int ks_max = p.ks_max, n = p.n, rpmax = p.rpmax;
    const int r = e->rank, rp = e->rp;
    const uint8_t *A = reinterpret_cast<const uint8_t *>(e->A);
    const float *fold = p.fold[m] + e->row_off;
    const float scale = p.scale;
    const uint16_t *xr = x + (size_t)p.perm[u] * d_in;
    for (int j0 = 0; j0 < r; j0 += kShrinkThreads / 32) {
        const int j = j0 + warp;
        if (j >= r) break;  // warp-uniform
        float acc = 0.f;
        for (int k0 = kbeg; k0 < kend; k0 += kShrinkDecKC) {
            uint2 av[kShrinkDecCh];
#pragma unroll
            for (int c = 0; c < kShrinkDecCh; ++c) {
                const int kk = k0 + lane * 8 + 256 * c;
                av[c] = kk < kend ? __ldg(reinterpret_cast<const uint2 *>(A + (size_t)j * d_in + kk)) : make_uint2(0, 0);
            }
            uint4 xv[kShrinkDecCh];
#pragma unroll
            for (int c = 0; c < kShrinkDecCh; ++c) {
                const int kk = k0 + lane * 8 + 256 * c;
                xv[c] = kk < kend ? __ldg(reinterpret_cast<const uint4 *>(xr + kk)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int c = 0; c < kShrinkDecCh; ++c) acc += dot8_i8_bf16(av[c], xv[c]);
        }
        const float v = warp_sum(acc);
        if (lane == 0) {
            if (ks == 1) trow[j] = scale * fold[j] * v;
            else partials[(((size_t)m * ks_max + kc) * n + u) * rpmax + j] = v;
        }
    }
    if (ks == 1) {
        for (int j = r + tid; j < rp; j += kShrinkThreads) trow[j] = 0.f;
        return;
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(p.counters + m * p.max_units + u, 1) == ks - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    for (int j = tid; j < rp; j += kShrinkThreads) {
        float v = 0.f;
        if (j < r)
            for (int c = 0; c < ks; ++c) v += __ldcg(partials + (((size_t)m * ks_max + c) * n + u) * rpmax + j);
        trow[j] = j < r ? scale * fold[j] * v : 0.f;
    }
    if (tid == 0) p.counters[m * p.max_units + u] = 0;
}

// Launched right after the gemm (on the gemm's trigger, which follows the gemm's own wait for the
// row plan), so it reads the plan, the pool and x without waiting, and runs on the resources the
// persistent gemm leaves free while the gemm streams W.  It never reads the gemm's results.  Block
// (0, 0) waits for the gemm before it exits: the grid then completes only after the gemm has, and
// the finalize's one wait covers both.
__global__ void __launch_bounds__(kShrinkThreads, 3) shrink_decode_kernel(const __grid_constant__ ShrinkParams p) {
    __shared__ int s_last;
    grid_dep_launch();
    shrink_decode_body(p, s_last);
    if (blockIdx.x == 0 && blockIdx.y == 0) grid_dep_wait();
}

// ============================================================================ gemm ==========
//
// Grouped rows.  One persistent CTA per SM, four roles: warp 0 is the TMA producer, lane 0 of
// warp 1 issues tcgen05.mma, warps 2-5 are the epilogue (TMEM lane quarter = warp % 4).  A tile
// is 128 rows of W (MMA M) by a 256-row chunk of the batch (MMA N); CTAs take whole tiles round
// robin in a grouped raster.  A tile's expand slots (one B stage each) enter the ring a few
// k-blocks into the previous tile; the epilogue copies each out of the ring, computes the slot's
// dot products and writes them into the tile's accumulator, which the MMAs then accumulate on.

struct Item {
    int32_t m, w_tile, chunk, kbn, nbs, tile;
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

// the j-th tile of CTA `cta`, its expand slots from the per-chunk table
__device__ bool rr_item(const GemmParams &p, int cta, int j, Item &it) {
    const int t = cta + j * p.n_cta;
    if (t >= p.total_tiles) return false;
    int m = 0;
    while (m + 1 < p.n_mod && p.mod[m + 1].tile_begin <= t) ++m;
    it.m = m;
    it.kbn = p.mod[m].k_blocks;
    it.tile = t;
    tile_coords(p, m, t - p.mod[m].tile_begin, it);
    it.nbs = p.chunk_nb ? p.chunk_nb[it.chunk] : 0;
    return true;
}

// tile j+1's B stages enter the ring after the first kGroupedLead k-blocks of tile j
constexpr int kGroupedLead = 4;

struct EpiCtx {
    const GemmParams *p;
    int n, nt, y_bf16;
    int etid;            // 0..127 among epilogue threads
    int o;               // TMEM lane = W row within the tile
    int lane_base;       // first TMEM lane of this warp
};

// Epilogue side of a B stage: delta[o, col] = sum_j B_a[o0 + o, j] t_col[j] for every row of every
// slot, written to the column of the tile's accumulator (32x32b.x1: this warp's 32 lanes).
__device__ __forceinline__ float dot8_bf16_f32(uint4 b, float4 ta, float4 tb) {
    float acc0 = bf16lo(b.x) * ta.x, acc1 = bf16hi(b.x) * ta.y;
    acc0 = fmaf(bf16lo(b.y), ta.z, acc0);
    acc1 = fmaf(bf16hi(b.y), ta.w, acc1);
    acc0 = fmaf(bf16lo(b.z), tb.x, acc0);
    acc1 = fmaf(bf16hi(b.z), tb.y, acc1);
    acc0 = fmaf(bf16lo(b.w), tb.z, acc0);
    acc1 = fmaf(bf16hi(b.w), tb.w, acc1);
    return acc0 + acc1;
}

// One slot: this lane's row of the slot's B (NCH 16-byte chunks, storage rank 8 NCH) is loaded
// once, then every row of the slot streams its t row against it.
template <int NCH>
__device__ __forceinline__ void expand_slot(const EpiCtx &c, uint32_t brow, uint32_t tslot, int tstride, int nrows,
                                            int q0, uint32_t tacc, int row0) {
    // lane o starts at chunk rot = o / (8 / NCH): the eight lanes of a quarter warp then hit eight
    // different 16-byte bank groups of their rows (rows are NCH * 16 bytes apart)
    const int rot = (c.o * NCH / 8) & (NCH - 1);
    uint4 b[NCH];
    const uint32_t mine = brow + (uint32_t)(c.o * NCH) * 16u;
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) b[ch] = lds_u128(mine + (uint32_t)((ch + rot) & (NCH - 1)) * 16u);
    for (int r = 0; r < nrows; ++r) {
        const uint32_t trow = tslot + (uint32_t)(r * tstride * 4);
        float acc[NCH];
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
            const uint32_t tc = trow + ((ch + rot) & (NCH - 1)) * 32;
            acc[ch] = dot8_bf16_f32(b[ch], lds128(tc), lds128(tc + 16));
        }
#pragma unroll
        for (int w = 1; w < NCH; w <<= 1)
#pragma unroll
            for (int ch = 0; ch + w < NCH; ch += 2 * w) acc[ch] += acc[ch + w];  // fixed pairwise order
        const int col = q0 + r - row0;  // the same for the whole warp: the guard is uniform
        if (q0 + r >= c.n || col < 0 || col >= c.nt) continue;
        tmem_st1(tacc + (uint32_t)col, acc[0]);
    }
}

__device__ void expand_stage(const EpiCtx &c, const uint8_t *sa, const uint8_t *sx, uint32_t tacc, int row0) {
    const BStageHdr *hdr = reinterpret_cast<const BStageHdr *>(sx);
    const int nslots = min(hdr->nslots, kPackSlots);
    const uint32_t a_base = smem_u32(sa), t_base = smem_u32(sx) + kStageHdrBytes;
    for (int e = 0; e < nslots; ++e) {
        const BSlotS sl = hdr->slot[e];
        const uint32_t brow = a_base + (uint32_t)sl.off * kBM * 2u;
        const uint32_t tslot = t_base + (uint32_t)sl.toff * 4;
        switch (sl.rp) {
            case 8: expand_slot<1>(c, brow, tslot, sl.tstride, sl.nrows, sl.q0, tacc, row0); break;
            case 16: expand_slot<2>(c, brow, tslot, sl.tstride, sl.nrows, sl.q0, tacc, row0); break;
            case 32: expand_slot<4>(c, brow, tslot, sl.tstride, sl.nrows, sl.q0, tacc, row0); break;
            case 64: expand_slot<8>(c, brow, tslot, sl.tstride, sl.nrows, sl.q0, tacc, row0); break;
            default: break;
        }
    }
}

// Drain: accumulator -> y through shared memory and TMA tensor stores of [16 columns][128 lanes]
// blocks: the blocks of a round are staged together (the round is as many blocks as the staging
// buffer holds), then one barrier and the round's stores back to back.
__device__ void drain(EpiCtx &c, const Item &it, int buf, uint32_t tmem_base, uint8_t *ys, uint32_t ys_bytes) {
    const GemmModule &M = c.p->mod[it.m];
    const int nt = c.nt, y_bf16 = c.y_bf16;
    const int row0 = it.chunk * nt;
    const int ncols = min(nt, c.n - row0);
    const int ncols16 = (ncols + 15) & ~15;
    const int o0 = it.w_tile * kBM;
    const uint32_t tacc = tmem_base + ((uint32_t)c.lane_base << 16) + (uint32_t)(buf * nt);
    const bool leader = c.etid == 0;
    const uint32_t esz = y_bf16 ? 2u : 4u;
    const uint32_t block_bytes = 16u * kBM * esz;
    const int round_blocks = (int)(ys_bytes / block_bytes);
    const CUtensorMap *tmY = &M.tmY;
    for (int c0 = 0; c0 < ncols16; c0 += 16) {
        uint32_t r[16];
        tmem_ld16(tacc + (uint32_t)c0, r);
        tmem_ld_wait();
        const int slot = (c0 >> 4) % round_blocks;
        if (slot == 0) {  // the previous round's stores must have read the buffer
            if (leader) bulk_wait_read<0>();
            named_bar_sync(1, 128);
        }
        uint8_t *dst = ys + (size_t)slot * block_bytes;
        if (!y_bf16) {
            float *f = reinterpret_cast<float *>(dst);
#pragma unroll
            for (int i = 0; i < 16; ++i) f[i * kBM + c.o] = __uint_as_float(r[i]);
        } else {
            uint16_t *h = reinterpret_cast<uint16_t *>(dst);
#pragma unroll
            for (int i = 0; i < 16; ++i) h[i * kBM + c.o] = __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(r[i])));
        }
        if (slot == round_blocks - 1 || c0 + 16 >= ncols16) {
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (leader) {
                for (int k = 0; k <= slot; ++k)
                    tma_store_2d(tmY, ys + (size_t)k * block_bytes, o0, row0 + c0 - 16 * (slot - k));
                bulk_commit();
            }
        }
    }
}

__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.n_stages;
    // Ring slot and round of fill k without an integer division in the loops:
    // k / S = umulhi(k, ceil(2^32 / S)), exact for k < 2^32 / 8 when S <= 8.
    const uint32_t ring_m = 0xFFFFFFFFu / (uint32_t)S + 1u;
    auto rround = [ring_m](uint32_t kk) -> uint32_t { return __umulhi(kk, ring_m); };
    auto rslot = [ring_m, S](uint32_t kk) -> uint32_t { return kk - __umulhi(kk, ring_m) * (uint32_t)S; };
    const uint32_t a_bytes = kBM * kBK * 2;
    const uint32_t b_bytes = (uint32_t)p.nt * kBK * 2;
    const uint32_t stage_bytes = a_bytes + b_bytes;
    const uint64_t wait_ns = p.wait_ns;
    uint8_t *ybuf = smem + (size_t)S * stage_bytes;  // epilogue y staging
    // A stage slot is filled with either W k-blocks (wfull, consumed by the MMA warp) or a B stage
    // (bfull, consumed by the epilogue).  Each consumer skips the other kind, so each kind has its
    // own barrier and every consumer keeps its own per-slot parity: a parity wait is only sound
    // when the waiter cannot fall two phases behind, which holds per kind but not across kinds.
    uint64_t *wfull = reinterpret_cast<uint64_t *>(ybuf + p.ybuf_bytes);
    uint64_t *bfull = wfull + S;
    uint64_t *empty = bfull + S;
    uint64_t *acc_full = empty + S;
    uint64_t *acc_free = acc_full + 2;
    uint64_t *mma_done = acc_free + 2;
    uint32_t *misc = reinterpret_cast<uint32_t *>(mma_done + 1);  // [0] tmem, [1] abort

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(wfull + s, 1);
            mbar_init(bfull + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_free + b, kEpiWarps);
        }
        mbar_init(mma_done, 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int m = 0; m < p.n_mod; ++m) {
            tma_prefetch_desc(&p.mod[m].tmW);
            tma_prefetch_desc(&p.mod[m].tmX);
        }
    }
    if (warp == 1) tmem_alloc(misc, (uint32_t)p.tmem_cols);
    grid_dep_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = misc[0];
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer (warp)
        const uint64_t pol_w = l2_policy_evict_normal();
        const uint64_t pol_x = l2_policy_evict_last();
        uint32_t k = 0;  // stage fills issued
        bool ok = true;
        // per slot (bit s): parity of the next W / B fill, kind and parity of the latest fill
        uint32_t wpar = 0, bpar = 0, last_b = 0, last_par = 0, filled = 0;
        auto note_fill = [&](int s, bool is_b) -> uint32_t {
            const uint32_t bit = 1u << s;
            const uint32_t par = ((is_b ? bpar : wpar) >> s) & 1u;
            if (is_b) bpar ^= bit; else wpar ^= bit;
            last_b = is_b ? (last_b | bit) : (last_b & ~bit);
            last_par = (last_par & ~bit) | (par << s);
            filled |= bit;
            return par;
        };
        // one stage slot: wait until it is free (lane 0), the answer goes to the whole warp
        auto acquire = [&](uint32_t kk) -> bool {
            int got = 1;
            if (lane == 0) got = mbar_wait(empty + rslot(kk), (rround(kk) & 1) ^ 1, abort_flag, p.err, wait_ns) ? 1 : 0;
            return __shfl_sync(0xffffffffu, got, 0) != 0;
        };
        auto issue_w = [&](const Item &t, int kb, uint32_t kk) {
            const GemmModule &M = p.mod[t.m];
            const uint32_t sl = rslot(kk);
            note_fill((int)sl, false);
            if (lane == 0) {
                uint8_t *sa = smem + (size_t)sl * stage_bytes;
                mbar_arrive_expect_tx(wfull + sl, stage_bytes);
                tma_load_2d(sa, &M.tmW, wfull + sl, kb * kBK, t.w_tile * kBM, pol_w);
                tma_load_2d(sa + a_bytes, &M.tmX, wfull + sl, kb * kBK, t.chunk * p.nt, pol_x);
            }
        };
        // a tile's next slot (walked with sg / r): a segment's rows in the chunk in runs of pf_ch
        auto issue_b = [&](const Item &t, int &sg, int &r, uint32_t kk) {
            const GemmModule &M = p.mod[t.m];
            const int o0 = t.w_tile * kBM, row0 = t.chunk * p.nt;
            const int orows = min(kBM, M.d_out - o0);
            const int row1 = min(p.n, row0 + p.nt);
            const uint32_t ring_s = rslot(kk);
            uint8_t *sa = smem + (size_t)ring_s * stage_bytes;
            uint8_t *sx = sa + a_bytes;
            uint64_t *bar = bfull + ring_s;
            note_fill((int)ring_s, true);
            if (lane != 0) return;
            const int ns = *p.n_seg;
            int s1 = 0, a = -1;
            for (; sg < ns; ++sg) {  // the next segment with an adapter and rows left in the chunk
                s1 = min(p.seg_start[sg + 1], row1);
                a = p.seg_adapter[sg];
                r = max(r, p.seg_start[sg]);
                if (a >= 0 && r < s1) break;
            }
            BStageHdr *hdr = reinterpret_cast<BStageHdr *>(sx);
            if (sg >= ns) {  // the chunk has fewer slots than counted: an empty stage
                report(p.err, LORA_DEVERR_BAD_SEGMENTS, t.chunk);
                hdr->nslots = 0;
                fence_proxy_async_smem();
                mbar_arrive(bar);
                return;
            }
            const int nr = min(p.pf_ch, s1 - r);
            const PoolEntry e = M.table[a];
            BSlotS sl;
            sl.q0 = r;
            sl.nrows = (int16_t)nr;
            sl.rp = (int16_t)e.rp;
            sl.off = 0;
            sl.tstride = (int16_t)p.rpmax;
            sl.toff = 0;
            hdr->nslots = 1;
            hdr->slot[0] = sl;
            fence_proxy_async_smem();  // the slot is refilled by TMA later
            const uint32_t bb = (uint32_t)(orows * e.rp * 2), tb = (uint32_t)(nr * p.rpmax * 4);
            mbar_arrive_expect_tx(bar, bb + tb);
            bulk_load(sa, e.B + (size_t)o0 * e.rp, bb, bar);
            bulk_load(sx + kStageHdrBytes, M.T + (size_t)r * p.rpmax, tb, bar);
            r += nr;
        };
        Item cur, nxt;
        bool has = rr_item(p, blockIdx.x, 0, cur);
        if (has) {
            int sg = p.chunk_seg0[cur.chunk], r = cur.chunk * p.nt;
            for (int q = 0; q < cur.nbs && ok; ++q, ++k) {
                if (!acquire(k)) {
                    ok = false;
                    break;
                }
                issue_b(cur, sg, r, k);
            }
        }
        for (int jt = 0; has && ok; ++jt) {
            const bool has_nxt = rr_item(p, blockIdx.x, jt + 1, nxt);
            const int lead = min(kGroupedLead, cur.kbn);
            int sg = has_nxt ? p.chunk_seg0[nxt.chunk] : 0, r = has_nxt ? nxt.chunk * p.nt : 0;
            for (int kb = 0; kb <= cur.kbn && ok; ++kb) {
                if (kb == lead && has_nxt)
                    for (int q = 0; q < nxt.nbs && ok; ++q, ++k) {
                        if (!acquire(k)) {
                            ok = false;
                            break;
                        }
                        issue_b(nxt, sg, r, k);
                    }
                if (kb == cur.kbn || !ok) continue;
                if (!acquire(k)) {
                    ok = false;
                    break;
                }
                issue_w(cur, kb, k);
                ++k;
            }
            cur = nxt;
            has = has_nxt;
        }
        // never leave the block with copies still landing in its shared memory: wait for the
        // latest fill of every slot
        if (lane == 0)
            for (int q = 0; q < S; ++q) {
                if (!((filled >> q) & 1u)) continue;
                const uint32_t a = smem_u32(((last_b >> q) & 1u) ? bfull + q : wfull + q);
                const uint64_t t0 = globaltimer();
                while (!mbar_try_wait(a, (last_par >> q) & 1u) && globaltimer() - t0 < kWaitBudgetNs) {
                }
            }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            const uint32_t idesc = idesc_bf16_f32(kBM, (uint32_t)p.nt);
            uint32_t k = 0, use0 = 0, use1 = 0, wpar = 0;
            bool ok = true;
            // one W k-block at stage k into accumulator column d; the epilogue wrote the tile's
            // expand into the accumulator first, so every k-block accumulates on top of it
            auto mma_stage = [&](uint32_t d) -> bool {
                const int s = (int)rslot(k);
                if (!mbar_wait(wfull + s, (wpar >> s) & 1u, abort_flag, p.err, wait_ns)) return false;
                wpar ^= 1u << s;
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + (size_t)s * stage_bytes);
                const uint64_t da = sdesc_kmajor_sw128(sa);
                const uint64_t db = sdesc_kmajor_sw128(sa + a_bytes);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) umma_bf16(d, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2), idesc, 1u);
                umma_commit(empty + s);
                return true;
            };
            Item cur, nxt;
            bool has = rr_item(p, blockIdx.x, 0, cur);
            if (has) k += (uint32_t)cur.nbs;
            for (int jt = 0; has && ok; ++jt) {
                const bool has_nxt = rr_item(p, blockIdx.x, jt + 1, nxt);
                const int buf = jt & 1;
                const uint32_t use = buf ? use1 : use0;
                if (!mbar_wait(acc_free + buf, use & 1, abort_flag, p.err, wait_ns)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * p.nt);
                const int lead = min(kGroupedLead, cur.kbn);
                for (int kb = 0; kb < cur.kbn; ++kb) {
                    if (kb == lead && has_nxt) k += (uint32_t)nxt.nbs;
                    if (!mma_stage(d)) {
                        ok = false;
                        break;
                    }
                    ++k;
                }
                if (!ok) break;
                if (lead == cur.kbn && has_nxt) k += (uint32_t)nxt.nbs;
                umma_commit(acc_full + buf);
                if (buf) ++use1; else ++use0;
                cur = nxt;
                has = has_nxt;
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
        c.etid = threadIdx.x - 64;
        c.lane_base = (warp & 3) * 32;
        c.o = c.lane_base + lane;
        c.n = p.n;
        c.nt = p.nt;
        c.y_bf16 = p.y_bf16;
        const uint32_t lane_off = (uint32_t)c.lane_base << 16;
        uint32_t bpar = 0;
        // wait for the B stage at ring slot kk (all 128 threads); false if the wait gave up
        auto wait_b = [&](uint32_t kk) -> bool {
            const int s = (int)rslot(kk);
            const bool ok = !named_bar_or(1, 128, !mbar_wait(bfull + s, (bpar >> s) & 1u, abort_flag, p.err, wait_ns));
            if (ok) bpar ^= 1u << s;
            return ok;
        };
        float z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0.f;
        uint32_t use0 = 0, use1 = 0;
        // the expand of tile t into accumulator buf (zeros + delta), then acc_free lets the MMA
        // warp start on it.  A B stage is copied into the y buffer first, so its ring slot is
        // given back at once.
        auto pre = [&](const Item &t, int buf, uint32_t k0) -> bool {
            const uint32_t tacc = tmem_base + lane_off + (uint32_t)(buf * p.nt);
            const int row0 = t.chunk * p.nt;
            for (int c0 = 0; c0 < p.nt; c0 += 16) tmem_st16(tacc + (uint32_t)c0, z);
            tmem_st_wait();
            for (int q = 0; q < t.nbs; ++q) {
                const uint32_t kk = k0 + (uint32_t)q;
                if (!wait_b(kk)) return false;
                const uint8_t *sa = smem + (size_t)rslot(kk) * stage_bytes;
                const uint8_t *sx = sa + a_bytes;
                const BStageHdr *hdr = reinterpret_cast<const BStageHdr *>(sx);
                // the slot's B rows ([128][rp], rank offset 0), then header and t rows
                const uint32_t bbytes = hdr->nslots > 0 ? (uint32_t)(kBM * hdr->slot[0].rp * 2) : 0u;
                const uint32_t tbytes = hdr->nslots > 0 ? (uint32_t)(hdr->slot[0].nrows * p.rpmax * 4) : 0u;
                if (c.etid == 0) bulk_wait_read<0>();  // y stores of the last drain have read the buffer
                named_bar_sync(1, 128);
                for (uint32_t off = (uint32_t)c.etid * 16; off < bbytes; off += 128 * 16)
                    *reinterpret_cast<uint4 *>(ybuf + off) = *reinterpret_cast<const uint4 *>(sa + off);
                for (uint32_t off = (uint32_t)c.etid * 16; off < kStageHdrBytes + tbytes; off += 128 * 16)
                    *reinterpret_cast<uint4 *>(ybuf + bbytes + off) = *reinterpret_cast<const uint4 *>(sx + off);
                named_bar_sync(1, 128);  // the copy is complete: the slot goes back
                if (c.etid == 0) mbar_arrive(empty + rslot(kk));
                expand_stage(c, ybuf, ybuf + bbytes, tacc, row0);
                named_bar_sync(1, 128);  // before the buffer is overwritten
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free + buf);
            return true;
        };
        Item cur, nxt;
        bool has = rr_item(p, blockIdx.x, 0, cur);
        bool ok = true;
        uint32_t kw = 0;  // ring position of the current tile's first k-block
        if (has) {
            ok = pre(cur, 0, 0);
            kw = (uint32_t)cur.nbs;
        }
        for (int jt = 0; has && ok; ++jt) {
            const bool has_nxt = rr_item(p, blockIdx.x, jt + 1, nxt);
            const int buf = jt & 1;
            const int lead = min(kGroupedLead, cur.kbn);
            if (has_nxt) ok = pre(nxt, buf ^ 1, kw + (uint32_t)lead);
            if (!ok) break;
            const uint32_t use = buf ? use1 : use0;
            ok = mbar_wait(acc_full + buf, use & 1, abort_flag, p.err, wait_ns);
            if (named_bar_or(1, 128, !ok)) break;
            tc_fence_after();
            drain(c, cur, buf, tmem_base, ybuf, (uint32_t)p.ybuf_bytes);
            tc_fence_before();
            __syncwarp();
            if (buf) ++use1; else ++use0;
            kw += (uint32_t)cur.kbn + (has_nxt ? (uint32_t)nxt.nbs : 0u);
            cur = nxt;
            has = has_nxt;
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

static size_t gemm_smem_bytes(int nt, int n_stages, int ybuf_bytes) {
    const size_t stage = (size_t)kBM * kBK * 2 + (size_t)nt * kBK * 2;
    return 1024 + stage * n_stages + (size_t)ybuf_bytes + 8 * (3 * (size_t)n_stages + 5) + 16;
}

bool plan_gemm(GemmParams &gp, size_t *smem_bytes) {
    // TMEM: two accumulators of nt columns (the expand is written into the accumulator before
    // the tile's MMAs); a dedicated y buffer, so every tile drains while the next one streams
    const int cols = 2 * gp.nt;
    gp.tmem_cols = 32;
    while (gp.tmem_cols < cols) gp.tmem_cols <<= 1;
    gp.ybuf_bytes = kYBufBytes;
    const size_t stage = (size_t)kBM * kBK * 2 + (size_t)gp.nt * kBK * 2;
    const size_t fixed = gemm_smem_bytes(gp.nt, 0, gp.ybuf_bytes);
    gp.n_stages = (int)std::min<size_t>(kMaxStages, (227 * 1024 - fixed - 24 * kMaxStages) / stage);
    *smem_bytes = gemm_smem_bytes(gp.nt, gp.n_stages, gp.ybuf_bytes);
    return gp.n_stages >= 2;
}

cudaError_t launch_prep_segments(const PrepParams &p, cudaStream_t s) {
    return launch_pdl(prep_segments_kernel, dim3(1), dim3(1024), 0, s, p);
}

cudaError_t launch_shrink(const ShrinkParams &p, int grid_x, int grid_y, cudaStream_t s) {
    if (p.by_segment) {
        if (!p.i8) return cudaErrorInvalidValue;  // bf16 decode batches shrink on the tensor cores
        return launch_pdl(shrink_decode_kernel, dim3(grid_x, grid_y), dim3(kShrinkThreads), 0, s, p);
    }
    return launch_pdl(shrink_kernel, dim3(grid_x, grid_y), dim3(kShrinkThreads), 0, s, p);
}

cudaError_t launch_gemm(const GemmParams &p, size_t smem_bytes, cudaStream_t s) {
    static size_t configured = 0;
    if (smem_bytes > configured) {
        cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
        if (e != cudaSuccess) return e;
        configured = smem_bytes;
    }
    return launch_pdl(gemm_kernel, dim3(p.n_cta), dim3(kGemmThreads), smem_bytes, s, p);
}

cudaError_t launch_table_write(PoolEntry *dst, PoolEntry value, cudaStream_t s) {
    table_write_kernel<<<1, 1, 0, s>>>(dst, value);
    return cudaGetLastError();
}

cudaError_t launch_table_write_many(const TableWrites &w, cudaStream_t s) {
    if (w.n <= 0) return cudaSuccess;
    table_write_many_kernel<<<1, kTableWritesMax, 0, s>>>(w);
    return cudaGetLastError();
}

cudaError_t launch_packed_load(const PackedJobs &jobs, cudaStream_t s) {
    if (jobs.n <= 0) return cudaSuccess;
    packed_load_kernel<<<dim3(jobs.n, 16), 256, 0, s>>>(jobs);
    return cudaGetLastError();
}

}  // namespace lora
