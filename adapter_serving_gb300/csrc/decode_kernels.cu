// decode_kernels.cu -- the decode path of the adapted linear layer y_i = W x_i + s B_a (A_a x_i),
// for a batch of at most 256 rows that each carry their own adapter id:
//
//   prep_decode_kernel      row grouping: stable sort of the rows by adapter id (the segments),
//                           id checks, and per projection the gather list of the distinct
//                           adapters' A rows (8-row groups)
//   decode_gemm_kernel      one persistent tcgen05 GEMM per call over two tile spaces, each split
//                           stream-K over the SMs: W tiles (128 rows of W: the base W x) and A tiles
//                           (128 gathered rows of the distinct adapters' A: the shrink A_a x).  Both
//                           multiply the same x k-blocks; base pieces go to the workspace, the
//                           shrink's t values (row j against its own adapter's rows only) to per-CTA
//                           partial buffers.  The W tiles need no row plan and run first
//   decode_finalize_kernel  per (W tile, 16 rows of the adapter-sorted batch): the base pieces added
//                           in k order, t (the parts summed in k order and scaled, here or by the
//                           gemm), the expand s B_a t on CUDA cores (B read once per adapter and
//                           block), y written
//
// The forward is "m07 -- Multi-Adapter (LoRA) Serving", section 6 "Deep Dive A: Batching
// Heterogeneous Adapters": one base GEMM shared by the batch plus a per-row adapter product
// gathered through an index vector inside the kernel; "the cost is bandwidth, not compute": W is
// read once per call and every distinct adapter's A and B once per call.  The shrink rides on the
// tensor cores because the base GEMM's operand stream is already there: an A tile costs the same
// bytes as the CUDA-core shrink and multiplies every row (the rows of other adapters are computed
// and dropped), which is free at decode, where the tensor pipe idles.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>

#include "lora_internal.h"
#include "prep_common.cuh"
#include "ptx.cuh"

namespace lora {

// ============================================================================ prep ==========

constexpr int kPrepGroups = 4;  // groups of 256 threads; group g builds projections g, g + 4
constexpr int kFinRows = 16;     // rows of the sorted batch per finalize block (a "row block")

// Exclusive prefix sum of 64-bit values over a group of 256 threads (8 warps) on named barrier
// `bar`; `total` receives the sum.
__device__ uint64_t group_scan256_u64(uint64_t v, uint64_t *s_warp, uint64_t &total, int bar) {
    const int lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) & 7;
    uint64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    named_bar_sync(bar, 256);
    uint64_t before = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const uint64_t t = s_warp[w];
        before += w < warp ? t : 0;
        tot += t;
    }
    named_bar_sync(bar, 256);  // s_warp may be reused
    total = tot;
    return before + x - v;
}

// Row grouping state the prep block keeps in shared memory (n <= 256 rows).
struct PrepShared {
    int id[LORA_MAX_DECODE_ROWS];                    // adapter id of row r (-1 = base only)
    int sorted[LORA_MAX_DECODE_ROWS];                // adapter id at sorted position q
    int perm[LORA_MAX_DECODE_ROWS];                  // row at sorted position q
    int cnt[4][LORA_MAX_DECODE_ROWS];                // partial position counts
    int seg_q0[LORA_MAX_DECODE_ROWS + 1];            // first position of segment s
    int rank[LORA_MAX_MODULES][LORA_MAX_DECODE_ROWS];  // rank at position q (0 = none)
    int arow[LORA_MAX_MODULES][LORA_MAX_DECODE_ROWS];  // first A-slab row of the adapter at q
    int scan[8];
};

// The gather list of every projection: each segment with an adapter of rank r takes ceil(r / 8)
// consecutive 8-row groups (its A rows in order), segments in sorted order; a row's t values sit
// at slot rows [8 g0, 8 g0 + r) of its segment's first group g0.
__device__ void build_groups(const PrepParams &p, const PrepShared &sh, int ns) {
    __shared__ uint64_t s_warp_all[kPrepGroups][8];
    const int g = threadIdx.x >> 8, tid = threadIdx.x & 255;
    const int bar = 1 + g;
    uint64_t *s_warp = s_warp_all[g];
    for (int m = g; m < p.n_mod; m += kPrepGroups) {
        int cnt = 0, q0 = 0, q1 = 0, r = 0, row = 0;
        if (tid < ns) {
            q0 = sh.seg_q0[tid];
            q1 = sh.seg_q0[tid + 1];
            r = sh.rank[m][q0];
            row = sh.arow[m][q0];
            if (sh.sorted[q0] >= 0 && r > 0) cnt = (r + kGroupRows - 1) / kGroupRows;
        }
        uint64_t tot = 0;
        const int g0 = (int)group_scan256_u64((uint64_t)cnt, s_warp, tot, bar);
        AGroup *G = p.groups[m];
        for (int k = 0; k < cnt; ++k) {
            AGroup a;
            a.row = row + kGroupRows * k;
            a.q0 = (int16_t)q0;
            a.q1 = (int16_t)q1;
            a.rbase = (int16_t)(kGroupRows * k);
            a.rank = (int16_t)r;
            a.pad_ = 0;
            G[g0 + k] = a;
        }
        // the segment's rows find their t parts through the first group
        if (cnt > 0)
            for (int q = q0; q < q1; ++q) p.rowinfo[m][sh.perm[q]].g0 = g0;
        if (tid == 0) p.n_groups[m] = (int)tot;
    }
}

// One block of 1024 threads, n <= 256 rows.  Position of row i in the stable order:
// #{j : id_j < id_i} + #{j < i : id_j == id_i}, counted by four threads per row over a quarter
// of the rows each.
__global__ void __launch_bounds__(256 * kPrepGroups) prep_decode_kernel(const PrepParams p) {
    __shared__ PrepShared sh;
    const int tid = threadIdx.x;
    const int n = p.n;
    grid_dep_wait();
    grid_dep_launch();
    bool seg_ok = true;
    if (p.ids == nullptr) {
        seg_ok = segments_valid_block(p);
        if (!seg_ok && tid == 0) report(p.err, LORA_DEVERR_BAD_SEGMENTS, 0);
    }
    // ---- ids, checked; every projection's rank and A row of the row's adapter (loads in flight first)
    int id = -1;
    int rank_row[LORA_MAX_MODULES], arow_row[LORA_MAX_MODULES], rp_row[LORA_MAX_MODULES];
    const uint16_t *B_row[LORA_MAX_MODULES];
    if (tid < n) {
        int where = tid;
        if (p.ids) {
            id = p.ids[tid];
        } else if (seg_ok) {
            where = seg_of(p.seg_start_in, p.n_seg_in, tid);
            id = p.seg_adapter_in[where];
        }
        if (id < -1 || id >= p.max_adapters) {
            report(p.err, LORA_DEVERR_BAD_ADAPTER, where);
            id = -1;
        }
#pragma unroll
        for (int m = 0; m < LORA_MAX_MODULES; ++m) {
            rank_row[m] = 1;
            arow_row[m] = 0;
            rp_row[m] = 0;
            B_row[m] = nullptr;
            if (id >= 0 && m < p.n_mod) {
                const PoolEntry *e = p.table[m] + id;
                rank_row[m] = e->rank;
                arow_row[m] = (int)e->row_off;
                rp_row[m] = e->rp;
                B_row[m] = e->B;
            }
        }
        bool ok = true;
#pragma unroll
        for (int m = 0; m < LORA_MAX_MODULES; ++m) ok = ok && rank_row[m] > 0;
        if (!ok) {
            report(p.err, LORA_DEVERR_NOT_LOADED, where);
            id = -1;
        }
        if (id < 0) {
#pragma unroll
            for (int m = 0; m < LORA_MAX_MODULES; ++m) rank_row[m] = 0;
        }
        sh.id[tid] = id;
        p.radapter[tid] = id;
#pragma unroll
        for (int m = 0; m < LORA_MAX_MODULES; ++m)
            if (m < p.n_mod) {
                RowInfo ri;
                ri.B = id >= 0 ? B_row[m] : nullptr;
                ri.rank = (int16_t)(id >= 0 ? rank_row[m] : 0);
                ri.rp = (int16_t)(id >= 0 ? rp_row[m] : 0);
                ri.g0 = 0;
                p.rowinfo[m][tid] = ri;
            }
    }
    __syncthreads();
    // ---- stable sort: four partial counts per row
    {
        const int row = tid & 255, part = tid >> 8;
        if (row < n) {
            const int v = sh.id[row];
            const int j0 = part * n / 4, j1 = (part + 1) * n / 4;
            int c = 0;
            for (int j = j0; j < j1; ++j) {
                const int u = sh.id[j];
                c += (u < v) || (u == v && j < row);
            }
            sh.cnt[part][row] = c;
        }
    }
    __syncthreads();
    if (tid < n) {
        const int pos = sh.cnt[0][tid] + sh.cnt[1][tid] + sh.cnt[2][tid] + sh.cnt[3][tid];
        p.perm[pos] = tid;
        p.qadapter[pos] = id;
        sh.perm[pos] = tid;
        sh.sorted[pos] = id;
#pragma unroll
        for (int m = 0; m < LORA_MAX_MODULES; ++m) {
            sh.rank[m][pos] = rank_row[m];
            sh.arow[m][pos] = arow_row[m];
        }
    }
    __syncthreads();
    // ---- segment starts: positions whose id differs from the one before; inclusive scan of the
    // flags (warp shuffles, then the 8 warp totals)
    int flag = 0;
    if (tid < 256) flag = (tid < n) && (tid == 0 || sh.sorted[tid] != sh.sorted[tid - 1]);
    int incl = flag;
    const int lane = tid & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (tid < 256 && lane == 31) sh.scan[tid >> 5] = incl;
    __syncthreads();
    int before = 0, ns = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        const int t = sh.scan[w];
        before += w < (tid >> 5) ? t : 0;
        ns += t;
    }
    if (flag) {
        const int seg = before + incl - 1;
        p.seg_start[seg] = tid;
        p.seg_adapter[seg] = sh.sorted[tid];
        sh.seg_q0[seg] = tid;
    }
    if (tid == 0) {
        *p.n_seg = ns;
        p.seg_start[ns] = n;
        sh.seg_q0[ns] = n;
    }
    // The finalize's row blocks heaviest first (when its blocks take more than one wave, the ones
    // with the most B to stage start first): a block's weight is the sum of the ranks of the
    // distinct adapters among its 16 positions (the first projection's), ties in block order.
    if (p.rb_order != nullptr) {
        __shared__ int s_weight[LORA_MAX_DECODE_ROWS / kFinRows];
        const int nrb = (n + kFinRows - 1) / kFinRows;
        if (tid < nrb) {
            int wgt = 0;
            for (int q = tid * kFinRows; q < min(n, (tid + 1) * kFinRows); ++q)
                if (sh.sorted[q] >= 0 && (q == tid * kFinRows || sh.sorted[q - 1] != sh.sorted[q])) wgt += sh.rank[0][q];
            s_weight[tid] = wgt;
        }
        __syncthreads();
        if (tid < nrb) {
            const int wgt = s_weight[tid];
            int pos = 0;
            for (int b = 0; b < nrb; ++b) pos += (s_weight[b] > wgt) || (s_weight[b] == wgt && b < tid);
            p.rb_order[pos] = tid;
        }
    }
    if (p.groups[0] != nullptr) {
        __syncthreads();  // the segment table is complete
        build_groups(p, sh, ns);
    }
}

// ============================================================================ gemm ==========
//
// Two launches per call, each a programmatic dependent of the one before it.
//
// decode_gemm_kernel: one CTA per SM (at most), warp roles: warp 0 is the TMA producer, lane 0 of
// warp 1 issues tcgen05.mma, warps 2-5 are the epilogue (TMEM lane quarter = warp % 4); with an
// int4 base, warps 6-9 convert W codes to bf16 between the TMA load and the MMA.  MMA M = 128 rows
// of W or of the gathered A rows, N = the batch (nt columns, column = row of the batch), K = d_in
// in 64-wide k-blocks.  Each of the two tile spaces is split stream-K: CTA c takes k-blocks
// [c T / N, (c + 1) T / N) of the W space (T = all W tiles' k-blocks, N = CTAs) and its share of
// the A space (whose size the prep decided on the device): the W range first, before anything
// waits for the row plan, unless x is the previous call's output.  Every item (a tile's k range
// held by one CTA) accumulates into one of two TMEM buffers, so the drain of one overlaps the MMAs
// of the next.  W items leave base pieces in the workspace half of the call's parity; A items
// leave, for every row j, its share of t_j (the rows of its own adapter only), added up in k order
// by the finalize or by the last CTA to finish the tile (a counter, no waiting).  The epilogue
// warps, once they have waited for the kernel before, let the dependent launch: the finalize's
// blocks take the resources the gemm leaves and wait, so they start the moment the gemm is done.
//
// decode_finalize_kernel: block (W tile, 16 rows of the batch), thread o = output row 128 tile + o:
//   base  = the tile's pieces in k order (the piece from k-block 0, then every later CTA's)
//   t_j   = s * (the A tiles' parts in k order), summed here or by the gemm, or the CUDA-core
//           shrink's row (int8 factors)
//   y[j, o] = base + sum_r B_a(j)[o, r] t_j[r]
// The rows' adapters and their B rows are fetched before the block waits for the gemm; after it,
// one round of loads (t and the pieces), the dot products and the stores.  B is read as
// the pool stores it ([d_out, rp]): a block reads one contiguous run of 128 rows of each row's
// adapter.

constexpr int kConvWarp0 = 2 + kEpiWarps;
constexpr int kDecThreads = 32 * (kConvWarp0);
constexpr int kDecThreadsW4 = 32 * (kConvWarp0 + kConvWarps);
constexpr uint32_t kPreL2 = 12;                // W k-blocks asked of L2 before the wait

// The A space of a call, computed from the prep's group counts (one thread).
struct DecShared {
    int32_t a_begin[LORA_MAX_MODULES + 1];  // first A-space k-block of each projection
    int32_t n_groups[LORA_MAX_MODULES];
    int32_t a_iters, a_ctas;
};

__device__ void dec_a_space(const DecodeParams &p, DecShared &d) {
    // every projection's group count in flight at once (one round trip, not one per projection)
    int gs[LORA_MAX_MODULES];
#pragma unroll
    for (int m = 0; m < LORA_MAX_MODULES; ++m) gs[m] = (m < p.n_mod && p.shrink_tc) ? __ldcg(p.mod[m].n_groups) : 0;
    int it = 0, kbn_max = 0;
#pragma unroll
    for (int m = 0; m < LORA_MAX_MODULES; ++m) {
        if (m >= p.n_mod) break;
        const int g = min(max(gs[m], 0), kDecMaxGroups);
        const int at = (g + kTileGroups - 1) / kTileGroups;
        d.n_groups[m] = g;
        d.a_begin[m] = it;
        it += at * p.mod[m].k_blocks;
        if (at > 0) kbn_max = max(kbn_max, p.mod[m].k_blocks);
    }
    d.a_begin[p.n_mod] = it;
    d.a_iters = it;
    d.a_ctas = decode_a_ctas(it, kbn_max, p.n_cta);
}

// The CTA whose range [c T / N, (c + 1) T / N) holds position x (32-bit arithmetic while T N
// fits, as it does for every shape a pool can hold).
__device__ __forceinline__ int cta_of(int64_t x, int64_t total, int n) {
    if (total * n < 0x7fffffff) return (int)(((uint32_t)(x + 1) * (uint32_t)n - 1u) / (uint32_t)total);
    return (int)(((x + 1) * n - 1) / total);
}

struct DItem {
    int32_t a;         // 0: W tile, 1: A tile
    int32_t m;         // projection
    int32_t tile;      // tile within the projection (W: rows 128 tile..; A: groups 16 tile..)
    int32_t kb0, kb1;  // the CTA's k-blocks of the tile
    int32_t it0;       // the tile's first k-block in its space
};

// A CTA's items come in two ranges, walked one after the other: its W range (W tiles of every
// projection, split evenly over the CTAs) and its share of the A space (known only from the row
// plan).  Which comes first is the call's choice (see the kernel).
struct DSched {
    int64_t x, e;
    int32_t phase, cta;
    // the W range
    __device__ void begin_w(const DecodeParams &p, int c) {
        cta = c;
        phase = 1;
        x = (int64_t)c * p.w_iters / p.n_cta;
        e = (int64_t)(c + 1) * p.w_iters / p.n_cta;
    }
    // the share of the A space
    __device__ void begin_a(const DecodeParams &p, int c, const DecShared &d) {
        cta = c;
        phase = 0;
        if (c < d.a_ctas) {
            x = (int64_t)c * d.a_iters / d.a_ctas;
            e = (int64_t)(c + 1) * d.a_iters / d.a_ctas;
        } else {
            x = e = 0;
        }
    }
    __device__ bool next(const DecodeParams &p, const DecShared *d, DItem &it) {
        if (phase == 0) {
            if (x < e) {
                int m = 0;
                while (m + 1 < p.n_mod && d->a_begin[m + 1] <= x) ++m;
                const int kbn = p.mod[m].k_blocks;
                const int local = (int)(x - d->a_begin[m]);
                const int at = local / kbn;
                it.a = 1;
                it.m = m;
                it.tile = at;
                it.kb0 = local - at * kbn;
                it.kb1 = (e - x) < (int64_t)(kbn - it.kb0) ? it.kb0 + (int)(e - x) : kbn;
                it.it0 = d->a_begin[m] + at * kbn;
                x += it.kb1 - it.kb0;
                return true;
            }
            phase = 2;
            return false;
        }
        if (phase == 1 && x < e) {
            int m = 0;
            while (m + 1 < p.n_mod && p.mod[m + 1].w_iter_begin <= x) ++m;
            const int kbn = p.mod[m].k_blocks;
            const int local = (int)(x - p.mod[m].w_iter_begin);
            const int lt = local / kbn;
            it.a = 0;
            it.m = m;
            it.tile = lt;
            it.kb0 = local - lt * kbn;
            it.kb1 = (e - x) < (int64_t)(kbn - it.kb0) ? it.kb0 + (int)(e - x) : kbn;
            it.it0 = p.mod[m].w_iter_begin + lt * kbn;
            x += it.kb1 - it.kb0;
            return true;
        }
        phase = 2;
        return false;
    }
};

// Base pieces are kept by batch row: the value of row j (the MMA's column j) for output row o of the
// tile sits at j * 128 + o.  A warp stores 128 contiguous bytes per column, and the finalize, whatever
// order it walks rows in, reads 512 contiguous bytes per row.

// W4: the int4 codes of one W k-block ([128 rows][32 bytes] as the TMA lays the box down) into the
// bf16 tile of the integers the MMA reads ([128 rows][64], 128-byte swizzle: the 16-byte chunk j of
// row r sits at chunk j ^ (r % 8)).  Packing: a 32-bit word holds 8 consecutive k elements; nibble s
// of the low half is element 2s and nibble s of the high half element 2s + 1, each stored as
// code + 8.  (0x4300 | u) read as bf16 is 128 + u, so one mask-or per pair and one bf16x2
// subtraction of 136 give two codes.  Thread ct of the kConvWarps * 32 converter threads takes
// 16-byte pieces ct, ct + 64, ...: piece i is half i % 2 of row i / 2.
__device__ __forceinline__ uint4 w4_bf16x8(uint32_t w) {
    const __nv_bfloat162 off = __floats2bfloat162_rn(136.f, 136.f);
    uint32_t r[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const uint32_t b = ((w >> (4 * s)) & 0x000F000Fu) | 0x43004300u;
        const __nv_bfloat162 h = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&b), off);
        r[s] = *reinterpret_cast<const uint32_t *>(&h);
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

__device__ __forceinline__ void convert_w4_kblock(uint32_t raw, uint32_t dst, int ct) {
#pragma unroll
    for (int i = 0; i < (kBM * 2) / (kConvWarps * 32); ++i) {
        const int idx = ct + i * kConvWarps * 32;
        const int r = idx >> 1, h = idx & 1;
        const uint4 w = lds_u128(raw + (uint32_t)idx * 16);
        const uint32_t row = dst + (uint32_t)r * 128;
        const uint32_t sw = (uint32_t)(r & 7);
        sts_u128(row + (((uint32_t)(4 * h + 0) ^ sw) << 4), w4_bf16x8(w.x));
        sts_u128(row + (((uint32_t)(4 * h + 1) ^ sw) << 4), w4_bf16x8(w.y));
        sts_u128(row + (((uint32_t)(4 * h + 2) ^ sw) << 4), w4_bf16x8(w.z));
        sts_u128(row + (((uint32_t)(4 * h + 3) ^ sw) << 4), w4_bf16x8(w.w));
    }
}

// two floats as a bf16x2 word (round to nearest even), the first in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// 8 bf16 of B against 8 fp32 t values
__device__ __forceinline__ float dot8_b(uint4 b, const float *t) {
    float a0 = bf16lo(b.x) * t[0], a1 = bf16hi(b.x) * t[1];
    a0 = fmaf(bf16lo(b.y), t[2], a0);
    a1 = fmaf(bf16hi(b.y), t[3], a1);
    a0 = fmaf(bf16lo(b.z), t[4], a0);
    a1 = fmaf(bf16hi(b.z), t[5], a1);
    a0 = fmaf(bf16lo(b.w), t[6], a0);
    a1 = fmaf(bf16hi(b.w), t[7], a1);
    return a0 + a1;
}
// 8 int8 codes of B against 8 fp32 t values (the int8 scales are already folded into t)
__device__ __forceinline__ float dot8_b(uint2 b, const float *t) {
    const float4 lo = i8x4(b.x), hi = i8x4(b.y);
    float a0 = lo.x * t[0], a1 = lo.y * t[1];
    a0 = fmaf(lo.z, t[2], a0);
    a1 = fmaf(lo.w, t[3], a1);
    a0 = fmaf(hi.x, t[4], a0);
    a1 = fmaf(hi.y, t[5], a1);
    a0 = fmaf(hi.z, t[6], a0);
    a1 = fmaf(hi.w, t[7], a1);
    return a0 + a1;
}


// W4: the base weights are int4 codes with one fp32 scale per output row ("12. Adapter Serving and
// Multi-Tenant Customization", section "Quantization": an INT4 base dequantised in the kernel,
// BF16 adapters, wide accumulation).  The codes enter the MMA as exact bf16 integers and the drain
// multiplies the accumulator by the row's scale.
template <bool W4>
__global__ void __launch_bounds__(W4 ? kDecThreadsW4 : kDecThreads, 1) decode_gemm_kernel(const __grid_constant__ DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ DecShared dsh;
    __shared__ int32_t perm_s[LORA_MAX_DECODE_ROWS];
    __shared__ int s_last;
    const int S = p.n_stages;
    // Ring slot and round of fill k without an integer division in the loops:
    // k / S = umulhi(k, ceil(2^32 / S)), exact for k < 2^32 / 8 when S <= 8.
    const uint32_t ring_m = 0xFFFFFFFFu / (uint32_t)S + 1u;
    auto rround = [ring_m](uint32_t kk) -> uint32_t { return __umulhi(kk, ring_m); };
    auto rslot = [ring_m, S](uint32_t kk) -> uint32_t { return kk - __umulhi(kk, ring_m) * (uint32_t)S; };
    const int nt = p.nt, kps = p.kps;
    // A stage holds one k-step (kps k-blocks of 64): the W or A operand (kps blocks of [128][64]
    // bf16), the x operand (kps blocks of [nt][64]), and with an int4 base the raw codes.  W
    // sub-block q sits at q * 16 KiB; an A tile's group g (8 rows) at g * kps KiB, its sub-block q at
    // + q KiB (so the 8-row atoms of one sub-block are kps KiB apart).
    const uint32_t sub_a = kBM * kBK * 2, sub_x = (uint32_t)nt * kBK * 2;
    const uint32_t a_bytes = (uint32_t)kps * sub_a;
    const uint32_t x_bytes = (uint32_t)kps * sub_x;
    const uint32_t stage_bytes = a_bytes + x_bytes + (W4 ? (uint32_t)(kps * kW4RawBytes) : 0u);
    const uint32_t w_fill = W4 ? (uint32_t)(kps * kW4RawBytes) : a_bytes;  // bytes of W one fill brings
    // one k-step's TMA box of a tensor map at (element or byte) column kx of k-step ks, row y
    auto load = [kps](void *dst, const CUtensorMap *tm, uint64_t *bar, int ks, int kcols, int y, uint64_t pol) {
        if (kps == 1) tma_load_2d(dst, tm, bar, ks * kcols, y, pol);
        else tma_load_3d(dst, tm, bar, 0, y, ks * kps, pol);
    };
    const uint64_t wait_ns = p.wait_ns;
    // Every fill (W or A k-block) completes one phase of its slot's wfull, so the phase of fill k
    // is round(k) & 1 for every waiter; with an int4 base the converters arrive on cfull for every
    // fill (converting W ones), and the MMA waits on cfull instead.
    uint64_t *wfull = reinterpret_cast<uint64_t *>(smem + (size_t)S * stage_bytes);
    uint64_t *cfull = wfull + S;
    uint64_t *empty = cfull + S;
    uint64_t *acc_full = empty + S;
    uint64_t *acc_free = acc_full + 2;
    uint64_t *mma_done = acc_free + 2;
    uint64_t *plan_ready = mma_done + 1;  // the A space and the row order are in shared memory
    uint32_t *misc = reinterpret_cast<uint32_t *>(plan_ready + 1);  // [0] tmem, [1] abort

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(wfull + s, 1);
            mbar_init(cfull + s, kConvWarps * 32);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_free + b, kEpiWarps);
        }
        mbar_init(mma_done, 1);
        mbar_init(plan_ready, 1);
        misc[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        for (int m = 0; m < p.n_mod; ++m) {
            tma_prefetch_desc(&p.mod[m].tmW);
            tma_prefetch_desc(&p.mod[m].tmX);
            if (p.shrink_tc) tma_prefetch_desc(&p.mod[m].tmA);
        }
    }
    if (warp == 1) tmem_alloc(misc, (uint32_t)p.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = misc[0];
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    const uint64_t pol_w = l2_policy_evict_first();  // W and A: read once per call
    const uint64_t pol_x = l2_policy_evict_last();   // x: read by every tile

    // The order of a CTA's items.  W first (p.w_first): the W tiles read only W, x and the workspace
    // of this call's parity, none of which the kernel before this one (the row plan, or the previous
    // call's finalize, which reads the other parity's pieces) writes -- the host checks that x is not
    // the previous call's y -- so they run while that kernel drains, and only the A tiles, which
    // read the row plan, wait for it (griddepcontrol.wait).  Otherwise every role waits first, the
    // A tiles come first, and the CTA's first W k-blocks are asked of L2 before the wait.
    const bool w_first = p.w_first != 0;
    if (!w_first && warp == 0 && lane == 0) {
        DSched sc;
        sc.begin_w(p, blockIdx.x);
        DItem it;
        uint32_t nf = 0;
        while (nf < kPreL2 && sc.next(p, nullptr, it)) {
            const DecodeModule &M = p.mod[it.m];
            for (int kb = it.kb0; kb < it.kb1 && nf < kPreL2; ++kb, ++nf) {
                if (kps == 1) tma_prefetch_2d(&M.tmW, W4 ? kb * (kBK / 2) : kb * kBK, it.tile * kBM);
                else tma_prefetch_3d(&M.tmW, 0, it.tile * kBM, kb * kps);
            }
        }
    }
    // the A range (and with A first, everything) waits for the plan, which the epilogue warps
    // publish after their own griddepcontrol.wait
    auto plan_wait = [&]() -> bool {
        grid_dep_wait();
        return mbar_wait(plan_ready, 0, abort_flag, p.err, wait_ns);
    };
    // item ranges in order: 0 = W (W first), 1 = A, 2 = W (A first)
    const int ph0 = w_first ? 0 : 1, ph1 = w_first ? 2 : 3;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer (warp)
        DItem it;
        uint32_t k = 0;  // stage fills issued
        bool ok = true;
        for (int ph = ph0; ok && ph < ph1; ++ph) {
        if (ph == 1) {
            int got = 1;
            grid_dep_wait();
            if (lane == 0) got = mbar_wait(plan_ready, 0, abort_flag, p.err, wait_ns) ? 1 : 0;
            if (!__shfl_sync(0xffffffffu, got, 0)) break;
        }
        DSched sc;
        if (ph == 1) sc.begin_a(p, blockIdx.x, dsh);
        else sc.begin_w(p, blockIdx.x);
        while (ok && sc.next(p, &dsh, it)) {
            const DecodeModule &M = p.mod[it.m];
            // A tile: lane l < 16 gathers group 16 tile + l (8 rows of one adapter's A) -- unless the
            // tile's groups are consecutive rows of the slab (adapters stored one after another):
            // then one 128-row box, laid out like a W tile (rows past the last group are computed
            // and dropped)
            // (rows past the slab, the copy fills zeros).  With one k-block per stage the gathers
            // go one box per run of consecutive groups instead: a run of length L splits into boxes
            // of L's binary digits, largest first (an adapter's groups are one run of 1, 2, 4 or 8),
            // and the lane at a box's first group issues it (box = log2 of its groups, -1: none).
            int arow = 0, box = -1;
            bool mine = false, runs = false;
            uint32_t a_tx = 0;
            if (it.a) {
                const int g = it.tile * kTileGroups + lane;
                mine = lane < kTileGroups && g < dsh.n_groups[it.m];
                if (mine) arow = M.groups[g].row;
                const int arow0 = __shfl_sync(0xffffffffu, arow, 0);
                const int prev = __shfl_up_sync(0xffffffffu, arow, 1);
                runs = M.a_runs && __all_sync(0xffffffffu, !mine || arow == arow0 + kGroupRows * lane);
                const unsigned valid = __ballot_sync(0xffffffffu, mine);
                // runs are cut at group 8 too, so no box is longer than 8 groups (64 rows)
                const unsigned starts = __ballot_sync(0xffffffffu, mine && (lane == 0 || lane == 8 || arow != prev + kGroupRows));
                if (M.a_boxes && mine) {
                    const unsigned upto = (2u << lane) - 1u;                  // lanes 0..lane
                    const int s0 = 31 - __clz(starts & upto);                 // this run's first lane
                    const int e = __ffs((starts | ~valid) & ~upto) - 1;       // the next run's (lanes >= 16 are not valid)
                    const int len = e - s0, pos = lane - s0;
                    const int tb = 31 - __clz(len - pos);                     // the box at pos, if one starts there
                    box = pos == ((len >> (tb + 1)) << (tb + 1)) ? tb : -1;
                }
                arow = runs ? arow0 : arow;
                a_tx = runs ? (uint32_t)(kps * kBM * kBK * 2) : (uint32_t)__popc(valid) * (uint32_t)(kps * kGroupRows * kBK * 2);
            }
            for (int kb = it.kb0; kb < it.kb1; ++kb, ++k) {
                const uint32_t sl = rslot(k);
                uint8_t *sa = smem + (size_t)sl * stage_bytes;
                {
                    int got = 1;
                    if (lane == 0) got = mbar_wait(empty + sl, (rround(k) & 1) ^ 1, abort_flag, p.err, wait_ns) ? 1 : 0;
                    if (!__shfl_sync(0xffffffffu, got, 0)) {
                        ok = false;
                        break;
                    }
                    if (it.a == 0) {
                        if (lane == 0) {
                            mbar_arrive_expect_tx(wfull + sl, w_fill + x_bytes);
                            if (W4) load(sa + a_bytes + x_bytes, &M.tmW, wfull + sl, kb, kBK / 2, it.tile * kBM, pol_w);
                            else load(sa, &M.tmW, wfull + sl, kb, kBK, it.tile * kBM, pol_w);
                        }
                    } else {
                        if (lane == 0) mbar_arrive_expect_tx(wfull + sl, a_tx + x_bytes);
                        __syncwarp();
                        if (runs) {
                            if (lane == 0) load(sa, &M.tmA128, wfull + sl, kb, kBK, arow, pol_w);
                        } else if (M.a_boxes) {
                            if (box >= 0)
                                load(sa + lane * (kGroupRows * kBK * 2), box == 0 ? &M.tmA : &M.tmAb[box - 1], wfull + sl, kb, kBK, arow, pol_w);
                        } else if (mine) {
                            load(sa + lane * (kps * kGroupRows * kBK * 2), &M.tmA, wfull + sl, kb, kBK, arow, pol_w);
                        }
                    }
                }
                if (lane == 0) load(sa + a_bytes, &M.tmX, wfull + sl, kb, kBK, 0, pol_x);
            }
        }
        }
        // never leave the block with copies still landing in its shared memory: wait for the
        // latest fill of every slot
        const uint32_t issued = k;
        if (lane == 0)
            for (uint32_t q = 0; q < (uint32_t)S && q < issued; ++q) mbar_drain(wfull + q, ((issued - 1 - q) / (uint32_t)S) & 1u, p.err);
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------ MMA issuer
            const uint32_t idesc = idesc_bf16_f32(kBM, (uint32_t)nt);
            DItem it;
            uint32_t k = 0, li = 0;
            bool ok = true;
            for (int ph = ph0; ok && ph < ph1; ++ph) {
            if (ph == 1 && !plan_wait()) break;
            DSched sc;
            if (ph == 1) sc.begin_a(p, blockIdx.x, dsh);
            else sc.begin_w(p, blockIdx.x);
            while (ok && sc.next(p, &dsh, it)) {
                const int buf = li & 1;
                // the producer's choice for an A tile: one 128-row box when its groups are
                // consecutive slab rows (then laid out like a W tile), else 8-row gathers
                bool gathered = false;
                if (it.a) {
                    const DecodeModule &Ma = p.mod[it.m];
                    const int ng = dsh.n_groups[it.m], g0 = it.tile * kTileGroups;
                    int rows[kTileGroups];  // all loads in flight at once
#pragma unroll
                    for (int i = 0; i < kTileGroups; ++i) rows[i] = g0 + i < ng ? __ldg(&Ma.groups[g0 + i].row) : 0;
                    gathered = !Ma.a_runs;
#pragma unroll
                    for (int i = 1; i < kTileGroups; ++i)
                        gathered = gathered || (g0 + i < ng && rows[i] != rows[0] + kGroupRows * i);
                }
                if (!mbar_wait(acc_free + buf, ((li >> 1) & 1) ^ 1, abort_flag, p.err, wait_ns)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * nt);
                for (int kb = it.kb0; kb < it.kb1; ++kb, ++k) {
                    const uint32_t s = rslot(k);
                    if (!mbar_wait((W4 ? cfull : wfull) + s, rround(k) & 1, abort_flag, p.err, wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)s * stage_bytes);
                    for (int q = 0; q < kps; ++q) {
                        // W (and a contiguous A tile): sub-block q at q * 16 KiB, 1 KiB atoms; a gathered
                        // A tile: at q KiB, atoms kps KiB apart
                        const uint64_t da = gathered ? sdesc_kmajor_sw128(sa + (uint32_t)q * 1024u, (uint32_t)kps * 1024u)
                                                     : sdesc_kmajor_sw128(sa + (uint32_t)q * sub_a);
                        const uint64_t db = sdesc_kmajor_sw128(sa + a_bytes + (uint32_t)q * sub_x);
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            umma_bf16(d, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2), idesc,
                                      (kb > it.kb0 || q > 0 || kk > 0) ? 1u : 0u);
                    }
                    umma_commit(empty + s);
                }
                if (!ok) break;
                umma_commit(acc_full + buf);
                ++li;
            }
            }
            umma_commit(mma_done);
            mbar_drain(mma_done, 0, p.err);
        }
    } else if (warp >= 2 && warp < 2 + kEpiWarps) {
        // ---------------------------------------------------------------- epilogue
        const int lane_base = (warp & 3) * 32;
        const int o = lane_base + lane;  // TMEM lane = row of the tile
        const uint32_t lane_off = (uint32_t)lane_base << 16;
        const size_t slot_elems = (size_t)kBM * nt;
        const int ncols16 = (p.n + 15) & ~15;
        // The plan: these warps wait for the kernel before this one, publish the A space and the row
        // order, and let the next kernel launch.  Every kernel before this one has completed, so
        // the finalize may read the row plan (and the factors) before its own wait; it waits for
        // this grid before reading anything this grid writes.
        grid_dep_wait();
        if (threadIdx.x == 64) {
            grid_dep_launch();
            dec_a_space(p, dsh);
        }
        for (int q = threadIdx.x - 64; q < p.n; q += 128) perm_s[q] = p.perm[q];
        named_bar_sync(1, 128);
        if (threadIdx.x == 64) mbar_arrive(plan_ready);
        DItem it;
        uint32_t li = 0;
        bool go = true;
        for (int ph = ph0; go && ph < ph1; ++ph) {
        DSched sc;
        if (ph == 1) sc.begin_a(p, blockIdx.x, dsh);
        else sc.begin_w(p, blockIdx.x);
        while (sc.next(p, &dsh, it)) {
            const int buf = li & 1;
            const bool ok = mbar_wait(acc_full + buf, (li >> 1) & 1, abort_flag, p.err, wait_ns);
            if (named_bar_or(1, 128, !ok)) {
                go = false;
                break;
            }
            tc_fence_after();
            const uint32_t tacc = tmem_base + lane_off + (uint32_t)(buf * nt);
            const DecodeModule &M = p.mod[it.m];
            if (it.a == 0) {
                // base piece -> its workspace slot
                float *const piece = it.kb0 == 0 ? p.home + (size_t)(M.w_tile_begin + it.tile) * slot_elems
                                                 : p.ctaw + (size_t)blockIdx.x * slot_elems;
                const int orow = it.tile * kBM + o;
                const float wsc = (W4 && orow < M.d_out) ? __ldg(M.w_scale + orow) : 1.f;
                for (int c0 = 0; c0 < ncols16; c0 += 16) {
                    uint32_t r[16];
                    tmem_ld16(tacc + (uint32_t)c0, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (c0 + i < p.n) __stcg(piece + (size_t)(c0 + i) * kBM + o, __uint_as_float(r[i]) * wsc);
                }
            } else {
                // shrink piece: lane o is slot row 128 tile + o; only the columns of the rows whose
                // adapter owns the slot row are kept (this CTA's part of their t values)
                const int a_first = cta_of(it.it0, dsh.a_iters, dsh.a_ctas);
                const int part = (int)blockIdx.x - a_first;
                const size_t pstride = (size_t)p.tp_rows * LORA_MAX_RANK;
                const int g = it.tile * kTileGroups + o / kGroupRows;  // this lane's group
                const bool gok = g < dsh.n_groups[it.m];
                // the projection's pointers, copied out of the parameters before the stores below
                float *const tpart = M.tpart;
                const AGroup *const groups = M.groups;
                // the lane's group and rank row; the groups are in segment order, so the batch rows
                // (sorted positions) of a warp's four groups are one range [wq0, wq1)
                int q0 = 0, q1 = 0, r = 0;
                if (gok) {
                    const AGroup ag = groups[g];
                    q0 = ag.q0;
                    q1 = ag.q1;
                    r = ag.rbase + (o & (kGroupRows - 1));
                    if (r >= ag.rank) q1 = q0;  // a padding row of the group: nothing to keep
                }
                const int wq0 = __shfl_sync(0xffffffffu, q0, 0);
                const int wq1 = (int)__reduce_max_sync(0xffffffffu, (unsigned)q1);
                // this CTA's part: per batch row of the range, one warp-wide TMEM load of its column
                // (four in flight), kept by the lanes whose group owns the row
                for (int qb = wq0; qb < wq1; qb += 4) {
                    uint32_t v[4];
                    int jc[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        jc[u] = perm_s[min(qb + u, wq1 - 1)];
                        v[u] = tmem_ld1(tacc + (uint32_t)jc[u]);
                    }
                    tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        if (qb + u >= q0 && qb + u < q1)
                            tpart[part * pstride + (size_t)jc[u] * LORA_MAX_RANK + r] = __uint_as_float(v[u]);
                }
                // t = s * (the parts added in k order): by the finalize (p.t_fin), else by the tile's
                // last CTA (a counter, no waiting), two rows' parts in flight
                if (!p.t_fin) {
                    const int na = cta_of(it.it0 + M.k_blocks - 1, dsh.a_iters, dsh.a_ctas) - a_first + 1;
                    float *const tfin = M.tfin;
                    const float scale = p.scale;
                    __threadfence();
                    named_bar_sync(1, 128);
                    if (o == 0) s_last = atomicAdd(M.acount + it.tile, 1) == na - 1;
                    named_bar_sync(1, 128);
                    if (s_last) {
                        __threadfence();
                        for (int qb = wq0; qb < wq1; qb += 2) {
                            bool own[2];
                            int jr[2];
                            float sum[2] = {0.f, 0.f};
#pragma unroll
                            for (int u = 0; u < 2; ++u) {
                                own[u] = qb + u >= q0 && qb + u < q1;
                                jr[u] = own[u] ? perm_s[qb + u] : 0;
                            }
                            for (int cp = 0; cp < na; cp += 8) {  // eight parts per row in flight, k order
                                float pt[2][8];
#pragma unroll
                                for (int u = 0; u < 2; ++u)
#pragma unroll
                                    for (int c = 0; c < 8; ++c)
                                        pt[u][c] = own[u] && cp + c < na
                                                       ? __ldcg(tpart + (size_t)(cp + c) * pstride + (size_t)jr[u] * LORA_MAX_RANK + r)
                                                       : 0.f;
#pragma unroll
                                for (int u = 0; u < 2; ++u)
#pragma unroll
                                    for (int c = 0; c < 8; ++c)
                                        if (cp + c < na) sum[u] = (cp + c == 0) ? pt[u][c] : sum[u] + pt[u][c];
                            }
#pragma unroll
                            for (int u = 0; u < 2; ++u)
                                if (own[u]) tfin[(size_t)jr[u] * LORA_MAX_RANK + r] = scale * sum[u];
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_free + buf);
            ++li;
        }
        }
    } else if (W4 && warp >= kConvWarp0) {
        // ---------------------------------------------------------------- int4 converters
        const int ct = threadIdx.x - 32 * kConvWarp0;
        DItem it;
        uint32_t k = 0;
        bool ok = true;
        for (int ph = ph0; ok && ph < ph1; ++ph) {
        if (ph == 1 && !plan_wait()) break;
        DSched sc;
        if (ph == 1) sc.begin_a(p, blockIdx.x, dsh);
        else sc.begin_w(p, blockIdx.x);
        while (ok && sc.next(p, &dsh, it)) {
            for (int kb = it.kb0; kb < it.kb1; ++kb, ++k) {
                const uint32_t s = rslot(k);
                if (!mbar_wait(wfull + s, rround(k) & 1, abort_flag, p.err, wait_ns)) {
                    ok = false;
                    break;
                }
                if (it.a == 0) {
                    uint8_t *sa = smem + (size_t)s * stage_bytes;
                    for (int q = 0; q < kps; ++q)
                        convert_w4_kblock(smem_u32(sa + a_bytes + x_bytes + q * kW4RawBytes), smem_u32(sa + q * sub_a), ct);
                    fence_proxy_async_smem();  // the MMA reads the tile through the async proxy
                }
                mbar_arrive(cfull + s);
            }
        }
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

// Where chunk ch (8 B values) of output row o of a B tile sits in shared memory, in chunks from the
// tile's start, for rows of nch chunks (nch = 1, 2, 4 or 8): the chunks of a row are XOR-rotated so
// that 8 threads reading the same chunk of 8 consecutive rows hit 8 different 16-byte bank groups.
__device__ __forceinline__ int bchunk_slot(int o, int ch, int nch) {
    return o * nch + (ch ^ (((o * nch) >> 3) & (nch - 1)));
}

// The B tiles (output rows o_base .. o_base + tile_rows - 1) of the rows k0 .. k1 - 1 (but those in
// `skip`, whose tile another row stages) into `buf`,
// every thread of the block copying consecutive chunks of each tile (coalesced), one cp.async group.
// Out of line: the finalize is short-lived and starts cold, so its code is kept small.
template <bool I8>
__device__ __noinline__ void fin_stage(const RowInfo *s_ri, const int *s_off, unsigned skip, int k0, int k1, uint8_t *buf,
                                       int o_base, int tile_rows) {
    using BChunk = typename std::conditional<I8, uint2, uint4>::type;
    constexpr int cu = sizeof(BChunk);
#pragma unroll 4
    for (int k = k0; k < k1; ++k) {
        const RowInfo ri = s_ri[k];
        if (ri.rank <= 0 || ((skip >> k) & 1u)) continue;
        const int lg = __ffs(ri.rp >> 3) - 1, nch = 1 << lg;  // chunks per row: 1, 2, 4 or 8
        const BChunk *src = reinterpret_cast<const BChunk *>(ri.B) + ((size_t)o_base << lg);
        const uint32_t dst = smem_u32(buf + s_off[k]);
        const int units = tile_rows << lg;
        for (int u = threadIdx.x; u < units; u += kBM) {
            const uint32_t d = dst + (uint32_t)bchunk_slot(u >> lg, u & (nch - 1), nch) * cu;
            if constexpr (I8) cp_async_8(d, src + u);
            else cp_async_16cg(d, src + u);
        }
    }
    cp_async_commit();
}

// The finalize's copy of the call's A space: where each projection's A tiles start, and how many CTAs
// share it (the gemm's DecShared without the group counts, which the finalize does not keep: the
// bytes count toward five blocks to an SM, see plan_decode_finalize).
struct FinAShared {
    int32_t a_begin[LORA_MAX_MODULES + 1];
    int32_t a_iters, a_ctas;
};

// ONE: every B tile of the block fits one buffer (a single pass); the expand then runs fully unrolled
// over the 16 rows with y in registers.  Otherwise passes through two buffers, y accumulating in
// shared memory (compact code: the kernel is short-lived and starts with a cold instruction cache).
template <bool I8, bool ONE, bool TF>
__global__ void __launch_bounds__(kBM, 5) decode_finalize_kernel(const __grid_constant__ DecodeParams p) {
    using BChunk = typename std::conditional<I8, uint2, uint4>::type;  // 8 elements of B
    // B tile buffers (fin_nbuf of fin_buf bytes), y [16][128] (base, then + expand), t [16][rpmax],
    // the rows' adapters, the pass plan
    extern __shared__ __align__(16) uint8_t fsm[];
    __shared__ FinAShared fds;  // the call's A space (where each A tile's t parts are)
    const int nbuf = p.fin_nbuf, buf_bytes = p.fin_buf, rpmax = p.rpmax;
    float *ys = reinterpret_cast<float *>(fsm + (size_t)nbuf * buf_bytes);
    float *ts = ys + kFinRows * kBM;
    RowInfo *s_ri = reinterpret_cast<RowInfo *>(ts + kFinRows * rpmax);
    int *s_off = reinterpret_cast<int *>(s_ri + kFinRows);  // [16] byte offset of row k's tile
    int *s_pend = s_off + kFinRows;                        // [17] end row of pass i
    int *s_j = s_pend + kFinRows + 1;                      // [16] batch row of row k
    int *s_skip = s_j + kFinRows;                          // rows staged by an earlier row (bit k)
    // the block's rows are the sorted positions c0 .. c0 + 15 (rows of one adapter are adjacent);
    // row blocks in the prep's order, heaviest first
    const int tid = threadIdx.x, tile = blockIdx.x;
    const int c0 = (p.rb_order != nullptr ? __ldcg(p.rb_order + blockIdx.y) : (int)blockIdx.y) * kFinRows;
    int m = 0;
    while (m + 1 < p.n_mod && p.mod[m + 1].w_tile_begin <= tile) ++m;
    // the projection's fields, copied out of the parameters once: a runtime-indexed parameter is
    // read through a generic pointer, which the compiler must reload after every store
    const DecodeModule &Mp = p.mod[m];
    const int w_tile_begin = Mp.w_tile_begin, k_blocks = Mp.k_blocks, d_out = Mp.d_out;
    const int w_iter_begin = Mp.w_iter_begin, m_tiles = Mp.m_tiles;
    const RowInfo *const rowinfo = Mp.rowinfo;
    const float *const tpart = Mp.tpart;
    const float *const tfin = Mp.tfin;
    constexpr bool t_fin = TF;  // the call's p.t_fin
    const size_t pstride = (size_t)p.tp_rows * LORA_MAX_RANK;
    const float scale = p.scale;
    const float *const Tm = Mp.T;
    void *const yv_base = Mp.y;
    const float *const home = p.home, *const ctaw = p.ctaw;
    const int n = p.n, nt = p.nt, shrink_tc = p.shrink_tc, y_bf16 = p.y_bf16;
    const int lt = tile - w_tile_begin;
    if (lt >= m_tiles || c0 >= n) {
        grid_dep_wait();
        return;
    }
    const int nrows = min(kFinRows, n - c0);
    const int o_base = lt * kBM;
    const bool o_ok = o_base + tid < d_out;
    const int tile_rows = min(kBM, d_out - o_base);
    // ---- before the gemm has finished: the rows' adapters (the row plan is complete: the gemm
    // launched this grid only after its own wait), the pass plan, and the first passes' B tiles.
    // Warp 0 plans in registers: lane k holds row k; passes are taken greedily in row order, and a
    // row with the adapter of the row before it reads that row's tile.
    if (tid < 32) {
        // lane m: the group count of the call's projection m (the A space), in flight with the rows'
        const int gm = (TF && shrink_tc && tid < p.n_mod) ? __ldcg(p.mod[tid].n_groups) : 0;
        RowInfo ri{nullptr, 0, 0, 0};
        int j = 0;
        if (tid < nrows) {
            j = __ldcg(p.perm + c0 + tid);
            const uint4 raw = __ldcg(reinterpret_cast<const uint4 *>(rowinfo + j));
            ri = *reinterpret_cast<const RowInfo *>(&raw);
        }
        const bool has = tid < nrows && ri.rank > 0;
        const int bytes = has ? kBM * (ri.rp >> 3) * (int)sizeof(BChunk) : 0;
        const unsigned long long bp = has ? reinterpret_cast<unsigned long long>(ri.B) : 0ull;
        const unsigned long long bprev = __shfl_up_sync(0xffffffffu, bp, 1);
        const bool same = has && tid > 0 && bprev == bp;  // the previous row's adapter
        const unsigned same_mask = __ballot_sync(0xffffffffu, same);
        int used = 0, np = 0, off = 0, last = 0;
        for (int k = 0; k < nrows; ++k) {
            const int b = __shfl_sync(0xffffffffu, bytes, k);
            if ((same_mask >> k) & 1u) {  // same pass as row k - 1: its tile
                if (tid == k) off = last;
                continue;
            }
            if (k > 0 && used + b > buf_bytes) {  // row k opens pass np + 1
                if (tid == 0) s_pend[np] = k;
                ++np;
                used = 0;
            }
            if (tid == k) off = used;
            last = used;
            used += b;
        }
        if (tid == 0) s_pend[np] = nrows;
        if (shrink_tc && t_fin) {
            // the call's A space as the gemm lays it out: projection m's tiles of 16 groups, each
            // k_blocks k-steps long, projections in order (lanes m < n_mod, a warp scan)
            const int kbm = tid < p.n_mod ? p.mod[tid].k_blocks : 0;
            const int at = (min(max(gm, 0), kDecMaxGroups) + kTileGroups - 1) / kTileGroups;
            const int am = at * kbm;
            int incl = am;
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += y;
            }
            const int total = __shfl_sync(0xffffffffu, incl, 31);
            const int kmax = (int)__reduce_max_sync(0xffffffffu, (unsigned)(at > 0 ? kbm : 0));
            if (tid < p.n_mod) fds.a_begin[tid] = incl - am;
            if (tid == 0) {
                fds.a_begin[p.n_mod] = total;
                fds.a_iters = total;
                fds.a_ctas = decode_a_ctas(total, kmax, p.n_cta);
            }
        }
        if (tid > np && tid <= kFinRows) s_pend[tid] = -1;
        if (tid < kFinRows) {
            s_ri[tid] = ri;
            s_off[tid] = off;
            s_j[tid] = j;
        }
        if (tid == 0) *s_skip = (int)same_mask;  // rows whose tile an earlier row stages
    }
    __syncthreads();
    int n_pass = 0;
    while (n_pass < kFinRows && s_pend[n_pass] >= 0) ++n_pass;
    const unsigned skip = (unsigned)*s_skip;
    for (int i = 0; i < min(nbuf, n_pass); ++i)
        fin_stage<I8>(s_ri, s_off, skip, i == 0 ? 0 : s_pend[i - 1], s_pend[i], fsm + (size_t)i * buf_bytes, o_base, tile_rows);
    // Where the gemm's outputs for this block are (not the outputs themselves), still before the
    // wait: the blocks start as the gemm's CTAs leave their SMs and wait there for the whole gemm,
    // so what they issue after the wait is the tail of the call.
    // base: the tile's stream-K pieces, the home slot and then CTAs c_first + 1 .. c_first + np - 1
    const size_t slot_elems = (size_t)kBM * nt;
    const int it0 = w_iter_begin + lt * k_blocks;
    const int c_first = cta_of(it0, p.w_iters, p.n_cta);
    const int np = cta_of(it0 + k_blocks - 1, p.w_iters, p.n_cta) - c_first + 1;
    const float *const q = home + (size_t)(w_tile_begin + lt) * slot_elems + tid;
    const float *const q1 = ctaw + (size_t)(c_first + 1) * slot_elems + tid;
    // t is [16 rows][rpmax / 4] float4 values; with fewer values than threads, tpv threads share one
    // value's A-tile parts (each adds every tpv-th part in k order, then the partial sums are added
    // in a fixed order), and both of a thread's values take their parts in one loop, so that the
    // parts' loads are in flight together.  A one-pass bf16 block has rank-8 rows only (16 tiles fill
    // its 32 KiB), so 32 values: one per thread at most.
    constexpr int kVals = (ONE && !I8) ? 1 : 2;
    const int lq = __ffs(rpmax >> 2) - 1;  // log2(rpmax / 4)
    const int nv = kFinRows << lq;
    const int tpv = TF && nv < kBM ? kBM / nv : 1, vpt = !TF ? 2 : nv > kBM ? nv / kBM : 1;
    const int sub = tid & (tpv - 1);
    // value i: its first t part (TF: parts pstride apart) or its t, and how many (0: none)
    const float *tp[2] = {tpart, tpart};
    int na[2] = {0, 0};
#pragma unroll
    for (int i = 0; i < kVals; ++i) {
        const int e = tid / tpv + i * (kBM / tpv), jj = e >> lq, r = (e & ((1 << lq) - 1)) * 4;
        if (i < vpt && jj < kFinRows && r < s_ri[jj].rank) {
            const int j = s_j[jj];
            if (shrink_tc && !t_fin) {
                if (sub == 0) {
                    tp[i] = tfin + (size_t)j * LORA_MAX_RANK + r;
                    na[i] = 1;
                }
            } else if (shrink_tc) {
                // t = s * (the A tile's parts): the tile of the group holding rank rows r .. r + 3
                // of the row's adapter, and the CTAs that shared it
                const int at = (s_ri[jj].g0 + r / kGroupRows) / kTileGroups;
                const int ia = fds.a_begin[m] + at * k_blocks;
                const int cf = cta_of(ia, fds.a_iters, fds.a_ctas);
                na[i] = cta_of(ia + k_blocks - 1, fds.a_iters, fds.a_ctas) - cf + 1;
                tp[i] = tpart + (size_t)j * LORA_MAX_RANK + r;
            } else if (sub == 0) {
                tp[i] = Tm + (size_t)j * rpmax + r;
                na[i] = 1;
            }
        }
    }
    grid_dep_wait();
    grid_dep_launch();
    // the gemm is complete: its A-tile counters start the next call at zero (even after a call
    // that gave up a wait)
    if (blockIdx.x == 0 && blockIdx.y == 0 && shrink_tc && !t_fin)
        for (int mm = 0; mm < p.n_mod; ++mm)
            for (int i = tid; i < kDecMaxGroups / kTileGroups; i += kBM) p.mod[mm].acount[i] = 0;
    // ---- after: the tile's base pieces and t (zero past each row's rank), the pieces' loads issued
    // first so that they are in flight while t's are.
    // base: the block's rows of every piece, added in k order; row k's values at s_j[k] * 128 + tid
    // (rows past n read row 0, unused); the first two pieces (most tiles have at most two) loaded here
    float v[kFinRows], f[kFinRows];
#pragma unroll
    for (int k = 0; k < kFinRows; ++k) {
        const int jo = s_j[k] * kBM;
        v[k] = __ldcg(q + jo);
        f[k] = np > 1 ? __ldcg(q1 + jo) : 0.f;
    }
    float4 tv[2];
    {
        float4 acc[2] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
        if constexpr (TF) {
            const int nmax = kVals > 1 ? max(na[0], na[1]) : na[0];
            for (int pc = sub; pc < nmax; pc += 4 * tpv) {  // four parts of each value in flight
                float4 pt[2][4];
#pragma unroll
                for (int i = 0; i < kVals; ++i)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        pt[i][c] = pc + c * tpv < na[i]
                                       ? __ldcg(reinterpret_cast<const float4 *>(tp[i] + (size_t)(pc + c * tpv) * pstride))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int i = 0; i < kVals; ++i)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        acc[i].x += pt[i][c].x;
                        acc[i].y += pt[i][c].y;
                        acc[i].z += pt[i][c].z;
                        acc[i].w += pt[i][c].w;
                    }
            }
        } else {
#pragma unroll
            for (int i = 0; i < kVals; ++i)
                if (na[i] > 0) acc[i] = __ldcg(reinterpret_cast<const float4 *>(tp[i]));
        }
#pragma unroll
        for (int i = 0; i < kVals; ++i) {
            // the value's partial sums, lanes sub = 0 .. tpv - 1 (every lane takes part)
            for (int off = 1; off < tpv; off <<= 1) {
                acc[i].x += __shfl_down_sync(0xffffffffu, acc[i].x, off);
                acc[i].y += __shfl_down_sync(0xffffffffu, acc[i].y, off);
                acc[i].z += __shfl_down_sync(0xffffffffu, acc[i].z, off);
                acc[i].w += __shfl_down_sync(0xffffffffu, acc[i].w, off);
            }
            tv[i] = shrink_tc && t_fin ? make_float4(scale * acc[i].x, scale * acc[i].y, scale * acc[i].z, scale * acc[i].w)
                                       : acc[i];
        }
    }
    // the pieces after the first two
    if (np > 1)
#pragma unroll
        for (int k = 0; k < kFinRows; ++k) v[k] += f[k];
    for (int pc = 2; pc < np; ++pc) {
        const float *qq = ctaw + (size_t)(c_first + pc) * slot_elems + tid;
#pragma unroll
        for (int k = 0; k < kFinRows; ++k) f[k] = __ldcg(qq + s_j[k] * kBM);
#pragma unroll
        for (int k = 0; k < kFinRows; ++k) v[k] += f[k];
    }
#pragma unroll
    for (int i = 0; i < kVals; ++i) {
        const int e = tid / tpv + i * (kBM / tpv), jj = e >> lq, r = (e & ((1 << lq) - 1)) * 4;
        if (i < vpt && sub == 0 && jj < kFinRows) {
            const int rank = s_ri[jj].rank;
            float4 v = tv[i];
            if (r + 1 >= rank) v.y = 0.f;
            if (r + 2 >= rank) v.z = 0.f;
            if (r + 3 >= rank) v.w = 0.f;
            *reinterpret_cast<float4 *>(ts + jj * rpmax + r) = v;
        }
    }
    if constexpr (ONE) {
        // ---- expand (every index into out[] is a compile-time constant: nothing goes through
        // local memory, which the L1-light carve-out would send to L2)
        cp_async_wait_all();
        __syncthreads();  // the tiles and t visible to every thread
        float out[kFinRows];
#pragma unroll
        for (int k = 0; k < kFinRows; ++k) {
            float d = 0.f;
            const RowInfo ri = s_ri[k];
            if (o_ok && ri.rank > 0) {
                const int nch = I8 ? ri.rp >> 3 : 1;  // 1, or 2 for int8 rank 16 (bf16: rank 8 only)
                const BChunk *bk = reinterpret_cast<const BChunk *>(fsm + s_off[k]);
                const float *tk = ts + k * rpmax;
                d = dot8_b(bk[bchunk_slot(tid, 0, nch)], tk);
                if (nch > 1) d += dot8_b(bk[bchunk_slot(tid, 1, nch)], tk + 8);
            }
            out[k] = v[k] + d;
        }
#pragma unroll
        for (int k = 0; k < kFinRows; ++k) ys[k * kBM + tid] = out[k];
    } else {
#pragma unroll
        for (int k = 0; k < kFinRows; ++k) ys[k * kBM + tid] = v[k];  // y column tid starts as the base
        // ---- expand, pass by pass: each thread adds B_a[o] . t to its own column of y
        for (int i = 0; i < n_pass; ++i) {
            if (i + 1 < n_pass) cp_async_wait_all_but_1();
            else cp_async_wait_all();
            __syncthreads();  // pass i's tiles (and, on the first pass, t) visible to every thread
            const uint8_t *buf = fsm + (size_t)(i % nbuf) * buf_bytes;
            if (o_ok)
                for (int k = i == 0 ? 0 : s_pend[i - 1]; k < s_pend[i]; ++k) {
                    const RowInfo ri = s_ri[k];
                    if (ri.rank <= 0) continue;
                    const int nch = ri.rp >> 3;
                    const BChunk *bk = reinterpret_cast<const BChunk *>(buf + s_off[k]);
                    const float *tk = ts + k * rpmax;
                    float d = 0.f;
                    for (int ch = 0; ch < nch; ++ch) d += dot8_b(bk[bchunk_slot(tid, ch, nch)], tk + 8 * ch);
                    ys[k * kBM + tid] += d;
                }
            if (i + nbuf < n_pass) {
                __syncthreads();  // every thread is done with this buffer
                fin_stage<I8>(s_ri, s_off, skip, s_pend[i + nbuf - 1], s_pend[i + nbuf], fsm + (size_t)(i % nbuf) * buf_bytes,
                              o_base, tile_rows);
            }
        }
    }
    // ---- y: each thread writes 16-byte runs of one row, a warp 512 (fp32) or 256 (bf16)
    // contiguous bytes per store
    __syncthreads();
    if (y_bf16) {
        for (int f = tid; f < nrows * 16; f += kBM) {  // runs of 8 outputs
            const int k = f >> 4, c8 = (f & 15) * 8;
            if (o_base + c8 < d_out) {
                const float *src = ys + k * kBM + c8;
                uint4 w;
                w.x = pack_bf16x2(src[0], src[1]);
                w.y = pack_bf16x2(src[2], src[3]);
                w.z = pack_bf16x2(src[4], src[5]);
                w.w = pack_bf16x2(src[6], src[7]);
                *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(yv_base) + (size_t)s_j[k] * d_out + o_base + c8) = w;
            }
        }
    } else {
        for (int f = tid; f < nrows * 32; f += kBM) {  // runs of 4 outputs
            const int k = f >> 5, c4 = (f & 31) * 4;
            if (o_base + c4 < d_out)
                *reinterpret_cast<float4 *>(static_cast<float *>(yv_base) + (size_t)s_j[k] * d_out + o_base + c4) =
                    *reinterpret_cast<const float4 *>(ys + k * kBM + c4);
        }
    }
}

// ====================================================================== launchers ==========

static size_t decode_stage_bytes(int nt, int kps, bool w4) {
    return (size_t)kps * ((size_t)kBM * kBK * 2 + (size_t)nt * kBK * 2 + (w4 ? kW4RawBytes : 0));
}
static size_t decode_smem_bytes(int nt, int kps, int n_stages, bool w4) {
    return 1024 + decode_stage_bytes(nt, kps, w4) * n_stages + 8 * (3 * (size_t)n_stages + 6) + 16;
}

bool plan_decode_gemm(DecodeParams &dp, size_t *smem_bytes) {
    int cols = 32;
    while (cols < 2 * dp.nt) cols <<= 1;  // two accumulators of nt columns
    dp.tmem_cols = cols;
    const bool w4 = dp.w4 != 0;
    const size_t stage = decode_stage_bytes(dp.nt, dp.kps, w4);
    // at most six k-blocks of stages in flight
    const size_t budget = 227 * 1024 - 2048;  // static shared memory (perm copy, A space)
    int s = (int)std::min<size_t>(6 / dp.kps, (budget - decode_smem_bytes(dp.nt, dp.kps, 0, w4)) / stage);
    dp.n_stages = s;
    *smem_bytes = decode_smem_bytes(dp.nt, dp.kps, s, w4);
    return s >= 2;
}

cudaError_t launch_prep_decode(const PrepParams &p, cudaStream_t s) {
    return launch_pdl(prep_decode_kernel, dim3(1), dim3(256 * kPrepGroups), 0, s, p);
}

cudaError_t launch_decode_gemm(const DecodeParams &p, size_t smem_bytes, cudaStream_t s) {
    static size_t configured[2] = {0, 0};
    const int v = p.w4 ? 1 : 0;
    void (*const kernels[2])(DecodeParams) = {decode_gemm_kernel<false>, decode_gemm_kernel<true>};
    if (smem_bytes > configured[v]) {
        cudaError_t e = cudaFuncSetAttribute(kernels[v], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
        if (e != cudaSuccess) return e;
        configured[v] = smem_bytes;
    }
    return launch_pdl(kernels[v], dim3(p.n_cta), dim3(p.w4 ? kDecThreadsW4 : kDecThreads), smem_bytes, s, p);
}

// The finalize's B buffers: one that holds a block's 16 tiles when they fit 32 KiB (one pass), else
// two of 16 KiB (one rank-64 tile), filled and drained in turn (a pass takes the rows whose tiles
// fit one buffer).  With y and t beside them a block holds at most 45,512 bytes of dynamic shared
// memory.  An SM of this part offers 233,472 bytes to its blocks, each block's share (with the
// 1 KiB the driver keeps per block) rounded up to 128 bytes: five blocks take 5 x 46,592 = 232,960.
// Nine more bytes per block would round each share up by another 128 and leave four blocks to an
// SM (the multi-pass launches of a batch of 256 rows then take a third wave).
constexpr size_t kFinSmemMax = 2 * 16384 + (size_t)kFinRows * kBM * 4 + (size_t)kFinRows * LORA_MAX_RANK * 4 +
                               kFinRows * sizeof(RowInfo) + (3 * kFinRows + 2) * sizeof(int);
static_assert(5 * ((kFinSmemMax + (sizeof(FinAShared) + 15) / 16 * 16 + 1024 + 127) / 128 * 128) <= 233472,
              "five finalize blocks to an SM");
void plan_decode_finalize(DecodeParams &dp, size_t *smem_bytes) {
    const int cu = dp.i8 ? 8 : 16;
    const int tile_max = kBM * std::max(1, dp.rpmax / 8) * cu;
    const int all = kFinRows * tile_max;
    constexpr int kOne = 32 * 1024, kTwo = 16 * 1024;
    dp.fin_nbuf = all <= kOne ? 1 : 2;
    dp.fin_buf = all <= kOne ? all : std::max(kTwo, tile_max);
    *smem_bytes = (size_t)dp.fin_nbuf * dp.fin_buf + kFinRows * kBM * 4 + (size_t)kFinRows * dp.rpmax * 4 +
                  kFinRows * sizeof(RowInfo) + (3 * kFinRows + 2) * sizeof(int);
}

cudaError_t launch_decode_finalize(const DecodeParams &p, size_t smem_bytes, cudaStream_t s) {
    // The finalize's blocks may land beside a gemm's CTAs (which hold most of shared memory), so they
    // ask for the same split of the SM's memory between L1 and shared memory.
    static size_t configured[6] = {0, 0, 0, 0, 0, 0};
    void (*const kernels[6])(DecodeParams) = {
        decode_finalize_kernel<false, false, false>, decode_finalize_kernel<true, false, false>,
        decode_finalize_kernel<false, true, false>,  decode_finalize_kernel<true, true, false>,
        decode_finalize_kernel<false, false, true>,  decode_finalize_kernel<false, true, true>};
    // int8 factors have no A tiles (t comes from the CUDA-core shrink)
    const int v = p.t_fin && !p.i8 ? 4 + (p.fin_nbuf == 1 ? 1 : 0) : (p.i8 ? 1 : 0) + (p.fin_nbuf == 1 ? 2 : 0);
    if (configured[v] == 0) {
        cudaError_t e = cudaFuncSetAttribute(kernels[v], cudaFuncAttributePreferredSharedMemoryCarveout,
                                             cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
    }
    if (smem_bytes > configured[v]) {
        cudaError_t e = cudaFuncSetAttribute(kernels[v], cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
        if (e != cudaSuccess) return e;
        configured[v] = smem_bytes;
    }
    const dim3 grid(p.w_tiles, (p.n + kFinRows - 1) / kFinRows);
    return launch_pdl(kernels[v], grid, dim3(kBM), smem_bytes, s, p);
}

}  // namespace lora
