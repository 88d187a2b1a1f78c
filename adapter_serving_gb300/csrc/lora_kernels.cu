// lora_kernels.cu -- the device side of the adapted linear layer y_i = W x_i + s B_a (A_a x_i).
//
//   prep_decode_kernel    row grouping: stable sort of the rows by adapter id, id checks, and
//                         the expand packs (which adapters' B slices share one B stage)
//   prep_segments_kernel  checks a given contiguous segment table (prefill), expand slots per
//                         row chunk
//   shrink_kernel         t_i = s * A_a x_i for every row (CUDA cores; bandwidth-bound), grouped
//   shrink_decode_kernel  rows and decode batches; the decode one also reads int8 factors
//   gemm_kernel           base W x_i on tcgen05 tensor cores into TMEM; the expand s B_a t_i from
//                         B stages in the same TMA ring on CUDA cores into a second TMEM buffer;
//                         both added on the way out
//   finalize_kernel       decode: the stream-K tiles split over CTAs, their pieces added in k order
//
// The forward is the one on "m07 -- Multi-Adapter (LoRA) Serving", section 6 "Deep Dive A:
// Batching Heterogeneous Adapters" (one batched base GEMM shared by the batch, plus a gathered
// per-row adapter product) and "LoRA, quotas and noisy neighbours", section "One weight read,
// many adapters" (rows tagged with their adapter, grouped, one kernel per layer).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <algorithm>
#include <cstdint>
#include <type_traits>
#include <utility>

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

// Row grouping state the prep block keeps in shared memory (decode, n <= 256 rows).
struct PrepShared {
    int id[LORA_MAX_DECODE_ROWS];                          // adapter id of row r (-1 = base only)
    int sorted[LORA_MAX_DECODE_ROWS];                      // adapter id at sorted position q
    int cnt[4][LORA_MAX_DECODE_ROWS];                      // partial position counts
    int seg_of[LORA_MAX_DECODE_ROWS];                      // segment of position q
    int seg_q0[LORA_MAX_DECODE_ROWS + 1];                  // first position of segment s
    int rp[LORA_MAX_MODULES][LORA_MAX_DECODE_ROWS];        // storage rank at position q (0 = none)
    const uint16_t *B[LORA_MAX_MODULES][LORA_MAX_DECODE_ROWS];  // B of the adapter at position q
    int scan[8];
};

// Expand packs of every module (decode).  A slot is one adapter segment's run of at most
// pack_ch positions.  Slots are ordered by storage rank (descending), then segment, then
// position, and laid end to end in rank units: as ranks are powers of two no slot crosses a
// multiple of 64, so pack j (one B stage) is exactly the slots in units [64 j, 64 j + 64).
// A slot at unit offset P keeps its t rows at floats [pack_ch * P, pack_ch * (P + rp)) of the
// module's packed T, so a pack's t rows are one contiguous range too.
// The prep block has kPrepGroups groups of 256 threads; group g builds the packs of modules
// g, g + kPrepGroups, ..., synchronising on its own named barrier.  Everything it needs about
// the segments (first position, rank, B) is already in shared memory.
constexpr int kPrepGroups = 4;

__device__ void build_packs(const PrepParams &p, const PrepShared &sh, int ns) {
    __shared__ uint64_t s_warp_all[kPrepGroups][8];
    __shared__ int s_first_all[kPrepGroups][320];
    __shared__ int s_unit_all[kPrepGroups][LORA_MAX_DECODE_ROWS];
    const int g = threadIdx.x >> 8, tid = threadIdx.x & 255;
    const int bar = 1 + g;
    uint64_t *s_warp = s_warp_all[g];
    int *s_first = s_first_all[g], *s_unit = s_unit_all[g];
    const int ch = p.pack_ch;
    for (int m = g; m < p.n_mod; m += kPrepGroups) {
        int q0 = 0, q1 = 0, rp = 0, nsl = 0, cls = 4;
        const uint16_t *B = nullptr;
        if (tid < ns) {
            q0 = sh.seg_q0[tid];
            q1 = sh.seg_q0[tid + 1];
            rp = sh.rp[m][q0];
            B = sh.B[m][q0];
            if (rp > 0) {
                nsl = (q1 - q0 + ch - 1) / ch;
                cls = rp == 64 ? 0 : rp == 32 ? 1 : rp == 16 ? 2 : 3;
            }
        }
        // slots before this segment's, per rank class, in one scan of four 16-bit counts
        uint64_t tot4;
        const uint64_t ex4 = group_scan256_u64(cls < 4 ? (uint64_t)nsl << (16 * cls) : 0, s_warp, tot4, bar);
        int slots_tot = 0, units_tot = 0, slot_base = 0, unit_base = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int tot = (int)((tot4 >> (16 * c)) & 0xffff);
            if (cls == c) {
                const int ex = (int)((ex4 >> (16 * c)) & 0xffff);
                slot_base = slots_tot + ex;
                unit_base = units_tot + ex * (64 >> c);
            }
            slots_tot += tot;
            units_tot += tot * (64 >> c);
        }
        const int PR = p.pack_ranks;
        const int npk = (units_tot + PR - 1) / PR;
        for (int k = 0; k < nsl; ++k) {
            const int P = unit_base + k * rp;
            if (P % PR == 0) s_first[P / PR] = slot_base + k;
        }
        if (tid < ns) s_unit[tid] = rp > 0 ? unit_base : -1;
        if (tid == 0) s_first[npk] = slots_tot;
        named_bar_sync(bar, 256);
        BPackG *packs = p.packs[m];
        for (int k = 0; k < nsl; ++k) {
            const int P = unit_base + k * rp, j = P / PR;
            const int e = slot_base + k - s_first[j];
            const int r0 = q0 + k * ch;
            BSlotG sl;
            sl.B = B;
            sl.q0 = (uint16_t)r0;
            sl.nrows = (uint8_t)min(ch, q1 - r0);
            sl.rp = (uint8_t)rp;
            sl.off = (uint8_t)(P % PR);
            sl.pad_[0] = sl.pad_[1] = sl.pad_[2] = 0;
            packs[j].slot[e] = sl;
            if (e == 0) {
                packs[j].tbegin = ch * PR * j;
                packs[j].tfloats = ch * min(PR, units_tot - PR * j);
                packs[j].nslots = s_first[j + 1] - s_first[j];
                packs[j].pad_ = 0;
            }
        }
        // where each position's t row goes: one thread per position
        for (int q = tid; q < p.n; q += 256) {
            const int sg = sh.seg_of[q], ub = s_unit[sg], r = sh.rp[m][q];
            const int d = q - sh.seg_q0[sg];
            p.tpos[m][q] = ub >= 0 ? ch * (ub + (d / ch) * r) + (d % ch) * r : -1;
        }
        if (tid == 0) p.n_packs[m] = npk;
        named_bar_sync(bar, 256);  // s_first and s_unit are reused by the group's next module
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
        seg_ok = segments_valid(p);
        if (!seg_ok && tid == 0) report(p.err, LORA_DEVERR_BAD_SEGMENTS, 0);
    }
    // ---- ids, checked; every module's rank and B of the row's adapter (all loads in flight first)
    int id = -1;
    int rp_row[LORA_MAX_MODULES];
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
        int rank[LORA_MAX_MODULES];
#pragma unroll
        for (int m = 0; m < LORA_MAX_MODULES; ++m) {
            rank[m] = 1;
            rp_row[m] = 0;
            B_row[m] = nullptr;
            if (id >= 0 && m < p.n_mod) {
                const PoolEntry *e = p.table[m] + id;
                rank[m] = e->rank;
                rp_row[m] = e->rp;
                B_row[m] = e->B;
            }
        }
        bool ok = true;
#pragma unroll
        for (int m = 0; m < LORA_MAX_MODULES; ++m) ok = ok && rank[m] > 0;
        if (!ok) {
            report(p.err, LORA_DEVERR_NOT_LOADED, where);
            id = -1;
        }
        if (id < 0) {
#pragma unroll
            for (int m = 0; m < LORA_MAX_MODULES; ++m) {
                rp_row[m] = 0;
                B_row[m] = nullptr;
            }
        }
        sh.id[tid] = id;
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
        sh.sorted[pos] = id;
#pragma unroll
        for (int m = 0; m < LORA_MAX_MODULES; ++m) {
            sh.rp[m][pos] = rp_row[m];
            sh.B[m][pos] = B_row[m];
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
    if (tid < n) sh.seg_of[tid] = before + incl - 1;
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
    if (p.packs[0] != nullptr) {
        __syncthreads();  // the segment table is complete
        build_packs(p, sh, ns);
    }
}

// Grouped rows (prefill): validate the table, copy it into the workspace with unusable
// adapters replaced by -1 (base only).  A malformed table becomes one base-only segment.
__global__ void __launch_bounds__(1024) prep_segments_kernel(const PrepParams p) {
    grid_dep_wait();
    grid_dep_launch();
    const bool ok = segments_valid(p);
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

// Four signed bytes as floats, exactly: bias each code to 0..255 (xor 0x80), place it in the low
// mantissa bits of 2^23 (byte permute), subtract 2^23 + 128.  Two full-rate operations per code.
__device__ __forceinline__ float4 i8x4(uint32_t v) {
    const uint32_t u = v ^ 0x80808080u;
    constexpr float kBias = 8388736.0f;  // 2^23 + 128
    return make_float4(__uint_as_float(__byte_perm(u, 0x4B000000u, 0x7650)) - kBias,
                       __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7651)) - kBias,
                       __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7652)) - kBias,
                       __uint_as_float(__byte_perm(u, 0x4B000000u, 0x7653)) - kBias);
}

// 8 int8 codes of A (a.x bytes 0..3, a.y bytes 0..3) against 8 bf16 values of x
__device__ __forceinline__ float dot8_bf16(uint2 a, uint4 b) {
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

__global__ void __launch_bounds__(kShrinkThreads) shrink_kernel(const __grid_constant__ ShrinkParams p) {
    __shared__ __align__(16) uint16_t xs[kShrinkRows * kShrinkKSub];
    __shared__ int s_last;
    grid_dep_wait();
    grid_dep_launch();
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
// I8: A holds int8 codes (8 per 8-byte load) and t_j is scaled by the row's fold scale.
template <bool I8>
__global__ void __launch_bounds__(kShrinkThreads, 3) shrink_decode_kernel(const __grid_constant__ ShrinkParams p) {
    using AChunk = typename std::conditional<I8, uint2, uint4>::type;  // 8 elements of A
    __shared__ int s_last;
    grid_dep_wait();
    grid_dep_launch();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int m = 0;
    while (m + 1 < p.n_mod && p.split_begin[m + 1] <= (int)blockIdx.y) ++m;
    const int kc = blockIdx.y - p.split_begin[m];
    if (kc >= p.ksplit[m]) return;
    // one block per sorted position: rows of a shared adapter spread over blocks (its A is read
    // from L2 after the first), so blocks stay balanced
    const int u = blockIdx.x;
    if (u >= p.n) return;
    const int qlo = u, qhi = u + 1;
    const int a = p.qadapter[u];
    const int d_in = p.d_in[m];
    if (a < 0) return;  // base-only position: no t row (every split of it returns here)
    const PoolEntry *e = p.table[m] + a;
    const int rp_u = e->rp;
    // The split width was chosen for the largest storage rank in the pool (about 128 KiB of A
    // per block); a lower-rank adapter takes proportionally wider splits, so fewer of them
    // (blocks past its count leave at once).  Ranks are powers of two, so widths stay multiples
    // of the 2048-wide step.
    int kcw = p.kc[m];
    for (int r2 = rp_u; r2 < p.rpmax && kcw < d_in; r2 <<= 1) kcw <<= 1;
    const int ks = (d_in + kcw - 1) / kcw;
    if (kc >= ks) return;
    const int kbeg = kc * kcw;
    const int kend = min(d_in, kbeg + kcw);
    const uint16_t *x = p.x[m];
    float *const T = p.T[m];
    const int32_t *const perm = p.perm;
    const int32_t *const tpos = p.tpos[m];
    // where position q's t row starts: its pack slot (expand packs) or its row
    auto t_at = [&](int q) -> float * { return T + (tpos ? (size_t)tpos[q] : (size_t)perm[q] * p.rpmax); };
    float *const partials = p.partials;
    const float scale = p.scale;
    const int ks_max = p.ks_max, n = p.n;
    const int rpmax = p.rpmax;
    int r = 0, rp = 0;
    const uint8_t *A = nullptr;  // bytes: bf16 elements or int8 codes
    const float *fold = nullptr;  // I8: scale of each of the adapter's rows
    {
        r = e->rank;
        rp = e->rp;
        A = reinterpret_cast<const uint8_t *>(e->A);
        if (I8) fold = p.fold[m] + e->row_off;
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
                AChunk av[kShrinkDecCh];
#pragma unroll
                for (int c = 0; c < kShrinkDecCh; ++c) {
                    const int kk = k0 + lane * 8 + 256 * c;
                    const size_t at = ((size_t)j * d_in + kk) * (I8 ? 1 : 2);
                    if (kk < kend) av[c] = __ldg(reinterpret_cast<const AChunk *>(A + at));
                    else av[c] = AChunk{};
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
                            t_at(qb + rr)[j] = (I8 ? scale * fold[j] : scale) * v;
                        else
                            partials[(((size_t)m * ks_max + kc) * n + (qb + rr)) * rpmax + j] = v;
                    }
                }
            }
        }
    }
    if (ks == 1) {
        for (int idx = tid; idx < (qhi - qlo) * (rp - r); idx += kShrinkThreads)
            t_at(qlo + idx / (rp - r))[r + idx % (rp - r)] = 0.f;
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
        t_at(q)[j] = (I8 && j < r ? scale * fold[j] : scale) * v;
    }
    if (tid == 0) p.counters[m * p.max_units + u] = 0;
}

// ============================================================================ gemm ==========
//
// One persistent CTA per SM, four roles: warp 0 is the TMA producer, lane 0 of warp 1 issues
// tcgen05.mma, warps 2-5 are the epilogue (TMEM lane quarter = warp % 4).  A tile is 128 rows
// of W (MMA M) by the rows of the batch or of a row chunk (MMA N).  Decode spreads the flattened
// (tile, W k-block) space evenly over the CTAs (stream-K), grouped rows take whole tiles round
// robin.  A tile's nb B stages (the expand, see BStageHdr) ride along with its k-blocks: pack j
// belongs to k-block floor(j kbn / nb) in the sense that the packs [P(kb), P(kb + 1)),
// P(kb) = floor(kb nb / kbn), follow k-block kb in the stage ring.  So a piece of a tile carries
// the packs in proportion to its k-blocks, and where the pieces split never depends on the
// adapters of the batch.

struct Item {
    int32_t m, w_tile, chunk, kb0, kb1, kbn, nbs, tile;
    int64_t it0;  // flattened index of the tile's first W k-block
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
    // whether next() has another item to give
    __device__ __forceinline__ bool more(const GemmParams &p) const {
        return p.stream_k ? x < e : cta + j * p.n_cta < p.total_tiles;
    }
    // `npk`: B stages per tile of each module (decode, shared memory)
    __device__ bool next(const GemmParams &p, const int32_t *npk, Item &it) {
        if (p.stream_k) {
            if (x >= e) return false;
            int m = 0;
            while (m + 1 < p.n_mod && p.mod[m + 1].iter_begin <= x) ++m;
            const int kbn = p.mod[m].k_blocks;
            const int64_t local = x - p.mod[m].iter_begin;
            const int lt = (int)(local / kbn);
            it.m = m;
            it.kbn = kbn;
            it.nbs = npk[m];
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
        it.nbs = p.chunk_nb ? p.chunk_nb[it.chunk] : 0;
        return true;
    }
};

// Grouped rows (round robin): the j-th tile of CTA `cta`, whole K, its expand slots from the
// per-chunk table.
__device__ bool rr_item(const GemmParams &p, int cta, int j, Item &it) {
    const int t = cta + j * p.n_cta;
    if (t >= p.total_tiles) return false;
    int m = 0;
    while (m + 1 < p.n_mod && p.mod[m + 1].tile_begin <= t) ++m;
    it.m = m;
    it.kbn = p.mod[m].k_blocks;
    it.kb0 = 0;
    it.kb1 = it.kbn;
    it.tile = t;
    it.it0 = 0;
    tile_coords(p, m, t - p.mod[m].tile_begin, it);
    it.nbs = p.chunk_nb ? p.chunk_nb[it.chunk] : 0;
    return true;
}

// Grouped rows: tile j+1's B stages enter the ring after the first kGroupedLead k-blocks of tile
// j, so its expand runs while tile j is multiplied; tile 0's come first.
constexpr int kGroupedLead = 4;

// The item's packs: [P(kb0), P(kb1)) with P(kb) = floor(kb nb / kbn).
__device__ __forceinline__ int pack_of(const Item &it, int kb) { return kb * it.nbs / it.kbn; }
__device__ __forceinline__ int item_b(const Item &it) { return pack_of(it, it.kb1) - pack_of(it, it.kb0); }

// Walks an item's k-blocks without a division per step: after k-block kb the packs
// [P(kb), P(kb + 1)) follow; acc = (kb nb) mod kbn, b = P(kb).
struct Mix {
    int nb, kbn, acc, b;
    __device__ __forceinline__ void begin(const Item &it) {
        nb = it.nbs;
        kbn = it.kbn;
        const int t = it.kb0 * nb;
        b = t / kbn;
        acc = t - b * kbn;
    }
    // number of packs that follow the current k-block (they start at `b` before the call)
    __device__ __forceinline__ int after_w() {
        acc += nb;
        int cnt = 0;
        while (acc >= kbn) {
            acc -= kbn;
            ++cnt;
        }
        return cnt;
    }
};

// Everything the epilogue reads per call, copied out of the kernel parameters once.  Parameters
// reached through a runtime module index are generic loads that the compiler must repeat after
// every store (they might alias); locals never are.
struct EpiCtx {
    const GemmParams *p;
    const int32_t *perm_s;  // decode: sorted position -> row (shared memory copy)
    int decode, n, nt, y_bf16, n_cta, pack_ch;
    int64_t total_iters;
    float *partials;
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
    int d_out;
};
__device__ __forceinline__ ModLocal mod_local(const GemmParams &p, int m) {
    const GemmModule &M = p.mod[m];
    return ModLocal{&M.tmY, M.y, M.d_out};
}

// ---- expand (B stages) ----------------------------------------------------------------
//
// Producer side: one B stage = the B slices (rows o0 .. o0+127 of each slot's adapter, [128][rp]
// bf16, one bulk copy each, at rank offset `off` of the A buffer) and the slots' t rows (one bulk
// copy after the header of the X buffer); the slot header is written with plain stores before
// the arrive that opens the stage.

// decode: pack j of module M, its 16-byte pieces held one per lane (lane 0: header, lane e + 1:
// slot e), already loaded.  Returns the bytes the copies bring.
__device__ __forceinline__ void produce_pack(const uint4 rec, const GemmModule &M, int o0, int orows, int pack_ch,
                                             uint8_t *sa, uint8_t *sx, uint64_t *full_bar, int lane, int esize) {
    const int nslots = __shfl_sync(0xffffffffu, (int)rec.z, 0);
    const int tbegin = __shfl_sync(0xffffffffu, (int)rec.x, 0);
    const int tfloats = __shfl_sync(0xffffffffu, (int)rec.y, 0);
    BStageHdr *hdr = reinterpret_cast<BStageHdr *>(sx);
    const bool mine = lane >= 1 && lane <= nslots;
    const uint8_t *B = reinterpret_cast<const uint8_t *>((uint64_t)rec.x | ((uint64_t)rec.y << 32));
    const int rp = (int)(rec.z >> 24), off = (int)(rec.w & 0xff);
    uint32_t bytes = 0;
    if (mine) {
        BSlotS sl;
        sl.q0 = (int)(rec.z & 0xffff);
        sl.nrows = (int16_t)((rec.z >> 16) & 0xff);
        sl.rp = (int16_t)rp;
        sl.off = (int16_t)off;
        sl.tstride = (int16_t)rp;
        sl.toff = pack_ch * off;
        hdr->slot[lane - 1] = sl;
        bytes = (uint32_t)(orows * rp * esize);
    }
    const bool plain = !mine || (rp == 8 && ((rec.z >> 16) & 0xff) == 1);
    const bool singles8 = __all_sync(0xffffffffu, plain);
    if (lane == 0) {
        hdr->nslots = nslots;
        hdr->singles8 = singles8 ? 1 : 0;
    }
    fence_proxy_async_smem();  // the slot is refilled by TMA later
    const uint32_t total = __reduce_add_sync(0xffffffffu, bytes) + (uint32_t)tfloats * 4;
    __syncwarp();
    if (lane == 0) mbar_arrive_expect_tx(full_bar, total);
    __syncwarp();
    if (mine) bulk_load(sa + off * kBM * esize, B + (size_t)o0 * rp * esize, bytes, full_bar);
    if (lane == 0 && tfloats > 0) bulk_load(sx + kStageHdrBytes, M.T + tbegin, (uint32_t)tfloats * 4, full_bar);
}

// Epilogue side: delta[o, col] = sum_j B_a[o0 + o, j] t_col[j] for every row of every slot of
// the stage, written to the column of the TMEM delta buffer (32x32b.x1: this warp's 32 lanes).
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

// 8 int8 codes of B against 8 fp32 t values (the int8 scales are already folded into t)
__device__ __forceinline__ float dot8_i8_f32(uint2 b, float4 ta, float4 tb) {
    const float4 lo = i8x4(b.x), hi = i8x4(b.y);
    float acc0 = lo.x * ta.x, acc1 = lo.y * ta.y;
    acc0 = fmaf(lo.z, ta.z, acc0);
    acc1 = fmaf(lo.w, ta.w, acc1);
    acc0 = fmaf(hi.x, tb.x, acc0);
    acc1 = fmaf(hi.y, tb.y, acc1);
    acc0 = fmaf(hi.z, tb.z, acc0);
    acc1 = fmaf(hi.w, tb.w, acc1);
    return acc0 + acc1;
}

// One slot of a B stage: this lane's row of the slot's B (NCH 16-byte chunks, storage rank 8 NCH)
// is loaded once, then every position of the slot streams its t row against it.
// I8: a row holds int8 codes, 8 per 8-byte chunk.
template <int NCH, bool I8>
__device__ __forceinline__ void expand_slot(const EpiCtx &c, uint32_t brow, uint32_t tslot, int tstride, int nrows,
                                            int q0, uint32_t tdel, int row0) {
    using BChunk = typename std::conditional<I8, uint2, uint4>::type;
    constexpr uint32_t kChunk = I8 ? 8 : 16;
    // lane o starts at chunk rot = o / (8 / NCH): the eight lanes of a quarter warp then hit eight
    // different 16-byte bank groups of their rows (rows are NCH * 16 bytes apart)
    const int rot = (c.o * NCH / 8) & (NCH - 1);
    BChunk b[NCH];
    const uint32_t mine = brow + (uint32_t)(c.o * NCH) * kChunk;
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
        const uint32_t at = mine + (uint32_t)((ch + rot) & (NCH - 1)) * kChunk;
        if constexpr (I8) b[ch] = lds_u64(at);
        else b[ch] = lds_u128(at);
    }
    for (int r = 0; r < nrows; ++r) {
        const uint32_t trow = tslot + (uint32_t)(r * tstride * 4);
        float acc[NCH];
#pragma unroll
        for (int ch = 0; ch < NCH; ++ch) {
            const uint32_t tc = trow + ((ch + rot) & (NCH - 1)) * 32;
            if constexpr (I8) acc[ch] = dot8_i8_f32(b[ch], lds128(tc), lds128(tc + 16));
            else acc[ch] = dot8_bf16_f32(b[ch], lds128(tc), lds128(tc + 16));
        }
#pragma unroll
        for (int w = 1; w < NCH; w <<= 1)
#pragma unroll
            for (int ch = 0; ch + w < NCH; ch += 2 * w) acc[ch] += acc[ch + w];  // fixed pairwise order
        const int q = q0 + r;  // the same for the whole warp: the guards below are uniform
        if (q < 0 || q >= c.n) continue;
        const int col = c.decode ? c.perm_s[q] : q - row0;
        if (col < 0 || col >= c.nt) continue;
        tmem_st1(tdel + (uint32_t)col, acc[0]);
    }
}

template <bool I8>
__device__ void expand_stage(const EpiCtx &c, const uint8_t *sa, const uint8_t *sx, uint32_t tdel, int row0) {
    constexpr uint32_t kEsize = I8 ? 1 : 2;
    const BStageHdr *hdr = reinterpret_cast<const BStageHdr *>(sx);
    const int nslots = min(hdr->nslots, kPackSlots);
    const uint32_t a_base = smem_u32(sa), t_base = smem_u32(sx) + kStageHdrBytes;
    if (hdr->singles8) {
        // rank-8 slots of one row each (distinct adapters): slot e's B rows sit at rank offset 8 e
        // and its t row at pack_ch * 8 e floats, so all loads go out before any arithmetic and
        // only the column lookup waits on the slot header
        for (int e0 = 0; e0 < nslots; e0 += 4) {
            typename std::conditional<I8, uint2, uint4>::type bv[4];
            float4 ta[4], tb[4];
            int q[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int e = e0 + u;
                q[u] = -1;
                if (e < nslots) {
                    if constexpr (I8) bv[u] = lds_u64(a_base + (uint32_t)e * 1024 + (uint32_t)c.o * 8);
                    else bv[u] = lds_u128(a_base + (uint32_t)e * 2048 + (uint32_t)c.o * 16);
                    ta[u] = lds128(t_base + (uint32_t)(e * c.pack_ch * 32));
                    tb[u] = lds128(t_base + (uint32_t)(e * c.pack_ch * 32) + 16);
                    q[u] = hdr->slot[e].q0;
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (q[u] >= 0 && q[u] < c.n) {  // the same for the whole warp
                    const int col = c.decode ? c.perm_s[q[u]] : q[u] - row0;
                    if (col >= 0 && col < c.nt) {
                        float v;
                        if constexpr (I8) v = dot8_i8_f32(bv[u], ta[u], tb[u]);
                        else v = dot8_bf16_f32(bv[u], ta[u], tb[u]);
                        tmem_st1(tdel + (uint32_t)col, v);
                    }
                }
            }
        }
        return;
    }
    for (int e = 0; e < nslots; ++e) {
        const BSlotS sl = hdr->slot[e];
        const uint32_t brow = a_base + (uint32_t)sl.off * kBM * kEsize;
        const uint32_t tslot = t_base + (uint32_t)sl.toff * 4;
        switch (sl.rp) {
            case 8: expand_slot<1, I8>(c, brow, tslot, sl.tstride, sl.nrows, sl.q0, tdel, row0); break;
            case 16: expand_slot<2, I8>(c, brow, tslot, sl.tstride, sl.nrows, sl.q0, tdel, row0); break;
            case 32: expand_slot<4, I8>(c, brow, tslot, sl.tstride, sl.nrows, sl.q0, tdel, row0); break;
            case 64: expand_slot<8, I8>(c, brow, tslot, sl.tstride, sl.nrows, sl.q0, tdel, row0); break;
            default: break;
        }
    }
}

// This CTA's share of 16 columns of a tile: accumulator (times the W row's scale, 1 for bf16
// weights) and/or expand delta, both TMEM loads in flight before the one wait.
__device__ __forceinline__ void own_cols16(uint32_t tacc, uint32_t tdel, bool with_acc, bool with_delta, int c0,
                                           float wsc, float (&v)[16]) {
    uint32_t r[16], d[16];
    if (with_acc) tmem_ld16(tacc + c0, r);
    if (with_delta) tmem_ld16(tdel + c0, d);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = (with_acc ? __uint_as_float(r[i]) * wsc : 0.f) + (with_delta ? __uint_as_float(d[i]) : 0.f);
}

// Partial tiles (stream-K pieces) are kept in column quads: element (column c, lane o) at
// ((c / 4) * 128 + o) * 4 + c % 4.  A thread's 16 columns are four 16-byte vectors and a warp
// stores or loads 512 contiguous bytes per instruction.
__device__ __forceinline__ float4 *piece_quads(float *piece, int c0, int o) {
    return reinterpret_cast<float4 *>(piece) + (size_t)(c0 >> 2) * kBM + o;
}

// Drain: accumulator (+ expand delta) -> y.  y goes out through shared memory and TMA tensor
// stores of [16 columns][128 lanes] blocks: the blocks of a round are staged together (the round
// is as many blocks as the staging buffer holds), then one barrier and the round's stores back to
// back.
//
// A tile split over several CTAs (stream-K) is not finished here: every CTA writes its piece of
// the tile to its workspace slot with plain vector stores and moves on, and finalize_kernel, the
// next launch, adds the pieces in k order (so the sum never depends on timing).  Finishing in the
// gemm kept the CTAs that held a tile's first k-block waiting for the others and then summing
// alone, 6-8 us after everyone else was done.
struct DrainBufs {
    uint8_t *ybuf;       // y staging (the expand ring, idle during a drain)
    uint32_t ybuf_bytes;
    uint8_t *stage;      // the stage buffers, free once the CTA's last item has been multiplied
    uint32_t stage_bytes;
};


__device__ void drain(EpiCtx &c, const Item &it, int buf, bool with_acc, bool with_delta, bool last, DrainBufs &db) {
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
    // Where y is staged: on the CTA's last item the stage buffers are idle (after any pieces pulled
    // in there); otherwise the kernel's y buffer if it has one.  With neither, plain stores.
    const uint32_t block_bytes = 16u * kBM * esz;
    uint8_t *ys = nullptr;
    int round_blocks = 0;
    auto set_staging = [&](uint32_t used) {
        if (last && used < db.stage_bytes) {
            ys = db.stage + used;
            round_blocks = (int)((db.stage_bytes - used) / block_bytes);
        } else {
            ys = db.ybuf;
            round_blocks = (int)(db.ybuf_bytes / block_bytes);
        }
    };
    const bool o_ok = o0 + c.o < M.d_out;
    // int4 base: the accumulator holds sum_k code[o, k] x[k]; the row's scale makes it W x
    const float wsc = (c.p->w4 && o_ok) ? __ldg(c.p->mod[it.m].w_scale + o0 + c.o) : 1.f;
    // block c0 of y: into its slot of the current round; the round's stores go out when it is full
    auto emit = [&](int c0, const float (&v)[16]) {
        if (round_blocks == 0) {  // plain stores: lane o writes output o0 + o of 16 rows
            if (!o_ok) return;
            const size_t base = (size_t)(row0 + c0) * M.d_out + o0 + c.o;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (c0 + i >= ncols) continue;
                if (!y_bf16) static_cast<float *>(M.y)[base + (size_t)i * M.d_out] = v[i];
                else static_cast<__nv_bfloat16 *>(M.y)[base + (size_t)i * M.d_out] = __float2bfloat16_rn(v[i]);
            }
            return;
        }
        const int slot = (c0 >> 4) % round_blocks;
        if (slot == 0) {  // the previous round's stores must have read the buffer
            if (leader) bulk_wait_read<0>();
            named_bar_sync(1, 128);
        }
        put16(ys + (size_t)slot * block_bytes, v);
        if (slot == round_blocks - 1 || c0 + 16 >= ncols16) {
            fence_proxy_async_smem();
            named_bar_sync(1, 128);
            if (leader) {
                for (int k = 0; k <= slot; ++k)
                    tma_store_2d(M.tmY, ys + (size_t)k * block_bytes, o0, row0 + c0 - 16 * (slot - k));
                bulk_commit();
            }
        }
    };

    if (head && it.kb1 == it.kbn) {
        set_staging(0);
        for (int c0 = 0; c0 < ncols16; c0 += 16) {
            float v[16];
            own_cols16(tacc, tdel, with_acc, with_delta, c0, wsc, v);
            emit(c0, v);
        }
        return;
    }

    // ---- partial tile (stream-K): the piece goes to this CTA's workspace slot (first or later
    // item of the CTA); finalize_kernel adds the pieces of the tile in k order once the grid is done
    const int64_t b_c = (int64_t)blockIdx.x * total_iters / n_cta;
    float *dst = partials + ((size_t)blockIdx.x * 2 + ((b_c >= it.it0) ? 0 : 1)) * slot_elems;
    for (int c0 = 0; c0 < ncols16; c0 += 16) {
        float v[16];
        own_cols16(tacc, tdel, with_acc, with_delta, c0, wsc, v);
        float4 *q = piece_quads(dst, c0, c.o);
#pragma unroll
        for (int k = 0; k < 4; ++k) __stcg(q + k * kBM, make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]));
    }
}

// ---- int4 base weights ------------------------------------------------------------------
//
// W is stored as 4-bit codes, two per byte, with one fp32 scale per output row ("12. Adapter
// Serving and Multi-Tenant Customization", section "Quantization": an INT4 base with BF16
// adapters, dequantised in the kernel, accumulated wide).  tcgen05's f16 kind takes bf16 on both sides, so the converter warps
// turn every W k-block's codes into a bf16 tile of the integers themselves (exact: |code| <= 7)
// between the TMA load and the MMA, and the drain multiplies the accumulator by the row's scale.
//
// Packing: a 32-bit word holds 8 consecutive k elements; nibble s (s = 0..3) of the low half is
// element 2s and nibble s of the high half element 2s + 1, each stored as code + 8 (1..15).
// (0x4300 | u) read as bf16 is 128 + u (u sits in the low mantissa bits), so one mask-or per pair
// and one bf16x2 subtraction of 136 give a pair of codes.  A zero nibble (the TMA fill past d_in)
// reads as -8 and meets x's zero fill there.
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

// One W k-block: the packed codes at `raw` ([128 rows][32 bytes], as TMA lays down the box) into
// the bf16 tile at `dst` ([128 rows][64], 128-byte swizzle: the 16-byte chunk j of row r sits at
// chunk j ^ (r % 8) of the row, as a TMA load with that swizzle would put it).  Thread ct of the
// kConvWarps * 32 converter threads takes 16-byte pieces ct, ct + 64, ...: piece i is half i % 2 of
// row i / 2, i.e. output chunks 4 (i % 2) .. 4 (i % 2) + 3.  A quarter warp reads 128 contiguous
// bytes and writes eight different chunk columns of four rows: no bank conflicts.
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

// I8: the adapters' B factors are int8 codes (their scales are folded into t by the shrink).
// W4: the base weights are int4 codes with row scales (decode only); two more warps convert them.
template <bool I8, bool W4>
__global__ void __launch_bounds__(W4 ? kGemmThreadsW4 : kGemmThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.n_stages;
    // Ring slot and round of fill k without an integer division in the loops (a runtime divide
    // is tens of dependent instructions, and the producer issues one fill per few hundred
    // cycles): k / S = umulhi(k, ceil(2^32 / S)), exact for k < 2^32 / 8 when S <= 8.
    const uint32_t ring_m = 0xFFFFFFFFu / (uint32_t)S + 1u;
    auto rround = [ring_m](uint32_t kk) -> uint32_t { return __umulhi(kk, ring_m); };
    auto rslot = [ring_m, S](uint32_t kk) -> uint32_t { return kk - __umulhi(kk, ring_m) * (uint32_t)S; };
    const int NB = p.n_acc;
    const uint32_t a_bytes = kBM * kBK * 2;
    const uint32_t b_bytes = (uint32_t)p.nt * kBK * 2;
    // W4: the stage also holds the k-block's packed codes after the x tile
    const uint32_t stage_bytes = a_bytes + b_bytes + (W4 ? (uint32_t)kW4RawBytes : 0u);
    const uint32_t w_tx = W4 ? (uint32_t)kW4RawBytes + b_bytes : a_bytes + b_bytes;  // bytes of one W fill
    uint8_t *ybuf = smem + (size_t)S * stage_bytes;  // epilogue y staging (may be empty)
    int32_t *perm_s = reinterpret_cast<int32_t *>(ybuf + p.ybuf_bytes);
    int32_t *npk = perm_s + LORA_MAX_DECODE_ROWS;  // [LORA_MAX_MODULES] packs per tile (decode)
    // A stage slot is filled with either W k-blocks (wfull, consumed by the MMA warp) or a B stage
    // (bfull, consumed by the epilogue).  Each consumer skips the other kind, so each kind has its
    // own barrier and every consumer keeps its own per-slot parity: a parity wait is only sound
    // when the waiter cannot fall two phases behind, which holds per kind but not across kinds.
    uint64_t *wfull = reinterpret_cast<uint64_t *>(npk + LORA_MAX_MODULES);
    uint64_t *bfull = wfull + S;
    uint64_t *empty = bfull + S;
    uint64_t *cfull = empty + S;  // W4: the slot's codes are converted (the MMA waits on this)
    uint64_t *acc_full = cfull + (W4 ? S : 0);
    uint64_t *acc_free = acc_full + 2;
    uint64_t *mma_done = acc_free + 2;
    uint32_t *misc = reinterpret_cast<uint32_t *>(mma_done + 1);  // [0] tmem, [1] abort

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(wfull + s, 1);
            mbar_init(bfull + s, 1);
            mbar_init(empty + s, 1);
            if (W4) mbar_init(cfull + s, kConvWarps * 32);
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
    // everything above overlaps the previous kernel on the stream; from here on its outputs
    // (segments, packs, t) and the inputs written before it are read.  The next kernel is let in
    // only as CTAs exit (no early trigger): launched early, a shrink's blocks would crowd three
    // to an SM onto the first SMs this grid's tail frees instead of spreading over all of them.
    grid_dep_wait();
    if (threadIdx.x == 0)
        for (int m = 0; m < p.n_mod; ++m) npk[m] = (p.stream_k && p.n_packs) ? p.n_packs[p.mod[m].npk_index] : 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = misc[0];
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer (warp)
        const uint64_t pol_w = p.decode ? l2_policy_evict_first() : l2_policy_evict_normal();
        const uint64_t pol_x = l2_policy_evict_last();
        Sched sc;
        sc.begin(p, blockIdx.x);
        Item it;
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
            if (lane == 0) got = mbar_wait(empty + rslot(kk), (rround(kk) & 1) ^ 1, abort_flag, p.err) ? 1 : 0;
            return __shfl_sync(0xffffffffu, got, 0) != 0;
        };
        // one W k-block of item t into stage kk
        auto issue_w = [&](const Item &t, int kb, uint32_t kk) {
            const GemmModule &M = p.mod[t.m];
            const uint32_t sl = rslot(kk);
            note_fill((int)sl, false);
            if (lane == 0) {
                uint8_t *sa = smem + (size_t)sl * stage_bytes;
                mbar_arrive_expect_tx(wfull + sl, w_tx);
                if (W4) tma_load_2d(sa + a_bytes + b_bytes, &M.tmW, wfull + sl, kb * (kBK / 2), t.w_tile * kBM, pol_w);
                else tma_load_2d(sa, &M.tmW, wfull + sl, kb * kBK, t.w_tile * kBM, pol_w);
                tma_load_2d(sa + a_bytes, &M.tmX, wfull + sl, kb * kBK, t.chunk * p.nt, pol_x);
            }
        };
        if (I8 || W4 || p.stream_k) {  // int8 factors, int4 base: decode only
            // ---- decode: stream-K items, packs after their k-blocks
            while (ok && sc.next(p, npk, it)) {
                const GemmModule &M = p.mod[it.m];
                const int o0 = it.w_tile * kBM;
                const int orows = min(kBM, M.d_out - o0);
                const int b1 = pack_of(it, it.kb1);
                Mix mx;
                mx.begin(it);
                // the first pack of the item's B stages, fetched ahead
                uint4 rec = make_uint4(0, 0, 0, 0);
                if (b1 > mx.b && lane <= kPackSlots) rec = __ldcg(reinterpret_cast<const uint4 *>(M.packs + mx.b) + lane);
                for (int kb = it.kb0; kb < it.kb1 && ok; ++kb) {
                    if (!acquire(k)) {
                        ok = false;
                        break;
                    }
                    issue_w(it, kb, k);
                    ++k;
                    const int nb = mx.after_w();
                    for (int q = 0; q < nb; ++q, ++mx.b, ++k) {
                        const int jb = mx.b;
                        if (!acquire(k)) {
                            ok = false;
                            break;
                        }
                        const uint32_t sl = rslot(k);
                        uint8_t *sa = smem + (size_t)sl * stage_bytes;
                        note_fill((int)sl, true);
                        const uint4 cur = rec;
                        if (jb + 1 < b1 && lane <= kPackSlots)
                            rec = __ldcg(reinterpret_cast<const uint4 *>(M.packs + jb + 1) + lane);
                        produce_pack(cur, M, o0, orows, p.pack_ch, sa, sa + a_bytes, bfull + sl, lane, I8 ? 1 : 2);
                    }
                }
            }
        } else if constexpr (!W4) {
            // ---- grouped rows: whole tiles round robin, each tile's slots one per B stage: a
            // segment's rows in the chunk in runs of pf_ch (walked with sg / r)
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
                    hdr->singles8 = 0;
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
                hdr->singles8 = 0;
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
            uint32_t k = 0, li = 0, use0 = 0, use1 = 0, wpar = 0;
            bool ok = true;
            // one W k-block at stage k into accumulator column d
            auto mma_stage = [&](uint32_t d, bool accumulate) -> bool {
                const int s = (int)rslot(k);
                if (!mbar_wait((W4 ? cfull : wfull) + s, (wpar >> s) & 1u, abort_flag, p.err)) return false;
                wpar ^= 1u << s;
                tc_fence_after();
                const uint32_t sa = smem_u32(smem + (size_t)s * stage_bytes);
                const uint64_t da = sdesc_kmajor_sw128(sa);
                const uint64_t db = sdesc_kmajor_sw128(sa + a_bytes);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    umma_bf16(d, da + (uint64_t)(kk * 2), db + (uint64_t)(kk * 2), idesc, (accumulate || kk > 0) ? 1u : 0u);
                umma_commit(empty + s);
                return true;
            };
            if (I8 || W4 || p.stream_k) {  // int8 factors, int4 base: decode only
                Sched sc;
                sc.begin(p, blockIdx.x);
                Item it;
                while (ok && sc.next(p, npk, it)) {
                    const int buf = li % NB;
                    const uint32_t use = buf ? use1 : use0;
                    if (!mbar_wait(acc_free + buf, (use & 1) ^ 1, abort_flag, p.err)) break;
                    tc_fence_after();
                    const uint32_t d = tmem_base + (uint32_t)(buf * p.nt);
                    Mix mx;
                    mx.begin(it);
                    for (int kb = it.kb0; kb < it.kb1; ++kb) {
                        if (!mma_stage(d, kb > it.kb0)) {
                            ok = false;
                            break;
                        }
                        k += 1 + (uint32_t)mx.after_w();  // the packs after it go to the epilogue
                    }
                    if (!ok) break;
                    umma_commit(acc_full + buf);
                    if (buf) ++use1; else ++use0;
                    ++li;
                }
            } else if constexpr (!W4) {
                // grouped rows: the epilogue writes each tile's expand into the accumulator first
                // and then arrives on acc_free, so every k-block accumulates on top of it
                Item cur, nxt;
                bool has = rr_item(p, blockIdx.x, 0, cur);
                if (has) k += (uint32_t)cur.nbs;
                for (int jt = 0; has && ok; ++jt) {
                    const bool has_nxt = rr_item(p, blockIdx.x, jt + 1, nxt);
                    const int buf = jt & 1;
                    const uint32_t use = buf ? use1 : use0;
                    if (!mbar_wait(acc_free + buf, use & 1, abort_flag, p.err)) break;
                    tc_fence_after();
                    const uint32_t d = tmem_base + (uint32_t)(buf * p.nt);
                    const int lead = min(kGroupedLead, cur.kbn);
                    for (int kb = 0; kb < cur.kbn; ++kb) {
                        if (kb == lead && has_nxt) k += (uint32_t)nxt.nbs;
                        if (!mma_stage(d, true)) {
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
            }
            umma_commit(mma_done);
            const uint32_t a = smem_u32(mma_done);
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(a, 0) && globaltimer() - t0 < kWaitBudgetNs) {
            }
        }
    } else if (W4 && warp >= 2 + kEpiWarps) {
        // ---------------------------------------------------------------- int4 converters
        // walk the same fills as the MMA warp: every W k-block, skipping the B stages after it
        const int ct = threadIdx.x - (64 + 32 * kEpiWarps);
        Sched sc;
        sc.begin(p, blockIdx.x);
        Item it;
        uint32_t k = 0, wpar = 0;
        bool ok = true;
        while (ok && sc.next(p, npk, it)) {
            Mix mx;
            mx.begin(it);
            for (int kb = it.kb0; kb < it.kb1; ++kb) {
                const int s = (int)rslot(k);
                if (!mbar_wait(wfull + s, (wpar >> s) & 1u, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                wpar ^= 1u << s;
                uint8_t *sa = smem + (size_t)s * stage_bytes;
                convert_w4_kblock(smem_u32(sa + a_bytes + b_bytes), smem_u32(sa), ct);
                fence_proxy_async_smem();  // the MMA reads the tile through the async proxy
                mbar_arrive(cfull + s);
                k += 1 + (uint32_t)mx.after_w();
            }
        }
    } else {
        // ---------------------------------------------------------------- epilogue
        EpiCtx c;
        c.p = &p;
        c.perm_s = perm_s;
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
        c.pack_ch = p.pack_ch;
        c.total_iters = p.total_iters;
        c.partials = p.partials;
        if (p.decode)
            for (int q = c.etid; q < p.n; q += 128) perm_s[q] = p.perm[q];
        named_bar_sync(1, 128);
        DrainBufs db;
        db.ybuf = ybuf;
        db.ybuf_bytes = (uint32_t)p.ybuf_bytes;
        db.stage = smem;
        db.stage_bytes = (uint32_t)S * stage_bytes;
        const uint32_t lane_off = (uint32_t)c.lane_base << 16;
        uint32_t bpar = 0;
        // wait for the B stage at ring slot kk (all 128 threads); false if the wait gave up
        auto wait_b = [&](uint32_t kk) -> bool {
            const int s = (int)rslot(kk);
            const bool ok = !named_bar_or(1, 128, !mbar_wait(bfull + s, (bpar >> s) & 1u, abort_flag, p.err));
            if (ok) bpar ^= 1u << s;
            return ok;
        };
        float z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0.f;
        if (I8 || W4 || p.stream_k) {  // int8 factors, int4 base: decode only
            Sched sc;
            sc.begin(p, blockIdx.x);
            Item cur;
            bool has_cur = sc.next(p, npk, cur);
            uint32_t k = 0, li = 0, use0 = 0, use1 = 0;
            while (has_cur) {
                const int buf = li % NB;
                const bool last = !sc.more(p);
                const int nbs = item_b(cur);
                bool ok = true;
                if (nbs > 0) {
                    // expand: zero this item's delta columns, then every B stage adds its slots' rows
                    const uint32_t tdel = tmem_base + lane_off + c.delta_col + (uint32_t)(buf * p.nt);
                    const int row0 = cur.chunk * p.nt;
                    const int ncols = p.decode ? p.n : min(p.nt, p.n - row0);
                    float z[16];
    #pragma unroll
                    for (int i = 0; i < 16; ++i) z[i] = 0.f;
                    for (int c0 = 0; c0 < ncols; c0 += 16) tmem_st16(tdel + (uint32_t)c0, z);
                    tmem_st_wait();
                    Mix mx;
                    mx.begin(cur);
                    for (int kb = cur.kb0; kb < cur.kb1 && ok; ++kb) {
                        ++k;  // the W k-block goes to the MMA warp
                        const int nb = mx.after_w();
                        for (int q = 0; q < nb; ++q, ++k) {
                            const int s = (int)rslot(k);
                            ok = wait_b(k);
                            if (!ok) break;
                            const uint8_t *sa = smem + (size_t)s * stage_bytes;
                            expand_stage<I8>(c, sa, sa + a_bytes, tdel, row0);
                            named_bar_sync(1, 128);  // every warp is done with the stage
                            if (c.etid == 0) mbar_arrive(empty + s);
                        }
                    }
                    tmem_st_wait();
                } else {
                    k += (uint32_t)(cur.kb1 - cur.kb0);
                }
                if (!ok) break;
                const uint32_t use = buf ? use1 : use0;
                ok = mbar_wait(acc_full + buf, use & 1, abort_flag, p.err);
                if (named_bar_or(1, 128, !ok)) break;
                tc_fence_after();
                drain(c, cur, buf, true, nbs > 0, last, db);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_free + buf);
                if (buf) ++use1; else ++use0;
                has_cur = sc.next(p, npk, cur);
                ++li;
            }
        } else if constexpr (!W4) {
            // ---- grouped rows: the expand of tile j+1 is written into its accumulator (zeros +
            // delta) while tile j is multiplied, then acc_free tells the MMA warp to start on it.
            // A B stage is copied into the y buffer first, so its ring slot is given back at once.
            uint32_t use0 = 0, use1 = 0;
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
                    expand_stage<I8>(c, ybuf, ybuf + bbytes, tacc, row0);
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
                ok = mbar_wait(acc_full + buf, use & 1, abort_flag, p.err);
                if (named_bar_or(1, 128, !ok)) break;
                tc_fence_after();
                drain(c, cur, buf, true, false, !has_nxt, db);
                tc_fence_before();
                __syncwarp();
                if (buf) ++use1; else ++use0;
                kw += (uint32_t)cur.kbn + (has_nxt ? (uint32_t)nxt.nbs : 0u);
                cur = nxt;
                has = has_nxt;
            }
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

// Stream-K finish: block (tile, 16-column block) of every tile whose k range was split over
// CTAs adds the CTAs' pieces in k order and writes those 16 columns of y (lane o of the block =
// output row o0 + o: plain stores, 128 contiguous bytes per warp and column).  Tiles done by one
// CTA were written by the gemm itself.  The CTAs of a split tile are found from the same
// flattened (tile, k-block) split as the gemm's.
__global__ void __launch_bounds__(kBM) finalize_kernel(const __grid_constant__ GemmParams p) {
    grid_dep_wait();
    grid_dep_launch();
    const int tile = blockIdx.x, c0 = blockIdx.y * 16, o = threadIdx.x;
    int m = 0;
    while (m + 1 < p.n_mod && p.mod[m + 1].tile_begin <= tile) ++m;
    const GemmModule &M = p.mod[m];
    const int lt = tile - M.tile_begin;
    if (lt >= M.m_tiles || c0 >= p.n) return;
    const int64_t it0 = M.iter_begin + (int64_t)lt * M.k_blocks;
    const int c_first = (int)(((it0 + 1) * p.n_cta - 1) / p.total_iters);
    const int c_last = (int)(((it0 + M.k_blocks) * p.n_cta - 1) / p.total_iters);
    if (c_first == c_last) return;  // one CTA held the whole tile
    const size_t slot_elems = (size_t)kBM * p.nt;
    auto quads = [&](int cta) {  // this thread's four column quads of CTA cta's piece
        const int64_t b_c = (int64_t)cta * p.total_iters / p.n_cta;
        const float *piece = p.partials + ((size_t)cta * 2 + ((b_c >= it0) ? 0 : 1)) * slot_elems;
        return reinterpret_cast<const float4 *>(piece) + (size_t)(c0 >> 2) * kBM + o;
    };
    // pieces in groups of up to three, every load of a group in flight before the adds (in k order)
    float v[16];
    for (int g0 = c_first; g0 <= c_last; g0 += 3) {
        const int ng = min(3, c_last - g0 + 1);
        float4 f[3][4];
#pragma unroll
        for (int j = 0; j < 3; ++j)
            if (j < ng) {
                const float4 *q = quads(g0 + j);
#pragma unroll
                for (int k = 0; k < 4; ++k) f[j][k] = __ldcg(q + k * kBM);
            }
#pragma unroll
        for (int j = 0; j < 3; ++j)
            if (j < ng) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float a[4] = {f[j][k].x, f[j][k].y, f[j][k].z, f[j][k].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[4 * k + e] = (g0 + j == c_first) ? a[e] : v[4 * k + e] + a[e];
                }
            }
    }
    const int orow = lt * kBM + o;  // decode: one row chunk, W tile = local tile index
    if (orow >= M.d_out) return;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        if (c0 + i >= p.n) break;
        const size_t at = (size_t)(c0 + i) * M.d_out + orow;
        if (p.y_bf16) static_cast<__nv_bfloat16 *>(M.y)[at] = __float2bfloat16_rn(v[i]);
        else static_cast<float *>(M.y)[at] = v[i];
    }
}

// ====================================================================== launchers ==========

size_t gemm_smem_bytes(int nt, int n_stages, int ybuf_bytes, bool w4) {
    const size_t stage = (size_t)kBM * kBK * 2 + (size_t)nt * kBK * 2 + (w4 ? kW4RawBytes : 0);
    return 1024 + stage * n_stages + (size_t)ybuf_bytes + 4 * LORA_MAX_DECODE_ROWS + 4 * LORA_MAX_MODULES +
           8 * ((w4 ? 4 : 3) * (size_t)n_stages + 5) + 16;
}

bool plan_gemm(GemmParams &gp, size_t *smem_bytes) {
    // TMEM.  Decode: n_acc accumulator buffers of nt columns, then one expand-delta buffer per
    // accumulator.  Grouped rows: two accumulators and no delta buffer (the expand is written into
    // the accumulator before the tile's MMAs).
    gp.n_acc = (!gp.stream_k || 4 * gp.nt <= 512) ? 2 : 1;
    const int cols = gp.stream_k ? 2 * gp.n_acc * gp.nt : gp.n_acc * gp.nt;
    gp.tmem_cols = 32;
    while (gp.tmem_cols < cols) gp.tmem_cols <<= 1;
    // y staging: decode drains stage y in the idle stage buffers (the finishing CTA's last item)
    // or store it plainly, which buys one more stage; grouped rows drain every tile while the next
    // one streams, so they keep a dedicated buffer
    gp.ybuf_bytes = gp.stream_k ? 0 : kYBufBytes;
    const bool w4 = gp.w4 != 0;
    const size_t stage = (size_t)kBM * kBK * 2 + (size_t)gp.nt * kBK * 2 + (w4 ? kW4RawBytes : 0);
    const size_t fixed = gemm_smem_bytes(gp.nt, 0, gp.ybuf_bytes, w4);
    gp.n_stages = (int)std::min<size_t>(kMaxStages, (227 * 1024 - fixed - (w4 ? 32 : 24) * kMaxStages) / stage);
    *smem_bytes = gemm_smem_bytes(gp.nt, gp.n_stages, gp.ybuf_bytes, w4);
    return gp.n_stages >= 2;
}

// Every hot-path kernel is launched as a programmatic dependent of the one before it on the
// stream: it may start (and run its prologue) while that one drains, and waits for it with
// griddepcontrol.wait before reading anything.
template <class... KArgs, class... Args>
static cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

cudaError_t launch_prep_decode(const PrepParams &p, cudaStream_t s) {
    return launch_pdl(prep_decode_kernel, dim3(1), dim3(256 * kPrepGroups), 0, s, p);
}

cudaError_t launch_prep_segments(const PrepParams &p, cudaStream_t s) {
    return launch_pdl(prep_segments_kernel, dim3(1), dim3(1024), 0, s, p);
}

cudaError_t launch_shrink(const ShrinkParams &p, int grid_x, int grid_y, cudaStream_t s) {
    if (p.by_segment && p.i8)
        return launch_pdl(shrink_decode_kernel<true>, dim3(grid_x, grid_y), dim3(kShrinkThreads), 0, s, p);
    if (p.by_segment) return launch_pdl(shrink_decode_kernel<false>, dim3(grid_x, grid_y), dim3(kShrinkThreads), 0, s, p);
    return launch_pdl(shrink_kernel, dim3(grid_x, grid_y), dim3(kShrinkThreads), 0, s, p);
}

cudaError_t launch_gemm(const GemmParams &p, size_t smem_bytes, cudaStream_t s) {
    static size_t configured[4] = {0, 0, 0, 0};
    const int v = (p.i8 ? 1 : 0) + (p.w4 ? 2 : 0);
    void (*const kernels[4])(GemmParams) = {gemm_kernel<false, false>, gemm_kernel<true, false>,
                                            gemm_kernel<false, true>, gemm_kernel<true, true>};
    auto kernel = kernels[v];
    if (smem_bytes > configured[v]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
        if (e != cudaSuccess) return e;
        configured[v] = smem_bytes;
    }
    return launch_pdl(kernel, dim3(p.n_cta), dim3(p.w4 ? kGemmThreadsW4 : kGemmThreads), smem_bytes, s, p);
}

cudaError_t launch_finalize(const GemmParams &p, cudaStream_t s) {
    return launch_pdl(finalize_kernel, dim3(p.total_tiles, (p.n + 15) / 16), dim3(kBM), 0, s, p);
}

cudaError_t launch_table_write(PoolEntry *dst, PoolEntry value, cudaStream_t s) {
    table_write_kernel<<<1, 1, 0, s>>>(dst, value);
    return cudaGetLastError();
}

}  // namespace lora
