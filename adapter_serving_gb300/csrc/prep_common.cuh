// prep_common.cuh -- device helpers of the row-grouping (prep) kernels of both paths: the error
// word, segment lookup and the check of a caller's segment table.
#pragma once
#include <cstdint>

#include "lora_internal.h"

namespace lora {

// First error wins: the code and where it was found (row or segment index).
__device__ __forceinline__ void report(int32_t *err, int32_t code, int32_t detail) {
    if (err && atomicCAS(err, 0, code) == 0) err[1] = detail;
}

// Largest s in [0, n_seg) with seg_start[s] <= q (seg_start non-decreasing, seg_start[0] = 0).
__device__ __forceinline__ int seg_of(const int32_t *seg_start, int n_seg, int q) {
    int lo = 0, hi = n_seg - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(seg_start + mid) <= q) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Whether the caller's segment table starts at 0, never decreases and ends at n (whole block).
__device__ __forceinline__ bool segments_valid_block(const PrepParams &p) {
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

}  // namespace lora
