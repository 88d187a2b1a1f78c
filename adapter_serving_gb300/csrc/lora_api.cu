// lora_api.cu -- host side of the C ABI declared in include/lora_gb300.h: the paged adapter
// pool (64-row pages per projection, carved into power-of-two runs of rank-vectors by a
// buddy allocator), the device-side (pointer, rank) table, the workspace, and the forward
// entry points that queue the prep / shrink / tcgen05 kernels.
//
// Paging follows "LoRA, quotas and noisy neighbours", section "Adapter weights and KV in one
// pool", and "12. Adapter Serving and Multi-Tenant Customization", sections "S-LoRA's unified
// paging" (fixed-size pages, gathered through indirection) and "vLLM's pre-allocated LoRA
// buffers" (capacity fixed at creation: max adapters, max rank).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <set>
#include <string>
#include <unordered_map>
#include <vector>

#include "lora_internal.h"

using namespace lora;

namespace {

thread_local std::string g_last_cuda_error;

int cuda_fail(cudaError_t e, const char *what) {
    g_last_cuda_error = std::string(what) + ": " + cudaGetErrorString(e);
    return LORA_ECUDA;
}

#define LORA_CUDA(call)                                 \
    do {                                                \
        cudaError_t e_ = (call);                        \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
    } while (0)

int storage_rank(int r) {
    int rp = 8;
    while (rp < r) rp <<= 1;
    return rp;
}
int order_of(int rp) { return rp == 8 ? 0 : rp == 16 ? 1 : rp == 32 ? 2 : 3; }

// Buddy allocator over one projection's pages: runs of 8/16/32/64 rows, aligned to their size,
// never crossing a 64-row page.
struct RowAllocator {
    std::set<int64_t> free_[4];
    int64_t free_rows = 0;
    void init(int64_t pages) {
        for (auto &f : free_) f.clear();
        for (int64_t p = 0; p < pages; ++p) free_[3].insert(p * LORA_PAGE_ROWS);
        free_rows = pages * LORA_PAGE_ROWS;
    }
    int64_t alloc(int order) {
        int o = order;
        while (o < 4 && free_[o].empty()) ++o;
        if (o == 4) return -1;
        int64_t off = *free_[o].begin();
        free_[o].erase(free_[o].begin());
        while (o > order) {  // split, keep the lower half
            --o;
            free_[o].insert(off + (int64_t(8) << o));
        }
        free_rows -= int64_t(8) << order;
        return off;
    }
    void release(int64_t off, int order) {
        free_rows += int64_t(8) << order;
        while (order < 3) {
            const int64_t buddy = off ^ (int64_t(8) << order);
            auto it = free_[order].find(buddy);
            if (it == free_[order].end()) break;
            free_[order].erase(it);
            off = std::min(off, buddy);
            ++order;
        }
        free_[order].insert(off);
    }
};

struct ModuleStore {
    int d_in = 0, d_out = 0;
    int64_t pages = 0;
    uint16_t *A = nullptr;  // [pages * 64, d_in] (bf16, or int8 codes in an int8 pool)
    uint16_t *B = nullptr;  // [pages * 64 * d_out] (rank-major runs of [d_out, rp])
    float *fold = nullptr;  // int8 pool: [pages * 64] scale of each stored row (A scale x B scale)
    CUtensorMap tmA[2];     // bf16 pool: the A slab for the decode gemm's A-tile gathers, box {64, 8}
    CUtensorMap tmA128[2];  // the same slab, box {64, 128}: A tiles whose 16 groups are consecutive rows
    bool a_runs = false;    // tmA128 made (the slab has at least 128 rows)
    CUtensorMap tmAb[3];    // the same slab, box {64, 16 / 32 / 64}, one k-block: runs of consecutive groups
    bool a_boxes = false;   // tmAb made
                            // ([0]: one k-block per box; [1]: two, when d_in % 64 == 0)
    RowAllocator rows;
};

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

// bf16 tensor [rows, cols] (row-major), 128-byte swizzle.  kps = 1: 2-D, box {64 cols, box_rows};
// kps = 2 (cols a multiple of 64): the 3-D view {64, rows, cols / 64} (strides: row, 128 bytes), box
// {64, box_rows, 2}: two consecutive k-blocks, each landing as a 2-D box would.
int lora::make_tmap(CUtensorMap *tm, const void *base, int64_t rows, int64_t cols, int box_rows, int kps) {
    auto fn = encode_fn();
    if (!fn) {
        g_last_cuda_error = "cuTensorMapEncodeTiled unavailable";
        return LORA_ECUDA;
    }
    CUresult r;
    cuuint32_t estr[3] = {1, 1, 1};
    if (kps == 1) {
        cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
        cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
        cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
        r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        if (cols % 64 != 0) {
            g_last_cuda_error = "two k-blocks per box need cols % 64 == 0";
            return LORA_EINVAL;
        }
        cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(cols / 64)};
        cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128};
        cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)kps};
        r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) {
        g_last_cuda_error = "cuTensorMapEncodeTiled failed (" + std::to_string((int)r) + ")";
        return LORA_ECUDA;
    }
    return LORA_OK;
}

// Bytes [rows, cols] (row-major; int4 base codes, two per byte), no swizzle: the shared-memory side
// is a dense [box_rows][box_cols] block (kps = 2: two of them, for k-blocks kb and kb + 1, from the
// 3-D view {box_cols, rows, cols / box_cols}).  256-byte L2 promotion, so a 32-byte box row still
// brings whole DRAM bursts into L2.
int lora::make_tmap_u8(CUtensorMap *tm, const void *base, int64_t rows, int64_t cols, int box_cols, int box_rows,
                       int kps) {
    auto fn = encode_fn();
    if (!fn) {
        g_last_cuda_error = "cuTensorMapEncodeTiled unavailable";
        return LORA_ECUDA;
    }
    CUresult r;
    cuuint32_t estr[3] = {1, 1, 1};
    if (kps == 1) {
        cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
        cuuint64_t strides[1] = {(cuuint64_t)cols};
        cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
        r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        if (cols % box_cols != 0) {
            g_last_cuda_error = "two k-blocks per box need cols % box_cols == 0";
            return LORA_EINVAL;
        }
        cuuint64_t dims[3] = {(cuuint64_t)box_cols, (cuuint64_t)rows, (cuuint64_t)(cols / box_cols)};
        cuuint64_t strides[2] = {(cuuint64_t)cols, (cuuint64_t)box_cols};
        cuuint32_t box[3] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows, (cuuint32_t)kps};
        r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) {
        g_last_cuda_error = "cuTensorMapEncodeTiled (int4 codes) failed (" + std::to_string((int)r) + ")";
        return LORA_ECUDA;
    }
    return LORA_OK;
}

// Output y [n, d_out] (row-major, fp32 or bf16), box {128 outputs, 16 rows}, no swizzle: the
// shared-memory side is a dense [16][128] block.  Rows past n and columns past d_out are clipped.
int lora::make_tmap_y(CUtensorMap *tm, void *y, int64_t n, int64_t d_out, bool bf16) {
    auto fn = encode_fn();
    if (!fn) {
        g_last_cuda_error = "cuTensorMapEncodeTiled unavailable";
        return LORA_ECUDA;
    }
    const int esz = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {(cuuint64_t)d_out, (cuuint64_t)(n > 0 ? n : 1)};
    cuuint64_t strides[1] = {(cuuint64_t)d_out * esz};
    cuuint32_t box[2] = {128, 16};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(tm, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, y, dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        g_last_cuda_error = "cuTensorMapEncodeTiled (y) failed (" + std::to_string((int)r) + ")";
        return LORA_ECUDA;
    }
    return LORA_OK;
}

struct lora_pool {
    int device = 0;
    int num_sms = 0;
    int n_modules = 0;
    ModuleStore mod[LORA_MAX_MODULES];
    int max_adapters = 0, max_rank = 0, max_rows = 0;
    bool i8 = false;                  // factors stored as int8 codes + per-row scales
    // a row plan (lora_plan_rows) stays usable while `gen` is unchanged: loads, unloads and
    // forwards that build their own grouping advance it
    uint64_t gen = 1, plan_gen = 0;
    int plan_n = 0;
    PoolEntry *d_table = nullptr;     // [n_modules][max_adapters]
    std::vector<PoolEntry> h_table;
    std::vector<int> rp_count;        // loaded entries per storage-rank order (for rpmax)
    // workspace
    int32_t *perm = nullptr, *seg_start = nullptr, *seg_adapter = nullptr, *n_seg = nullptr, *err = nullptr;
    int32_t *qadapter = nullptr;      // [max_rows] decode: adapter of each sorted position
    int32_t *radapter = nullptr;      // [256] decode: validated adapter of each row
    float *T = nullptr;               // [LORA_MAX_MODULES][max_rows][64] CUDA-core shrink result
    float *shrink_part = nullptr;     // [LORA_MAX_MODULES][ks_cap][256][64]
    int32_t *shrink_cnt = nullptr;    // [LORA_MAX_MODULES][256]
    AGroup *groups = nullptr;         // [LORA_MAX_MODULES][kDecMaxGroups] decode: A gather lists
    int32_t *n_groups = nullptr;      // [LORA_MAX_MODULES]
    RowInfo *rowinfo = nullptr;       // [LORA_MAX_MODULES][256] decode: each row's adapter (B, rank, slot)
    float *tpart = nullptr;           // [LORA_MAX_MODULES][kDecMaxParts][tp_rows][64] t partial sums
    float *home = nullptr;            // [2][w_tiles_cap][128 * nt_cap] decode base pieces from k-block 0
    float *ctaw = nullptr;            // [2][num_sms][128 * nt_cap] decode base pieces from inside a tile
    int call_parity = 0;              // the half of home / ctaw the next decode call writes
    int32_t *rb_order = nullptr;      // [16] the finalize's row blocks, heaviest first (written by the prep)
    float *tfin = nullptr;            // [LORA_MAX_MODULES][tp_rows][64] decode t (summed in the gemm)
    int32_t *acount = nullptr;        // [LORA_MAX_MODULES][kDecMaxGroups / 16] A-tile completion counters
    int tp_rows = 0, nt_cap = 0, w_tiles_cap = 0;
    uint64_t wait_ns = kWaitBudgetNs;  // budget of one in-kernel wait
    int32_t *chunk_seg0 = nullptr;    // [chunk_cap] grouped rows: first segment of each chunk
    int32_t *chunk_nb = nullptr;      // [chunk_cap] grouped rows: expand slots of each chunk
    int chunk_cap = 0;
    int ks_cap = 0;
    // kernel timing: pending event pairs per kernel kind
    bool profiling = false;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> prof_pending[4];
    std::vector<cudaEvent_t> prof_free;
    // lora_layer_step_host: the stream the outputs go down on, and one event per stage
    cudaStream_t d2h = nullptr, h2d = nullptr;
    std::vector<cudaEvent_t> stage_done;
    cudaEvent_t inputs_ready = nullptr, downloads_done = nullptr;
    // per device buffer set (keyed by its ids buffer): the compute that last read its inputs, the
    // downloads that last read its outputs -- the next call on the same set waits for those only
    struct BufSet {
        const void *key = nullptr;
        cudaEvent_t in_free = nullptr, out_free = nullptr;
        bool used = false;
        uint64_t last = 0;
    };
    BufSet bufsets[4];
    uint64_t host_calls = 0;
    int last_n = 0;                   // rows of the most recent forward
    bool last_decode = false;
    std::vector<void *> allocations;

    PoolEntry &entry(int m, int a) { return h_table[(size_t)m * max_adapters + a]; }
    int rpmax() const {
        for (int o = 3; o >= 0; --o)
            if (rp_count[o] > 0) return 8 << o;
        return 8;
    }
};

static int dev_alloc(lora_pool *p, void **ptr, size_t bytes) {
    cudaError_t e = cudaMalloc(ptr, std::max<size_t>(bytes, 256));
    if (e != cudaSuccess) {
        cudaGetLastError();
        g_last_cuda_error = std::string("cudaMalloc: ") + cudaGetErrorString(e);
        return LORA_ENOMEM;
    }
    p->allocations.push_back(*ptr);
    return LORA_OK;
}

void lora::set_last_error(const char *why) { g_last_cuda_error = why; }

extern "C" {

int lora_version(void) { return 10000; }

const char *lora_status_string(int s) {
    switch (s) {
        case LORA_OK: return "ok";
        case LORA_EINVAL: return "invalid argument";
        case LORA_ENOTLOADED: return "adapter not resident";
        case LORA_ENOMEM: return "out of pool pages or device memory";
        case LORA_ECUDA: return "CUDA error";
        case LORA_EUNSUPPORTED: return "unsupported request";
        case LORA_EDEVICE: return "device-side error recorded";
        case LORA_EPINNED: return "pinning guard: no new adapters while the cache is pinned";
        default: return "unknown status";
    }
}

const char *lora_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

int lora_pool_destroy(lora_pool *p) {
    if (!p) return LORA_EINVAL;
    cudaSetDevice(p->device);
    cudaDeviceSynchronize();
    for (void *a : p->allocations) cudaFree(a);
    for (auto &v : p->prof_pending)
        for (auto &e : v) {
            cudaEventDestroy(e.first);
            cudaEventDestroy(e.second);
        }
    for (auto e : p->prof_free) cudaEventDestroy(e);
    for (auto e : p->stage_done) cudaEventDestroy(e);
    for (auto &b : p->bufsets) {
        if (b.in_free) cudaEventDestroy(b.in_free);
        if (b.out_free) cudaEventDestroy(b.out_free);
    }
    if (p->inputs_ready) cudaEventDestroy(p->inputs_ready);
    if (p->downloads_done) cudaEventDestroy(p->downloads_done);
    if (p->d2h) cudaStreamDestroy(p->d2h);
    if (p->h2d) cudaStreamDestroy(p->h2d);
    delete p;
    return LORA_OK;
}

int lora_pool_create(const lora_pool_desc *d, lora_pool **out) {
    if (!d || !out || !d->d_in || !d->d_out) return LORA_EINVAL;
    if (d->n_modules < 1 || d->n_modules > LORA_MAX_MODULES) return LORA_EINVAL;
    if (d->max_adapters < 1 || d->max_rank < 1 || d->max_rank > LORA_MAX_RANK || d->max_rows < 1) return LORA_EINVAL;
    if (d->factor_dtype != LORA_FACTOR_BF16 && d->factor_dtype != LORA_FACTOR_I8) return LORA_EINVAL;
    for (int m = 0; m < d->n_modules; ++m) {
        if (d->d_in[m] < 8 || d->d_out[m] < 8 || d->d_in[m] % 8 || d->d_out[m] % 8) return LORA_EINVAL;
        if (d->pages && d->pages[m] < 0) return LORA_EINVAL;
    }
    *out = nullptr;
    int device = 0, num_sms = 0;
    LORA_CUDA(cudaGetDevice(&device));
    LORA_CUDA(cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, device));
    lora_pool *p = new lora_pool();
    p->device = device;
    p->num_sms = num_sms;
    p->n_modules = d->n_modules;
    p->max_adapters = d->max_adapters;
    p->max_rank = d->max_rank;
    p->max_rows = d->max_rows;
    p->i8 = d->factor_dtype == LORA_FACTOR_I8;
    p->rp_count.assign(4, 0);
    const size_t esize = p->i8 ? 1 : 2;
    const int rp_cap = storage_rank(d->max_rank);
    int rc;
    for (int m = 0; m < p->n_modules; ++m) {
        ModuleStore &s = p->mod[m];
        s.d_in = d->d_in[m];
        s.d_out = d->d_out[m];
        s.pages = d->pages ? d->pages[m]
                           : ((int64_t)d->max_adapters * rp_cap + LORA_PAGE_ROWS - 1) / LORA_PAGE_ROWS;
        const size_t rows = (size_t)s.pages * LORA_PAGE_ROWS;
        if ((rc = dev_alloc(p, (void **)&s.A, rows * s.d_in * esize)) ||
            (rc = dev_alloc(p, (void **)&s.B, rows * s.d_out * esize)) ||
            (p->i8 && (rc = dev_alloc(p, (void **)&s.fold, rows * 4)))) {
            lora_pool_destroy(p);
            return rc;
        }
        s.rows.init(s.pages);
    }
    p->h_table.assign((size_t)p->n_modules * p->max_adapters, PoolEntry{nullptr, nullptr, 0, 0, -1});
    const size_t tbytes = p->h_table.size() * sizeof(PoolEntry);
    if ((rc = dev_alloc(p, (void **)&p->d_table, tbytes))) {
        lora_pool_destroy(p);
        return rc;
    }
    // workspace
    int max_din = 0, max_dout = 0;
    for (int m = 0; m < p->n_modules; ++m) {
        max_din = std::max(max_din, p->mod[m].d_in);
        max_dout = std::max(max_dout, p->mod[m].d_out);
    }
    p->ks_cap = (max_din + 511) / 512;
    const size_t R = (size_t)p->max_rows;
    p->chunk_cap = (int)(R / 256 + 2);  // row chunks of 256 (grouped rows)
    const int dec_rows = std::min(p->max_rows, LORA_MAX_DECODE_ROWS);
    p->tp_rows = dec_rows;
    p->nt_cap = (dec_rows + 15) & ~15;
    p->w_tiles_cap = 0;
    for (int m = 0; m < p->n_modules; ++m) p->w_tiles_cap += (p->mod[m].d_out + kBM - 1) / kBM;
    const size_t piece = (size_t)kBM * p->nt_cap * 4;
    if ((rc = dev_alloc(p, (void **)&p->perm, (R + 1) * 4)) || (rc = dev_alloc(p, (void **)&p->seg_start, (R + 2) * 4)) ||
        (rc = dev_alloc(p, (void **)&p->seg_adapter, (R + 1) * 4)) || (rc = dev_alloc(p, (void **)&p->n_seg, 16)) ||
        (rc = dev_alloc(p, (void **)&p->qadapter, (R + 1) * 4)) ||
        (rc = dev_alloc(p, (void **)&p->radapter, (size_t)LORA_MAX_DECODE_ROWS * 4)) ||
        (rc = dev_alloc(p, (void **)&p->err, 16)) ||
        (rc = dev_alloc(p, (void **)&p->T, (size_t)LORA_MAX_MODULES * R * LORA_MAX_RANK * 4)) ||
        (rc = dev_alloc(p, (void **)&p->shrink_part,
                        (size_t)LORA_MAX_MODULES * p->ks_cap * LORA_MAX_DECODE_ROWS * LORA_MAX_RANK * 4)) ||
        (rc = dev_alloc(p, (void **)&p->shrink_cnt, (size_t)LORA_MAX_MODULES * LORA_MAX_DECODE_ROWS * 4)) ||
        (rc = dev_alloc(p, (void **)&p->groups, sizeof(AGroup) * LORA_MAX_MODULES * kDecMaxGroups)) ||
        (rc = dev_alloc(p, (void **)&p->n_groups, (size_t)4 * LORA_MAX_MODULES)) ||
        (rc = dev_alloc(p, (void **)&p->rowinfo, sizeof(RowInfo) * LORA_MAX_MODULES * LORA_MAX_DECODE_ROWS)) ||
        (rc = dev_alloc(p, (void **)&p->tpart,
                        (size_t)4 * LORA_MAX_MODULES * kDecMaxParts * p->tp_rows * LORA_MAX_RANK)) ||
        (rc = dev_alloc(p, (void **)&p->tfin, (size_t)4 * LORA_MAX_MODULES * p->tp_rows * LORA_MAX_RANK)) ||
        (rc = dev_alloc(p, (void **)&p->rb_order, (size_t)4 * (LORA_MAX_DECODE_ROWS / 16))) ||
        (rc = dev_alloc(p, (void **)&p->acount, (size_t)4 * LORA_MAX_MODULES * (kDecMaxGroups / kTileGroups))) ||
        (rc = dev_alloc(p, (void **)&p->home, 2 * piece * p->w_tiles_cap)) ||
        (rc = dev_alloc(p, (void **)&p->ctaw, 2 * piece * p->num_sms)) ||
        (rc = dev_alloc(p, (void **)&p->chunk_seg0, (size_t)4 * p->chunk_cap)) ||
        (rc = dev_alloc(p, (void **)&p->chunk_nb, (size_t)4 * p->chunk_cap))) {
        lora_pool_destroy(p);
        return rc;
    }
    // the decode gemm gathers A rows of a bf16 pool straight from the slab, 8 rows per box
    for (int m = 0; m < p->n_modules && !p->i8; ++m) {
        ModuleStore &ms = p->mod[m];
        const int64_t rows = (int64_t)ms.pages * LORA_PAGE_ROWS;
        if (ms.pages > 0 && ((rc = make_tmap(&ms.tmA[0], ms.A, rows, ms.d_in, kGroupRows, 1)) ||
                             (ms.d_in % 64 == 0 && (rc = make_tmap(&ms.tmA[1], ms.A, rows, ms.d_in, kGroupRows, 2))))) {
            lora_pool_destroy(p);
            return rc;
        }
        if (rows >= kBM) {
            if ((rc = make_tmap(&ms.tmA128[0], ms.A, rows, ms.d_in, kBM, 1)) ||
                (ms.d_in % 64 == 0 && (rc = make_tmap(&ms.tmA128[1], ms.A, rows, ms.d_in, kBM, 2)))) {
                lora_pool_destroy(p);
                return rc;
            }
            ms.a_runs = true;
        }
        if (ms.pages > 0) {  // at least 64 rows
            for (int j = 0; j < 3; ++j)
                if ((rc = make_tmap(&ms.tmAb[j], ms.A, rows, ms.d_in, kGroupRows << (j + 1), 1))) {
                    lora_pool_destroy(p);
                    return rc;
                }
            ms.a_boxes = true;
        }
    }
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess) e = cudaMemset(p->d_table, 0, tbytes);
    if (e == cudaSuccess) e = cudaMemset(p->err, 0, 16);
    if (e == cudaSuccess) e = cudaMemset(p->n_seg, 0, 16);
    if (e == cudaSuccess) e = cudaMemset(p->acount, 0, (size_t)4 * LORA_MAX_MODULES * (kDecMaxGroups / kTileGroups));
    if (e == cudaSuccess) e = cudaMemset(p->shrink_cnt, 0, (size_t)LORA_MAX_MODULES * LORA_MAX_DECODE_ROWS * 4);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        lora_pool_destroy(p);
        return cuda_fail(e, "pool init");
    }
    *out = p;
    return LORA_OK;
}

int lora_pool_query(const lora_pool *p, int32_t a, int32_t m, int32_t *rank, int64_t *row_off) {
    if (!p || m < 0 || m >= p->n_modules || a < 0 || a >= p->max_adapters) return LORA_EINVAL;
    const PoolEntry &e = p->h_table[(size_t)m * p->max_adapters + a];
    if (rank) *rank = e.rank;
    if (row_off) *row_off = e.rank > 0 ? e.row_off : -1;
    return LORA_OK;
}

int lora_pool_free_rows(const lora_pool *p, int32_t m, int64_t *free_rows) {
    if (!p || !free_rows || m < 0 || m >= p->n_modules) return LORA_EINVAL;
    *free_rows = p->mod[m].rows.free_rows;
    return LORA_OK;
}

static void release_entry(lora_pool *p, int m, int a) {
    PoolEntry &e = p->entry(m, a);
    if (e.rank > 0) {
        p->mod[m].rows.release(e.row_off, order_of(e.rp));
        p->rp_count[order_of(e.rp)]--;
    }
    e = PoolEntry{nullptr, nullptr, 0, 0, -1};
}

// The copies and host bookkeeping of one bf16 load, queued on s; *dst / *val receive the table
// write that publishes it (also on failure: the cleared entry).
static int load_one(lora_pool *p, int32_t a, int32_t m, const void *A, const void *B, int32_t rank, cudaStream_t s,
                    PoolEntry **dst, PoolEntry *val) {
    *dst = nullptr;
    if (!p || !A || !B || m < 0 || m >= p->n_modules || a < 0 || a >= p->max_adapters) return LORA_EINVAL;
    if (rank < 1 || rank > p->max_rank || p->i8) return LORA_EINVAL;
    ++p->gen;
    ModuleStore &ms = p->mod[m];
    const int rp = storage_rank(rank);
    // a reload replaces the old factors; free first so the rows can be reused
    release_entry(p, m, a);
    *dst = p->d_table + (size_t)m * p->max_adapters + a;
    const int64_t off = ms.rows.alloc(order_of(rp));
    if (off < 0) {
        *val = p->entry(m, a);
        return LORA_ENOMEM;
    }
    uint16_t *Ad = ms.A + (size_t)off * ms.d_in;
    uint16_t *Bd = ms.B + (size_t)off * ms.d_out;
    LORA_CUDA(cudaMemcpyAsync(Ad, A, (size_t)rank * ms.d_in * 2, cudaMemcpyDefault, s));
    if (rank < rp) LORA_CUDA(cudaMemsetAsync(Ad + (size_t)rank * ms.d_in, 0, (size_t)(rp - rank) * ms.d_in * 2, s));
    if (rank == rp) {
        LORA_CUDA(cudaMemcpyAsync(Bd, B, (size_t)ms.d_out * rank * 2, cudaMemcpyDefault, s));
    } else {
        LORA_CUDA(cudaMemsetAsync(Bd, 0, (size_t)ms.d_out * rp * 2, s));
        LORA_CUDA(cudaMemcpy2DAsync(Bd, (size_t)rp * 2, B, (size_t)rank * 2, (size_t)rank * 2, ms.d_out,
                                    cudaMemcpyDefault, s));
    }
    PoolEntry e{Ad, Bd, rank, rp, off};
    p->entry(m, a) = e;
    p->rp_count[order_of(rp)]++;
    *val = e;
    return LORA_OK;
}

int lora_pool_load(lora_pool *p, int32_t a, int32_t m, const void *A, const void *B, int32_t rank,
                   lora_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    PoolEntry *dst;
    PoolEntry val;
    const int rc = load_one(p, a, m, A, B, rank, s, &dst, &val);
    if (dst) LORA_CUDA(launch_table_write(dst, val, s));
    return rc;
}

int lora_pool_load_many(lora_pool *p, int32_t n, const lora_load_item *items, int32_t *n_done, lora_stream_t stream) {
    if (n_done) *n_done = 0;
    if (!p || n < 0 || (n > 0 && !items)) return LORA_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    TableWrites w;
    w.n = 0;
    int rc = LORA_OK, i = 0;
    for (; i < n; ++i) {
        PoolEntry *dst;
        PoolEntry val;
        const lora_load_item &it = items[i];
        rc = load_one(p, it.adapter, it.module, it.A, it.B, it.rank, s, &dst, &val);
        if (dst) {
            w.dst[w.n] = dst;
            w.v[w.n] = val;
            if (++w.n == kTableWritesMax) {
                LORA_CUDA(launch_table_write_many(w, s));
                w.n = 0;
            }
        }
        if (rc != LORA_OK) break;
    }
    LORA_CUDA(launch_table_write_many(w, s));
    if (n_done) *n_done = i;
    return rc;
}

int lora_pool_load_packed(lora_pool *p, int32_t n, const lora_packed_item *items, const void *host_blob,
                          void *dev_staging, int64_t blob_bytes, int32_t *n_done, lora_stream_t stream) {
    if (n_done) *n_done = 0;
    if (!p || n < 0 || blob_bytes < 0 || (n > 0 && (!items || !host_blob || !dev_staging)) || p->i8) return LORA_EINVAL;
    if (reinterpret_cast<uintptr_t>(dev_staging) & 15) return LORA_EINVAL;
    for (int i = 0; i < n; ++i) {  // every item checked before anything is queued
        const lora_packed_item &it = items[i];
        if (it.module < 0 || it.module >= p->n_modules || it.adapter < 0 || it.adapter >= p->max_adapters) return LORA_EINVAL;
        if (it.rank < 1 || it.rank > p->max_rank || it.a_offset < 0 || it.b_offset < 0) return LORA_EINVAL;
        const ModuleStore &ms = p->mod[it.module];
        if (it.a_offset % 16 || it.b_offset % 2 || it.a_offset + (int64_t)it.rank * ms.d_in * 2 > blob_bytes ||
            it.b_offset + (int64_t)ms.d_out * it.rank * 2 > blob_bytes)
            return LORA_EINVAL;
    }
    if (n == 0) return LORA_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    LORA_CUDA(cudaMemcpyAsync(dev_staging, host_blob, (size_t)blob_bytes, cudaMemcpyHostToDevice, s));
    const uint8_t *stage = static_cast<const uint8_t *>(dev_staging);
    ++p->gen;
    PackedJobs jobs;
    jobs.n = 0;
    int rc = LORA_OK, i = 0;
    for (; i < n; ++i) {
        const lora_packed_item &it = items[i];
        ModuleStore &ms = p->mod[it.module];
        const int rp = storage_rank(it.rank);
        release_entry(p, it.module, it.adapter);  // a reload replaces the old factors
        PoolEntry *dst = p->d_table + (size_t)it.module * p->max_adapters + it.adapter;
        const int64_t off = ms.rows.alloc(order_of(rp));
        if (off < 0) {
            LORA_CUDA(launch_packed_load(jobs, s));
            LORA_CUDA(launch_table_write(dst, p->entry(it.module, it.adapter), s));  // cleared
            jobs.n = 0;
            rc = LORA_ENOMEM;
            break;
        }
        PoolEntry e{ms.A + (size_t)off * ms.d_in, ms.B + (size_t)off * ms.d_out, it.rank, rp, off};
        p->entry(it.module, it.adapter) = e;
        p->rp_count[order_of(rp)]++;
        jobs.j[jobs.n++] = PackedJob{stage + it.a_offset, stage + it.b_offset, dst, e, ms.d_in, ms.d_out};
        if (jobs.n == kPackedMax) {
            LORA_CUDA(launch_packed_load(jobs, s));
            jobs.n = 0;
        }
    }
    LORA_CUDA(launch_packed_load(jobs, s));
    if (n_done) *n_done = i;
    return rc;
}

int lora_pool_unload_many(lora_pool *p, int32_t n, const int32_t *ids, int32_t *n_done, lora_stream_t stream) {
    if (n_done) *n_done = 0;
    if (!p || n < 0 || (n > 0 && !ids)) return LORA_EINVAL;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ++p->gen;
    TableWrites w;
    w.n = 0;
    int rc = LORA_OK, i = 0;
    for (; i < n; ++i) {
        const int a = ids[i];
        if (a < 0 || a >= p->max_adapters) {
            rc = LORA_EINVAL;
            break;
        }
        bool any = false;
        for (int m = 0; m < p->n_modules; ++m) {
            if (p->entry(m, a).rank <= 0) continue;
            any = true;
            release_entry(p, m, a);
            w.dst[w.n] = p->d_table + (size_t)m * p->max_adapters + a;
            w.v[w.n] = p->entry(m, a);
            if (++w.n == kTableWritesMax) {
                LORA_CUDA(launch_table_write_many(w, s));
                w.n = 0;
            }
        }
        if (!any) {
            rc = LORA_ENOTLOADED;
            break;
        }
    }
    LORA_CUDA(launch_table_write_many(w, s));
    if (n_done) *n_done = i;
    return rc;
}

int lora_pool_load_i8(lora_pool *p, int32_t a, int32_t m, const int8_t *qA, const float *sA, const int8_t *qB,
                      const float *sB, int32_t rank, lora_stream_t stream) {
    if (!p || !qA || !qB || !sA || !sB || m < 0 || m >= p->n_modules || a < 0 || a >= p->max_adapters)
        return LORA_EINVAL;
    if (rank < 1 || rank > p->max_rank || !p->i8) return LORA_EINVAL;
    ++p->gen;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    ModuleStore &ms = p->mod[m];
    const int rp = storage_rank(rank);
    release_entry(p, m, a);
    const int64_t off = ms.rows.alloc(order_of(rp));
    if (off < 0) {
        LORA_CUDA(launch_table_write(p->d_table + (size_t)m * p->max_adapters + a, p->entry(m, a), s));
        return LORA_ENOMEM;
    }
    int8_t *Ad = reinterpret_cast<int8_t *>(ms.A) + (size_t)off * ms.d_in;
    int8_t *Bd = reinterpret_cast<int8_t *>(ms.B) + (size_t)off * ms.d_out;
    LORA_CUDA(cudaMemcpyAsync(Ad, qA, (size_t)rank * ms.d_in, cudaMemcpyDefault, s));
    if (rank < rp) LORA_CUDA(cudaMemsetAsync(Ad + (size_t)rank * ms.d_in, 0, (size_t)(rp - rank) * ms.d_in, s));
    if (rank == rp) {
        LORA_CUDA(cudaMemcpyAsync(Bd, qB, (size_t)ms.d_out * rank, cudaMemcpyDefault, s));
    } else {
        LORA_CUDA(cudaMemsetAsync(Bd, 0, (size_t)ms.d_out * rp, s));
        LORA_CUDA(cudaMemcpy2DAsync(Bd, (size_t)rp, qB, (size_t)rank, (size_t)rank, ms.d_out, cudaMemcpyDefault, s));
    }
    // one fp32 scale per stored row; pageable source, so the call returns once it is staged
    std::vector<float> fold((size_t)rp, 0.f);
    for (int j = 0; j < rank; ++j) fold[(size_t)j] = sA[j] * sB[j];
    LORA_CUDA(cudaMemcpyAsync(ms.fold + off, fold.data(), (size_t)rp * 4, cudaMemcpyHostToDevice, s));
    PoolEntry e{reinterpret_cast<const uint16_t *>(Ad), reinterpret_cast<const uint16_t *>(Bd), rank, rp, off};
    p->entry(m, a) = e;
    p->rp_count[order_of(rp)]++;
    LORA_CUDA(launch_table_write(p->d_table + (size_t)m * p->max_adapters + a, e, s));
    return LORA_OK;
}

int lora_quantize_rows_int8(const void *src, int64_t rows, int64_t cols, int8_t *codes, float *scales) {
    if (rows < 0 || cols < 1 || (rows > 0 && (!src || !codes || !scales))) return LORA_EINVAL;
    const uint16_t *b = static_cast<const uint16_t *>(src);
    auto f32 = [](uint16_t h) {
        const uint32_t u = (uint32_t)h << 16;
        float f;
        std::memcpy(&f, &u, 4);
        return f;
    };
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *row = b + r * cols;
        float mx = 0.f;
        for (int64_t c = 0; c < cols; ++c) mx = std::max(mx, std::fabs(f32(row[c])));
        const float sc = mx / 127.0f;
        scales[r] = sc;
        for (int64_t c = 0; c < cols; ++c) {
            float q = 0.f;
            if (sc > 0.f) q = std::min(127.0f, std::max(-127.0f, std::nearbyint(f32(row[c]) / sc)));
            codes[r * cols + c] = (int8_t)q;
        }
    }
    return LORA_OK;
}

int lora_quantize_w4(const void *src, int64_t rows, int64_t cols, uint8_t *packed, float *scales) {
    if (rows < 0 || cols < 8 || cols % 8 != 0 || (rows > 0 && (!src || !packed || !scales))) return LORA_EINVAL;
    const uint16_t *b = static_cast<const uint16_t *>(src);
    auto f32 = [](uint16_t h) {
        const uint32_t u = (uint32_t)h << 16;
        float f;
        std::memcpy(&f, &u, 4);
        return f;
    };
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *row = b + r * cols;
        float mx = 0.f;
        for (int64_t c = 0; c < cols; ++c) mx = std::max(mx, std::fabs(f32(row[c])));
        const float sc = mx / 7.0f;
        scales[r] = sc;
        for (int64_t w = 0; w < cols / 8; ++w) {
            uint32_t word = 0;
            for (int e = 0; e < 8; ++e) {
                float q = 0.f;
                if (sc > 0.f) q = std::min(7.0f, std::max(-7.0f, std::nearbyint(f32(row[8 * w + e]) / sc)));
                const uint32_t u = (uint32_t)((int)q + 8);  // 1..15
                word |= u << ((e & 1) * 16 + (e >> 1) * 4);  // element 2s: nibble s; 2s + 1: nibble s of the high half
            }
            uint8_t *dst = packed + r * (cols / 2) + 4 * w;
            for (int k = 0; k < 4; ++k) dst[k] = (uint8_t)(word >> (8 * k));  // little-endian, on any host
        }
    }
    return LORA_OK;
}

int lora_pool_unload(lora_pool *p, int32_t a, lora_stream_t stream) {
    if (!p || a < 0 || a >= p->max_adapters) return LORA_EINVAL;
    ++p->gen;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    bool any = false;
    for (int m = 0; m < p->n_modules; ++m) {
        if (p->entry(m, a).rank > 0) {
            any = true;
            release_entry(p, m, a);
            LORA_CUDA(launch_table_write(p->d_table + (size_t)m * p->max_adapters + a, p->entry(m, a), s));
        }
    }
    return any ? LORA_OK : LORA_ENOTLOADED;
}

int lora_build_segments(const int32_t *ids, int32_t n, int32_t *perm, int32_t *seg_start, int32_t *seg_adapter,
                        int32_t *n_seg) {
    if (n < 0 || !seg_start || !n_seg || (n > 0 && (!ids || !perm || !seg_adapter))) return LORA_EINVAL;
    std::vector<int32_t> order(n);
    for (int i = 0; i < n; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return ids[x] < ids[y]; });
    int ns = 0;
    for (int q = 0; q < n; ++q) {
        perm[q] = order[q];
        if (q == 0 || ids[order[q]] != ids[order[q - 1]]) {
            seg_start[ns] = q;
            seg_adapter[ns] = ids[order[q]];
            ++ns;
        }
    }
    seg_start[ns] = n;
    *n_seg = ns;
    return LORA_OK;
}

int lora_pool_last_segments(lora_pool *p, int32_t *perm, int32_t *seg_start, int32_t *seg_adapter, int32_t *n_seg,
                            int32_t *n) {
    if (!p) return LORA_EINVAL;
    LORA_CUDA(cudaSetDevice(p->device));
    LORA_CUDA(cudaDeviceSynchronize());
    int32_t ns = 0;
    LORA_CUDA(cudaMemcpy(&ns, p->n_seg, 4, cudaMemcpyDeviceToHost));
    if (ns < 0 || ns > p->max_rows + 1) ns = 0;
    if (n) *n = p->last_n;
    if (n_seg) *n_seg = ns;
    if (perm && p->last_decode && p->last_n > 0)
        LORA_CUDA(cudaMemcpy(perm, p->perm, (size_t)p->last_n * 4, cudaMemcpyDeviceToHost));
    if (seg_start) LORA_CUDA(cudaMemcpy(seg_start, p->seg_start, (size_t)(ns + 1) * 4, cudaMemcpyDeviceToHost));
    if (seg_adapter && ns > 0) LORA_CUDA(cudaMemcpy(seg_adapter, p->seg_adapter, (size_t)ns * 4, cudaMemcpyDeviceToHost));
    return LORA_OK;
}

int lora_last_device_error(lora_pool *p, int32_t *code, int32_t *detail) {
    if (!p) return LORA_EINVAL;
    LORA_CUDA(cudaSetDevice(p->device));
    LORA_CUDA(cudaDeviceSynchronize());
    int32_t h[2] = {0, 0};
    LORA_CUDA(cudaMemcpy(h, p->err, 8, cudaMemcpyDeviceToHost));
    LORA_CUDA(cudaMemset(p->err, 0, 8));
    if (code) *code = h[0];
    if (detail) *detail = h[1];
    return LORA_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ profiling --------------

static cudaEvent_t prof_event(lora_pool *p) {
    if (!p->prof_free.empty()) {
        cudaEvent_t e = p->prof_free.back();
        p->prof_free.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

// Runs `launch` between two recorded events when profiling is on.
template <class F>
static cudaError_t timed_launch(lora_pool *p, int kind, cudaStream_t s, F &&launch) {
    if (!p->profiling) return launch();
    cudaEvent_t a = prof_event(p), b = prof_event(p);
    if (!a || !b) return launch();
    cudaEventRecord(a, s);
    cudaError_t e = launch();
    cudaEventRecord(b, s);
    p->prof_pending[kind].push_back({a, b});
    return e;
}

extern "C" int lora_pool_set_wait_budget(lora_pool *p, uint64_t budget_ns) {
    if (!p) return LORA_EINVAL;
    p->wait_ns = budget_ns ? budget_ns : kWaitBudgetNs;
    return LORA_OK;
}

extern "C" int lora_profile_enable(lora_pool *p, int32_t enable) {
    if (!p) return LORA_EINVAL;
    p->profiling = enable != 0;
    return LORA_OK;
}

extern "C" int lora_profile_read(lora_pool *p, int32_t kind, int32_t *launches, double *total_ms) {
    if (!p || kind < 0 || kind > 3) return LORA_EINVAL;
    LORA_CUDA(cudaSetDevice(p->device));
    LORA_CUDA(cudaDeviceSynchronize());
    double tot = 0;
    for (auto &pr : p->prof_pending[kind]) {
        float ms = 0;
        LORA_CUDA(cudaEventElapsedTime(&ms, pr.first, pr.second));
        tot += ms;
        p->prof_free.push_back(pr.first);
        p->prof_free.push_back(pr.second);
    }
    if (launches) *launches = (int32_t)p->prof_pending[kind].size();
    if (total_ms) *total_ms = tot;
    p->prof_pending[kind].clear();
    return LORA_OK;
}

// ------------------------------------------------------------------ forward ----------------

namespace {
std::mutex g_out_mu;
std::unordered_map<cudaStream_t, std::vector<ByteRange>> g_out;  // guarded by g_out_mu
}  // namespace

void lora::note_stream_outputs(cudaStream_t s, const ByteRange *r, int n) {
    std::lock_guard<std::mutex> lk(g_out_mu);
    g_out[s].assign(r, r + n);
}

bool lora::overlaps_stream_outputs(cudaStream_t s, const ByteRange *r, int n) {
    std::lock_guard<std::mutex> lk(g_out_mu);
    auto it = g_out.find(s);
    if (it == g_out.end()) return false;
    for (const ByteRange &o : it->second)
        for (int i = 0; i < n; ++i)
            if (r[i].lo < o.hi && o.lo < r[i].hi) return true;
    return false;
}

// mode: kOwnGrouping (group the rows, then the call's kernels), kBuildPlan (group the rows and
// build the gather lists of every module of the pool, nothing else), kUsePlan (the call's kernels
// on the last plan)
enum { kOwnGrouping = 0, kBuildPlan = 1, kUsePlan = 2 };

// One projection as the forward sees it: lora_module_io, or lora_module_io_w4 (w_scale set).
struct IoDesc {
    int32_t module;
    const void *x;
    const void *W;  // bf16 [d_out, d_in], or int4 codes [d_out, d_in / 2] bytes
    const float *w_scale;
    void *y;
};

// Decode (n <= 256): prep (unless planned), the int8 shrink on CUDA cores (int8 pools), the gemm
// (W tiles, and for bf16 pools the A tiles of the shrink), the finalize (expand, y).
static int decode_call(lora_pool *p, int n_io, const IoDesc *io, int n, float scale, int y_dtype, cudaStream_t s,
                       bool w4, const int *slot_of) {
    cudaError_t e;
    const int nt = (n + 15) & ~15;
    const int rpmax = p->rpmax();
    // int8 factors: the CUDA-core shrink, launched after the gemm (which needs no t) so that it
    // runs beside the gemm's W stream; the finalize then waits for both
    ShrinkParams sp{};
    int shrink_splits = 0;
    if (p->i8) {
        sp.n_mod = n_io;
        sp.n = n;
        sp.rpmax = rpmax;
        sp.by_segment = 1;
        sp.max_units = LORA_MAX_DECODE_ROWS;
        sp.ks_max = p->ks_cap;
        sp.scale = scale;
        sp.i8 = 1;
        sp.perm = p->perm;
        sp.qadapter = p->qadapter;
        sp.partials = p->shrink_part;
        sp.counters = p->shrink_cnt;
        // split width: about 128 KiB of A codes per block, in whole 2048-wide steps
        int kc_dec = kShrinkDecKC;
        while (kc_dec * rpmax < 128 * 1024) kc_dec += kShrinkDecKC;
        int splits = 0;
        for (int i = 0; i < n_io; ++i) {
            const ModuleStore &ms = p->mod[io[i].module];
            sp.x[i] = static_cast<const uint16_t *>(io[i].x);
            sp.table[i] = p->d_table + (size_t)io[i].module * p->max_adapters;
            sp.fold[i] = ms.fold;
            sp.T[i] = p->T + (size_t)slot_of[i] * p->max_rows * LORA_MAX_RANK;
            sp.d_in[i] = ms.d_in;
            sp.kc[i] = std::min(kc_dec, ms.d_in);
            sp.ksplit[i] = (ms.d_in + sp.kc[i] - 1) / sp.kc[i];
            if (sp.ksplit[i] > p->ks_cap) return LORA_EUNSUPPORTED;
            sp.split_begin[i] = splits;
            splits += sp.ksplit[i];
        }
        sp.split_begin[n_io] = splits;
        shrink_splits = splits;
    }

    DecodeParams dp;
    memset(&dp, 0, sizeof dp);
    dp.n_mod = n_io;
    dp.n = n;
    dp.nt = nt;
    dp.tp_rows = p->tp_rows;
    dp.shrink_tc = p->i8 ? 0 : 1;
    dp.w4 = w4 ? 1 : 0;
    dp.i8 = p->i8 ? 1 : 0;
    dp.y_bf16 = y_dtype == LORA_DTYPE_BF16 ? 1 : 0;
    dp.rpmax = rpmax;
    dp.scale = scale;
    dp.perm = p->perm;
    dp.rb_order = p->rb_order;
    dp.radapter = p->radapter;
    // base pieces in the workspace half of this call's parity: the previous call's finalize may
    // still read the other half while this call's W tiles run
    dp.home = p->home + (size_t)p->call_parity * p->w_tiles_cap * kBM * p->nt_cap;
    dp.ctaw = p->ctaw + (size_t)p->call_parity * p->num_sms * kBM * p->nt_cap;
    dp.err = p->err;
    dp.wait_ns = p->wait_ns;
    {
        ByteRange xr[LORA_MAX_MODULES] = {};
        for (int i = 0; i < n_io; ++i) {
            const uintptr_t lo = reinterpret_cast<uintptr_t>(io[i].x);
            xr[i] = ByteRange{lo, lo + (uintptr_t)n * p->mod[io[i].module].d_in * 2};
        }
        dp.w_first = overlaps_stream_outputs(s, xr, n_io) ? 0 : 1;
    }
    // Where the A tiles' t parts are added up.  In the finalize when a batch of more than 128 rows
    // can put tens of rows on one adapter (a tile's last CTA would add them one row range after
    // another, at the end of its W stream) or the ranks are small (few values per finalize block);
    // otherwise once per tile in the gemm, so that the many finalize blocks of wide projections
    // read t directly.
    dp.t_fin = (nt > 128 || rpmax <= 16) ? 1 : 0;
    // two k-blocks per pipeline stage (half the TMA requests, above all for the 8-row A gathers)
    // when every projection's d_in is a whole number of k-blocks and the batch fills at most 128
    // columns (a stage of a 256-row batch would leave only two in shared memory)
    dp.kps = nt <= 128 ? 2 : 1;
    for (int i = 0; i < n_io; ++i)
        if (p->mod[io[i].module].d_in % 64 != 0) dp.kps = 1;
    int iters = 0, tiles = 0;
    for (int i = 0; i < n_io; ++i) {
        const ModuleStore &ms = p->mod[io[i].module];
        DecodeModule &dm = dp.mod[i];
        int rc;
        if (w4) {
            rc = make_tmap_u8(&dm.tmW, io[i].W, ms.d_out, ms.d_in / 2, kBK / 2, kBM, dp.kps);
            dm.w_scale = io[i].w_scale;
        } else {
            rc = make_tmap(&dm.tmW, io[i].W, ms.d_out, ms.d_in, kBM, dp.kps);
        }
        if (rc) return rc;
        if ((rc = make_tmap(&dm.tmX, io[i].x, n, ms.d_in, nt, dp.kps))) return rc;
        if (!p->i8) {
            dm.tmA = ms.tmA[dp.kps - 1];
            dm.tmA128 = ms.tmA128[dp.kps - 1];
            dm.a_runs = ms.a_runs ? 1 : 0;
            dm.a_boxes = (dp.kps == 1 && ms.a_boxes) ? 1 : 0;
            if (dm.a_boxes)
                for (int j = 0; j < 3; ++j) dm.tmAb[j] = ms.tmAb[j];
        }
        const int sl = slot_of[i];
        dm.groups = p->groups + (size_t)sl * kDecMaxGroups;
        dm.n_groups = p->n_groups + sl;
        dm.rowinfo = p->rowinfo + (size_t)sl * LORA_MAX_DECODE_ROWS;
        dm.T = p->T + (size_t)sl * p->max_rows * LORA_MAX_RANK;
        dm.tpart = p->tpart + (size_t)sl * kDecMaxParts * p->tp_rows * LORA_MAX_RANK;
        dm.tfin = p->tfin + (size_t)sl * p->tp_rows * LORA_MAX_RANK;
        dm.acount = p->acount + (size_t)sl * (kDecMaxGroups / kTileGroups);
        dm.y = io[i].y;
        dm.d_in = ms.d_in;
        dm.d_out = ms.d_out;
        dm.m_tiles = (ms.d_out + kBM - 1) / kBM;
        dm.k_blocks = ((ms.d_in + kBK - 1) / kBK + dp.kps - 1) / dp.kps;  // k-steps
        dm.w_iter_begin = iters;
        dm.w_tile_begin = tiles;
        tiles += dm.m_tiles;
        iters += dm.m_tiles * dm.k_blocks;
    }
    if (tiles > p->w_tiles_cap) return LORA_EUNSUPPORTED;  // a projection named twice in one call
    dp.w_tiles = tiles;
    dp.w_iters = iters;
    // every CTA gets at least 4 k-blocks of the W space, so all its ranges are non-empty
    dp.n_cta = std::max(1, std::min(p->num_sms, iters / 4));
    size_t smem = 0;
    if (!plan_decode_gemm(dp, &smem)) return LORA_EUNSUPPORTED;
    e = timed_launch(p, LORA_KERNEL_GEMM, s, [&] { return launch_decode_gemm(dp, smem, s); });
    if (e != cudaSuccess) return cuda_fail(e, "gemm kernel");
    if (p->i8) {
        e = timed_launch(p, LORA_KERNEL_SHRINK, s, [&] { return launch_shrink(sp, n, shrink_splits, s); });
        if (e != cudaSuccess) return cuda_fail(e, "shrink kernel");
    }
    size_t fsmem = 0;
    plan_decode_finalize(dp, &fsmem);
    e = timed_launch(p, LORA_KERNEL_FINALIZE, s, [&] { return launch_decode_finalize(dp, fsmem, s); });
    if (e != cudaSuccess) return cuda_fail(e, "finalize kernel");
    p->call_parity ^= 1;
    return LORA_OK;
}

// Grouped rows (n > 256, contiguous segments): prep, shrink, gemm with the expand in its ring.
static int grouped_call(lora_pool *p, int n_io, const IoDesc *io, int n, float scale, int y_dtype, cudaStream_t s) {
    cudaError_t e;
    const int nt = 256;
    const int rpmax = p->rpmax();
    ShrinkParams sp{};
    sp.n_mod = n_io;
    sp.n = n;
    sp.rpmax = rpmax;
    sp.by_segment = 0;
    sp.max_units = LORA_MAX_DECODE_ROWS;
    sp.ks_max = p->ks_cap;
    sp.scale = scale;
    sp.seg_start = p->seg_start;
    sp.seg_adapter = p->seg_adapter;
    sp.n_seg = p->n_seg;
    for (int i = 0; i < n_io; ++i) {
        const ModuleStore &ms = p->mod[io[i].module];
        sp.x[i] = static_cast<const uint16_t *>(io[i].x);
        sp.table[i] = p->d_table + (size_t)io[i].module * p->max_adapters;
        sp.T[i] = p->T + (size_t)i * p->max_rows * LORA_MAX_RANK;
        sp.d_in[i] = ms.d_in;
        sp.kc[i] = ms.d_in;
        sp.ksplit[i] = 1;
        sp.split_begin[i] = i;
    }
    sp.split_begin[n_io] = n_io;
    const int units = (n + kShrinkGroupRows - 1) / kShrinkGroupRows;
    e = timed_launch(p, LORA_KERNEL_SHRINK, s, [&] { return launch_shrink(sp, units, n_io, s); });
    if (e != cudaSuccess) return cuda_fail(e, "shrink kernel");

    GemmParams gp;
    memset(&gp, 0, sizeof gp);
    gp.n_mod = n_io;
    gp.n = n;
    gp.nt = nt;
    gp.n_chunks = (n + nt - 1) / nt;
    gp.rpmax = rpmax;
    gp.y_bf16 = y_dtype == LORA_DTYPE_BF16 ? 1 : 0;
    gp.raster_group = 8;
    gp.wait_ns = p->wait_ns;
    int tiles = 0;
    for (int i = 0; i < n_io; ++i) {
        const ModuleStore &ms = p->mod[io[i].module];
        GemmModule &gm = gp.mod[i];
        int rc;
        if ((rc = make_tmap(&gm.tmW, io[i].W, ms.d_out, ms.d_in, kBM))) return rc;
        if ((rc = make_tmap(&gm.tmX, io[i].x, n, ms.d_in, nt))) return rc;
        if ((rc = make_tmap_y(&gm.tmY, io[i].y, n, ms.d_out, y_dtype == LORA_DTYPE_BF16))) return rc;
        gm.y = io[i].y;
        gm.T = sp.T[i];
        gm.table = sp.table[i];
        gm.d_in = ms.d_in;
        gm.d_out = ms.d_out;
        gm.m_tiles = (ms.d_out + kBM - 1) / kBM;
        gm.k_blocks = (ms.d_in + kBK - 1) / kBK;
        gm.tile_begin = tiles;
        tiles += gm.m_tiles * gp.n_chunks;
    }
    gp.total_tiles = tiles;
    gp.n_cta = std::min(p->num_sms, tiles);
    gp.chunk_seg0 = p->chunk_seg0;
    gp.chunk_nb = p->chunk_nb;
    gp.pf_ch = pf_ch(nt, rpmax);
    size_t smem = 0;
    if (!plan_gemm(gp, &smem)) return LORA_EUNSUPPORTED;
    gp.seg_start = p->seg_start;
    gp.seg_adapter = p->seg_adapter;
    gp.n_seg = p->n_seg;
    gp.err = p->err;
    e = timed_launch(p, LORA_KERNEL_GEMM, s, [&] { return launch_gemm(gp, smem, s); });
    if (e != cudaSuccess) return cuda_fail(e, "gemm kernel");
    return LORA_OK;
}

static int forward_impl(lora_pool *p, int n_io, const IoDesc *io, const int32_t *ids,
                        const int32_t *seg_start, const int32_t *seg_adapter, int n_seg, int n, float scale,
                        int y_dtype, cudaStream_t s, int mode = kOwnGrouping, bool w4 = false) {
    if (!p) return LORA_EINVAL;
    if (mode == kUsePlan) {
        if (p->plan_gen != p->gen) return LORA_EINVAL;  // no plan, or the pool changed since
        n = p->plan_n;
    }
    if (mode == kBuildPlan) {
        if (!ids || n < 0 || n > std::min(p->max_rows, LORA_MAX_DECODE_ROWS)) return LORA_EINVAL;
        ++p->gen;
        p->plan_gen = 0;
        if (n == 0) {
            p->plan_gen = p->gen;
            p->plan_n = 0;
            return LORA_OK;
        }
    } else {
        if (!io || n_io < 1 || n_io > LORA_MAX_MODULES || n < 0 || n > p->max_rows) return LORA_EINVAL;
        if (y_dtype != LORA_DTYPE_F32 && y_dtype != LORA_DTYPE_BF16) return LORA_EINVAL;
        for (int i = 0; i < n_io; ++i)
            if (io[i].module < 0 || io[i].module >= p->n_modules) return LORA_EINVAL;
        if (mode == kOwnGrouping) ++p->gen;  // this call's grouping overwrites any plan
    }
    if (n == 0) return LORA_OK;  // empty batch: nothing to read or write
    for (int i = 0; mode != kBuildPlan && i < n_io; ++i) {
        const IoDesc &m = io[i];
        if (!m.x || !m.W || !m.y) return LORA_EINVAL;
        if (!aligned16(m.x) || !aligned16(m.W) || !aligned16(m.y)) return LORA_EINVAL;
        if (w4 && (!m.w_scale || (reinterpret_cast<uintptr_t>(m.w_scale) & 3))) return LORA_EINVAL;
        // int4 codes: a packed row (d_in / 2 bytes) is a whole number of 16-byte TMA strides
        if (w4 && p->mod[m.module].d_in % 32 != 0) return LORA_EUNSUPPORTED;
    }
    if (mode == kOwnGrouping && ids == nullptr && (!seg_start || !seg_adapter || n_seg < 1 || n_seg > n))
        return LORA_EINVAL;
    const bool decode = n <= LORA_MAX_DECODE_ROWS;
    if ((ids || p->i8 || w4) && !decode) return LORA_EUNSUPPORTED;
    // the plan covers every module of the pool; a planned call finds module m's lists at slot m
    const int n_prep = mode == kBuildPlan ? p->n_modules : n_io;
    int slot_of[LORA_MAX_MODULES];
    for (int i = 0; i < n_prep; ++i) slot_of[i] = mode == kOwnGrouping ? i : (mode == kBuildPlan ? i : io[i].module);
    auto pool_module = [&](int i) { return mode == kBuildPlan ? i : io[i].module; };

    // ---- prep: row grouping / checks
    if (mode != kUsePlan) {
        PrepParams pp{};
        pp.ids = ids;
        pp.seg_start_in = seg_start;
        pp.seg_adapter_in = seg_adapter;
        pp.n_seg_in = n_seg;
        pp.n = n;
        pp.max_adapters = p->max_adapters;
        pp.n_mod = n_prep;
        for (int i = 0; i < n_prep; ++i) pp.table[i] = p->d_table + (size_t)pool_module(i) * p->max_adapters;
        pp.perm = p->perm;
        pp.seg_start = p->seg_start;
        pp.seg_adapter = p->seg_adapter;
        pp.n_seg = p->n_seg;
        pp.err = p->err;
        pp.qadapter = p->qadapter;
        if (decode) {
            pp.radapter = p->radapter;
            pp.rb_order = p->rb_order;
            pp.n_groups = p->n_groups;
            for (int i = 0; i < n_prep; ++i) {
                if (!p->i8) pp.groups[i] = p->groups + (size_t)slot_of[i] * kDecMaxGroups;
                pp.rowinfo[i] = p->rowinfo + (size_t)slot_of[i] * LORA_MAX_DECODE_ROWS;
            }
        } else {
            if ((n + 255) / 256 > p->chunk_cap) return LORA_EUNSUPPORTED;
            pp.nt = 256;
            pp.pf_ch = pf_ch(256, p->rpmax());
            pp.chunk_seg0 = p->chunk_seg0;
            pp.chunk_nb = p->chunk_nb;
        }
        cudaError_t e = timed_launch(p, LORA_KERNEL_PREP, s,
                                     [&] { return decode ? launch_prep_decode(pp, s) : launch_prep_segments(pp, s); });
        if (e != cudaSuccess) return cuda_fail(e, "prep kernel");
        p->last_n = n;
        p->last_decode = decode;
    }
    if (mode == kBuildPlan) {
        p->plan_gen = p->gen;
        p->plan_n = n;
        return LORA_OK;
    }
    const int rc = decode ? decode_call(p, n_io, io, n, scale, y_dtype, s, w4, slot_of)
                          : grouped_call(p, n_io, io, n, scale, y_dtype, s);
    if (rc == LORA_OK) {
        ByteRange yr[LORA_MAX_MODULES] = {};
        const size_t es = y_dtype == LORA_DTYPE_BF16 ? 2 : 4;
        for (int i = 0; i < n_io; ++i) {
            const uintptr_t lo = reinterpret_cast<uintptr_t>(io[i].y);
            yr[i] = ByteRange{lo, lo + (uintptr_t)((size_t)n * p->mod[io[i].module].d_out * es)};
        }
        note_stream_outputs(s, yr, n_io);
    }
    return rc;
}

namespace {
// the projections of a call as IoDesc; false if n_io is out of range or io is missing
bool io_descs(int32_t n_io, const lora_module_io *io, IoDesc (&d)[LORA_MAX_MODULES]) {
    if (!io || n_io < 1 || n_io > LORA_MAX_MODULES) return false;
    for (int i = 0; i < n_io; ++i) d[i] = IoDesc{io[i].module, io[i].x, io[i].W, nullptr, io[i].y};
    return true;
}
bool io_descs(int32_t n_io, const lora_module_io_w4 *io, IoDesc (&d)[LORA_MAX_MODULES]) {
    if (!io || n_io < 1 || n_io > LORA_MAX_MODULES) return false;
    for (int i = 0; i < n_io; ++i) d[i] = IoDesc{io[i].module, io[i].x, io[i].W_codes, io[i].W_scale, io[i].y};
    return true;
}

template <class Io>
int layer_forward(lora_pool *p, int32_t n_io, const Io *io, const int32_t *ids, int32_t n, float scale,
                  int32_t y_dtype, lora_stream_t stream, bool w4) {
    IoDesc d[LORA_MAX_MODULES];
    if (!io_descs(n_io, io, d)) return LORA_EINVAL;
    if (!ids && n > 0) return LORA_EINVAL;
    if (n == 0) return forward_impl(p, n_io, d, nullptr, nullptr, nullptr, 0, 0, scale, y_dtype, nullptr, kOwnGrouping, w4);
    if (n > LORA_MAX_DECODE_ROWS) return LORA_EUNSUPPORTED;
    return forward_impl(p, n_io, d, ids, nullptr, nullptr, 0, n, scale, y_dtype, reinterpret_cast<cudaStream_t>(stream),
                        kOwnGrouping, w4);
}

template <class Io>
int layer_forward_planned(lora_pool *p, int32_t n_io, const Io *io, float scale, int32_t y_dtype,
                          lora_stream_t stream, bool w4) {
    IoDesc d[LORA_MAX_MODULES];
    if (!io_descs(n_io, io, d)) return LORA_EINVAL;
    return forward_impl(p, n_io, d, nullptr, nullptr, nullptr, 0, 0, scale, y_dtype,
                        reinterpret_cast<cudaStream_t>(stream), kUsePlan, w4);
}
}  // namespace

extern "C" {

int lora_layer_forward(lora_pool *p, int32_t n_io, const lora_module_io *io, const int32_t *ids, int32_t n,
                       float scale, int32_t y_dtype, lora_stream_t stream) {
    return layer_forward(p, n_io, io, ids, n, scale, y_dtype, stream, false);
}

int lora_layer_forward_w4(lora_pool *p, int32_t n_io, const lora_module_io_w4 *io, const int32_t *ids, int32_t n,
                          float scale, int32_t y_dtype, lora_stream_t stream) {
    return layer_forward(p, n_io, io, ids, n, scale, y_dtype, stream, true);
}

int lora_linear_forward(lora_pool *p, int32_t module, const void *x, const void *W, const int32_t *ids, int32_t n,
                        float scale, void *y, int32_t y_dtype, lora_stream_t stream) {
    lora_module_io io{module, x, W, y};
    return lora_layer_forward(p, 1, &io, ids, n, scale, y_dtype, stream);
}

int lora_plan_rows(lora_pool *p, const int32_t *ids, int32_t n, lora_stream_t stream) {
    return forward_impl(p, 0, nullptr, ids, nullptr, nullptr, 0, n, 1.f, LORA_DTYPE_F32,
                        reinterpret_cast<cudaStream_t>(stream), kBuildPlan);
}

int lora_layer_forward_planned(lora_pool *p, int32_t n_io, const lora_module_io *io, float scale, int32_t y_dtype,
                               lora_stream_t stream) {
    return layer_forward_planned(p, n_io, io, scale, y_dtype, stream, false);
}

int lora_layer_forward_planned_w4(lora_pool *p, int32_t n_io, const lora_module_io_w4 *io, float scale,
                                  int32_t y_dtype, lora_stream_t stream) {
    return layer_forward_planned(p, n_io, io, scale, y_dtype, stream, true);
}

int lora_layer_step(lora_pool *p, const int32_t *ids, int32_t n, int32_t n_stages, const int32_t *stage_n,
                    const lora_module_io *io, float scale, int32_t y_dtype, lora_stream_t stream) {
    if (!p || n_stages < 0 || (n_stages > 0 && (!stage_n || !io))) return LORA_EINVAL;
    for (int st = 0; st < n_stages; ++st)
        if (stage_n[st] < 1) return LORA_EINVAL;
    int rc = lora_plan_rows(p, ids, n, stream);
    if (rc != LORA_OK) return rc;
    for (int st = 0, off = 0; st < n_stages; off += stage_n[st], ++st)
        if ((rc = lora_layer_forward_planned(p, stage_n[st], io + off, scale, y_dtype, stream)) != LORA_OK) return rc;
    return LORA_OK;
}

}  // extern "C"

namespace {
int planned_forward(lora_pool *p, int32_t n_io, const lora_module_io *io, float scale, int32_t y_dtype,
                    lora_stream_t stream) {
    return lora_layer_forward_planned(p, n_io, io, scale, y_dtype, stream);
}
int planned_forward(lora_pool *p, int32_t n_io, const lora_module_io_w4 *io, float scale, int32_t y_dtype,
                    lora_stream_t stream) {
    return lora_layer_forward_planned_w4(p, n_io, io, scale, y_dtype, stream);
}

// lora_layer_step_host and its int4-base twin: IO is lora_module_io or lora_module_io_w4 (module,
// x and y are what this code reads of it)
template <class IO>
int step_host(lora_pool *p, const int32_t *host_ids, int32_t *row_adapter_ids, int32_t n, int32_t n_stages,
              const int32_t *stage_n, const IO *io, const void *const *host_x, void *const *host_y, float scale,
              int32_t y_dtype, lora_stream_t stream) {
    if (!p || !host_ids || !row_adapter_ids || n < 0 || n_stages < 0 || (n_stages > 0 && (!stage_n || !io || !host_x || !host_y)))
        return LORA_EINVAL;
    if (y_dtype != LORA_DTYPE_F32 && y_dtype != LORA_DTYPE_BF16) return LORA_EINVAL;
    int total = 0;
    for (int st = 0; st < n_stages; ++st) {
        if (stage_n[st] < 1) return LORA_EINVAL;
        for (int i = total; i < total + stage_n[st]; ++i)
            if (io[i].module < 0 || io[i].module >= p->n_modules || io[i].x != io[total].x || !host_y[i]) return LORA_EINVAL;
        if (!host_x[st]) return LORA_EINVAL;
        total += stage_n[st];
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    LORA_CUDA(cudaSetDevice(p->device));
    if (!p->d2h) LORA_CUDA(cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking));
    if (!p->h2d) LORA_CUDA(cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking));
    if (!p->inputs_ready) LORA_CUDA(cudaEventCreateWithFlags(&p->inputs_ready, cudaEventDisableTiming));
    if (!p->downloads_done) LORA_CUDA(cudaEventCreateWithFlags(&p->downloads_done, cudaEventDisableTiming));
    while ((int)p->stage_done.size() < n_stages) {
        cudaEvent_t e;
        LORA_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
        p->stage_done.push_back(e);
    }
    // the buffer set of this call (least recently used slot for a new one)
    lora_pool::BufSet *bs = nullptr;
    for (auto &b : p->bufsets)
        if (b.key == row_adapter_ids) bs = &b;
    if (!bs) {
        bs = &p->bufsets[0];
        for (auto &b : p->bufsets)
            if (b.last < bs->last) bs = &b;
        if (!bs->in_free) LORA_CUDA(cudaEventCreateWithFlags(&bs->in_free, cudaEventDisableTiming));
        if (!bs->out_free) LORA_CUDA(cudaEventCreateWithFlags(&bs->out_free, cudaEventDisableTiming));
        bs->key = row_adapter_ids;
        bs->used = false;
    }
    bs->last = ++p->host_calls;
    // inputs in, on the pool's upload stream: after the last compute that read this set's inputs,
    // so they may go up while an earlier call (another set) still computes
    if (bs->used) LORA_CUDA(cudaStreamWaitEvent(p->h2d, bs->in_free, 0));
    LORA_CUDA(cudaMemcpyAsync(row_adapter_ids, host_ids, (size_t)n * 4, cudaMemcpyHostToDevice, p->h2d));
    for (int st = 0, off = 0; st < n_stages; off += stage_n[st], ++st)
        LORA_CUDA(cudaMemcpyAsync(const_cast<void *>(io[off].x), host_x[st], (size_t)n * p->mod[io[off].module].d_in * 2,
                                  cudaMemcpyHostToDevice, p->h2d));
    LORA_CUDA(cudaEventRecord(p->inputs_ready, p->h2d));
    // the step on `stream`: once its inputs are in and this set's outputs of an earlier call are out
    LORA_CUDA(cudaStreamWaitEvent(s, p->inputs_ready, 0));
    if (bs->used) LORA_CUDA(cudaStreamWaitEvent(s, bs->out_free, 0));
    int rc = lora_plan_rows(p, row_adapter_ids, n, stream);
    if (rc != LORA_OK) return rc;
    // each stage, then its outputs out on the pool's download stream while the next stage (or the
    // next call) computes
    const size_t esz = y_dtype == LORA_DTYPE_F32 ? 4 : 2;
    for (int st = 0, off = 0; st < n_stages; off += stage_n[st], ++st) {
        if ((rc = planned_forward(p, stage_n[st], io + off, scale, y_dtype, stream)) != LORA_OK) return rc;
        LORA_CUDA(cudaEventRecord(p->stage_done[(size_t)st], s));
        LORA_CUDA(cudaStreamWaitEvent(p->d2h, p->stage_done[(size_t)st], 0));
        for (int i = off; i < off + stage_n[st]; ++i)
            LORA_CUDA(cudaMemcpyAsync(host_y[i], io[i].y, (size_t)n * p->mod[io[i].module].d_out * esz,
                                      cudaMemcpyDeviceToHost, p->d2h));
    }
    LORA_CUDA(cudaEventRecord(bs->in_free, s));
    LORA_CUDA(cudaEventRecord(bs->out_free, p->d2h));
    bs->used = true;
    return LORA_OK;
}
}  // namespace

extern "C" {

int lora_layer_step_host(lora_pool *p, const int32_t *host_ids, int32_t *row_adapter_ids, int32_t n, int32_t n_stages,
                         const int32_t *stage_n, const lora_module_io *io, const void *const *host_x,
                         void *const *host_y, float scale, int32_t y_dtype, lora_stream_t stream) {
    return step_host(p, host_ids, row_adapter_ids, n, n_stages, stage_n, io, host_x, host_y, scale, y_dtype, stream);
}

int lora_layer_step_host_w4(lora_pool *p, const int32_t *host_ids, int32_t *row_adapter_ids, int32_t n,
                            int32_t n_stages, const int32_t *stage_n, const lora_module_io_w4 *io,
                            const void *const *host_x, void *const *host_y, float scale, int32_t y_dtype,
                            lora_stream_t stream) {
    return step_host(p, host_ids, row_adapter_ids, n, n_stages, stage_n, io, host_x, host_y, scale, y_dtype, stream);
}

int lora_pool_host_wait(lora_pool *p, lora_stream_t stream) {
    if (!p) return LORA_EINVAL;
    if (!p->d2h) return LORA_OK;
    LORA_CUDA(cudaEventRecord(p->downloads_done, p->d2h));
    LORA_CUDA(cudaStreamWaitEvent(reinterpret_cast<cudaStream_t>(stream), p->downloads_done, 0));
    return LORA_OK;
}

int lora_segment_forward(lora_pool *p, int32_t n_io, const lora_module_io *io, const int32_t *seg_start,
                         const int32_t *seg_adapter, int32_t n_seg, int32_t n, float scale, int32_t y_dtype,
                         lora_stream_t stream) {
    IoDesc d[LORA_MAX_MODULES];
    if (!io_descs(n_io, io, d)) return LORA_EINVAL;
    if (n == 0) return forward_impl(p, n_io, d, nullptr, nullptr, nullptr, 0, 0, scale, y_dtype, nullptr);
    if (!seg_start || !seg_adapter) return LORA_EINVAL;
    return forward_impl(p, n_io, d, nullptr, seg_start, seg_adapter, n_seg, n, scale, y_dtype,
                        reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ------------------------------------------------------------------ layer gates -----------

struct lora_layer_gate {
    int device = 0;
    std::vector<cudaEvent_t> ev;
};

int lora_layer_gate_create(int32_t n_layers, lora_layer_gate **out) {
    if (!out || n_layers < 1) return LORA_EINVAL;
    *out = nullptr;
    auto *g = new lora_layer_gate;
    if (cudaGetDevice(&g->device) != cudaSuccess) {
        delete g;
        return cuda_fail(cudaGetLastError(), "cudaGetDevice");
    }
    g->ev.assign((size_t)n_layers, nullptr);
    for (auto &e : g->ev) {
        const cudaError_t ce = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
        if (ce != cudaSuccess) {
            lora_layer_gate_destroy(g);
            return cuda_fail(ce, "cudaEventCreateWithFlags");
        }
    }
    *out = g;
    return LORA_OK;
}

int lora_layer_gate_destroy(lora_layer_gate *g) {
    if (!g) return LORA_EINVAL;
    for (auto e : g->ev)
        if (e) cudaEventDestroy(e);
    delete g;
    return LORA_OK;
}

int lora_layer_gate_mark(lora_layer_gate *g, int32_t layer, lora_stream_t copy_stream) {
    if (!g || layer < 0 || layer >= (int32_t)g->ev.size()) return LORA_EINVAL;
    LORA_CUDA(cudaEventRecord(g->ev[(size_t)layer], reinterpret_cast<cudaStream_t>(copy_stream)));
    return LORA_OK;
}

int lora_layer_gate_wait(lora_layer_gate *g, int32_t layer, lora_stream_t compute_stream) {
    if (!g || layer < 0 || layer >= (int32_t)g->ev.size()) return LORA_EINVAL;
    // loads already finished need no wait: leaving it out keeps the compute stream's kernels
    // back to back (each launches early on the one before, which a stream wait would prevent)
    const cudaError_t q = cudaEventQuery(g->ev[(size_t)layer]);
    if (q == cudaSuccess) return LORA_OK;
    if (q != cudaErrorNotReady) return cuda_fail(q, "cudaEventQuery");
    LORA_CUDA(cudaStreamWaitEvent(reinterpret_cast<cudaStream_t>(compute_stream), g->ev[(size_t)layer], 0));
    return LORA_OK;
}
