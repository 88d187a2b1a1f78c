// lora_internal.h -- structures shared by the host side (pool, API) and the kernels.
#pragma once
#include <cstdint>
#include <string>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/lora_gb300.h"

namespace lora {

// One (adapter, module) entry of the device-side indirection table.  Kernels read the
// factor addresses from here at run time, so captured graphs survive loads and unloads.
struct alignas(32) PoolEntry {
    const uint16_t *A;  // [rp, d_in] bf16, rows >= rank are zero
    const uint16_t *B;  // [d_out, rp] bf16, columns >= rank are zero
    int32_t rank;       // 0 = not resident
    int32_t rp;         // storage rank: power of two in {8, 16, 32, 64}
    int64_t row_off;    // first pool row (host bookkeeping)
};
static_assert(sizeof(PoolEntry) == 32, "PoolEntry layout");

constexpr int kBM = 128;       // W rows per tile (MMA M)
constexpr int kBK = 64;        // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int kEpiWarps = 4;   // epilogue warps (one per TMEM lane quarter)
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxWin = 256;        // segments one tile's expand can touch (= max rows per tile)
constexpr int kMaxStages = 8;
constexpr int kShrinkThreads = 256;
constexpr int kShrinkRows = 8;      // rows per register block in the shrink
constexpr int kShrinkKSub = 1024;   // K elements staged in shared memory per step
constexpr int kShrinkGroupRows = 64;  // rows per shrink block on the grouped (prefill) path
constexpr int kShrinkDecCh = 8;       // decode shrink: 16-byte chunks of A per lane and pass
constexpr int kShrinkDecKC = 256 * kShrinkDecCh;  // decode shrink: K per block (split width)
constexpr int kShrinkDecRows = 4;     // decode shrink: rows sharing one register load of A

struct GemmModule {
    CUtensorMap tmW;  // W [d_out, d_in]: box {64, 128}, 128B swizzle
    CUtensorMap tmX;  // X [n, d_in]:    box {64, nt},  128B swizzle
    CUtensorMap tmY;  // y [n, d_out]:   box {128, 16}, fp32 or bf16, no swizzle (epilogue stores)
    void *y;
    const float *T;            // scaled shrink result, sorted positions, [n][rpmax]
    const PoolEntry *table;    // this module's entries [max_adapters]
    int32_t d_in, d_out;
    int32_t m_tiles, k_blocks;
    int64_t iter_begin;        // flattened (tile, k-block) index where this module starts
    int32_t tile_begin;        // first global tile index of this module
    int32_t pad_;
};

struct GemmParams {
    GemmModule mod[LORA_MAX_MODULES];
    int32_t n_mod;
    int32_t n;             // rows
    int32_t nt;            // rows per chunk (MMA N), multiple of 16, <= 256
    int32_t n_chunks;
    int32_t decode;        // 1: one chunk, TMEM column = original row, init maps q -> perm[q]
    int32_t stream_k;      // 1: contiguous (tile, k-block) ranges per CTA; 0: whole tiles round robin
    int32_t n_cta;
    int32_t total_tiles;
    int64_t total_iters;
    int32_t rpmax;         // T row stride
    int32_t y_bf16;
    int32_t n_stages;
    int32_t ring_chunks;   // per epilogue thread: 16-byte pieces of B rows staged per batch
    int32_t raster_group;  // W tiles per raster group (round robin)
    int32_t tmem_cols;
    int32_t n_acc;         // accumulator + delta buffer pairs in TMEM (2 when 4 * nt <= 512, else 1)
    const int32_t *perm;
    const int32_t *seg_start;
    const int32_t *seg_adapter;
    const int32_t *n_seg;
    float *partials;       // [n_cta][2][kBM * nt]
    int32_t *tile_counters;
    int32_t *err;          // [0] code, [1] detail
};

struct ShrinkParams {
    const uint16_t *x[LORA_MAX_MODULES];
    const PoolEntry *table[LORA_MAX_MODULES];
    float *T[LORA_MAX_MODULES];
    int32_t d_in[LORA_MAX_MODULES];
    int32_t ksplit[LORA_MAX_MODULES];
    int32_t kc[LORA_MAX_MODULES];       // K elements per split
    int32_t split_begin[LORA_MAX_MODULES + 1];
    int32_t n_mod;
    int32_t n;
    int32_t rpmax;
    int32_t by_segment;   // 1: one block per segment (decode); 0: one block per 64 rows
    int32_t max_units;
    int32_t ks_max;
    float scale;
    const int32_t *perm;  // null: identity
    const int32_t *seg_start;
    const int32_t *seg_adapter;
    const int32_t *n_seg;
    float *partials;      // [n_mod][ks_max][n][rpmax]
    int32_t *counters;    // [n_mod][max_units]
};

struct PrepParams {
    const int32_t *ids;          // decode ids (device) or null
    const int32_t *seg_start_in; // segment table (device) or null
    const int32_t *seg_adapter_in;
    int32_t n_seg_in;
    int32_t n;
    int32_t max_adapters;
    int32_t n_mod;
    const PoolEntry *table[LORA_MAX_MODULES];
    int32_t *perm;
    int32_t *seg_start;
    int32_t *seg_adapter;
    int32_t *n_seg;
    int32_t *err;
};

static_assert(sizeof(GemmParams) <= 32764, "gemm parameters exceed the kernel parameter space");

// tensor maps (lora_api.cu): bf16 [rows, cols] operand, box {64, box_rows}, 128-byte swizzle; and
// the output y [n, d_out] (fp32 or bf16), box {128, 16}, for the epilogue's TMA stores
int make_tmap(CUtensorMap *tm, const void *base, int64_t rows, int64_t cols, int box_rows);
int make_tmap_y(CUtensorMap *tm, void *y, int64_t n, int64_t d_out, bool bf16);

// launchers (lora_kernels.cu)
cudaError_t launch_prep_decode(const PrepParams &p, cudaStream_t s);
cudaError_t launch_prep_segments(const PrepParams &p, cudaStream_t s);
cudaError_t launch_shrink(const ShrinkParams &p, int grid_x, int grid_y, cudaStream_t s);
cudaError_t launch_gemm(const GemmParams &p, size_t smem_bytes, cudaStream_t s);
cudaError_t launch_table_write(PoolEntry *dst, PoolEntry value, cudaStream_t s);
size_t gemm_smem_bytes(int nt, int n_stages, int ring_chunks, int rpmax);

// lora_api.cu: sets the string lora_last_cuda_error() returns on this thread
void set_last_error(const char *why);
inline void set_last_error(const std::string &why) { set_last_error(why.c_str()); }

}  // namespace lora
