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
    int64_t row_off;    // first row of A in the module's A slab (the gathers' TMA coordinate)
};
static_assert(sizeof(PoolEntry) == 32, "PoolEntry layout");

constexpr uint64_t kWaitBudgetNs = 2000000000ull;  // default in-kernel wait budget: 2 s, far above any legitimate wait
constexpr int kBM = 128;       // W rows per tile (MMA M)
constexpr int kBK = 64;        // K per pipeline stage (one 128-byte swizzle row of bf16)
constexpr int kEpiWarps = 4;   // epilogue warps (one per TMEM lane quarter)
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;
// int4 base weights: converter warps unpack each W k-block's codes into the bf16 tile the MMA reads
constexpr int kConvWarps = 4;
constexpr int kW4RawBytes = kBM * kBK / 2;  // packed codes of one W k-block (two per byte)
constexpr int kMaxStages = 8;
constexpr int kShrinkThreads = 256;
constexpr int kShrinkRows = 8;      // rows per register block in the shrink
constexpr int kShrinkKSub = 1024;   // K elements staged in shared memory per step
constexpr int kShrinkGroupRows = 64;  // rows per shrink block on the grouped (prefill) path
constexpr int kShrinkDecCh = 8;       // decode shrink: 16-byte chunks of A per lane and pass
constexpr int kShrinkDecKC = 256 * kShrinkDecCh;  // decode shrink: K per block (split width)
constexpr int kShrinkDecRows = 4;     // decode shrink: rows sharing one register load of A

// ============================================================== decode (n <= 256 rows) ======
//
// The shrink runs on the tensor cores inside the base GEMM: the A rows of the batch's distinct
// adapters are gathered, 8 rows per TMA box, into 128-row "A tiles" that multiply the same x
// k-blocks as the W tiles.  An 8-row group of one adapter's A rows is the unit of the gather.
constexpr int kGroupRows = 8;
constexpr int kTileGroups = kBM / kGroupRows;   // groups per A tile
constexpr int kDecMaxGroups = LORA_MAX_DECODE_ROWS * (LORA_MAX_RANK / kGroupRows);
// an A tile's k range is split over at most this many CTAs (its t partial sums, one per CTA)
constexpr int kDecMaxParts = 32;

struct AGroup {
    int32_t row;     // first A-slab row of the group (the gather's TMA row coordinate)
    int16_t q0, q1;  // sorted positions [q0, q1) whose rows use the adapter
    int16_t rbase;   // rank index of the group's first row
    int16_t rank;    // the adapter's rank for this projection
    int32_t pad_;
};
static_assert(sizeof(AGroup) == 16, "AGroup layout");

// What the finalize needs about one row's adapter for one projection, written by the prep.
struct RowInfo {
    const uint16_t *B;  // the adapter's B [d_out, rp] (bytes for int8 factors); null: base only
    int16_t rank, rp;
    int32_t g0;         // bf16 factors: the first gathered group of the row's adapter (its t parts)
};
static_assert(sizeof(RowInfo) == 16, "RowInfo layout");

// Decode tensor maps cover kps 64-wide k-blocks per box (a "k-step", one pipeline stage).  With
// kps = 1 they are 2-D ({k, row}); with kps = 2 they are 3-D views {64 elements, row, k-block}
// (k-block stride 128 bytes), whose box {64, rows, 2} lands as two k-blocks one after the other,
// each in the layout a 2-D box would give.
struct DecodeModule {
    CUtensorMap tmW;  // W [d_out, d_in] bf16, box {64, 128(, kps)}, 128B swizzle; int4 base: codes
                      // [d_out, d_in / 2] bytes, box {32, 128(, kps)}, no swizzle
    CUtensorMap tmX;  // x [n, d_in] bf16, box {64, nt(, kps)}, 128B swizzle
    CUtensorMap tmA;  // A slab [rows, d_in] bf16, box {64, 8(, kps)}, 128B swizzle (bf16 factors)
    CUtensorMap tmA128;  // the same slab, box {64, 128(, kps)}: an A tile whose groups are consecutive rows
    CUtensorMap tmAb[3]; // kps = 1: the same slab, box {64, 16 / 32 / 64}: 2 / 4 / 8 consecutive groups
    const float *w_scale;      // int4 base: [d_out] fp32 row scales
    const AGroup *groups;      // [kDecMaxGroups] this projection's gathered groups
    const int32_t *n_groups;   // device: number of groups
    const RowInfo *rowinfo;    // [n] per row: its adapter's B, rank, slot row
    const float *T;            // int8 factors: t rows [n][rpmax] from the CUDA-core shrink
    float *tpart;              // [kDecMaxParts][tp_rows][64] t partial sums of the A tiles
    float *tfin;               // [tp_rows][64] t = s * (sum of the parts), by each A tile's last CTA (t_fin = 0)
    int32_t *acount;           // [kDecMaxGroups / 16] CTAs done with each A tile (t_fin = 0; the finalize resets it)
    void *y;
    int32_t d_in, d_out, m_tiles;
    int32_t k_blocks;          // k-steps of a tile (kps k-blocks of 64 each)
    int32_t w_iter_begin;      // first (W tile, k-step) index of this projection
    int32_t w_tile_begin;      // first W tile of this projection
    int32_t a_runs;            // 1: tmA128 is valid (the slab has at least 128 rows)
    int32_t a_boxes;           // 1: tmAb is valid and kps = 1 (gathers go as one box per run of groups)
};

struct DecodeParams {
    DecodeModule mod[LORA_MAX_MODULES];
    int32_t n_mod;
    int32_t n;            // rows
    int32_t nt;           // MMA N: rows rounded up to 16 (<= 256)
    int32_t tp_rows;      // row stride of tpart
    int32_t n_cta;
    int32_t n_stages;
    int32_t kps;          // 64-wide k-blocks per pipeline stage (1 or 2)
    int32_t tmem_cols;
    int32_t w_iters;      // W tile k-steps of all projections (the W stream-K space)
    int32_t w_tiles;
    int32_t shrink_tc;    // 1: the shrink is the A tiles (bf16 factors); 0: t comes from T
    int32_t w4;
    int32_t y_bf16;
    int32_t i8;           // factors are int8 codes (B read as bytes in the expand)
    int32_t rpmax;        // row stride of T; the largest storage rank in the pool
    int32_t fin_nbuf;     // the finalize's B tile buffers (1 or 2)
    int32_t fin_buf;      // bytes of one
    float scale;
    const int32_t *perm;      // sorted position -> row
    const int32_t *rb_order;  // the finalize's row blocks (16 sorted positions each) in launch order; null: in order
    const int32_t *radapter;  // row -> validated adapter id (-1: base only)
    float *home;          // [w_tiles][kBM * nt] base pieces that start at k-block 0 of their tile
    float *ctaw;          // [n_cta][kBM * nt] base pieces that start inside their tile
    int32_t *err;         // [0] code, [1] detail
    uint64_t wait_ns;     // budget of one in-kernel wait
    int32_t w_first;      // 1: each CTA runs its W range before it waits for the kernel before it
    int32_t t_fin;        // 1: the finalize adds the A tiles' t parts; 0: each tile's last CTA does (tfin)
};
static_assert(sizeof(DecodeParams) <= 32764, "decode parameters exceed the kernel parameter space");

// The outputs (y) of the library's last forward on a stream.  Its kernels let the next kernel on the
// stream start before they finish, so a decode call reads its x before its griddepcontrol.wait only
// when x overlaps none of them.
struct ByteRange {
    uintptr_t lo, hi;  // [lo, hi)
};
void note_stream_outputs(cudaStream_t s, const ByteRange *r, int n);
bool overlaps_stream_outputs(cudaStream_t s, const ByteRange *r, int n);

// ========================================================== grouped rows (prefill) ==========
//
// The expand (delta = B_a t) of a tile runs from "B stages" that follow the tile's W k-blocks in
// the same TMA ring: a stage holds the 128-row slice of B of one slot (one adapter with a run of
// rows that use it) and those rows' t rows; the epilogue warps compute the dot products from
// shared memory into the tile's accumulator before its MMAs start.
constexpr int kPackSlots = 16;
constexpr int kStageHdrBytes = 512;  // slot header at the start of a B stage's X buffer
constexpr int kYBufBytes = 32768;    // epilogue y staging

// shared-memory slot header of a B stage, written by the producer, read by the epilogue
struct BSlotS {
    int32_t q0;       // first row of the slot
    int16_t nrows;
    int16_t rp;
    int16_t off;      // rank offset: the slot's B rows start at off * 128 * 2 bytes of the A buffer
    int16_t tstride;  // floats between consecutive t rows
    int32_t toff;     // first float of the slot's t rows in the stage's t area
};
struct BStageHdr {
    int32_t nslots;
    int32_t pad_[3];
    BSlotS slot[kPackSlots];
};
static_assert(sizeof(BStageHdr) <= kStageHdrBytes, "B stage header");

struct GemmModule {
    CUtensorMap tmW;  // W [d_out, d_in]: box {64, 128}, 128B swizzle
    CUtensorMap tmX;  // X [n, d_in]:    box {64, nt},  128B swizzle
    CUtensorMap tmY;  // y [n, d_out]:   box {128, 16}, fp32 or bf16, no swizzle (epilogue stores)
    void *y;
    const float *T;            // shrink result [n][rpmax]
    const PoolEntry *table;    // this module's entries [max_adapters]
    int32_t d_in, d_out;
    int32_t m_tiles, k_blocks;
    int32_t tile_begin;        // first global tile index of this module
};

struct GemmParams {
    GemmModule mod[LORA_MAX_MODULES];
    int32_t n_mod;
    int32_t n;             // rows
    int32_t nt;            // rows per chunk (MMA N), multiple of 16, <= 256
    int32_t n_chunks;
    int32_t n_cta;
    int32_t total_tiles;
    int32_t rpmax;         // T row stride
    int32_t y_bf16;
    int32_t n_stages;
    int32_t raster_group;  // W tiles per raster group (round robin)
    int32_t tmem_cols;
    int32_t ybuf_bytes;    // dedicated y staging in shared memory
    const int32_t *seg_start;
    const int32_t *seg_adapter;
    const int32_t *n_seg;
    const int32_t *chunk_seg0;  // first segment touching each row chunk
    const int32_t *chunk_nb;    // B stages (slots) of each row chunk
    int32_t pf_ch;              // rows per slot
    int32_t *err;          // [0] code, [1] detail
    uint64_t wait_ns;      // budget of one in-kernel wait
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
    int32_t by_segment;   // 1: one block per sorted position (decode); 0: one block per 64 rows
    int32_t max_units;
    int32_t ks_max;
    float scale;
    const int32_t *perm;  // null: identity
    const int32_t *seg_start;
    const int32_t *seg_adapter;
    const int32_t *n_seg;
    const int32_t *qadapter;                // decode: adapter of each sorted position
    float *partials;      // [n_mod][ks_max][n][rpmax]
    int32_t *counters;    // [n_mod][max_units]
    // int8 factors: A rows are int8 codes and t_j is multiplied by fold[m][row_off + j] (the
    // product of the rank row's A and B scales)
    int32_t i8;
    const float *fold[LORA_MAX_MODULES];
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
    int32_t *qadapter;                // decode: [n] adapter of each sorted position
    int32_t *radapter;                // decode: [n] validated adapter of each row
    // decode: the gathered A groups of every projection (null: not built)
    AGroup *groups[LORA_MAX_MODULES];
    int32_t *n_groups;                // [n_mod]
    RowInfo *rowinfo[LORA_MAX_MODULES];  // decode: [n] per row: its adapter's B, rank, slot row
    int32_t *rb_order;                // decode: [ceil(n / 16)] the finalize's row blocks, heaviest first (null: not built)
    // grouped rows: per row chunk of nt rows
    int32_t nt;
    int32_t pf_ch;
    int32_t *chunk_seg0;
    int32_t *chunk_nb;
};

static_assert(sizeof(GemmParams) <= 32764, "gemm parameters exceed the kernel parameter space");

// tensor maps (lora_api.cu): bf16 [rows, cols] operand, box {64, box_rows}, 128-byte swizzle (with
// kps = 2: the 3-D view {64, rows, cols / 64}, box {64, box_rows, 2}); and
// the output y [n, d_out] (fp32 or bf16), box {128, 16}, for the epilogue's TMA stores
int make_tmap(CUtensorMap *tm, const void *base, int64_t rows, int64_t cols, int box_rows, int kps = 1);
// bytes [rows, cols] (row-major), box {box_cols, box_rows}, no swizzle, 256-byte L2 promotion
int make_tmap_u8(CUtensorMap *tm, const void *base, int64_t rows, int64_t cols, int box_cols, int box_rows, int kps = 1);
int make_tmap_y(CUtensorMap *tm, void *y, int64_t n, int64_t d_out, bool bf16);

// launchers (lora_kernels.cu: grouped rows, shrink; decode_kernels.cu: decode)
cudaError_t launch_prep_decode(const PrepParams &p, cudaStream_t s);
cudaError_t launch_prep_segments(const PrepParams &p, cudaStream_t s);
cudaError_t launch_shrink(const ShrinkParams &p, int grid_x, int grid_y, cudaStream_t s);
cudaError_t launch_gemm(const GemmParams &p, size_t smem_bytes, cudaStream_t s);
cudaError_t launch_decode_gemm(const DecodeParams &p, size_t smem_bytes, cudaStream_t s);
void plan_decode_finalize(DecodeParams &dp, size_t *smem_bytes);
cudaError_t launch_decode_finalize(const DecodeParams &p, size_t smem_bytes, cudaStream_t s);
cudaError_t launch_table_write(PoolEntry *dst, PoolEntry value, cudaStream_t s);
// Up to kTableWritesMax table entries written by one launch (the entries ride in the parameters).
constexpr int kTableWritesMax = 64;
struct TableWrites {
    PoolEntry *dst[kTableWritesMax];
    PoolEntry v[kTableWritesMax];
    int32_t n;
};
cudaError_t launch_table_write_many(const TableWrites &w, cudaStream_t s);
// Packed loads: one item's factors from a device staging buffer into its pool rows, zero-padded
// to the storage rank, then its table entry.  Up to kPackedMax items per launch (parameters).
constexpr int kPackedMax = 96;
struct PackedJob {
    const uint8_t *srcA;  // bf16 [rank, d_in] in the staging buffer
    const uint8_t *srcB;  // bf16 [d_out, rank]
    PoolEntry *dst;       // the table entry to publish
    PoolEntry val;        // its value (val.A, val.B: the rows in the pool)
    int32_t d_in, d_out;
};
struct PackedJobs {
    PackedJob j[kPackedMax];
    int32_t n;
};
cudaError_t launch_packed_load(const PackedJobs &jobs, cudaStream_t s);
// TMEM buffers, stage count and shared memory of a gemm launch; false if no two stages fit
bool plan_gemm(GemmParams &gp, size_t *smem_bytes);
bool plan_decode_gemm(DecodeParams &dp, size_t *smem_bytes);
// grouped rows: positions per slot so that a slot's B rows, header and t rows fit the y buffer the
// epilogue copies a B stage into (and the t rows fit the stage's X buffer)
inline int pf_ch(int nt, int rpmax) {
    const int c = (kYBufBytes - kStageHdrBytes - kBM * rpmax * 2) / (rpmax * 4);
    return c < nt ? c : nt;
}
// decode: CTAs of the A-tile (shrink) space for `a_iters` k-blocks, so that an A tile of at most
// `kbn_max` k-blocks is shared by at most kDecMaxParts CTAs (every range is at least
// ceil(kbn_max / (kDecMaxParts - 1)) k-blocks long)
__host__ __device__ inline int decode_a_ctas(int a_iters, int kbn_max, int n_cta) {
    if (a_iters <= 0) return 0;
    const int lq = (kbn_max + kDecMaxParts - 2) / (kDecMaxParts - 1);
    int na = a_iters / (lq > 0 ? lq : 1);
    if (na > n_cta) na = n_cta;
    return na < 1 ? 1 : na;
}

// Every hot-path kernel is launched as a programmatic dependent of the one before it on the
// stream: it may start (and run its prologue) while that one drains, and waits for it with
// griddepcontrol.wait before reading anything it may have written.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
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
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// lora_api.cu: sets the string lora_last_cuda_error() returns on this thread
void set_last_error(const char *why);
inline void set_last_error(const std::string &why) { set_last_error(why.c_str()); }

}  // namespace lora
