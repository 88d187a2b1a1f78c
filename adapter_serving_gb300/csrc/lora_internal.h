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
// int4 base weights: converter warps unpack each W k-block's codes into the bf16 tile the MMA reads
constexpr int kConvWarps = 2;
constexpr int kGemmThreadsW4 = kGemmThreads + 32 * kConvWarps;
constexpr int kW4RawBytes = kBM * kBK / 2;  // packed codes of one W k-block (two per byte)
constexpr int kMaxWin = 256;        // segments one tile's expand can touch (= max rows per tile)
constexpr int kMaxStages = 8;
constexpr int kShrinkThreads = 256;
constexpr int kShrinkRows = 8;      // rows per register block in the shrink
constexpr int kShrinkKSub = 1024;   // K elements staged in shared memory per step
constexpr int kShrinkGroupRows = 64;  // rows per shrink block on the grouped (prefill) path
constexpr int kShrinkDecCh = 8;       // decode shrink: 16-byte chunks of A per lane and pass
constexpr int kShrinkDecKC = 256 * kShrinkDecCh;  // decode shrink: K per block (split width)
constexpr int kShrinkDecRows = 4;     // decode shrink: rows sharing one register load of A

// ---- expand stages --------------------------------------------------------------------
// The expand (delta = B_a t) of a tile runs from "B stages" that follow the tile's W k-blocks in
// the same TMA ring: a stage holds the 128-row slices of B of a group of slots (a slot is one
// adapter with a run of positions that use it) and those positions' t rows; the epilogue warps
// compute the dot products from shared memory into the tile's TMEM delta buffer.

// storage ranks per B stage: as many 128-row B slices as the stage's 16 KiB A buffer holds
constexpr int kPackRanks = 64;       // bf16 factors
constexpr int kPackRanksI8 = 128;    // int8 factors
constexpr int kPackSlots = kPackRanksI8 / 8;
constexpr int kStageHdrBytes = 512;  // slot header at the start of a B stage's X buffer
constexpr int kYBufBytes = 32768;    // epilogue y staging

// decode: one group of slots ("pack"), written by prep, read by the TMA producer
struct BSlotG {
    const uint16_t *B;  // adapter's B for this module, [d_out, rp]
    uint16_t q0;        // first sorted position of the slot
    uint8_t nrows;      // positions in the slot (<= pack_ch)
    uint8_t rp;         // storage rank
    uint8_t off;        // rank offset within the pack
    uint8_t pad_[3];
};
static_assert(sizeof(BSlotG) == 16, "BSlotG layout");
struct BPackG {
    int32_t tbegin;   // first float of the pack's t rows in the module's packed T
    int32_t tfloats;  // floats of t rows
    int32_t nslots;
    int32_t pad_;
    BSlotG slot[kPackSlots];
};
static_assert(sizeof(BPackG) == 16 * (1 + kPackSlots), "BPackG layout");

// shared-memory slot header of a B stage, written by the producer, read by the epilogue
struct BSlotS {
    int32_t q0;       // first position (decode: sorted position; grouped rows: row)
    int16_t nrows;
    int16_t rp;
    int16_t off;      // rank offset: the slot's B rows start at off * 128 * (element bytes) of the A buffer
    int16_t tstride;  // floats between consecutive t rows
    int32_t toff;     // first float of the slot's t rows in the stage's t area
};
struct BStageHdr {
    int32_t nslots;
    int32_t singles8;  // every slot has rank 8 and one row (the epilogue's fast path)
    int32_t pad_[2];
    BSlotS slot[kPackSlots];
};
static_assert(sizeof(BStageHdr) <= kStageHdrBytes, "B stage header");

// rows per decode slot: the t rows of a full pack (pack_ranks fp32 per row) must fit the X buffer
// (nt * 128 bytes) after the header
__host__ __device__ constexpr int pack_ch(int nt, int pack_ranks) {
    return (nt * 128 - kStageHdrBytes) / (pack_ranks * 4) < 8 ? (nt * 128 - kStageHdrBytes) / (pack_ranks * 4) : 8;
}
// packs of one module (decode, n <= 256 rows): at most one per slot
constexpr int kMaxPacks = LORA_MAX_DECODE_ROWS + LORA_MAX_DECODE_ROWS / 7 + 1;
// packed t of one module: pack_ch floats per rank unit, 64 units per pack
constexpr size_t kPackedTFloats = (size_t)8 * kPackRanks * kMaxPacks;

struct GemmModule {
    CUtensorMap tmW;  // W [d_out, d_in]: box {64, 128}, 128B swizzle
    CUtensorMap tmX;  // X [n, d_in]:    box {64, nt},  128B swizzle
    CUtensorMap tmY;  // y [n, d_out]:   box {128, 16}, fp32 or bf16, no swizzle (epilogue stores)
    // int4 base (GemmParams::w4): tmW is the packed codes [d_out, d_in / 2] bytes, box {32, 128},
    // no swizzle (its 256-byte L2 promotion brings each row's next k-blocks into L2 with the first)
    const float *w_scale;      // int4 base: [d_out] fp32 row scales
    void *y;
    const float *T;            // shrink result: decode packed per pack, grouped rows [n][rpmax]
    const PoolEntry *table;    // this module's entries [max_adapters]
    const BPackG *packs;       // decode: this module's packs
    int32_t d_in, d_out;
    int32_t m_tiles, k_blocks;
    int64_t iter_begin;        // flattened (tile, W k-block) index where this module starts
    int32_t tile_begin;        // first global tile index of this module
    int32_t npk_index;         // decode: this module's entry of GemmParams::n_packs
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
    int64_t total_iters;       // W k-blocks of all tiles (the stream-K space)
    int32_t rpmax;         // T row stride
    int32_t y_bf16;
    int32_t i8;            // factors are int8 codes (B stages carry 1-byte elements)
    int32_t w4;            // base weights are int4 codes with one fp32 scale per output row (decode)
    int32_t n_stages;
    int32_t raster_group;  // W tiles per raster group (round robin)
    int32_t tmem_cols;
    int32_t n_acc;         // accumulator + delta buffer pairs in TMEM (2 when 4 * nt <= 512, else 1)
    int32_t ybuf_bytes;    // dedicated y staging in shared memory (0: stage buffers / plain stores)
    const int32_t *perm;
    const int32_t *seg_start;
    const int32_t *seg_adapter;
    const int32_t *n_seg;
    const int32_t *n_packs;     // decode: [n_mod] B stages per tile of each module
    const int32_t *chunk_seg0;  // grouped rows: first segment touching each row chunk
    const int32_t *chunk_nb;    // grouped rows: B stages (slots) of each row chunk
    int32_t pack_ch;            // decode: positions per slot
    int32_t pf_ch;              // grouped rows: positions per slot
    float *partials;       // [n_cta][2][kBM * nt] stream-K pieces (a CTA's first and later item)
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
    const int32_t *tpos[LORA_MAX_MODULES];  // decode: where position q's t row starts in T
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
    // decode: expand packs per module
    BPackG *packs[LORA_MAX_MODULES];
    int32_t *tpos[LORA_MAX_MODULES];  // [n] float offset of position q's t row in the packed T
    int32_t *n_packs;                 // [n_mod]
    int32_t pack_ch;
    int32_t pack_ranks;               // decode: storage ranks per pack (kPackRanks or kPackRanksI8)
    // grouped rows: per row chunk of nt rows
    int32_t nt;
    int32_t pf_ch;
    int32_t *chunk_seg0;
    int32_t *chunk_nb;
};

static_assert(sizeof(GemmParams) <= 32764, "gemm parameters exceed the kernel parameter space");

// tensor maps (lora_api.cu): bf16 [rows, cols] operand, box {64, box_rows}, 128-byte swizzle; and
// the output y [n, d_out] (fp32 or bf16), box {128, 16}, for the epilogue's TMA stores
int make_tmap(CUtensorMap *tm, const void *base, int64_t rows, int64_t cols, int box_rows);
// bytes [rows, cols] (row-major), box {box_cols, box_rows}, no swizzle, 256-byte L2 promotion
int make_tmap_u8(CUtensorMap *tm, const void *base, int64_t rows, int64_t cols, int box_cols, int box_rows);
int make_tmap_y(CUtensorMap *tm, void *y, int64_t n, int64_t d_out, bool bf16);

// launchers (lora_kernels.cu)
cudaError_t launch_prep_decode(const PrepParams &p, cudaStream_t s);
cudaError_t launch_prep_segments(const PrepParams &p, cudaStream_t s);
cudaError_t launch_shrink(const ShrinkParams &p, int grid_x, int grid_y, cudaStream_t s);
cudaError_t launch_gemm(const GemmParams &p, size_t smem_bytes, cudaStream_t s);  // p.i8, p.w4 pick the instantiation
cudaError_t launch_finalize(const GemmParams &p, cudaStream_t s);  // decode: sum split tiles' pieces into y
cudaError_t launch_table_write(PoolEntry *dst, PoolEntry value, cudaStream_t s);
size_t gemm_smem_bytes(int nt, int n_stages, int ybuf_bytes, bool w4 = false);
// TMEM buffers, stage count and shared memory of a gemm launch; false if no two stages fit
bool plan_gemm(GemmParams &gp, size_t *smem_bytes);
// decode packs of one module: at most one pack per slot
inline int pack_cap(int n, int ch) { return n + (n + ch - 1) / ch + 1; }
// grouped rows: positions per slot so that a slot's B rows, header and t rows fit the y buffer the
// epilogue copies a B stage into (and the t rows fit the stage's X buffer)
inline int pf_ch(int nt, int rpmax) {
    const int c = (kYBufBytes - kStageHdrBytes - kBM * rpmax * 2) / (rpmax * 4);
    return c < nt ? c : nt;
}

// lora_api.cu: sets the string lora_last_cuda_error() returns on this thread
void set_last_error(const char *why);
inline void set_last_error(const std::string &why) { set_last_error(why.c_str()); }

}  // namespace lora
