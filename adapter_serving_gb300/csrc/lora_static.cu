// lora_static.cu -- lora_linear_forward_static: the decode forward for callers that must not
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all: a serving runtime that has already handed every
// byte of HBM to its own allocator (the KV cache and its own pre-sized LoRA buffers), where a
// stray cudaMalloc would fail or fragment memory that runtime accounts for; or code embedded in
// another framework whose allocation policy forbids raw device allocations.  Such callers also
// keep their adapters in their own fixed buffers instead of in a lora_pool.  This entry point
// serves them: the caller passes the inputs, the output and its stacked adapter factors, and
// every piece of per-call scratch (row grouping, shrink result and partial sums, stream-K
// partial tiles, counters, the factor table) lives in one file-scope device array, sized once,
// that each GPU loading this library holds until the process exits.  It runs the same row
// grouping, shrink and tcgen05 kernels as lora_linear_forward.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <string>

#include "lora_internal.h"

using namespace lora;

namespace {

// ---- limits of the static path and the scratch layout they imply -----------------------
constexpr int kStMaxRows = 128;       // decode rows per call
constexpr int kStMaxDin = 16384;      // shrink K splits: d_in / 2048 <= 8
constexpr int kStMaxDout = 32768;     // stream-K tile counters: d_out / 128 <= 256
constexpr int kStMaxAdapters = 4096;  // factor table entries
constexpr int kStMaxCta = 160;        // stream-K partial-tile slots
constexpr int kStKsMax = kStMaxDin / kShrinkDecKC;
constexpr int kStMaxUnits = LORA_MAX_DECODE_ROWS;  // shrink counter stride (one per segment)

constexpr size_t al(size_t v) { return (v + 255) & ~size_t(255); }
constexpr size_t kOffTable = 0;
constexpr size_t kOffPerm = al(kOffTable + sizeof(PoolEntry) * kStMaxAdapters);
constexpr size_t kOffSegStart = al(kOffPerm + 4 * 256);
constexpr size_t kOffSegAdapter = al(kOffSegStart + 4 * 272);
constexpr size_t kOffNSeg = al(kOffSegAdapter + 4 * 256);
constexpr size_t kOffQAdapter = al(kOffNSeg + 16);
constexpr size_t kOffErr = al(kOffQAdapter + 4 * 256);                     // from here up to kOffT:
constexpr size_t kOffShrinkCnt = al(kOffErr + 16);                // cleared at every call
constexpr size_t kOffT = al(kOffShrinkCnt + 4 * kStMaxUnits);  // packed t of the expand
constexpr size_t kOffPacks = al(kOffT + 4 * kPackedTFloats);
constexpr size_t kOffTpos = al(kOffPacks + sizeof(BPackG) * kMaxPacks);
constexpr size_t kOffNPacks = al(kOffTpos + 4 * LORA_MAX_DECODE_ROWS);
constexpr size_t kOffShrinkPart = al(kOffNPacks + 16);
constexpr size_t kOffGemmPart = al(kOffShrinkPart + 4 * (size_t)kStKsMax * kStMaxRows * LORA_MAX_RANK);
constexpr size_t kStaticBytes = al(kOffGemmPart + 4 * (size_t)kStMaxCta * 2 * kBM * kStMaxRows);
static_assert(kOffT % 256 == 0 && kOffShrinkPart % 256 == 0 && kOffGemmPart % 256 == 0, "alignment");
static_assert(kStaticBytes <= (24u << 20), "the static scratch stays at most 24 MiB");

}  // namespace

// The scratch itself.  Host code must never hand this name to a kernel: on the host it only
// stands for the symbol, so its device address is fetched with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_lora_static_scratch[kStaticBytes];

namespace {

std::mutex g_addr_mutex;
unsigned char *g_addr[64] = {};  // device address of the scratch, per device ordinal
int g_sms[64] = {};

__global__ void static_table_kernel(PoolEntry *table, const uint16_t *A, const uint16_t *B, int n_adapters,
                                    int rank, int d_in, int d_out) {
    const int a = blockIdx.x * blockDim.x + threadIdx.x;
    if (a < n_adapters)
        table[a] = PoolEntry{A + (size_t)a * rank * d_in, B + (size_t)a * d_out * rank, rank, rank, 0};
}

// Returns `status` and leaves the reason where lora_last_cuda_error() reads it.
int fail(int status, const std::string &why) {
    set_last_error(why);
    return status;
}

}  // namespace

extern "C" int lora_linear_forward_static(const void *x, const void *W, int32_t d_in, int32_t d_out,
                                          const int32_t *row_adapter_ids, int32_t n, const void *A_stack,
                                          const void *B_stack, int32_t n_adapters, int32_t rank, float scale,
                                          void *y, int32_t y_dtype, lora_stream_t stream) {
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (n == 0) return LORA_OK;
    if (!x || !W || !row_adapter_ids || !y || n < 0 || (n_adapters > 0 && (!A_stack || !B_stack)))
        return fail(LORA_EINVAL, "null pointer or negative row count");
    if (y_dtype != LORA_DTYPE_F32 && y_dtype != LORA_DTYPE_BF16) return fail(LORA_EINVAL, "y_dtype");
    if (d_in < 8 || d_out < 8 || d_in % 8 || d_out % 8) return fail(LORA_EINVAL, "d_in, d_out: multiples of 8");
    if (rank != 8 && rank != 16 && rank != 32 && rank != 64)
        return fail(LORA_EINVAL, "rank must be 8, 16, 32 or 64 (zero-pad other ranks)");
    if (n > kStMaxRows || d_in > kStMaxDin || d_out > kStMaxDout || n_adapters < 0 || n_adapters > kStMaxAdapters)
        return fail(LORA_EUNSUPPORTED, "exceeds the static scratch: n <= 128, d_in <= 16384, d_out <= 32768, "
                                       "n_adapters <= 4096");
    const void *ptrs[] = {x, W, y, A_stack, B_stack};
    for (const void *ptr : ptrs)
        if (ptr && (reinterpret_cast<uintptr_t>(ptr) & 15)) return fail(LORA_EINVAL, "pointers: 16-byte aligned");

    // set-up once per device: the scratch's device address
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(LORA_ECUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(LORA_EUNSUPPORTED, "device ordinal above 63");
    unsigned char *scratch;
    int num_sms;
    {
        std::lock_guard<std::mutex> lock(g_addr_mutex);
        if (!g_addr[dev]) {
            void *ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_lora_static_scratch);
            if (e != cudaSuccess)
                return fail(LORA_ECUDA, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e));
            int sms = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return fail(LORA_ECUDA, std::string("SM count: ") + cudaGetErrorString(e));
            g_addr[dev] = static_cast<unsigned char *>(ptr);
            g_sms[dev] = sms;
        }
        scratch = g_addr[dev];
        num_sms = std::min(g_sms[dev], kStMaxCta);
    }
    PoolEntry *table = reinterpret_cast<PoolEntry *>(scratch + kOffTable);
    int32_t *perm = reinterpret_cast<int32_t *>(scratch + kOffPerm);
    int32_t *seg_start = reinterpret_cast<int32_t *>(scratch + kOffSegStart);
    int32_t *seg_adapter = reinterpret_cast<int32_t *>(scratch + kOffSegAdapter);
    int32_t *n_seg = reinterpret_cast<int32_t *>(scratch + kOffNSeg);
    int32_t *err = reinterpret_cast<int32_t *>(scratch + kOffErr);
    int32_t *qadapter = reinterpret_cast<int32_t *>(scratch + kOffQAdapter);
    float *T = reinterpret_cast<float *>(scratch + kOffT);
    BPackG *packs = reinterpret_cast<BPackG *>(scratch + kOffPacks);
    int32_t *tpos = reinterpret_cast<int32_t *>(scratch + kOffTpos);
    int32_t *n_packs = reinterpret_cast<int32_t *>(scratch + kOffNPacks);
    const int nt = (n + 15) & ~15;

    // the previous call leaves its contents behind: zero the counters and the error word
    e = cudaMemsetAsync(scratch + kOffErr, 0, kOffT - kOffErr, s);
    if (e != cudaSuccess) return fail(LORA_ECUDA, std::string("clear counters: ") + cudaGetErrorString(e));
    if (n_adapters > 0) {
        static_table_kernel<<<(n_adapters + 127) / 128, 128, 0, s>>>(table, static_cast<const uint16_t *>(A_stack),
                                                                    static_cast<const uint16_t *>(B_stack),
                                                                    n_adapters, rank, d_in, d_out);
        if ((e = cudaGetLastError()) != cudaSuccess)
            return fail(LORA_ECUDA, std::string("table kernel: ") + cudaGetErrorString(e));
    }

    PrepParams pp{};
    pp.ids = row_adapter_ids;
    pp.n = n;
    pp.max_adapters = n_adapters;
    pp.n_mod = 1;
    pp.table[0] = table;
    pp.perm = perm;
    pp.seg_start = seg_start;
    pp.seg_adapter = seg_adapter;
    pp.n_seg = n_seg;
    pp.err = err;
    pp.qadapter = qadapter;
    pp.packs[0] = packs;
    pp.tpos[0] = tpos;
    pp.n_packs = n_packs;
    pp.pack_ranks = kPackRanks;
    pp.pack_ch = pack_ch(nt, kPackRanks);
    if ((e = launch_prep_decode(pp, s)) != cudaSuccess)
        return fail(LORA_ECUDA, std::string("prep kernel: ") + cudaGetErrorString(e));

    const int rpmax = rank;
    ShrinkParams sp{};
    sp.n_mod = 1;
    sp.n = n;
    sp.rpmax = rpmax;
    sp.by_segment = 1;
    sp.max_units = kStMaxUnits;
    sp.ks_max = kStKsMax;
    sp.scale = scale;
    sp.perm = perm;
    sp.seg_start = seg_start;
    sp.seg_adapter = seg_adapter;
    sp.n_seg = n_seg;
    sp.qadapter = qadapter;
    sp.partials = reinterpret_cast<float *>(scratch + kOffShrinkPart);
    sp.counters = reinterpret_cast<int32_t *>(scratch + kOffShrinkCnt);
    sp.x[0] = static_cast<const uint16_t *>(x);
    sp.table[0] = table;
    sp.T[0] = T;
    sp.tpos[0] = tpos;
    sp.d_in[0] = d_in;
    sp.kc[0] = std::min(kShrinkDecKC, d_in);
    sp.ksplit[0] = (d_in + sp.kc[0] - 1) / sp.kc[0];
    sp.split_begin[0] = 0;
    sp.split_begin[1] = sp.ksplit[0];
    if ((e = launch_shrink(sp, n, sp.ksplit[0], s)) != cudaSuccess)
        return fail(LORA_ECUDA, std::string("shrink kernel: ") + cudaGetErrorString(e));

    GemmParams gp;
    memset(&gp, 0, sizeof gp);
    gp.n_mod = 1;
    gp.n = n;
    gp.nt = nt;
    gp.n_chunks = 1;
    gp.decode = 1;
    gp.stream_k = 1;
    gp.rpmax = rpmax;
    gp.y_bf16 = y_dtype == LORA_DTYPE_BF16 ? 1 : 0;
    gp.raster_group = 8;
    GemmModule &gm = gp.mod[0];
    if (make_tmap(&gm.tmW, W, d_out, d_in, kBM) || make_tmap(&gm.tmX, x, n, d_in, gp.nt) ||
        make_tmap_y(&gm.tmY, y, n, d_out, y_dtype == LORA_DTYPE_BF16))
        return LORA_ECUDA;  // the reason is already recorded
    gm.y = y;
    gm.T = T;
    gm.table = table;
    gm.d_in = d_in;
    gm.d_out = d_out;
    gm.m_tiles = (d_out + kBM - 1) / kBM;
    gm.k_blocks = (d_in + kBK - 1) / kBK;
    gm.iter_begin = 0;
    gm.tile_begin = 0;
    gm.packs = packs;
    gp.total_tiles = gm.m_tiles;
    gp.total_iters = (int64_t)gm.m_tiles * gm.k_blocks;
    gp.n_cta = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms, gp.total_iters / 4));
    gp.n_packs = n_packs;
    gp.pack_ch = pack_ch(nt, kPackRanks);
    size_t smem = 0;
    if (!plan_gemm(gp, &smem)) return fail(LORA_EUNSUPPORTED, "no two pipeline stages fit shared memory");
    gp.perm = perm;
    gp.seg_start = seg_start;
    gp.seg_adapter = seg_adapter;
    gp.n_seg = n_seg;
    gp.partials = reinterpret_cast<float *>(scratch + kOffGemmPart);
    gp.err = err;
    if ((e = launch_gemm(gp, smem, s)) != cudaSuccess)
        return fail(LORA_ECUDA, std::string("gemm kernel: ") + cudaGetErrorString(e));
    if ((e = launch_finalize(gp, s)) != cudaSuccess)  // split tiles' pieces -> y
        return fail(LORA_ECUDA, std::string("finalize kernel: ") + cudaGetErrorString(e));
    return LORA_OK;
}
