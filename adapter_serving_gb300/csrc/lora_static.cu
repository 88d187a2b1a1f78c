// lora_static.cu -- lora_linear_forward_static: the decode forward for callers that must not
// allocate device memory.
//
// Some callers cannot call cudaMalloc at all: a serving runtime that has already handed every
// byte of HBM to its own allocator (the KV cache and its own pre-sized LoRA buffers), where a
// stray cudaMalloc would fail or fragment memory that runtime accounts for; or code embedded in
// another framework whose allocation policy forbids raw device allocations.  Such callers also
// keep their adapters in their own fixed buffers instead of in a lora_pool.  This entry point
// serves them: the caller passes the inputs, the output and its stacked adapter factors, and
// every piece of per-call scratch (row grouping, the A gather list, the shrink's partial t sums,
// the base pieces of the stream-K split, the factor table) lives in one file-scope device array,
// sized once, that each GPU loading this library holds until the process exits.  It runs the same
// prep, tcgen05 gemm and finalize kernels as lora_linear_forward.
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
constexpr int kStMaxDout = 16384;     // one base-piece slot per 128-row tile of W: d_out / 128 <= 128
constexpr int kStMaxAdapters = 4096;  // factor table entries
constexpr int kStMaxCta = 160;        // base pieces that start inside a tile: one slot per CTA
constexpr int kStMaxTiles = kStMaxDout / kBM;
constexpr int kStNt = kStMaxRows;     // MMA N for the largest batch

constexpr size_t al(size_t v) { return (v + 255) & ~size_t(255); }
constexpr size_t kOffTable = 0;
constexpr size_t kOffPerm = al(kOffTable + sizeof(PoolEntry) * kStMaxAdapters);
constexpr size_t kOffSegStart = al(kOffPerm + 4 * (kStMaxRows + 1));
constexpr size_t kOffSegAdapter = al(kOffSegStart + 4 * (kStMaxRows + 2));
constexpr size_t kOffNSeg = al(kOffSegAdapter + 4 * (kStMaxRows + 1));
constexpr size_t kOffQAdapter = al(kOffNSeg + 16);
constexpr size_t kOffRAdapter = al(kOffQAdapter + 4 * (kStMaxRows + 1));
constexpr size_t kOffGroups = al(kOffRAdapter + 4 * (kStMaxRows + 1));
constexpr size_t kOffNGroups = al(kOffGroups + sizeof(AGroup) * kStMaxRows * (LORA_MAX_RANK / kGroupRows));
constexpr size_t kOffRowInfo = al(kOffNGroups + 16);
constexpr size_t kOffErr = al(kOffRowInfo + sizeof(RowInfo) * kStMaxRows);  // cleared at every call
constexpr size_t kOffTpart = al(kOffErr + 16);
constexpr size_t kOffHome = al(kOffTpart + 4 * (size_t)kDecMaxParts * kStMaxRows * LORA_MAX_RANK);
constexpr size_t kOffCtaw = al(kOffHome + 4 * (size_t)kStMaxTiles * kBM * kStNt);
constexpr size_t kStaticBytes = al(kOffCtaw + 4 * (size_t)kStMaxCta * kBM * kStNt);
static_assert(kOffTpart % 256 == 0 && kOffHome % 256 == 0 && kOffCtaw % 256 == 0, "alignment");
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
        table[a] = PoolEntry{A + (size_t)a * rank * d_in, B + (size_t)a * d_out * rank, rank, rank, (int64_t)a * rank};
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
    if (n > kStMaxRows || d_out > kStMaxDout || n_adapters < 0 || n_adapters > kStMaxAdapters)
        return fail(LORA_EUNSUPPORTED, "exceeds the static scratch: n <= 128, d_out <= 16384, n_adapters <= 4096");
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
    int32_t *err = reinterpret_cast<int32_t *>(scratch + kOffErr);
    const int nt = (n + 15) & ~15;

    // the previous call leaves its contents behind: clear the error word (everything else is
    // written before it is read)
    e = cudaMemsetAsync(scratch + kOffErr, 0, 16, s);
    if (e != cudaSuccess) return fail(LORA_ECUDA, std::string("clear the error word: ") + cudaGetErrorString(e));
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
    pp.seg_start = reinterpret_cast<int32_t *>(scratch + kOffSegStart);
    pp.seg_adapter = reinterpret_cast<int32_t *>(scratch + kOffSegAdapter);
    pp.n_seg = reinterpret_cast<int32_t *>(scratch + kOffNSeg);
    pp.err = err;
    pp.qadapter = reinterpret_cast<int32_t *>(scratch + kOffQAdapter);
    pp.radapter = reinterpret_cast<int32_t *>(scratch + kOffRAdapter);
    pp.groups[0] = reinterpret_cast<AGroup *>(scratch + kOffGroups);
    pp.n_groups = reinterpret_cast<int32_t *>(scratch + kOffNGroups);
    pp.rowinfo[0] = reinterpret_cast<RowInfo *>(scratch + kOffRowInfo);
    if ((e = launch_prep_decode(pp, s)) != cudaSuccess)
        return fail(LORA_ECUDA, std::string("prep kernel: ") + cudaGetErrorString(e));

    DecodeParams dp;
    memset(&dp, 0, sizeof dp);
    dp.n_mod = 1;
    dp.n = n;
    dp.nt = nt;
    dp.tp_rows = kStMaxRows;
    dp.shrink_tc = 1;
    dp.y_bf16 = y_dtype == LORA_DTYPE_BF16 ? 1 : 0;
    dp.rpmax = rank;
    dp.scale = scale;
    dp.perm = perm;
    dp.radapter = pp.radapter;
    dp.home = reinterpret_cast<float *>(scratch + kOffHome);
    dp.ctaw = reinterpret_cast<float *>(scratch + kOffCtaw);
    dp.err = err;
    dp.wait_ns = kWaitBudgetNs;
    DecodeModule &dm = dp.mod[0];
    dp.kps = (d_in % 64 == 0) ? 2 : 1;  // two k-blocks per pipeline stage where d_in allows
    // the stacked A factors are the slab the A tiles gather from: adapter a's rows start at a * rank
    const int64_t a_rows = n_adapters > 0 ? (int64_t)n_adapters * rank : kGroupRows;
    if (make_tmap(&dm.tmW, W, d_out, d_in, kBM, dp.kps) || make_tmap(&dm.tmX, x, n, d_in, nt, dp.kps) ||
        make_tmap(&dm.tmA, n_adapters > 0 ? A_stack : W, a_rows, d_in, kGroupRows, dp.kps))
        return LORA_ECUDA;  // the reason is already recorded
    dm.a_runs = 0;
    dm.a_boxes = 0;
    if (a_rows >= kBM) {  // A tiles of consecutive adapters' rows: one 128-row box
        if (make_tmap(&dm.tmA128, A_stack, a_rows, d_in, kBM, dp.kps)) return LORA_ECUDA;
        dm.a_runs = 1;
    }
    dm.groups = pp.groups[0];
    dm.n_groups = pp.n_groups;
    dm.rowinfo = pp.rowinfo[0];
    dm.tpart = reinterpret_cast<float *>(scratch + kOffTpart);
    dp.t_fin = 1;  // the finalize adds the A tiles' t parts (no counters in the scratch)
    dm.y = y;
    dm.d_in = d_in;
    dm.d_out = d_out;
    dm.m_tiles = (d_out + kBM - 1) / kBM;
    dm.k_blocks = ((d_in + kBK - 1) / kBK + dp.kps - 1) / dp.kps;  // k-steps
    dp.w_tiles = dm.m_tiles;
    dp.w_iters = dm.m_tiles * dm.k_blocks;
    dp.n_cta = std::max(1, std::min(num_sms, dp.w_iters / 4));
    size_t smem = 0;
    if (!plan_decode_gemm(dp, &smem)) return fail(LORA_EUNSUPPORTED, "no two pipeline stages fit shared memory");
    if ((e = launch_decode_gemm(dp, smem, s)) != cudaSuccess)
        return fail(LORA_ECUDA, std::string("gemm kernel: ") + cudaGetErrorString(e));
    size_t fsmem = 0;
    plan_decode_finalize(dp, &fsmem);
    if ((e = launch_decode_finalize(dp, fsmem, s)) != cudaSuccess)  // pieces + expand -> y
        return fail(LORA_ECUDA, std::string("finalize kernel: ") + cudaGetErrorString(e));
    const uintptr_t ylo = reinterpret_cast<uintptr_t>(y);
    const ByteRange yr{ylo, ylo + (uintptr_t)((size_t)n * d_out * (y_dtype == LORA_DTYPE_BF16 ? 2 : 4))};
    note_stream_outputs(s, &yr, 1);
    return LORA_OK;
}
