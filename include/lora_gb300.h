/*
 * lora_gb300.h -- C ABI of the GB300 (sm_103a) multi-tenant LoRA adapted linear layer.
 *
 * The operation.  One adapted linear layer over a batch whose rows each carry their own
 * adapter id:
 *
 *     y_i = W x_i + s * B_a (A_a x_i),      a = adapter of row i,
 *
 * with W: [d_out, d_in], A_a: [r, d_in], B_a: [d_out, r]
 * ("m07 -- Multi-Adapter (LoRA) Serving", section 2 "Scale Numbers", the factor shapes, and
 * section 6 "Deep Dive A: Batching Heterogeneous Adapters", y = Wx + (B.A)x.(alpha/r) -- the
 * scale s is passed in directly; "12. Adapter Serving and Multi-Tenant Customization",
 * section "What an adapter adds to a forward pass").  A row whose adapter id is -1 is a
 * base-only request and gets W x_i alone ("12. Adapter Serving ...", section "Scheduling
 * with adapter awareness", the base-only group).  The base projection reads W once per call
 * for the whole batch; every DISTINCT adapter's factors are read once per call ("m07",
 * section 6, "The cost is bandwidth, not compute").  Factors are gathered inside the kernels
 * through a device-side indirection table, so a captured CUDA graph stays valid across
 * loads ("12. Adapter Serving ...", section "CUDA graphs": adapter addresses are read from a
 * buffer, not baked into the graph).  Factor storage is paged ("LoRA, quotas and noisy
 * neighbours", section "Adapter weights and KV in one pool"; "12. Adapter Serving ...",
 * section "S-LoRA's unified paging").
 *
 * Conventions for every entry point:
 *  - Return value: LORA_OK (0) or a negative LORA_E* status; nothing aborts the process and
 *    no kernel traps.  lora_status_string() names a status.
 *  - Tensors are dense row-major; bf16 means IEEE bfloat16 (16-bit) values.
 *  - "device" pointers are CUDA device memory (or managed memory) of the current device;
 *    "host or device" pointers may be either (copied with UVA).  Pointers passed to the
 *    forward calls must be 16-byte aligned.
 *  - Caller-owned buffers are only borrowed for the duration of the call (for asynchronous
 *    calls: until the work queued on `stream` has run).  The pool owns its factor pages,
 *    its table and its workspace.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls that take a
 *    stream are asynchronous with respect to the host.  All calls on one pool must be
 *    ordered with each other (one stream, or explicit events): the pool's workspace and
 *    table are shared by its calls.
 *  - The forward kernels are programmatic dependents of the kernel before them on the stream
 *    (they may start while it drains), and a decode call streams its W tiles -- reading W and
 *    x -- before it waits for that kernel.  An x that the library's previous forward on the
 *    same stream wrote is detected, and that call waits first.  An x or W produced by another
 *    library's kernel that itself lets dependents start early
 *    (cudaTriggerProgrammaticLaunchCompletion) before it has written them must be separated
 *    from the forward by an event or a stream synchronisation.
 *  - Shapes: d_in and d_out must be multiples of 8; 1 <= rank <= 64.
 */
#ifndef LORA_GB300_H
#define LORA_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct lora_pool lora_pool;
typedef struct CUstream_st *lora_stream_t; /* == cudaStream_t */

/* status codes */
#define LORA_OK 0
#define LORA_EINVAL (-1)       /* bad argument: null pointer, shape, rank, id out of range */
#define LORA_ENOTLOADED (-2)   /* adapter (or a module of it) is not resident */
#define LORA_ENOMEM (-3)       /* no free pages in the pool, or a device allocation failed */
#define LORA_ECUDA (-5)        /* a CUDA runtime call failed (see lora_last_cuda_error) */
#define LORA_EUNSUPPORTED (-6) /* valid request the library does not handle (see each call) */
#define LORA_EDEVICE (-7)      /* a kernel recorded an error (see lora_last_device_error) */
#define LORA_EPINNED (-8)      /* the adapter cache's pinning guard refuses a new adapter */

/* output element types */
#define LORA_DTYPE_F32 0
#define LORA_DTYPE_BF16 1

#define LORA_MAX_MODULES 8     /* projections per pool and per layer call */
#define LORA_MAX_RANK 64
#define LORA_PAGE_ROWS 64      /* rank-vectors per page */
#define LORA_MAX_DECODE_ROWS 256

/* device-side error codes reported by lora_last_device_error */
#define LORA_DEVERR_NONE 0
#define LORA_DEVERR_BAD_ADAPTER 1 /* row/segment names an id outside [-1, max_adapters) */
#define LORA_DEVERR_NOT_LOADED 2  /* row/segment names an adapter not resident for a module */
#define LORA_DEVERR_TIMEOUT 3     /* a bounded in-kernel wait gave up (kernel returned early) */
#define LORA_DEVERR_BAD_SEGMENTS 4 /* segment table not increasing / not covering the rows */

/*
 * Pool geometry, fixed at creation.
 *  n_modules       number of projections (1..LORA_MAX_MODULES)
 *  d_in, d_out     [n_modules] host arrays: projection m maps d_in[m] -> d_out[m]
 *  max_adapters    adapter ids are 0 .. max_adapters-1
 *  max_rank        largest rank a load may use (1..64)
 *  pages           [n_modules] host array or NULL: number of 64-row pages reserved for
 *                  module m.  A rank-r factor pair takes ceil-pow2(max(r, 8)) rows of one
 *                  page (A rows d_in wide, B stored as [d_out, rows]).  NULL reserves
 *                  enough for every adapter at max_rank.
 *  max_rows        largest row count (decode rows or prefill tokens) one forward may pass;
 *                  sizes the workspace.
 *  factor_dtype    LORA_FACTOR_BF16 (0: bf16 factors, lora_pool_load) or LORA_FACTOR_I8 (int8
 *                  codes with one fp32 scale per rank row of A and of B transposed,
 *                  lora_pool_load_i8; decode forwards only)
 */
typedef struct {
    int32_t n_modules;
    const int32_t *d_in;
    const int32_t *d_out;
    int32_t max_adapters;
    int32_t max_rank;
    const int64_t *pages;
    int32_t max_rows;
    int32_t factor_dtype;
} lora_pool_desc;

#define LORA_FACTOR_BF16 0
#define LORA_FACTOR_I8 1

/*
 * lora_pool_create -- allocate the paged factor pool, its (pointer, rank) table and the
 * workspace on the current CUDA device.  *out receives the pool.  Synchronous.
 * Errors: EINVAL (bad desc), ENOMEM, ECUDA.
 */
int lora_pool_create(const lora_pool_desc *desc, lora_pool **out);

/* lora_pool_destroy -- synchronize the device and free everything the pool owns. */
int lora_pool_destroy(lora_pool *pool);

/*
 * lora_pool_load -- make adapter `adapter_id` resident for projection `module`.
 *  A     host or device bf16 [rank, d_in]     (copied; caller keeps ownership)
 *  B     host or device bf16 [d_out, rank]
 * Pages are taken from the module's free list; the factors are copied in on `stream`
 * (zero-padded to the storage rank) and the table entry is written on `stream` after the
 * copy, so forwards queued later on `stream` see the adapter.  Loading an id that is
 * already resident for this module replaces it.  Host-side bookkeeping is synchronous.
 * Errors: EINVAL (id, module, rank, null), ENOMEM (no free rows), ECUDA.
 */
int lora_pool_load(lora_pool *pool, int32_t adapter_id, int32_t module, const void *A,
                   const void *B, int32_t rank, lora_stream_t stream);

/*
 * lora_pool_load_many -- lora_pool_load for n items in one call: each item's copies are queued
 * on `stream` in item order, and the table entries are then written by one kernel launch per 64
 * items instead of one per item (the host cost of a load is its launches).  Items apply in order,
 * so a later item for the same (adapter, module) replaces an earlier one.  The call stops at the
 * first item that fails: the items before it are loaded and published, *n_done (may be null)
 * counts them, and the failing item leaves its (adapter, module) entry as lora_pool_load would:
 * untouched for EINVAL (bad id, module, rank or pointer), cleared for ENOMEM (no free rows).
 */
typedef struct {
    int32_t adapter;
    int32_t module;
    int32_t rank;
    const void *A;  /* host or device bf16 [rank, d_in] */
    const void *B;  /* host or device bf16 [d_out, rank] */
} lora_load_item;
int lora_pool_load_many(lora_pool *pool, int32_t n, const lora_load_item *items, int32_t *n_done,
                        lora_stream_t stream);

/*
 * lora_pool_load_packed -- many bf16 loads from one packed host buffer: a single host->device copy
 * of the whole blob into the caller's device staging buffer, then one kernel (per 96 items) that
 * scatters every item's factors into its pool rows, zero-padded to the storage rank, and
 * publishes its table entry.  Two launches however many items: the form for loading a cold
 * adapter's factors for a layer while other layers run (see lora_layer_gate).
 *  host_blob    host bf16 factors, pinned for an asynchronous copy; item i's A ([rank, d_in],
 *               row-major) starts at byte a_offset (a multiple of 16), its B ([d_out, rank])
 *               at b_offset (even)
 *  dev_staging  device buffer of at least blob_bytes, 16-byte aligned, the caller's; it must not
 *               be written while the call's kernels may still read it (same stream: in order)
 * Every item is checked before anything is queued (EINVAL: bad id, module, rank or offset; then
 * nothing is loaded).  Items then apply in order; ENOMEM (no free rows) stops at that item, whose
 * entry is left cleared; *n_done (may be null) counts the items loaded.  Same visibility as
 * lora_pool_load: forwards queued later on `stream` see the adapters.
 */
typedef struct {
    int32_t adapter;
    int32_t module;
    int32_t rank;
    int32_t pad_;
    int64_t a_offset;
    int64_t b_offset;
} lora_packed_item;
int lora_pool_load_packed(lora_pool *pool, int32_t n, const lora_packed_item *items, const void *host_blob,
                          void *dev_staging, int64_t blob_bytes, int32_t *n_done, lora_stream_t stream);

/*
 * lora_pool_unload_many -- lora_pool_unload for n adapters, the table entries cleared by one
 * kernel launch per 64.  Stops at the first id that is out of range (EINVAL) or resident in no
 * module (ENOTLOADED); *n_done (may be null) counts the adapters unloaded.
 */
int lora_pool_unload_many(lora_pool *pool, int32_t n, const int32_t *adapter_ids, int32_t *n_done,
                          lora_stream_t stream);

/*
 * lora_pool_unload -- release adapter `adapter_id` from every module.  The table entries
 * are cleared on `stream`; the rows return to the free lists at once, so a later load may
 * reuse them: order it after every forward that still reads the adapter.
 * Errors: EINVAL, ENOTLOADED (resident in no module).
 */
int lora_pool_unload(lora_pool *pool, int32_t adapter_id, lora_stream_t stream);

/*
 * lora_pool_query -- host-side view of one table entry: *rank (0 if not resident) and
 * *row_offset (first pool row of its pages).  Either output may be NULL.
 */
int lora_pool_query(const lora_pool *pool, int32_t adapter_id, int32_t module, int32_t *rank,
                    int64_t *row_offset);

/* lora_pool_free_rows -- free (rank-vector) rows left in module `module`'s pages. */
int lora_pool_free_rows(const lora_pool *pool, int32_t module, int64_t *free_rows);

/*
 * lora_build_segments -- host-side row grouping: a stable sort of rows by adapter id
 * (ascending, -1 first, ties keep row order).  ("m07", section 6: the index vector
 * sequence -> adapter slot; "LoRA, quotas and noisy neighbours", section "One weight read,
 * many adapters": rows tagged with their adapter and grouped.)
 *  row_ids      host int32 [n]
 *  perm         host int32 [n]     out: perm[p] = row at sorted position p
 *  seg_start    host int32 [n+1]   out: group s covers sorted positions [seg_start[s], seg_start[s+1])
 *  seg_adapter  host int32 [n]     out: adapter id of group s
 *  n_seg        host int32         out: number of groups
 * The same grouping is computed on the device inside lora_layer_forward.  Errors: EINVAL.
 */
int lora_build_segments(const int32_t *row_ids, int32_t n, int32_t *perm, int32_t *seg_start,
                        int32_t *seg_adapter, int32_t *n_seg);

/*
 * lora_quantize_rows_int8 -- host-side symmetric int8 quantization with one scale per row
 * ("m07 -- Multi-Adapter (LoRA) Serving", section 9 "Bottlenecks and Evolution", item 3:
 * adapters tolerate int8; half the bytes).  For each row, in fp32: scale = max|v| / 127,
 * code = round-half-to-even(v / scale) clipped to [-127, 127]; a zero row gets scale 0.
 *  src     host bf16 [rows, cols]
 *  codes   host int8 [rows, cols]    out
 *  scales  host fp32 [rows]          out
 * For an adapter, quantize A [r, d_in] by rows and B transposed ([r, d_out]) by rows, so both
 * scales belong to one rank index.  Errors: EINVAL.
 */
int lora_quantize_rows_int8(const void *src, int64_t rows, int64_t cols, int8_t *codes, float *scales);

/*
 * lora_pool_load_i8 -- lora_pool_load for an int8 pool: the adapter's factors as codes and
 * scales, factor = code * scale.
 *  qA      host or device int8 [rank, d_in]     sA  host fp32 [rank]  (scale of A's row j)
 *  qB      host or device int8 [d_out, rank]    sB  host fp32 [rank]  (scale of B's column j)
 * Stored like the bf16 factors (rows >= rank zero) plus, per stored row, sA[j] * sB[j] in fp32,
 * which the shrink applies to t_j.  Errors: EINVAL (bf16 pool, shapes, rank), ENOMEM, ECUDA.
 */
int lora_pool_load_i8(lora_pool *pool, int32_t adapter_id, int32_t module, const int8_t *qA, const float *sA,
                      const int8_t *qB, const float *sB, int32_t rank, lora_stream_t stream);

/* Policy of the adapter-aware batch former (lora_form_batch). */
typedef struct {
    int32_t max_batch;     /* most requests in one step, >= 1 */
    int32_t max_distinct;  /* cap on the adapters of one step ("m07", section 6: 32), >= 0 */
    int32_t min_batch;     /* the cap binds only once the batch holds this many requests, >= 0 */
    int32_t tail_slots;    /* places reserved for the oldest single-request adapters
                              ("m07", revision R1: 4 of the 32); 0 = none */
    double max_queue_ms;   /* age deadline: older requests are admitted first ("m07", section 6,
                              "The fairness cost": 200 ms); <= 0 = no deadline */
} lora_batch_policy;

/*
 * lora_form_batch -- host-side batch former: picks the requests of the next step from the
 * waiting queue so that the step reads few distinct adapters.  ("m07 -- Multi-Adapter (LoRA)
 * Serving", section 6 "Deep Dive A", "The adapter-aware scheduler" and "The fairness cost, which
 * must be stated"; revision R1, reserved tail slots; "12. Adapter Serving and Multi-Tenant
 * Customization", section "Scheduling with adapter awareness".)  In batch order it admits
 *   1. every request older than max_queue_ms (oldest first);
 *   2. up to tail_slots of the oldest remaining requests whose adapter has exactly one waiting
 *      request;
 *   3. the remaining requests grouped by adapter, largest group first (ties: first arrival),
 *      each group whole while there is room.  Once the batch holds max_distinct adapters and at
 *      least min_batch requests, groups that would add a new adapter are passed over; groups of
 *      adapters already admitted and the base-only group (-1) still come in.
 *  queue_adapter    host int32 [n_queue]   adapter id of each waiting request (-1 = base only),
 *                                          in arrival order
 *  queue_waited_ms  host double [n_queue]  how long each request has waited
 *  out_idx          host int32 [min(n_queue, max_batch)]  out: queue indices of the batch, in
 *                                          batch order
 *  out_n            out: requests in the batch
 *  out_distinct     out: distinct adapters (ids >= 0) in the batch
 * Pure host code; no device is touched.  Errors: EINVAL (null pointer, negative count, a policy
 * field out of range, an id < -1, a NaN wait).
 */
int lora_form_batch(const int32_t *queue_adapter, const double *queue_waited_ms, int32_t n_queue,
                    const lora_batch_policy *policy, int32_t *out_idx, int32_t *out_n, int32_t *out_distinct);

/*
 * Adapter cache -- host-side residency decisions for the device pool.  ("m07 -- Multi-Adapter
 * (LoRA) Serving", section 7 "Deep Dive B", "Eviction, and the trap in it": value =
 * requests_last_hour / size_bytes, evict lowest value first, never an adapter with in-flight
 * requests, and stop admitting new adapters while pinned bytes exceed a share of the budget;
 * revision R3: that share is 80% once the budget is sized by Little's law.)  The cache only
 * decides; the caller unloads and loads on the pool (lora_pool_unload / lora_pool_load, any
 * stream).  Pure host code; one cache per pool, not thread-safe.
 *
 * lora_cache_create   budget_bytes >= 0, guard_fraction in [0, 1], window_s > 0 (the pages: an
 *                     hour).  Errors: EINVAL.
 * lora_cache_acquire  a sequence starts on `adapter` (bytes = what it holds in the pool) at time
 *                     now_s: counts one request, and takes a reference.  If the adapter is
 *                     resident nothing else happens (*must_load = 0).  Otherwise, unless the
 *                     pinning guard refuses (EPINNED), room is made by evicting unreferenced
 *                     adapters lowest value first (ties: older latest request, then smaller id);
 *                     their ids go to evict[0 .. *n_evict) and the caller must unload them before
 *                     loading `adapter` (*must_load = 1).  ENOMEM: even evicting every
 *                     unreferenced adapter would not make room; nothing changed.  EINVAL: bad
 *                     argument, a time earlier than the previous call's, a resident adapter
 *                     acquired with another size, or more evictions than evict_cap.
 * lora_cache_release  a sequence on `adapter` ended: drops one reference.  EINVAL if it holds none.
 * lora_cache_stats    resident bytes, pinned bytes (resident with references), resident adapters.
 * lora_cache_resident whether `adapter` is resident, and its references.
 */
typedef struct lora_cache lora_cache;
int lora_cache_create(int64_t budget_bytes, double guard_fraction, double window_s, lora_cache **out);
int lora_cache_destroy(lora_cache *cache);
int lora_cache_acquire(lora_cache *cache, int32_t adapter, int64_t bytes, double now_s, int32_t *evict,
                       int32_t evict_cap, int32_t *n_evict, int32_t *must_load);
int lora_cache_release(lora_cache *cache, int32_t adapter);
int lora_cache_stats(const lora_cache *cache, int64_t *used_bytes, int64_t *pinned_bytes, int32_t *resident);
int lora_cache_resident(const lora_cache *cache, int32_t adapter, int32_t *resident, int32_t *ref);

/*
 * Layer gates -- adapter loads pipelined across the layers of a forward pass ("12. Adapter
 * Serving and Multi-Tenant Customization", section "Switching cost: I/O, not compute": a cold
 * adapter's factors are a copy, not a computation, so the factors a later layer needs can arrive
 * while the earlier layers run).  A gate holds one CUDA event per layer, each layer with its own
 * pool.  The loader queues layer l's loads on a copy stream (lora_pool_load / _load_many on that
 * layer's pool) and then calls lora_layer_gate_mark(gate, l, copy_stream); the forward queues
 * lora_layer_gate_wait(gate, l, compute_stream) just before layer l's first call, so the compute
 * stream waits for layer l's copies only, never for a later layer's.  A layer never marked, or
 * whose copies have already finished when the wait is queued, adds no wait (a stream wait between
 * two forwards keeps the second from launching early on the first).  One wait may also cover
 * several layers: marks of layers l .. l + g - 1 waited for before layer l.  Marking a layer again replaces its event (the waits queued after see the
 * newest mark).  Unloads that free pages a queued forward still reads must be ordered after it
 * (e.g. the copy stream waits for the compute stream before the step's unloads).
 * lora_layer_gate_create  n_layers >= 1; uses the current device.  Errors: EINVAL, ECUDA.
 * lora_layer_gate_mark / _wait   Errors: EINVAL (layer out of range), ECUDA.
 */
typedef struct lora_layer_gate lora_layer_gate;
int lora_layer_gate_create(int32_t n_layers, lora_layer_gate **out);
int lora_layer_gate_destroy(lora_layer_gate *gate);
int lora_layer_gate_mark(lora_layer_gate *gate, int32_t layer, lora_stream_t copy_stream);
int lora_layer_gate_wait(lora_layer_gate *gate, int32_t layer, lora_stream_t compute_stream);

/* One projection of a layer call. */
typedef struct {
    int32_t module;  /* pool module index */
    const void *x;   /* device bf16 [n, d_in]; projections may share x */
    const void *W;   /* device bf16 [d_out, d_in] */
    void *y;         /* device [n, d_out], element type y_dtype (fp32 or bf16) */
} lora_module_io;

/*
 * lora_layer_forward -- decode step: y = W x + s B_a A_a x for every projection in `io`,
 * rows tagged by `row_adapter_ids` (device int32 [n], -1 = base only).  The rows are
 * grouped by adapter on the device; every distinct adapter's factors are read once.
 *  n_io       1..LORA_MAX_MODULES projections, each with its own W and y (x may be shared)
 *  n          rows, 0 <= n <= min(LORA_MAX_DECODE_ROWS, max_rows); n == 0 does nothing
 *  scale      s
 *  y_dtype    LORA_DTYPE_F32 or LORA_DTYPE_BF16 (fp32 accumulate either way)
 * Asynchronous on `stream`.  An id outside [-1, max_adapters) or an adapter not resident
 * for one of the modules is recorded in the device error word (lora_last_device_error) and
 * that row gets the base term only.  Errors: EINVAL, EUNSUPPORTED (n > 256: use
 * lora_segment_forward with grouped rows), ECUDA.
 */
int lora_layer_forward(lora_pool *pool, int32_t n_io, const lora_module_io *io,
                       const int32_t *row_adapter_ids, int32_t n, float scale, int32_t y_dtype,
                       lora_stream_t stream);

/* lora_linear_forward -- lora_layer_forward for one projection. */
int lora_linear_forward(lora_pool *pool, int32_t module, const void *x, const void *W,
                        const int32_t *row_adapter_ids, int32_t n, float scale, void *y,
                        int32_t y_dtype, lora_stream_t stream);

/*
 * lora_segment_forward -- prefill / grouped rows: rows come as contiguous segments, one
 * adapter per segment ("m07", section 6 "Prefill is different, and worse": variable-length
 * segments; "LoRA, quotas and noisy neighbours", section "One weight read, many adapters").
 *  seg_start    device int32 [n_seg+1], seg_start[0] = 0, non-decreasing, seg_start[n_seg] = n
 *  seg_adapter  device int32 [n_seg], -1 = base only
 *  n            rows (tokens), 0 <= n <= max_rows
 * Same outputs and error reporting as lora_layer_forward; any n up to max_rows.
 */
int lora_segment_forward(lora_pool *pool, int32_t n_io, const lora_module_io *io,
                         const int32_t *seg_start, const int32_t *seg_adapter, int32_t n_seg,
                         int32_t n, float scale, int32_t y_dtype, lora_stream_t stream);

/*
 * lora_linear_forward_static -- lora_linear_forward for callers that must not allocate device
 * memory.  The pages have no counterpart to this call.
 *
 * Who needs it: a caller that cannot call cudaMalloc -- a serving runtime that has already
 * handed all of HBM to its own allocator (KV cache, its own fixed LoRA buffers), where an extra
 * allocation would fail or break its accounting, or code embedded in a framework that forbids
 * raw device allocations.  Such a caller cannot create a lora_pool either, so it passes its
 * adapters as stacked buffers it already owns.  Every per-call scratch buffer (row grouping,
 * shrink result and partial sums, stream-K partial tiles, counters, the factor table) lives in
 * one file-scope device array of this library, at most 24 MiB, which every GPU that loads the
 * library keeps until the process exits.  Nothing is allocated by this call.
 *
 *  x, W, y        as lora_linear_forward (device, 16-byte aligned); d_in, d_out multiples of 8
 *  row_adapter_ids device int32 [n]; -1 = base only; an id outside [-1, n_adapters) is served
 *                 base only
 *  A_stack        device bf16 [n_adapters, rank, d_in]   (adapter a's A at offset a*rank*d_in)
 *  B_stack        device bf16 [n_adapters, d_out, rank]  (adapter a's B at offset a*d_out*rank)
 *  rank           8, 16, 32 or 64, the same for every adapter (zero-pad smaller ranks)
 * Limits of the scratch: n <= 128, d_out <= 16384 (one base-piece slot per 128 rows of W),
 * n_adapters <= 4096; d_in is not limited.  Larger requests return LORA_EUNSUPPORTED, bad
 * arguments LORA_EINVAL, and lora_last_cuda_error() then names the reason.
 * This call has no device error report: unlike the pooled calls (lora_last_device_error), it
 * does not say when a row named an out-of-range id (that row gets the base term) or when a
 * bounded in-kernel wait ran out (after the 2 s budget the kernels return early and y is
 * undefined).  LORA_OK means the work was queued, not that the device finished it cleanly.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress) for
 * that device, so make that first call before any stream capture.
 * All calls share the one array and it keeps the previous call's contents (the counters in it
 * are cleared by every call): calls that can overlap on the GPU -- on different streams, or
 * from several host threads -- race and corrupt each other's results; order them.
 * Asynchronous on `stream`.
 */
int lora_linear_forward_static(const void *x, const void *W, int32_t d_in, int32_t d_out,
                               const int32_t *row_adapter_ids, int32_t n, const void *A_stack,
                               const void *B_stack, int32_t n_adapters, int32_t rank, float scale,
                               void *y, int32_t y_dtype, lora_stream_t stream);

/*
 * lora_plan_rows -- group a decode batch's rows once for every projection of the pool (the
 * index vector of "m07", section 6, is one per batch): stable sort by adapter id, id checks
 * (device error word), each row's adapter per projection, and every projection's gather list of
 * the batch's distinct adapters' A rows (8-row groups, the shrink's tiles).  Then
 * lora_layer_forward_planned runs any projections of the pool on that batch without grouping
 * again.
 *  row_adapter_ids  device int32 [n], -1 = base only; 0 <= n <= min(LORA_MAX_DECODE_ROWS, max_rows)
 * Asynchronous on `stream`.  The plan lives in the pool's workspace: lora_pool_load / _load_i8 /
 * _unload and every forward that groups its own rows end it.  Errors: EINVAL, ECUDA.
 */
int lora_plan_rows(lora_pool *pool, const int32_t *row_adapter_ids, int32_t n, lora_stream_t stream);

/*
 * lora_layer_step -- one layer of a decode step in one call: lora_plan_rows on the batch, then
 * lora_layer_forward_planned for each stage in order (stage st runs stage_n[st] >= 1 projections
 * that share an input, e.g. q/k/v, then o).  io holds the stages' entries one after another.
 * Same outputs, errors and error word as those calls; stops at the first error.
 */
int lora_layer_step(lora_pool *pool, const int32_t *row_adapter_ids, int32_t n, int32_t n_stages,
                    const int32_t *stage_n, const lora_module_io *io, float scale, int32_t y_dtype,
                    lora_stream_t stream);

/*
 * lora_layer_step_host -- lora_layer_step with the step's inputs and outputs in host memory, one
 * call per step.  The ids (host_ids -> row_adapter_ids, device int32 [n]) and every stage's input
 * (host_x[st] -> that stage's io[].x, bf16 [n, d_in]) go up on an upload stream of the pool's; the
 * rows are planned and the stages run on `stream`; each stage's outputs (io[i].y -> host_y[i],
 * [n, d_out] of y_dtype) come down on a download stream of the pool's while the next stage -- or
 * the next call -- computes.  The projections of a stage share one device x.
 * Serving loop: alternate two sets of device buffers (ids, x, y; a set is known by its ids
 * buffer): a call's inputs then go up while the previous call computes, and its outputs come down
 * while the next one does.  A call waits only for the earlier calls on the same set (its inputs
 * consumed, its outputs downloaded).  The outputs are in host memory once `stream` has passed a
 * later lora_pool_host_wait(pool, stream), which makes `stream` wait for every download queued so
 * far.  Host buffers should be pinned (pageable memory makes the copies synchronous); the host
 * inputs may be rewritten, and the host outputs read, only after that point.  The device buffers
 * are the caller's, borrowed.  Errors: EINVAL, and those of lora_layer_step.
 */
int lora_layer_step_host(lora_pool *pool, const int32_t *host_ids, int32_t *row_adapter_ids, int32_t n,
                         int32_t n_stages, const int32_t *stage_n, const lora_module_io *io,
                         const void *const *host_x, void *const *host_y, float scale, int32_t y_dtype,
                         lora_stream_t stream);

/* lora_pool_host_wait -- make `stream` wait for every download lora_layer_step_host has queued. */
int lora_pool_host_wait(lora_pool *pool, lora_stream_t stream);

/*
 * lora_layer_forward_planned -- lora_layer_forward on the rows of the last lora_plan_rows (same
 * n, same ids): shrink and base + expand only.  `io` may name any modules of the pool, in any
 * calls, as long as the plan is current.  Errors: EINVAL (no current plan, or as
 * lora_layer_forward), EUNSUPPORTED, ECUDA.
 */
int lora_layer_forward_planned(lora_pool *pool, int32_t n_io, const lora_module_io *io, float scale,
                               int32_t y_dtype, lora_stream_t stream);

/*
 * int4 base weights with bf16 (or int8) adapters ("12. Adapter Serving ...", section
 * "Quantization": the base quantized to INT4 while the adapters stay BF16; the kernel dequantizes
 * the base, adds the adapter term and accumulates wide, and one batch mixes adapted and base-only
 * rows).  W is symmetric int4 with one fp32 scale per output row:
 *     W[o, k] = scale[o] * code[o, k],   code in [-7, 7],   scale[o] = max_k |W[o, k]| / 7
 * and the forward computes y_i = scale * (code x_i) + s B_a A_a x_i with fp32 accumulation (the
 * codes enter the tensor-core product as exact bf16 integers; the row scale multiplies the
 * accumulator).
 *
 * lora_quantize_w4 -- host quantizer.  src: host bf16 [rows, cols] (cols a multiple of 8); writes
 * packed [rows, cols / 2] bytes and scales [rows].  code = round-half-even(v / scale) in fp32,
 * clipped to [-7, 7]; a zero row gets scale 0 and codes 0.  Packed layout: every 8 consecutive
 * elements e0..e7 of a row form one little-endian 32-bit word; element 2s (s = 0..3) is stored at
 * bits [4s, 4s + 4) and element 2s + 1 at bits [16 + 4s, 20 + 4s), each as code + 8 (1..15).
 * Errors: EINVAL.
 */
int lora_quantize_w4(const void *src, int64_t rows, int64_t cols, uint8_t *packed, float *scales);

/* One projection of an int4-base call. */
typedef struct {
    int32_t module;       /* pool module index */
    const void *x;        /* device bf16 [n, d_in] */
    const void *W_codes;  /* device [d_out, d_in / 2] bytes, lora_quantize_w4's layout; 16-byte aligned */
    const float *W_scale; /* device fp32 [d_out] */
    void *y;              /* device [n, d_out], fp32 or bf16 */
} lora_module_io_w4;

/*
 * lora_layer_forward_w4 / lora_layer_forward_planned_w4 -- lora_layer_forward and
 * lora_layer_forward_planned with int4 base weights.  Decode batches only (n <= 256); the module's
 * d_in must be a multiple of 32.  The pool's factors may be bf16 or int8.  x, W_codes, W_scale and
 * y are caller-owned device memory, borrowed for the call (x, W_codes, y 16-byte aligned, W_scale
 * 4-byte aligned).  Same row ids, error word and errors as the bf16 calls: EINVAL also for a
 * missing or misaligned W_scale, EUNSUPPORTED also for d_in % 32 != 0 or n > 256.
 */
int lora_layer_forward_w4(lora_pool *pool, int32_t n_io, const lora_module_io_w4 *io,
                          const int32_t *row_adapter_ids, int32_t n, float scale, int32_t y_dtype,
                          lora_stream_t stream);
int lora_layer_forward_planned_w4(lora_pool *pool, int32_t n_io, const lora_module_io_w4 *io, float scale,
                                  int32_t y_dtype, lora_stream_t stream);

/*
 * lora_layer_step_host_w4 -- lora_layer_step_host with int4 base weights: the same host I/O, buffer
 * sets, streams and lora_pool_host_wait, each stage run by lora_layer_forward_planned_w4.  Errors:
 * EINVAL, and those of lora_layer_forward_planned_w4.
 */
int lora_layer_step_host_w4(lora_pool *pool, const int32_t *host_ids, int32_t *row_adapter_ids, int32_t n,
                            int32_t n_stages, const int32_t *stage_n, const lora_module_io_w4 *io,
                            const void *const *host_x, void *const *host_y, float scale, int32_t y_dtype,
                            lora_stream_t stream);

/*
 * lora_pool_last_segments -- synchronize the device and copy out the row grouping the most
 * recent forward on this pool used (computed on the device for lora_layer_forward; the
 * checked copy of the given table for lora_segment_forward).  Host outputs:
 *  perm         int32 [n]      sorted position -> row (identity for grouped rows with n > 256;
 *                              left untouched then)
 *  seg_start    int32 [n+1], seg_adapter int32 [n], *n_seg, *n (rows of that forward).
 * Any output pointer may be NULL.  Errors: EINVAL, ECUDA.
 */
int lora_pool_last_segments(lora_pool *pool, int32_t *perm, int32_t *seg_start, int32_t *seg_adapter,
                            int32_t *n_seg, int32_t *n);

/*
 * lora_last_device_error -- synchronize the device, then read and clear the pool's device
 * error word.  *code is a LORA_DEVERR_* value, *detail the row/segment it concerns.
 */
int lora_last_device_error(lora_pool *pool, int32_t *code, int32_t *detail);

/*
 * lora_pool_set_wait_budget -- the wall-clock budget of each bounded in-kernel wait of this pool's
 * forwards (a wait for a TMA copy to land, for an MMA, for a free pipeline slot or accumulator).
 * A wait that runs out records LORA_DEVERR_TIMEOUT in the device error word; the kernel stops
 * issuing work, waits for the copies and MMAs it has already issued, frees its tensor memory and
 * returns, so the context stays usable.  That call's outputs are undefined; later calls are not
 * affected.  0 restores the default of 2 s, far above any legitimate wait.  A budget of a few
 * microseconds makes a correct call give up: that is how the bounded waits are exercised without
 * hanging or faulting a GPU.  Host-side setting, takes effect for forwards queued after it.
 * Errors: EINVAL.
 */
int lora_pool_set_wait_budget(lora_pool *pool, uint64_t budget_ns);

/*
 * Kernel timing.  While enabled, every forward on this pool records a CUDA event pair on its
 * stream around each kernel it launches:
 *  LORA_KERNEL_PREP      row grouping / checks (and the decode gather lists)
 *  LORA_KERNEL_SHRINK    t = s A x on CUDA cores (grouped rows; decode with int8 factors)
 *  LORA_KERNEL_GEMM      tcgen05 base (decode: with the shrink's A tiles for bf16 factors;
 *                        grouped rows: with the expand)
 *  LORA_KERNEL_FINALIZE  decode: base pieces summed, the expand s B t, y written
 * lora_profile_read synchronizes, returns the number of launches and their summed device
 * time in milliseconds for one kind, and clears that kind.  Timing adds two event records
 * per launch and separates launches that otherwise overlap; leave it off for throughput
 * runs.  Errors: EINVAL, ECUDA.
 */
#define LORA_KERNEL_PREP 0
#define LORA_KERNEL_SHRINK 1
#define LORA_KERNEL_GEMM 2
#define LORA_KERNEL_FINALIZE 3
int lora_profile_enable(lora_pool *pool, int32_t enable);
int lora_profile_read(lora_pool *pool, int32_t kernel, int32_t *launches, double *total_ms);

/* lora_last_cuda_error -- the last CUDA error string seen by this library (thread-local). */
const char *lora_last_cuda_error(void);

/* lora_status_string -- a constant string naming a LORA_* status. */
const char *lora_status_string(int status);

/* lora_version -- ABI version (major * 10000 + minor * 100 + patch). */
int lora_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LORA_GB300_H */
