/*
 * ls_api.h — C ABI of the layer-streaming library (liblstream.so).
 *
 * Layer-streamed execution: model parameters stay in host memory, cut into
 * parameter-bearing segments. While the active segment computes on the GPU, the
 * parameters of the next `prefetch_depth` segments are copied into a fixed-slot
 * pool in device memory, which turns a serial load-then-compute loop into a
 * rolling pipeline.
 *   - "feat: prefetch streamed layers during compute" (stable-diffusion.cpp PR
 *     #1905), Summary and "Effective behavior" table: prefetch depth, resident
 *     prefix as a maximum (-1 = auto), budget rules, synchronous fallback, and a
 *     versioned parameter struct whose undersized (older) form stays valid.
 *   - "feat: pool VRAM for streamed layer" (stable-diffusion.cpp PR #1906),
 *     Summary and the pool "Effective behavior" table: one contiguous pool of
 *     equal slots, peak slot count only, degradation down to one slot, the
 *     mandatory one-slot pool.
 *   - "layer split: overlap the stages' hand-off" (Strata #1120), description
 *     and "Changes since #936": a ready word per hand-off buffer raised by the
 *     writer's last block after a system fence, a bounded wait on the reader's
 *     side that sets an error word, and a test hook that drops the Nth publish.
 *   - "prefill: a layer split's idle card streams a share of a one-chunk
 *     prompt's experts" (Strata #663), What: a copy kernel reading mapped host
 *     memory with 16-byte loads instead of copy-engine uploads, and expert
 *     grouping through a row table and group bounds.
 *
 * Conventions for every call:
 *   - Return values are ls_status (int32_t). Negative = failure, nothing
 *     half-done is left behind unless stated. Positive = warning; results valid.
 *   - Pointers named *_dev are CUDA device pointers on the context's device;
 *     *_host are host pointers. Streams are passed as `void*` holding a
 *     cudaStream_t (NULL = the legacy default stream).
 *   - A context is not thread-safe: calls on one context must not overlap.
 *   - ls_last_error() gives a one-line human-readable reason for the last failure
 *     on that context.
 */
#ifndef LS_API_H
#define LS_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LS_PARAMS_VERSION 1

typedef int32_t ls_status;
enum {
    LS_OK = 0,
    LS_WARN_MANDATORY_SLOT = 1,  /* budget below one slot: the one-slot pool was taken anyway */
    LS_WARN_SYNC_FALLBACK = 2,   /* asynchronous prefetch unavailable: continued synchronously */
    LS_ERR_INVALID_ARG = -1,
    LS_ERR_VERSION = -2,         /* params.version unknown or struct_size too small */
    LS_ERR_OOM = -3,             /* even the one-slot pool (or a synchronous load) could not be allocated */
    LS_ERR_HANDOFF_TIMEOUT = -4, /* a ready word stayed down past wait_limit_ms; that run's output is invalid */
    LS_ERR_CUDA = -5,            /* a CUDA call failed; see ls_last_error */
    LS_ERR_STATE = -6,           /* call out of order (e.g. ls_run before ls_register_segments) */
    LS_ERR_UNSUPPORTED = -7,     /* shape or alignment the kernels do not handle */
    LS_ERR_BOUNDS = -8           /* params.debug_checks found a canary overwritten or an invalid MoE row
                                    table; see ls_last_error (the run's output is invalid) */
};

/* Segment kinds: what one segment computes (x: [tokens, hidden] activations). */
enum {
    LS_KIND_LINEAR_GELU_F32 = 0,      /* y = GELU(x W^T + b); tensors W[F,H] f32, b[F] f32 */
    LS_KIND_FFN_GELU_BF16 = 1,        /* y = x + GELU(x W1^T + b1) W2^T + b2; W1[F,H], b1[F], W2[H,F], b2[H] bf16 */
    LS_KIND_FFN_GELU_SHARED_BF16 = 2, /* y = x + GELU((x P^T) W1^T + b1) W2^T + b2; P[H,H] (shared), W1, b1, W2, b2 */
    LS_KIND_SWIGLU_BF16 = 3,          /* y = x + (SiLU(x G^T) * (x U^T)) D^T; G[F,H], U[F,H], D[H,F] bf16 */
    LS_KIND_MOE_SWIGLU_BF16 = 4       /* y = x + sum_k w_k SwiGLU_{e_k}(x); expert-major G_e[F,H], U_e[F,H], D_e[H,F] */
};

enum { LS_DTYPE_F32 = 0, LS_DTYPE_BF16 = 1 };

/* Schedule event kinds (ls_sched_event.kind). */
enum {
    LS_EV_SHARED_LOAD = 0,   /* a deduplicated shared tensor copied into the shared region (run 0) */
    LS_EV_LOAD_RESIDENT = 1, /* a resident-prefix segment copied synchronously before a run's first
                                step (run 0, or the first run after a plan change grew the prefix) */
    LS_EV_LOAD_SYNC = 2,     /* a streamed segment copied on the compute stream right before use */
    LS_EV_PREFETCH = 3,      /* a streamed segment queued on the copy stream ahead of use */
    LS_EV_ACTIVATE = 4,      /* the segment's compute was issued, reading its slot */
    LS_EV_EVICT = 5          /* a resident released under memory pressure (pool off, at a step) or at a
                                plan change (step -1), or a stale cross-run prefetch (step -1) */
};

enum { LS_COPY_AUTO = 0, LS_COPY_KERNEL = 1, LS_COPY_ENGINE = 2 };

/* Optional device allocator for parameter memory (pool, shared region,
 * per-load buffers with the pool off). alloc returns NULL on failure. free is
 * called with the stream on which the memory was last used; the allocator must
 * not hand the memory out again for work not ordered after that stream point.
 * Default (both NULL): cudaMallocAsync / cudaFreeAsync. */
typedef void* (*ls_alloc_fn)(void* user, size_t bytes, void* stream);
typedef void (*ls_free_fn)(void* user, void* ptr, size_t bytes, void* stream);

/* Versioned parameters. The caller sets struct_size = sizeof(ls_params) as it
 * was compiled; fields past struct_size take their defaults, so a binary built
 * against an older, shorter struct keeps working. The minimum accepted size
 * covers the four controls up to use_pool. ls_params_init() fills defaults. */
typedef struct ls_params {
    uint32_t struct_size;
    uint32_t version;          /* LS_PARAMS_VERSION */
    int32_t prefetch_depth;    /* >= 0; 0 (default) = synchronous streaming */
    int32_t resident_layers;   /* -1 = auto (default), 0 = none, N = at most N leading segments */
    int64_t max_vram_bytes;    /* parameter budget in bytes; 0 (default) = no segmentation, all resident */
    int32_t use_pool;          /* 1 = one contiguous slot pool; 0 (default) = one allocation per load */
    /* ---- end of the minimum struct ---- */
    int32_t wait_limit_ms;     /* bound of every device-side wait, 1..600000; default 30000 */
    int32_t copy_path;         /* LS_COPY_AUTO (default: both paths timed on each segment's load at
                                  registration, chosen per segment), _KERNEL, _ENGINE (every segment) */
    int32_t copy_ctas;         /* CTAs of the copy kernel; 0 = default */
    int32_t reserve_sms;       /* SMs the GEMMs leave free while a copy kernel runs; -1 = default */
    int32_t device;            /* CUDA device ordinal; -1 (default) = the current device */
    ls_alloc_fn alloc_fn;      /* optional, see above */
    ls_free_fn free_fn;
    void* alloc_user;
    /* test hooks (all 0 = off) */
    int64_t test_alloc_cap_bytes; /* parameter allocations beyond this many live bytes fail */
    int32_t test_fail_async;      /* the first prefetch finds asynchronous transfer unavailable */
    int32_t test_drop_publish;    /* the Nth publish (1-based, over the context's life) leaves its ready word down */
    int32_t kernel_timing;        /* 1 = bracket every launch with CUDA events (see ls_get_kernel_times);
                                     2 = also keep a per-launch trace (see ls_get_trace). Launches
                                     then run without programmatic dependent launch, so that each
                                     event pair times its kernel alone.
                                     3 = trace only the copies and, per segment, one "compute" span
                                     from the end of the hand-off wait to the segment's last kernel;
                                     launches keep programmatic dependent launch */
    int32_t cross_run_prefetch;   /* 1 = the prefetch window crosses the run boundary: the last steps of
                                     a run also queue the next run's first streamed segments (when the
                                     ring is a full depth + 1 slots; never for the MoE kind, whose next
                                     loads depend on the next run's routing). 0 (default) = every run
                                     starts its window afresh ("feat: prefetch streamed layers during
                                     compute", maintainer review: no cross-forward state). The prefetch
                                     of a run that never comes is released at ls_replan or destroy. */
    int64_t expert_cache_bytes;   /* MoE kind: device memory for hot experts of streamed layers, on top of
                                     max_vram_bytes (0 = none). It holds K = bytes / expert-blob bytes
                                     experts: in each pass, the K (layer, expert) pairs routed in the most
                                     earlier passes (ties to the lower expert, then layer); a hot expert is
                                     copied in when its layer next loads it from the host, and a routed
                                     expert found there is read in place by the grouped GEMMs instead of
                                     crossing the host link. Bits are unchanged; the schedule's load bytes count
                                     the host copies only. */
    int32_t debug_checks;         /* 1 = bounds checks that need no sanitizer: a 256-byte canary after every
                                     pool slot, after the shared region and after every per-load buffer
                                     (pool off), filled at allocation and verified after each ls_run (and
                                     before a per-load buffer is freed); the MoE row table and group bounds
                                     are validated on the device after routing. A violation fails the run
                                     with LS_ERR_BOUNDS. Canaries are device memory beyond max_vram_bytes.
                                     0 (default) = off */
    int32_t test_corrupt_canary;  /* test hook (debug_checks only): N > 0 overwrites the canary of pool slot
                                     N - 1 once, right after registration */
    int32_t test_kernel_copy_stride; /* test hook (copy_path AUTO only): N > 0 skips the timing and puts the
                                     loads of the segments whose index is a multiple of N on the copy
                                     kernel, the others on the copy engine */
} ls_params;

/* One tensor of a segment: host memory owned by the caller, kept alive and
 * unchanged until ls_ctx_destroy. Pageable memory is registered (pinned and
 * mapped) by the library and unregistered at destroy; memory that is already
 * pinned is used as is. */
typedef struct ls_tensor_desc {
    const void* host_ptr;
    uint64_t bytes;
    int32_t dtype;             /* LS_DTYPE_* */
    int32_t ndim;              /* 1 or 2 */
    int64_t shape[2];          /* row-major; weights are [out, in] */
} ls_tensor_desc;

typedef struct ls_segment_desc {
    int32_t kind;              /* LS_KIND_* (all segments of one context share the kind) */
    int32_t n_tensors;
    const ls_tensor_desc* tensors;
} ls_segment_desc;

/* Marks tensor `tensor_index` of segment `segment` as shared parameter
 * `shared_id`. Tensors with the same id are one parameter: it is copied once
 * into a resident shared region and every segment reads that copy. */
typedef struct ls_shared_ref {
    int32_t segment;
    int32_t tensor_index;
    int32_t shared_id;         /* >= 0 */
} ls_shared_ref;

/* Router input of the MoE kind: logits [n_segments, tokens, n_experts] fp32,
 * row-major, on the device (ls_run) or on the host (ls_run_host). */
typedef struct ls_moe_routing {
    const float* logits;
    int32_t top_k;             /* 1..8 */
} ls_moe_routing;

typedef struct ls_sched_event {
    int32_t run;               /* 0-based index of the ls_run call on this context */
    int32_t step;              /* segment step the event belongs to; -1 = before step 0 */
    int32_t kind;              /* LS_EV_* */
    int32_t segment;           /* segment index (shared id for SHARED_LOAD) */
    int32_t slot;              /* logical slot (-1 for SHARED_LOAD) */
    int32_t reserved;
    int64_t bytes;             /* bytes moved over the host link by this event (0 for ACTIVATE/EVICT) */
} ls_sched_event;

typedef struct ls_stats {
    uint32_t struct_size;      /* set by the caller, as for ls_params */
    int32_t n_segments;
    int32_t residents;         /* current resident prefix R */
    int32_t depth;             /* current effective prefetch depth */
    int32_t ring_slots;        /* Q: slots cycling through streamed segments */
    int32_t pool_slots;        /* P = R + Q (planned) */
    int32_t warnings;          /* bit (1 << w) for each warning w raised so far */
    int32_t copy_path;         /* LS_COPY_KERNEL or LS_COPY_ENGINE when every segment's loads take that
                                  path; LS_COPY_AUTO when the segments differ (kernel_copy_segments) */
    int64_t slot_bytes;        /* S */
    int64_t shared_bytes;
    int64_t pool_bytes;        /* bytes of the pool allocation (0 with the pool off) */
    int64_t runs;
    int64_t prefetch_queued;
    int64_t prefetch_activated;
    int64_t sync_loads;
    int64_t resident_loads;
    int64_t shared_loads;
    int64_t evictions;
    int64_t sync_fallbacks;
    int64_t pool_degradations;
    int64_t bytes_loaded;
    double copy_kernel_gbs;    /* registration-time timing of both copy paths over the segments' loads (0 if not timed) */
    double copy_engine_gbs;
    int64_t graph_captures;    /* passes captured into a CUDA graph by ls_run_graph */
    int64_t graph_replays;     /* passes issued as a replay of the captured graph */
    int64_t expert_cache_hits; /* routed experts of streamed layers served from the expert cache */
    int64_t expert_host_loads; /* routed experts of streamed layers copied from the host */
    int64_t debug_violations;  /* runs failed by params.debug_checks */
    int64_t kernel_copy_segments; /* segments whose loads go through the copy kernel */
} ls_stats;

/* Per-kernel timing, accumulated over runs while params.kernel_timing is on.
 * Each launch is bracketed by CUDA events on the stream it is launched on. */
typedef struct ls_kernel_time {
    char name[32];             /* kernel class, e.g. "copy_h2slot", "gemm_up", "gemm_down" */
    int64_t launches;
    double total_ms;
} ls_kernel_time;

/* One launch of the per-launch trace (kernel_timing = 2): times in ms from the
 * first launch recorded since the previous ls_sync. */
typedef struct ls_trace_event {
    char name[32];
    int32_t stream;            /* 0 = the caller's (compute) stream, 1 = the context's copy stream */
    int32_t segment;           /* segment the launch belongs to, -1 if none */
    double start_ms;
    double end_ms;
} ls_trace_event;

typedef struct ls_ctx ls_ctx;

/* Fill *p with defaults (struct_size = sizeof(ls_params), version = 1). */
void ls_params_init(ls_params* p);

/* Validate the params and create an empty context. Host only: no GPU work.
 * Errors: LS_ERR_INVALID_ARG (NULL, negative depth, resident < -1, negative
 * budget, wait_limit_ms out of range), LS_ERR_VERSION. */
ls_status ls_ctx_create(const ls_params* params, ls_ctx** out);

/* Register the segments (host pointers) and the shared-parameter map, plan the
 * slots, allocate the pool (degrading the slot count on allocation failure),
 * copy the shared parameters, and time the copy paths. Under LS_COPY_AUTO (with
 * something streamed) every segment's load is copied once by each path into the
 * first slot, so registration moves about twice the stack's private bytes over
 * the host link (~0.6 s for 58 GB at 211 GB/s, longer where the copy engine reads
 * slowly). n_segments >= 1.
 * Returns LS_WARN_MANDATORY_SLOT when the budget is below one slot,
 * LS_ERR_OOM when not even one slot could be allocated, LS_ERR_UNSUPPORTED for
 * tensor shapes or kinds the kernels do not handle. Once per context. */
ls_status ls_register_segments(ls_ctx* ctx, const ls_segment_desc* segs, int32_t n_segments,
                               const ls_shared_ref* shared_map, int32_t n_shared);

/* One pass over every segment: y = segment_{N-1}(... segment_0(x)).
 * x_dev / y_dev: [tokens, hidden] row-major, bf16 (f32 for the fp32 kind),
 * caller-owned device memory; they may not alias. Stream-ordered on `stream`;
 * returns after that stream has finished the pass (the error word is read
 * then). routing is required for the MoE kind and ignored otherwise.
 * LS_ERR_HANDOFF_TIMEOUT: a hand-off wait ran out; y is invalid, the context
 * stays usable. LS_WARN_SYNC_FALLBACK: this pass fell back to synchronous loads. */
ls_status ls_run(ls_ctx* ctx, const void* x_dev, void* y_dev, int64_t tokens, void* stream,
                 const ls_moe_routing* routing);

/* ls_run without the final host synchronisation: the pass is queued on
 * `stream` and the call returns (for the MoE kind after one short sync that
 * reads which experts are routed). Consecutive passes of one context are
 * ordered after each other even on different streams. Device-side errors
 * (hand-off timeouts, failed kernels) are reported by the next ls_sync. */
ls_status ls_run_async(ls_ctx* ctx, const void* x_dev, void* y_dev, int64_t tokens, void* stream,
                       const ls_moe_routing* routing);

/* Wait for every queued pass of the context and report the first device error
 * (LS_ERR_HANDOFF_TIMEOUT, LS_ERR_CUDA) since the previous ls_sync, else LS_OK. */
ls_status ls_sync(ls_ctx* ctx);

/* ls_run from host buffers: copies x_host (and the MoE logits, given on the
 * host) to the device, runs the pass, copies y back into y_host. Pinned host
 * buffers give asynchronous copies; pageable ones work too. */
ls_status ls_run_host(ls_ctx* ctx, const void* x_host, void* y_host, int64_t tokens,
                      const ls_moe_routing* routing_host);

/* ls_run_host without the final synchronisation: the copy of x_host (and the logits) in,
 * the pass and the copy of y back into y_host are queued, in that order, on the context's
 * own stream, and the call returns (for the MoE kind after the routing sync of ls_run_async,
 * which also waits for the previous pass's compute). Consecutive calls pipeline: a pass's
 * inputs are copied in once the previous pass has finished with the staging buffers, while
 * the weight copies of the passes keep the host link busy. The host buffers must stay valid,
 * and y_host unread, until ls_sync returns; ls_sync also reports the passes' device errors.
 * Pinned host buffers are needed for the copies to be asynchronous (CUDA copies pageable
 * memory synchronously). Errors as ls_run_host. */
ls_status ls_run_host_async(ls_ctx* ctx, const void* x_host, void* y_host, int64_t tokens,
                            const ls_moe_routing* routing_host);

/* Copy up to `cap` logged events (oldest first) into out; *n_out = total logged. */
ls_status ls_get_schedule(ls_ctx* ctx, ls_sched_event* out, int64_t cap, int64_t* n_out);

/* Counters and the current plan. out->struct_size must be set by the caller. */
ls_status ls_get_stats(ls_ctx* ctx, ls_stats* out);

/* Switch per-launch timing (the kernel_timing field of ls_params: 0 to 3)
 * for the passes issued from now on. With timing on, kernels launch without
 * programmatic dependent launch (a kernel placed early would otherwise start its
 * event pair while the kernel before it still runs), and event records between
 * launches cost the stream a little time, so a throughput measurement runs with
 * timing off and a separate set of passes collects the per-kernel times. LS_ERR_STATE while passes issued
 * by ls_run_async have not been collected by ls_sync; LS_ERR_INVALID_ARG for a
 * mode outside 0..3. The pages define no such call: it is instrumentation. */
ls_status ls_set_kernel_timing(ls_ctx* ctx, int32_t mode);

/* One pass, like ls_run_async, issued as a CUDA graph: the first steady-state
 * pass (no shared, resident or synchronous-fallback work left) is captured with
 * its copy and compute streams, and later passes replay it while x_dev, y_dev,
 * tokens and the pass's schedule stay the same (a change re-captures). This
 * removes the host's per-launch cost, which dominates passes of small stacks
 * ("layer split: overlap the stages' hand-off", Summary: host launch and sync on
 * the critical path). The graph sets the slots' ready words to 0 at its start,
 * then raises them with the epochs fixed at capture. Passes that are not steady
 * (the first runs, after a plan change) run as ordinary passes.
 * The schedule log and counters advance as for ls_run_async. LS_ERR_UNSUPPORTED
 * for the MoE kind (routing is read back on the host every pass), with the pool
 * off, or with cross_run_prefetch; other errors as for ls_run_async. The graph is
 * dropped at ls_replan, at ls_ctx_destroy and when a larger token count replaces
 * the workspaces. Complete with ls_sync. */
ls_status ls_run_graph(ls_ctx* ctx, const void* x_dev, void* y_dev, int64_t tokens, void* stream);

/* New streaming controls between runs ("feat: prefetch streamed layers during
 * compute", Summary: residents are evicted from the end of the prefix under
 * memory pressure, and stale residents and prefetches are released when the
 * plan changes; "feat: pool VRAM for streamed layer", Summary: a sufficiently
 * large pool is reused and reduced caps are remembered). The next run plans
 * with the same rules as ls_register_segments, under any remembered reduced
 * pool slot count; a remembered synchronous fallback stays. Before that run's
 * first step:
 *  - prefetches already queued for it (cross_run_prefetch) are released;
 *  - residents beyond the new prefix are released, last first (LS_EV_EVICT, step -1);
 *  - pool on: the pool is kept when its slot count does not change. Otherwise it
 *    is freed and a pool of the new count is allocated (fewer slots on failure).
 *    That empties every slot, so the whole new prefix is loaded again;
 *  - newly resident segments are loaded (LS_EV_LOAD_RESIDENT).
 * Returns LS_OK or LS_WARN_MANDATORY_SLOT (the new budget is below one slot);
 * LS_ERR_STATE while passes from ls_run_async await ls_sync;
 * LS_ERR_INVALID_ARG for a negative depth or budget or a resident cap below -1;
 * LS_ERR_OOM when not even a one-slot pool can be allocated, after which the
 * context cannot run (destroy it). Blocks until queued copies finish. */
ls_status ls_replan(ls_ctx* ctx, int32_t prefetch_depth, int32_t resident_layers, int64_t max_vram_bytes);

/* Copy up to cap kernel-time records into out; *n_out = number of classes.
 * reset != 0 clears the accumulators afterwards. */
ls_status ls_get_kernel_times(ls_ctx* ctx, ls_kernel_time* out, int32_t cap, int32_t* n_out, int32_t reset);

/* Copy up to cap trace records of the passes completed by the last ls_sync. */
ls_status ls_get_trace(ls_ctx* ctx, ls_trace_event* out, int64_t cap, int64_t* n_out);

/* Release everything the context owns (pool, buffers, streams, registrations). NULL is a no-op. */
void ls_ctx_destroy(ls_ctx* ctx);

const char* ls_status_string(ls_status s);
const char* ls_last_error(const ls_ctx* ctx);

/* Run the context's scheduler without a GPU: the same planning and event
 * logic as ls_register_segments + `runs` x ls_run, with device work replaced by
 * byte accounting (test_alloc_cap_bytes and test_fail_async apply).
 * seg_slot_bytes[n]: each segment's 256-byte-aligned private footprint.
 * shared_bytes[n_shared]: the distinct shared tensors' bytes, by shared id
 * (shared_ids[i] is the id of shared_bytes[i]). load_bytes: NULL (a load moves
 * the segment's footprint) or [runs][n] bytes per load. run_status[runs]
 * receives each run's status (LS_ERR_OOM at registration leaves it untouched).
 * events: up to cap written; *n_events = total. */
/* ls_simulate driven by a script instead of a run count: script[4 * i ..] =
 * {op, depth, resident, max_vram_bytes}, op 0 = one run (the other three
 * ignored), op 1 = ls_replan with those controls. step_status[n_steps] receives
 * each step's status; the script stops at the first error. Loads move each
 * segment's footprint. Other arguments as for ls_simulate. */
ls_status ls_simulate_script(const ls_params* params, const int64_t* seg_slot_bytes, int32_t n,
                             const int64_t* shared_bytes, const int32_t* shared_ids, int32_t n_shared,
                             const int64_t* script, int32_t n_steps, ls_sched_event* events, int64_t cap,
                             int64_t* n_events, ls_stats* stats, ls_status* step_status);

ls_status ls_simulate(const ls_params* params, const int64_t* seg_slot_bytes, int32_t n,
                      const int64_t* shared_bytes, const int32_t* shared_ids, int32_t n_shared,
                      int32_t runs, const int64_t* load_bytes, ls_sched_event* events,
                      int64_t cap, int64_t* n_events, ls_stats* stats, ls_status* run_status);

/* Pinned, device-mapped host memory for segment tensors (no counterpart on the pages,
 * which pin the caller's memory; this is the driver's own pinned allocation, portable
 * across devices). Memory from ls_host_alloc is used as is by ls_register_segments (it is
 * not registered again). ls_host_alloc: LS_ERR_OOM when the driver refuses;
 * ls_host_free(NULL) does nothing; freeing memory a context still uses is undefined. */
ls_status ls_host_alloc(uint64_t bytes, void** out);
ls_status ls_host_free(void* p);

/* Idle-stage helper of a two-stage layer split ("prefill: a layer split's idle card
 * streams a share of a one-chunk prompt's experts", Strata #663, What). While one stage
 * computes its MoE layers the other card idles; it takes a share of each layer's routed
 * experts, streams them over its own host link, computes their (token, k) rows and hands
 * the rows back through mapped host memory (lsk_moe_group_masked, lsk_moe_rows_copy and
 * lsk_wait_ready in ls_kernels.h are the device steps). Each row is computed on one card
 * by the same kernels, so the combined layer has the bits of the unsplit one. Measured on
 * one GPU only: the two cards' steps run one after the other there.
 *
 * ls_helper_share: the share for a one-chunk prompt of `tokens` tokens,
 * min(0.45, 0.5 - tokens/16384), and 0 (helper off) when that is below 0.3. */
double ls_helper_share(int64_t tokens);

/* Which of a layer's routed experts the helper takes: routed[E] (nonzero = routed in this
 * pass, host memory) -> helper_mask[E] (1 = the helper's, host memory). The helper takes
 * floor(share * routed count) experts, the highest-numbered routed ones; the active card
 * keeps the others. LS_ERR_INVALID_ARG for NULL pointers, E < 0 or share outside [0, 1]. */
ls_status ls_helper_split(const uint8_t* routed, int32_t E, double share, uint8_t* helper_mask);

#ifdef __cplusplus
}
#endif
#endif /* LS_API_H */
