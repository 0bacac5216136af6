// Layer-streaming runtime: contexts, registration, the GPU executor and the C ABI.
//
// The scheduler (ls_sched.h) decides what happens at each step; the executor here
// turns each decision into device work:
//   load (prefetch)  copy stream: wait until the slot's previous occupant has
//                    computed (event), then the host-to-slot copy, whose last
//                    CTA raises the slot's ready word to a fresh epoch.
//   load (sync)      the same copy on the compute stream (stream order is the
//                    hand-off; the ready word is raised too).
//   activate         compute stream: the segment's kernels; the first kernel
//                    that reads streamed weights waits for the ready word
//                    (bounded), then "slot free" is recorded for the copy stream.
// No host synchronisation happens inside a pass; ls_run synchronises once at the
// end and then reads the error word the bounded waits write on timeout
// ("layer split: overlap the stages' hand-off", Changes since #936).
#include <cuda_runtime.h>

#include <algorithm>
#include <tuple>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <new>
#include <optional>
#include <string>
#include <vector>

#include "common.cuh"
#include "kernels.h"
#include "ls_api.h"
#include "ls_sched.h"

using namespace ls;

namespace {

constexpr size_t MIN_PARAMS_SIZE = offsetof(ls_params, use_pool) + sizeof(int32_t);
constexpr int64_t ALIGN = 256;
inline int64_t align_up(int64_t n) { return (n + ALIGN - 1) / ALIGN * ALIGN; }

struct TensorRec {
    const void* host = nullptr;
    const void* dev = nullptr;  // device-visible address of the host memory
    uint64_t bytes = 0;
    int dtype = 0, ndim = 0;
    int64_t shape[2] = {0, 0};
    int64_t off = 0;            // offset in the slot (private) or in the shared region (shared)
    int shared_id = -1;
};

struct SegRec {
    std::vector<TensorRec> t;
    int64_t slot_bytes = 0;     // aligned private footprint
    int64_t load_bytes = 0;     // exact private bytes
    bool kernel_ok = true;      // all sources 16-byte aligned
    bool use_kernel = false;    // this segment's loads go through the copy kernel
    CopyRange* ranges_dev = nullptr;
    int n_ranges = 0;
    int64_t n_chunks = 0;
};

struct SharedRec {
    int id;
    const void* host;
    const void* dev;
    uint64_t bytes;
    int64_t off;
};

}  // namespace

struct ls_ctx {
    ls_params prm{};
    int device = 0;
    std::string err;
    bool registered = false;
    int kind = -1;
    int N = 0, H = 0, F = 0, E = 0;
    std::vector<SegRec> segs;
    std::vector<SharedRec> shared;
    std::vector<std::pair<void*, size_t>> host_registered;
    Scheduler sched;
    // device memory
    void* shared_dev = nullptr;
    void* pool = nullptr;
    int64_t pool_bytes = 0;
    int64_t slot_stride = 0;             // bytes between slots (slot size + canary with debug_checks)
    int pool_slots = 0;
    int64_t shared_bytes_dev = 0;        // the shared region's bytes before its canary
    int64_t debug_violations = 0;
    std::vector<void*> seg_buf;          // pool off: current buffer of each segment
    uint32_t* ready = nullptr;           // [P] ready words
    uint32_t* tickets = nullptr;         // [P] last-CTA tickets
    std::vector<uint32_t> slot_epoch;
    std::vector<cudaEvent_t> slot_free;
    uint32_t* err_word = nullptr;        // mapped pinned host
    uint32_t* err_word_dev = nullptr;
    cudaStream_t copy_stream = nullptr;
    cudaStream_t own_stream = nullptr;
    cudaEvent_t alloc_event = nullptr;
    cudaEvent_t run_done = nullptr;          // end of the last queued pass
    std::vector<cudaStream_t> pending;       // streams with queued passes
    int copy_path = LS_COPY_ENGINE;          // summary: ENGINE, KERNEL, or AUTO when segments differ
    int kernel_copy_segments = 0;            // segments whose loads go through the copy kernel
    int copy_ctas = 0;
    int reserve_sms = 0;
    double gbs_kernel = 0, gbs_engine = 0;
    int64_t publishes = 0;
    // per-run segment state
    std::vector<uint32_t> seg_epoch;
    std::vector<void*> seg_ptr;
    std::vector<int> seg_slot;
    // workspaces
    int64_t ws_tokens = 0;
    void* act[2] = {nullptr, nullptr};  // fp32 kind: ping-pong activations
    void* xb = nullptr;                 // bf16 kinds: bf16 operand copy of the residual stream
    float* xf = nullptr;                // bf16 kinds: fp32 residual stream (updated in place)
    void* hbuf = nullptr;
    void* ubuf = nullptr;
    float* splitk_ws = nullptr;         // partial tiles of split-K GEMMs at <= 128 tokens (kept for life)
    // MoE workspaces
    int top_k = 0;
    int* moe_sel = nullptr;
    float* moe_w = nullptr;
    int* moe_table = nullptr;
    int* moe_bounds = nullptr;
    uint8_t* moe_used = nullptr;
    uint8_t* moe_used_host = nullptr;      // mapped: routed experts, then the ones to copy from the host
    uint8_t* moe_used_host_dev = nullptr;  // its device address (the copy kernel's expert mask)
    // expert cache of streamed MoE layers
    void* ecache = nullptr;
    int ecache_K = 0;
    int64_t ecache_eb = 0;                 // bytes of one expert blob (G, U, D)
    std::vector<int64_t> ecache_counts;    // [N * E] earlier passes in which the pair was routed
    std::vector<int> ecache_slot;          // [N * E] cache slot of a hot pair, else -1
    // [N][2][E] first B row of each expert's gate/up and down matrices for this pass: in the
    // slot, or (top bit set) in the cache, where hits are read in place
    int* ecache_rows_host = nullptr;       // pinned
    int* ecache_rows_dev = nullptr;
    std::vector<char> ecache_filled;       // [N * E] its blob is in the cache
    std::vector<std::vector<std::pair<int, int>>> ecache_hits, ecache_fills;  // per layer, this pass
    int64_t n_ecache_hits = 0, n_ecache_host = 0;
    void* moe_xs = nullptr;
    void* moe_hs = nullptr;
    float* moe_y = nullptr;
    // host-buffer entry point staging
    void* stage_x = nullptr;
    void* stage_y = nullptr;
    float* stage_logits = nullptr;
    int64_t stage_tokens = 0;
    cudaError_t cuda_err = cudaSuccess;
    // kernel timing (params.kernel_timing)
    struct TimerClass {
        std::string name;
        int64_t launches = 0;
        double total_ms = 0;
    };
    std::vector<TimerClass> tclass;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> tev;  // event pool
    std::vector<int> tev_class;                              // class of each used pair
    std::vector<int> tev_stream, tev_seg;
    size_t tev_used = 0;
    int cur_seg = -1;
    std::vector<ls_trace_event> trace;
    // graph replay of a steady-state pass (ls_run_graph)
    bool capturing = false;               // issuing into a stream capture
    bool capture_stream_ops = true;       // publish inside a capture as a stream memory operation
    cudaStream_t graph_stream = nullptr;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t graph_exec = nullptr;
    cudaEvent_t graph_in = nullptr, graph_out = nullptr, graph_fork = nullptr, graph_join = nullptr;
    const void* graph_x = nullptr;
    void* graph_y = nullptr;
    int64_t graph_T = 0;
    std::vector<ls_sched_event> graph_events;  // the captured pass's schedule (run field 0)
    int64_t graph_captures = 0, graph_replays = 0;
};

namespace {

void set_err(ls_ctx* c, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    c->err = buf;
}

// Regions named by a canary violation (bits 8.. of the error word): pool slot i is i.
constexpr uint32_t CANARY_REGION_SHARED = 0x8000;
constexpr uint32_t CANARY_REGION_SEGMENT = 0x10000;  // + segment: a per-load buffer with the pool off
constexpr uint32_t CHECK_REGION_MOE = 0x20000;       // + layer: that layer's MoE routing tables

#define CK(call)                                                                      \
    do {                                                                              \
        cudaError_t e_ = (call);                                                      \
        if (e_ != cudaSuccess) {                                                      \
            set_err(c, "%s failed: %s", #call, cudaGetErrorString(e_));               \
            return LS_ERR_CUDA;                                                       \
        }                                                                             \
    } while (0)

void* dev_alloc(ls_ctx* c, size_t bytes, cudaStream_t s) {
    if (bytes == 0) return nullptr;
    if (c->prm.alloc_fn) return c->prm.alloc_fn(c->prm.alloc_user, bytes, s);
    void* p = nullptr;
    if (cudaMallocAsync(&p, bytes, s) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return p;
}

void dev_free(ls_ctx* c, void* p, size_t bytes, cudaStream_t s) {
    if (!p) return;
    if (c->prm.free_fn) {
        c->prm.free_fn(c->prm.alloc_user, p, bytes, s);
        return;
    }
    cudaFreeAsync(p, s);
}

inline void track(ls_ctx* c, cudaError_t e) {
    if (e != cudaSuccess && c->cuda_err == cudaSuccess) c->cuda_err = e;
}

// Bracket one launch with events on its own stream (only with kernel_timing on). Modes
// 1 and 2 bracket every launch; mode 3 brackets only the copies and, per segment, the
// compute kernels after the hand-off wait as one "compute" span.
inline bool ktime_on(const ls_ctx* c, const char* name) {
    const int m = c->prm.kernel_timing;
    const bool segment_span = strcmp(name, "compute") == 0;
    if (m == 1 || m == 2) return !segment_span;
    if (m == 3) return segment_span || strncmp(name, "copy_", 5) == 0;
    return false;
}
struct KTime {
    ls_ctx* c;
    cudaStream_t s;
    size_t idx = (size_t)-1;
    KTime(ls_ctx* ctx, const char* name, cudaStream_t st) : c(ctx), s(st) {
        if (!ktime_on(c, name)) return;
        int cls = -1;
        for (size_t i = 0; i < c->tclass.size(); ++i)
            if (c->tclass[i].name == name) cls = (int)i;
        if (cls < 0) {
            c->tclass.push_back({name, 0, 0});
            cls = (int)c->tclass.size() - 1;
        }
        if (c->tev_used == c->tev.size()) {  // grow the pool in batches, not per launch
            const size_t grow = c->tev.empty() ? 4096 : c->tev.size();
            for (size_t g = 0; g < grow; ++g) {
                cudaEvent_t a, b;
                if (cudaEventCreate(&a) != cudaSuccess) break;
                if (cudaEventCreate(&b) != cudaSuccess) {
                    cudaEventDestroy(a);
                    break;
                }
                c->tev.push_back({a, b});
                c->tev_class.push_back(-1);
                c->tev_stream.push_back(0);
                c->tev_seg.push_back(-1);
            }
            cudaGetLastError();
            if (c->tev_used == c->tev.size()) return;
        }
        idx = c->tev_used++;
        c->tev_class[idx] = cls;
        c->tev_stream[idx] = s == c->copy_stream ? 1 : 0;
        c->tev_seg[idx] = c->cur_seg;
        track(c, cudaEventRecord(c->tev[idx].first, s));
    }
    ~KTime() {
        if (idx != (size_t)-1) track(c, cudaEventRecord(c->tev[idx].second, s));
    }
};

// After the run's final synchronisation: fold the recorded pairs into the classes.
void collect_times(ls_ctx* c) {
    const bool tracing = c->prm.kernel_timing >= 2;
    if (tracing) c->trace.clear();
    for (size_t i = 0; i < c->tev_used; ++i) {
        float ms = 0;
        if (cudaEventElapsedTime(&ms, c->tev[i].first, c->tev[i].second) == cudaSuccess) {
            c->tclass[c->tev_class[i]].launches += 1;
            c->tclass[c->tev_class[i]].total_ms += ms;
        } else {
            cudaGetLastError();
        }
        if (tracing) {
            ls_trace_event t{};
            snprintf(t.name, sizeof(t.name), "%s", c->tclass[c->tev_class[i]].name.c_str());
            t.stream = c->tev_stream[i];
            t.segment = c->tev_seg[i];
            float a = 0, b = 0;
            if (cudaEventElapsedTime(&a, c->tev[0].first, c->tev[i].first) != cudaSuccess ||
                cudaEventElapsedTime(&b, c->tev[0].first, c->tev[i].second) != cudaSuccess)
                cudaGetLastError();
            t.start_ms = a;
            t.end_ms = b;
            c->trace.push_back(t);
        }
    }
    c->tev_used = 0;
}

// --------------------------------------------------------------------------- copies
void issue_copy(ls_ctx* c, int seg, void* dst, int slot, uint32_t epoch, cudaStream_t s, bool use_kernel,
                const uint8_t* expert_mask) {
    SegRec& sr = c->segs[seg];
    const bool publish = !(c->prm.test_drop_publish > 0 && ++c->publishes == c->prm.test_drop_publish);
    // expert cache: hits stay where the cache holds them (the GEMMs read them there); hot
    // experts that come from the host this time are copied into the cache after the publish
    const bool cached = c->ecache_K > 0 && expert_mask;
    auto cache_copies = [&](const std::vector<std::pair<int, int>>& list, bool into_slot) {
        for (auto& h : list) {
            uint8_t* sl = (uint8_t*)dst + (int64_t)h.first * c->ecache_eb;
            uint8_t* ca = (uint8_t*)c->ecache + (int64_t)h.second * c->ecache_eb;
            track(c, cudaMemcpyAsync(into_slot ? sl : ca, into_slot ? ca : sl, (size_t)c->ecache_eb,
                                     cudaMemcpyDeviceToDevice, s));
        }
    };
    if (use_kernel && sr.kernel_ok) {
        KTime kt(c, "copy_h2slot", s);
        track(c, launch_copy_h2slot(sr.ranges_dev, sr.n_ranges, sr.n_chunks, dst, expert_mask,
                                    expert_mask ? 3 : 1, c->ready + slot, c->tickets + slot, epoch,
                                    publish, c->copy_ctas, s));
        if (cached) cache_copies(c->ecache_fills[seg], false);
        return;
    }
    // copy engine: one copy per tensor (contiguous neighbours merged), then publish
    KTime kt(c, "copy_engine", s);
    const bool moe = c->kind == LS_KIND_MOE_SWIGLU_BF16;
    int64_t run_dst = 0, run_len = 0;
    const uint8_t* host_src0 = nullptr;
    auto flush = [&]() {
        if (run_len > 0)
            track(c, cudaMemcpyAsync((uint8_t*)dst + run_dst, host_src0, run_len, cudaMemcpyHostToDevice, s));
        run_len = 0;
    };
    for (size_t i = 0; i < sr.t.size(); ++i) {
        const TensorRec& t = sr.t[i];
        if (t.shared_id >= 0) continue;
        if (moe && expert_mask && !c->moe_used_host[(int64_t)seg * c->E + i / 3]) {
            flush();
            continue;
        }
        const uint8_t* src = (const uint8_t*)t.host;
        if (run_len > 0 && src == host_src0 + run_len && t.off == run_dst + run_len) {
            run_len += (int64_t)t.bytes;
        } else {
            flush();
            host_src0 = src;
            run_dst = t.off;
            run_len = (int64_t)t.bytes;
        }
    }
    flush();
    track(c, launch_publish(c->ready + slot, epoch, publish, s, !c->capturing || c->capture_stream_ops,
                            c->capturing));
    if (cached) cache_copies(c->ecache_fills[seg], false);
}

// --------------------------------------------------------------------------- compute
const void* tptr(ls_ctx* c, int seg, int i) {
    const TensorRec& t = c->segs[seg].t[i];
    if (t.shared_id >= 0) return (const uint8_t*)c->shared_dev + t.off;
    return (const uint8_t*)c->seg_ptr[seg] + t.off;
}

int gemm_ctas(ls_ctx* c) {
    int sms = gemm_num_sms();
    int r = c->reserve_sms;
    if (r < 0) r = 0;
    return std::max(1, sms - r);
}

struct RunCtx {
    const void* x;
    void* y;
    int64_t T;
    cudaStream_t s;
    uint64_t wait_ns;
};

// Activations between segments: the fp32 kind ping-pongs two buffers; the bf16
// kinds carry the residual stream in fp32 (xf, updated in place: every output
// element reads and writes only its own residual element) plus its bf16
// rounding (xb) as the next GEMM operand. Segment 0 reads the caller's bf16 x;
// the last segment writes the caller's bf16 y.
void compute_segment(ls_ctx* c, const RunCtx& rc, int seg, bool wait) {
    const int N = c->N;
    const bool first = seg == 0, last = seg == N - 1;
    const void* xin = first ? rc.x : (c->kind == LS_KIND_LINEAR_GELU_F32 ? c->act[(seg - 1) & 1] : c->xb);
    void* xout = last ? rc.y : (c->kind == LS_KIND_LINEAR_GELU_F32 ? c->act[seg & 1] : c->xb);
    const void* rin = first ? rc.x : (const void*)c->xf;   // residual input
    const bool rin_f32 = !first;
    float* xout32 = last ? nullptr : c->xf;                // fp32 residual output
    const int T = (int)rc.T, H = c->H, F = c->F;
    const int slot = c->seg_slot[seg];
    const uint32_t epoch = c->seg_epoch[seg];
    const uint32_t code = DERR_HANDOFF_TIMEOUT | ((uint32_t)slot << 8);
    // Kernels overlap their prologue with the previous kernel's tail (programmatic
    // dependent launch) except while events bracket each launch (timing modes 1 and 2):
    // an event pair then times its kernel alone.
    const bool pdl = c->prm.kernel_timing == 0 || c->prm.kernel_timing == 3;
    std::optional<KTime> span;  // mode 3: the segment's compute kernels after the hand-off wait
    auto open_span = [&]() {
        if (c->prm.kernel_timing == 3 && !span) span.emplace(c, "compute", rc.s);
    };
    // A prefetched segment's kernels start behind a one-CTA wait on the slot's
    // ready word. The wait is its own launch: a spinning waiter must hold almost
    // nothing, so the copy it waits for can always find SMs to run on.
    auto wait_slot = [&]() {
        KTime kt(c, "wait_ready", rc.s);
        // the GEMM behind it may be placed early only if nothing on the copy stream needs an
        // SM (no copy or publish kernel that the placed CTAs could starve; device-to-device
        // copies of the expert cache may run as kernels too)
        const bool early = c->kernel_copy_segments == 0 && publish_needs_no_sm() &&
                           (!c->capturing || c->capture_stream_ops) && c->ecache_K == 0 && pdl;
        track(c, launch_wait_ready(c->ready + slot, epoch, rc.wait_ns, c->err_word_dev, code, rc.s, early));
        open_span();
    };
    GemmDesc w0;
    w0.err_word = c->err_word_dev;
    w0.pdl = pdl;
    w0.splitk_ws = c->splitk_ws;
    w0.splitk_ws_bytes = c->splitk_ws ? gemm_split_ws_max() : 0;
    const int ctas = gemm_ctas(c);
    if (!wait) open_span();
    switch (c->kind) {
        case LS_KIND_LINEAR_GELU_F32: {
            if (wait) wait_slot();
            KTime kt(c, "linear_gelu_f32", rc.s);
            track(c, launch_linear_gelu_f32((const float*)xin, (const float*)tptr(c, seg, 0),
                                            (const float*)tptr(c, seg, 1), (float*)xout, T, H, F, rc.s, pdl));
            break;
        }
        case LS_KIND_FFN_GELU_BF16:
        case LS_KIND_FFN_GELU_SHARED_BF16: {
            const bool proj = c->kind == LS_KIND_FFN_GELU_SHARED_BF16;
            const int o = proj ? 1 : 0;
            const void* a1 = xin;
            if (proj) {  // reads only the resident shared projection: runs before the wait

                GemmDesc g;
                g.pdl = pdl;
                g.epi = EPI_STORE;
                g.A = xin; g.lda = H; g.a_rows = T;
                g.B = tptr(c, seg, 0); g.ldb = H; g.b_rows = H;
                g.M = T; g.N = H; g.K = H;
                g.C = c->ubuf; g.ldc = H;
                g.err_word = c->err_word_dev;
                KTime kt(c, "gemm_proj", rc.s);
                track(c, launch_gemm_bf16(g, ctas, rc.s));
                a1 = c->ubuf;
            }
            if (wait) wait_slot();
            GemmDesc g1 = w0;
            g1.epi = EPI_BIAS_GELU;
            g1.A = a1; g1.lda = H; g1.a_rows = T;
            g1.B = tptr(c, seg, o + 0); g1.ldb = H; g1.b_rows = F;
            g1.bias = tptr(c, seg, o + 1);
            g1.M = T; g1.N = F; g1.K = H;
            g1.C = c->hbuf; g1.ldc = F;
            {
                KTime kt(c, "gemm_up", rc.s);
                track(c, launch_gemm_bf16(g1, ctas, rc.s));
            }
            GemmDesc g2 = w0;
            g2.epi = EPI_BIAS_RESID;
            g2.A = c->hbuf; g2.lda = F; g2.a_rows = T;
            g2.B = tptr(c, seg, o + 2); g2.ldb = F; g2.b_rows = H;
            g2.bias = tptr(c, seg, o + 3);
            g2.resid = rin; g2.resid_f32 = rin_f32; g2.ldr = H;
            g2.M = T; g2.N = H; g2.K = F;
            g2.C = xout; g2.ldc = H; g2.C32 = xout32;
            KTime kt(c, "gemm_down", rc.s);
            track(c, launch_gemm_bf16(g2, ctas, rc.s));
            break;
        }
        case LS_KIND_SWIGLU_BF16: {
            if (wait) wait_slot();
            GemmDesc g1 = w0;
            g1.epi = EPI_SWIGLU;
            g1.A = xin; g1.lda = H; g1.a_rows = T;
            g1.B = tptr(c, seg, 0); g1.ldb = H; g1.b_rows = 2 * (int64_t)F;
            g1.b2_row_off = F;
            g1.M = T; g1.N = F; g1.K = H;
            g1.C = c->hbuf; g1.ldc = F;
            {
                KTime kt(c, "gemm_up", rc.s);
                track(c, launch_gemm_bf16(g1, ctas, rc.s));
            }
            GemmDesc g2 = w0;
            g2.epi = EPI_RESID;
            g2.A = c->hbuf; g2.lda = F; g2.a_rows = T;
            g2.B = tptr(c, seg, 2); g2.ldb = F; g2.b_rows = H;
            g2.resid = rin; g2.resid_f32 = rin_f32; g2.ldr = H;
            g2.M = T; g2.N = H; g2.K = F;
            g2.C = xout; g2.ldc = H; g2.C32 = xout32;
            KTime kt(c, "gemm_down", rc.s);
            track(c, launch_gemm_bf16(g2, ctas, rc.s));
            break;
        }
        case LS_KIND_MOE_SWIGLU_BF16: {
            const int k = c->top_k, E = c->E;
            const int rows = T * k;
            const int* table = c->moe_table + (int64_t)seg * rows;
            const int* bounds = c->moe_bounds + (int64_t)seg * (E + 1);
            {
                KTime kt(c, "moe_gather", rc.s);
                track(c, launch_moe_gather(xin, table, rows, k, H, c->moe_xs, rc.s));
            }
            const int64_t eb = c->segs[seg].slot_bytes / E;  // bytes per expert (G, U, D packed)
            const void* base = c->seg_ptr[seg];
            if (wait) wait_slot();
            GemmDesc g1 = w0;
            g1.epi = EPI_SWIGLU;
            g1.A = c->moe_xs; g1.lda = H; g1.a_rows = rows;
            g1.B = base; g1.ldb = H; g1.b_rows = c->segs[seg].slot_bytes / (2 * (int64_t)H);
            g1.b2_row_off = F;
            g1.M = rows; g1.N = F; g1.K = H;
            g1.C = c->moe_hs; g1.ldc = F;
            g1.group_bounds = bounds; g1.n_groups = E;
            g1.b_group_stride_rows = (int)(eb / (2 * (int64_t)H));
            g1.b_base_row = 0;
            const bool in_cache = c->ecache_K > 0 && seg >= c->sched.residents();
            if (in_cache) {  // hot experts of streamed layers are read where the cache holds them
                g1.group_b_row = c->ecache_rows_dev + (size_t)seg * 2 * E;
                g1.B2 = c->ecache;
                g1.b2_rows = (int64_t)c->ecache_K * (eb / (2 * (int64_t)H));
            }
            {
                KTime kt(c, "gemm_up", rc.s);
                track(c, launch_gemm_bf16(g1, ctas, rc.s));
            }
            GemmDesc g2 = w0;
            g2.epi = EPI_SCALE_F32;
            g2.A = c->moe_hs; g2.lda = F; g2.a_rows = rows;
            g2.B = base; g2.ldb = F; g2.b_rows = c->segs[seg].slot_bytes / (2 * (int64_t)F);
            g2.M = rows; g2.N = H; g2.K = F;
            g2.C = c->moe_y; g2.ldc = H;
            g2.group_bounds = bounds; g2.n_groups = E;
            g2.b_group_stride_rows = (int)(eb / (2 * (int64_t)F));
            g2.b_base_row = (int)(2 * (int64_t)F * H * 2 / (2 * (int64_t)F));
            g2.row_table = table;
            g2.row_weight = c->moe_w + (int64_t)seg * rows;
            if (in_cache) {
                g2.group_b_row = c->ecache_rows_dev + (size_t)seg * 2 * E + E;
                g2.B2 = c->ecache;
                g2.b2_rows = (int64_t)c->ecache_K * (eb / (2 * (int64_t)F));
            }
            {
                KTime kt(c, "gemm_down", rc.s);
                track(c, launch_gemm_bf16(g2, ctas, rc.s));
            }
            KTime kt(c, "moe_combine", rc.s);
            track(c, launch_moe_combine(rin, rin_f32, c->moe_y, T, k, H, xout, xout32, rc.s));
            break;
        }
    }
}

// --------------------------------------------------------------------------- executors
struct GpuExec : Executor {
    ls_ctx* c;
    RunCtx rc;
    explicit GpuExec(ls_ctx* ctx) : c(ctx) { rc = RunCtx{nullptr, nullptr, 0, nullptr, 0}; }

    // With debug_checks every allocation carries a canary after its last byte.
    int64_t canary() const { return c->prm.debug_checks ? CANARY_BYTES : 0; }
    bool alloc_shared(int64_t bytes) override {
        c->shared_dev = dev_alloc(c, (size_t)(bytes + canary()), c->copy_stream);
        c->shared_bytes_dev = bytes;
        if (c->shared_dev && canary())
            track(c, launch_canary((uint8_t*)c->shared_dev + bytes, 0, 1, false, nullptr, 0, c->copy_stream));
        return c->shared_dev != nullptr;
    }
    bool alloc_pool(int slots, int64_t slot_bytes) override {
        const int64_t stride = slot_bytes + canary();
        c->pool = dev_alloc(c, (size_t)(slots * stride), c->copy_stream);
        c->pool_bytes = slots * stride;
        c->slot_stride = stride;
        c->pool_slots = slots;
        if (c->pool && canary())
            track(c, launch_canary((uint8_t*)c->pool + slot_bytes, stride, slots, false, nullptr, 0, c->copy_stream));
        return c->pool != nullptr;
    }
    bool alloc_segment(int seg, int64_t bytes) override {
        c->seg_buf[seg] = dev_alloc(c, (size_t)(bytes + canary()), rc.s);
        if (c->seg_buf[seg] && canary())
            track(c, launch_canary((uint8_t*)c->seg_buf[seg] + bytes, 0, 1, false, nullptr, 0, rc.s));
        return c->seg_buf[seg] != nullptr;
    }
    // pool off: a per-load buffer's canary is checked right before the buffer is freed
    void check_segment_canary(int seg, cudaStream_t s) {
        if (!canary() || !c->seg_buf[seg]) return;
        track(c, launch_canary((uint8_t*)c->seg_buf[seg] + c->segs[seg].slot_bytes, 0, 1, true, c->err_word_dev,
                               CANARY_REGION_SEGMENT + (uint32_t)seg, s));
    }
    void free_segment(int seg) override {
        check_segment_canary(seg, rc.s);
        dev_free(c, c->seg_buf[seg], (size_t)(c->segs[seg].slot_bytes + canary()), rc.s);
        c->seg_buf[seg] = nullptr;
    }
    void begin_run(int) override {}
    void load_shared(int id) override {
        for (auto& s : c->shared)
            if (s.id == id)
                track(c, cudaMemcpyAsync((uint8_t*)c->shared_dev + s.off, s.host, s.bytes,
                                         cudaMemcpyHostToDevice, rc.s));
    }
    void load(int seg, int slot, int kind, int64_t) override {
        c->cur_seg = seg;
        void* dst = c->prm.use_pool ? (uint8_t*)c->pool + (int64_t)slot * c->slot_stride : c->seg_buf[seg];
        const uint32_t epoch = ++c->slot_epoch[slot];
        c->seg_epoch[seg] = epoch;
        c->seg_ptr[seg] = dst;
        c->seg_slot[seg] = slot;
        // a streamed MoE load moves the experts routed in this pass; a resident keeps all of
        // them, since later passes may route to any
        const uint8_t* mask = c->kind == LS_KIND_MOE_SWIGLU_BF16 && kind != LS_EV_LOAD_RESIDENT
                                  ? c->moe_used_host_dev + (int64_t)seg * c->E
                                  : nullptr;
        const bool kern = c->segs[seg].use_kernel;
        if (kind == LS_EV_PREFETCH) {
            track(c, cudaStreamWaitEvent(c->copy_stream, c->slot_free[slot], 0));
            if (!c->prm.use_pool) {  // the buffer was allocated in compute-stream order
                track(c, cudaEventRecord(c->alloc_event, rc.s));
                track(c, cudaStreamWaitEvent(c->copy_stream, c->alloc_event, 0));
            }
            issue_copy(c, seg, dst, slot, epoch, c->copy_stream, kern, mask);
        } else {
            issue_copy(c, seg, dst, slot, epoch, rc.s, kern, mask);
        }
    }
    void activate(int seg, int slot, bool via_queue) override {
        c->cur_seg = seg;
        compute_segment(c, rc, seg, via_queue);
        track(c, cudaEventRecord(c->slot_free[slot], rc.s));
    }
    void evict(int seg, int) override {
        check_segment_canary(seg, rc.s);
        dev_free(c, c->seg_buf[seg], (size_t)(c->segs[seg].slot_bytes + canary()), rc.s);
        c->seg_buf[seg] = nullptr;
    }
    void free_pool() override {
        dev_free(c, c->pool, (size_t)c->pool_bytes, c->copy_stream);
        c->pool = nullptr;
        c->pool_bytes = 0;
        c->pool_slots = 0;
    }
};

struct DryExec : Executor {
    bool alloc_shared(int64_t) override { return true; }
    bool alloc_pool(int, int64_t) override { return true; }
    bool alloc_segment(int, int64_t) override { return true; }
    void free_segment(int) override {}
    void begin_run(int) override {}
    void load_shared(int) override {}
    void load(int, int, int, int64_t) override {}
    void activate(int, int, bool) override {}
    void evict(int, int) override {}
    void free_pool() override {}
};

ls_status check_params(const ls_params* p, ls_params* out, std::string* why) {
    if (!p) {
        *why = "params is NULL";
        return LS_ERR_INVALID_ARG;
    }
    if (p->version != LS_PARAMS_VERSION) {
        *why = "unknown params version";
        return LS_ERR_VERSION;
    }
    if (p->struct_size < MIN_PARAMS_SIZE) {
        *why = "params struct_size below the minimum";
        return LS_ERR_VERSION;
    }
    ls_params d;
    ls_params_init(&d);
    size_t n = std::min<size_t>(p->struct_size, sizeof(ls_params));
    memcpy(&d, p, n);
    d.struct_size = sizeof(ls_params);
    if (d.prefetch_depth < 0) { *why = "prefetch_depth < 0"; return LS_ERR_INVALID_ARG; }
    if (d.resident_layers < -1) { *why = "resident_layers < -1"; return LS_ERR_INVALID_ARG; }
    if (d.max_vram_bytes < 0) { *why = "max_vram_bytes < 0"; return LS_ERR_INVALID_ARG; }
    if (d.use_pool != 0 && d.use_pool != 1) { *why = "use_pool must be 0 or 1"; return LS_ERR_INVALID_ARG; }
    if (d.wait_limit_ms < 1 || d.wait_limit_ms > 600000) {
        *why = "wait_limit_ms must be in 1..600000 (device waits are always bounded)";
        return LS_ERR_INVALID_ARG;
    }
    if (d.copy_path < LS_COPY_AUTO || d.copy_path > LS_COPY_ENGINE) { *why = "bad copy_path"; return LS_ERR_INVALID_ARG; }
    if (d.copy_ctas < 0 || d.test_alloc_cap_bytes < 0 || d.test_drop_publish < 0 || d.kernel_timing < 0 ||
        d.kernel_timing > 3 || d.test_kernel_copy_stride < 0) {
        *why = "negative count";
        return LS_ERR_INVALID_ARG;
    }
    if ((d.alloc_fn == nullptr) != (d.free_fn == nullptr)) { *why = "alloc_fn and free_fn go together"; return LS_ERR_INVALID_ARG; }
    if (d.cross_run_prefetch != 0 && d.cross_run_prefetch != 1) { *why = "cross_run_prefetch must be 0 or 1"; return LS_ERR_INVALID_ARG; }
    if (d.expert_cache_bytes < 0) { *why = "expert_cache_bytes < 0"; return LS_ERR_INVALID_ARG; }
    if (d.debug_checks != 0 && d.debug_checks != 1) { *why = "debug_checks must be 0 or 1"; return LS_ERR_INVALID_ARG; }
    if (d.test_corrupt_canary < 0) { *why = "test_corrupt_canary < 0"; return LS_ERR_INVALID_ARG; }
    *out = d;
    return LS_OK;
}

// Pin and map every host range that is not pinned yet. Exactly the tensors'
// bytes are registered (ranges that overlap or touch are merged), never whole
// pages: a page-rounded range would also register the neighbouring bytes of
// other allocations, and a copy of the caller's that straddles the end of a
// registered range is refused by the driver.
ls_status pin_host(ls_ctx* c, std::vector<std::pair<const void*, uint64_t>>& ranges) {
    std::vector<std::pair<uintptr_t, uintptr_t>> todo;
    for (auto& r : ranges) {
        if (!r.first || !r.second) continue;
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, r.first) == cudaSuccess && a.type == cudaMemoryTypeHost) continue;
        cudaGetLastError();
        todo.push_back({(uintptr_t)r.first, (uintptr_t)r.first + r.second});
    }
    std::sort(todo.begin(), todo.end());
    std::vector<std::pair<uintptr_t, uintptr_t>> merged;
    for (auto& r : todo) {
        if (!merged.empty() && r.first <= merged.back().second)
            merged.back().second = std::max(merged.back().second, r.second);
        else
            merged.push_back(r);
    }
    for (auto& r : merged) {
        cudaError_t e = cudaHostRegister((void*)r.first, r.second - r.first,
                                         cudaHostRegisterMapped | cudaHostRegisterPortable);
        if (e != cudaSuccess) {
            cudaGetLastError();
            set_err(c, "cudaHostRegister of %zu bytes failed: %s", (size_t)(r.second - r.first),
                    cudaGetErrorString(e));
            return LS_ERR_CUDA;
        }
        c->host_registered.push_back({(void*)r.first, r.second - r.first});
    }
    return LS_OK;
}

const void* mapped_ptr(const void* host) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, host) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.devicePointer;
}

ls_status validate_layout(ls_ctx* c) {
    const int k = c->kind;
    auto shape_is = [](const TensorRec& t, int64_t a, int64_t b) {
        return b < 0 ? (t.ndim == 1 && t.shape[0] == a) : (t.ndim == 2 && t.shape[0] == a && t.shape[1] == b);
    };
    for (int s = 0; s < c->N; ++s) {
        const auto& t = c->segs[s].t;
        bool ok = true;
        const int dt = k == LS_KIND_LINEAR_GELU_F32 ? LS_DTYPE_F32 : LS_DTYPE_BF16;
        for (auto& x : t) {
            ok &= x.dtype == dt;
            ok &= x.bytes == (uint64_t)(x.shape[0] * (x.ndim == 2 ? x.shape[1] : 1) * (dt == LS_DTYPE_F32 ? 4 : 2));
        }
        if (k == LS_KIND_LINEAR_GELU_F32)
            ok &= t.size() == 2 && t[0].ndim == 2 && shape_is(t[1], t[0].shape[0], -1);
        else if (k == LS_KIND_FFN_GELU_BF16 || k == LS_KIND_FFN_GELU_SHARED_BF16) {
            int o = k == LS_KIND_FFN_GELU_SHARED_BF16 ? 1 : 0;
            ok &= (int)t.size() == 4 + o;
            if (ok) {
                int64_t Fh = t[o].shape[0], Hh = t[o].shape[1];
                ok &= shape_is(t[o + 1], Fh, -1) && shape_is(t[o + 2], Hh, Fh) && shape_is(t[o + 3], Hh, -1);
                if (o) ok &= shape_is(t[0], Hh, Hh) && t[0].shared_id >= 0;
                for (int i = o; i < 4 + o; ++i) ok &= t[i].shared_id < 0;
            }
        } else if (k == LS_KIND_SWIGLU_BF16) {
            ok &= t.size() == 3;
            if (ok) {
                int64_t Fh = t[0].shape[0], Hh = t[0].shape[1];
                ok &= shape_is(t[1], Fh, Hh) && shape_is(t[2], Hh, Fh);
                ok &= t[1].off == t[0].off + (int64_t)t[0].bytes;  // G and U adjacent: one [2F, H] view
            }
        } else if (k == LS_KIND_MOE_SWIGLU_BF16) {
            ok &= t.size() % 3 == 0 && !t.empty() && t.size() / 3 <= 256;
            if (ok) {
                int64_t Fh = t[0].shape[0], Hh = t[0].shape[1];
                int64_t eb = 3 * Fh * Hh * 2;
                for (size_t e = 0; e < t.size() / 3 && ok; ++e) {
                    ok &= shape_is(t[3 * e], Fh, Hh) && shape_is(t[3 * e + 1], Fh, Hh) && shape_is(t[3 * e + 2], Hh, Fh);
                    ok &= t[3 * e].off == (int64_t)e * eb && t[3 * e + 1].off == t[3 * e].off + Fh * Hh * 2 &&
                          t[3 * e + 2].off == t[3 * e].off + 2 * Fh * Hh * 2;
                }
            }
        } else {
            ok = false;
        }
        if (!ok) {
            set_err(c, "segment %d: tensors do not match kind %d's layout", s, k);
            return LS_ERR_UNSUPPORTED;
        }
    }
    // dims of the stack
    const auto& t0 = c->segs[0].t;
    if (k == LS_KIND_LINEAR_GELU_F32) {
        c->F = (int)t0[0].shape[0];
        c->H = (int)t0[0].shape[1];
        if (c->F != c->H) {
            set_err(c, "fp32 linear stack: out features must equal in features");
            return LS_ERR_UNSUPPORTED;
        }
    } else {
        int o = k == LS_KIND_FFN_GELU_SHARED_BF16 ? 1 : 0;
        c->F = (int)t0[o].shape[0];
        c->H = (int)t0[o].shape[1];
        if (k == LS_KIND_MOE_SWIGLU_BF16) c->E = (int)(t0.size() / 3);
        if ((c->H % 8) || (c->F % 8)) {
            set_err(c, "bf16 kinds need hidden and ffn sizes that are multiples of 8");
            return LS_ERR_UNSUPPORTED;
        }
    }
    for (int s = 1; s < c->N; ++s) {
        int o = k == LS_KIND_FFN_GELU_SHARED_BF16 ? 1 : 0;
        if (c->segs[s].t.size() != t0.size() || c->segs[s].t[o].shape[0] != t0[o].shape[0] ||
            c->segs[s].t[o].shape[1] != t0[o].shape[1]) {
            set_err(c, "segment %d has other dimensions than segment 0", s);
            return LS_ERR_UNSUPPORTED;
        }
    }
    return LS_OK;
}

ls_status build_ranges(ls_ctx* c, SegRec& sr) {
    std::vector<CopyRange> v;
    int64_t chunk = 0;
    for (auto& t : sr.t) {
        if (t.shared_id >= 0) continue;
        if (((uintptr_t)t.dev & 15) != 0) sr.kernel_ok = false;
        CopyRange r{};
        r.src = t.dev;
        r.dst_off = t.off;
        r.n16 = (int64_t)(t.bytes / 16);
        r.tail = (int32_t)(t.bytes % 16);
        r.chunk_begin = chunk;
        chunk += std::max<int64_t>(1, copy_chunks_for(r.n16));
        v.push_back(r);
    }
    for (auto& r : v)  // every range ends inside the slot (the layout is built above; a cheap guard)
        if (r.dst_off < 0 || r.dst_off + r.n16 * 16 + r.tail > sr.slot_bytes) {
            set_err(c, "internal: a copy range ends past its slot");
            return LS_ERR_INVALID_ARG;
        }
    sr.n_ranges = (int)v.size();
    sr.n_chunks = chunk;
    if (v.empty()) return LS_OK;
    CK(cudaMalloc(&sr.ranges_dev, v.size() * sizeof(CopyRange)));
    CK(cudaMemcpy(sr.ranges_dev, v.data(), v.size() * sizeof(CopyRange), cudaMemcpyHostToDevice));
    return LS_OK;
}

// The copy path of every segment's loads. A forced path applies to every segment (the copy
// kernel only where the segment's sources are 16-byte aligned). AUTO times both paths on
// each segment's own load, once each after an untimed warm-up of both (copy stream, into the
// first slot or a scratch buffer): how fast the copy engine reads pinned host memory differs
// between regions of the same host buffer. On GB300 hosts whose memory had been through large
// allocate-and-free cycles, the copy engine read the first ~14 GB of a 58 GB stack at a third
// to a tenth of the link rate while the copy kernel's loads read the same pages at the full
// rate, so one segment's timing does not speak for the others.
ls_status autotune_copy(ls_ctx* c) {
    const Plan& p = c->sched.plan();
    const int N = p.N;
    const int forced = c->prm.copy_path;
    auto summarize = [&]() {
        c->kernel_copy_segments = 0;
        for (int i = 0; i < N; ++i) c->kernel_copy_segments += c->segs[i].use_kernel ? 1 : 0;
        c->copy_path = c->kernel_copy_segments == 0   ? LS_COPY_ENGINE
                       : c->kernel_copy_segments == N ? LS_COPY_KERNEL
                                                      : LS_COPY_AUTO;
    };
    if (forced != LS_COPY_AUTO || p.N - p.R <= 0) {  // forced, or nothing streamed
        for (int i = 0; i < N; ++i) c->segs[i].use_kernel = forced == LS_COPY_KERNEL && c->segs[i].kernel_ok;
        summarize();
        return LS_OK;
    }
    if (c->prm.test_kernel_copy_stride > 0) {  // test hook: a fixed mix of the two paths
        for (int i = 0; i < N; ++i)
            c->segs[i].use_kernel = i % c->prm.test_kernel_copy_stride == 0 && c->segs[i].kernel_ok;
        summarize();
        return LS_OK;
    }
    int64_t max_slot = 0;
    for (int i = 0; i < N; ++i) max_slot = std::max(max_slot, c->segs[i].slot_bytes);
    void* dst = c->pool;
    void* scratch = nullptr;
    if (!dst) {
        CK(cudaMalloc(&scratch, (size_t)max_slot));
        dst = scratch;
    }
    if (c->kind == LS_KIND_MOE_SWIGLU_BF16) {  // time with every expert routed
        CK(cudaMemset(c->moe_used, 1, (size_t)N * c->E));
        memset(c->moe_used_host, 1, (size_t)N * c->E);
    }
    cudaEvent_t e0, e1;
    CK(cudaEventCreate(&e0));
    CK(cudaEventCreate(&e1));
    const int saved_drop = c->prm.test_drop_publish;
    const int saved_timing = c->prm.kernel_timing;
    c->prm.test_drop_publish = 0;
    c->prm.kernel_timing = 0;
    uint32_t epoch = 0x80000000u;
    auto time_load = [&](int seg, bool kern, float* ms) -> ls_status {
        const uint8_t* mask = c->kind == LS_KIND_MOE_SWIGLU_BF16 ? c->moe_used + (int64_t)seg * c->E : nullptr;
        CK(cudaEventRecord(e0, c->copy_stream));
        issue_copy(c, seg, dst, 0, epoch++, c->copy_stream, kern, mask);
        CK(cudaEventRecord(e1, c->copy_stream));
        CK(cudaEventSynchronize(e1));
        CK(c->cuda_err);
        CK(cudaEventElapsedTime(ms, e0, e1));
        return LS_OK;
    };
    // The copy kernel occupies SM issue slots and registers next to the segment's GEMMs
    // while the copy engine uses none, so a segment takes the kernel only when it is
    // clearly faster on that segment's load (by more than KERNEL_MARGIN).
    constexpr double KERNEL_MARGIN = 1.15;
    double bytes_k = 0, bytes_e = 0, ms_k = 0, ms_e = 0;
    float ms = 0;
    ls_status st = LS_OK;
    for (int kern = 0; kern < 2 && st == LS_OK; ++kern)  // warm-up of both paths
        if (!kern || c->segs[N - 1].kernel_ok) st = time_load(N - 1, kern != 0, &ms);
    // One reading per path and segment, in segment order as a pass reads them: the engine's
    // reading of a segment comes after the other segments' loads. A second engine reading of
    // the same segment right after its first was fast for host regions that the engine read
    // slowly in every pass, so it is not taken.
    for (int seg = 0; seg < N && st == LS_OK; ++seg) {
        SegRec& sr = c->segs[seg];
        sr.use_kernel = false;
        if (sr.load_bytes == 0) continue;
        float me = 0, mk = 0;
        if ((st = time_load(seg, false, &me)) != LS_OK) break;
        bytes_e += (double)sr.load_bytes;
        ms_e += me;
        if (!sr.kernel_ok) continue;
        if ((st = time_load(seg, true, &mk)) != LS_OK) break;
        bytes_k += (double)sr.load_bytes;
        ms_k += mk;
        sr.use_kernel = (double)mk * KERNEL_MARGIN < (double)me;
    }
    c->prm.test_drop_publish = saved_drop;
    c->prm.kernel_timing = saved_timing;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (st != LS_OK) {
        if (scratch) cudaFree(scratch);
        return st;
    }
    CK(cudaMemsetAsync(c->ready, 0, sizeof(uint32_t) * std::max(1, p.P), c->copy_stream));
    CK(cudaStreamSynchronize(c->copy_stream));
    if (scratch) cudaFree(scratch);
    c->gbs_kernel = ms_k > 0 ? bytes_k / (ms_k * 1e-3) / 1e9 : 0;
    c->gbs_engine = ms_e > 0 ? bytes_e / (ms_e * 1e-3) / 1e9 : 0;
    summarize();
    return LS_OK;
}

// Waits for the work this context queued: its passes' streams, the copy stream, the
// host-buffer stream and the graph stream. Other streams of the device are not waited on.
void sync_ctx_streams(ls_ctx* c) {
    for (cudaStream_t s : c->pending) cudaStreamSynchronize(s);
    for (cudaStream_t s : {c->copy_stream, c->own_stream, c->graph_stream})
        if (s) cudaStreamSynchronize(s);
}

// Workspaces are stream-ordered allocations on the copy stream, so replacing them
// never synchronises the whole device (a plain cudaFree would).
void free_workspaces(ls_ctx* c) {
    for (void** p : {&c->act[0], &c->act[1], &c->xb, (void**)&c->xf, &c->hbuf, &c->ubuf, &c->moe_xs, &c->moe_hs,
                     (void**)&c->moe_sel, (void**)&c->moe_w, (void**)&c->moe_table, (void**)&c->moe_y})
        if (*p) {
            cudaFreeAsync(*p, c->copy_stream);
            *p = nullptr;
        }
    c->ws_tokens = 0;
}

ls_status ensure_workspace(ls_ctx* c, int64_t T) {
    if (T <= c->ws_tokens) return LS_OK;
    sync_ctx_streams(c);   // no queued pass of this context uses the old workspaces any more
    free_workspaces(c);
    cudaStream_t a = c->copy_stream;
    if (c->N > 1 && c->kind == LS_KIND_LINEAR_GELU_F32) {
        CK(cudaMallocAsync(&c->act[0], (size_t)T * c->H * 4, a));
        CK(cudaMallocAsync(&c->act[1], (size_t)T * c->H * 4, a));
    } else if (c->N > 1) {
        CK(cudaMallocAsync(&c->xb, (size_t)T * c->H * 2, a));
        CK(cudaMallocAsync((void**)&c->xf, (size_t)T * c->H * 4, a));
    }
    if (c->kind == LS_KIND_FFN_GELU_BF16 || c->kind == LS_KIND_FFN_GELU_SHARED_BF16 || c->kind == LS_KIND_SWIGLU_BF16)
        CK(cudaMallocAsync(&c->hbuf, (size_t)T * c->F * 2, a));
    if (c->kind == LS_KIND_FFN_GELU_SHARED_BF16) CK(cudaMallocAsync(&c->ubuf, (size_t)T * c->H * 2, a));
    if (c->kind == LS_KIND_MOE_SWIGLU_BF16) {
        const int64_t rows = T * 8;
        CK(cudaMallocAsync((void**)&c->moe_sel, (size_t)c->N * rows * sizeof(int), a));
        CK(cudaMallocAsync((void**)&c->moe_w, (size_t)c->N * rows * sizeof(float), a));
        CK(cudaMallocAsync((void**)&c->moe_table, (size_t)c->N * rows * sizeof(int), a));
        CK(cudaMallocAsync(&c->moe_xs, (size_t)rows * c->H * 2, a));
        CK(cudaMallocAsync(&c->moe_hs, (size_t)rows * c->F * 2, a));
        CK(cudaMallocAsync((void**)&c->moe_y, (size_t)rows * c->H * sizeof(float), a));
    }
    // dense bf16 kinds: the split-K workspace of small token counts, allocated once, so that a
    // given token count always takes the same path (and gives the same bits)
    if (!c->splitk_ws && (c->kind == LS_KIND_FFN_GELU_BF16 || c->kind == LS_KIND_FFN_GELU_SHARED_BF16 ||
                          c->kind == LS_KIND_SWIGLU_BF16))
        CK(cudaMallocAsync((void**)&c->splitk_ws, (size_t)gemm_split_ws_max(), a));
    CK(cudaStreamSynchronize(a));   // the new workspaces are usable on any stream
    c->ws_tokens = T;
    return LS_OK;
}

}  // namespace

// =========================================================================== C ABI
extern "C" {

void ls_params_init(ls_params* p) {
    if (!p) return;
    memset(p, 0, sizeof(*p));
    p->struct_size = sizeof(ls_params);
    p->version = LS_PARAMS_VERSION;
    p->prefetch_depth = 0;
    p->resident_layers = -1;
    p->max_vram_bytes = 0;
    p->use_pool = 0;
    p->wait_limit_ms = 30000;
    p->copy_path = LS_COPY_AUTO;
    p->copy_ctas = 0;
    p->reserve_sms = -1;
    p->device = -1;
    p->cross_run_prefetch = 0;
}

const char* ls_status_string(ls_status s) {
    switch (s) {
        case LS_OK: return "ok";
        case LS_WARN_MANDATORY_SLOT: return "warning: budget below one slot, mandatory one-slot pool used";
        case LS_WARN_SYNC_FALLBACK: return "warning: asynchronous prefetch unavailable, continued synchronously";
        case LS_ERR_INVALID_ARG: return "invalid argument";
        case LS_ERR_VERSION: return "unsupported params version or struct size";
        case LS_ERR_OOM: return "out of device memory (not even one slot)";
        case LS_ERR_HANDOFF_TIMEOUT: return "hand-off wait timed out (ready word stayed down)";
        case LS_ERR_CUDA: return "CUDA error";
        case LS_ERR_STATE: return "call out of order";
        case LS_ERR_UNSUPPORTED: return "unsupported shape, kind or alignment";
        case LS_ERR_BOUNDS: return "debug check failed (canary overwritten or invalid routing table)";
    }
    return "unknown status";
}

const char* ls_last_error(const ls_ctx* ctx) { return ctx ? ctx->err.c_str() : "null context"; }

ls_status ls_ctx_create(const ls_params* params, ls_ctx** out) {
    if (!out) return LS_ERR_INVALID_ARG;
    *out = nullptr;
    ls_params p;
    std::string why;
    ls_status st = check_params(params, &p, &why);
    if (st != LS_OK) return st;
    ls_ctx* c = new ls_ctx();
    c->prm = p;
    *out = c;
    return LS_OK;
}

static void release_resources(ls_ctx* c);

static ls_status register_impl(ls_ctx* c, const ls_segment_desc* segs, int32_t n, const ls_shared_ref* shared_map,
                               int32_t n_shared);

ls_status ls_register_segments(ls_ctx* c, const ls_segment_desc* segs, int32_t n, const ls_shared_ref* shared_map,
                               int32_t n_shared) {
    if (!c) return LS_ERR_INVALID_ARG;
    if (c->registered) {
        set_err(c, "segments are already registered");
        return LS_ERR_STATE;
    }
    ls_status st = register_impl(c, segs, n, shared_map, n_shared);
    if (st < 0) release_resources(c);  // a failed registration leaves nothing behind
    return st;
}

static ls_status register_impl(ls_ctx* c, const ls_segment_desc* segs, int32_t n, const ls_shared_ref* shared_map,
                               int32_t n_shared) {
    if (c->registered) {
        set_err(c, "segments are already registered");
        return LS_ERR_STATE;
    }
    if (!segs || n < 1 || (n_shared > 0 && !shared_map) || n_shared < 0) {
        set_err(c, "bad segment list");
        return LS_ERR_INVALID_ARG;
    }
    if (c->prm.device >= 0) CK(cudaSetDevice(c->prm.device));
    CK(cudaGetDevice(&c->device));
    c->N = n;
    c->kind = segs[0].kind;
    c->segs.assign(n, SegRec());
    std::vector<std::pair<const void*, uint64_t>> host_ranges;
    for (int s = 0; s < n; ++s) {
        if (segs[s].kind != c->kind || segs[s].n_tensors < 1 || !segs[s].tensors) {
            set_err(c, "segment %d: bad kind or tensor list", s);
            return LS_ERR_INVALID_ARG;
        }
        for (int i = 0; i < segs[s].n_tensors; ++i) {
            const ls_tensor_desc& d = segs[s].tensors[i];
            if (!d.host_ptr || d.bytes == 0 || d.ndim < 1 || d.ndim > 2) {
                set_err(c, "segment %d tensor %d: bad descriptor", s, i);
                return LS_ERR_INVALID_ARG;
            }
            TensorRec t;
            t.host = d.host_ptr;
            t.bytes = d.bytes;
            t.dtype = d.dtype;
            t.ndim = d.ndim;
            t.shape[0] = d.shape[0];
            t.shape[1] = d.ndim == 2 ? d.shape[1] : 1;
            c->segs[s].t.push_back(t);
            host_ranges.push_back({d.host_ptr, d.bytes});
        }
    }
    for (int i = 0; i < n_shared; ++i) {
        const ls_shared_ref& r = shared_map[i];
        if (r.segment < 0 || r.segment >= n || r.tensor_index < 0 ||
            r.tensor_index >= (int)c->segs[r.segment].t.size() || r.shared_id < 0) {
            set_err(c, "shared map entry %d out of range", i);
            return LS_ERR_INVALID_ARG;
        }
        c->segs[r.segment].t[r.tensor_index].shared_id = r.shared_id;
    }
    // dedup shared tensors by id (the first occurrence is the copy that is loaded)
    std::map<int, SharedRec> sh;
    for (int s = 0; s < n; ++s)
        for (auto& t : c->segs[s].t) {
            if (t.shared_id < 0) continue;
            auto it = sh.find(t.shared_id);
            if (it == sh.end()) {
                sh[t.shared_id] = SharedRec{t.shared_id, t.host, nullptr, t.bytes, 0};
            } else if (it->second.bytes != t.bytes) {
                set_err(c, "shared id %d registered with two sizes", t.shared_id);
                return LS_ERR_INVALID_ARG;
            }
        }
    int64_t off = 0;
    for (auto& kv : sh) {
        kv.second.off = off;
        off += align_up((int64_t)kv.second.bytes);
        c->shared.push_back(kv.second);
    }
    for (int s = 0; s < n; ++s) {
        int64_t o = 0, lb = 0;
        for (auto& t : c->segs[s].t) {
            if (t.shared_id >= 0) {
                t.off = sh[t.shared_id].off;
                continue;
            }
            t.off = o;
            o += align_up((int64_t)t.bytes);
            lb += (int64_t)t.bytes;
        }
        c->segs[s].slot_bytes = o;
        c->segs[s].load_bytes = lb;
        if (o == 0) {
            set_err(c, "segment %d has no private parameters", s);
            return LS_ERR_INVALID_ARG;
        }
    }
    ls_status st = validate_layout(c);
    if (st != LS_OK) return st;
    st = pin_host(c, host_ranges);
    if (st != LS_OK) return st;
    for (int s = 0; s < n; ++s)
        for (auto& t : c->segs[s].t) {
            t.dev = mapped_ptr(t.host);
            if (!t.dev) {
                set_err(c, "segment %d: host memory is not device-mapped", s);
                return LS_ERR_CUDA;
            }
        }
    for (auto& s : c->shared) s.dev = mapped_ptr(s.host);
    for (auto& s : c->segs) {
        st = build_ranges(c, s);
        if (st != LS_OK) return st;
    }
    // streams, words, events
    prepare_copy_kernels();
    CK(cudaStreamCreateWithFlags(&c->copy_stream, cudaStreamNonBlocking));
    CK(cudaEventCreateWithFlags(&c->alloc_event, cudaEventDisableTiming));
    CK(cudaEventCreateWithFlags(&c->run_done, cudaEventDisableTiming));
    CK(cudaHostAlloc((void**)&c->err_word, sizeof(uint32_t), cudaHostAllocMapped | cudaHostAllocPortable));
    *c->err_word = 0;
    CK(cudaHostGetDevicePointer((void**)&c->err_word_dev, c->err_word, 0));
    std::vector<int64_t> seg_slot(n);
    for (int s = 0; s < n; ++s) seg_slot[s] = c->segs[s].slot_bytes;
    std::vector<std::pair<int, int64_t>> shared_bytes;
    for (auto& s : c->shared) shared_bytes.push_back({s.id, (int64_t)s.bytes});
    {
        ls_params sp = c->prm;
        // a MoE segment's next loads depend on the next run's routing: no cross-run window
        if (c->kind == LS_KIND_MOE_SWIGLU_BF16) sp.cross_run_prefetch = 0;
        c->sched.configure(sp, seg_slot, shared_bytes);
    }
    GpuExec ex(c);
    ls_status plan_st = c->sched.register_memory(ex);
    if (plan_st < 0) {
        set_err(c, "could not allocate the parameter memory (not even one slot)");
        return plan_st;
    }
    // per-slot words and events for any plan a later ls_replan may choose (P <= N)
    const int P = std::max(1, n);
    CK(cudaMalloc(&c->ready, sizeof(uint32_t) * P));
    CK(cudaMalloc(&c->tickets, sizeof(uint32_t) * P));
    CK(cudaMemset(c->ready, 0, sizeof(uint32_t) * P));
    CK(cudaMemset(c->tickets, 0, sizeof(uint32_t) * P));
    c->slot_epoch.assign(P, 0);
    c->slot_free.assign(P, nullptr);
    for (int i = 0; i < P; ++i) CK(cudaEventCreateWithFlags(&c->slot_free[i], cudaEventDisableTiming));
    c->seg_buf.assign(n, nullptr);
    c->seg_epoch.assign(n, 0);
    c->seg_ptr.assign(n, nullptr);
    c->seg_slot.assign(n, 0);
    if (c->kind == LS_KIND_MOE_SWIGLU_BF16) {
        CK(cudaMalloc(&c->moe_bounds, sizeof(int) * (size_t)n * (c->E + 1)));
        CK(cudaMalloc(&c->moe_used, (size_t)n * c->E));
        CK(cudaHostAlloc((void**)&c->moe_used_host, (size_t)n * c->E, cudaHostAllocMapped));
        CK(cudaHostGetDevicePointer((void**)&c->moe_used_host_dev, c->moe_used_host, 0));
        memset(c->moe_used_host, 1, (size_t)n * c->E);
        if (c->prm.expert_cache_bytes > 0) {
            c->ecache_eb = c->segs[0].slot_bytes / c->E;
            const int64_t k = std::min<int64_t>(c->prm.expert_cache_bytes / c->ecache_eb, (int64_t)n * c->E);
            if (k > 0) {
                c->ecache = dev_alloc(c, (size_t)(k * c->ecache_eb), c->copy_stream);
                if (!c->ecache) {
                    set_err(c, "could not allocate the expert cache (%lld bytes)", (long long)(k * c->ecache_eb));
                    return LS_ERR_OOM;
                }
                c->ecache_K = (int)k;
                c->ecache_counts.assign((size_t)n * c->E, 0);
                c->ecache_slot.assign((size_t)n * c->E, -1);
                c->ecache_filled.assign((size_t)n * c->E, 0);
                c->ecache_hits.assign(n, {});
                c->ecache_fills.assign(n, {});
                const size_t rb = sizeof(int) * (size_t)n * 2 * c->E;
                CK(cudaHostAlloc((void**)&c->ecache_rows_host, rb, cudaHostAllocDefault));
                CK(cudaMalloc(&c->ecache_rows_dev, rb));
            }
        }
    }
    const int sms = gemm_num_sms();
    c->copy_ctas = c->prm.copy_ctas > 0 ? c->prm.copy_ctas : sms;
    c->reserve_sms = c->prm.reserve_sms >= 0 ? c->prm.reserve_sms : 0;
    CK(cudaStreamSynchronize(c->copy_stream));
    st = autotune_copy(c);
    if (st != LS_OK) return st;
    if (c->prm.debug_checks && c->prm.test_corrupt_canary > 0 && c->pool &&
        c->prm.test_corrupt_canary <= c->pool_slots) {  // test hook: an overrun past one slot, made by the host
        uint8_t* cn = (uint8_t*)c->pool + (int64_t)(c->prm.test_corrupt_canary - 1) * c->slot_stride + c->sched.plan().S;
        CK(cudaMemset(cn, 0, 8));
    }
    if (c->cuda_err != cudaSuccess) {
        set_err(c, "registration: %s", cudaGetErrorString(c->cuda_err));
        return LS_ERR_CUDA;
    }
    c->registered = true;
    return plan_st;
}

// params.debug_checks: compare the canaries of every pool slot and of the shared region, in
// stream order after the pass's last kernel (copies in flight write inside their slots).
static void check_canaries(ls_ctx* c, cudaStream_t s) {
    if (c->pool && c->pool_slots > 0)
        track(c, launch_canary((uint8_t*)c->pool + c->sched.plan().S, c->slot_stride, c->pool_slots, true,
                               c->err_word_dev, 0, s));
    if (c->shared_dev)
        track(c, launch_canary((uint8_t*)c->shared_dev + c->shared_bytes_dev, 0, 1, true, c->err_word_dev,
                               CANARY_REGION_SHARED, s));
}

static void destroy_graph(ls_ctx* c) {
    if (c->graph_exec) cudaGraphExecDestroy(c->graph_exec);
    if (c->graph) cudaGraphDestroy(c->graph);
    c->graph_exec = nullptr;
    c->graph = nullptr;
    c->graph_events.clear();
    cudaGetLastError();
}

// The expert cache's decisions for the pass whose routing moe_used_host holds: the hot set
// is the K pairs of streamed layers routed in the most earlier passes (ties to the lower
// expert, then layer, so that equal counts spread the cache over the layers); leaving
// pairs give back their slot, entering ones take the lowest free slots in rank order; a
// routed hot pair is a hit once filled, else it is filled from this pass's host copy. Hits
// are then cleared from moe_used_host, which becomes the set of experts to copy from the
// host, and the row tables tell the GEMMs where each expert's matrices are.
static void ecache_plan_pass(ls_ctx* c) {
    const int N = c->N, E = c->E, R = c->sched.residents();
    // B rows per expert blob in the gate/up view (rows of H elements) and the down view
    // (rows of F elements); the down matrix starts 2F x H elements into the blob
    const int up_rows = (int)(c->ecache_eb / (2 * (int64_t)c->H));
    const int dn_rows = (int)(c->ecache_eb / (2 * (int64_t)c->F)), dn_base = 2 * c->H;
    std::vector<std::tuple<int64_t, int, int>> cand;
    for (int l = R; l < N; ++l)
        for (int e = 0; e < E; ++e)
            if (c->ecache_counts[(size_t)l * E + e] > 0) cand.emplace_back(-c->ecache_counts[(size_t)l * E + e], e, l);
    std::sort(cand.begin(), cand.end());
    if ((int)cand.size() > c->ecache_K) cand.resize(c->ecache_K);
    std::vector<char> hot((size_t)N * E, 0);
    for (auto& t : cand) hot[(size_t)std::get<2>(t) * E + std::get<1>(t)] = 1;
    std::vector<int> free_slots;
    std::vector<char> taken(c->ecache_K, 0);
    for (size_t i = 0; i < hot.size(); ++i) {
        if (c->ecache_slot[i] >= 0 && !hot[i]) {
            c->ecache_slot[i] = -1;
            c->ecache_filled[i] = 0;
        }
        if (c->ecache_slot[i] >= 0) taken[c->ecache_slot[i]] = 1;
    }
    for (int k = c->ecache_K - 1; k >= 0; --k)
        if (!taken[k]) free_slots.push_back(k);  // popped from the back: lowest first
    for (int l = 0; l < N; ++l) {
        c->ecache_hits[l].clear();
        c->ecache_fills[l].clear();
    }
    for (auto& t : cand) {
        const int e = std::get<1>(t), l = std::get<2>(t);
        const size_t i = (size_t)l * E + e;
        if (c->ecache_slot[i] < 0) {
            c->ecache_slot[i] = free_slots.back();
            free_slots.pop_back();
        }
    }
    for (int l = R; l < N; ++l)
        for (int e = 0; e < E; ++e) c->ecache_counts[(size_t)l * E + e] += c->moe_used_host[(size_t)l * E + e];
    for (int l = R; l < N; ++l)
        for (int e = 0; e < E; ++e) {
            const size_t i = (size_t)l * E + e;
            if (!c->moe_used_host[i]) continue;
            if (hot[i] && c->ecache_filled[i]) {
                c->ecache_hits[l].push_back({e, c->ecache_slot[i]});
                c->moe_used_host[i] = 0;  // nothing to move: the GEMMs read it in the cache
                ++c->n_ecache_hits;
            } else {
                if (hot[i]) {
                    c->ecache_fills[l].push_back({e, c->ecache_slot[i]});
                    c->ecache_filled[i] = 1;
                }
                ++c->n_ecache_host;
            }
        }
    for (int l = R; l < N; ++l) {
        int* up = c->ecache_rows_host + (size_t)l * 2 * E;
        int* dn = up + E;
        for (int e = 0; e < E; ++e) {
            up[e] = e * up_rows;
            dn[e] = dn_base + e * dn_rows;
        }
        for (auto& h : c->ecache_hits[l]) {
            up[h.first] = (int)(0x80000000u | (uint32_t)(h.second * up_rows));
            dn[h.first] = (int)(0x80000000u | (uint32_t)(dn_base + h.second * dn_rows));
        }
    }
}

// Checks, workspaces and (MoE) routing of one pass on the caller's stream; fills the
// bytes each load will move. The pass itself is issued by the caller of this.
static ls_status prepare_pass(ls_ctx* c, const void* x_dev, void* y_dev, int64_t tokens, cudaStream_t s,
                              const ls_moe_routing* routing, std::vector<int64_t>& load_bytes) {
    if (!c->registered) {
        set_err(c, "ls_run before ls_register_segments");
        return LS_ERR_STATE;
    }
    if (!x_dev || !y_dev || tokens < 1 || tokens > (1 << 24) || x_dev == y_dev) {
        set_err(c, "bad run arguments");
        return LS_ERR_INVALID_ARG;
    }
    const bool moe = c->kind == LS_KIND_MOE_SWIGLU_BF16;
    if (moe && (!routing || !routing->logits || routing->top_k < 1 || routing->top_k > 8 ||
                routing->top_k > c->E)) {
        set_err(c, "the MoE kind needs routing logits and 1 <= top_k <= min(8, experts)");
        return LS_ERR_INVALID_ARG;
    }
    if ((int64_t)tokens * (moe ? routing->top_k : 1) > (int64_t)INT32_MAX / 4) {
        set_err(c, "too many tokens");
        return LS_ERR_INVALID_ARG;
    }
    CK(cudaSetDevice(c->device));
    if (tokens > c->ws_tokens) {
        ls_status sy = ls_sync(c);  // workspaces are about to be replaced
        if (sy < 0) return sy;
        destroy_graph(c);           // a captured pass points at the old ones
    }
    ls_status st = ensure_workspace(c, tokens);
    if (st != LS_OK) return st;
    if (std::find(c->pending.begin(), c->pending.end(), s) == c->pending.end()) c->pending.push_back(s);
    CK(cudaStreamWaitEvent(s, c->run_done, 0));  // passes share workspaces: keep them in order
    load_bytes.assign(c->N, 0);
    for (int i = 0; i < c->N; ++i) load_bytes[i] = c->segs[i].load_bytes;
    if (moe) {
        c->top_k = routing->top_k;
        const int E = c->E, k = c->top_k;
        {
            KTime kt(c, "moe_route_group", s);
            CK(launch_moe_route(routing->logits, c->N, (int)tokens, E, k, c->moe_sel, c->moe_w, s));
            CK(launch_moe_group(c->moe_sel, c->N, (int)tokens, E, k, c->moe_table, c->moe_bounds, c->moe_used, s));
        }
        if (c->prm.debug_checks)
            CK(launch_moe_check(c->moe_sel, c->moe_table, c->moe_bounds, c->N, (int)tokens, k, E, c->err_word_dev,
                                CHECK_REGION_MOE, s));
        CK(cudaMemcpyAsync(c->moe_used_host, c->moe_used, (size_t)c->N * E, cudaMemcpyDeviceToHost, s));
        CK(cudaStreamSynchronize(s));
        if (c->ecache_K > 0) {
            ecache_plan_pass(c);
            // the host table is rewritten only after the next pass's routing synchronisation,
            // which this copy precedes on the same stream
            CK(cudaMemcpyAsync(c->ecache_rows_dev, c->ecache_rows_host, sizeof(int) * (size_t)c->N * 2 * E,
                               cudaMemcpyHostToDevice, s));
        }
        const int64_t eb = c->segs[0].slot_bytes / E;
        const int R = c->sched.residents();  // residents are loaded whole (see GpuExec::load)
        for (int l = R; l < c->N; ++l) {
            int64_t used = 0;
            for (int e = 0; e < E; ++e) used += c->moe_used_host[(int64_t)l * E + e];
            load_bytes[l] = used * eb;
        }
    }
    return LS_OK;
}

ls_status ls_run_async(ls_ctx* c, const void* x_dev, void* y_dev, int64_t tokens, void* stream,
                       const ls_moe_routing* routing) {
    if (!c) return LS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    std::vector<int64_t> load_bytes;
    ls_status pst = prepare_pass(c, x_dev, y_dev, tokens, s, routing, load_bytes);
    if (pst != LS_OK) return pst;
    GpuExec ex(c);
    ex.rc = RunCtx{x_dev, y_dev, tokens, s, (uint64_t)c->prm.wait_limit_ms * 1000000ull};
    ls_status rs = c->sched.run(ex, load_bytes.data());
    if (c->prm.debug_checks) check_canaries(c, s);
    track(c, cudaEventRecord(c->run_done, s));
    if (rs < 0) set_err(c, "run %d: %s", c->sched.runs() - 1, ls_status_string(rs));
    return rs;
}

static bool same_events(const std::vector<ls_sched_event>& a, const std::vector<ls_sched_event>& b) {
    if (a.size() != b.size()) return false;
    for (size_t i = 0; i < a.size(); ++i)
        if (a[i].step != b[i].step || a[i].kind != b[i].kind || a[i].segment != b[i].segment ||
            a[i].slot != b[i].slot || a[i].bytes != b[i].bytes)
            return false;
    return true;
}

ls_status ls_run_graph(ls_ctx* c, const void* x_dev, void* y_dev, int64_t tokens, void* stream) {
    if (!c) return LS_ERR_INVALID_ARG;
    if (c->registered && (c->kind == LS_KIND_MOE_SWIGLU_BF16 || !c->prm.use_pool || c->prm.cross_run_prefetch)) {
        set_err(c, "ls_run_graph needs the pool, no cross-run window and a kind without per-pass routing");
        return LS_ERR_UNSUPPORTED;
    }
    cudaStream_t s = (cudaStream_t)stream;
    std::vector<int64_t> lb;
    ls_status pst = prepare_pass(c, x_dev, y_dev, tokens, s, nullptr, lb);
    if (pst != LS_OK) return pst;
    // the schedule this pass will follow, from a copy of the scheduler
    Scheduler probe = c->sched.without_log();
    DryExec dex;
    const ls_status prs = probe.run(dex, lb.data());
    std::vector<ls_sched_event> ev(probe.log().begin(), probe.log().end());
    bool steady = prs == LS_OK;
    for (auto& e : ev) {
        e.run = 0;
        steady = steady && (e.kind == LS_EV_PREFETCH || e.kind == LS_EV_LOAD_SYNC || e.kind == LS_EV_ACTIVATE);
    }
    if (!steady) {  // shared or resident loads, evictions, a fallback: an ordinary pass
        GpuExec ex(c);
        ex.rc = RunCtx{x_dev, y_dev, tokens, s, (uint64_t)c->prm.wait_limit_ms * 1000000ull};
        ls_status rs = c->sched.run(ex, lb.data());
        track(c, cudaEventRecord(c->run_done, s));
        if (rs < 0) set_err(c, "run %d: %s", c->sched.runs() - 1, ls_status_string(rs));
        return rs;
    }
    if (!c->graph_stream) {
        CK(cudaStreamCreateWithFlags(&c->graph_stream, cudaStreamNonBlocking));
        for (cudaEvent_t* e : {&c->graph_in, &c->graph_out, &c->graph_fork, &c->graph_join})
            CK(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
    }
    if (std::find(c->pending.begin(), c->pending.end(), c->graph_stream) == c->pending.end())
        c->pending.push_back(c->graph_stream);
    CK(cudaEventRecord(c->graph_in, s));
    CK(cudaStreamWaitEvent(c->graph_stream, c->graph_in, 0));
    const bool reuse = c->graph_exec && c->graph_x == x_dev && c->graph_y == y_dev && c->graph_T == tokens &&
                       same_events(ev, c->graph_events);
    if (reuse) {
        c->sched.run(dex, lb.data());  // the log and counters advance as for an issued pass
        ++c->graph_replays;
    } else {
        destroy_graph(c);
        // what a capture advances without running anything: restored if it has to be redone
        const Scheduler saved_sched = c->sched;
        const auto saved_slot_epoch = c->slot_epoch;
        const auto saved_seg_epoch = c->seg_epoch;
        const auto saved_seg_ptr = c->seg_ptr;
        const auto saved_seg_slot = c->seg_slot;
        const auto saved_publishes = c->publishes;
        const int saved_timing = c->prm.kernel_timing;
        cudaError_t e = cudaSuccess;
        ls_status rs = LS_OK;
        for (int attempt = 0; attempt < 2; ++attempt) {
            c->prm.kernel_timing = 0;
            c->capturing = true;
            cudaStream_t gs = c->graph_stream;
            rs = LS_OK;
            e = cudaStreamBeginCapture(gs, cudaStreamCaptureModeThreadLocal);
            if (e == cudaSuccess) {
                // ready words restart at every replay: the pass's epochs are fixed in the graph
                track(c, cudaMemsetAsync(c->ready, 0, sizeof(uint32_t) * std::max(1, c->N), gs));
                track(c, cudaEventRecord(c->graph_fork, gs));
                track(c, cudaStreamWaitEvent(c->copy_stream, c->graph_fork, 0));  // the copy stream joins
                for (cudaEvent_t f : c->slot_free) track(c, cudaEventRecord(f, gs));
                GpuExec ex(c);
                ex.rc = RunCtx{x_dev, y_dev, tokens, gs, (uint64_t)c->prm.wait_limit_ms * 1000000ull};
                rs = c->sched.run(ex, lb.data());
                track(c, cudaEventRecord(c->graph_join, c->copy_stream));
                track(c, cudaStreamWaitEvent(gs, c->graph_join, 0));
                cudaGraph_t g = nullptr;
                e = cudaStreamEndCapture(gs, &g);
                c->graph = g;
            }
            c->capturing = false;
            c->prm.kernel_timing = saved_timing;
            if (e == cudaSuccess && c->cuda_err == cudaSuccess)
                e = cudaGraphInstantiate(&c->graph_exec, c->graph, 0);
            if (e == cudaSuccess && c->cuda_err == cudaSuccess && rs == LS_OK) break;
            // failed: nothing ran; put the bookkeeping back as before the capture
            if (e == cudaSuccess) e = c->cuda_err;
            c->cuda_err = cudaSuccess;
            cudaGetLastError();
            destroy_graph(c);
            c->sched = saved_sched;
            c->slot_epoch = saved_slot_epoch;
            c->seg_epoch = saved_seg_epoch;
            c->seg_ptr = saved_seg_ptr;
            c->seg_slot = saved_seg_slot;
            c->publishes = saved_publishes;
            if (attempt == 0 && c->capture_stream_ops) {
                c->capture_stream_ops = false;  // the driver refused the memory operation in a graph
                continue;
            }
            set_err(c, "run %d: graph capture failed: %s", c->sched.runs(), cudaGetErrorString(e));
            return LS_ERR_CUDA;
        }
        c->graph_x = x_dev;
        c->graph_y = y_dev;
        c->graph_T = tokens;
        c->graph_events = ev;
        ++c->graph_captures;
    }
    CK(cudaGraphLaunch(c->graph_exec, c->graph_stream));
    CK(cudaEventRecord(c->graph_out, c->graph_stream));
    CK(cudaStreamWaitEvent(s, c->graph_out, 0));
    // slot events were last recorded inside the capture: record them again in plain stream order
    for (cudaEvent_t f : c->slot_free) track(c, cudaEventRecord(f, s));
    track(c, cudaEventRecord(c->run_done, s));
    return LS_OK;
}

ls_status ls_sync(ls_ctx* c) {
    if (!c) return LS_ERR_INVALID_ARG;
    if (!c->registered) return LS_OK;
    CK(cudaSetDevice(c->device));
    cudaError_t e = cudaSuccess;
    for (cudaStream_t s : c->pending) {
        cudaError_t e1 = cudaStreamSynchronize(s);
        if (e == cudaSuccess) e = e1;
    }
    cudaError_t e2 = cudaStreamSynchronize(c->copy_stream);
    if (e == cudaSuccess) e = e2;
    c->pending.clear();
    if (c->prm.kernel_timing) collect_times(c);
    if (e == cudaSuccess) e = c->cuda_err;
    c->cuda_err = cudaSuccess;
    const uint32_t ew = *(volatile uint32_t*)c->err_word;
    *(volatile uint32_t*)c->err_word = 0;
    if (e != cudaSuccess) {
        set_err(c, "run %d: %s", c->sched.runs() - 1, cudaGetErrorString(e));
        return LS_ERR_CUDA;
    }
    if (ew != 0) {
        if ((ew & 0xff) == DERR_HANDOFF_TIMEOUT) {
            set_err(c, "run %d: the ready word of slot %u stayed down for %d ms", c->sched.runs() - 1, ew >> 8,
                    c->prm.wait_limit_ms);
            return LS_ERR_HANDOFF_TIMEOUT;
        }
        if ((ew & 0xff) == DERR_BOUNDS) {
            ++c->debug_violations;
            const uint32_t r = ew >> 8;
            if (r >= CHECK_REGION_MOE)
                set_err(c, "run %d: debug check failed: MoE row table or group bounds of layer %u are invalid",
                        c->sched.runs() - 1, r - CHECK_REGION_MOE);
            else if (r >= CANARY_REGION_SEGMENT)
                set_err(c, "run %d: debug check failed: canary after the buffer of segment %u overwritten",
                        c->sched.runs() - 1, r - CANARY_REGION_SEGMENT);
            else if (r == CANARY_REGION_SHARED)
                set_err(c, "run %d: debug check failed: canary after the shared region overwritten", c->sched.runs() - 1);
            else
                set_err(c, "run %d: debug check failed: canary after pool slot %u overwritten", c->sched.runs() - 1, r);
            return LS_ERR_BOUNDS;
        }
        set_err(c, "run %d: device error word 0x%x", c->sched.runs() - 1, ew);
        return LS_ERR_CUDA;
    }
    return LS_OK;
}

ls_status ls_replan(ls_ctx* c, int32_t prefetch_depth, int32_t resident_layers, int64_t max_vram_bytes) {
    if (!c) return LS_ERR_INVALID_ARG;
    if (!c->registered) {
        set_err(c, "ls_replan before ls_register_segments");
        return LS_ERR_STATE;
    }
    if (!c->pending.empty()) {
        set_err(c, "ls_replan: passes are queued; call ls_sync first");
        return LS_ERR_STATE;
    }
    if (prefetch_depth < 0 || resident_layers < -1 || max_vram_bytes < 0) {
        set_err(c, "ls_replan: depth and budget must be >= 0, resident_layers >= -1");
        return LS_ERR_INVALID_ARG;
    }
    CK(cudaSetDevice(c->device));
    // queued copies (a cross-run prefetch) land before their slots change hands
    CK(cudaStreamSynchronize(c->copy_stream));
    GpuExec ex(c);
    ex.rc = RunCtx{nullptr, nullptr, 0, c->copy_stream, 0};
    destroy_graph(c);
    const ls_status st = c->sched.replan(ex, prefetch_depth, resident_layers, max_vram_bytes);
    CK(cudaStreamSynchronize(c->copy_stream));  // releases and the new pool are in place
    if (c->cuda_err != cudaSuccess) {
        set_err(c, "ls_replan: %s", cudaGetErrorString(c->cuda_err));
        c->cuda_err = cudaSuccess;
        return LS_ERR_CUDA;
    }
    c->prm.prefetch_depth = prefetch_depth;
    c->prm.resident_layers = resident_layers;
    c->prm.max_vram_bytes = max_vram_bytes;
    if (st == LS_ERR_OOM) set_err(c, "ls_replan: not even a one-slot pool could be allocated; the context cannot run");
    return st;
}

ls_status ls_run(ls_ctx* c, const void* x_dev, void* y_dev, int64_t tokens, void* stream,
                 const ls_moe_routing* routing) {
    ls_status st = ls_run_async(c, x_dev, y_dev, tokens, stream, routing);
    ls_status sy = c ? ls_sync(c) : LS_ERR_INVALID_ARG;
    if (st < 0) return st;
    if (sy < 0) return sy;
    return st;
}

// ls_run_host (sync) and ls_run_host_async (!sync): the inputs' copies, the pass and the
// output's copy, queued in that order on the context's own stream
static ls_status run_host(ls_ctx* c, const void* x_host, void* y_host, int64_t tokens,
                          const ls_moe_routing* routing_host, bool sync) {
    if (!c) return LS_ERR_INVALID_ARG;
    if (!c->registered) {
        set_err(c, "ls_run_host before ls_register_segments");
        return LS_ERR_STATE;
    }
    if (!x_host || !y_host || tokens < 1) {
        set_err(c, "bad run arguments");
        return LS_ERR_INVALID_ARG;
    }
    const bool moe = c->kind == LS_KIND_MOE_SWIGLU_BF16;
    if (moe && (!routing_host || !routing_host->logits)) {
        set_err(c, "the MoE kind needs routing logits");
        return LS_ERR_INVALID_ARG;
    }
    CK(cudaSetDevice(c->device));
    if (!c->own_stream) CK(cudaStreamCreateWithFlags(&c->own_stream, cudaStreamNonBlocking));
    const size_t es = c->kind == LS_KIND_LINEAR_GELU_F32 ? 4 : 2;
    const size_t xb = (size_t)tokens * c->H * es;
    if (tokens > c->stage_tokens) {
        ls_status sy = ls_sync(c);
        if (sy < 0) return sy;
        if (c->stage_x) cudaFree(c->stage_x);
        if (c->stage_y) cudaFree(c->stage_y);
        if (c->stage_logits) cudaFree(c->stage_logits);
        c->stage_x = c->stage_y = nullptr;
        c->stage_logits = nullptr;
        CK(cudaMalloc(&c->stage_x, xb));
        CK(cudaMalloc(&c->stage_y, xb));
        if (moe) CK(cudaMalloc((void**)&c->stage_logits, (size_t)c->N * tokens * c->E * sizeof(float)));
        c->stage_tokens = tokens;
    }
    CK(cudaMemcpyAsync(c->stage_x, x_host, xb, cudaMemcpyHostToDevice, c->own_stream));
    ls_moe_routing r{};
    if (moe) {
        CK(cudaMemcpyAsync(c->stage_logits, routing_host->logits, (size_t)c->N * tokens * c->E * sizeof(float),
                           cudaMemcpyHostToDevice, c->own_stream));
        r.logits = c->stage_logits;
        r.top_k = routing_host->top_k;
    }
    // the pass, then the copy back in the same stream, then a single synchronisation
    ls_status st = ls_run_async(c, c->stage_x, c->stage_y, tokens, c->own_stream, moe ? &r : nullptr);
    if (st < 0) {
        ls_sync(c);
        return st;
    }
    CK(cudaMemcpyAsync(y_host, c->stage_y, xb, cudaMemcpyDeviceToHost, c->own_stream));
    if (!sync) return st;
    const ls_status sy = ls_sync(c);
    if (sy < 0) return sy;
    return st;
}

ls_status ls_run_host(ls_ctx* c, const void* x_host, void* y_host, int64_t tokens, const ls_moe_routing* routing_host) {
    return run_host(c, x_host, y_host, tokens, routing_host, true);
}

ls_status ls_run_host_async(ls_ctx* c, const void* x_host, void* y_host, int64_t tokens,
                            const ls_moe_routing* routing_host) {
    return run_host(c, x_host, y_host, tokens, routing_host, false);
}

ls_status ls_get_schedule(ls_ctx* c, ls_sched_event* out, int64_t cap, int64_t* n_out) {
    if (!c || !n_out || cap < 0 || (cap > 0 && !out)) return LS_ERR_INVALID_ARG;
    const auto& log = c->sched.log();
    *n_out = (int64_t)log.size();
    const int64_t n = std::min<int64_t>(cap, (int64_t)log.size());
    if (n > 0) memcpy(out, log.data(), sizeof(ls_sched_event) * n);
    return LS_OK;
}

ls_status ls_get_stats(ls_ctx* c, ls_stats* out) {
    if (!c || !out || out->struct_size < offsetof(ls_stats, slot_bytes)) return LS_ERR_INVALID_ARG;
    ls_stats s;
    memset(&s, 0, sizeof(s));
    s.struct_size = sizeof(s);
    if (c->registered || c->sched.plan().N > 0) c->sched.fill_stats(s);
    s.copy_path = c->copy_path;
    s.kernel_copy_segments = c->kernel_copy_segments;
    s.copy_kernel_gbs = c->gbs_kernel;
    s.copy_engine_gbs = c->gbs_engine;
    s.graph_captures = c->graph_captures;
    s.graph_replays = c->graph_replays;
    s.expert_cache_hits = c->n_ecache_hits;
    s.expert_host_loads = c->n_ecache_host;
    s.debug_violations = c->debug_violations;
    const uint32_t n = std::min<uint32_t>(out->struct_size, sizeof(s));
    memcpy(out, &s, n);
    out->struct_size = n;
    return LS_OK;
}

ls_status ls_get_trace(ls_ctx* c, ls_trace_event* out, int64_t cap, int64_t* n_out) {
    if (!c || !n_out || cap < 0 || (cap > 0 && !out)) return LS_ERR_INVALID_ARG;
    *n_out = (int64_t)c->trace.size();
    const int64_t n = std::min<int64_t>(cap, (int64_t)c->trace.size());
    if (n > 0) memcpy(out, c->trace.data(), sizeof(ls_trace_event) * n);
    return LS_OK;
}

ls_status ls_set_kernel_timing(ls_ctx* c, int32_t mode) {
    if (!c || mode < 0 || mode > 3) return LS_ERR_INVALID_ARG;
    if (!c->pending.empty()) {
        set_err(c, "ls_set_kernel_timing: passes are queued; call ls_sync first");
        return LS_ERR_STATE;
    }
    c->prm.kernel_timing = mode;
    return LS_OK;
}

ls_status ls_get_kernel_times(ls_ctx* c, ls_kernel_time* out, int32_t cap, int32_t* n_out, int32_t reset) {
    if (!c || !n_out || cap < 0 || (cap > 0 && !out)) return LS_ERR_INVALID_ARG;
    *n_out = (int32_t)c->tclass.size();
    for (int32_t i = 0; i < cap && i < (int32_t)c->tclass.size(); ++i) {
        memset(&out[i], 0, sizeof(out[i]));
        snprintf(out[i].name, sizeof(out[i].name), "%s", c->tclass[i].name.c_str());
        out[i].launches = c->tclass[i].launches;
        out[i].total_ms = c->tclass[i].total_ms;
    }
    if (reset)
        for (auto& t : c->tclass) {
            t.launches = 0;
            t.total_ms = 0;
        }
    return LS_OK;
}

static void release_resources(ls_ctx* c) {
    if (c->N > 0) {
        cudaSetDevice(c->device);
        sync_ctx_streams(c);
        free_workspaces(c);
        if (c->splitk_ws) cudaFreeAsync(c->splitk_ws, c->copy_stream);
        for (int s = 0; s < (int)c->seg_buf.size(); ++s)
            if (c->seg_buf[s])
                dev_free(c, c->seg_buf[s], (size_t)(c->segs[s].slot_bytes + (c->prm.debug_checks ? CANARY_BYTES : 0)),
                         c->copy_stream);
        if (c->pool) dev_free(c, c->pool, (size_t)c->pool_bytes, c->copy_stream);
        if (c->shared_dev) dev_free(c, c->shared_dev, 0, c->copy_stream);
        if (c->ecache) dev_free(c, c->ecache, (size_t)(c->ecache_K * c->ecache_eb), c->copy_stream);
        if (c->copy_stream) cudaStreamSynchronize(c->copy_stream);
        for (auto& sr : c->segs)
            if (sr.ranges_dev) cudaFree(sr.ranges_dev);
        for (void* p : {(void*)c->ready, (void*)c->tickets, (void*)c->moe_bounds, (void*)c->moe_used, c->stage_x,
                        c->stage_y, (void*)c->stage_logits})
            if (p) cudaFree(p);
        if (c->moe_used_host) cudaFreeHost(c->moe_used_host);
        if (c->ecache_rows_host) cudaFreeHost(c->ecache_rows_host);
        if (c->ecache_rows_dev) cudaFree(c->ecache_rows_dev);
        if (c->err_word) cudaFreeHost(c->err_word);
        for (auto e : c->slot_free)
            if (e) cudaEventDestroy(e);
        for (auto& e : c->tev) {
            cudaEventDestroy(e.first);
            cudaEventDestroy(e.second);
        }
        if (c->alloc_event) cudaEventDestroy(c->alloc_event);
        if (c->run_done) cudaEventDestroy(c->run_done);
        if (c->copy_stream) cudaStreamDestroy(c->copy_stream);
        if (c->own_stream) cudaStreamDestroy(c->own_stream);
        destroy_graph(c);
        for (cudaEvent_t e : {c->graph_in, c->graph_out, c->graph_fork, c->graph_join})
            if (e) cudaEventDestroy(e);
        if (c->graph_stream) cudaStreamDestroy(c->graph_stream);
        for (auto& r : c->host_registered) cudaHostUnregister(r.first);
        cudaGetLastError();
    }
    // back to an empty, unregistered context
    ls_params prm = c->prm;
    std::string err = c->err;
    c->~ls_ctx();
    new (c) ls_ctx();
    c->prm = prm;
    c->err = err;
}

void ls_ctx_destroy(ls_ctx* c) {
    if (!c) return;
    release_resources(c);
    delete c;
}

static void copy_out(const Scheduler& sched, bool planned, ls_sched_event* events, int64_t cap, int64_t* n_events,
                     ls_stats* stats, ls_status* bad) {
    const auto& log = sched.log();
    *n_events = (int64_t)log.size();
    const int64_t m = std::min<int64_t>(cap, (int64_t)log.size());
    if (m > 0) memcpy(events, log.data(), sizeof(ls_sched_event) * m);
    if (stats) {
        if (stats->struct_size < offsetof(ls_stats, slot_bytes)) {
            *bad = LS_ERR_INVALID_ARG;
            return;
        }
        ls_stats s;
        memset(&s, 0, sizeof(s));
        if (planned) sched.fill_stats(s);
        s.copy_path = LS_COPY_AUTO;
        const uint32_t sz = std::min<uint32_t>(stats->struct_size, sizeof(s));
        memcpy(stats, &s, sz);
        stats->struct_size = sz;
    }
}

ls_status ls_simulate_script(const ls_params* params, const int64_t* seg_slot_bytes, int32_t n,
                             const int64_t* shared_bytes, const int32_t* shared_ids, int32_t n_shared,
                             const int64_t* script, int32_t n_steps, ls_sched_event* events, int64_t cap,
                             int64_t* n_events, ls_stats* stats, ls_status* step_status) {
    ls_params p;
    std::string why;
    ls_status st = check_params(params, &p, &why);
    if (st != LS_OK) return st;
    if (!seg_slot_bytes || n < 1 || n_steps < 0 || (n_steps > 0 && !script) ||
        (n_shared > 0 && (!shared_bytes || !shared_ids)) || !n_events || (cap > 0 && !events))
        return LS_ERR_INVALID_ARG;
    std::vector<int64_t> seg(seg_slot_bytes, seg_slot_bytes + n);
    for (int64_t b : seg)
        if (b <= 0) return LS_ERR_INVALID_ARG;
    std::vector<std::pair<int, int64_t>> sh;
    for (int i = 0; i < n_shared; ++i) sh.push_back({shared_ids[i], shared_bytes[i]});
    Scheduler sched;
    sched.configure(p, seg, sh);
    DryExec ex;
    ls_status reg = sched.register_memory(ex);
    if (reg >= 0) {
        for (int i = 0; i < n_steps; ++i) {
            const int64_t* op = script + 4 * (int64_t)i;
            ls_status rs;
            if (op[0] == 0)
                rs = sched.run(ex, nullptr);
            else if (op[0] == 1 && op[1] >= 0 && op[2] >= -1 && op[3] >= 0)
                rs = sched.replan(ex, (int)op[1], (int)op[2], op[3]);
            else
                rs = LS_ERR_INVALID_ARG;
            if (step_status) step_status[i] = rs;
            if (rs < 0) break;
        }
    }
    ls_status bad = LS_OK;
    copy_out(sched, reg >= 0 && sched.usable(), events, cap, n_events, stats, &bad);
    return bad != LS_OK ? bad : reg;
}

ls_status ls_simulate(const ls_params* params, const int64_t* seg_slot_bytes, int32_t n, const int64_t* shared_bytes,
                      const int32_t* shared_ids, int32_t n_shared, int32_t runs, const int64_t* load_bytes,
                      ls_sched_event* events, int64_t cap, int64_t* n_events, ls_stats* stats,
                      ls_status* run_status) {
    ls_params p;
    std::string why;
    ls_status st = check_params(params, &p, &why);
    if (st != LS_OK) return st;
    if (!seg_slot_bytes || n < 1 || runs < 0 || (n_shared > 0 && (!shared_bytes || !shared_ids)) || !n_events ||
        (cap > 0 && !events))
        return LS_ERR_INVALID_ARG;
    std::vector<int64_t> seg(seg_slot_bytes, seg_slot_bytes + n);
    for (int64_t b : seg)
        if (b <= 0) return LS_ERR_INVALID_ARG;
    std::vector<std::pair<int, int64_t>> sh;
    for (int i = 0; i < n_shared; ++i) sh.push_back({shared_ids[i], shared_bytes[i]});
    Scheduler sched;
    sched.configure(p, seg, sh);
    DryExec ex;
    ls_status reg = sched.register_memory(ex);
    if (reg >= 0) {
        for (int r = 0; r < runs; ++r) {
            ls_status rs = sched.run(ex, load_bytes ? load_bytes + (int64_t)r * n : nullptr);
            if (run_status) run_status[r] = rs;
        }
    }
    const auto& log = sched.log();
    *n_events = (int64_t)log.size();
    const int64_t m = std::min<int64_t>(cap, (int64_t)log.size());
    if (m > 0) memcpy(events, log.data(), sizeof(ls_sched_event) * m);
    if (stats) {
        if (stats->struct_size < offsetof(ls_stats, slot_bytes)) return LS_ERR_INVALID_ARG;
        ls_stats s;
        memset(&s, 0, sizeof(s));
        if (reg >= 0) sched.fill_stats(s);
        s.copy_path = LS_COPY_AUTO;
        const uint32_t sz = std::min<uint32_t>(stats->struct_size, sizeof(s));
        memcpy(stats, &s, sz);
        stats->struct_size = sz;
    }
    return reg;
}

}  // extern "C"
