// Standalone C entry points of the device kernels (see ls_kernels.h).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ls_kernels.h"

using namespace ls;

namespace {

uint32_t* g_err_host = nullptr;
uint32_t* g_err_dev = nullptr;
std::mutex g_err_mu;

uint32_t* err_dev() {
    std::lock_guard<std::mutex> g(g_err_mu);
    if (!g_err_host) {
        if (cudaHostAlloc((void**)&g_err_host, sizeof(uint32_t), cudaHostAllocMapped | cudaHostAllocPortable) !=
            cudaSuccess) {
            cudaGetLastError();
            g_err_host = nullptr;
            return nullptr;
        }
        *g_err_host = 0;
        cudaHostGetDevicePointer((void**)&g_err_dev, g_err_host, 0);
    }
    return g_err_dev;
}

inline ls_status st(cudaError_t e) {
    if (e == cudaSuccess) return LS_OK;
    if (e == cudaErrorInvalidValue) return LS_ERR_INVALID_ARG;
    return LS_ERR_CUDA;
}

}  // namespace

extern "C" {

int32_t lsk_num_sms(void) { return gemm_num_sms(); }

uint32_t lsk_device_error(void) {
    if (!g_err_host) return 0;
    uint32_t v = *(volatile uint32_t*)g_err_host;
    *(volatile uint32_t*)g_err_host = 0;
    return v;
}

ls_status lsk_copy_h2slot(void* dst_dev, const void* src_host, uint64_t bytes, int32_t ctas, uint32_t* ready_dev,
                          uint32_t* ticket_dev, uint32_t epoch, void* stream) {
    if (!dst_dev || !src_host || !ready_dev || !ticket_dev) return LS_ERR_INVALID_ARG;
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, src_host) != cudaSuccess || a.type != cudaMemoryTypeHost || !a.devicePointer) {
        cudaGetLastError();
        return LS_ERR_INVALID_ARG;
    }
    if (((uintptr_t)a.devicePointer & 15) || ((uintptr_t)dst_dev & 15)) return LS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    CopyRange r{};
    r.src = a.devicePointer;
    r.dst_off = 0;
    r.n16 = (int64_t)(bytes / 16);
    r.tail = (int32_t)(bytes % 16);
    r.chunk_begin = 0;
    const int64_t chunks = bytes ? std::max<int64_t>(1, copy_chunks_for(r.n16)) : 0;
    CopyRange* rd = nullptr;
    if (chunks) {
        if (cudaMallocAsync(&rd, sizeof(CopyRange), s) != cudaSuccess) return LS_ERR_CUDA;
        if (cudaMemcpyAsync(rd, &r, sizeof(r), cudaMemcpyHostToDevice, s) != cudaSuccess) return LS_ERR_CUDA;
    }
    int c = ctas > 0 ? ctas : gemm_num_sms();
    cudaError_t e = launch_copy_h2slot(rd, chunks ? 1 : 0, chunks, dst_dev, nullptr, 1, ready_dev, ticket_dev, epoch,
                                       true, c, s);
    if (rd) cudaFreeAsync(rd, s);
    return st(e);
}

ls_status lsk_wait_ready(const uint32_t* ready_dev, uint32_t epoch, int32_t limit_ms, uint32_t* err_host,
                         int32_t slot, void* stream) {
    if (!ready_dev || !err_host || limit_ms < 1 || limit_ms > 600000) return LS_ERR_INVALID_ARG;
    uint32_t* ed = nullptr;
    if (cudaHostGetDevicePointer((void**)&ed, err_host, 0) != cudaSuccess) {
        cudaGetLastError();
        return LS_ERR_INVALID_ARG;
    }
    return st(launch_wait_ready(ready_dev, epoch, (uint64_t)limit_ms * 1000000ull, ed,
                                DERR_HANDOFF_TIMEOUT | ((uint32_t)slot << 8), (cudaStream_t)stream));
}

// A memory pool per device for the entry points' short-lived scratch (the split-K partial
// tiles): freed blocks stay in the pool (no release threshold), so calls in a loop do not map
// and unmap device memory each time. Other allocators' pools are left alone.
static cudaMemPool_t scratch_pool() {
    static std::mutex mu;
    static cudaMemPool_t pools[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> g(mu);
    if (!pools[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        if (cudaMemPoolCreate(&pools[dev], &props) != cudaSuccess) {
            cudaGetLastError();
            pools[dev] = nullptr;
            return nullptr;
        }
        uint64_t keep = UINT64_MAX;
        cudaMemPoolSetAttribute(pools[dev], cudaMemPoolAttrReleaseThreshold, &keep);
        cudaGetLastError();
    }
    return pools[dev];
}

ls_status lsk_gemm_bf16(int32_t epilogue, const void* A, const void* B, int64_t b_rows, int32_t b2_row_off,
                        const void* bias, const void* resid, int32_t resid_f32, void* C, void* C32, int32_t M,
                        int32_t N, int32_t K, int32_t max_ctas, void* stream) {
    if (epilogue < LSK_EPI_STORE || epilogue > LSK_EPI_RESID) return LS_ERR_INVALID_ARG;
    if ((epilogue == LSK_EPI_BIAS_GELU || epilogue == LSK_EPI_BIAS_RESID) && !bias) return LS_ERR_INVALID_ARG;
    if ((epilogue == LSK_EPI_BIAS_RESID || epilogue == LSK_EPI_RESID) && !resid) return LS_ERR_INVALID_ARG;
    if (!A || !B || !C || M < 0 || N <= 0 || K <= 0) return LS_ERR_INVALID_ARG;
    if (b_rows < (epilogue == LSK_EPI_SWIGLU ? (int64_t)b2_row_off + N : N)) return LS_ERR_INVALID_ARG;
    GemmDesc d;
    d.epi = epilogue;
    d.A = A; d.lda = K; d.a_rows = M;
    d.B = B; d.ldb = K; d.b_rows = b_rows;
    d.b2_row_off = b2_row_off;
    d.bias = bias;
    d.resid = resid; d.ldr = N;
    d.resid_f32 = resid_f32 != 0;
    d.C = C; d.ldc = N;
    d.C32 = C32;
    d.M = M; d.N = N; d.K = K;
    d.err_word = err_dev();
    // a small GEMM split along K needs a workspace for its partial tiles: stream-ordered, from
    // a memory pool of this library's own that keeps freed memory for the next call
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t ws = gemm_split_ws_bytes(M, N, K, epilogue);
    if (ws > 0) {
        cudaMemPool_t pool = scratch_pool();
        if (!pool || cudaMallocFromPoolAsync((void**)&d.splitk_ws, (size_t)ws, pool, s) != cudaSuccess) {
            cudaGetLastError();
            return LS_ERR_OOM;
        }
        d.splitk_ws_bytes = ws;
    }
    const cudaError_t e = launch_gemm_bf16(d, max_ctas, s);
    if (d.splitk_ws) cudaFreeAsync(d.splitk_ws, s);
    return st(e);
}

int32_t lsk_gemm_tile_n(int32_t epilogue, int32_t M, int32_t N) {
    if (epilogue < LSK_EPI_STORE || epilogue > LSK_EPI_RESID || M < 1 || N < 1) return 0;
    if (epilogue == LSK_EPI_SWIGLU) return 128;
    return M > 128 ? gemm_pair_tile_n(M, N) : 256;
}

ls_status lsk_gemm_grouped_bf16(int32_t epilogue, const void* A, const void* B, int64_t b_rows, int32_t b_base_row,
                                int32_t b_group_stride_rows, int32_t b2_row_off, const int32_t* group_bounds,
                                int32_t n_groups, const int32_t* row_table, const float* row_weight, void* C,
                                int32_t M, int32_t N, int32_t K, int32_t max_ctas, void* stream) {
    if (epilogue != LSK_EPI_SWIGLU && epilogue != LSK_EPI_SCALE_F32) return LS_ERR_INVALID_ARG;
    if (!A || !B || !C || !group_bounds || n_groups < 1 || M < 0 || N <= 0 || K <= 0) return LS_ERR_INVALID_ARG;
    if (epilogue == LSK_EPI_SCALE_F32 && (!row_table || !row_weight)) return LS_ERR_INVALID_ARG;
    GemmDesc d;
    d.epi = epilogue;
    d.A = A; d.lda = K; d.a_rows = M;
    d.B = B; d.ldb = K; d.b_rows = b_rows;
    d.b2_row_off = b2_row_off;
    d.C = C; d.ldc = N;
    d.M = M; d.N = N; d.K = K;
    d.group_bounds = group_bounds;
    d.n_groups = n_groups;
    d.b_group_stride_rows = b_group_stride_rows;
    d.b_base_row = b_base_row;
    d.row_table = row_table;
    d.row_weight = row_weight;
    d.err_word = err_dev();
    return st(launch_gemm_bf16(d, max_ctas, (cudaStream_t)stream));
}

ls_status lsk_linear_gelu_f32(const float* x, const float* w, const float* b, float* y, int32_t T, int32_t H,
                              int32_t F, void* stream) {
    if (!x || !w || !b || !y || T < 0 || H <= 0 || F <= 0) return LS_ERR_INVALID_ARG;
    return st(launch_linear_gelu_f32(x, w, b, y, T, H, F, (cudaStream_t)stream));
}

ls_status lsk_moe_route(const float* logits, int32_t n_layers, int32_t T, int32_t E, int32_t k, int32_t* sel,
                        float* weight, void* stream) {
    if (!logits || !sel || !weight || n_layers < 0 || T < 0) return LS_ERR_INVALID_ARG;
    return st(launch_moe_route(logits, n_layers, T, E, k, sel, weight, (cudaStream_t)stream));
}

ls_status lsk_moe_group(const int32_t* sel, int32_t n_layers, int32_t T, int32_t E, int32_t k, int32_t* row_table,
                        int32_t* group_bounds, uint8_t* expert_used, void* stream) {
    if (!sel || !row_table || !group_bounds || T < 0 || k < 1) return LS_ERR_INVALID_ARG;
    return st(launch_moe_group(sel, n_layers, T, E, k, row_table, group_bounds, expert_used, (cudaStream_t)stream));
}

ls_status lsk_moe_group_masked(const int32_t* sel, int32_t n_layers, int32_t T, int32_t E, int32_t k,
                               const uint8_t* expert_mask, int32_t* row_table, int32_t* group_bounds,
                               uint8_t* expert_used, void* stream) {
    if (!sel || !expert_mask || !row_table || !group_bounds || T < 0 || k < 1) return LS_ERR_INVALID_ARG;
    return st(launch_moe_group(sel, n_layers, T, E, k, row_table, group_bounds, expert_used, (cudaStream_t)stream,
                               expert_mask));
}

// The device address of p: p itself for device memory, the mapped address for pinned host
// memory; NULL when the device cannot reach p.
static const void* device_address(const void* p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
    if (a.type == cudaMemoryTypeHost) return a.devicePointer;
    return nullptr;
}

ls_status lsk_moe_rows_copy(const float* src, const int32_t* src_table, float* dst, const int32_t* dst_table,
                            int32_t rows, int32_t H, uint32_t* ready_dev, uint32_t* ticket_dev, uint32_t epoch,
                            int32_t ctas, void* stream) {
    if (!src || !dst || rows < 0 || H < 4 || (H % 4) || (ready_dev && !ticket_dev)) return LS_ERR_INVALID_ARG;
    const float* s = static_cast<const float*>(device_address(src));
    float* d = static_cast<float*>(const_cast<void*>(device_address(dst)));
    if (!s || !d || ((uintptr_t)s & 15) || ((uintptr_t)d & 15)) return LS_ERR_INVALID_ARG;
    const int c = ctas > 0 ? ctas : gemm_num_sms();
    return st(launch_moe_rows_copy(s, src_table, d, dst_table, rows, H, ready_dev, ticket_dev, epoch, c,
                                   (cudaStream_t)stream));
}

ls_status ls_host_alloc(uint64_t bytes, void** out) {
    if (!out || bytes == 0) return LS_ERR_INVALID_ARG;
    *out = nullptr;
    if (cudaHostAlloc(out, (size_t)bytes, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess) {
        cudaGetLastError();
        *out = nullptr;
        return LS_ERR_OOM;
    }
    return LS_OK;
}

ls_status ls_host_free(void* p) {
    if (!p) return LS_OK;
    if (cudaFreeHost(p) != cudaSuccess) {
        cudaGetLastError();
        return LS_ERR_INVALID_ARG;
    }
    return LS_OK;
}

double ls_helper_share(int64_t tokens) {
    // "prefill: a layer split's idle card streams a share of a one-chunk prompt's experts",
    // What: min(0.45, 0.5 - T/16384), off below 0.3
    const double s = std::min(0.45, 0.5 - (double)tokens / 16384.0);
    return s >= 0.3 ? s : 0.0;
}

ls_status ls_helper_split(const uint8_t* routed, int32_t E, double share, uint8_t* helper_mask) {
    if (!routed || !helper_mask || E < 0 || !(share >= 0.0 && share <= 1.0)) return LS_ERR_INVALID_ARG;
    int n = 0;
    for (int e = 0; e < E; ++e) n += routed[e] != 0;
    const int n_h = (int)std::floor(share * n);
    // the helper takes the n_h highest-numbered routed experts
    int left = n_h;
    for (int e = E - 1; e >= 0; --e) {
        helper_mask[e] = (routed[e] && left > 0) ? 1 : 0;
        if (helper_mask[e]) --left;
    }
    return LS_OK;
}

ls_status lsk_moe_gather(const void* x, const int32_t* row_table, int32_t rows, int32_t k, int32_t H,
                         void* x_sorted, void* stream) {
    if (!x || !row_table || !x_sorted || rows < 0 || k < 1) return LS_ERR_INVALID_ARG;
    return st(launch_moe_gather(x, row_table, rows, k, H, x_sorted, (cudaStream_t)stream));
}

ls_status lsk_moe_combine(const void* x, int32_t x_f32, const float* y, int32_t T, int32_t k, int32_t H, void* out,
                          float* out32, void* stream) {
    if (!x || !y || !out || T < 0 || k < 1 || k > 8) return LS_ERR_INVALID_ARG;
    return st(launch_moe_combine(x, x_f32 != 0, y, T, k, H, out, out32, (cudaStream_t)stream));
}

ls_status lsk_moe_check(const int32_t* sel, const int32_t* table, const int32_t* bounds, int32_t n_layers, int32_t T,
                        int32_t k, int32_t E, uint32_t* err_host, void* stream) {
    if (!sel || !table || !bounds || !err_host || n_layers < 0 || T < 0 || k < 1 || E < 1) return LS_ERR_INVALID_ARG;
    uint32_t* ed = nullptr;
    if (cudaHostGetDevicePointer((void**)&ed, err_host, 0) != cudaSuccess) {
        cudaGetLastError();
        return LS_ERR_INVALID_ARG;
    }
    return st(launch_moe_check(sel, table, bounds, n_layers, T, k, E, ed, 0x20000u, (cudaStream_t)stream));
}

}  // extern "C"
