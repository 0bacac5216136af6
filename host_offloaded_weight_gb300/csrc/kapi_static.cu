// lsk_copy_h2slot_static: the host-to-slot copy and publish without any device
// allocation (see ls_kernels.h).
//
// Callers that cannot allocate device memory: a process whose device memory is
// all owned by another allocator (a framework's caching pool that already holds
// the card), or a latency-critical loop in which cudaMalloc/cudaFree must not
// run because they can synchronise the whole device. The regular entry point
// allocates a small range table per call; this one keeps the table and the
// CTAs' ticket word in a fixed array that every device holds from the moment
// the library is loaded until the process exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "ls_kernels.h"

using namespace ls;

namespace {

// Layout: [0, 256) the ticket word (the CTAs' arrival counter); then
// LSK_STATIC_MAX_RANGES range records.
constexpr size_t TICKET_BYTES = 256;
constexpr size_t SCRATCH_BYTES = TICKET_BYTES + LSK_STATIC_MAX_RANGES * sizeof(CopyRange);
static_assert(SCRATCH_BYTES == LSK_STATIC_SCRATCH_BYTES, "the header states the scratch size");

static __device__ __align__(256) unsigned char g_copy_scratch[SCRATCH_BYTES];

// Device address of g_copy_scratch, looked up with the device current the first
// time a call runs on that device, and again whenever the device's current
// context is not the one the address was looked up in (after cudaDeviceReset the
// module is loaded anew, and an address kept from the old context would be stale).
// In host code the name g_copy_scratch is only a host-side shadow, never a
// device address.
constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void* g_scratch_dev[MAX_DEVICES] = {nullptr};
CUcontext g_scratch_ctx[MAX_DEVICES] = {nullptr};

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
        cudaGetLastError();
    });
    return fn;
}

cudaError_t scratch_for_current_device(unsigned char** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
    // make the device's primary context current (it already is after any earlier
    // runtime call on this device), so that the context read below is the one the
    // kernel will run in
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    CUcontext ctx = nullptr;
    CtxGetCurrentFn get = ctx_get_current_fn();
    if (!get || get(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_scratch_dev[dev] || g_scratch_ctx[dev] != ctx) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_copy_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_dev[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = static_cast<unsigned char*>(g_scratch_dev[dev]);
    return cudaSuccess;
}

}  // namespace

extern "C" ls_status lsk_copy_h2slot_static(void* dst_dev, const void* const* src_hosts, const uint64_t* bytes,
                                            const uint64_t* dst_offsets, int32_t n_ranges, int32_t ctas,
                                            uint32_t* ready_dev, uint32_t epoch, void* stream) {
    if (n_ranges < 1 || n_ranges > LSK_STATIC_MAX_RANGES) return LS_ERR_INVALID_ARG;  // the table holds 64
    if (!dst_dev || !src_hosts || !bytes || !dst_offsets || !ready_dev) return LS_ERR_INVALID_ARG;
    if ((uintptr_t)dst_dev & 15) return LS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    // The range table is staged from this call's stack frame. A graph captured from
    // the call would keep that stack address and read whatever lies there at each
    // replay, so a capturing stream is refused before anything else is done.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
        cudaGetLastError();
        return LS_ERR_INVALID_ARG;
    }
    if (cap != cudaStreamCaptureStatusNone) return LS_ERR_INVALID_ARG;
    CopyRange table[LSK_STATIC_MAX_RANGES];
    int64_t chunks = 0;
    for (int i = 0; i < n_ranges; ++i) {
        if (!src_hosts[i] || (dst_offsets[i] & 15)) return LS_ERR_INVALID_ARG;
        cudaPointerAttributes a;
        if (cudaPointerGetAttributes(&a, src_hosts[i]) != cudaSuccess || a.type != cudaMemoryTypeHost ||
            !a.devicePointer) {
            cudaGetLastError();
            return LS_ERR_INVALID_ARG;  // not pinned and mapped
        }
        if ((uintptr_t)a.devicePointer & 15) return LS_ERR_INVALID_ARG;
        CopyRange r{};
        r.src = a.devicePointer;
        r.dst_off = (int64_t)dst_offsets[i];
        r.n16 = (int64_t)(bytes[i] / 16);
        r.tail = (int32_t)(bytes[i] % 16);
        r.chunk_begin = chunks;
        chunks += std::max<int64_t>(1, copy_chunks_for(r.n16));
        table[i] = r;
    }
    unsigned char* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) {
        cudaGetLastError();
        return LS_ERR_CUDA;
    }
    uint32_t* ticket = reinterpret_cast<uint32_t*>(scratch);
    CopyRange* ranges = reinterpret_cast<CopyRange*>(scratch + TICKET_BYTES);
    // the ticket must start at zero; the table is rewritten by every call
    if (cudaMemsetAsync(ticket, 0, sizeof(uint32_t), s) != cudaSuccess ||
        cudaMemcpyAsync(ranges, table, sizeof(CopyRange) * n_ranges, cudaMemcpyHostToDevice, s) != cudaSuccess) {
        cudaGetLastError();
        return LS_ERR_CUDA;
    }
    const int c = ctas > 0 ? ctas : gemm_num_sms();
    cudaError_t e = launch_copy_h2slot(ranges, n_ranges, chunks, dst_dev, nullptr, 1, ready_dev, ticket, epoch,
                                       true, c, s);
    return e == cudaSuccess ? LS_OK : LS_ERR_CUDA;
}
