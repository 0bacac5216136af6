// Host-to-slot copy, ready-word publish and bounded wait.
//
// copy_h2slot: the segment's tensors live in pinned, mapped host memory; the
// kernel reads them through their device-visible addresses with 16-byte
// vector loads (several in flight per thread) and writes them into the slot
// ("prefill: a layer split's idle card streams a share of a one-chunk prompt's
// experts", What: a copy kernel with 16-byte loads from mapped host memory
// instead of copy-engine uploads). After its last store every CTA issues a
// system-scope fence and takes a ticket; the CTA that takes the last ticket
// raises the slot's ready word to the load's epoch ("layer split: overlap the
// stages' hand-off", description: payload, system fence, the last block
// raises the flag).
//
// wait_ready: the consumer side. One thread spins with an acquire load until
// the slot's ready word equals the expected epoch, bounded by a time limit;
// on timeout it records the error word and returns so the stream drains
// ("layer split: overlap the stages' hand-off", Changes since #936: bounded
// wait, error word, the host fails the window). A wait that finds the error
// word already set returns at once, so one lost hand-off costs one limit.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace ls {

// One chunk = CHUNK_UNITS 16-byte units of one range.
// 256 threads x 8 loads of 16 B in flight: small enough (about 16K registers per
// CTA) to sit on an SM next to a GEMM CTA.
static constexpr int COPY_THREADS = 256;
static constexpr int COPY_UNROLL = 8;
static constexpr int64_t CHUNK_UNITS = (int64_t)COPY_THREADS * COPY_UNROLL;

__global__ void __launch_bounds__(COPY_THREADS, 4)
copy_h2slot_kernel(const CopyRange* __restrict__ ranges, int n_ranges, int64_t n_chunks,
                   uint8_t* __restrict__ dst_base, const uint8_t* __restrict__ group_mask, int ranges_per_group,
                   uint32_t* ready, uint32_t* ticket, uint32_t epoch, int publish) {
    for (int64_t c = blockIdx.x; c < n_chunks; c += gridDim.x) {
        // find the range holding chunk c (ranges are few; chunk_begin is sorted)
        int lo = 0, hi = n_ranges - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (ranges[mid].chunk_begin <= c) lo = mid; else hi = mid - 1;
        }
        const CopyRange& r = ranges[lo];
        if (group_mask && !group_mask[lo / ranges_per_group]) continue;
        const int64_t u0 = (c - r.chunk_begin) * CHUNK_UNITS;
        const uint4* src = reinterpret_cast<const uint4*>(r.src);
        uint4* dst = reinterpret_cast<uint4*>(dst_base + r.dst_off);
        uint4 v[COPY_UNROLL];
#pragma unroll
        for (int i = 0; i < COPY_UNROLL; ++i) {
            int64_t u = u0 + (int64_t)i * COPY_THREADS + threadIdx.x;
            if (u < r.n16) v[i] = __ldg(src + u);
        }
#pragma unroll
        for (int i = 0; i < COPY_UNROLL; ++i) {
            int64_t u = u0 + (int64_t)i * COPY_THREADS + threadIdx.x;
            if (u < r.n16) dst[u] = v[i];
        }
        // tail bytes (< 16) of the range, done by the chunk that holds the range's end
        if (r.tail && threadIdx.x == 0 && u0 + CHUNK_UNITS >= r.n16) {
            const uint8_t* s8 = reinterpret_cast<const uint8_t*>(r.src) + r.n16 * 16;
            uint8_t* d8 = dst_base + r.dst_off + r.n16 * 16;
            for (int b = 0; b < r.tail; ++b) d8[b] = s8[b];
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence_system();
        unsigned prev = atomicAdd(ticket, 1u);
        if (prev == gridDim.x - 1) {  // every CTA has fenced its stores
            *ticket = 0;              // next launch on this slot is stream-ordered after us
            __threadfence();
            if (publish) st_release_gpu(ready, epoch);
        }
    }
}

__global__ void publish_kernel(uint32_t* ready, uint32_t epoch, int publish) {
    __threadfence_system();
    if (publish) st_release_gpu(ready, epoch);
}

__global__ void wait_ready_kernel(const uint32_t* ready, uint32_t epoch, uint64_t limit_ns,
                                  uint32_t* err_word, uint32_t code, int early_dependents) {
    // The GEMM behind this wait may be placed now (it reads the weights only after
    // this kernel has completed) - but only when the copy this waits for needs no SM:
    // placed GEMM CTAs fill every SM, and a copy or publish kernel could then never
    // run, so the wait would run out instead of ending.
    if (early_dependents) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x != 0) return;
    if (*(volatile uint32_t*)err_word) return;
    if (ld_acquire_gpu(ready) == epoch) return;
    const uint64_t t0 = globaltimer_ns();
    unsigned ns = 32;
    while (ld_acquire_gpu(ready) != epoch) {
        if (globaltimer_ns() - t0 > limit_ns) {
            raise_error(err_word, code);
            return;
        }
        __nanosleep(ns);
        if (ns < 256) ns <<= 1;
    }
}

int64_t copy_chunks_for(int64_t n16) { return (n16 + CHUNK_UNITS - 1) / CHUNK_UNITS; }

cudaError_t launch_copy_h2slot(const CopyRange* ranges_dev, int n_ranges, int64_t n_chunks,
                               void* dst_base, const uint8_t* group_mask_dev, int ranges_per_group, uint32_t* ready,
                               uint32_t* ticket, uint32_t epoch, bool publish, int ctas,
                               cudaStream_t s) {
    if (n_chunks <= 0 || n_ranges <= 0) {
        publish_kernel<<<1, 1, 0, s>>>(ready, epoch, publish ? 1 : 0);
        return cudaGetLastError();
    }
    int grid = (int)(n_chunks < ctas ? n_chunks : ctas);
    if (grid < 1) grid = 1;
    copy_h2slot_kernel<<<grid, COPY_THREADS, 0, s>>>(ranges_dev, n_ranges, n_chunks,
                                                     reinterpret_cast<uint8_t*>(dst_base), group_mask_dev,
                                                     ranges_per_group, ready, ticket, epoch,
                                                     publish ? 1 : 0);
    return cudaGetLastError();
}

// After a copy-engine load the ready word is raised by a stream memory
// operation: it runs in stream order after the copy, behind a memory barrier,
// and needs no SM, so it is not held up by GEMM CTAs that fill every SM (a
// publish kernel was, and the next copy queued behind it). If the driver does
// not offer stream memory operations, or the stream is being captured into a
// graph (stream_op false), a one-thread kernel publishes instead.
typedef CUresult (*WriteValueFn)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);

static WriteValueFn write_value_fn() {
    static WriteValueFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<WriteValueFn>(p);
        cudaGetLastError();
    });
    return fn;
}

static bool use_mem_op = true;

bool publish_needs_no_sm() { return use_mem_op && write_value_fn() != nullptr; }

cudaError_t launch_publish(uint32_t* ready, uint32_t epoch, bool publish, cudaStream_t s, bool stream_op,
                           bool capturing) {
    if (!publish) return cudaSuccess;  // the drop hook: the word stays down
    if (capturing && stream_op) {     // a graph node; a refusal fails the capture, which is retried
        WriteValueFn fn = write_value_fn();
        if (fn && fn((CUstream)s, (CUdeviceptr)ready, epoch, CU_STREAM_WRITE_VALUE_DEFAULT) == CUDA_SUCCESS)
            return cudaSuccess;
        return cudaErrorStreamCaptureUnsupported;
    }
    if (use_mem_op && stream_op) {
        WriteValueFn fn = write_value_fn();
        if (fn && fn((CUstream)s, (CUdeviceptr)ready, epoch, CU_STREAM_WRITE_VALUE_DEFAULT) == CUDA_SUCCESS)
            return cudaSuccess;
        use_mem_op = false;
    }
    publish_kernel<<<1, 1, 0, s>>>(ready, epoch, 1);
    return cudaGetLastError();
}

// An SM's shared-memory carveout stays as it is while any CTA is resident. A copy or wait CTA
// placed under the default carveout kept GEMM CTAs (~230 KB of shared memory each) off its SM
// until it ended: in a MoE pass, a layer's GEMMs then waited out the whole next copy (5.7 ms
// instead of 0.3) whenever the copy kernel reached the SMs first. Neither kernel uses shared
// memory, so both ask for the largest carveout, under which a GEMM CTA fits beside them.
void prepare_copy_kernels() {
    cudaFuncSetAttribute(copy_h2slot_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
    cudaFuncSetAttribute(wait_ready_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
    cudaGetLastError();
}

cudaError_t launch_wait_ready(const uint32_t* ready, uint32_t epoch, uint64_t limit_ns,
                              uint32_t* err_word, uint32_t code, cudaStream_t s, bool early_dependents) {
    wait_ready_kernel<<<1, 32, 0, s>>>(ready, epoch, limit_ns, err_word, code, early_dependents ? 1 : 0);
    return cudaGetLastError();
}

}  // namespace ls
