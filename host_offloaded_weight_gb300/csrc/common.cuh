// Shared device helpers (sm_103a). Every spin in this library is bounded by the
// global nanosecond timer and reports through an error word instead of hanging.
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ls {

// error codes written into the device error word (low byte = source)
enum : uint32_t {
    DERR_HANDOFF_TIMEOUT = 0x01,  // a ready word stayed down (bits 8.. = slot)
    DERR_GEMM_TIMEOUT = 0x02,     // an mbarrier wait inside a GEMM ran out (bits 8.. = role)
    DERR_BAD_ARG = 0x03,          // a kernel found an argument it cannot handle
    DERR_BOUNDS = 0x04,           // a debug check failed (bits 8.. = region or layer)
};

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Record an error in the error word (mapped host memory, read by the host after
// the stream drains). The first writer usually wins; a race only mixes codes of
// errors that happened anyway.
__device__ __forceinline__ void raise_error(uint32_t* err_word, uint32_t code) {
    if (!err_word) return;
    volatile uint32_t* w = err_word;
    if (*w == 0u) *w = code;
    __threadfence_system();
}

}  // namespace ls
