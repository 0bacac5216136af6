// Debug checks that stand in for a memory sanitizer (params.debug_checks).
//
// canary_kernel: every pool slot, the shared region and every per-load buffer get a
// 256-byte canary right after their last byte. It is filled with a fixed pattern when
// the memory is allocated and compared after each pass: a copy or a kernel that writes
// past the end of its slot changes it. The comparison only reads the canary.
//
// moe_check_kernel: the routing tables the grouped GEMMs and the combine index with
// (row table and group bounds, "prefill: a layer split's idle card streams a share of
// a one-chunk prompt's experts", What) are checked against the expert choice they were
// built from: bounds from 0 to T*k, never decreasing, and group e holding exactly the
// rows routed to expert e in increasing order. A violation is recorded in the error
// word; no index read from the tables is used to address memory here.
#include "common.cuh"
#include "kernels.h"

namespace ls {

static constexpr unsigned long long CANARY_PATTERN = 0xC0FFEE00D15EA5E5ull;
static constexpr int CANARY_WORDS = (int)(CANARY_BYTES / 8);

__global__ void canary_kernel(uint8_t* base, int64_t stride, int count, int check, uint32_t* err_word,
                              uint32_t region0) {
    for (int r = blockIdx.x; r < count; r += gridDim.x) {
        unsigned long long* w = reinterpret_cast<unsigned long long*>(base + (int64_t)r * stride);
        for (int i = threadIdx.x; i < CANARY_WORDS; i += blockDim.x) {
            const unsigned long long want = CANARY_PATTERN ^ (unsigned long long)i;
            if (!check)
                w[i] = want;
            else if (w[i] != want)
                raise_error(err_word, DERR_BOUNDS | ((region0 + (uint32_t)r) << 8));
        }
    }
}

cudaError_t launch_canary(void* base, int64_t stride, int count, bool check, uint32_t* err_word, uint32_t region0,
                          cudaStream_t s) {
    if (count <= 0 || !base) return cudaSuccess;
    const int grid = count < 1024 ? count : 1024;
    canary_kernel<<<grid, 32, 0, s>>>(reinterpret_cast<uint8_t*>(base), stride, count, check ? 1 : 0, err_word,
                                      region0);
    return cudaGetLastError();
}

static constexpr int CHECK_THREADS = 256;

// One CTA per layer.
__global__ void __launch_bounds__(CHECK_THREADS)
moe_check_kernel(const int* __restrict__ sel_all, const int* __restrict__ table_all,
                 const int* __restrict__ bounds_all, int T, int k, int E, uint32_t* err_word, uint32_t region0) {
    const int layer = blockIdx.x;
    const int n = T * k;
    const int* sel = sel_all + (int64_t)layer * n;
    const int* table = table_all + (int64_t)layer * n;
    const int* bounds = bounds_all + (int64_t)layer * (E + 1);
    const uint32_t code = DERR_BOUNDS | ((region0 + (uint32_t)layer) << 8);
    bool bad = false;
    if (threadIdx.x == 0 && (bounds[0] != 0 || bounds[E] != n)) bad = true;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int lo = bounds[e], hi = bounds[e + 1];
        if (lo > hi || lo < 0 || hi > n) {
            bad = true;
            continue;
        }
        // the rows of group e: routed to e, strictly increasing (so each appears once)
        for (int i = lo; i < hi; ++i) {
            const int r = table[i];
            if (r < 0 || r >= n || sel[r] != e || (i > lo && table[i - 1] >= r)) {
                bad = true;
                break;
            }
        }
    }
    // every row's expert is one of the E groups: together with the above, the groups hold
    // exactly the n rows, so the table is a permutation
    for (int r = threadIdx.x; r < n; r += blockDim.x)
        if (sel[r] < 0 || sel[r] >= E) bad = true;
    if (bad) raise_error(err_word, code);
}

cudaError_t launch_moe_check(const int* sel, const int* row_table, const int* bounds, int n_layers, int T, int k,
                             int E, uint32_t* err_word, uint32_t region0, cudaStream_t s) {
    if (n_layers <= 0 || T <= 0) return cudaSuccess;
    moe_check_kernel<<<n_layers, CHECK_THREADS, 0, s>>>(sel, row_table, bounds, T, k, E, err_word, region0);
    return cudaGetLastError();
}

}  // namespace ls
