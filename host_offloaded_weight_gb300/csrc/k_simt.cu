// fp32 linear + bias + GELU for the tiny fp32 stack: y = GELU(x W^T + b).
// At 8 tokens this is a latency problem, not a throughput one: one warp per
// output column n reads row n of W with coalesced loads, keeps x in shared
// memory, and reduces each token's dot product with a fixed butterfly, so the
// result is the same on every run. A lane's W values of a 256-column chunk are
// all requested before the first use (one memory latency per chunk, not eight),
// and the kernel is launched behind its predecessor (programmatic dependent
// launch): it waits for that kernel only before its first global read.
#include "common.cuh"
#include "kernels.h"

namespace ls {

static constexpr int SIMT_WARPS = 8;
static constexpr int SIMT_MAX_T = 16;
static constexpr int SIMT_KCHUNK = 8;  // W values per lane requested together

__global__ void __launch_bounds__(SIMT_WARPS * 32)
linear_gelu_f32_kernel(const float* __restrict__ x, const float* __restrict__ w,
                       const float* __restrict__ b, float* __restrict__ y, int T, int H, int F) {
    extern __shared__ float xs[];  // [tc][H] for the current token chunk
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x * SIMT_WARPS + warp;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the previous kernel's output is x
    for (int t0 = 0; t0 < T; t0 += SIMT_MAX_T) {
        const int tc = min(SIMT_MAX_T, T - t0);
        __syncthreads();
        for (int i = threadIdx.x; i < tc * H; i += blockDim.x) xs[i] = x[(int64_t)t0 * H + i];
        __syncthreads();
        if (n >= F) continue;
        float acc[SIMT_MAX_T];
#pragma unroll
        for (int t = 0; t < SIMT_MAX_T; ++t) acc[t] = 0.f;
        const float* wr = w + (int64_t)n * H;
        for (int k0 = 0; k0 < H; k0 += 32 * SIMT_KCHUNK) {
            float wv[SIMT_KCHUNK];
#pragma unroll
            for (int i = 0; i < SIMT_KCHUNK; ++i) {  // all of the chunk's loads in flight
                const int k = k0 + 32 * i + lane;
                wv[i] = k < H ? __ldg(wr + k) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < SIMT_KCHUNK; ++i) {
                const int k = k0 + 32 * i + lane;
                if (k >= H) break;
#pragma unroll
                for (int t = 0; t < SIMT_MAX_T; ++t)
                    if (t < tc) acc[t] = fmaf(xs[t * H + k], wv[i], acc[t]);
            }
        }
#pragma unroll
        for (int t = 0; t < SIMT_MAX_T; ++t) {
            float v = acc[t];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            acc[t] = v;
        }
        if (lane == 0) {
            const float bn = b[n];
            for (int t = 0; t < tc; ++t) {
                const float z = acc[t] + bn;
                y[(int64_t)(t0 + t) * F + n] = 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
            }
        }
    }
}

cudaError_t launch_linear_gelu_f32(const float* x, const float* w, const float* b, float* y, int T,
                                   int H, int F, cudaStream_t s, bool pdl) {
    if (T <= 0) return cudaSuccess;
    size_t smem = (size_t)SIMT_MAX_T * H * sizeof(float);
    if (smem > 200 * 1024) return cudaErrorInvalidValue;
    static size_t attr = 0;
    if (smem > 48 * 1024 && smem > attr) {
        cudaError_t e = cudaFuncSetAttribute(linear_gelu_f32_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attr = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((F + SIMT_WARPS - 1) / SIMT_WARPS);
    cfg.blockDim = dim3(SIMT_WARPS * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, linear_gelu_f32_kernel, x, w, b, y, T, H, F);
}

}  // namespace ls
