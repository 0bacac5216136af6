// MoE routing, expert grouping, row gather and weighted combine.
//
// "prefill: a layer split's idle card streams a share of a one-chunk prompt's
// experts" (What) runs the expert layer as: route, group the token rows by
// expert into a row table with group bounds, a grouped expert GEMM, then a
// combine. Here:
//   route    one warp per (layer, token): top-k of the fp32 logits (larger
//            first, ties to the lower expert index), then a softmax over the k
//            chosen logits in fp32.
//   group    one CTA per layer: a stable counting sort of the (token, k) rows
//            by expert. Rows of one expert keep (token, k) order, so the row
//            table does not depend on thread timing.
//   gather   x rows copied into expert order for the grouped GEMM.
//   combine  out[t] = x[t] + sum_{j<k} Y[t*k + j] in fixed j order (fp32), one
//            rounding to bf16 (plus the fp32 value for the residual stream). Y
//            holds w[t,j] * expert output, written by the grouped
//            down-projection's epilogue.
#include "common.cuh"
#include "kernels.h"

namespace ls {

static constexpr int MOE_MAX_E = 256;
static constexpr int MOE_MAX_K = 8;

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

__global__ void moe_route_kernel(const float* __restrict__ logits, int rows, int E, int k,
                                 int* __restrict__ sel, float* __restrict__ weight) {
    const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp_global >= rows) return;
    const float* lg = logits + (int64_t)warp_global * E;
    constexpr int PER = MOE_MAX_E / 32;
    float v[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        int e = lane + 32 * i;
        v[i] = e < E ? lg[e] : -INFINITY;
    }
    float chosen[MOE_MAX_K];
    int chosen_idx[MOE_MAX_K];
    unsigned taken = 0;  // bit i: this lane's candidate lane + 32 i is already chosen
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1u) && better(v[i], e, bv, bi)) { bv = v[i]; bi = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        chosen[j] = bv;
        chosen_idx[j] = bi;
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    }
    if (lane == 0) {
        float sum = 0.f, ex[MOE_MAX_K];
        for (int j = 0; j < k; ++j) {
            ex[j] = expf(chosen[j] - chosen[0]);
            sum += ex[j];
        }
        for (int j = 0; j < k; ++j) {
            sel[(int64_t)warp_global * k + j] = chosen_idx[j];
            weight[(int64_t)warp_global * k + j] = ex[j] / sum;
        }
    }
}

static constexpr int GROUP_THREADS = 1024;
static constexpr int GROUP_WARPS = GROUP_THREADS / 32;

// mask_all (may be NULL): [n_layers, E]; rows routed to an expert whose mask byte is 0 are
// left out, so the table holds the kept rows only (bounds[E] = their count).
__global__ void __launch_bounds__(GROUP_THREADS)
moe_group_kernel(const int* __restrict__ sel_all, int T, int E, int k, int* __restrict__ table_all,
                 int* __restrict__ bounds_all, uint8_t* __restrict__ used_all, const uint8_t* __restrict__ mask_all) {
    extern __shared__ int sm[];
    int* counts = sm;                    // [E]
    int* bounds = counts + E;            // [E + 1]
    int* cnt = bounds + E + 1;           // [GROUP_WARPS][E]
    const int layer = blockIdx.x;
    const int n = T * k;
    const int* sel = sel_all + (int64_t)layer * n;
    int* table = table_all + (int64_t)layer * n;
    const uint8_t* mask = mask_all ? mask_all + (int64_t)layer * E : nullptr;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < E; i += blockDim.x) counts[i] = 0;
    for (int i = threadIdx.x; i < GROUP_WARPS * E; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < n; i += blockDim.x)
        if (!mask || mask[sel[i]]) atomicAdd(&counts[sel[i]], 1);
    __syncthreads();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int e = 0; e < E; ++e) {
            bounds[e] = acc;
            acc += counts[e];
        }
        bounds[E] = acc;
    }
    // per-warp counts over a contiguous chunk of rows
    const int chunk = (n + GROUP_WARPS - 1) / GROUP_WARPS;
    const int c0 = warp * chunk, c1 = min(n, c0 + chunk);
    const unsigned lt = (1u << lane) - 1u;
    for (int b = c0; b < c1; b += 32) {
        const int i = b + lane;
        const bool act = i < c1 && (!mask || mask[sel[i]]);
        const int e = act ? sel[i] : -1 - lane;  // inactive lanes never match a real expert
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (act && (peers & lt) == 0) cnt[warp * E + e] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // base of each warp's rows inside each expert's group
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int acc = bounds[e];
        for (int w = 0; w < GROUP_WARPS; ++w) {
            int c = cnt[w * E + e];
            cnt[w * E + e] = acc;
            acc += c;
        }
    }
    __syncthreads();
    for (int b = c0; b < c1; b += 32) {
        const int i = b + lane;
        const bool act = i < c1 && (!mask || mask[sel[i]]);
        const int e = act ? sel[i] : -1 - lane;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        if (act) table[cnt[warp * E + e] + __popc(peers & lt)] = i;
        __syncwarp();
        if (act && (peers & lt) == 0) cnt[warp * E + e] += __popc(peers);
        __syncwarp();
    }
    for (int e = threadIdx.x; e <= E; e += blockDim.x) bounds_all[(int64_t)layer * (E + 1) + e] = bounds[e];
    if (used_all)
        for (int e = threadIdx.x; e < E; e += blockDim.x) used_all[(int64_t)layer * E + e] = counts[e] > 0;
}

__global__ void moe_gather_kernel(const uint4* __restrict__ x, const int* __restrict__ table, int rows,
                                  int k, int h16, uint4* __restrict__ xs) {
    const int r = blockIdx.x;
    if (r >= rows) return;
    const int t = table[r] / k;
    for (int i = threadIdx.x; i < h16; i += blockDim.x) xs[(int64_t)r * h16 + i] = x[(int64_t)t * h16 + i];
}

// K = top-k as a template parameter: the K row loads of a thread are all in flight before
// the first add; the adds run in j order (0 + y0) + y1 + ..., as for any K.
template <int K>
__global__ void moe_combine_kernel(const void* __restrict__ x, int x_f32, const float* __restrict__ y,
                                   int T, int H, __nv_bfloat16* __restrict__ out, float* __restrict__ out32) {
    const int64_t idx = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (idx >= (int64_t)T * H) return;
    const int t = (int)(idx / H), c = (int)(idx % H);
    float4 v[K];
#pragma unroll
    for (int j = 0; j < K; ++j) v[j] = __ldg(reinterpret_cast<const float4*>(y + ((int64_t)t * K + j) * H + c));
    float4 xr;
    if (x_f32) {
        xr = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(x) + idx);
    } else {
        const __nv_bfloat162* xb = reinterpret_cast<const __nv_bfloat162*>(reinterpret_cast<const __nv_bfloat16*>(x) + idx);
        const float2 a = __bfloat1622float2(xb[0]), b = __bfloat1622float2(xb[1]);
        xr = make_float4(a.x, a.y, b.x, b.y);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < K; ++j) {
        acc.x += v[j].x;
        acc.y += v[j].y;
        acc.z += v[j].z;
        acc.w += v[j].w;
    }
    const float4 o4 = make_float4(xr.x + acc.x, xr.y + acc.y, xr.z + acc.z, xr.w + acc.w);
    __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(out + idx);
    o[0] = __floats2bfloat162_rn(o4.x, o4.y);
    o[1] = __floats2bfloat162_rn(o4.z, o4.w);
    if (out32) *reinterpret_cast<float4*>(out32 + idx) = o4;
}

// dst[dst_table ? dst_table[i] : i] = src[src_table ? src_table[i] : i] for i < rows, fp32
// rows of H (H % 4 == 0) with 16-byte accesses; either side may be mapped pinned host
// memory (the hand-off of result rows between two cards without peer access). With
// `ready`, the last CTA raises ready[0] = epoch after a system fence, as the slot copy does.
__global__ void moe_rows_copy_kernel(const float4* __restrict__ src, const int* __restrict__ src_table,
                                     float4* __restrict__ dst, const int* __restrict__ dst_table, int rows, int h4,
                                     uint32_t* ready, uint32_t* ticket, uint32_t epoch) {
    for (int r = blockIdx.x; r < rows; r += gridDim.x) {
        const int64_t si = src_table ? src_table[r] : r;
        const int64_t di = dst_table ? dst_table[r] : r;
        for (int i = threadIdx.x; i < h4; i += blockDim.x) dst[di * h4 + i] = src[si * h4 + i];
    }
    if (!ready) return;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence_system();
        const unsigned prev = atomicAdd(ticket, 1u);
        if (prev == gridDim.x - 1) {
            *ticket = 0;
            __threadfence();
            st_release_gpu(ready, epoch);
        }
    }
}

cudaError_t launch_moe_rows_copy(const float* src, const int* src_table, float* dst, const int* dst_table, int rows,
                                 int H, uint32_t* ready, uint32_t* ticket, uint32_t epoch, int ctas, cudaStream_t s) {
    if ((H % 4) != 0 || rows < 0 || (ready && !ticket)) return cudaErrorInvalidValue;
    int grid = rows < ctas ? rows : ctas;
    if (grid < 1) grid = 1;
    moe_rows_copy_kernel<<<grid, 256, 0, s>>>(reinterpret_cast<const float4*>(src), src_table,
                                              reinterpret_cast<float4*>(dst), dst_table, rows, H / 4, ready, ticket,
                                              epoch);
    return cudaGetLastError();
}

cudaError_t launch_moe_route(const float* logits, int n_layers, int T, int E, int k, int* sel,
                             float* weight, cudaStream_t s) {
    if (E < 1 || E > MOE_MAX_E || k < 1 || k > MOE_MAX_K || k > E) return cudaErrorInvalidValue;
    const int rows = n_layers * T;
    if (rows <= 0) return cudaSuccess;
    const int threads = 256;
    const int grid = (int)(((int64_t)rows * 32 + threads - 1) / threads);
    moe_route_kernel<<<grid, threads, 0, s>>>(logits, rows, E, k, sel, weight);
    return cudaGetLastError();
}

cudaError_t launch_moe_group(const int* sel, int n_layers, int T, int E, int k, int* row_table,
                             int* group_bounds, uint8_t* expert_used, cudaStream_t s, const uint8_t* expert_mask) {
    if (E < 1 || E > MOE_MAX_E || n_layers <= 0) return cudaErrorInvalidValue;
    size_t smem = (size_t)(E + E + 1 + GROUP_WARPS * E) * sizeof(int);
    static size_t attr = 0;
    if (smem > 48 * 1024 && smem > attr) {
        cudaError_t e = cudaFuncSetAttribute(moe_group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        attr = smem;
    }
    moe_group_kernel<<<n_layers, GROUP_THREADS, smem, s>>>(sel, T, E, k, row_table, group_bounds, expert_used,
                                                           expert_mask);
    return cudaGetLastError();
}

cudaError_t launch_moe_gather(const void* x, const int* row_table, int rows, int k, int H,
                              void* x_sorted, cudaStream_t s) {
    if ((H % 8) != 0) return cudaErrorInvalidValue;
    if (rows <= 0) return cudaSuccess;
    moe_gather_kernel<<<rows, 128, 0, s>>>(reinterpret_cast<const uint4*>(x), row_table, rows, k, H / 8,
                                          reinterpret_cast<uint4*>(x_sorted));
    return cudaGetLastError();
}

cudaError_t launch_moe_combine(const void* x, bool x_f32, const float* y, int T, int k, int H, void* out,
                               float* out32, cudaStream_t s) {
    if ((H % 4) != 0) return cudaErrorInvalidValue;
    const int64_t n4 = (int64_t)T * H / 4;
    if (n4 <= 0) return cudaSuccess;
    const int threads = 256;
    const int grid = (int)((n4 + threads - 1) / threads);
    __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out);
    const int xf = x_f32 ? 1 : 0;
    switch (k) {
        case 1: moe_combine_kernel<1><<<grid, threads, 0, s>>>(x, xf, y, T, H, o, out32); break;
        case 2: moe_combine_kernel<2><<<grid, threads, 0, s>>>(x, xf, y, T, H, o, out32); break;
        case 3: moe_combine_kernel<3><<<grid, threads, 0, s>>>(x, xf, y, T, H, o, out32); break;
        case 4: moe_combine_kernel<4><<<grid, threads, 0, s>>>(x, xf, y, T, H, o, out32); break;
        case 5: moe_combine_kernel<5><<<grid, threads, 0, s>>>(x, xf, y, T, H, o, out32); break;
        case 6: moe_combine_kernel<6><<<grid, threads, 0, s>>>(x, xf, y, T, H, o, out32); break;
        case 7: moe_combine_kernel<7><<<grid, threads, 0, s>>>(x, xf, y, T, H, o, out32); break;
        case 8: moe_combine_kernel<8><<<grid, threads, 0, s>>>(x, xf, y, T, H, o, out32); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace ls
