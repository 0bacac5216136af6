// bf16 GEMM on the sm_103a tensor cores: C[M,N] = A[M,K] * B[N,K]^T, fp32
// accumulation in tensor memory, with the segment's elementwise work fused into
// the epilogue (bias, GELU, residual add, SiLU-gated product, routing weight).
//
// Structure (one persistent CTA per SM, 320 threads):
//   warp 0     TMA producer: 128x64 A tile and 256x64 B tile (or two 128x64 B
//              tiles for the gate/up pair) per stage, 128-byte swizzle, into a
//              4-stage shared-memory ring guarded by full/empty mbarriers.
//   warp 1     allocates 512 TMEM columns (two 128x256 fp32 accumulators) and
//              issues tcgen05.mma (M=128, K=16 per instruction) from one thread;
//              tcgen05.commit releases smem stages and hands finished
//              accumulators to the epilogue.
//   warps 2-9  epilogue: two warps per TMEM lane quarter, each taking half of
//              the tile's columns: tcgen05.ld of its 32 lanes (one output row
//              per thread), fused elementwise work in registers, then a 32x32
//              transpose through a swizzled shared buffer so that residual
//              loads and output stores are coalesced row segments. The second
//              accumulator lets the next tile's mainloop run meanwhile.
// Tiles are visited in a fixed order and each output element is produced by
// one thread from one fixed-order accumulation, so results do not depend on
// the grid size or on where the weights live.
//
// Dense GEMMs with more than 128 rows use the pair-CTA form below (256 x W tiles
// over a 2-CTA cluster, W in {256, 224, 192, 160} chosen per shape, 10 or 18
// warps); single-CTA 128x256 tiles serve the grouped mode and short problems.
//
// Grouped mode (expert GEMM of the MoE stack): rows of A are already sorted by
// expert; group g owns rows [group_bounds[g], group_bounds[g+1]) and reads its
// own B matrix at row b_base_row + g * b_group_stride_rows of the B view.
//
// Every mbarrier wait is bounded in time; on expiry the CTA records an error
// word, stops issuing work, waits (bounded) for its own copies and MMAs, frees
// its TMEM and exits. The GEMM never waits on another kernel: a persistent
// grid that spins on a flag would hold the SMs its producer needs.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

#include <algorithm>
#include <cstdint>
#include <mutex>
#include <unordered_map>

namespace ls {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int ACC_COLS = 256;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = ACC_COLS * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + 32 * EPI_WARPS;
constexpr int EPI_BUF_BYTES = 32 * 32 * 4;  // one 32x32 fp32 transpose buffer per epilogue warp
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + EPI_WARPS * EPI_BUF_BYTES + 1024 + 256;
constexpr uint64_t MBAR_LIMIT_NS = 2000000000ull;  // 2 s: far above any legitimate stall
constexpr int MAX_GROUPS = 256;

struct GemmParams {
    CUtensorMap tmA;
    CUtensorMap tmB;
    CUtensorMap tmC;    // pair kernel: bf16 output, 32x32 box, 64-byte swizzle
    CUtensorMap tmC32;  // pair kernel: fp32 output copy, 32x32 box, 128-byte swizzle
    CUtensorMap tmB2;   // grouped: a second B view (the expert cache), same row pitch and box
    int M, N, K;
    int num_m_tiles, num_n_tiles, num_k_blocks, num_tiles;
    int b2_row_off;
    const __nv_bfloat16* bias;
    const void* resid;       // bf16, or fp32 when resid_f32
    int resid_f32;
    int64_t ldr;
    void* C;
    int64_t ldc;
    float* C32;              // optional fp32 copy of the output (same ldc)
    const int* group_bounds;
    int n_groups;
    int b_group_stride_rows;
    int b_base_row;
    const int* row_table;
    const float* row_weight;
    const int* group_b_row;  // grouped, optional: first B row of group g's matrix; top bit set = in tmB2
    uint32_t* err;
    uint64_t mbar_limit_ns;  // bound of every internal mbarrier wait
    int pdl;                 // host side: launch with programmatic stream serialization
    int splits;              // EPI_PARTIAL: K slices; slice s of tile t is work item s * num_tiles + t
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait; false (with the error word set) if the phase did not complete in
// time. The common case (phase already complete) stays inline: an out-of-line
// call per k-block cost the MMA issuer about a third of its rate.
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, uint32_t* err, uint32_t role,
                                            uint64_t limit_ns);
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* err, uint32_t role,
                                          uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_slow(bar, parity, err, role, limit_ns);
}
__device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, uint32_t* err, uint32_t role,
                                            uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            raise_error(err, DERR_GEMM_TIMEOUT | (role << 8));
            return false;
        }
    }
    return true;
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// Programmatic dependent launch: a GEMM is launched while the kernel before it in
// the stream is still running, so its prologue (barriers, TMEM, descriptors)
// overlaps that kernel's tail. grid_dep_wait() blocks until the previous kernel
// has completed and its writes are visible, and comes before this kernel's first
// global-memory access; grid_dep_launch() lets the next kernel start early.
// Both are no-ops for a launch without the attribute.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// Lane l of the warp writes r[0..31] into its TMEM lane, 32 consecutive columns from taddr.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Instruction descriptor of kind::f16: D fp32, A and B bf16, both K-major.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}
// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// ------------------------------------------------------------------ tile mapping
struct Tile {
    int a_row;     // first A row of the tile
    int row_end;   // rows >= row_end are padding (not stored)
    int b_row;     // first B row of the tile
    int n0;        // first output column
    int b_map;     // 1: B rows are in the second view (tmB2)
};

template <bool GROUPED, bool DUAL>
__device__ __forceinline__ Tile tile_of(const GemmParams& p, int t, const int* s_mt_prefix) {
    constexpr int BN = DUAL ? ACC_COLS / 2 : ACC_COLS;
    Tile r;
    if (!GROUPED) {
        int m = t % p.num_m_tiles, n = t / p.num_m_tiles;
        r.a_row = m * BM;
        r.row_end = p.M;
        r.n0 = n * BN;
        r.b_row = r.n0;
        r.b_map = 0;
    } else {
        // column tiles innermost: the CTAs of one wave share each row tile of A (read once
        // from DRAM instead of once per column tile) and a group's row tiles of B
        int n = t % p.num_n_tiles, mt = t / p.num_n_tiles;
        int lo = 0, hi = p.n_groups - 1;  // last group g with prefix[g] <= mt
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (s_mt_prefix[mid] <= mt) lo = mid; else hi = mid - 1;
        }
        int g = lo;
        int g0 = p.group_bounds[g];
        r.a_row = g0 + (mt - s_mt_prefix[g]) * BM;
        r.row_end = p.group_bounds[g + 1];
        r.n0 = n * BN;
        if (p.group_b_row) {  // per-group placement: the slot or the second view
            const int v = p.group_b_row[g];
            r.b_map = v < 0 ? 1 : 0;
            r.b_row = (v & 0x7fffffff) + r.n0;
        } else {
            r.b_map = 0;
            r.b_row = p.b_base_row + g * p.b_group_stride_rows + r.n0;
        }
    }
    return r;
}

__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }
// GELU(v) = v/2 (1 + erf(v/sqrt 2)) with erf by Abramowitz & Stegun, Handbook of
// Mathematical Functions, formula 7.1.28: for z >= 0,
//   erf(z) = 1 - (1 + a1 z + a2 z^2 + a3 z^3 + a4 z^4 + a5 z^5 + a6 z^6)^-16,
// |error| <= 3e-7 (odd extension for z < 0); evaluated in fp32 the sixteenth
// power amplifies rounding to at most 2e-6 in erf. With z = |v|/sqrt 2 and
// q = 1 - erf(z), both signs reduce to GELU(v) = max(v, 0) - (|v|/2) q.
// The argument's scale and the 1/2 are folded into the polynomial, taken in u = |v|:
// b_i = c a_i 2^(-i/2) with b_0 = c = 2^(1/16), so that (b(u))^16 = 2 (1 + ... + a6 z^6)^16 and
// GELU(v) = max(v, 0) - u / b(u)^16 (the same function; two multiplications fewer per pair).
// One approximate reciprocal per element (the only special-function op; +inf
// gives 0); the rest runs two elements per instruction on the packed fp32
// pipe. All of it sits far below the bf16 rounding of the output.
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 gelu2(float2 v) {
    const float2 u = make_float2(fabsf(v.x), fabsf(v.y));
    float2 p = __ffma2_rn(f2(5.6213e-06f), u, f2(5.105521e-05f));
    p = __ffma2_rn(p, u, f2(3.9686136e-05f));
    p = __ffma2_rn(p, u, f2(3.4227392e-03f));
    p = __ffma2_rn(p, u, f2(2.2076998e-02f));
    p = __ffma2_rn(p, u, f2(5.2075163e-02f));
    p = __ffma2_rn(p, u, f2(1.0442737f));
    p = __fmul2_rn(p, p);
    p = __fmul2_rn(p, p);
    p = __fmul2_rn(p, p);
    p = __fmul2_rn(p, p);
    const float2 q = make_float2(rcp_approx(p.x), rcp_approx(p.y));
    return __ffma2_rn(make_float2(-u.x, -u.y), q, make_float2(fmaxf(v.x, 0.f), fmaxf(v.y, 0.f)));
}
// in place over an even-length register array
template <int N>
__device__ __forceinline__ void gelu_inplace(float* v) {
#pragma unroll
    for (int j = 0; j < N; j += 2) {
        const float2 g = gelu2(make_float2(v[j], v[j + 1]));
        v[j] = g.x;
        v[j + 1] = g.y;
    }
}
__device__ __forceinline__ float silu_f(float v) { return v / (1.0f + __expf(-v)); }

// 32x32 fp32 staging of one warp, held as 32 rows x 8 float4 and XOR-swizzled
// at float4 granularity: float4 (r, c4) sits at r*8 + (c4 ^ (r & 7)). Row-wise
// writes (lane r writes its row) and row-segment reads (8 lanes read one row)
// are both free of bank conflicts within each quarter-warp phase.
__device__ __forceinline__ int sw4(int r, int c4) { return r * 8 + (c4 ^ (r & 7)); }

// Epilogue of one 32x32 chunk: lane l holds row row0 + l of the chunk in v[]
// (and u[] for the gate/up pair), columns n .. n+31. Elementwise work runs
// row-wise in registers; everything that touches global memory goes through
// the warp's staging buffer, so each instruction reads or writes four whole
// 32-column row segments with 16-byte (fp32) or 8-byte (bf16) accesses per lane.
// EPI_SCALE_F32: lane l also holds row_dst (the row table's entry for row row0 + l)
// and row_w (the routing weight of that destination row), loaded once per tile.
template <int EPI>
__device__ __forceinline__ void epilogue_chunk(const GemmParams& p, int row0, int row_end, int n, float* v,
                                               const float* u, float* buf, int row_dst = 0, float row_w = 0.f,
                                               int64_t c_off = 0) {
    const int lane = threadIdx.x & 31;
    float4* b4 = reinterpret_cast<float4*>(buf);
    const int c4 = lane & 7;              // this lane's float4 column in the transposed phase
    const int col = n + 4 * c4;           // N % 8 == 0, so a group of 4 never straddles N
    const bool col_ok = col < p.N;
    if (EPI == EPI_BIAS_GELU || EPI == EPI_BIAS_RESID) {
        const uint16_t* bb = reinterpret_cast<const uint16_t*>(p.bias) + n;
        if (n + 32 <= p.N) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
                uint4 q = *reinterpret_cast<const uint4*>(bb + j);
                const uint16_t* h = reinterpret_cast<const uint16_t*>(&q);
#pragma unroll
                for (int i = 0; i < 8; ++i) v[j + i] += bf2f(h[i]);
            }
        } else {
            for (int j = 0; j < 32; ++j) v[j] += (n + j < p.N ? bf2f(bb[j]) : 0.f);
        }
    }
    if (EPI == EPI_BIAS_GELU) gelu_inplace<32>(v);
    if (EPI == EPI_SWIGLU) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = silu_f(v[j]) * u[j];
    }
    if (EPI == EPI_BIAS_RESID || EPI == EPI_RESID) {
        float4 rv[8];
#pragma unroll
        for (int it = 0; it < 8; ++it) {  // all eight loads in flight before any use
            const int row = row0 + it * 4 + (lane >> 3);
            rv[it] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (row < row_end && col_ok) {
                if (p.resid_f32) {
                    rv[it] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.resid) +
                                                              (int64_t)row * p.ldr + col);
                } else {
                    const uint2 h = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.resid) +
                                                                    (int64_t)row * p.ldr + col);
                    rv[it] = make_float4(bf2f(h.x & 0xffff), bf2f(h.x >> 16), bf2f(h.y & 0xffff), bf2f(h.y >> 16));
                }
            }
        }
#pragma unroll
        for (int it = 0; it < 8; ++it) b4[sw4(it * 4 + (lane >> 3), c4)] = rv[it];
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 t = b4[sw4(lane, j)];
            v[4 * j] += t.x;
            v[4 * j + 1] += t.y;
            v[4 * j + 2] += t.z;
            v[4 * j + 3] += t.w;
        }
        __syncwarp();
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) b4[sw4(lane, j)] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    __syncwarp();
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int row = row0 + it * 4 + (lane >> 3);
        // every lane takes part in the shuffles, before any of them skips its row
        const int dst = EPI == EPI_SCALE_F32 ? __shfl_sync(0xffffffffu, row_dst, it * 4 + (lane >> 3)) : 0;
        const float w = EPI == EPI_SCALE_F32 ? __shfl_sync(0xffffffffu, row_w, it * 4 + (lane >> 3)) : 0.f;
        if (row >= row_end || !col_ok) continue;
        const float4 o = b4[sw4(it * 4 + (lane >> 3), c4)];
        if (EPI == EPI_SCALE_F32) {
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.C) + (int64_t)dst * p.ldc + col) =
                make_float4(w * o.x, w * o.y, w * o.z, w * o.w);
        } else if (EPI == EPI_PARTIAL) {
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.C) + c_off + (int64_t)row * p.ldc + col) = o;
        } else {
            if ((EPI == EPI_BIAS_RESID || EPI == EPI_RESID) && p.C32)
                *reinterpret_cast<float4*>(p.C32 + (int64_t)row * p.ldc + col) = o;
            __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y), hi = __floats2bfloat162_rn(o.z, o.w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.C) + (int64_t)row * p.ldc + col) = pk;
        }
    }
    __syncwarp();
}

template <int EPI, bool DUAL, bool GROUPED>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_bf16_tc(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + STAGES * STAGE_BYTES + EPI_WARPS * EPI_BUF_BYTES;
    // barrier layout: full[S], empty[S], tfull[2], tempty[2], done; then tmem base word
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * STAGES + 4);
    uint32_t* tmem_slot =
        reinterpret_cast<uint32_t*>(gbase + STAGES * STAGE_BYTES + EPI_WARPS * EPI_BUF_BYTES + 8 * (2 * STAGES + 5));
    __shared__ int s_mt_prefix[MAX_GROUPS + 1];
    __shared__ volatile int s_abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), EPI_WARPS);
        }
        mbar_init(done_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    grid_dep_wait();
    if (GROUPED && threadIdx.x == 32) {
        int acc = 0;
        for (int g = 0; g < p.n_groups; ++g) {
            s_mt_prefix[g] = acc;
            int rows = p.group_bounds[g + 1] - p.group_bounds[g];
            acc += (rows + BM - 1) / BM;
        }
        s_mt_prefix[p.n_groups] = acc;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    int num_tiles = p.num_tiles;
    if (GROUPED) num_tiles = s_mt_prefix[p.n_groups] * p.num_n_tiles;
    const int kb_n = p.num_k_blocks;
    // split K (EPI_PARTIAL): work item t is K slice t / num_tiles of tile t % num_tiles
    const int n_items = EPI == EPI_PARTIAL ? num_tiles * p.splits : num_tiles;
    auto kb_lo = [&](int t) { return EPI == EPI_PARTIAL ? (int)((int64_t)(t / num_tiles) * kb_n / p.splits) : 0; };
    auto kb_hi = [&](int t) {
        return EPI == EPI_PARTIAL ? (int)((int64_t)(t / num_tiles + 1) * kb_n / p.splits) : kb_n;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tmA);
            tma_prefetch_desc(&p.tmB);
            if (GROUPED && p.group_b_row) tma_prefetch_desc(&p.tmB2);
            bool ok = true;
            int it = 0;
            uint32_t issued_mask = 0;
            for (int t = blockIdx.x; t < n_items && ok; t += gridDim.x) {
                const Tile tl = tile_of<GROUPED, DUAL>(p, t % num_tiles, s_mt_prefix);
                for (int kb = kb_lo(t); kb < kb_hi(t); ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, p.err, 1, p.mbar_limit_ns)) {
                        ok = false;
                        s_abort = 1;
                        break;
                    }
                    const uint32_t sa = base + s * STAGE_BYTES;
                    const uint32_t sb = sa + A_BYTES;
                    mbar_expect_tx(full_bar(s), STAGE_BYTES);
                    tma_load_2d(sa, &p.tmA, full_bar(s), kb * BK, tl.a_row);
                    const CUtensorMap* mb = (GROUPED && tl.b_map) ? &p.tmB2 : &p.tmB;
                    if (DUAL) {
                        tma_load_2d(sb, mb, full_bar(s), kb * BK, tl.b_row);
                        tma_load_2d(sb + B_BYTES / 2, mb, full_bar(s), kb * BK, tl.b_row + p.b2_row_off);
                    } else {
                        tma_load_2d(sb, mb, full_bar(s), kb * BK, tl.b_row);
                    }
                    issued_mask |= 1u << s;
                }
            }
            grid_dep_launch();  // every load is issued: the next kernel may start placing CTAs
            // drain: every stage's last armed phase must have landed before exit
            for (int s = 0; s < STAGES; ++s) {
                if (!(issued_mask & (1u << s))) continue;
                // the last issue on stage s had index <= it-1 with (index % STAGES) == s
                int last = it - 1 - ((it - 1 - s) % STAGES + STAGES) % STAGES;
                mbar_wait(full_bar(s), (uint32_t)(last / STAGES) & 1u, p.err, 5, p.mbar_limit_ns);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC = DUAL ? make_idesc(BM, ACC_COLS / 2) : make_idesc(BM, ACC_COLS);
            int it = 0, tcount = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < n_items && ok; t += gridDim.x, ++tcount) {
                const int buf = tcount & 1;
                const uint32_t tph = (uint32_t)(tcount >> 1) & 1u;
                if (!mbar_wait(tempty_bar(buf), tph ^ 1u, p.err, 2, p.mbar_limit_ns) || s_abort) {
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * ACC_COLS);
                const int kb0 = kb_lo(t);
                for (int kb = kb0; kb < kb_hi(t); ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                    if (!mbar_wait(full_bar(s), ph, p.err, 3, p.mbar_limit_ns)) {
                        ok = false;
                        s_abort = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + s * STAGE_BYTES;
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t ad = make_sdesc(sa + kk * 32);
                        const uint32_t acc = (kb > kb0 || kk > 0) ? 1u : 0u;
                        if (DUAL) {
                            umma_bf16(d, ad, make_sdesc(sb + kk * 32), IDESC, acc);
                            umma_bf16(d + ACC_COLS / 2, ad, make_sdesc(sb + B_BYTES / 2 + kk * 32), IDESC, acc);
                        } else {
                            umma_bf16(d, ad, make_sdesc(sb + kk * 32), IDESC, acc);
                        }
                    }
                    umma_commit(empty_bar(s));
                }
                if (ok) umma_commit(tfull_bar(buf));
            }
            // every MMA issued by this thread has completed once done_bar flips
            umma_commit(done_bar);
            mbar_wait(done_bar, 0, p.err, 6, p.mbar_limit_ns);
        }
    } else {
        // ------------------------------------------------------------ epilogue (warps 2..9)
        const int q = warp & 3;                 // TMEM lane quarter this warp may read
        const int half = (warp - 2) >> 2;       // which half of the tile's columns
        float* ebuf = reinterpret_cast<float*>(gbase + STAGES * STAGE_BYTES + (warp - 2) * EPI_BUF_BYTES);
        int tcount = 0;
        for (int t = blockIdx.x; t < n_items; t += gridDim.x, ++tcount) {
            const int buf = tcount & 1;
            const uint32_t tph = (uint32_t)(tcount >> 1) & 1u;
            // the row table and routing weights of this warp's 32 rows are inputs: read them
            // before the accumulator is ready, once per tile (lane l: row row0 + l)
            const Tile tl = tile_of<GROUPED, DUAL>(p, t % num_tiles, s_mt_prefix);
            // split K: slice t / num_tiles writes its partial tile into its own M x N plane
            const int64_t c_off = EPI == EPI_PARTIAL ? (int64_t)(t / num_tiles) * p.M * p.ldc : 0;
            const int row0 = tl.a_row + q * 32;            // first row of this warp's 32
            const int row_end = tl.row_end < p.M ? tl.row_end : p.M;
            int row_dst = 0;
            float row_w = 0.f;
            if (EPI == EPI_SCALE_F32 && row0 + lane < row_end) {
                row_dst = p.row_table[row0 + lane];
                row_w = p.row_weight[row_dst];
            }
            // warp-uniform outcome: the warp's TMEM loads and its single arrive below need every lane
            if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar(buf), tph, p.err, 4, p.mbar_limit_ns) && !s_abort)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * ACC_COLS);
            constexpr int CHUNKS = DUAL ? ACC_COLS / 64 : ACC_COLS / 32;
            constexpr int PER_WARP = CHUNKS / (EPI_WARPS / 4);
#pragma unroll 1
            for (int c = half * PER_WARP; c < (half + 1) * PER_WARP; ++c) {
                uint32_t r[32], r2[32];
                tmem_ld32(tbase + c * 32, r);
                if (DUAL) tmem_ld32(tbase + ACC_COLS / 2 + c * 32, r2);
                tmem_ld_wait();
                const int n = tl.n0 + c * 32;
                if (n < p.N && row0 < row_end) {      // uniform across the warp
                    float v[32], u[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        v[j] = __uint_as_float(r[j]);
                        u[j] = DUAL ? __uint_as_float(r2[j]) : 0.f;
                    }
                    epilogue_chunk<EPI>(p, row0, row_end, n, v, u, ebuf, row_dst, row_w, c_off);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(buf));  // one arrive per warp
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// ------------------------------------------------------------------ pair-CTA (cta_group::2) kernel
// A 2-CTA cluster computes a 256 x BN tile: CTA r loads its 128 rows of A and
// its BN/2 rows of B (for the gate/up pair, BN = 256: the leader 128 rows of G,
// the peer 128 of U), so each SM takes in half of B; the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256) reading both CTAs' shared memory and
// writing each CTA's 128 rows into that CTA's TMEM. Both CTAs' TMA loads
// complete on the leader's full barrier; the leader's commits arrive on both
// CTAs' barriers; both epilogues release the accumulator on the leader's
// barrier. All waits are bounded, and both CTAs always reach the closing
// cluster barrier before TMEM is freed.
constexpr int S2_A = 128 * 64 * 2;             // this CTA's 128 rows of A
__host__ __device__ constexpr int s2_b_bytes(int bn) { return (bn / 2) * 64 * 2; }  // its BN/2 rows of B
__host__ __device__ constexpr int s2_stage_bytes(int bn) { return S2_A + s2_b_bytes(bn); }
constexpr int S2_STG_BF = 32 * 32 * 2;         // 32x32 bf16 output staging tile (64-byte rows)
constexpr int S2_STG_F32 = 32 * 32 * 4;        // 32x32 fp32 output staging tile (128-byte rows)
// Residual epilogues also write the fp32 copy: their staging takes room from the
// mainloop stages and they run 8 epilogue warps (their residual registers need 168
// per thread, the cap of a 10-warp CTA). The others run 16 epilogue warps (4 per TMEM
// lane quarter, 96 registers) so that more warps hide each other's latencies; every
// epilogue warp single-buffers its staging tiles. The mainloop takes as many stages
// as the rest of shared memory holds (at most 8). ONE (residual epilogues where every
// CTA pair has at most one tile): that tile is the pair's last, so its fp32 and bf16
// chunks are staged in the mainloop's stage memory, free once its MMAs are done, and
// no staging tile takes room from the stages.
__host__ __device__ constexpr bool s2_out_f32(int epi) { return epi == EPI_BIAS_RESID || epi == EPI_RESID; }
__host__ __device__ constexpr int s2_nbuf(int) { return 1; }
__host__ __device__ constexpr int s2_epi_warps(int epi) { return s2_out_f32(epi) ? 8 : 16; }
__host__ __device__ constexpr int s2_threads(int epi) { return 64 + 32 * s2_epi_warps(epi); }
__host__ __device__ constexpr int s2_warp_bytes(int epi, bool one = false) {
    return one ? 0 : s2_nbuf(epi) * (S2_STG_BF + (s2_out_f32(epi) ? S2_STG_F32 : 0));
}
__host__ __device__ constexpr int s2_stages(int epi, int bn, bool one = false) {
    return (232448 - 1024 - 256 - s2_epi_warps(epi) * s2_warp_bytes(epi, one)) / s2_stage_bytes(bn) < 8
               ? (232448 - 1024 - 256 - s2_epi_warps(epi) * s2_warp_bytes(epi, one)) / s2_stage_bytes(bn)
               : 8;
}
__host__ __device__ constexpr int s2_smem_bytes(int epi, int bn, bool one = false) {
    return s2_stages(epi, bn, one) * s2_stage_bytes(bn) + s2_epi_warps(epi) * s2_warp_bytes(epi, one) + 1024 + 256;
}
static_assert(s2_stages(EPI_BIAS_RESID, 256, true) == 7 && s2_stages(EPI_RESID, 160, true) == 8 &&
                  8 * S2_STG_F32 <= s2_stages(EPI_RESID, 160, true) * s2_stage_bytes(160),
              "one-tile residual layout: the fp32 staging fits in the stage memory");
static_assert(s2_stages(EPI_BIAS_RESID, 256) == 5 && s2_stages(EPI_STORE, 256) == 6, "stages at BN = 256");
static_assert(s2_smem_bytes(EPI_BIAS_RESID, 160) <= 232448 && s2_smem_bytes(EPI_STORE, 160) <= 232448, "shared memory");

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
    return out;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void remote_arrive(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void tma_load_2d_2sm(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster, int c0,
                                                int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma2_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void umma2_commit_both(uint32_t bar) {
    const uint16_t mask = 0x3;
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}

// Bulk tensor store from shared memory (issued by one thread; completion tracked
// per thread in bulk groups).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(src), "r"(c0), "r"(c1)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&t);
}
// v[j] += bias[n0 + j] for the columns below N.
__device__ __forceinline__ void add_bias_row(const GemmParams& p, int n0, float (&v)[32]) {
    const uint16_t* bb = reinterpret_cast<const uint16_t*>(p.bias) + n0;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (n0 + 8 * g >= p.N) break;
        const uint4 qv = *reinterpret_cast<const uint4*>(bb + 8 * g);
        const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[8 * g + 2 * i] += bf2f((uint16_t)(w[i] & 0xffff));
            v[8 * g + 2 * i + 1] += bf2f((uint16_t)(w[i] >> 16));
        }
    }
}
// The bias of one 32-column chunk held across the warp: lane j has bias[n0 + j] (0 past N).
// Read before the accumulator is ready (the bias is an input), it is then broadcast to every
// row by shuffles: the epilogue touches no global memory for it after the wait.
__device__ __forceinline__ float bias_lane(const GemmParams& p, int n0) {
    const int c = n0 + (int)(threadIdx.x & 31);
    return c < p.N ? bf2f(reinterpret_cast<const uint16_t*>(p.bias)[c]) : 0.f;
}
__device__ __forceinline__ void add_bias_lanes(float b, float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] += __shfl_sync(0xffffffffu, b, j);
}
// Four residual values at (row, col .. col+3), zeros past M or N (N % 8 == 0, so a
// group of four never straddles N).
__device__ __forceinline__ float4 load_resid4(const GemmParams& p, int row, int col) {
    if (row >= p.M || col >= p.N) return make_float4(0.f, 0.f, 0.f, 0.f);
    if (p.resid_f32)
        return *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.resid) + (int64_t)row * p.ldr + col);
    const uint2 h = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(p.resid) + (int64_t)row * p.ldr + col);
    return make_float4(bf2f((uint16_t)(h.x & 0xffff)), bf2f((uint16_t)(h.x >> 16)), bf2f((uint16_t)(h.y & 0xffff)),
                       bf2f((uint16_t)(h.y >> 16)));
}
// The residual's 32 columns n0.. of one row, as fp32 bit patterns (zeros past M or N).
__device__ __forceinline__ void load_resid_row32(const GemmParams& p, int row, int n0, uint32_t (&r)[32]) {
    float4 x[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) x[g] = load_resid4(p, row, n0 + 4 * g);
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        r[4 * g] = __float_as_uint(x[g].x);
        r[4 * g + 1] = __float_as_uint(x[g].y);
        r[4 * g + 2] = __float_as_uint(x[g].z);
        r[4 * g + 3] = __float_as_uint(x[g].w);
    }
}
__device__ __forceinline__ void st_shared_f4(uint32_t addr, float4 v) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr)
                 : "memory");
    return v;
}

template <int EPI, bool DUAL, int BN, bool ONE = false>
__global__ void __launch_bounds__(s2_threads(EPI), 1) gemm_bf16_tc2(const __grid_constant__ GemmParams p) {
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256 && (!DUAL || BN == 256), "tile width");
    static_assert(!ONE || s2_out_f32(EPI), "one-tile layout: residual epilogues");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    constexpr int S2_STAGES = s2_stages(EPI, BN, ONE);
    constexpr int S2_STAGE = s2_stage_bytes(BN);
    constexpr int WSB = s2_warp_bytes(EPI, ONE);
    constexpr bool OUT32 = s2_out_f32(EPI);
    constexpr int NBUF = s2_nbuf(EPI);
    const uint32_t stg0 = base + S2_STAGES * S2_STAGE;  // epilogue staging tiles, WSB bytes per warp
    constexpr int EW = s2_epi_warps(EPI);
    const uint32_t bar0 = stg0 + EW * WSB;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S2_STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * S2_STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * S2_STAGES + 2 + b); };
    const uint32_t done_bar = bar0 + 8u * (2 * S2_STAGES + 4);
    uint32_t* tmem_slot =
        reinterpret_cast<uint32_t*>(gbase + (bar0 - base) + 8 * (2 * S2_STAGES + 5));
    __shared__ volatile int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int cluster_id = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        s_abort = 0;
        for (int s = 0; s < S2_STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull_bar(b), 1);
            mbar_init(tempty_bar(b), 2 * EW);
        }
        mbar_init(done_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        tmem_alloc2(smem_u32(tmem_slot), 512);
        tmem_relinquish2();
    }
    tc_fence_before();
    cluster_sync();  // barriers of both CTAs initialised, TMEM allocated in both
    tc_fence_after();
    grid_dep_wait();
    const uint32_t tmem_base = *tmem_slot;
    const int num_m2 = (p.M + 255) / 256;
    const int num_tiles = num_m2 * p.num_n_tiles;  // num_n_tiles counts BN (dual: 128) columns
    const int kb_n = p.num_k_blocks;

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&p.tmA);
            tma_prefetch_desc(&p.tmB);
            int it = 0;
            uint32_t issued_mask = 0;
            bool ok = true;
            for (int t = cluster_id; t < num_tiles && ok; t += n_clusters) {
                const int m2 = t % num_m2, n = t / num_m2;
                const int a_row = m2 * 256 + (int)rank * 128;
                // dense: the pair covers 256 columns; gate/up pair: 128 columns of G (leader) and of U (peer)
                const int b_row = DUAL ? n * 128 + (rank ? p.b2_row_off : 0) : n * BN + (int)rank * (BN / 2);
                for (int kb = 0; kb < kb_n; ++kb, ++it) {
                    const int s = it % S2_STAGES;
                    const uint32_t ph = (uint32_t)(it / S2_STAGES) & 1u;
                    if (!mbar_wait(empty_bar(s), ph ^ 1u, p.err, 1, p.mbar_limit_ns)) {
                        ok = false;
                        s_abort = 1;
                        break;
                    }
                    const uint32_t sa = base + s * S2_STAGE;
                    const uint32_t sb = sa + S2_A;
                    const uint32_t leader_full = mapa(full_bar(s), 0);
                    if (leader) mbar_expect_tx(full_bar(s), 2 * S2_STAGE);
                    tma_load_2d_2sm(sa, &p.tmA, leader_full, kb * BK, a_row);
                    tma_load_2d_2sm(sb, &p.tmB, leader_full, kb * BK, b_row);
                    issued_mask |= 1u << s;
                }
            }
            grid_dep_launch();  // every load is issued: the next kernel may start placing CTAs
            // the leader's full barrier tracks both CTAs' loads: drain there (leader only)
            if (leader)
                for (int s = 0; s < S2_STAGES; ++s) {
                    if (!(issued_mask & (1u << s))) continue;
                    int last = it - 1 - ((it - 1 - s) % S2_STAGES + S2_STAGES) % S2_STAGES;
                    mbar_wait(full_bar(s), (uint32_t)(last / S2_STAGES) & 1u, p.err, 5, p.mbar_limit_ns);
                }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            constexpr uint32_t IDESC = make_idesc(256, BN);
            int it = 0, tcount = 0;
            bool ok = true;
            for (int t = cluster_id; t < num_tiles && ok; t += n_clusters, ++tcount) {
                const int buf = tcount & 1;
                const uint32_t tph = (uint32_t)(tcount >> 1) & 1u;
                if (!mbar_wait(tempty_bar(buf), tph ^ 1u, p.err, 2, p.mbar_limit_ns) || s_abort) {
                    s_abort = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(buf * ACC_COLS);
                for (int kb = 0; kb < kb_n; ++kb, ++it) {
                    const int s = it % S2_STAGES;
                    const uint32_t ph = (uint32_t)(it / S2_STAGES) & 1u;
                    if (!mbar_wait(full_bar(s), ph, p.err, 3, p.mbar_limit_ns)) {
                        ok = false;
                        s_abort = 1;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = base + s * S2_STAGE;
                    const uint32_t sb = sa + S2_A;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma2_bf16(d, make_sdesc(sa + kk * 32), make_sdesc(sb + kk * 32), IDESC,
                                   (kb > 0 || kk > 0) ? 1u : 0u);
                    umma2_commit_both(empty_bar(s));
                }
                if (ok) umma2_commit_both(tfull_bar(buf));
            }
            umma2_commit_both(done_bar);
            mbar_wait(done_bar, 0, p.err, 6, p.mbar_limit_ns);
        }
    } else {
        // Epilogue: warp (q, half) owns TMEM lanes q*32.. (its 32 output rows, one per
        // thread) and a contiguous 4/EW share of the tile's 32-column chunks (shares
        // differ by one chunk at most when they do not divide). A chunk is finished in
        // registers, written into a swizzled staging tile and sent out by one bulk
        // tensor store that runs while the warp moves on; the tensor map clips
        // rows >= M and columns >= N.
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const uint32_t stg = stg0 + (uint32_t)(warp - 2) * WSB;
        const uint32_t leader_tempty0 = mapa(tempty_bar(0), 0), leader_tempty1 = mapa(tempty_bar(1), 0);
        const bool want32 = OUT32 && p.C32 != nullptr;
        if (lane == 0) {
            tma_prefetch_desc(&p.tmC);
            if (want32) tma_prefetch_desc(&p.tmC32);
        }
        constexpr int CHUNKS = DUAL ? ACC_COLS / 64 : BN / 32;
        constexpr int WPQ = EW / 4;                                // warps per TMEM lane quarter
        constexpr int PER_WARP = (CHUNKS + WPQ - 1) / WPQ;         // the largest share
        const int c_begin = half * CHUNKS / WPQ;
        const int n_chunks = (half + 1) * CHUNKS / WPQ - c_begin;  // this warp's share
        // Residual epilogues read the residual while the accumulator is still being
        // computed: coalesced loads (8 lanes cover one row's 32 columns, 4 rows per
        // instruction) for the tile's first two chunks go out before the wait, each
        // later chunk's as soon as a register set frees up. The fp32 staging tile
        // turns each chunk into one row per lane (its layout is the 128-byte swizzle
        // the output store reads).
        const int c4 = lane & 7, rsub = lane >> 3;
        auto issue = [&](int rbase, int n0, float4 (&g)[8]) {
#pragma unroll
            for (int it = 0; it < 8; ++it) g[it] = load_resid4(p, rbase + it * 4 + rsub, n0 + 4 * c4);
        };
        auto release = [&](int b) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) remote_arrive(b ? leader_tempty1 : leader_tempty0);  // one arrive per warp
        };
        int sb = 0;
        // Chunk output: v (row per lane) goes into the swizzled staging tiles and out by
        // bulk tensor stores. The caller has made sure the staging tiles are free.
        // ONE: the cluster's one tile is its last, so all of the stage memory is free for its
        // epilogue: each warp gets ONE_NS pairs of fp32 and bf16 staging tiles there (one per
        // chunk where they fit), and a chunk waits only for the stores of the chunk ONE_NS before
        constexpr int ONE_SLOT = S2_STG_F32 + S2_STG_BF;
        constexpr int ONE_FIT = S2_STAGES * S2_STAGE / (EW * ONE_SLOT);
        constexpr int ONE_NS = ONE_FIT < PER_WARP ? ONE_FIT : PER_WARP;
        static_assert(!ONE || ONE_NS >= 1, "one-tile staging in the stage memory");
        auto store_chunk = [&](float (&v)[32], int n0, int row0, int slot) {
            const uint32_t one_slot = base + (uint32_t)(((warp - 2) * ONE_NS + slot) * ONE_SLOT);
            const uint32_t s32 = ONE ? one_slot : stg + NBUF * S2_STG_BF + (uint32_t)sb * S2_STG_F32;
            const uint32_t sbf = ONE ? one_slot + S2_STG_F32 : stg + (uint32_t)sb * S2_STG_BF;
            // 64-byte swizzle: 16-byte unit j of row r sits at unit j ^ ((r >> 1) & 3)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                st_shared_v4(sbf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4), pack_bf16(v[8 * j], v[8 * j + 1]),
                             pack_bf16(v[8 * j + 2], v[8 * j + 3]), pack_bf16(v[8 * j + 4], v[8 * j + 5]),
                             pack_bf16(v[8 * j + 6], v[8 * j + 7]));
            if (want32) {
                // 128-byte swizzle: 16-byte unit j of row r sits at unit j ^ (r & 7)
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    st_shared_v4(s32 + lane * 128 + ((j ^ (lane & 7)) << 4), __float_as_uint(v[4 * j]),
                                 __float_as_uint(v[4 * j + 1]), __float_as_uint(v[4 * j + 2]),
                                 __float_as_uint(v[4 * j + 3]));
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
                tma_store_2d(&p.tmC, sbf, n0, row0);
                if (want32) tma_store_2d(&p.tmC32, s32, n0, row0);
                bulk_commit();
            }
            if (NBUF == 2) sb ^= 1;
        };
        int tcount = 0;
        for (int t = cluster_id; t < num_tiles; t += n_clusters, ++tcount) {
            const int buf = tcount & 1;
            const uint32_t tph = (uint32_t)(tcount >> 1) & 1u;
            const int m2 = t % num_m2, n = t / num_m2;
            const int row0 = m2 * 256 + (int)rank * 128 + q * 32;
            const int nbase = DUAL ? n * 128 : n * BN;
            // GELU epilogue: the bias of this warp's first two chunks, one value per lane (more
            // chunks are rare: they read theirs after the wait)
            const bool has_bias = EPI == EPI_BIAS_GELU;
            const float bl0 = has_bias && n_chunks > 0 ? bias_lane(p, nbase + c_begin * 32) : 0.f;
            const float bl1 = has_bias && n_chunks > 1 ? bias_lane(p, nbase + (c_begin + 1) * 32) : 0.f;
            auto bias_of = [&](int i, int n0) { return i == 0 ? bl0 : i == 1 ? bl1 : bias_lane(p, n0); };
            // A CTA's last tile leaves the other accumulator buffer unused: its residual
            // goes there (row per lane, as the accumulator) while the MMAs still run, so the
            // epilogue after the last accumulator reads no global memory.
            const bool last = OUT32 && (ONE || t + n_clusters >= num_tiles);
            const uint32_t rbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)((buf ^ 1) * ACC_COLS);
            float4 g[2][8];
            if (last) {
#pragma unroll 1
                for (int i = 0; i < n_chunks; ++i) {
                    uint32_t rr[32];
                    load_resid_row32(p, row0 + lane, nbase + (c_begin + i) * 32, rr);
                    tmem_st32(rbase + (c_begin + i) * 32, rr);
                }
                tmem_st_wait();
            } else if (OUT32) {
                issue(row0, nbase + c_begin * 32, g[0]);
                if (n_chunks > 1) issue(row0, nbase + (c_begin + 1) * 32, g[1]);
            }
            // warp-uniform outcome: TMEM loads and the single arrive below need every lane
            if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar(buf), tph, p.err, 4, p.mbar_limit_ns) && !s_abort)) {
                s_abort = 1;
                break;
            }
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * ACC_COLS);
            if (last) {
#pragma unroll 1
                for (int i = 0; i < n_chunks; ++i) {
                    const int c = c_begin + i;
                    const int n0 = nbase + c * 32;
                    uint32_t r[32], rr[32];
                    tmem_ld32(tbase + c * 32, r);
                    tmem_ld32(rbase + c * 32, rr);
                    tmem_ld_wait();
                    if (n0 < p.N && row0 < p.M) {  // uniform across the warp
                        float v[32];
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                        if (EPI == EPI_BIAS_RESID) add_bias_row(p, n0, v);
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] += __uint_as_float(rr[j]);
                        if (!ONE || i >= ONE_NS) {
                            // the stores that last used these staging tiles have read them
                            if (lane == 0) bulk_wait_read<ONE ? ONE_NS - 1 : 0>();
                            __syncwarp();
                        }
                        store_chunk(v, n0, row0, ONE ? i % ONE_NS : 0);
                    }
                }
                release(buf);
                continue;
            }
            // unrolled only where the residual registers rotate (static indexing)
#pragma unroll (OUT32 ? PER_WARP : 1)
            for (int i = 0; i < PER_WARP; ++i) {
                // a fixed trip count keeps the ring's indexing static; shares one chunk
                // short skip the last pass
                const bool have = i < n_chunks;
                const int c = c_begin + i;
                const int n0 = nbase + c * 32;
                uint32_t r[32], r2[32];
                if (have) {
                    tmem_ld32(tbase + c * 32, r);
                    if (DUAL) tmem_ld32(tbase + ACC_COLS / 2 + c * 32, r2);
                    tmem_ld_wait();
                }
                if (have && n0 < p.N && row0 < p.M) {  // uniform across the warp
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
                    if (EPI == EPI_BIAS_GELU) {
                        add_bias_lanes(bias_of(i, n0), v);
                        gelu_inplace<32>(v);
                    }
                    const uint32_t s32 = stg + NBUF * S2_STG_BF + (uint32_t)sb * S2_STG_F32;
                    if (OUT32) {
                        if (EPI == EPI_BIAS_RESID) add_bias_row(p, n0, v);
                        if (lane == 0) bulk_wait_read<0>();  // the previous chunk's stores have left the staging tiles
                        __syncwarp();
#pragma unroll
                        for (int it = 0; it < 8; ++it) st_shared_f4(s32 + 16u * sw4(it * 4 + rsub, c4), g[i & 1][it]);
                        __syncwarp();
                        // each lane reads (and below overwrites) only its own row
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 t4 = ld_shared_f4(s32 + 16u * sw4(lane, j));
                            v[4 * j] += t4.x; v[4 * j + 1] += t4.y; v[4 * j + 2] += t4.z; v[4 * j + 3] += t4.w;
                        }
                    }
                    if (EPI == EPI_SWIGLU) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = silu_f(v[j]) * __uint_as_float(r2[j]);
                    }
                    if (!OUT32) {
                        // the staging tile about to be written was last read by the store NBUF chunks ago
                        if (lane == 0) bulk_wait_read<NBUF - 1>();
                        __syncwarp();
                    }
                    store_chunk(v, n0, row0, 0);
                }
                if (OUT32 && i + 2 < n_chunks) issue(row0, n0 + 64, g[i & 1]);
            }
            release(buf);
        }
        if (lane == 0) bulk_wait_all();  // stores complete before the CTA exits
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the pair's MMAs and epilogues are done before either CTA frees TMEM
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc2(tmem_base, 512);
    }
}
// ------------------------------------------------------------------ split-K reduction
// C = epilogue(sum over s of part[s]) for a GEMM whose K was cut into `splits` slices: the
// partial tiles are added in slice order (fixed, so the bits do not depend on timing), then
// the same elementwise epilogue as the unsplit kernels (bias, GELU, residual) runs on the
// sum. One thread per 4 consecutive columns.
template <int EPI>
__global__ void splitk_reduce_kernel(const float* __restrict__ part, int splits, int M, int N,
                                     const __nv_bfloat16* __restrict__ bias, const void* __restrict__ resid,
                                     int resid_f32, int64_t ldr, __nv_bfloat16* __restrict__ C, int64_t ldc,
                                     float* __restrict__ C32) {
    const int64_t i4 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int n4 = N / 4;
    if (i4 >= (int64_t)M * n4) return;
    const int row = (int)(i4 / n4), col = (int)(i4 % n4) * 4;
    const int64_t plane = (int64_t)M * N;
    float v[4] = {0.f, 0.f, 0.f, 0.f};
    const float* src = part + (int64_t)row * N + col;
    for (int s0 = 0; s0 < splits; s0 += 8) {  // eight slices' loads in flight, then added in order
        float4 t[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            t[j] = s0 + j < splits ? __ldcg(reinterpret_cast<const float4*>(src + (s0 + j) * plane))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (s0 + j < splits) { v[0] += t[j].x; v[1] += t[j].y; v[2] += t[j].z; v[3] += t[j].w; }
    }
    if (EPI == EPI_BIAS_GELU || EPI == EPI_BIAS_RESID) {
        const uint2 h = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(bias) + col);
        v[0] += bf2f((uint16_t)(h.x & 0xffff)); v[1] += bf2f((uint16_t)(h.x >> 16));
        v[2] += bf2f((uint16_t)(h.y & 0xffff)); v[3] += bf2f((uint16_t)(h.y >> 16));
    }
    if (EPI == EPI_BIAS_GELU) gelu_inplace<4>(v);
    if (EPI == EPI_BIAS_RESID || EPI == EPI_RESID) {
        if (resid_f32) {
            const float4 r = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(resid) + (int64_t)row * ldr + col);
            v[0] += r.x; v[1] += r.y; v[2] += r.z; v[3] += r.w;
        } else {
            const uint2 h = *reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(resid) + (int64_t)row * ldr + col);
            v[0] += bf2f((uint16_t)(h.x & 0xffff)); v[1] += bf2f((uint16_t)(h.x >> 16));
            v[2] += bf2f((uint16_t)(h.y & 0xffff)); v[3] += bf2f((uint16_t)(h.y >> 16));
        }
        if (C32) *reinterpret_cast<float4*>(C32 + (int64_t)row * ldc + col) = make_float4(v[0], v[1], v[2], v[3]);
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]), hi = __floats2bfloat162_rn(v[2], v[3]);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(C + (int64_t)row * ldc + col) = pk;
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D view [rows, cols] of 2- or 4-byte elements with row stride ld (elements);
// box = box_cols x box_rows.
struct MapSpec {
    const void* p;
    int64_t rows, cols, ld;
    int box_cols, box_rows;
    int esize;    // 2: bf16, 4: fp32
    int swizzle;  // bytes: 64 or 128
    bool operator==(const MapSpec& o) const {
        return p == o.p && rows == o.rows && cols == o.cols && ld == o.ld && box_cols == o.box_cols &&
               box_rows == o.box_rows && esize == o.esize && swizzle == o.swizzle;
    }
};
struct MapSpecHash {
    size_t operator()(const MapSpec& k) const {
        size_t h = std::hash<const void*>()(k.p);
        h ^= std::hash<int64_t>()(k.rows * 1000003 + k.cols * 31 + k.ld) + 0x9e3779b9 + (h << 6) + (h >> 2);
        h ^= std::hash<int64_t>()(((int64_t)k.box_cols << 24) ^ ((int64_t)k.box_rows << 8) ^ (k.esize << 4) ^
                                  k.swizzle) + 0x9e3779b9 + (h << 6) + (h >> 2);
        return h;
    }
};

bool make_tmap(CUtensorMap* m, const MapSpec& k) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)k.cols, (cuuint64_t)k.rows};
    cuuint64_t strides[1] = {(cuuint64_t)(k.ld * k.esize)};
    cuuint32_t box[2] = {(cuuint32_t)k.box_cols, (cuuint32_t)k.box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, k.esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(k.p), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    k.swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool cached_tmap(CUtensorMap* out, const MapSpec& k) {
    static std::mutex mu;
    static std::unordered_map<MapSpec, CUtensorMap, MapSpecHash> cache;
    std::lock_guard<std::mutex> g(mu);
    auto it = cache.find(k);
    if (it != cache.end()) {
        *out = it->second;
        return true;
    }
    if (!make_tmap(out, k)) return false;
    if (cache.size() > 4096) cache.clear();
    cache.emplace(k, *out);
    return true;
}
// bf16 operand view: 64-element (128-byte) K box, 128-byte swizzle
bool cached_tmap(CUtensorMap* out, const void* ptr, int64_t rows, int64_t cols, int64_t ld, int box) {
    return cached_tmap(out, MapSpec{ptr, rows, cols, ld, BK, box, 2, 128});
}

template <int EPI, bool DUAL, bool GROUPED>
cudaError_t launch_t(const GemmParams& p, int grid, cudaStream_t s) {
    auto kern = gemm_bf16_tc<EPI, DUAL, GROUPED>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = p.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int EPI, bool DUAL, int BN, bool ONE = false>
cudaError_t launch_t2(const GemmParams& p, int clusters, cudaStream_t s) {
    auto kern = gemm_bf16_tc2<EPI, DUAL, BN, ONE>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, s2_smem_bytes(EPI, BN, ONE));
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters);
    cfg.blockDim = dim3(s2_threads(EPI));
    cfg.dynamicSmemBytes = s2_smem_bytes(EPI, BN, ONE);
    cfg.stream = s;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = p.pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int EPI, bool ONE = false>
cudaError_t launch_t2_bn(const GemmParams& p, int bn, int clusters, cudaStream_t s) {
    switch (bn) {
        case 256: return launch_t2<EPI, false, 256, ONE>(p, clusters, s);
        case 224: return launch_t2<EPI, false, 224, ONE>(p, clusters, s);
        case 192: return launch_t2<EPI, false, 192, ONE>(p, clusters, s);
        case 160: return launch_t2<EPI, false, 160, ONE>(p, clusters, s);
    }
    return cudaErrorInvalidValue;
}

template <int EPI>
cudaError_t launch_splitk_reduce(const float* part, int splits, const GemmDesc& d, cudaStream_t s) {
    const int64_t n4 = (int64_t)d.M * (d.N / 4);
    const int threads = 256;
    splitk_reduce_kernel<EPI><<<(int)((n4 + threads - 1) / threads), threads, 0, s>>>(
        part, splits, d.M, d.N, reinterpret_cast<const __nv_bfloat16*>(d.bias), d.resid, d.resid_f32 ? 1 : 0, d.ldr,
        reinterpret_cast<__nv_bfloat16*>(d.C), d.ldc, reinterpret_cast<float*>(d.C32));
    return cudaGetLastError();
}

}  // namespace

int gemm_split_k(int64_t M, int64_t N, int64_t K, int epi) {
    if (M <= 0 || M > BM || N <= 0 || K <= 0) return 1;
    if (epi != EPI_STORE && epi != EPI_BIAS_GELU && epi != EPI_BIAS_RESID && epi != EPI_RESID) return 1;
    const int64_t tiles = (N + ACC_COLS - 1) / ACC_COLS;
    const int64_t kb = (K + BK - 1) / BK;
    // enough K slices to give every SM a work item, each at least two k-blocks long, but no
    // more than the slices whose fp32 partial tiles (M x N x 4 bytes each) together weigh
    // about what the weights do (N x K x 2 bytes): beyond that the partials' traffic costs
    // more than the parallelism gains
    const int64_t sp = std::min<int64_t>(std::min<int64_t>(gemm_num_sms() / tiles, kb / 2),
                                         std::max<int64_t>(2, K / (2 * M)));
    return sp >= 2 ? (int)sp : 1;
}

int64_t gemm_split_ws_bytes(int64_t M, int64_t N, int64_t K, int epi) {
    const int sp = gemm_split_k(M, N, K, epi);
    return sp > 1 ? (int64_t)sp * M * N * (int64_t)sizeof(float) : 0;
}

int64_t gemm_split_ws_max() { return (int64_t)gemm_num_sms() * BM * ACC_COLS * (int64_t)sizeof(float); }

// Tile width of a dense pair GEMM. A k-block of a 256 x BN tile costs about the time
// of BN + 1024 columns: measured on GB300, narrowing the tile from 256 to 160
// columns shortens a k-block by only ~8 %; the MMAs set the pace (with the loads
// taken out the loop is <10 % faster) and a 160-wide instruction runs at ~75 % of
// the 256-wide one's rate. The width taken
// minimises waves x (BN + 1024) over all of the device's CTA pairs: the fewest
// waves, then the narrowest tile. It depends only on the shape and the device,
// never on the grid a call is given, so a result's bits do not depend on the grid.
int gemm_pair_tile_n(int64_t M, int64_t N) {
    const int64_t clusters = std::max(1, gemm_num_sms() / 2);
    const int64_t m2 = (M + 255) / 256;
    int best = 256;
    int64_t best_cost = INT64_MAX;
    for (int bn : {256, 224, 192, 160}) {
        const int64_t tiles = m2 * ((N + bn - 1) / bn);
        const int64_t cost = ((tiles + clusters - 1) / clusters) * (bn + 1024);
        if (cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

int gemm_num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 1;
    }
    return n;
}

cudaError_t launch_gemm_bf16(const GemmDesc& d, int max_ctas, cudaStream_t s) {
    const bool dual = d.epi == EPI_SWIGLU;
    const bool grouped = d.group_bounds != nullptr;
    if (d.M < 0 || d.N <= 0 || d.K <= 0 || (d.K % 8) || (d.N % 8) || (d.lda % 8) || (d.ldb % 8) ||
        (reinterpret_cast<uintptr_t>(d.A) & 15) || (reinterpret_cast<uintptr_t>(d.B) & 15))
        return cudaErrorInvalidValue;
    if (d.epi != EPI_SCALE_F32 && ((d.ldc % 8) || (reinterpret_cast<uintptr_t>(d.C) & 15)))
        return cudaErrorInvalidValue;
    if ((d.epi == EPI_BIAS_RESID || d.epi == EPI_RESID) &&
        ((d.ldr % 8) || (reinterpret_cast<uintptr_t>(d.resid) & 15) || !d.resid))
        return cudaErrorInvalidValue;
    if (d.C32 && ((d.epi != EPI_BIAS_RESID && d.epi != EPI_RESID) || (reinterpret_cast<uintptr_t>(d.C32) & 15)))
        return cudaErrorInvalidValue;
    if (grouped && (d.n_groups < 1 || d.n_groups > MAX_GROUPS)) return cudaErrorInvalidValue;
    if (d.M == 0) return cudaSuccess;
    GemmParams p;
    memset(&p, 0, sizeof(p));
    const int BN = dual ? ACC_COLS / 2 : ACC_COLS;
    if (!cached_tmap(&p.tmA, d.A, d.a_rows > 0 ? d.a_rows : d.M, d.K, d.lda, BM)) return cudaErrorInvalidValue;
    if (!cached_tmap(&p.tmB, d.B, d.b_rows > 0 ? d.b_rows : d.N, d.K, d.ldb, BN)) return cudaErrorInvalidValue;
    p.M = d.M;
    p.N = d.N;
    p.K = d.K;
    p.num_m_tiles = (d.M + BM - 1) / BM;
    p.num_n_tiles = (d.N + BN - 1) / BN;
    p.num_k_blocks = (d.K + BK - 1) / BK;
    p.num_tiles = p.num_m_tiles * p.num_n_tiles;
    p.b2_row_off = d.b2_row_off;
    p.bias = reinterpret_cast<const __nv_bfloat16*>(d.bias);
    p.resid = d.resid;
    p.resid_f32 = d.resid_f32 ? 1 : 0;
    p.ldr = d.ldr;
    p.C = d.C;
    p.ldc = d.ldc;
    p.C32 = reinterpret_cast<float*>(d.C32);
    p.group_bounds = d.group_bounds;
    p.n_groups = d.n_groups;
    p.b_group_stride_rows = d.b_group_stride_rows;
    p.b_base_row = d.b_base_row;
    p.row_table = d.row_table;
    p.row_weight = d.row_weight;
    p.group_b_row = nullptr;
    if (d.group_b_row) {  // grouped only: B rows of some groups live in a second view
        if (!grouped || !d.B2 || d.b2_rows < 1 || (reinterpret_cast<uintptr_t>(d.B2) & 15) ||
            !cached_tmap(&p.tmB2, d.B2, d.b2_rows, d.K, d.ldb, BN))
            return cudaErrorInvalidValue;
        p.group_b_row = d.group_b_row;
    }
    p.err = d.err_word;
    p.mbar_limit_ns = MBAR_LIMIT_NS;
    p.pdl = d.pdl ? 1 : 0;
    p.splits = 1;
    int tiles = p.num_tiles;
    if (grouped) {
        // sum over groups of ceil(rows/BM) <= M/BM + n_groups
        tiles = (p.num_m_tiles + d.n_groups) * p.num_n_tiles;
        if (d.max_tiles_hint > 0 && d.max_tiles_hint < tiles) tiles = d.max_tiles_hint;
    }
    int sms = gemm_num_sms();
    int grid = max_ctas > 0 ? (max_ctas < sms ? max_ctas : sms) : sms;
    if (!grouped && d.M > BM) {
        // pair-CTA tiles of 256 rows; the choice depends only on the shape, so the
        // bits do not depend on the grid size
        const int bn2 = dual ? 256 : gemm_pair_tile_n(d.M, d.N);
        if (!cached_tmap(&p.tmA, d.A, d.a_rows > 0 ? d.a_rows : d.M, d.K, d.lda, 128) ||
            !cached_tmap(&p.tmB, d.B, d.b_rows > 0 ? d.b_rows : d.N, d.K, d.ldb, dual ? 128 : bn2 / 2))
            return cudaErrorInvalidValue;
        if (!dual) p.num_n_tiles = (d.N + bn2 - 1) / bn2;
        // output views for the bulk tensor stores (32x32 boxes; clipped at M and N)
        if (!cached_tmap(&p.tmC, MapSpec{d.C, d.M, d.N, d.ldc, 32, 32, 2, 64})) return cudaErrorInvalidValue;
        if (d.C32 && !cached_tmap(&p.tmC32, MapSpec{d.C32, d.M, d.N, d.ldc, 32, 32, 4, 128}))
            return cudaErrorInvalidValue;
        const int pair_tiles = ((d.M + 255) / 256) * p.num_n_tiles;
        int clusters = grid / 2;
        if (clusters > pair_tiles) clusters = pair_tiles;
        if (clusters < 1) clusters = 1;
        // every cluster with one tile: the residual epilogues' one-tile layout (more stages; the
        // same arithmetic, so the bits do not change with the grid)
        const bool one = pair_tiles <= clusters;
        switch (d.epi) {
            case EPI_STORE: return launch_t2_bn<EPI_STORE>(p, bn2, clusters, s);
            case EPI_BIAS_GELU: return launch_t2_bn<EPI_BIAS_GELU>(p, bn2, clusters, s);
            case EPI_BIAS_RESID:
                return one ? launch_t2_bn<EPI_BIAS_RESID, true>(p, bn2, clusters, s)
                           : launch_t2_bn<EPI_BIAS_RESID>(p, bn2, clusters, s);
            case EPI_RESID:
                return one ? launch_t2_bn<EPI_RESID, true>(p, bn2, clusters, s)
                           : launch_t2_bn<EPI_RESID>(p, bn2, clusters, s);
            case EPI_SWIGLU: return launch_t2<EPI_SWIGLU, true, 256>(p, clusters, s);
        }
        return cudaErrorInvalidValue;
    }
    // a small dense GEMM with few tiles: its K slices go to separate CTAs, and a reduction adds
    // their partial tiles in slice order and runs the epilogue
    const int splits = grouped || dual ? 1 : gemm_split_k(d.M, d.N, d.K, d.epi);
    if (splits > 1 && d.splitk_ws && d.splitk_ws_bytes >= gemm_split_ws_bytes(d.M, d.N, d.K, d.epi) &&
        !(reinterpret_cast<uintptr_t>(d.splitk_ws) & 15)) {
        GemmParams q = p;
        q.splits = splits;
        q.C = d.splitk_ws;
        q.ldc = d.N;
        q.C32 = nullptr;
        int g2 = grid < tiles * splits ? grid : tiles * splits;
        if (g2 < 1) g2 = 1;
        cudaError_t e = launch_t<EPI_PARTIAL, false, false>(q, g2, s);
        if (e != cudaSuccess) return e;
        switch (d.epi) {
            case EPI_STORE: return launch_splitk_reduce<EPI_STORE>(d.splitk_ws, splits, d, s);
            case EPI_BIAS_GELU: return launch_splitk_reduce<EPI_BIAS_GELU>(d.splitk_ws, splits, d, s);
            case EPI_BIAS_RESID: return launch_splitk_reduce<EPI_BIAS_RESID>(d.splitk_ws, splits, d, s);
            case EPI_RESID: return launch_splitk_reduce<EPI_RESID>(d.splitk_ws, splits, d, s);
        }
        return cudaErrorInvalidValue;
    }
    if (grid > tiles) grid = tiles;
    if (grid < 1) grid = 1;
    switch (d.epi) {
        case EPI_STORE:
            return grouped ? cudaErrorInvalidValue : launch_t<EPI_STORE, false, false>(p, grid, s);
        case EPI_BIAS_GELU:
            return grouped ? cudaErrorInvalidValue : launch_t<EPI_BIAS_GELU, false, false>(p, grid, s);
        case EPI_BIAS_RESID:
            return grouped ? cudaErrorInvalidValue : launch_t<EPI_BIAS_RESID, false, false>(p, grid, s);
        case EPI_RESID:
            return grouped ? cudaErrorInvalidValue : launch_t<EPI_RESID, false, false>(p, grid, s);
        case EPI_SWIGLU:
            return grouped ? launch_t<EPI_SWIGLU, true, true>(p, grid, s)
                           : launch_t<EPI_SWIGLU, true, false>(p, grid, s);
        case EPI_SCALE_F32:
            return grouped ? launch_t<EPI_SCALE_F32, false, true>(p, grid, s) : cudaErrorInvalidValue;
    }
    return cudaErrorInvalidValue;
}

}  // namespace ls
