// Internal kernel launchers of the layer-streaming library (not part of the C ABI).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace ls {

// ---------------------------------------------------------------- copy path
struct CopyRange {
    const void* src;      // device-visible address of mapped pinned host memory
    int64_t dst_off;      // byte offset inside the destination slot
    int64_t n16;          // whole 16-byte units
    int64_t chunk_begin;  // first chunk index of this range in the launch
    int32_t tail;         // trailing bytes (< 16)
    int32_t pad;
};
int64_t copy_chunks_for(int64_t n16);
cudaError_t launch_copy_h2slot(const CopyRange* ranges_dev, int n_ranges, int64_t n_chunks,
                               void* dst_base, const uint8_t* group_mask_dev, int ranges_per_group, uint32_t* ready,
                               uint32_t* ticket, uint32_t epoch, bool publish, int ctas,
                               cudaStream_t s);
cudaError_t launch_publish(uint32_t* ready, uint32_t epoch, bool publish, cudaStream_t s,
                           bool stream_op = true, bool capturing = false);
// early_dependents: let the next kernel be placed while this one waits - only when the
// awaited copy needs no SM (copy engine + stream-operation publish).
cudaError_t launch_wait_ready(const uint32_t* ready, uint32_t epoch, uint64_t limit_ns,
                              uint32_t* err_word, uint32_t code, cudaStream_t s, bool early_dependents = false);
// True when a publish after a copy-engine load is a stream memory operation (no SM).
bool publish_needs_no_sm();
// Asks, on the current device, for the largest shared-memory carveout for the copy and wait
// kernels (called once per context, outside any stream capture; a hint, errors ignored).
void prepare_copy_kernels();

// ---------------------------------------------------------------- fp32 linear + GELU
cudaError_t launch_linear_gelu_f32(const float* x, const float* w, const float* b, float* y, int T,
                                   int H, int F, cudaStream_t s, bool pdl = true);

// ---------------------------------------------------------------- tcgen05 GEMM
enum GemmEpilogue : int {
    EPI_STORE = 0,      // C = acc                          -> bf16
    EPI_BIAS_GELU = 1,  // C = GELU(acc + bias)             -> bf16
    EPI_BIAS_RESID = 2, // C = acc + bias + R               -> bf16
    EPI_SWIGLU = 3,     // dual B: C = SiLU(acc_g) * acc_u  -> bf16
    EPI_RESID = 4,      // C = acc + R                      -> bf16
    EPI_SCALE_F32 = 5,  // grouped: Y[row_table[i]] = w[row_table[i]] * acc -> fp32
    EPI_PARTIAL = 6,    // internal (split K): the fp32 accumulator of one K slice, as is
};

struct GemmDesc {
    int epi = EPI_STORE;
    // A: [M, K] bf16 row-major (lda elements); B: [rows, K] bf16 row-major (ldb elements)
    const void* A = nullptr;
    int64_t lda = 0;
    int64_t a_rows = 0;          // rows addressable through A (>= M)
    const void* B = nullptr;
    int64_t ldb = 0;
    int64_t b_rows = 0;          // rows addressable through B
    int M = 0, N = 0, K = 0;
    int b2_row_off = 0;          // dual: second B matrix starts this many rows after the first
    const void* bias = nullptr;  // [N] bf16
    const void* resid = nullptr; // [M, ldr] bf16 (fp32 with resid_f32)
    bool resid_f32 = false;
    int64_t ldr = 0;
    void* C = nullptr;
    int64_t ldc = 0;
    void* C32 = nullptr;         // residual epilogues: optional fp32 copy of C (ldc)
    // grouped (expert) mode: M is the total row count; groups split it
    const int* group_bounds = nullptr;  // [n_groups + 1], device
    int n_groups = 0;
    int b_group_stride_rows = 0;        // B rows between consecutive groups' matrices
    int b_base_row = 0;                 // B row of group 0's matrix
    const int* row_table = nullptr;     // EPI_SCALE_F32: destination row of sorted row i
    const float* row_weight = nullptr;  // EPI_SCALE_F32: weight by destination row
    int max_tiles_hint = 0;             // grouped: upper bound of tiles (grid sizing)
    // grouped, optional: group g's matrix starts at B row group_b_row[g] (device, [n_groups]);
    // with the top bit set, at row (group_b_row[g] & 0x7fffffff) of B2 [b2_rows, K] instead
    // (same ldb): experts read in place from the expert cache
    const int* group_b_row = nullptr;
    const void* B2 = nullptr;
    int64_t b2_rows = 0;
    // dense GEMMs with M <= 128 and few tiles (see gemm_split_k): fp32 workspace for the K
    // slices' partial tiles; without one (or too small) the GEMM runs unsplit
    float* splitk_ws = nullptr;
    int64_t splitk_ws_bytes = 0;
    uint32_t* err_word = nullptr;       // mapped host word for internal timeouts
    // programmatic dependent launch: the prologue overlaps the previous kernel's tail.
    // Off where events bracket each launch, so that an event pair times this kernel alone.
    bool pdl = true;
};

// max_ctas <= 0: one CTA per SM.
cudaError_t launch_gemm_bf16(const GemmDesc& d, int max_ctas, cudaStream_t s);
int gemm_num_sms();
// Tile width (output columns) of the dense pair-CTA GEMM for an M x N output.
int gemm_pair_tile_n(int64_t M, int64_t N);
// K slices of a dense single-CTA GEMM (M <= 128, not the gate/up pair): 1 when it is not split.
// A function of the shape and the device only, so the bits do not depend on the grid.
int gemm_split_k(int64_t M, int64_t N, int64_t K, int epi);
// Workspace bytes the split needs (0 when not split); at most GEMM_SPLITK_WS_MAX.
int64_t gemm_split_ws_bytes(int64_t M, int64_t N, int64_t K, int epi);
int64_t gemm_split_ws_max();

// ---------------------------------------------------------------- MoE
cudaError_t launch_moe_route(const float* logits, int n_layers, int T, int E, int k, int* sel,
                             float* weight, cudaStream_t s);
// expert_mask (may be NULL): [n_layers, E]; rows of masked-out experts are left out of the table.
cudaError_t launch_moe_group(const int* sel, int n_layers, int T, int E, int k, int* row_table,
                             int* group_bounds, uint8_t* expert_used, cudaStream_t s,
                             const uint8_t* expert_mask = nullptr);
// Row hand-off: dst[dst_table ? dst_table[i] : i] = src[src_table ? src_table[i] : i] (fp32 rows
// of H); with ready, the last CTA publishes ready[0] = epoch after a system fence.
cudaError_t launch_moe_rows_copy(const float* src, const int* src_table, float* dst, const int* dst_table, int rows,
                                 int H, uint32_t* ready, uint32_t* ticket, uint32_t epoch, int ctas, cudaStream_t s);
cudaError_t launch_moe_gather(const void* x, const int* row_table, int rows, int k, int H,
                              void* x_sorted, cudaStream_t s);
// out = x + sum_j y[t*k+j]; x bf16 (or fp32 with x_f32); out bf16, plus out32 fp32 if given
cudaError_t launch_moe_combine(const void* x, bool x_f32, const float* y, int T, int k, int H, void* out,
                               float* out32, cudaStream_t s);

// ---------------------------------------------------------------- debug checks
// Canaries: `count` regions of CANARY_BYTES at base, base + stride, ...; fill writes the
// pattern, check compares it and raises DERR_BOUNDS | (region0 + r) << 8 on a mismatch.
constexpr int64_t CANARY_BYTES = 256;
cudaError_t launch_canary(void* base, int64_t stride, int count, bool check, uint32_t* err_word,
                          uint32_t region0, cudaStream_t s);
// Validates a MoE routing of n_layers layers (sel [L, T*k], row_table [L, T*k], bounds
// [L, E+1]): bounds start at 0, end at T*k and never decrease; the rows of group e are
// the rows routed to expert e, in increasing order, so the table is a permutation of
// 0..T*k-1. Reads only inside those arrays. Raises DERR_BOUNDS | (region0 + layer) << 8.
cudaError_t launch_moe_check(const int* sel, const int* row_table, const int* bounds, int n_layers, int T,
                             int k, int E, uint32_t* err_word, uint32_t region0, cudaStream_t s);

}  // namespace ls
