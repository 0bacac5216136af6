/*
 * ls_kernels.h — the library's device kernels as standalone C entry points.
 *
 * ls_run drives these kernels itself; these entry points exist so that each
 * kernel can be checked and timed alone, in the launch configuration ls_run
 * uses. All pointers named *_dev are device memory on the current device;
 * `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 * Calls are asynchronous: they return once the work is queued. Return values
 * are ls_status codes from ls_api.h (LS_ERR_INVALID_ARG for shapes or
 * alignments a kernel does not handle, LS_ERR_CUDA for a failed launch).
 * A bounded wait that expires inside a kernel sets the library's device error
 * word, read and cleared with lsk_device_error().
 */
#ifndef LS_KERNELS_H
#define LS_KERNELS_H

#include <stdint.h>

#include "ls_api.h"

#ifdef __cplusplus
extern "C" {
#endif

/* GEMM epilogues (C[M,N] = A[M,K] B[N,K]^T, fp32 accumulation, bf16 operands). */
enum {
    LSK_EPI_STORE = 0,      /* C = acc -> bf16 */
    LSK_EPI_BIAS_GELU = 1,  /* C = GELU(acc + bias) -> bf16; GELU(z) = z Phi(z) */
    LSK_EPI_BIAS_RESID = 2, /* C = acc + bias + R -> bf16 */
    LSK_EPI_SWIGLU = 3,     /* two B matrices (rows b2_row_off apart): C = SiLU(A Bg^T) * (A Bu^T) -> bf16 */
    LSK_EPI_RESID = 4,      /* C = acc + R -> bf16 */
    LSK_EPI_SCALE_F32 = 5   /* grouped only: C[row_table[i]] = row_weight[row_table[i]] * acc -> fp32 */
};

/* Number of SMs of the current device (the default CTA count of the GEMMs). */
int32_t lsk_num_sms(void);

/* Read and clear the device error word of the standalone entry points (0 = none). */
uint32_t lsk_device_error(void);

/* Host-to-device copy with the copy kernel (16-byte loads of mapped pinned host
 * memory), then ready_dev[0] = epoch after a system fence, raised by the last CTA.
 * src_host must be pinned (page-locked and mapped) and 16-byte aligned; dst_dev
 * 16-byte aligned. ticket_dev: one zeroed uint32 the CTAs count on (left at 0).
 * ctas <= 0: one per SM. "layer split: overlap the stages' hand-off" (publish
 * order); "prefill: a layer split's idle card streams a share of a one-chunk
 * prompt's experts", What (16-byte copy kernel). */
ls_status lsk_copy_h2slot(void* dst_dev, const void* src_host, uint64_t bytes, int32_t ctas,
                          uint32_t* ready_dev, uint32_t* ticket_dev, uint32_t epoch, void* stream);

/* lsk_copy_h2slot for callers that cannot allocate device memory: callers
 * whose device memory is all owned by another allocator (a framework's caching
 * pool holding the card), and latency-critical loops that must not call
 * cudaMalloc/cudaFree because those can synchronise the device. The pages have
 * no counterpart of this call; it is an interface convenience of this library.
 *
 * It copies n_ranges host ranges (src_hosts[i], bytes[i]) to dst_dev +
 * dst_offsets[i] with the same copy kernel, then raises ready_dev[0] = epoch
 * after a system fence (last CTA). It allocates nothing: the range table and the
 * CTAs' ticket word live in a fixed device array of LSK_STATIC_SCRATCH_BYTES
 * bytes, defined in the library, that every device which loads the library
 * holds until the process exits.
 *   - n_ranges must be 1..LSK_STATIC_MAX_RANGES; more returns LS_ERR_INVALID_ARG
 *     before any work is queued.
 *   - Sources must be pinned and mapped, sources, dst_dev and the offsets
 *     16-byte aligned (LS_ERR_INVALID_ARG otherwise).
 *   - The first call on a device, and the first after that device's context has
 *     been replaced (cudaDeviceReset), looks up the array's device address with
 *     that device current (cudaGetSymbolAddress).
 *   - A call whose stream is being captured into a CUDA graph returns
 *     LS_ERR_INVALID_ARG before any work is queued: the range table is staged
 *     from the call's own stack frame, which a replay would read again long after
 *     the call has returned.
 *   - Every call shares the one array per device and each call overwrites it
 *     (the ticket is cleared by the call itself). Calls whose work overlaps on
 *     the GPU (different streams, no ordering between them) race on the array.
 *   - The range table is copied from a host array on `stream` as pageable
 *     memory; the call returns once that copy has been staged. */
#define LSK_STATIC_MAX_RANGES 64
#define LSK_STATIC_SCRATCH_BYTES (256 + 64 * 40)
ls_status lsk_copy_h2slot_static(void* dst_dev, const void* const* src_hosts, const uint64_t* bytes,
                                 const uint64_t* dst_offsets, int32_t n_ranges, int32_t ctas, uint32_t* ready_dev,
                                 uint32_t epoch, void* stream);

/* One thread waits until ready_dev[0] == epoch, at most limit_ms; on expiry it
 * writes err_host[0] (pinned, mapped host memory) = 1 | (slot << 8) and returns. */
ls_status lsk_wait_ready(const uint32_t* ready_dev, uint32_t epoch, int32_t limit_ms, uint32_t* err_host,
                         int32_t slot, void* stream);

/* Dense tcgen05 GEMM with a fused epilogue. A_dev [M,K], B_dev [b_rows,K] (b_rows
 * >= N, or >= b2_row_off + N for SWIGLU), bias [N], R [M,N], C [M,N]; bf16
 * row-major, dense, except R, which is fp32 when resid_f32 != 0. The residual
 * epilogues also write the fp32 result to C32_dev [M,N] when it is not NULL.
 * K and N multiples of 8, pointers 16-byte aligned. max_ctas <= 0: one CTA per SM.
 * A small GEMM (M <= 128, not SWIGLU) whose 256-column tiles leave SMs idle is split along
 * K: the slices' fp32 partial tiles go to a workspace this call takes on `stream` from a
 * memory pool of the library's own, which keeps freed blocks for later calls (stream-ordered,
 * at most one 128 x 256 fp32 tile per SM; LS_ERR_OOM if refused), and a reduction adds them
 * in slice order before the epilogue. The slice count depends only on
 * the shape and the device, so the bits do not depend on max_ctas. */
ls_status lsk_gemm_bf16(int32_t epilogue, const void* A_dev, const void* B_dev, int64_t b_rows,
                        int32_t b2_row_off, const void* bias_dev, const void* resid_dev, int32_t resid_f32,
                        void* C_dev, void* C32_dev, int32_t M, int32_t N, int32_t K, int32_t max_ctas,
                        void* stream);

/* Output columns of one tile of lsk_gemm_bf16 for this shape on the current device:
 * the pair-CTA GEMM (M > 128, not SWIGLU) takes 256 x W tiles, W in {256, 224, 192,
 * 160}: the fewest waves of tiles over all of the device's CTA pairs, then the
 * narrowest tile (a k-block's time is modelled as W + 1024 columns, most of it
 * independent of W); SWIGLU tiles cover 128 columns of each
 * matrix, the single-CTA GEMM (M <= 128) 256 columns. Depends only on the shape and
 * the device, not on max_ctas. Returns 0 for an invalid epilogue or shape. */
int32_t lsk_gemm_tile_n(int32_t epilogue, int32_t M, int32_t N);

/* Grouped (expert) GEMM: rows of A_dev [M,K] are sorted by group;
 * group g = rows [group_bounds[g], group_bounds[g+1]) multiplies B rows
 * starting at b_base_row + g * b_group_stride_rows (SWIGLU: second matrix
 * b2_row_off rows further). Epilogue SWIGLU (C bf16 [M,N], sorted rows) or
 * SCALE_F32 (C fp32 [*,N] scattered through row_table with row_weight). */
ls_status lsk_gemm_grouped_bf16(int32_t epilogue, const void* A_dev, const void* B_dev, int64_t b_rows,
                                int32_t b_base_row, int32_t b_group_stride_rows, int32_t b2_row_off,
                                const int32_t* group_bounds_dev, int32_t n_groups,
                                const int32_t* row_table_dev, const float* row_weight_dev, void* C_dev,
                                int32_t M, int32_t N, int32_t K, int32_t max_ctas, void* stream);

/* y[T,F] = GELU(x[T,H] W[F,H]^T + b[F]), fp32. */
ls_status lsk_linear_gelu_f32(const float* x_dev, const float* w_dev, const float* b_dev, float* y_dev,
                              int32_t T, int32_t H, int32_t F, void* stream);

/* Routing of n_layers x T tokens: sel [n_layers,T,k] = top-k expert ids of the
 * fp32 logits [n_layers,T,E] (larger first, ties to the lower index); weight =
 * softmax over the k chosen logits (fp32). E <= 256, k <= 8. */
ls_status lsk_moe_route(const float* logits_dev, int32_t n_layers, int32_t T, int32_t E, int32_t k,
                        int32_t* sel_dev, float* weight_dev, void* stream);

/* Per layer: stable counting sort of the rows t*k+j by expert -> row_table
 * [n_layers, T*k], group_bounds [n_layers, E+1], expert_used [n_layers, E]
 * (may be NULL). */
ls_status lsk_moe_group(const int32_t* sel_dev, int32_t n_layers, int32_t T, int32_t E, int32_t k,
                        int32_t* row_table_dev, int32_t* group_bounds_dev, uint8_t* expert_used_dev,
                        void* stream);

/* lsk_moe_group over a subset of the experts: expert_mask_dev [n_layers, E] (1 = keep);
 * rows routed to a masked-out expert are left out, so row_table holds only the kept rows,
 * still grouped by expert in (token, k) order, and group_bounds[E] is their count. The
 * split of a layer between the active card and the idle-stage helper (see
 * ls_helper_split): each card groups the rows of its own experts. */
ls_status lsk_moe_group_masked(const int32_t* sel_dev, int32_t n_layers, int32_t T, int32_t E, int32_t k,
                               const uint8_t* expert_mask_dev, int32_t* row_table_dev, int32_t* group_bounds_dev,
                               uint8_t* expert_used_dev, void* stream);

/* Hand-off of fp32 result rows (H floats each, H % 4 == 0): for i < rows,
 * dst[dst_table ? dst_table[i] : i] = src[src_table ? src_table[i] : i], with 16-byte
 * loads and stores ("prefill: a layer split's idle card streams a share of a one-chunk
 * prompt's experts", What: result rows go through mapped host memory and are read by
 * copy kernels on the device that needs them). src and dst are device memory or pinned,
 * mapped host memory (host pointers are translated); tables are device int32 arrays or
 * NULL. With ready_dev, the last CTA raises ready_dev[0] = epoch after a system fence
 * (ticket_dev: one zeroed uint32, left at 0), so a reader can lsk_wait_ready on it.
 * ctas <= 0: one per SM. */
ls_status lsk_moe_rows_copy(const float* src, const int32_t* src_table, float* dst, const int32_t* dst_table,
                            int32_t rows, int32_t H, uint32_t* ready_dev, uint32_t* ticket_dev, uint32_t epoch,
                            int32_t ctas, void* stream);

/* x_sorted[i] = x[row_table[i] / k] for i < rows; bf16 rows of H (H % 8 == 0). */
ls_status lsk_moe_gather(const void* x_dev, const int32_t* row_table_dev, int32_t rows, int32_t k, int32_t H,
                         void* x_sorted_dev, void* stream);

/* out[t] = x[t] + sum_{j<k} y[t*k + j] (fp32 sum in j order, one bf16 rounding), 1 <= k <= 8.
 * x is bf16, or fp32 when x_f32 != 0; out32_dev (may be NULL) gets the fp32 sum. */
ls_status lsk_moe_combine(const void* x_dev, int32_t x_f32, const float* y_dev, int32_t T, int32_t k, int32_t H,
                          void* out_dev, float* out32_dev, void* stream);

/* The routing check of params.debug_checks (no counterpart on the pages; it stands in for
 * a memory sanitizer). For n_layers layers of a MoE routing - sel_dev [L, T*k] int32 (the
 * expert of row t*k + j), row_table_dev [L, T*k] int32 and group_bounds_dev [L, E+1] int32
 * as lsk_moe_group writes them - it checks that the bounds run from 0 to T*k without
 * decreasing and that group e holds exactly the rows routed to expert e, in increasing
 * order. It only reads the three arrays; an invalid layer sets err_host[0] (pinned, mapped
 * host memory) = 4 | ((0x20000 + layer) << 8) if it is still 0. Returns LS_OK once
 * queued; the outcome is in err_host after the stream drains. */
ls_status lsk_moe_check(const int32_t* sel_dev, const int32_t* row_table_dev, const int32_t* group_bounds_dev,
                        int32_t n_layers, int32_t T, int32_t k, int32_t E, uint32_t* err_host, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* LS_KERNELS_H */
