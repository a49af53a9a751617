/*
 * libmoe: a B300 (sm_103a) MoE expert layer behind a plain C ABI.
 *
 * The layer is the one described in "Efficient MoE Training for Biological
 * Foundation Models" (NVIDIA Developer Blog): top-k routing, a permute of the
 * routed tokens into contiguous per-expert groups, a grouped FC1 GEMM
 * (gate and up projections, out_features = 2*intermediate_size), SwiGLU
 * scaled by the routing probabilities ("ScaledSwiGLU"), a grouped FC2
 * ("down") GEMM and the weighted combine, forward and backward, in BF16 and
 * in MXFP8 (E4M3 elements, one E8M0 scale per 32 consecutive values).
 *
 * Conventions for every call
 *  - All pointers are DEVICE pointers unless stated otherwise; the caller
 *    owns every buffer. The library never allocates device memory.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *    default stream) and never synchronise the host, except
 *    moe_device_error.
 *  - BF16 tensors are passed as void* and hold IEEE bfloat16 values,
 *    row-major with the stated leading dimension.
 *  - Arguments are checked on the host; a bad argument returns MOE_ERR_ARG
 *    and enqueues nothing. A failed launch returns MOE_ERR_CUDA.
 *  - Kernels that detect a bad value (an expert index out of range) or give
 *    up a bounded wait record a flag in a device error word instead of
 *    trapping; moe_device_error reads and clears it.
 *
 * Notation: T tokens, H hidden size, F FFN (intermediate) size, E experts,
 * k experts per token, R = T*k routed rows, R_pad = rows after padding each
 * expert group to a multiple of `align`.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

typedef struct CUstream_st* moe_stream_t;

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_ARG = 1,          /* invalid argument; nothing was enqueued */
  MOE_ERR_UNSUPPORTED = 2,  /* valid but not supported (shape or device) */
  MOE_ERR_CUDA = 3,         /* a CUDA runtime call failed */
  MOE_ERR_DEVICE = 4        /* the device error word was set */
};

/* Device error word flags (moe_device_error). */
#define MOE_DEVERR_BAD_INDEX 0x1u   /* an expert index outside [0, E), or a gathered row past its source */
#define MOE_DEVERR_TIMEOUT 0x2u     /* a bounded wait in a pipelined kernel gave up */
#define MOE_DEVERR_CAPACITY 0x4u    /* more padded rows than the buffer holds */
#define MOE_DEVERR_LAYOUT 0x8u      /* group offsets not aligned as the call requires */

/* Human-readable name of a status code. Static string; never NULL. */
MOE_API const char* moe_status_string(int status);

/* Synchronises `stream`, then reads and clears the device error word of the
 * current device. *flags (host pointer) receives the MOE_DEVERR_* bits.
 * Returns MOE_ERR_DEVICE when any bit was set, MOE_OK otherwise. */
MOE_API int moe_device_error(moe_stream_t stream, unsigned* flags);

/* moe_selftest_wait_timeout: a diagnostic of the failure detection above.
 * Launches one CTA in which two warps wait, with the bounded wait every
 * pipelined kernel of this library uses, on an mbarrier that nothing arrives
 * at. After the library's wait limit (2 s) the wait gives up, sets
 * MOE_DEVERR_TIMEOUT and the kernel returns; the context stays usable and a
 * following moe_device_error reports the bit. Nothing else is touched. */
MOE_API int moe_selftest_wait_timeout(moe_stream_t stream);

/* moe_selftest_tile_order: a host-side diagnostic of the grouped GEMMs' tile
 * scheduler; no GPU work. For one expert's grid of mtiles x ntiles output
 * tiles, writes the m-tile and n-tile that the kernels process as the expert's
 * local tile t (0 <= t < mtiles * ntiles) into mt[t] and nt[t] (host arrays).
 * The kernels run an expert's tiles in bands when neither operand fits in its
 * L2 share: band_rows is that share in operand rows of K elements, tile_m and
 * tile_n the operand rows one tile reads of A and of B, prefer_m the order of
 * an expert that is not banded (m-tiles fastest when non-zero), and
 * min_band_tiles the smallest band (the kernels pass two waves of tiles).
 * The grouped GEMMs pass band_rows = (32 MiB / element bytes) / K.
 * Returns MOE_ERR_ARG for non-positive sizes, a negative band_rows, null
 * arrays or a grid of 2^31 tiles or more. */
MOE_API int moe_selftest_tile_order(int mtiles, int ntiles, int tile_m, int tile_n,
                                    long long band_rows, int prefer_m, int min_band_tiles,
                                    int32_t* mt, int32_t* nt);

/* ------------------------------------------------------------------------
 * Routing. "How MoE Architecture Cuts Costs and Boosts Efficiency: Efficient
 * Training of Biological Foundation Models", the Router paragraph (top-K
 * routing); "Efficient MoE Training ...", §Challenge 1 (routing_weights).
 *
 * moe_route: for each token t, the k experts with the largest logits (ties
 * to the lower expert index; +0 and -0 are equal), in descending order, and
 * w[t, j] = softmax over those k logits.
 *   logits  [T, E] fp32, row-major.      idx [T, k] int32 (out).
 *   w       [T, k] fp32 (out).
 * Requires 1 <= k <= E <= 256, k <= 8, T >= 0. NaN logits give unspecified
 * (but in-range) indices.
 */
MOE_API int moe_route(const float* logits, int T, int E, int k, int32_t* idx, float* w,
              moe_stream_t stream);

/* moe_route_backward: gradient of the loss with respect to the logits.
 * dp holds partial sums of dL/dw: for routed row i = t*k + j the partials are
 * dp[row(i) * ld_dp + c], c = 0..n_part-1, with row(i) = dest[i] when dest is
 * not NULL and row(i) = i otherwise. They are summed in increasing c (a fixed
 * order, so the result is deterministic) into g_j, and
 *   dlogits[t, e] = w_j * (g_j - sum_i w_i g_i)  if e = idx[t, j],  else 0.
 *   w, idx [T, k] as produced by moe_route.   dlogits [T, E] fp32 (out).
 */
MOE_API int moe_route_backward(const float* dp, long long ld_dp, int n_part, const int32_t* dest,
                       const float* w, const int32_t* idx, int T, int E, int k,
                       float* dlogits, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Router projection and auxiliary load-balancing loss. "How MoE Architecture
 * Cuts Costs and Boosts Efficiency: ...", the Router paragraph (a score for
 * every expert per token; the top K are kept) and "Engineering Challenges of
 * Efficient Training" (an auxiliary load-balancing loss added to the
 * training objective penalises uneven expert load).
 *
 * moe_router_forward:
 *   logits[t, e] = sum_h x[t, h] * w_r[h, e]   (exact bf16 products summed in
 *                  fp32 on warp-level tensor-core MMAs; 128-column chunks of H
 *                  go to 8 warps whose sums are added in warp order, so the
 *                  result is deterministic)
 *   idx, w       = moe_route(logits, k)
 *   aux          = [L_aux, f_0..f_{E-1}, P_0..P_{E-1}] (fp32, 1 + 2E values) with
 *                  f_e = #{(t, j): idx[t, j] = e} / (T*k), P_e = mean over t of
 *                  softmax_e(logits[t, :]) over all E, L_aux = E * sum_e f_e * P_e
 *                  (1 for perfectly balanced routing).
 *   x [T, H] bf16 (16-byte aligned), w_r [H, E] bf16, logits [T, E] fp32 (out),
 *   idx [T, k] int32 and w [T, k] fp32 (out), aux (out).
 *   workspace: at least moe_router_workspace_size(T, H, E) bytes, 256-aligned.
 *   Requires H % 64 == 0, 1 <= k <= min(E, 8), E <= 256.
 *   Every sum over tokens is taken in a fixed order: results are
 *   deterministic.
 * moe_router_backward: given dlogits_route = dL/dlogits from the experts'
 * path (moe_route_backward; may be NULL) and the weight aux_coeff of L_aux in
 * the training loss,
 *   dlogits[t, e] = dlogits_route[t, e]
 *                   + aux_coeff * (E/T) * s[t, e] * (f_e - sum_i f_i * s[t, i])
 *   (s = softmax(logits[t, :]); the top-k selection has no gradient),
 *   dx_out[t, h]  = dx_in[t, h] + sum_e dlogits[t, e] * w_r[h, e]  (bf16;
 *                   dx_in may be NULL or equal dx_out, e.g. the experts' dX),
 *   dw_r[h, e]    = sum_t x[t, h] * dlogits[t, e]  (bf16).
 *   Both contractions run on warp-level bf16 MMAs with fp32 accumulation;
 *   dlogits enters them as two bf16 terms, hi = bf16(dl) and
 *   lo = bf16(dl - hi), about 16 significant bits (the dropped remainder is
 *   below 2^-16 |dl|). Token sums are taken in a fixed order.
 *   logits and aux as written by moe_router_forward; dlogits [T, E] fp32 (out;
 *   may be the same buffer as dlogits_route). w_r, dx_in and dx_out 16-byte
 *   aligned.
 */
MOE_API size_t moe_router_workspace_size(int T, int H, int E);
MOE_API int moe_router_forward(const void* x, const void* w_r, int T, int H, int E, int k,
                               float* logits, int32_t* idx, float* w, float* aux,
                               void* workspace, size_t workspace_bytes, moe_stream_t stream);
MOE_API int moe_router_backward(const void* x, const void* w_r, const float* logits,
                                const float* aux, const float* dlogits_route, float aux_coeff,
                                int T, int H, int E, float* dlogits, const void* dx_in,
                                void* dx_out, void* dw_r, void* workspace,
                                size_t workspace_bytes, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Expert sort: the per-expert token lists and split sizes of
 * "Efficient MoE Training ...", §Challenge 1, built as a stable counting
 * sort of the T*k routed rows by expert.
 *
 * moe_rows_padded_max: host-side upper bound on R_pad for any routing:
 *   T*k + E*(align-1). Needs no device access.
 * moe_permute_plan_workspace_size: bytes of device workspace that
 *   moe_permute_plan needs (a multiple of 256).
 *
 * moe_permute_plan:
 *   idx      [T, k] int32 expert of each routed row (input).
 *   counts   [E] int32 (out): rows routed to each expert (the split sizes).
 *   offsets  [E+1] int32 (out): exclusive prefix sum of counts rounded up to
 *            `align`; offsets[E] = R_pad. Expert e owns Xp rows
 *            [offsets[e], offsets[e+1]).
 *   dest     [T*k] int32 (out): Xp row of routed row i = t*k + j. Inside an
 *            expert group the rows keep increasing i (token, then slot).
 *   src      [src_rows] int32 (out): inverse of dest, -1 on padding rows and
 *            on every row at or beyond R_pad. src_rows must be at least
 *            moe_rows_padded_max(T, E, k, align).
 *   workspace, workspace_bytes: device scratch, at least
 *            moe_permute_plan_workspace_size(T, E, k) bytes, 256-aligned.
 * Requires 1 <= k <= E <= 1024, 1 <= align <= 4096, T*k < 2^31.
 * An index outside [0, E) sets MOE_DEVERR_BAD_INDEX and that row is dropped.
 */
MOE_API long long moe_rows_padded_max(int T, int E, int k, int align);
MOE_API size_t moe_permute_plan_workspace_size(int T, int E, int k);
MOE_API int moe_permute_plan(const int32_t* idx, int T, int E, int k, int align, int32_t* counts,
                     int32_t* offsets, int32_t* dest, int32_t* src, long long src_rows,
                     void* workspace, size_t workspace_bytes, moe_stream_t stream);

/* moe_permute_plan_static: moe_permute_plan for callers that cannot
 * allocate device memory (engines that give a plugin no workspace and forbid
 * allocation after start-up, or latency-critical loops that cannot afford
 * cudaMalloc's implicit device synchronisation). The sources have no
 * counterpart of this call; it exists only for such callers.
 *   Arguments and results are those of moe_permute_plan, without the
 *   workspace: the scratch is a fixed array of MOE_PLAN_STATIC_SCRATCH_INTS
 *   int32 (1 MiB) inside the library, held on every GPU that loads the
 *   library until the process exits. The caller still passes all inputs and
 *   outputs; nothing is allocated.
 *   Limit: ceil(T*k / 1024) * E <= MOE_PLAN_STATIC_SCRATCH_INTS, else
 *   MOE_ERR_UNSUPPORTED and nothing is enqueued.
 *   The first call on each device looks up the array's device address (with
 *   that device current) and keeps it; make that first call before any
 *   stream capture. The kept address does not survive cudaDeviceReset: do not
 *   call this entry point again in a process that reset the device.
 *   Each device holds its own copy of the array. Calls on the same device
 *   share it: calls that overlap on that GPU (other streams, threads) race
 *   and must be serialised by the caller. Each call overwrites the scratch it
 *   reads, so nothing carries over between calls.
 */
#define MOE_PLAN_STATIC_SCRATCH_INTS 262144
MOE_API int moe_permute_plan_static(const int32_t* idx, int T, int E, int k, int align,
                                    int32_t* counts, int32_t* offsets, int32_t* dest,
                                    int32_t* src, long long src_rows, moe_stream_t stream);

/* moe_permute: the gather that makes each expert's rows contiguous
 * ("Efficient MoE Training ...", §Challenge 1, GroupedLinear "gathering ...
 * input tokens"): xp[dest[t*k + j]] = x[t]; padding rows
 * [offsets[e] + counts[e], offsets[e+1]) are set to zero.
 *   x [T, H] bf16.  xp [R_pad, H] bf16 (out).
 *   w, p_rows: optional (both NULL or both set): p_rows[dest[i]] = w[i]
 *   (fp32 [R_pad], 0 on padding rows), the per-row routing weight used by
 *   the scaled-SwiGLU epilogue.
 *   xp may be NULL when p_rows is set: then only p_rows is written (the
 *   MXFP8 path gathers x inside mxfp8_quantize instead) and x is not read.
 * Requires H % 8 == 0 and 16-byte aligned x and xp. */
MOE_API int moe_permute(const void* x, const int32_t* dest, const int32_t* offsets,
                const int32_t* counts, const float* w, int T, int H, int E, int k, void* xp,
                float* p_rows, moe_stream_t stream);

/* moe_unpermute: the combine (index_add of "Efficient MoE Training ...",
 * §Challenge 1): out[t] = sum_{j<k} w[t, j] * y[dest[t*k + j]], accumulated
 * in fp32 in slot order j = 0..k-1 and rounded once to bf16. w = NULL means
 * all weights 1 (used when the weights were already applied, and for the
 * backward of moe_permute).
 *   y [R_pad, H] bf16.  out [T, H] bf16 (out).  Requires H % 8 == 0. */
MOE_API int moe_unpermute(const void* y, const int32_t* dest, const float* w, int T, int H, int k,
                  void* out, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * MXFP8 quantisation ("Efficient MoE Training ...", §Challenge 2: a scale
 * for each block of 32 consecutive values; OCP Microscaling Formats v1.0):
 * per block, e = clamp(floor(log2(max|v|)) - 8, -127, 127) (all-zero block:
 * -127), scale byte e + 127, element = E4M3(v * 2^-e) rounded to nearest
 * even and saturated to +-448; a block holding Inf or NaN gets scale 0xFF
 * and element bytes 0x7F.
 *
 * Scale layout (MXFP8 operand with MN rows and K columns, data [MN, K]
 * e4m3 with K contiguous): 512-byte tiles, one per 128 rows x 128 columns;
 * tile (i, j) starts at byte (i*(K/128) + j)*512, and inside it the scale of
 * row r = 32a + b (b < 32, a < 4) and 32-column block c (c < 4) is byte
 * 16b + 4a + c. This is the order in which tcgen05 block-scaled MMAs take
 * scales from tensor memory.
 *
 * mxfp8_quantize: input rows r = 0..rows-1 are read from in + row(r)*ld,
 * with row(r) = r when src is NULL, else row(r) = src[r] / src_div, and a
 * zero row when src[r] < 0 (this fuses moe_permute into the quantiser).
 *   dirs & 1 (row-wise, blocks along a row):  q_row [rows, cols] e4m3,
 *       s_row tiled with MN = rows, K = cols.
 *   dirs & 2 (column-wise, blocks of 32 rows, stored transposed):
 *       q_col [cols, rows] e4m3, s_col tiled with MN = cols, K = rows.
 * Requires rows % 128 == 0, cols % 128 == 0, ld >= cols, ld % 8 == 0. */
#define MOE_QUANT_ROWWISE 1
#define MOE_QUANT_COLWISE 2
MOE_API int mxfp8_quantize(const void* in, long long rows, int cols, long long ld, const int32_t* src,
                   int src_div, int dirs, uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                   uint8_t* s_col, moe_stream_t stream);

/* mxfp8_scales_to_canonical: the scales of an MXFP8 operand with MN rows and
 * K columns, given in the tiled layout above, rewritten row-major:
 * canon[r * (K/32) + c] = scale byte of row r and 32-column block c (the
 * plain [MN, K/32] E8M0 array of the OCP MX format, one byte per block of
 * 32 consecutive values, "Efficient MoE Training ...", §Challenge 2). For
 * tests and for handing scales to other software; the GEMMs read only the
 * tiled layout.
 *   tiled: mn*kdim/32 bytes (in).  canon: mn*kdim/32 bytes (out); the two
 *   must not overlap and both must be 4-byte aligned.
 *   Requires mn % 128 == 0 and kdim % 128 == 0 (mn == 0 does nothing). */
MOE_API int mxfp8_scales_to_canonical(const uint8_t* tiled, long long mn, int kdim,
                                      uint8_t* canon, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * MXFP4 activation compression (the hgpu.org abstract on MXFP4 training of
 * MoE models on Hopper: activations are kept in MXFP4 while the GEMMs run in
 * FP8; FP8 goes to FP4 and back without a BF16 round trip, and the
 * column-wise copy is derived from the row-wise one with new block scales).
 *
 * MXFP4 (OCP Microscaling v1.0): 32-element blocks, E8M0 scale byte
 * e + 127 with e = clamp(floor(log2(max|v|)) - 2, -127, 127) (all-zero
 * block: -127); E2M1 codes (sign bit 3; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6
 * for codes 0..7) = the nearest magnitude to |v| * 2^-e, ties to the even
 * code, saturating at 6; the sign is kept for zeros. A block holding Inf or
 * NaN gets scale 0xFF and codes 0. Two codes per byte, element 2i in the low
 * nibble: data [MN, K] is stored as [MN, K/2] bytes. Scales use the 512-byte
 * tiled layout of mxfp8_quantize (MN rows, K columns).
 *
 * Each conversion decodes its input exactly and applies the output format's
 * rule, so its result equals quantising the decoded values. Matrices are
 * [rows, cols] with row-wise blocks along cols; rows % 128 == 0,
 * cols % 128 == 0; data pointers 16-byte aligned. The caller owns every
 * buffer; nothing is allocated. MOE_ERR_ARG on a bad argument.
 *
 * mxfp4_from_mxfp8: row-wise MXFP8 (q8 [rows, cols] e4m3, s8) -> row-wise
 *   MXFP4 (q4 [rows, cols/2], s4) over the same blocks.
 * mxfp8_from_mxfp4: row-wise MXFP4 -> row-wise MXFP8 by the mxfp8_quantize
 *   rule (lossless: every MXFP4 value is an MXFP8 value).
 * mxfp4_rowwise_to_colwise: row-wise MXFP4 -> column-wise MXFP4 stored
 *   transposed (q4c [cols, rows/2], s4c tiled with MN = cols, K = rows):
 *   blocks of 32 rows, scales computed from the decoded values.
 * mxfp8_colwise_from_mxfp4_rowwise: the column-wise MXFP4 of the previous
 *   call, de-quantised to column-wise MXFP8 (q8c [cols, rows], s8c tiled
 *   with MN = cols, K = rows): the operand layout of an MXFP8 wgrad GEMM. */
MOE_API int mxfp4_from_mxfp8(const uint8_t* q8, const uint8_t* s8, long long rows, int cols,
                             uint8_t* q4, uint8_t* s4, moe_stream_t stream);
MOE_API int mxfp8_from_mxfp4(const uint8_t* q4, const uint8_t* s4, long long rows, int cols,
                             uint8_t* q8, uint8_t* s8, moe_stream_t stream);
MOE_API int mxfp4_rowwise_to_colwise(const uint8_t* q4, const uint8_t* s4, long long rows,
                                     int cols, uint8_t* q4c, uint8_t* s4c, moe_stream_t stream);
MOE_API int mxfp8_colwise_from_mxfp4_rowwise(const uint8_t* q4, const uint8_t* s4,
                                             long long rows, int cols, uint8_t* q8c,
                                             uint8_t* s8c, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Grouped GEMM on tcgen05 tensor cores: one launch for all experts, each with
 * its own weights and its own number of rows ("Efficient MoE Training ...",
 * §Challenge 1: GroupedLinear takes per-expert token counts, split_sizes, and
 * submits all local experts as one grouped operation).
 *
 * Groups: expert e owns rows [offsets[e], offsets[e+1]) of the row-indexed
 * operands; offsets is the device array written by moe_permute_plan.
 *
 * moe_grouped_gemm_bf16, mode MOE_GEMM_FPROP (forward and dgrad):
 *   C[r, n] = sum_k A[r, k] * B_e(k, n) for every row r of group e.
 *   A [rows, K] bf16, C [rows, N] bf16 (fp32 accumulation, one rounding).
 *   b_layout 0: B_e stored [K, N] at B + e*K*N (N contiguous).
 *   b_layout 1: B_e stored [N, K] at B + e*N*K (K contiguous), i.e. B_e^T.
 *   M is ignored. Requires N % 128 == 0, K % 64 == 0.
 * mode MOE_GEMM_WGRAD (weight gradients):
 *   C_e[m, n] = sum over rows r of group e of A[r, m] * B[r, n];
 *   C_e = C + e*M*N, [M, N] bf16. A [rows, M], B [rows, N] bf16.
 *   Experts with no rows get C_e = 0. Requires M % 128 == 0, N % 128 == 0,
 *   and every group size a multiple of 64 (else MOE_DEVERR_LAYOUT).
 * All of A, B, C 16-byte aligned; 1 <= E <= 256; rows < 2^31.
 *
 * Row gather (the permute-free operands of "Efficient MoE Training ...",
 * §Challenge 3: the fused path "avoids materializing some intermediate
 * results"): an operand whose rows are the permuted rows can instead be
 * read straight from its un-permuted source. With a moe_row_gather g, row r
 * of the operand is row g.src[r] / g.src_div of the source tensor (which has
 * g.src_rows rows and the operand's columns), and a zero row where
 * g.src[r] < 0 (padding). g.src is moe_permute_plan's src map (src_div = k),
 * at least `rows` entries. The source pointer is passed in place of the
 * operand, 16-byte aligned. Requires src_rows < 2^31, src_div >= 1. A source
 * row >= src_rows is read as a zero row and sets MOE_DEVERR_BAD_INDEX.
 * The gathered rows are copied into the GEMM's shared-memory stages by
 * 16-byte asynchronous copies, the other operand by TMA.
 */
#define MOE_GEMM_FPROP 0
#define MOE_GEMM_WGRAD 1
typedef struct moe_row_gather {
  const int32_t* src;  /* device, [rows]: flat routed index of each permuted row, -1 padding */
  int src_div;         /* source row = src[r] / src_div */
  long long src_rows;  /* rows of the source tensor */
} moe_row_gather;
/* ga, gb: optional gathers of A and B (NULL: the operand is stored permuted).
 * FPROP gathers only A (gb must be NULL); WGRAD may gather either operand. */
MOE_API int moe_grouped_gemm_bf16(int mode, const void* A, const void* B, int b_layout,
                                  const int32_t* offsets, int E, long long rows, int M, int N,
                                  int K, void* C, const moe_row_gather* ga,
                                  const moe_row_gather* gb, moe_stream_t stream);

/* moe_fc1_swiglu_bf16: the fused gate_up GroupedLinear + ScaledSwiGLU of
 * "Efficient MoE Training ...", §Challenge 3. For every row r of group e:
 *   [g | u] = xp[r] * W1_e  (W1_e stored [H, 2F], gate = columns [0, F)),
 *   gu[r] = [g | u] rounded to bf16 (kept for the backward),
 *   h[r, f] = silu(g_f) * u_f * p_rows[r]  (bf16), silu(z) = z / (1 + e^-z).
 *   xp [rows, H], w1 [E, H, 2F], gu [rows, 2F], h [rows, F] bf16;
 *   p_rows [rows] fp32 (moe_permute's per-row routing weight).
 *   gx: optional row gather of xp (xp is then the tokens x [src_rows, H]).
 * Requires H % 64 == 0, F % 64 == 0. */
MOE_API int moe_fc1_swiglu_bf16(const void* xp, const void* w1, const int32_t* offsets,
                                const float* p_rows, int E, long long rows, int H, int F,
                                void* gu, void* h, const moe_row_gather* gx, moe_stream_t stream);

/* moe_swiglu_bwd_parts: number of partial sums per row that
 * moe_fc2_dgrad_swiglu_bwd_bf16 writes to dp_part (0 if F is unsupported). */
MOE_API int moe_swiglu_bwd_parts(int F);

/* moe_fc2_dgrad_swiglu_bwd_bf16: the matching fused backward. For every row
 * r of group e: dH = dy2[r] * W2_e^T (W2_e stored [F, H]); with g, u from gu
 * and p = p_rows[r]: a = silu(g)*u, dA = dH*p,
 *   dy1[r] = [dA*u*silu'(g) | dA*silu(g)]  (bf16, [rows, 2F]),
 *   dp_part[r, c] = sum over the c-th block of F columns of dH*a (fp32),
 *   c < moe_swiglu_bwd_parts(F); sum them with moe_route_backward.
 * silu'(z) = s(z)*(1 + z*(1 - s(z))), s the logistic function.
 * gdy: optional row gather of dy2 (dy2 is then the upstream gradient
 * [src_rows, H] in token order).
 * Requires H % 64 == 0, F % 128 == 0. */
MOE_API int moe_fc2_dgrad_swiglu_bwd_bf16(const void* dy2, const void* w2,
                                          const int32_t* offsets, const float* p_rows,
                                          const void* gu, int E, long long rows, int H, int F,
                                          void* dy1, float* dp_part, const moe_row_gather* gdy,
                                          moe_stream_t stream);

/* ------------------------------------------------------------------------
 * MXFP8 grouped GEMMs on the block-scaled tcgen05 MMA ("Efficient MoE
 * Training ...", §Challenge 2: MXFP8 GEMMs on Blackwell's block-scaled
 * tensor-core instructions; §Challenge 3: the fused grouped MLP with
 * quantisation folded in). Every operand is an MXFP8 tensor as written by
 * mxfp8_quantize: E4M3 data [MN, K] with K contiguous and the tiled scale
 * layout, with 32-blocks along the reduction dimension K. Accumulation is
 * fp32; the result is the exact dot product of the dequantised operands up to
 * fp32 summation order.
 *
 * moe_grouped_gemm_mxfp8, mode MOE_GEMM_FPROP:
 *   C[r, n] = sum_k A[r, k] * B_e[n, k] for every row r of group e, with
 *   B_e[n, k] = B[e*b_row_stride + n, e*b_k_stride + k]: a row-wise copy of
 *   per-expert [N, K] weights uses (b_row_stride = N, b_k_stride = 0); a
 *   column-wise copy of per-expert [K, N] weights, stored [N, E*K], uses
 *   (0, K). A is [a_rows, a_cols = K], C [a_rows, N] bf16. N % 128 == 0
 *   (a tail of 128 columns past a multiple of 256 is masked), K % 128 == 0.
 * mode MOE_GEMM_WGRAD:
 *   C_e[m, n] = sum over rows r of group e of A[m, r] * B[n, r] with A
 *   [M, a_cols] and B [N, b_cols] the column-wise (transposed) copies,
 *   a_cols = b_cols = rows. C = E x [M, N] bf16. M % 128 == 0, N % 256 == 0.
 * All a_rows, a_cols, b_rows, b_cols are multiples of 128; group offsets
 * must be multiples of 128 (else MOE_DEVERR_LAYOUT). */
MOE_API int moe_grouped_gemm_mxfp8(int mode, const uint8_t* a, const uint8_t* sa,
                                   long long a_rows, long long a_cols, const uint8_t* b,
                                   const uint8_t* sb, long long b_rows, long long b_cols,
                                   long long b_row_stride, long long b_k_stride,
                                   const int32_t* offsets, int E, int M, int N, int K, void* C,
                                   moe_stream_t stream);

/* moe_fc1_swiglu_mxfp8: FC1 + ScaledSwiGLU + requantisation, MXFP8.
 *   xq, sx: row-wise MXFP8 of the permuted tokens [rows, H].
 *   w1t, sw1t: column-wise MXFP8 of W1 viewed as [E*H, 2F], i.e. data
 *   [2F, E*H] (blocks along H).
 *   For every row r of group e: [g | u] = x_r * W1_e (fp32),
 *   gu[r] = [g | u] in bf16, h = silu(g)*u*p_rows[r] (fp32), written as
 *   row-wise MXFP8 hq_row [rows, F] + sh_row and column-wise MXFP8 (blocks of
 *   32 rows, transposed) hq_col [F, rows] + sh_col. hq_col and sh_col may
 *   both be NULL: then no column-wise copy is computed or written.
 * Requires rows, H, F multiples of 128. */
MOE_API int moe_fc1_swiglu_mxfp8(const uint8_t* xq, const uint8_t* sx, long long rows, int H,
                                 const uint8_t* w1t, const uint8_t* sw1t, const int32_t* offsets,
                                 const float* p_rows, int E, int F, void* gu, uint8_t* hq_row,
                                 uint8_t* sh_row, uint8_t* hq_col, uint8_t* sh_col,
                                 moe_stream_t stream);

/* moe_fc2_dgrad_swiglu_bwd_mxfp8: FC2 dgrad + SwiGLU backward, MXFP8.
 *   dy2q, sdy2: row-wise MXFP8 of the permuted upstream gradient [rows, H].
 *   w2q, sw2: row-wise MXFP8 of W2 viewed as [E*F, H] (blocks along H).
 *   dH = dy2 * W2_e^T; with g, u from gu and p = p_rows[r]:
 *   dY1 = [dA*u*silu'(g) | dA*silu(g)] (dA = dH*p) written as row-wise MXFP8
 *   dy1q_row [rows, 2F] + sdy1_row and column-wise dy1q_col [2F, rows] +
 *   sdy1_col; dp_part [rows, 2*ceil(F/256)] fp32: partial sums of
 *   dH*silu(g)*u (their sum over c is dL/dp of the row).
 * Requires rows, H, F multiples of 128. */
MOE_API int moe_fc2_dgrad_swiglu_bwd_mxfp8(const uint8_t* dy2q, const uint8_t* sdy2,
                                           long long rows, int H, const uint8_t* w2q,
                                           const uint8_t* sw2, const int32_t* offsets,
                                           const float* p_rows, const void* gu, int E, int F,
                                           uint8_t* dy1q_row, uint8_t* sdy1_row,
                                           uint8_t* dy1q_col, uint8_t* sdy1_col, float* dp_part,
                                           moe_stream_t stream);

/* ------------------------------------------------------------------------
 * The whole layer ("Efficient MoE Training ...", §Challenge 1 per-expert
 * loop, §Challenge 3 fused gate_up -> ScaledSwiGLU -> down), forward and
 * backward, as one call each over a caller-owned device workspace that also
 * carries the state saved between the two calls.
 *
 * Forward:  out[t] = sum_j w[t,j] * (silu(x W1_e[:, :F]) * (x W1_e[:, F:])) W2_e,
 *           e = idx[t, j] from moe_route(logits).
 *   logits [T, E] fp32; x [T, H] bf16; w1 [E, H, 2F] bf16 (gate | up);
 *   w2 [E, F, H] bf16; out [T, H] bf16.
 * Backward: gradients of L = sum(out * dout):
 *   dx [T, H] bf16, dw1 [E, H, 2F] bf16, dw2 [E, F, H] bf16,
 *   dlogits [T, E] fp32 (through the top-k softmax weights only).
 *   Must follow moe_layer_forward with the same cfg, weights and workspace.
 * Precision:
 *   MOE_PRECISION_BF16: bf16 operands, fp32 accumulation; [g|u], H and the
 *     permuted activations are kept in bf16. The permuted copies of x and
 *     dOut are made by moe_permute rather than read through row gathers
 *     (moe_row_gather): a gathered GEMM operand costs one TMA request per
 *     four 128-byte rows, far more time than the copy.
 *   MOE_PRECISION_MXFP8 (§Challenge 2 and 3): x, W1, W2 and dOut are
 *     quantised to MXFP8 (the permutes of x and dOut are fused into their
 *     quantisation; both weights are quantised once per forward, row- and
 *     column-wise); the FC1 epilogue emits H and the FC2-dgrad epilogue emits
 *     dY1 as MXFP8 in both directions; every GEMM takes operands whose
 *     32-blocks run along its reduction dimension (row-wise for forward and
 *     dgrad, column-wise within an expert group for wgrad). [g|u] is kept in
 *     bf16 for the SwiGLU backward.
 *   MOE_PRECISION_MXFP8_ACT4 (the hgpu.org abstract on MXFP4 MoE training on
 *     Hopper: FP8 compute, activations kept in MXFP4): as MXFP8, except the
 *     two activations that the weight gradients need, X (gathered) and H,
 *     are carried from the forward to the backward only as row-wise MXFP4
 *     (parts MOE_PART_X4Q_ROW, MOE_PART_H4Q_ROW: half the bytes of one FP8
 *     copy), made directly from their row-wise MXFP8 copies
 *     (mxfp4_from_mxfp8). The backward rebuilds their column-wise MXFP8
 *     operands with mxfp8_colwise_from_mxfp4_rowwise before the two wgrad
 *     GEMMs, so dW1 and dW2 see X and H quantised FP8 -> FP4 -> column-wise
 *     FP4. The row-wise FP8 copies of X and H are dead after the forward, so
 *     in this mode the column-wise FP8 parts of X and H occupy the same bytes
 *     as their row-wise parts (moe_layer_workspace_part reports the same
 *     offsets): after the backward, those bytes hold the rebuilt column-wise
 *     copies. The forward writes no column-wise H. The workspace is therefore
 *     smaller than in MXFP8 mode by one FP8 copy of X and of H, less their
 *     MXFP4 copies.
 * Requirements: H % 128 == 0 (H % 256 == 0 for MXFP8), F % 128 == 0,
 * 1 <= k <= 8, k <= E <= 256, align a multiple of 128 (groups are padded with
 * zero rows). moe_layer_workspace_size returns 0 for an unsupported cfg. The
 * workspace must be 256-byte aligned.
 * moe_layer_workspace_part gives the byte offset and size of one saved
 * intermediate (MOE_PART_*) inside the workspace, for inspection; parts of
 * the other precision have size 0. R_max = T*k + E*(align-1), rounded up to
 * a multiple of 128 in MXFP8 mode. MXFP8 parts come in fours: data of the
 * row-wise copy [rows, cols], its tiled scales, data of the column-wise copy
 * [cols, rows] and its tiled scales (layouts as in mxfp8_quantize).
 */
#define MOE_PRECISION_BF16 0
#define MOE_PRECISION_MXFP8 1
#define MOE_PRECISION_MXFP8_ACT4 2
typedef struct moe_layer_config {
  int T, H, F, E, k;
  int align;
  int precision;
} moe_layer_config;

#define MOE_PART_IDX 0      /* int32 [T, k] */
#define MOE_PART_W 1        /* fp32 [T, k] */
#define MOE_PART_COUNTS 2   /* int32 [E] */
#define MOE_PART_OFFSETS 3  /* int32 [E + 1] */
#define MOE_PART_DEST 4     /* int32 [T * k] */
#define MOE_PART_SRC 5      /* int32 [R_max] */
#define MOE_PART_PROWS 7    /* fp32 [R_max]: routing weight of each permuted row */
#define MOE_PART_XP 8       /* bf16 [R_max, H] */
#define MOE_PART_GU 9       /* bf16 [R_max, 2F] */
#define MOE_PART_H 10       /* bf16 [R_max, F] */
#define MOE_PART_Y2 11      /* bf16 [R_max, H]: FC2 output */
#define MOE_PART_DY2 12     /* bf16 [R_max, H]: dOut gathered (BF16 mode) */
#define MOE_PART_DY1 13     /* bf16 [R_max, 2F]: [dg | du] (BF16 mode) */
#define MOE_PART_DXP 14     /* bf16 [R_max, H]: FC1 dgrad output */
#define MOE_PART_DP 15      /* fp32 [R_max, n_part]: partial sums of dL/dw per row */
#define MOE_PART_XQ_ROW 16  /* MXFP8 x gathered: [R_max, H] (+ 17, 18, 19) */
#define MOE_PART_W1Q_ROW 20 /* MXFP8 W1 viewed [E*H, 2F] (+ 21, 22, 23) */
#define MOE_PART_W2Q_ROW 24 /* MXFP8 W2 viewed [E*F, H] (+ 25, 26, 27) */
#define MOE_PART_HQ_ROW 28  /* MXFP8 H: [R_max, F] (+ 29, 30, 31) */
#define MOE_PART_DY2Q_ROW 32 /* MXFP8 dOut gathered: [R_max, H] (+ 33, 34, 35) */
#define MOE_PART_DY1Q_ROW 36 /* MXFP8 dY1: [R_max, 2F] (+ 37, 38, 39) */
#define MOE_PART_DY1S_COL 39
#define MOE_PART_X4Q_ROW 40 /* MXFP8_ACT4: MXFP4 x gathered [R_max, H/2] bytes (+ 41: scales) */
#define MOE_PART_H4Q_ROW 42 /* MXFP8_ACT4: MXFP4 H [R_max, F/2] bytes (+ 43: scales) */

MOE_API size_t moe_layer_workspace_size(const moe_layer_config* cfg);
MOE_API int moe_layer_workspace_part(const moe_layer_config* cfg, int part, size_t* offset,
                                     size_t* bytes);
MOE_API int moe_layer_forward(const moe_layer_config* cfg, const float* logits, const void* x,
                              const void* w1, const void* w2, void* out, void* workspace,
                              size_t workspace_bytes, moe_stream_t stream);
MOE_API int moe_layer_backward(const moe_layer_config* cfg, const void* dout, const void* w1,
                               const void* w2, void* dx, void* dw1, void* dw2, float* dlogits,
                               void* workspace, size_t workspace_bytes, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
