/*
 * mm_moe.h -- C ABI of the GB300 (sm_103a) MoE routing / permute / MXFP8
 * expert-FFN library (libmm_moe.so).
 *
 * Operations and the pages that define them:
 *   mm_moe_init_routing   MoeInitRoutingV3 (CANN ops-transformer,
 *                         moe/moe_init_routing_v3): "计算公式" steps 1-3 and 5,
 *                         parameter table (quantMode, expertTokensNumType,
 *                         rowIdxType, expandedScaleOut).
 *   mm_moe_token_permute  moe_token_permute article ("CANN ops-transformer 的
 *                         moe_token_permute 算子"): sections 功能说明,
 *                         参数说明, 返回值说明, 约束说明.
 *   mm_mega_moe           MegaMoE README (ops-transformer, mc2/mega_moe):
 *                         "A8W8-FP quantization scenario" stages 1-4,
 *                         "Activation function formulas" (swiglu), parameter
 *                         table and the MXFP constraints on weight shapes;
 *                         run at epWorldSize = 1, so dispatch and combine are
 *                         a local permute and a local weighted sum.
 *   mm_mx_quantize        the Q_MX operation of the same README (group 32,
 *                         shared E8M0 exponent, FP8 elements).
 *
 * Conventions shared by every entry point
 *   Memory     every pointer is a device pointer unless stated otherwise.
 *              The caller owns every buffer; the library allocates no device
 *              memory.  Entry points that need scratch memory say how much
 *              through a *_workspace_size query; the caller passes a device
 *              buffer of at least that many bytes, 256-byte aligned.
 *   Streams    `stream` is a cudaStream_t (NULL = legacy default stream).
 *              All work is enqueued asynchronously on it; the call returns
 *              before the GPU finishes.  Calls on one stream may reuse one
 *              workspace; concurrent calls need separate workspaces.
 *   Errors     the return value is checked before anything is enqueued:
 *              invalid shapes or codes give MM_ERR_INVALID_ARG, valid but
 *              unimplemented options MM_ERR_UNSUPPORTED, a short workspace
 *              MM_ERR_WORKSPACE (nothing is truncated silently), a failed
 *              CUDA call MM_ERR_CUDA.  Data-dependent problems found on the
 *              GPU are OR-ed as MM_DEVERR_* bits into *dev_err (an int32 in
 *              device memory, may be NULL); kernels never trap.
 *   Flatten    the expanded row j of token i and choice k is j = i*K + k
 *              (row-major flatten of the [N, K] index matrix).
 *   Layouts    all matrices are row-major and dense.
 */
#ifndef MM_MOE_H_
#define MM_MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MM_OK = 0,
  MM_ERR_INVALID_ARG = 1,
  MM_ERR_UNSUPPORTED = 2,
  MM_ERR_WORKSPACE = 3,
  MM_ERR_CUDA = 4
} mm_status;

/* Bits OR-ed into *dev_err by the kernels. */
#define MM_DEVERR_EXPERT_RANGE 1 /* an expert id outside [0, expert_num): row left out */
#define MM_DEVERR_DUPLICATE_ID 2 /* a token lists one expert twice (MegaMoE forbids it) */
#define MM_DEVERR_TIMEOUT 4      /* a bounded wait inside a kernel gave up */
#define MM_DEVERR_BOUNDS 8       /* checked build only (mm_checked_build): an index computed on
                                    the GPU fell outside the buffer it addresses; that access
                                    was skipped */

/* Element type codes.  The FP8 / FP4 codes are the MegaMoE dtype codes
 * (dispatchQuantOutDtype: 23 = FLOAT8_E5M2, 24 = FLOAT8_E4M3FN,
 * 296 = FLOAT4_E2M1).  FLOAT4_E2M1 arrays here are packed two codes per
 * byte along the contiguous dimension, element 2i in bits 0-3 and element
 * 2i+1 in bits 4-7 (the pages store them in Ascend's FRACTAL_NZ_C0_32
 * format instead). */
#define MM_DT_FLOAT32 0
#define MM_DT_FLOAT16 1
#define MM_DT_INT32 3
#define MM_DT_INT64 9
#define MM_DT_FP8_E5M2 23
#define MM_DT_FP8_E4M3FN 24
#define MM_DT_BFLOAT16 27
#define MM_DT_FP4_E2M1 296

/* Quant-mode codes of moe_token_permute and MoeInitRoutingV3:
 * -1 none, 2 MXFP8 E5M2, 3 MXFP8 E4M3FN; 9 MXFP4 E2M1 (moe_token_permute only). */
#define MM_QUANT_NONE (-1)
#define MM_QUANT_MXFP8_E5M2 2
#define MM_QUANT_MXFP8_E4M3FN 3
#define MM_QUANT_MXFP4_E2M1 9

/* Layouts of the E8M0 weight scales passed to mm_mega_moe. */
#define MM_WSCALE_ROWS 0     /* the pages' (E, N_out, CeilDiv(K_red, 64), 2) */
#define MM_WSCALE_PREPARED 1 /* output of mm_prepare_weight_scales */

/* Human-readable name of a status code (static string). */
const char* mm_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int mm_version(void);

/* ------------------------------------------------------------------------
 * mm_moe_init_routing -- MoeInitRoutingV3, Dropless, active expert range
 * [0, expert_num), quantMode -1 / 2 / 3 / 9 (another range, and the key_value
 * count type: mm_moe_init_routing_v3 below).
 *
 *   sortedRowIdx          = keyValueSort(expertIdx, rowIdx)      (step 1)
 *   expandedRowIdx[sortedRowIdx[d]] = d                           (step 2)
 *   expert_tokens         = histogram of the sorted ids           (step 3)
 *   expandedX[d]          = Q(x[sortedRowIdx[d] / K])             (step 5)
 * Ties in the sort keep ascending j (a stable sort), so rows of one expert
 * are in ascending token order.
 *
 * x                 [num_rows, h] of x_dtype (bf16 / fp16 / fp32; quantised
 *                   modes take bf16 or fp16).  Row size in bytes must be a
 *                   multiple of 16.
 * expert_idx        [num_rows, k] int32, values in [0, expert_num).
 * quant_mode        MM_QUANT_NONE (expanded_x has x's type), an MXFP8 mode
 *                   (expanded_x FP8, h a multiple of 16), or MM_QUANT_MXFP4_E2M1
 *                   (quantMode 9: expanded_x [num_rows*k, h/2] packed E2M1, two
 *                   codes per byte, element 2i in bits 0-3).
 * expert_tokens_num_type  0: expert_tokens is the inclusive cumsum of the
 *                   counts; 1: the counts (expertTokensNumType 0 / 1).
 * expanded_x        [num_rows*k, h] output.
 * expanded_scale    [num_rows*k, AlignUp(CeilDiv(h, 32), 2)] E8M0 output in
 *                   the MX modes (padding column 0); ignored otherwise.
 * expanded_row_idx  [num_rows*k] int32 scatter index (rowIdxType 1), or NULL.
 * sorted_row_idx    [num_rows*k] int32 gather index (rowIdxType 0), or NULL.
 * expert_tokens     [expert_num] int64, or NULL.  With num_rows = 0 only
 *                   expert_tokens is written (all zeros).
 * Rows whose id is out of range are left out: their expanded_row_idx is -1,
 * the tail of sorted_row_idx is -1, the matching tail rows of expanded_x are
 * not written, and MM_DEVERR_EXPERT_RANGE is raised.
 * Limits: num_rows*k < 16777215 (the sort limit of the permute article),
 * 1 <= expert_num <= 10240.
 * ---------------------------------------------------------------------- */
mm_status mm_moe_init_routing_workspace_size(int64_t num_rows, int64_t k, int64_t expert_num,
                                             size_t* bytes);
mm_status mm_moe_init_routing(const void* x, int x_dtype, const int32_t* expert_idx,
                              int64_t num_rows, int64_t h, int64_t k, int64_t expert_num,
                              int quant_mode, int expert_tokens_num_type, void* expanded_x,
                              uint8_t* expanded_scale, int32_t* expanded_row_idx,
                              int32_t* sorted_row_idx, int64_t* expert_tokens, void* workspace,
                              size_t workspace_bytes, int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * mm_moe_init_routing_v3 -- MoeInitRoutingV3, Dropless, with the active
 * expert range (activeExpertRangeOptional = [active_expert_start,
 * active_expert_end), computation step 6) and the three count types.
 *
 * Only ids in the range are sorted: they fill the first availableIdxNum =
 * |{ids in the range}| rows of expanded_x / expanded_scale and of
 * sorted_row_idx (whose tail is -1); the other ids get expanded_row_idx -1
 * and no row.  Ids in [0, expert_num) but outside the range are not errors;
 * ids outside [0, expert_num) raise MM_DEVERR_EXPERT_RANGE.
 * 0 <= active_expert_start < active_expert_end <= expert_num, else
 * MM_ERR_INVALID_ARG.
 * expert_tokens_num_type  0: expert_tokens [end - start] inclusive cumsum;
 *                   1: [end - start] counts; 2 (key_value): [expert_num, 2]
 *                   int64 pairs (expert id, count) of the range's experts with
 *                   a non-zero count, in ascending id, the rows after them 0
 *                   (expert_num <= 5120 in this mode).
 * Other arguments as mm_moe_init_routing; the workspace is sized by
 * mm_moe_init_routing_v3_workspace_size.
 * ---------------------------------------------------------------------- */
mm_status mm_moe_init_routing_v3_workspace_size(int64_t num_rows, int64_t k, int64_t expert_num,
                                                size_t* bytes);
mm_status mm_moe_init_routing_v3(const void* x, int x_dtype, const int32_t* expert_idx,
                                 int64_t num_rows, int64_t h, int64_t k, int64_t expert_num,
                                 int64_t active_expert_start, int64_t active_expert_end,
                                 int quant_mode, int expert_tokens_num_type, void* expanded_x,
                                 uint8_t* expanded_scale, int32_t* expanded_row_idx,
                                 int32_t* sorted_row_idx, int64_t* expert_tokens, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * mm_moe_token_permute -- moe_token_permute with padded_mode = false.
 *
 *   sortedIndicesFirst = stable argSort(indices.flatten())
 *   sorted_indices     = argSort(sortedIndicesFirst)   (the inverse map)
 *   permuted[d]        = Q(tokens[sortedIndicesFirst[d] / topk]),  d < M
 *
 * tokens          [n, h] of tokens_dtype (fp16 / bf16 / fp32; quantised modes
 *                 take fp16 / bf16).
 * indices         [n, topk] (topk = 1 for 1-D indices) of indices_dtype
 *                 (MM_DT_INT32 / MM_DT_INT64), values in [0, num_experts).
 * num_experts     exclusive upper bound of the index values.  The article's
 *                 API infers it from the data; here the caller states it
 *                 (the counting sort needs the key range).
 * num_out_tokens  0: M = F = n*topk; > 0: M = min(num_out_tokens, F);
 *                 < 0: M = max(F + num_out_tokens, 0).
 * padded_mode     must be 0 (MM_ERR_UNSUPPORTED otherwise, as in the article).
 * quant_mode      MM_QUANT_NONE, MM_QUANT_MXFP8_E5M2, MM_QUANT_MXFP8_E4M3FN, or
 *                 MM_QUANT_MXFP4_E2M1 (the article's quant_mode 9: 32-element
 *                 groups, emax 2, two codes per byte, element 2i in bits 0-3).
 * permuted_tokens [M, h] output (tokens' type, or FP8); MXFP4: [M, h/2] bytes.
 * expanded_scale  [M, AlignUp(CeilDiv(h, 32), 2)] E8M0 output (MXFP8 modes);
 *                 MXFP4: [M, CeilDiv(h, 64), 2], the same number of columns.
 * sorted_indices  [F] int32 output, never truncated.
 * Limits: F < 16777215.
 * ---------------------------------------------------------------------- */
int64_t mm_moe_token_permute_out_rows(int64_t num_indices, int64_t num_out_tokens);
mm_status mm_moe_token_permute_workspace_size(int64_t num_indices, int64_t num_experts,
                                              size_t* bytes);
mm_status mm_moe_token_permute(const void* tokens, int tokens_dtype, const void* indices,
                               int indices_dtype, int64_t n, int64_t topk, int64_t h,
                               int64_t num_experts, int64_t num_out_tokens, int padded_mode,
                               int quant_mode, void* permuted_tokens, uint8_t* expanded_scale,
                               int32_t* sorted_indices, void* workspace, size_t workspace_bytes,
                               int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * mm_mega_moe -- MegaMoE, A8W8-FP / A8W4-FP / A4W4-FP scenarios, epWorldSize = 1:
 *
 *   X_hat_e, S_X,e = Q_MX(x[T_e])                                 stage 1
 *   G_e = DQ(X_hat_e) DQ(W1_e^(G))^T, U_e = DQ(X_hat_e) DQ(W1_e^(U))^T
 *   A_e = SiLU(G_e) * U_e,  A_hat_e, S_A,e = Q_MX(A_e)             stage 2
 *   O_e = DQ(A_hat_e) DQ(W2_e)^T                                  stage 3
 *   Y[i] = sum_k W[i,k] O[pi(i,k)] + sum_s O_s^shared[i]          stage 4
 *
 * x                  [bs, h] bf16 (dispatch_quant_mode 4), or FP8 codes of
 *                    dispatch_quant_out_dtype (dispatch_quant_mode 0; packed
 *                    FP4 [bs, h/2] when that type is 296).
 * x_scales           dispatch_quant_mode 0: E8M0 scales of x, [bs, h/32]
 *                    (the pages' scales input, (BS, CeilDiv(H, 32))); NULL
 *                    otherwise.
 * topk_ids           [bs, k] int32, distinct per token, in [0, moe_expert_num).
 *                    An id outside that range raises MM_DEVERR_EXPERT_RANGE and
 *                    its (token, k) term is left out of Y (and of the counts);
 *                    a repeated id raises MM_DEVERR_DUPLICATE_ID.
 * topk_weights       [bs, k], topk_weights_dtype MM_DT_FLOAT32 or MM_DT_BFLOAT16.
 * weight1            [E, 2*intermediate, h] FP8 (weight_dtype 23 / 24), or
 *                    FLOAT4_E2M1 (weight_dtype 296, the A8W4-FP scenario:
 *                    [E, 2*intermediate, h/2] packed bytes); rows [0, I) are
 *                    the gate (SiLU) branch, [I, 2I) the up branch.
 * weight2            [E, h, intermediate] of the same type (FP4: [E, h, I/2]).
 * weight_scales1/2   E8M0, MM_WSCALE_ROWS: [E, 2I, CeilDiv(h,64), 2] and
 *                    [E, h, CeilDiv(I,64), 2]; MM_WSCALE_PREPARED: the
 *                    outputs of mm_prepare_weight_scales for those arrays.
 * shared_weight*     same layouts with leading dimension shared_expert_num
 *                    (0..4; NULL when 0); shared_weight_dtype 23 / 24 / 296.
 * ep_world_size      must be 1.
 * max_recv_token_num 0, or >= bs*k (the rows this rank receives at ep = 1).
 * dispatch_quant_mode 4 (MX quantisation inside the operator) or 0
 *                    (pre-quantised pass-through: x and x_scales are X_hat, S_X);
 * dispatch_quant_out_dtype 23 / 24 is also the type of A_hat (FP8 with either
 *                    weight type: A8W8-FP, A8W4-FP).  296 (FLOAT4_E2M1) is
 *                    the A4W4-FP scenario ("A4W4-FP quantization scenario"):
 *                    the routed weights must be FP4 too (else
 *                    MM_ERR_UNSUPPORTED); X_hat is packed MXFP4, GEMM1 multiplies
 *                    FP4 by FP4, and A_hat is re-quantised to MXFP8 E4M3, so
 *                    GEMM2 is A8W4.
 * shared_quant_out_dtype  the shared experts' own input quantisation type (the
 *                    parameter table's sharedExpertQuantOutDtype): 0 for the
 *                    dispatch type, or 23 / 24 / 296 (any shared weight type;
 *                    with 296 their A_hat is E4M3, as in A4W4-FP).  The
 *                    shared rows are quantised in a pass of their own; with
 *                    dispatch_quant_mode 0 only 0 or the dispatch type is
 *                    accepted (MM_ERR_INVALID_ARG otherwise).
 * combine_quant_mode must be 0.
 * activation         "swiglu" (or NULL), "swiglustep", "swigluoai", "situglu" or
 *                    "gelu", with activation_params as the README's parameter
 *                    table gives them: swiglu / swiglustep [] or [clamp];
 *                    swigluoai [] or [clamp, alpha, beta] (defaults: clamp off,
 *                    alpha 1.702, beta 1.0); situglu [], [beta] or [beta,
 *                    linear_beta] (beta 1.0 when empty); gelu [FLT_MAX] only.
 *                    A clamp of 0 or FLT_MAX means no clamp.  Formulas:
 *                    "Activation function formulas".  Under gelu the whole
 *                    2*intermediate-wide Linear1 output is activated, so
 *                    weight2 is [E, h, 2*intermediate] (scales likewise) and
 *                    A_hat has 2*intermediate columns.  Bad parameter lists
 *                    give MM_ERR_INVALID_ARG, other names MM_ERR_UNSUPPORTED.
 * y                  [bs, h] bf16 output.
 * The call may be captured in a CUDA graph on `stream` (its kernels are
 * ordinary launches while the stream is capturing); the workspace and the
 * outputs then belong to the graph's replays.
 * expert_token_nums  [E] int32 output (rows per expert), or NULL.  With
 *                    bs = 0 only this is written (all zeros).
 * expanded_row_idx   [bs*k] int32 output pi(i, k) (position of row j = i*k+k'
 *                    in expert-sorted order), or NULL.
 * act_q, act_scale   optional diagnostic outputs of A_hat in expert-sorted
 *                    row order: [bs*k, W] FP8 and [bs*k, W/32] E8M0 with W = I
 *                    (2I under gelu); NULL to skip.
 * dispatch_q, dispatch_scale  optional diagnostic outputs of the dispatched
 *                    X_hat (stage 1) in expert-sorted row order: [bs*k, h]
 *                    FP8 codes of dispatch_quant_out_dtype ([bs*k, h/2] packed
 *                    FP4 under A4W4-FP) and [bs*k, h/32] E8M0; NULL to skip
 *                    (both or neither).
 * Shape limits: h and intermediate multiples of 128; k <= 32;
 * moe_expert_num <= 2048.
 * ---------------------------------------------------------------------- */
mm_status mm_mega_moe_workspace_size(int64_t bs, int64_t h, int64_t k, int64_t moe_expert_num,
                                     int64_t intermediate, int64_t shared_expert_num,
                                     int weight_scale_layout, size_t* bytes);
mm_status mm_mega_moe(const void* x, const uint8_t* x_scales, const int32_t* topk_ids,
                      const void* topk_weights, int topk_weights_dtype, const uint8_t* weight1, const uint8_t* weight2,
                      const uint8_t* weight_scales1, const uint8_t* weight_scales2,
                      int weight_dtype, int weight_scale_layout, const uint8_t* shared_weight1,
                      const uint8_t* shared_weight2, const uint8_t* shared_weight_scales1,
                      const uint8_t* shared_weight_scales2, int shared_weight_dtype,
                      int64_t shared_expert_num, int64_t bs, int64_t h, int64_t k,
                      int64_t moe_expert_num, int64_t ep_world_size, int64_t intermediate,
                      int64_t max_recv_token_num, int64_t dispatch_quant_mode,
                      int64_t dispatch_quant_out_dtype, int64_t shared_quant_out_dtype,
                      int64_t combine_quant_mode, const char* activation, const float* activation_params,
                      int64_t n_activation_params, void* y, int32_t* expert_token_nums,
                      int32_t* expanded_row_idx, uint8_t* act_q, uint8_t* act_scale,
                      uint8_t* dispatch_q, uint8_t* dispatch_scale,
                      void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Weight preparation (one-time, at weight-load time).
 *
 * mm_prepare_weight_scales rearranges E8M0 weight scales from the pages'
 * (E, N_out, CeilDiv(K_red, 64), 2) layout into the tile layout the grouped
 * GEMMs read (MM_WSCALE_PREPARED), the way the pages require FRACTAL_NZ
 * weight formats for some scenarios.  which = 1 for weightScales1 (N_out =
 * 2I), 2 for weightScales2 (N_out = H).  The layout is [E][pair][K_red/128]
 * [2][512 B]: each 512-byte tile holds the scales of 128 rows x 128 k in the
 * order the tensor-core scale copy reads them, and the two tiles of one GEMM
 * n tile sit side by side (which = 1: gate rows 128p.. with up rows
 * I + 128p..; which = 2: rows 256p..; rows past N_out read as zero).  src and
 * dst are device buffers; dst holds mm_prepared_weight_scales_size bytes.
 * K_red must be a multiple of 128, and with which = 1 N_out a multiple of
 * 256; other sizes give MM_ERR_INVALID_ARG.
 * ---------------------------------------------------------------------- */
mm_status mm_prepared_weight_scales_size(int which, int64_t experts, int64_t n_out, int64_t k_red,
                                         size_t* bytes);
mm_status mm_prepare_weight_scales(const uint8_t* src, int which, int64_t experts,
                                   int64_t n_out, int64_t k_red, uint8_t* dst, void* stream);

/* ------------------------------------------------------------------------
 * mm_mx_quantize -- Q_MX along each row (MegaMoE A8W8-FP stage 1; with
 * out_dtype 296 the MXFP4 E2M1 weights of the A8W4-FP scenario): groups of
 * 32 consecutive elements share one E8M0 exponent s = floor(log2 amax) -
 * emax (8 for E4M3FN, 15 for E5M2, 2 for E2M1), clamped to [-127, 127];
 * elements are FP8 / FP4(v * 2^-s), nearest-even, saturated to the largest
 * finite value.
 *
 * src     [rows, cols] of src_dtype (fp32 / bf16 / fp16); cols a multiple of 16.
 * q       [rows, cols] FP8 output of out_dtype (23 / 24), or [rows, cols/2]
 *         packed FP4 bytes (296).
 * scales  [rows, scale_cols] E8M0 output, scale_cols >= CeilDiv(cols, 32);
 *         columns past CeilDiv(cols, 32) are written as 0.
 * ---------------------------------------------------------------------- */
mm_status mm_mx_quantize(const void* src, int src_dtype, int64_t rows, int64_t cols, int out_dtype,
                         uint8_t* q, uint8_t* scales, int64_t scale_cols, void* stream);

/* ------------------------------------------------------------------------
 * mm_selftest_wait_timeout -- exercises the failure path of the kernels'
 * bounded waits.  The operator pages have no counterpart; it exists so that
 * a caller (and the tests) can check, without any fault, that a wait which
 * never completes ends: one CTA waits on an mbarrier that nothing arrives at,
 * gives up after limit_ns nanoseconds of %globaltimer time (the GEMM kernels
 * use the same wait with a 2 s limit), OR-s MM_DEVERR_TIMEOUT into *dev_err
 * and returns; the context stays usable.
 *
 * limit_ns   in (0, 10 s]; dev_err: device int32, required.  Asynchronous on
 * stream; MM_ERR_INVALID_ARG for a bad limit or a null dev_err.
 * ---------------------------------------------------------------------- */
mm_status mm_selftest_wait_timeout(int64_t limit_ns, int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Expert parallelism: dispatch to ranks and combine (MegaMoE README, A8W8-FP
 * scenario stage 1, where the quantised tokens travel to the ranks that hold
 * their experts, and stage 4, where the GMM2 rows go back to their source
 * rank to be weighted and summed, with epWorldSize > 1; parameter table
 * epWorldSize / moeExpertNum; the A4W4-FP scenario sends MXFP4 rows).  Rank r holds experts [r*E/W, (r+1)*E/W).
 * The exchange between ranks is the caller's collective (an all-to-all with
 * the counts below as split sizes); each rank runs mm_moe_expert_ffn on the
 * rows it receives (its local experts) and sends the resulting rows back in
 * the order received.
 *
 * mm_moe_ep_dispatch -- on the source rank: the flattened ids j = i*K + k
 *   are sorted by destination rank id / (E/W), stably (rows of one rank in
 *   ascending j); every token is MX-quantised once (group 32, E8M0 shared
 *   exponent, dispatch_quant_out_dtype 23 / 24, or 296 for packed FP4 E2M1)
 *   and its row stored at its K positions.
 * x                 [num_rows, h] bf16 / fp16 (x_dtype), h a multiple of 128.
 * topk_ids          [num_rows, k] int32 in [0, moe_expert_num); k <= 32.
 * moe_expert_num    E, a multiple of ep_world_size W.
 * send_x            [num_rows*k, h] FP8 codes ([num_rows*k, h/2] packed FP4),
 *                   rank-sorted (output).
 * send_scales       [num_rows*k, h/32] E8M0 (output).
 * send_expert       [num_rows*k] int32: the row's expert on its destination
 *                   rank, id % (E/W) (output).
 * rank_counts       [W] int64: rows for each rank, the send split sizes.
 * expanded_row_idx  [num_rows*k] int32: position of row j in the send
 *                   order; -1 for an id out of range (row left out,
 *                   MM_DEVERR_EXPERT_RANGE set).
 * workspace         mm_moe_ep_dispatch_workspace_size bytes.
 * num_rows = 0 only zeroes rank_counts.
 *
 * mm_moe_combine -- Y[i] = sum_k W[i,k] * expert_rows[row_idx[i*k + k']]
 *   + sum_s shared_rows[s][i], accumulated in fp32 in the order k' = 0..k-1
 *   then s, rounded to bf16 once; row_idx < 0 leaves the term out (MegaMoE
 *   stage 4).  On the source rank: expert_rows = the returned rows in send
 *   order, row_idx = expanded_row_idx of mm_moe_ep_dispatch, shared_rows =
 *   the rank's own shared experts' outputs for its tokens (they take part in
 *   no exchange).
 * expert_rows       [*, h] bf16 (expert_rows_dtype MM_DT_BFLOAT16), h a multiple
 *                   of 8; or MXFP8 codes (23 / 24: combineQuantMode 3 / 4, the
 *                   rows quantised for the exchange) with expert_scales
 *                   [*, h/32] E8M0, h a multiple of 32: each routed term is
 *                   DQ_MX of its row.
 * row_idx           [num_rows*k] int32; num_rows*k below 16777215, the row
 *                   limit of mm_moe_ep_dispatch.  Entries >= 0 must index
 *                   rows of expert_rows: the call is not given that buffer's
 *                   row count and cannot check them.
 * topk_weights      [num_rows, k] fp32 or bf16 (topk_weights_dtype).
 * shared_rows       [n_shared, num_rows, h] bf16, n_shared 0..4 (NULL when 0);
 *                   k + n_shared <= 36.
 * y                 [num_rows, h] bf16 output.
 * ---------------------------------------------------------------------- */
mm_status mm_moe_ep_dispatch_workspace_size(int64_t num_rows, int64_t k, int64_t ep_world_size, size_t* bytes);
mm_status mm_moe_ep_dispatch(const void* x, int x_dtype, const int32_t* topk_ids, int64_t num_rows, int64_t h,
                             int64_t k, int64_t moe_expert_num, int64_t ep_world_size,
                             int64_t dispatch_quant_out_dtype, uint8_t* send_x, uint8_t* send_scales,
                             int32_t* send_expert, int64_t* rank_counts, int32_t* expanded_row_idx,
                             void* workspace, size_t workspace_bytes, int32_t* dev_err, void* stream);
mm_status mm_moe_combine(const void* expert_rows, int expert_rows_dtype, const uint8_t* expert_scales,
                         const int32_t* row_idx, const void* topk_weights, int topk_weights_dtype,
                         int64_t num_rows, int64_t h, int64_t k, const void* shared_rows, int64_t n_shared,
                         void* y, void* stream);

/* ------------------------------------------------------------------------
 * mm_moe_expert_ffn -- the expert side of expert parallelism (MegaMoE README,
 * A8W8-FP scenario stages 2-3 on the rows a rank receives): for every
 * received row r, out[r] = GMM2(act(GMM1(DQ_MX(x[r]))), Q_MX between them)
 * with the weights of its local expert expert_ids[r], the bf16 result
 * written at row r itself (the order in which the rows go back to their
 * source ranks).  The same arithmetic as mm_mega_moe with top-K 1, gating
 * weight 1, pass-through quantisation and no shared experts, bit for bit,
 * without its combine pass.
 * x                 [rows, h] FP8 codes of x_dtype (23 | 24), or [rows, h/2]
 *                   packed FP4 codes (x_dtype 296, A4W4-FP: FP4 weights
 *                   required); x_scales [rows, h/32] E8M0 (required when
 *                   rows > 0).
 * expert_ids        [rows] int32 local expert ids in [0, local_experts); an
 *                   id outside the range leaves its row of out unwritten and
 *                   raises MM_DEVERR_EXPERT_RANGE.
 * weights, scales, weight_dtype, weight_scale_layout, activation: as for
 *                   mm_mega_moe, with E = local_experts.
 * out               [rows, h] bf16.  expert_token_nums [local_experts] int32
 *                   rows per expert (may be NULL).
 * Workspace from mm_moe_expert_ffn_workspace_size; errors as mm_mega_moe.
 * ---------------------------------------------------------------------- */
mm_status mm_moe_expert_ffn_workspace_size(int64_t rows, int64_t h, int64_t local_experts, int64_t intermediate,
                                           int weight_scale_layout, size_t* bytes);
mm_status mm_moe_expert_ffn(const uint8_t* x, const uint8_t* x_scales, int x_dtype, const int32_t* expert_ids,
                            int64_t rows, int64_t h, const uint8_t* weight1, const uint8_t* weight2,
                            const uint8_t* weight_scales1, const uint8_t* weight_scales2, int weight_dtype,
                            int weight_scale_layout, int64_t local_experts, int64_t intermediate,
                            const char* activation, const float* activation_params, int64_t n_activation_params,
                            void* out, int32_t* expert_token_nums, void* workspace, size_t workspace_bytes,
                            int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * mm_moe_init_routing_noalloc -- the same routing and permute as
 * mm_moe_init_routing (same arguments and outputs), for callers that cannot
 * give the library device scratch memory: for example a host program or
 * plug-in that reaches this library only through this C interface and has
 * no device allocator of its own, or one that must not call cudaMalloc /
 * cudaFree while it serves requests (those calls can synchronise the device
 * and fragment memory).  The operator pages have no counterpart of this
 * entry point; it exists only for such callers.
 *
 * No allocation: the caller passes inputs and outputs only.  The scratch the
 * kernels need lives in one fixed array of MM_NOALLOC_SCRATCH_BYTES inside
 * the library, which every GPU that loads the library holds until the
 * process exits.  With R = num_rows * k expanded rows and E = expert_num
 * the scratch is 4 * E * min(CeilDiv(R, 256), 512) bytes of histograms,
 * about 8 * E bytes of offsets, and 4 * R bytes of scatter index only when
 * expanded_row_idx is NULL (each piece rounded up to 256 bytes).  At
 * E = 256 every R below the sort limit fits when the caller passes
 * expanded_row_idx, and R up to 916,928 without it; from E = 2041 up, no
 * problem of 131,072 rows or more fits.  A problem that does not fit is
 * rejected with MM_ERR_WORKSPACE before anything is enqueued.
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  A failed lookup returns MM_ERR_CUDA.
 * Sharing: every call uses the same array and it keeps the last call's
 * contents; the one word that must start at zero (a grid-barrier counter)
 * is cleared on the stream by each call.  Calls whose kernels may overlap
 * on the GPU, e.g. on different streams without ordering, race on the
 * array; order them on one stream.  Launches are counted and timed by
 * mm_timing_read like those of mm_moe_init_routing.
 * ---------------------------------------------------------------------- */
#define MM_NOALLOC_SCRATCH_BYTES (4u << 20)
mm_status mm_moe_init_routing_noalloc(const void* x, int x_dtype, const int32_t* expert_idx,
                                      int64_t num_rows, int64_t h, int64_t k, int64_t expert_num,
                                      int quant_mode, int expert_tokens_num_type, void* expanded_x,
                                      uint8_t* expanded_scale, int32_t* expanded_row_idx,
                                      int32_t* sorted_row_idx, int64_t* expert_tokens,
                                      int32_t* dev_err, void* stream);

/* ------------------------------------------------------------------------
 * Stage timing and launch counts (diagnostics; not part of the pages' API).
 *
 * mm_timing_enable(1) makes every following call record a CUDA event pair
 * on its stream around each of its stages (MM_STAGE_*); mm_timing_enable(0)
 * stops that.  mm_timing_read waits for the recorded events, writes for
 * each stage s < n the device time summed over all recorded calls
 * (stage_ms[s], milliseconds) and the number of kernels launched since the
 * previous read (stage_launches[s], counted whether timing is on or not),
 * then resets both.  Host-side state only; not thread-safe across
 * concurrent callers on different streams.
 * ---------------------------------------------------------------------- */
#define MM_STAGE_WSCALE 0   /* weight-scale layout conversion */
#define MM_STAGE_ROUTE 1    /* histogram, scan, stable scatter */
#define MM_STAGE_DISPATCH 2 /* permute / MX quantisation */
#define MM_STAGE_GEMM1 3    /* grouped GEMM1 + swiglu + MX requant */
#define MM_STAGE_GEMM2 4    /* grouped GEMM2 */
#define MM_STAGE_COMBINE 5  /* weighted top-K combine */
#define MM_STAGE_DIAG 6     /* optional diagnostic outputs */
#define MM_STAGE_COUNT 7
mm_status mm_timing_enable(int on);
mm_status mm_timing_read(double* stage_ms, int64_t* stage_launches, int n);
/* mm_timing_select: which stages record their event pair while timing is on
 * (bit s = stage s; all stages by default).  Each event record between two
 * kernels costs the stream a few microseconds, so a measurement of the whole
 * call can keep the pair of one stage only.  MM_ERR_INVALID_ARG for bits at
 * or above MM_STAGE_COUNT. */
mm_status mm_timing_select(uint32_t stage_mask);

/* ------------------------------------------------------------------------
 * Routing implementation (diagnostics; not part of the pages' API).  Every
 * routing path computes the same stable counting sort (MoeInitRoutingV3,
 * formula steps 1-3) bit for bit; this selects which one the following
 * calls of every entry point use, process-wide:
 *   MM_ROUTE_AUTO      one thread-block cluster of up to 16 CTAs
 *                      (distributed shared memory, two cluster barriers)
 *                      for up to 131072 ids and 4096 keys; otherwise one
 *                      cooperative grid launch; under
 *                      stream capture, or where the grid does not fit,
 *                      four ordinary kernels
 *   MM_ROUTE_CLUSTER   the cluster kernel whenever the key count allows it
 *   MM_ROUTE_GRID      the cooperative grid launch (not under capture)
 *   MM_ROUTE_KERNELS   the four kernels
 * A path that cannot run for a problem falls through to the next one in
 * that order.  Returns MM_ERR_INVALID_ARG for any other value.  Host-side
 * state only.
 * ---------------------------------------------------------------------- */
#define MM_ROUTE_AUTO 0
#define MM_ROUTE_CLUSTER 1
#define MM_ROUTE_GRID 2
#define MM_ROUTE_KERNELS 3
mm_status mm_set_routing_path(int path);

/* ------------------------------------------------------------------------
 * Checked build (a debug aid; not part of the pages' API).  The same
 * sources compiled with MM_CHECK give libmm_moe_check.so, whose kernels
 * test every index they compute on the GPU (a routed row's slot against
 * the expanded-row count, a padded row against the grouped-layout
 * capacity, a GEMM tile against the tile count of its segment and of the
 * buffers, a combine term's row against the expert-row buffer) before the
 * access it guards; a failed test skips the access and ORs
 * MM_DEVERR_BOUNDS into *dev_err, so an internal inconsistency shows up as
 * a status bit instead of a memory fault.  The ABI is identical.
 * mm_checked_build returns 1 in that library and 0 in libmm_moe.so.
 * ---------------------------------------------------------------------- */
int mm_checked_build(void);

#ifdef __cplusplus
}
#endif

#endif /* MM_MOE_H_ */
