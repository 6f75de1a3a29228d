// Internal interfaces between the C-ABI layer and the kernel files.
#pragma once

#include "mm_common.cuh"

namespace mm {

// ---- routing (route.cu) ----------------------------------------------------
struct RoutePlan {
  int64_t rows;         // R = N * K flattened ids
  int num_experts;      // E
  int chunk;            // ids per warp chunk (multiple of 32)
  int units;            // number of chunks
  int warps_per_block;  // chunks per block (smem: warps * E * 4 bytes)
};

// Sort keys of the routing: key = (id - off) / div for the ids with a key in
// [0, num_experts); ids outside [0, limit) raise MM_DEVERR_EXPERT_RANGE.
struct KeyMap {
  int div;
  int off;
  int64_t limit;
};

struct RouteOutputs {
  int32_t* expanded_row_idx = nullptr;   // [R] scatter index (or null)
  int32_t* sorted_row_idx = nullptr;     // [R] gather index (or null)
  int32_t* pad_row = nullptr;            // [R] row in the 128-row padded grouped layout (or null)
  int64_t* expert_tokens = nullptr;      // [E] int64 counts / cumsum (or null)
  int tokens_cumsum = 0;
  int32_t* expert_token_nums = nullptr;  // [E] int32 counts (or null)
  int32_t* seg_rows = nullptr;           // [E + S] rows per GEMM segment (or null)
  int32_t* seg_mprefix = nullptr;        // [E + S + 1] prefix of 128-row tiles (or null)
  int n_shared = 0;                      // S shared segments ...
  int shared_rows = 0;                   // ... of this many rows each
  int key_div = 1;                       // sort key = id / key_div (ids < num_experts * key_div)
  int32_t* sorted_rem = nullptr;         // [R] id % key_div at each sorted position (or null)
  int key_off = 0;                       // key_div 1: sort key = id - key_off (an active expert range)
  int64_t id_limit = 0;                  // ids outside [0, id_limit) are errors (0: num_experts * key_div);
                                         // other ids without a key are left out silently
  int64_t pad_limit = 0;                 // rows of the padded layout pad_row addresses (checked build)
};

struct RouteScanArgs {
  int32_t* hist;
  int32_t* totals;
  int num_experts, units;
  int64_t rows;
  int32_t* offsets;
  int32_t* sorted_row_idx;
  int64_t* expert_tokens;
  int tokens_cumsum;
  int32_t* expert_token_nums;
  int32_t* seg_rows;
  int32_t* seg_mprefix;
  int n_shared, shared_rows;
};

RoutePlan route_plan(int64_t rows, int num_experts);
size_t route_workspace_bytes(const RoutePlan& p);
// int32 words of the offsets workspace: offsets [E + 1], totals [E] and the
// fused launch's grid-barrier counter
int64_t route_offsets_words(int num_experts);
// hist: [E * units] int32, offsets: [route_offsets_words(E)] int32 (both
// workspace)
// *launches (optional) receives the number of kernels launched: 1 (one
// cluster launch or one cooperative launch) or 4.
// MoeInitRoutingV3 expertTokensNumType 2 (key_value): out [out_rows, 2] int64
// = (first + e, counts[e]) for each e < n with counts[e] != 0, in ascending e,
// then zeros.
cudaError_t launch_key_value_counts(const int64_t* counts, int n, int64_t first, int64_t out_rows, int64_t* out,
                                    cudaStream_t st);
cudaError_t launch_route(const RoutePlan& p, const void* ids, bool ids64, int32_t* hist, int32_t* offsets,
                         RouteOutputs o, int32_t* dev_err, cudaStream_t st, int* launches = nullptr);
// Routing implementation used from now on, process-wide: 0 automatic (one
// cluster of up to 16 CTAs up to 131072 ids and 4096 keys, else the cooperative grid launch,
// else four kernels), 1 cluster, 2 cooperative grid, 3 four kernels (a path
// that cannot run falls through to the next).
void set_route_path(int path);

// ---- combine of rows given by an index (combine.cu) ------------------------
// Y[i] = sum_k W[i,k] * rows[row_idx[i*K + k]] (row_idx < 0: term left out),
// fp32 in k order, one bf16 rounding (MegaMoE stage 4 / EP combine).
cudaError_t launch_combine_rows(const __nv_bfloat16* rows, const int32_t* row_idx, const void* gate, int gate_bf16,
                                int64_t n, int64_t h, int k, const __nv_bfloat16* shared_rows, int n_shared,
                                __nv_bfloat16* y, cudaStream_t st, const uint8_t* rows_q = nullptr,
                                const uint8_t* rows_sf = nullptr, int rows_fmt = 0);

// ---- permute / quantise (permute.cu) -------------------------------------
struct PermuteArgs {
  const void* src;          // [n, h] source rows
  int src_dtype;            // MM_DT_BFLOAT16 / FLOAT16 / FLOAT32, or FP8 with src_scales
  const uint8_t* src_scales;  // pre-quantised source: E8M0 [n, h/32] (tile-layout output only)
  int64_t n, h;             // rows, row length (elements)
  int k;                    // destinations per row from dest[] (row i -> dest[i*k + t])
  const int32_t* dest;      // [n*k] destination rows (< 0: skipped; null: identity, k must be 1)
  int64_t dest_limit;       // destinations >= dest_limit are skipped (num_out_tokens)
  const int32_t* ids;       // [n, k] expert ids for the duplicate check (or null)
  int n_extra;              // extra destinations per row: extra_base[s] * 128 + i
  const int32_t* extra_base;  // [n_extra] tile index of each extra segment (device)
  int out_fmt;              // -1 copy, 23 / 24 FP8
  void* out;                // [*, h] output rows
  int64_t out_stride;       // bytes between output rows (0: the row's own size, h or h / 2 for packed FP4)
  uint8_t* scales;          // E8M0 output
  int64_t scale_cols;       // row layout: scale row stride; 0 = GEMM tile layout
  int32_t* dev_err;
  int32_t* dest_inv;        // optional [dest_limit]: dest_inv[dest[i*k + t]] = i*k + t (routed destinations)
};
cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t st);

// Tile layout of E8M0 weight scales (mm_prepare_weight_scales): 512-byte
// tiles of 128 rows x 128 k, two per GEMM n tile and k-block side by side
// ([E][pair][k-block][2][512 B]) so one 1 KB copy brings a stage's B scales.
// which = 1 (weight1, n_out = 2I): pair p = gate rows [128p, +128) and up
// rows [I + 128p, +128); which = 2: rows [256p, +256).
int64_t prepared_npairs(int64_t n_out, int which);
cudaError_t launch_prepare_wscales(const uint8_t* src, int64_t experts, int64_t n_out, int64_t k_red, int which,
                                   uint8_t* dst, cudaStream_t st);

// ---- grouped GEMMs (gemm.cu) ----------------------------------------------
struct GemmLaunch {
  int mode;                   // 1: GEMM1 + swiglu + MX requant; 2: GEMM2 -> bf16
  const uint8_t* a;           // [rows_cap, K] FP8 A (padded grouped layout), or packed FP4 [rows_cap, K/2]
  int64_t rows_cap;
  const uint8_t* sfa;         // A scales, tile layout
  const uint8_t* b;           // routed weights [E, N, K] FP8
  const uint8_t* sfb;         // routed prepared scales
  const uint8_t* b_sh;        // shared weights [S, N, K] (or null)
  const uint8_t* sfb_sh;
  int n_routed, n_shared;
  const int32_t* seg_rows;    // [n_routed + n_shared]
  const int32_t* seg_mprefix; // [n_routed + n_shared + 1]
  int64_t K, N;
  int a_fmt, b_fmt, b_fmt_sh; // 23 / 24, or 296 (packed FP4 E2M1)
  int a_fmt_sh;               // A type of the shared segments (their own input quantisation)
  int64_t a_stride;           // bytes between rows of a (0: K, or K / 2 for packed FP4)
  int act_fmt;                // mode 1: type of A_hat (23 / 24)
  int act_fmt_sh;             // mode 1: type of the shared segments' A_hat
  int inter;                  // mode 1: I (= N / 2)
  int act;                    // mode 1: MM_ACT_* (A_hat width I, or 2I for gelu)
  float act_c, act_alpha, act_beta, act_beta_lin;  // clamp (+inf: off), swigluoai alpha / beta,
                                                   // situglu beta / linear beta (0: off)
  uint8_t* act_q;             // mode 1 outputs
  uint8_t* act_sf;
  __nv_bfloat16* out;         // mode 2 output [rows_cap, N], or [rows of out_row, N]
  const int32_t* out_row;     // mode 2, optional: padded row r is written to output row out_row[r]
  int64_t out_rows;           // rows of out when out_row is set (checked build)
  int32_t* dev_err;
};
cudaError_t launch_gemm(const GemmLaunch& g, cudaStream_t st);

// ---- combine (combine.cu) --------------------------------------------------
struct CombineArgs {
  const __nv_bfloat16* o;     // [rows_cap, h] expert outputs (padded grouped layout)
  const __nv_bfloat16* o_sh;  // optional [n_shared, n, h] shared-expert rows (else in o at their segments)
  const uint8_t* oq;          // optional: the routed rows as MXFP8 codes [*, h] (oq_fmt 23 / 24) ...
  const uint8_t* oq_sf;       // ... with E8M0 scales [*, h / 32] (then o is unused)
  int oq_fmt;
  const int32_t* pad_row;     // [n*k]
  const void* gate;           // [n, k] fp32 or bf16
  int gate_bf16;
  int n_shared;
  const int32_t* seg_mprefix; // shared segment s starts at tile seg_mprefix[n_routed + s]
  int n_routed;
  int64_t n, h;
  int k;
  __nv_bfloat16* y;           // [n, h]
  int64_t rows_cap;           // rows of o (checked build)
  int32_t* dev_err;
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st);

// diagnostic: padded grouped rows -> expert-sorted dense rows
struct UnpadArgs {
  const uint8_t* src_q;       // [rows_cap, qbytes]
  const uint8_t* src_sf;      // tile layout, cols/128 groups4
  const int32_t* pad_row;     // [rows]
  const int32_t* expanded_row_idx;  // [rows]
  int64_t rows, cols;         // cols: elements of a row (cols / 32 scale groups)
  int64_t qbytes;             // bytes of a row of codes: cols, or cols / 2 for packed FP4
  int64_t src_stride;         // bytes between rows of src_q (0: qbytes)
  uint8_t* dst_q;             // [rows, qbytes]
  uint8_t* dst_sf;            // [rows, cols/32]
  int64_t rows_cap;           // rows of src_q (checked build)
  int32_t* dev_err;
};
cudaError_t launch_unpad(const UnpadArgs& a, cudaStream_t st);

// SMs of the current device (queried once per device)
int num_sms();
// one CTA waits on an mbarrier that nothing completes, gives up after
// limit_ns and raises MM_DEVERR_TIMEOUT (the bounded-wait failure path)
cudaError_t launch_selftest_wait_timeout(uint64_t limit_ns, int32_t* dev_err, cudaStream_t st);

// ---- C-ABI helpers shared by the entry points (abi.cu) -------------------
// One stage of one call for mm_timing_read: the constructor records the
// begin event on the stream (while timing is enabled), finish() the end
// event and adds the number of kernels the stage launched.
struct StageScope {
  int stage;
  cudaStream_t st;
  bool active;
  StageScope(int s, cudaStream_t stream);
  void finish(int kernels);
};

// Argument checks of mm_moe_init_routing that do not involve the workspace
// (also used by mm_moe_init_routing_noalloc).
mm_status validate_init_routing(const void* x, int x_dtype, const int32_t* expert_idx, int64_t num_rows,
                                int64_t h, int64_t k, int64_t expert_num, int quant_mode, int expert_tokens_num_type,
                                const void* expanded_x, const uint8_t* expanded_scale);
// element format of expanded_x for a quant mode (-1: copy)
int init_routing_out_fmt(int quant_mode);

}  // namespace mm
