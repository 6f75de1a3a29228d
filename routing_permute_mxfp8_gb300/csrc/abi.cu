// C-ABI entry points of libmm_moe: argument checks (before anything is
// enqueued), workspace carving and the launch sequence of each operation.
#include <float.h>
#include <math.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "mm_route.cuh"

using namespace mm;

namespace {

constexpr int64_t kSortLimit = 16777215;  // permute article, 约束说明

// Carves 256-byte aligned pieces out of a workspace; with base == nullptr it
// only adds up the sizes.
struct Carver {
  uint8_t* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  template <typename T>
  T* take(int64_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += (size_t)round_up(count * (int64_t)sizeof(T), 256);
    return p;
  }
};

bool is_src_dtype(int dt) { return dt == MM_DT_BFLOAT16 || dt == MM_DT_FLOAT16 || dt == MM_DT_FLOAT32; }
int dt_size(int dt) { return dt == MM_DT_FLOAT32 ? 4 : 2; }
bool is_fp8(int64_t dt) { return dt == MM_DT_FP8_E4M3FN || dt == MM_DT_FP8_E5M2; }
// expert weight types: FP8 (A8W8-FP) or FP4 E2M1 (A8W4-FP)
bool is_mx_weight(int64_t dt) { return is_fp8(dt) || dt == MM_DT_FP4_E2M1; }
int quant_fmt(int quant_mode) {
  if (quant_mode == MM_QUANT_MXFP4_E2M1) return MM_DT_FP4_E2M1;
  return quant_mode == MM_QUANT_MXFP8_E5M2 ? MM_DT_FP8_E5M2
                                           : (quant_mode == MM_QUANT_MXFP8_E4M3FN ? MM_DT_FP8_E4M3FN : -1);
}
mm_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MM_OK : MM_ERR_CUDA; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// ---- mm_moe_init_routing / mm_moe_token_permute share the routing part ----
struct RoutingWs {
  int32_t* hist;
  int32_t* offsets;
  int32_t* exp_idx;
};

RoutingWs carve_routing(Carver& c, const RoutePlan& p) {
  RoutingWs w;
  w.hist = c.take<int32_t>((int64_t)p.num_experts * p.units);
  w.offsets = c.take<int32_t>(route_offsets_words(p.num_experts));
  w.exp_idx = c.take<int32_t>(p.rows);
  return w;
}

// ---- mm_mega_moe ----
struct MegaDims {
  int64_t bs, h, k, e, inter, s, rows, rows_cap;
  int64_t aw_max;  // widest A_hat: 2I (gelu keeps the whole Linear1 output)
};

struct MegaWs {
  int32_t *hist, *offsets, *seg_rows, *seg_mprefix, *exp_idx, *pad_row, *pad_inv;
  uint8_t *xq, *xsf, *aq, *asf;
  __nv_bfloat16* o;
  uint8_t *wsf1, *wsf2, *swsf1, *swsf2;
};

MegaDims mega_dims(int64_t bs, int64_t h, int64_t k, int64_t e, int64_t inter, int64_t s) {
  MegaDims d;
  d.bs = bs;
  d.h = h;
  d.k = k;
  d.e = e;
  d.inter = inter;
  d.s = s;
  d.rows = bs * k;
  d.aw_max = 2 * inter;
  // each segment pads to whole 128-row tiles
  d.rows_cap = kBM * (ceil_div(d.rows, kBM) + e) + s * round_up(bs, kBM);
  return d;
}

MegaWs carve_mega(Carver& c, const MegaDims& d, const RoutePlan& p, int wscale_layout) {
  MegaWs w;
  const int64_t nseg = d.e + d.s;
  w.hist = c.take<int32_t>((int64_t)p.num_experts * p.units);
  w.offsets = c.take<int32_t>(route_offsets_words((int)d.e));
  w.seg_rows = c.take<int32_t>(nseg);
  w.seg_mprefix = c.take<int32_t>(nseg + 1);
  w.exp_idx = c.take<int32_t>(d.rows);
  w.pad_row = c.take<int32_t>(d.rows);
  w.pad_inv = c.take<int32_t>(d.rows_cap);
  w.xq = c.take<uint8_t>(d.rows_cap * d.h);
  w.xsf = c.take<uint8_t>(d.rows_cap / kBM * (d.h / 128) * kSfChunk);
  w.aq = c.take<uint8_t>(d.rows_cap * d.aw_max);
  w.asf = c.take<uint8_t>(d.rows_cap / kBM * (d.aw_max / 128) * kSfChunk);
  w.o = c.take<__nv_bfloat16>(d.rows_cap * d.h);
  w.wsf1 = w.wsf2 = w.swsf1 = w.swsf2 = nullptr;
  if (wscale_layout == MM_WSCALE_ROWS) {
    w.wsf1 = c.take<uint8_t>(d.e * 2 * prepared_npairs(2 * d.inter, 1) * (d.h / 128) * kSfChunk);
    w.wsf2 = c.take<uint8_t>(d.e * 2 * prepared_npairs(d.h, 2) * (d.aw_max / 128) * kSfChunk);
    if (d.s > 0) {
      w.swsf1 = c.take<uint8_t>(d.s * 2 * prepared_npairs(2 * d.inter, 1) * (d.h / 128) * kSfChunk);
      w.swsf2 = c.take<uint8_t>(d.s * 2 * prepared_npairs(d.h, 2) * (d.aw_max / 128) * kSfChunk);
    }
  }
  return w;
}

mm_status check_mega_shapes(int64_t bs, int64_t h, int64_t k, int64_t e, int64_t inter, int64_t s) {
  if (bs < 0 || h <= 0 || k <= 0 || e <= 0 || inter <= 0 || s < 0) return MM_ERR_INVALID_ARG;
  if (k > 32 || k > e || e > 2048 || s > 4) return MM_ERR_INVALID_ARG;
  if (bs * k >= kSortLimit) return MM_ERR_INVALID_ARG;
  if (h % 128 != 0 || inter % 128 != 0) return MM_ERR_UNSUPPORTED;
  if (h < 256) return MM_ERR_UNSUPPORTED;
  return MM_OK;
}

}  // namespace

namespace mm {

// ---- stage timing (diagnostic, off by default) ----------------------------
// While enabled, every entry point records a CUDA event pair around each of
// its stages on the caller's stream; mm_timing_read sums the device time.
// Launch counts are kept whether or not timing is on.
struct StageTimer {
  std::mutex mu;
  bool on = false;
  uint32_t mask = (1u << MM_STAGE_COUNT) - 1;  // stages that record events
  std::vector<cudaEvent_t> pool;
  std::vector<cudaEvent_t> open[MM_STAGE_COUNT];  // begin, end, begin, end, ...
  int64_t launches[MM_STAGE_COUNT] = {0};
};
StageTimer& timer() {
  static StageTimer t;
  return t;
}

static cudaEvent_t take_event(StageTimer& t) {
  if (!t.pool.empty()) {
    cudaEvent_t ev = t.pool.back();
    t.pool.pop_back();
    return ev;
  }
  cudaEvent_t ev = nullptr;
  cudaEventCreate(&ev);
  return ev;
}

StageScope::StageScope(int s, cudaStream_t stream) : stage(s), st(stream), active(false) {
  StageTimer& t = timer();
  std::lock_guard<std::mutex> g(t.mu);
  if (t.on && ((t.mask >> stage) & 1u)) {
    cudaEvent_t ev = take_event(t);
    if (ev && cudaEventRecord(ev, st) == cudaSuccess) {
      t.open[stage].push_back(ev);
      active = true;
    }
  }
}

void StageScope::finish(int kernels) {
  StageTimer& t = timer();
  std::lock_guard<std::mutex> g(t.mu);
  t.launches[stage] += kernels;
  if (active) {
    cudaEvent_t ev = take_event(t);
    if (ev && cudaEventRecord(ev, st) == cudaSuccess) {
      t.open[stage].push_back(ev);
    } else {
      t.pool.push_back(t.open[stage].back());
      t.open[stage].pop_back();
    }
    active = false;
  }
}

mm_status validate_init_routing(const void* x, int x_dtype, const int32_t* expert_idx, int64_t num_rows,
                                int64_t h, int64_t k, int64_t expert_num, int quant_mode, int expert_tokens_num_type,
                                const void* expanded_x, const uint8_t* expanded_scale) {
  if (num_rows < 0 || k <= 0 || expert_num <= 0 || expert_num > 10240) return MM_ERR_INVALID_ARG;
  if (num_rows * k >= kSortLimit) return MM_ERR_INVALID_ARG;
  if (h <= 0 || !is_src_dtype(x_dtype)) return MM_ERR_INVALID_ARG;
  // quantMode -1, 2 / 3 (MXFP8) and 9 (MXFP4 E2M1, two codes per byte)
  if (quant_mode != MM_QUANT_NONE && quant_mode != MM_QUANT_MXFP8_E5M2 && quant_mode != MM_QUANT_MXFP8_E4M3FN &&
      quant_mode != MM_QUANT_MXFP4_E2M1)
    return MM_ERR_UNSUPPORTED;
  if (expert_tokens_num_type != 0 && expert_tokens_num_type != 1) return MM_ERR_UNSUPPORTED;
  const bool quant = quant_mode != MM_QUANT_NONE;
  if (quant ? (h % 16 != 0) : ((h * dt_size(x_dtype)) % 16 != 0)) return MM_ERR_UNSUPPORTED;
  if (num_rows * k == 0) return MM_OK;  // nothing is read or written but the counts
  if (!x || !expert_idx || !expanded_x || (quant && !expanded_scale)) return MM_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(expanded_x)) return MM_ERR_INVALID_ARG;
  return MM_OK;
}

int init_routing_out_fmt(int quant_mode) { return quant_fmt(quant_mode); }

}  // namespace mm

namespace {

// The activation and its activation_params (MegaMoE parameter table,
// "activation_params"): swiglu / swiglustep [] or [clamp]; swigluoai [] or
// [clamp, alpha, beta] (alpha 1.702, beta 1.0 by default); situglu [],
// [beta] or [beta, linear_beta] (beta 1.0 by default); gelu exactly [FLT_MAX]
// (a placeholder).  A clamp of 0 or the float maximum disables clamping;
// a clamp must be >= 0 and not NaN, alpha and beta finite, the situglu
// betas finite and > 0.
struct ActSpec {
  int kind = MM_ACT_SWIGLU;
  float c = INFINITY, alpha = 1.702f, beta = 1.0f, beta_lin = 0.0f;
};

mm_status parse_activation(const char* act, const float* p, int64_t n, ActSpec* out) {
  ActSpec a;
  if (n < 0 || (n > 0 && !p)) return MM_ERR_INVALID_ARG;
  const char* name = act ? act : "swiglu";
  auto clamp_of = [](float c, float* dst) {
    if (!(c >= 0.0f)) return false;  // negative or NaN
    *dst = (c == 0.0f || c >= FLT_MAX) ? INFINITY : c;
    return true;
  };
  if (strcmp(name, "swiglu") == 0 || strcmp(name, "swiglustep") == 0) {
    a.kind = name[6] == 0 ? MM_ACT_SWIGLU : MM_ACT_SWIGLUSTEP;
    if (n > 1) return MM_ERR_INVALID_ARG;
    if (n == 1 && !clamp_of(p[0], &a.c)) return MM_ERR_INVALID_ARG;
  } else if (strcmp(name, "swigluoai") == 0) {
    a.kind = MM_ACT_SWIGLUOAI;
    if (n != 0 && n != 3) return MM_ERR_INVALID_ARG;
    if (n == 3) {
      if (!clamp_of(p[0], &a.c) || !isfinite(p[1]) || !isfinite(p[2])) return MM_ERR_INVALID_ARG;
      a.alpha = p[1];
      a.beta = p[2];
    }
  } else if (strcmp(name, "situglu") == 0) {
    a.kind = MM_ACT_SITUGLU;
    if (n > 2) return MM_ERR_INVALID_ARG;
    if (n >= 1) a.beta = p[0];
    if (n == 2) a.beta_lin = p[1];
    if (!(isfinite(a.beta) && a.beta > 0.0f)) return MM_ERR_INVALID_ARG;
    if (n == 2 && !(isfinite(a.beta_lin) && a.beta_lin > 0.0f)) return MM_ERR_INVALID_ARG;
  } else if (strcmp(name, "gelu") == 0) {
    a.kind = MM_ACT_GELU;
    if (n != 1 || p[0] != FLT_MAX) return MM_ERR_INVALID_ARG;
  } else {
    return MM_ERR_UNSUPPORTED;
  }
  *out = a;
  return MM_OK;
}

}  // namespace

extern "C" {

const char* mm_status_string(int status) {
  switch (status) {
    case MM_OK: return "ok";
    case MM_ERR_INVALID_ARG: return "invalid argument";
    case MM_ERR_UNSUPPORTED: return "unsupported option";
    case MM_ERR_WORKSPACE: return "workspace too small";
    case MM_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int mm_version(void) { return 100; }

mm_status mm_timing_enable(int on) {
  StageTimer& t = timer();
  std::lock_guard<std::mutex> g(t.mu);
  t.on = on != 0;
  return MM_OK;
}

int mm_checked_build(void) { return kChecked ? 1 : 0; }

mm_status mm_set_routing_path(int path) {
  if (path < MM_ROUTE_AUTO || path > MM_ROUTE_KERNELS) return MM_ERR_INVALID_ARG;
  set_route_path(path);
  return MM_OK;
}

mm_status mm_timing_select(uint32_t stage_mask) {
  if (stage_mask >> MM_STAGE_COUNT) return MM_ERR_INVALID_ARG;
  StageTimer& t = timer();
  std::lock_guard<std::mutex> g(t.mu);
  t.mask = stage_mask;
  return MM_OK;
}

mm_status mm_timing_read(double* stage_ms, int64_t* stage_launches, int n) {
  if (n < 0 || (n > 0 && (!stage_ms || !stage_launches))) return MM_ERR_INVALID_ARG;
  StageTimer& t = timer();
  std::lock_guard<std::mutex> g(t.mu);
  mm_status st = MM_OK;
  for (int s = 0; s < MM_STAGE_COUNT; ++s) {
    double ms = 0.0;
    std::vector<cudaEvent_t>& v = t.open[s];
    for (size_t i = 0; i + 1 < v.size(); i += 2) {
      float f = 0.f;
      if (cudaEventSynchronize(v[i + 1]) != cudaSuccess || cudaEventElapsedTime(&f, v[i], v[i + 1]) != cudaSuccess)
        st = MM_ERR_CUDA;
      ms += f;
    }
    for (cudaEvent_t ev : v) t.pool.push_back(ev);
    v.clear();
    if (s < n) {
      stage_ms[s] = ms;
      stage_launches[s] = t.launches[s];
    }
    t.launches[s] = 0;
  }
  return st;
}

// ------------------------------------------------------------------------
mm_status mm_moe_init_routing_workspace_size(int64_t num_rows, int64_t k, int64_t expert_num, size_t* bytes) {
  if (!bytes || num_rows < 0 || k <= 0 || expert_num <= 0 || expert_num > 10240) return MM_ERR_INVALID_ARG;
  if (num_rows * k >= kSortLimit) return MM_ERR_INVALID_ARG;
  Carver c(nullptr);
  carve_routing(c, route_plan(num_rows * k, (int)expert_num));
  *bytes = c.off;
  return MM_OK;
}

mm_status mm_moe_init_routing_v3_workspace_size(int64_t num_rows, int64_t k, int64_t expert_num, size_t* bytes) {
  mm_status s = mm_moe_init_routing_workspace_size(num_rows, k, expert_num, bytes);
  if (s == MM_OK) *bytes += (size_t)round_up(expert_num * (int64_t)sizeof(int64_t), 256);  // key_value counts
  return s;
}

// MoeInitRoutingV3, Dropless, with the active expert range [start, end)
// (activeExpertRangeOptional; computation step 6) and the three count
// types; mm_moe_init_routing is the full range with types 0 / 1.
static mm_status init_routing_impl(bool v3, const void* x, int x_dtype, const int32_t* expert_idx, int64_t num_rows,
                                   int64_t h, int64_t k, int64_t expert_num, int64_t start, int64_t end,
                                   int quant_mode, int expert_tokens_num_type, void* expanded_x,
                                   uint8_t* expanded_scale, int32_t* expanded_row_idx, int32_t* sorted_row_idx,
                                   int64_t* expert_tokens, void* workspace, size_t workspace_bytes,
                                   int32_t* dev_err, void* stream) {
  size_t need = 0;
  mm_status s = v3 ? mm_moe_init_routing_v3_workspace_size(num_rows, k, expert_num, &need)
                   : mm_moe_init_routing_workspace_size(num_rows, k, expert_num, &need);
  if (s != MM_OK) return s;
  if (start < 0 || end <= start || end > expert_num) return MM_ERR_INVALID_ARG;
  const bool key_value = expert_tokens_num_type == 2;
  if (key_value && !v3) return MM_ERR_UNSUPPORTED;
  if (key_value && expert_num > 5120) return MM_ERR_INVALID_ARG;
  s = validate_init_routing(x, x_dtype, expert_idx, num_rows, h, k, expert_num, quant_mode,
                            key_value ? 1 : expert_tokens_num_type, expanded_x, expanded_scale);
  if (s != MM_OK) return s;
  const int64_t rows = num_rows * k;
  const int64_t ne = end - start;  // experts of the active range
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows == 0)  // no rows: every expert's count (and the cumsum) is 0
    return expert_tokens ? cuda_status(cudaMemsetAsync(
                               expert_tokens, 0, (size_t)(key_value ? 2 * expert_num : ne) * sizeof(int64_t), st))
                         : MM_OK;
  if (!workspace || workspace_bytes < need) return MM_ERR_WORKSPACE;
  const RoutePlan plan = route_plan(rows, (int)ne);
  Carver c(workspace);
  RoutingWs w = carve_routing(c, plan);
  int64_t* kv_counts = key_value ? c.take<int64_t>(expert_num) : nullptr;
  RouteOutputs o;
  o.expanded_row_idx = expanded_row_idx ? expanded_row_idx : w.exp_idx;
  o.sorted_row_idx = sorted_row_idx;
  o.expert_tokens = key_value ? (expert_tokens ? kv_counts : nullptr) : expert_tokens;
  o.tokens_cumsum = expert_tokens_num_type == 0;
  o.key_off = (int)start;
  o.id_limit = expert_num;
  StageScope sr(MM_STAGE_ROUTE, st);
  int nl = 0;
  cudaError_t e = launch_route(plan, expert_idx, false, w.hist, w.offsets, o, dev_err, st, &nl);
  if (e == cudaSuccess && key_value && expert_tokens) {
    e = launch_key_value_counts(kv_counts, (int)ne, start, expert_num, expert_tokens, st);
    ++nl;
  }
  sr.finish(nl);
  if (e != cudaSuccess) return MM_ERR_CUDA;
  PermuteArgs a = {};
  a.src = x;
  a.src_dtype = x_dtype;
  a.n = num_rows;
  a.h = h;
  a.k = (int)k;
  a.dest = o.expanded_row_idx;
  a.dest_limit = rows;
  a.out_fmt = quant_fmt(quant_mode);
  a.out = expanded_x;
  a.scales = expanded_scale;
  a.scale_cols = round_up(ceil_div(h, 32), 2);
  a.dev_err = dev_err;
  StageScope sd(MM_STAGE_DISPATCH, st);
  e = launch_permute(a, st);
  sd.finish(1);
  return cuda_status(e);
}

mm_status mm_moe_init_routing(const void* x, int x_dtype, const int32_t* expert_idx, int64_t num_rows, int64_t h,
                              int64_t k, int64_t expert_num, int quant_mode, int expert_tokens_num_type,
                              void* expanded_x, uint8_t* expanded_scale, int32_t* expanded_row_idx,
                              int32_t* sorted_row_idx, int64_t* expert_tokens, void* workspace,
                              size_t workspace_bytes, int32_t* dev_err, void* stream) {
  if (expert_num <= 0 || expert_num > 10240) return MM_ERR_INVALID_ARG;
  return init_routing_impl(false, x, x_dtype, expert_idx, num_rows, h, k, expert_num, 0, expert_num, quant_mode,
                           expert_tokens_num_type, expanded_x, expanded_scale, expanded_row_idx, sorted_row_idx,
                           expert_tokens, workspace, workspace_bytes, dev_err, stream);
}

mm_status mm_moe_init_routing_v3(const void* x, int x_dtype, const int32_t* expert_idx, int64_t num_rows, int64_t h,
                                 int64_t k, int64_t expert_num, int64_t active_expert_start,
                                 int64_t active_expert_end, int quant_mode, int expert_tokens_num_type,
                                 void* expanded_x, uint8_t* expanded_scale, int32_t* expanded_row_idx,
                                 int32_t* sorted_row_idx, int64_t* expert_tokens, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_err, void* stream) {
  return init_routing_impl(true, x, x_dtype, expert_idx, num_rows, h, k, expert_num, active_expert_start,
                           active_expert_end, quant_mode, expert_tokens_num_type, expanded_x, expanded_scale,
                           expanded_row_idx, sorted_row_idx, expert_tokens, workspace, workspace_bytes, dev_err,
                           stream);
}

// ------------------------------------------------------------------------
int64_t mm_moe_token_permute_out_rows(int64_t num_indices, int64_t num_out_tokens) {
  if (num_out_tokens == 0) return num_indices;
  if (num_out_tokens > 0) return num_out_tokens < num_indices ? num_out_tokens : num_indices;
  const int64_t m = num_indices + num_out_tokens;
  return m > 0 ? m : 0;
}

mm_status mm_moe_token_permute_workspace_size(int64_t num_indices, int64_t num_experts, size_t* bytes) {
  if (!bytes || num_indices < 0 || num_indices >= kSortLimit || num_experts <= 0 || num_experts > 10240)
    return MM_ERR_INVALID_ARG;
  Carver c(nullptr);
  carve_routing(c, route_plan(num_indices, (int)num_experts));
  *bytes = c.off;
  return MM_OK;
}

mm_status mm_moe_token_permute(const void* tokens, int tokens_dtype, const void* indices, int indices_dtype,
                               int64_t n, int64_t topk, int64_t h, int64_t num_experts, int64_t num_out_tokens,
                               int padded_mode, int quant_mode, void* permuted_tokens, uint8_t* expanded_scale,
                               int32_t* sorted_indices, void* workspace, size_t workspace_bytes,
                               int32_t* dev_err, void* stream) {
  if (n < 0 || topk <= 0 || h <= 0 || !is_src_dtype(tokens_dtype)) return MM_ERR_INVALID_ARG;
  if (indices_dtype != MM_DT_INT32 && indices_dtype != MM_DT_INT64) return MM_ERR_INVALID_ARG;
  size_t need = 0;
  const int64_t f = n * topk;
  mm_status s = mm_moe_token_permute_workspace_size(f, num_experts, &need);
  if (s != MM_OK) return s;
  if (padded_mode != 0) return MM_ERR_UNSUPPORTED;
  if (quant_mode != MM_QUANT_NONE && quant_mode != MM_QUANT_MXFP8_E5M2 && quant_mode != MM_QUANT_MXFP8_E4M3FN &&
      quant_mode != MM_QUANT_MXFP4_E2M1)
    return MM_ERR_UNSUPPORTED;
  const bool quant = quant_mode != MM_QUANT_NONE;
  if (quant && tokens_dtype == MM_DT_FLOAT32) return MM_ERR_UNSUPPORTED;  // the article: fp16 / bf16
  if (quant ? (h % 16 != 0) : ((h * dt_size(tokens_dtype)) % 16 != 0)) return MM_ERR_UNSUPPORTED;
  if (f == 0) return MM_OK;
  const int64_t m = mm_moe_token_permute_out_rows(f, num_out_tokens);
  if (!tokens || !indices || !sorted_indices || (m > 0 && !permuted_tokens) || (quant && m > 0 && !expanded_scale))
    return MM_ERR_INVALID_ARG;
  if (!aligned16(tokens) || (m > 0 && !aligned16(permuted_tokens))) return MM_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < need) return MM_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const RoutePlan plan = route_plan(f, (int)num_experts);
  Carver c(workspace);
  RoutingWs w = carve_routing(c, plan);
  RouteOutputs o;
  o.expanded_row_idx = sorted_indices;
  StageScope sr(MM_STAGE_ROUTE, st);
  int nl = 0;
  cudaError_t e =
      launch_route(plan, indices, indices_dtype == MM_DT_INT64, w.hist, w.offsets, o, dev_err, st, &nl);
  sr.finish(nl);
  if (e != cudaSuccess) return MM_ERR_CUDA;
  if (m == 0) return MM_OK;
  PermuteArgs a = {};
  a.src = tokens;
  a.src_dtype = tokens_dtype;
  a.n = n;
  a.h = h;
  a.k = (int)topk;
  a.dest = sorted_indices;
  a.dest_limit = m;
  a.out_fmt = quant_fmt(quant_mode);
  a.out = permuted_tokens;
  a.scales = expanded_scale;
  a.scale_cols = round_up(ceil_div(h, 32), 2);
  a.dev_err = dev_err;
  StageScope sd(MM_STAGE_DISPATCH, st);
  e = launch_permute(a, st);
  sd.finish(1);
  return cuda_status(e);
}

// ------------------------------------------------------------------------
mm_status mm_mega_moe_workspace_size(int64_t bs, int64_t h, int64_t k, int64_t moe_expert_num,
                                     int64_t intermediate, int64_t shared_expert_num, int weight_scale_layout,
                                     size_t* bytes) {
  if (!bytes) return MM_ERR_INVALID_ARG;
  mm_status s = check_mega_shapes(bs, h, k, moe_expert_num, intermediate, shared_expert_num);
  if (s != MM_OK) return s;
  if (weight_scale_layout != MM_WSCALE_ROWS && weight_scale_layout != MM_WSCALE_PREPARED)
    return MM_ERR_INVALID_ARG;
  const MegaDims d = mega_dims(bs, h, k, moe_expert_num, intermediate, shared_expert_num);
  Carver c(nullptr);
  carve_mega(c, d, route_plan(d.rows, (int)d.e), weight_scale_layout);
  *bytes = c.off;
  return MM_OK;
}

// The MegaMoE step; rows_out: the expert side of expert parallelism
// (top-K 1, no gating weights, no shared experts): GEMM2 writes each input
// row's expert output to y at that row's position and there is no combine.
static mm_status mega_moe_impl(bool rows_out, const void* x, const uint8_t* x_scales, const int32_t* topk_ids,
                               const void* topk_weights, int topk_weights_dtype,
                      const uint8_t* weight1, const uint8_t* weight2, const uint8_t* weight_scales1,
                      const uint8_t* weight_scales2, int weight_dtype, int weight_scale_layout,
                      const uint8_t* shared_weight1, const uint8_t* shared_weight2,
                      const uint8_t* shared_weight_scales1, const uint8_t* shared_weight_scales2,
                      int shared_weight_dtype, int64_t shared_expert_num, int64_t bs, int64_t h, int64_t k,
                      int64_t moe_expert_num, int64_t ep_world_size, int64_t intermediate,
                      int64_t max_recv_token_num, int64_t dispatch_quant_mode, int64_t dispatch_quant_out_dtype,
                      int64_t shared_quant_out_dtype, int64_t combine_quant_mode, const char* activation,
                      const float* activation_params, int64_t n_activation_params, void* y,
                      int32_t* expert_token_nums, int32_t* expanded_row_idx, uint8_t* act_q, uint8_t* act_scale,
                      uint8_t* dispatch_q, uint8_t* dispatch_scale, void* workspace, size_t workspace_bytes,
                      int32_t* dev_err, void* stream) {
  size_t need = 0;
  mm_status s = mm_mega_moe_workspace_size(bs, h, k, moe_expert_num, intermediate, shared_expert_num,
                                           weight_scale_layout, &need);
  if (s != MM_OK) return s;
  if (ep_world_size != 1) return MM_ERR_UNSUPPORTED;
  if (combine_quant_mode != 0) return MM_ERR_UNSUPPORTED;
  // 4: MX quantisation inside the operator; 0: pre-quantised pass-through
  // (x holds codes of dispatch_quant_out_dtype, x_scales its E8M0 scales).
  // An FP4 E2M1 dispatch is the A4W4-FP scenario: FP4 routed weights, and
  // A_hat re-quantised to MXFP8 E4M3 so that GEMM2 is A8W4.
  if (dispatch_quant_mode != 4 && dispatch_quant_mode != 0) return MM_ERR_UNSUPPORTED;
  if (!is_mx_weight(dispatch_quant_out_dtype) || !is_mx_weight(weight_dtype)) return MM_ERR_UNSUPPORTED;
  const bool a4w4 = dispatch_quant_out_dtype == MM_DT_FP4_E2M1;
  if (a4w4 && weight_dtype != MM_DT_FP4_E2M1) return MM_ERR_UNSUPPORTED;
  const int act_fmt = a4w4 ? MM_DT_FP8_E4M3FN : (int)dispatch_quant_out_dtype;
  // the shared experts' own input type (the parameter table's
  // sharedExpertQuantOutDtype; 0: the dispatch type), with the same rules
  if (shared_quant_out_dtype != 0 && !is_mx_weight(shared_quant_out_dtype)) return MM_ERR_UNSUPPORTED;
  const int sx_fmt = shared_expert_num > 0 && shared_quant_out_dtype != 0 ? (int)shared_quant_out_dtype
                                                                          : (int)dispatch_quant_out_dtype;
  if (dispatch_quant_mode == 0 && sx_fmt != dispatch_quant_out_dtype) return MM_ERR_INVALID_ARG;
  const int act_fmt_sh = sx_fmt == MM_DT_FP4_E2M1 ? MM_DT_FP8_E4M3FN : sx_fmt;
  // X_hat rows: FP8 (h bytes) or packed FP4 (h / 2); an FP8 stride for both
  // when routed and shared rows differ in width
  const int64_t xw = a4w4 ? h / 2 : h;
  const int64_t xstride = (sx_fmt == MM_DT_FP4_E2M1) == a4w4 ? xw : h;
  if (shared_expert_num > 0 && !is_mx_weight(shared_weight_dtype)) return MM_ERR_UNSUPPORTED;
  if (bs > 0 && (dispatch_quant_mode == 0) != (x_scales != nullptr)) return MM_ERR_INVALID_ARG;
  ActSpec act;
  s = parse_activation(activation, activation_params, n_activation_params, &act);
  if (s != MM_OK) return s;
  const int64_t aw = act.kind == MM_ACT_GELU ? 2 * intermediate : intermediate;
  if (!rows_out && topk_weights_dtype != MM_DT_FLOAT32 && topk_weights_dtype != MM_DT_BFLOAT16)
    return MM_ERR_INVALID_ARG;
  const int64_t rows = bs * k;
  if (max_recv_token_num != 0 && max_recv_token_num < rows) return MM_ERR_INVALID_ARG;
  if (bs == 0)  // no tokens: Y is empty and every expert received 0 rows
    return expert_token_nums ? cuda_status(cudaMemsetAsync(expert_token_nums, 0,
                                                           (size_t)moe_expert_num * sizeof(int32_t),
                                                           static_cast<cudaStream_t>(stream)))
                             : MM_OK;
  if (!x || !topk_ids || (!topk_weights && !rows_out) || !weight1 || !weight2 || !weight_scales1 ||
      !weight_scales2 || !y)
    return MM_ERR_INVALID_ARG;
  if (shared_expert_num > 0 &&
      (!shared_weight1 || !shared_weight2 || !shared_weight_scales1 || !shared_weight_scales2))
    return MM_ERR_INVALID_ARG;
  if ((act_q == nullptr) != (act_scale == nullptr)) return MM_ERR_INVALID_ARG;
  if ((dispatch_q == nullptr) != (dispatch_scale == nullptr)) return MM_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || !aligned16(weight1) || !aligned16(weight2) ||
      !aligned16(weight_scales1) || !aligned16(weight_scales2) || (act_q && !aligned16(act_q)) ||
      (dispatch_q && !aligned16(dispatch_q)))
    return MM_ERR_INVALID_ARG;
  if (shared_expert_num > 0 && (!aligned16(shared_weight1) || !aligned16(shared_weight2) ||
                                !aligned16(shared_weight_scales1) || !aligned16(shared_weight_scales2)))
    return MM_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < need) return MM_ERR_WORKSPACE;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const MegaDims d = mega_dims(bs, h, k, moe_expert_num, intermediate, shared_expert_num);
  const RoutePlan plan = route_plan(d.rows, (int)d.e);
  Carver c(workspace);
  MegaWs w = carve_mega(c, d, plan, weight_scale_layout);
  cudaError_t e;

  // 0. weight scales into the GEMM tile layout (skipped when prepared once)
  const uint8_t *wsf1 = weight_scales1, *wsf2 = weight_scales2;
  const uint8_t *swsf1 = shared_weight_scales1, *swsf2 = shared_weight_scales2;
  if (weight_scale_layout == MM_WSCALE_ROWS) {
    StageScope sw(MM_STAGE_WSCALE, st);
    e = launch_prepare_wscales(weight_scales1, d.e, 2 * d.inter, d.h, 1, w.wsf1, st);
    if (e == cudaSuccess) e = launch_prepare_wscales(weight_scales2, d.e, d.h, aw, 2, w.wsf2, st);
    if (e == cudaSuccess && d.s > 0)
      e = launch_prepare_wscales(shared_weight_scales1, d.s, 2 * d.inter, d.h, 1, w.swsf1, st);
    if (e == cudaSuccess && d.s > 0)
      e = launch_prepare_wscales(shared_weight_scales2, d.s, d.h, aw, 2, w.swsf2, st);
    sw.finish(d.s > 0 ? 4 : 2);
    if (e != cudaSuccess) return MM_ERR_CUDA;
    wsf1 = w.wsf1;
    wsf2 = w.wsf2;
    swsf1 = w.swsf1;
    swsf2 = w.swsf2;
  }

  // 1. routing: stable counting sort, inverse map, counts, GEMM segment table
  RouteOutputs o;
  o.expanded_row_idx = expanded_row_idx ? expanded_row_idx : w.exp_idx;
  o.pad_row = w.pad_row;
  o.pad_limit = d.rows_cap;
  o.expert_token_nums = expert_token_nums;
  o.seg_rows = w.seg_rows;
  o.seg_mprefix = w.seg_mprefix;
  o.n_shared = (int)d.s;
  o.shared_rows = (int)d.bs;
  StageScope sr(MM_STAGE_ROUTE, st);
  int nl = 0;
  e = launch_route(plan, topk_ids, false, w.hist, w.offsets, o, dev_err, st, &nl);
  sr.finish(nl);
  if (e != cudaSuccess) return MM_ERR_CUDA;

  // 2. dispatch: MX quantisation of each token, stored at its K expert rows
  //    (and once per shared expert) in the padded grouped layout
  PermuteArgs pa = {};
  pa.src = x;
  pa.src_dtype = dispatch_quant_mode == 0 ? (int)dispatch_quant_out_dtype : MM_DT_BFLOAT16;
  pa.src_scales = x_scales;
  pa.n = d.bs;
  pa.h = d.h;
  pa.k = (int)d.k;
  pa.dest = w.pad_row;
  pa.dest_limit = d.rows_cap;
  pa.ids = topk_ids;
  pa.n_extra = (int)d.s;
  pa.extra_base = w.seg_mprefix + d.e;
  pa.out_fmt = (int)dispatch_quant_out_dtype;
  pa.out = w.xq;
  pa.out_stride = xstride;
  pa.scales = w.xsf;
  pa.scale_cols = 0;
  pa.dev_err = dev_err;
  pa.dest_inv = rows_out ? w.pad_inv : nullptr;
  const bool split = sx_fmt != dispatch_quant_out_dtype;  // the shared rows in their own type
  if (split) pa.n_extra = 0;
  StageScope sd(MM_STAGE_DISPATCH, st);
  e = launch_permute(pa, st);
  if (e == cudaSuccess && split) {
    PermuteArgs ps = pa;
    ps.k = 0;
    ps.dest = nullptr;
    ps.ids = nullptr;
    ps.dest_inv = nullptr;
    ps.n_extra = (int)d.s;
    ps.out_fmt = sx_fmt;
    e = launch_permute(ps, st);
  }
  sd.finish(split ? 2 : 1);
  if (e != cudaSuccess) return MM_ERR_CUDA;

  // 3. GEMM1 + swiglu + MX requantisation
  GemmLaunch g1 = {};
  g1.mode = 1;
  g1.a = w.xq;
  g1.rows_cap = d.rows_cap;
  g1.sfa = w.xsf;
  g1.b = weight1;
  g1.sfb = wsf1;
  g1.b_sh = shared_weight1;
  g1.sfb_sh = swsf1;
  g1.n_routed = (int)d.e;
  g1.n_shared = (int)d.s;
  g1.seg_rows = w.seg_rows;
  g1.seg_mprefix = w.seg_mprefix;
  g1.K = d.h;
  g1.N = 2 * d.inter;
  g1.a_fmt = (int)dispatch_quant_out_dtype;
  g1.a_fmt_sh = sx_fmt;
  g1.a_stride = xstride;
  g1.act_fmt = act_fmt;
  g1.act_fmt_sh = act_fmt_sh;
  g1.b_fmt = weight_dtype;
  g1.b_fmt_sh = shared_weight_dtype;
  g1.inter = (int)d.inter;
  g1.act = act.kind;
  g1.act_c = act.c;
  g1.act_alpha = act.alpha;
  g1.act_beta = act.beta;
  g1.act_beta_lin = act.beta_lin;
  g1.act_q = w.aq;
  g1.act_sf = w.asf;
  g1.dev_err = dev_err;
  StageScope s1(MM_STAGE_GEMM1, st);
  e = launch_gemm(g1, st);
  s1.finish(1);
  if (e != cudaSuccess) return MM_ERR_CUDA;

  // 4. GEMM2 -> bf16 expert rows
  GemmLaunch g2 = g1;
  g2.mode = 2;
  g2.a = w.aq;
  g2.a_fmt = act_fmt;
  g2.a_fmt_sh = act_fmt_sh;
  g2.a_stride = 0;
  g2.sfa = w.asf;
  g2.b = weight2;
  g2.sfb = wsf2;
  g2.b_sh = shared_weight2;
  g2.sfb_sh = swsf2;
  g2.K = aw;
  g2.N = d.h;
  g2.act_q = nullptr;
  g2.act_sf = nullptr;
  g2.out = rows_out ? static_cast<__nv_bfloat16*>(y) : w.o;
  g2.out_row = rows_out ? w.pad_inv : nullptr;
  g2.out_rows = d.rows;
  StageScope s2(MM_STAGE_GEMM2, st);
  e = launch_gemm(g2, st);
  s2.finish(1);
  if (e != cudaSuccess) return MM_ERR_CUDA;

  // 5. combine (the expert side of expert parallelism has none: its rows
  //    go back to their source ranks)
  if (!rows_out) {
    CombineArgs ca = {};
    ca.o = w.o;
    ca.pad_row = w.pad_row;
    ca.gate = topk_weights;
    ca.gate_bf16 = topk_weights_dtype == MM_DT_BFLOAT16;
    ca.n_shared = (int)d.s;
    ca.seg_mprefix = w.seg_mprefix;
    ca.n_routed = (int)d.e;
    ca.n = d.bs;
    ca.h = d.h;
    ca.k = (int)d.k;
    ca.y = static_cast<__nv_bfloat16*>(y);
    ca.rows_cap = d.rows_cap;
    ca.dev_err = dev_err;
    StageScope sc(MM_STAGE_COMBINE, st);
    e = launch_combine(ca, st);
    sc.finish(1);
    if (e != cudaSuccess) return MM_ERR_CUDA;
  }

  // optional diagnostic copies of X_hat and A_hat in expert-sorted order
  if (dispatch_q) {
    UnpadArgs ua = {};
    ua.src_q = w.xq;
    ua.src_sf = w.xsf;
    ua.pad_row = w.pad_row;
    ua.expanded_row_idx = o.expanded_row_idx;
    ua.rows = d.rows;
    ua.cols = d.h;
    ua.qbytes = xw;
    ua.src_stride = xstride;
    ua.dst_q = dispatch_q;
    ua.dst_sf = dispatch_scale;
    ua.rows_cap = d.rows_cap;
    ua.dev_err = dev_err;
    StageScope su(MM_STAGE_DIAG, st);
    e = launch_unpad(ua, st);
    su.finish(1);
    if (e != cudaSuccess) return MM_ERR_CUDA;
  }
  if (act_q) {
    UnpadArgs ua = {};
    ua.src_q = w.aq;
    ua.src_sf = w.asf;
    ua.pad_row = w.pad_row;
    ua.expanded_row_idx = o.expanded_row_idx;
    ua.rows = d.rows;
    ua.cols = aw;
    ua.qbytes = aw;
    ua.dst_q = act_q;
    ua.dst_sf = act_scale;
    ua.rows_cap = d.rows_cap;
    ua.dev_err = dev_err;
    StageScope su(MM_STAGE_DIAG, st);
    e = launch_unpad(ua, st);
    su.finish(1);
    if (e != cudaSuccess) return MM_ERR_CUDA;
  }
  return MM_OK;
}

mm_status mm_mega_moe(const void* x, const uint8_t* x_scales, const int32_t* topk_ids, const void* topk_weights,
                      int topk_weights_dtype, const uint8_t* weight1, const uint8_t* weight2,
                      const uint8_t* weight_scales1, const uint8_t* weight_scales2, int weight_dtype,
                      int weight_scale_layout, const uint8_t* shared_weight1, const uint8_t* shared_weight2,
                      const uint8_t* shared_weight_scales1, const uint8_t* shared_weight_scales2,
                      int shared_weight_dtype, int64_t shared_expert_num, int64_t bs, int64_t h, int64_t k,
                      int64_t moe_expert_num, int64_t ep_world_size, int64_t intermediate,
                      int64_t max_recv_token_num, int64_t dispatch_quant_mode, int64_t dispatch_quant_out_dtype,
                      int64_t shared_quant_out_dtype, int64_t combine_quant_mode, const char* activation,
                      const float* activation_params, int64_t n_activation_params, void* y,
                      int32_t* expert_token_nums, int32_t* expanded_row_idx, uint8_t* act_q, uint8_t* act_scale,
                      uint8_t* dispatch_q, uint8_t* dispatch_scale, void* workspace, size_t workspace_bytes,
                      int32_t* dev_err, void* stream) {
  return mega_moe_impl(false, x, x_scales, topk_ids, topk_weights, topk_weights_dtype, weight1, weight2,
                       weight_scales1, weight_scales2, weight_dtype, weight_scale_layout, shared_weight1,
                       shared_weight2, shared_weight_scales1, shared_weight_scales2, shared_weight_dtype,
                       shared_expert_num, bs, h, k, moe_expert_num, ep_world_size, intermediate, max_recv_token_num,
                       dispatch_quant_mode, dispatch_quant_out_dtype, shared_quant_out_dtype, combine_quant_mode,
                       activation,
                       activation_params, n_activation_params, y, expert_token_nums, expanded_row_idx, act_q,
                       act_scale, dispatch_q, dispatch_scale, workspace, workspace_bytes, dev_err, stream);
}

// ------------------------------------------------------------------------
// The expert side of expert parallelism (MegaMoE README, A8W8-FP stages 2-3
// on the rows a rank receives): GEMM1 + activation + GEMM2 of each row's
// local expert, the result written at the row's own position.
mm_status mm_moe_expert_ffn_workspace_size(int64_t rows, int64_t h, int64_t local_experts, int64_t intermediate,
                                           int weight_scale_layout, size_t* bytes) {
  return mm_mega_moe_workspace_size(rows, h, 1, local_experts, intermediate, 0, weight_scale_layout, bytes);
}

mm_status mm_moe_expert_ffn(const uint8_t* x, const uint8_t* x_scales, int x_dtype, const int32_t* expert_ids,
                            int64_t rows, int64_t h, const uint8_t* weight1, const uint8_t* weight2,
                            const uint8_t* weight_scales1, const uint8_t* weight_scales2, int weight_dtype,
                            int weight_scale_layout, int64_t local_experts, int64_t intermediate,
                            const char* activation, const float* activation_params, int64_t n_activation_params,
                            void* out, int32_t* expert_token_nums, void* workspace, size_t workspace_bytes,
                            int32_t* dev_err, void* stream) {
  return mega_moe_impl(true, x, x_scales, expert_ids, nullptr, 0,
                       weight1, weight2, weight_scales1, weight_scales2, weight_dtype, weight_scale_layout, nullptr,
                       nullptr, nullptr, nullptr, 0, 0, rows, h, 1, local_experts, 1, intermediate, 0, 0, x_dtype, 0, 0,
                       activation, activation_params, n_activation_params, out, expert_token_nums, nullptr, nullptr,
                       nullptr, nullptr, nullptr, workspace, workspace_bytes, dev_err, stream);
}

// ------------------------------------------------------------------------
// Expert parallelism (MegaMoE README, A8W8-FP stage 1 / stage 4 with
// epWorldSize > 1): the source-side dispatch and the combine; the exchange
// between ranks is the caller's collective.
mm_status mm_moe_ep_dispatch_workspace_size(int64_t num_rows, int64_t k, int64_t ep_world_size, size_t* bytes) {
  if (!bytes || num_rows < 0 || k <= 0 || k > 32 || ep_world_size <= 0 || ep_world_size > 10240)
    return MM_ERR_INVALID_ARG;
  if (num_rows * k >= kSortLimit) return MM_ERR_INVALID_ARG;
  Carver c(nullptr);
  carve_routing(c, route_plan(num_rows * k, (int)ep_world_size));
  *bytes = c.off;
  return MM_OK;
}

mm_status mm_moe_ep_dispatch(const void* x, int x_dtype, const int32_t* topk_ids, int64_t num_rows, int64_t h,
                             int64_t k, int64_t moe_expert_num, int64_t ep_world_size,
                             int64_t dispatch_quant_out_dtype, uint8_t* send_x, uint8_t* send_scales,
                             int32_t* send_expert, int64_t* rank_counts, int32_t* expanded_row_idx, void* workspace,
                             size_t workspace_bytes, int32_t* dev_err, void* stream) {
  size_t need = 0;
  mm_status s = mm_moe_ep_dispatch_workspace_size(num_rows, k, ep_world_size, &need);
  if (s != MM_OK) return s;
  if (moe_expert_num <= 0 || moe_expert_num % ep_world_size != 0 || k > moe_expert_num) return MM_ERR_INVALID_ARG;
  if (x_dtype != MM_DT_BFLOAT16 && x_dtype != MM_DT_FLOAT16) return MM_ERR_INVALID_ARG;
  if (!is_mx_weight(dispatch_quant_out_dtype)) return MM_ERR_UNSUPPORTED;  // FP8, or FP4 (A4W4-FP)
  if (h <= 0 || h % 128 != 0) return MM_ERR_UNSUPPORTED;
  const int64_t rows = num_rows * k;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows == 0)  // nothing to send: every rank receives 0 rows
    return rank_counts ? cuda_status(cudaMemsetAsync(rank_counts, 0, (size_t)ep_world_size * sizeof(int64_t), st))
                       : MM_OK;
  if (!x || !topk_ids || !send_x || !send_scales || !send_expert || !rank_counts || !expanded_row_idx)
    return MM_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(send_x)) return MM_ERR_INVALID_ARG;
  if (!workspace || workspace_bytes < need) return MM_ERR_WORKSPACE;
  // stable sort of the flattened ids by destination rank = id / (E / W);
  // within a rank the rows stay in (token, choice) order
  const RoutePlan plan = route_plan(rows, (int)ep_world_size);
  Carver c(workspace);
  RoutingWs w = carve_routing(c, plan);
  RouteOutputs o;
  o.expanded_row_idx = expanded_row_idx;
  o.expert_tokens = rank_counts;
  o.tokens_cumsum = 0;
  o.key_div = (int)(moe_expert_num / ep_world_size);
  o.sorted_rem = send_expert;
  StageScope sr(MM_STAGE_ROUTE, st);
  int nl = 0;
  cudaError_t e = launch_route(plan, topk_ids, false, w.hist, w.offsets, o, dev_err, st, &nl);
  sr.finish(nl);
  if (e != cudaSuccess) return MM_ERR_CUDA;
  // Q_MX of each token once, stored at its K positions of the send buffer
  PermuteArgs a = {};
  a.src = x;
  a.src_dtype = x_dtype;
  a.n = num_rows;
  a.h = h;
  a.k = (int)k;
  a.dest = expanded_row_idx;
  a.dest_limit = rows;
  a.ids = topk_ids;
  a.out_fmt = (int)dispatch_quant_out_dtype;
  a.out = send_x;
  a.scales = send_scales;
  a.scale_cols = h / 32;
  a.dev_err = dev_err;
  StageScope sd(MM_STAGE_DISPATCH, st);
  e = launch_permute(a, st);
  sd.finish(1);
  return cuda_status(e);
}

mm_status mm_moe_combine(const void* expert_rows, int expert_rows_dtype, const uint8_t* expert_scales,
                         const int32_t* row_idx, const void* topk_weights, int topk_weights_dtype, int64_t num_rows,
                         int64_t h, int64_t k, const void* shared_rows, int64_t n_shared, void* y, void* stream) {
  if (num_rows < 0 || h <= 0 || k <= 0 || n_shared < 0 || n_shared > 4 || k + n_shared > 36)
    return MM_ERR_INVALID_ARG;
  if (num_rows * k >= kSortLimit) return MM_ERR_INVALID_ARG;  // the dispatch's row limit
  if (topk_weights_dtype != MM_DT_FLOAT32 && topk_weights_dtype != MM_DT_BFLOAT16) return MM_ERR_INVALID_ARG;
  // bf16 rows, or MXFP8 rows of the combine exchange (combineQuantMode 3 / 4)
  const bool q = expert_rows_dtype != MM_DT_BFLOAT16;
  if (q && !is_fp8(expert_rows_dtype)) return MM_ERR_UNSUPPORTED;
  if (h % 8 != 0 || (q && h % 32 != 0)) return MM_ERR_UNSUPPORTED;
  if (num_rows == 0) return MM_OK;
  if (!expert_rows || !row_idx || !topk_weights || !y || !aligned16(expert_rows) || !aligned16(y))
    return MM_ERR_INVALID_ARG;
  if (q && !expert_scales) return MM_ERR_INVALID_ARG;
  if (n_shared > 0 && (!shared_rows || !aligned16(shared_rows))) return MM_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  StageScope sc(MM_STAGE_COMBINE, st);
  const cudaError_t e = launch_combine_rows(
      q ? nullptr : static_cast<const __nv_bfloat16*>(expert_rows), row_idx, topk_weights,
      topk_weights_dtype == MM_DT_BFLOAT16, num_rows, h, (int)k, static_cast<const __nv_bfloat16*>(shared_rows),
      (int)n_shared, static_cast<__nv_bfloat16*>(y), st, q ? static_cast<const uint8_t*>(expert_rows) : nullptr,
      q ? expert_scales : nullptr, q ? expert_rows_dtype : 0);
  sc.finish(1);
  return cuda_status(e);
}

// ------------------------------------------------------------------------
mm_status mm_selftest_wait_timeout(int64_t limit_ns, int32_t* dev_err, void* stream) {
  if (limit_ns <= 0 || limit_ns > 10000000000ll || !dev_err) return MM_ERR_INVALID_ARG;
  return cuda_status(launch_selftest_wait_timeout((uint64_t)limit_ns, dev_err, static_cast<cudaStream_t>(stream)));
}

// ------------------------------------------------------------------------
mm_status mm_prepared_weight_scales_size(int which, int64_t experts, int64_t n_out, int64_t k_red,
                                         size_t* bytes) {
  if (!bytes || (which != 1 && which != 2) || experts <= 0 || n_out <= 0 || k_red <= 0 || k_red % 128 != 0)
    return MM_ERR_INVALID_ARG;
  if (which == 1 && n_out % 256 != 0) return MM_ERR_INVALID_ARG;  // 2I with I a multiple of 128
  *bytes = (size_t)(experts * 2 * prepared_npairs(n_out, which) * (k_red / 128) * kSfChunk);
  return MM_OK;
}

mm_status mm_prepare_weight_scales(const uint8_t* src, int which, int64_t experts, int64_t n_out,
                                   int64_t k_red, uint8_t* dst, void* stream) {
  size_t need;
  mm_status s = mm_prepared_weight_scales_size(which, experts, n_out, k_red, &need);
  if (s != MM_OK) return s;
  if (!src || !dst || (reinterpret_cast<uintptr_t>(src) & 3) || (reinterpret_cast<uintptr_t>(dst) & 3))
    return MM_ERR_INVALID_ARG;
  return cuda_status(launch_prepare_wscales(src, experts, n_out, k_red, which, dst,
                                            static_cast<cudaStream_t>(stream)));
}

mm_status mm_mx_quantize(const void* src, int src_dtype, int64_t rows, int64_t cols, int out_dtype, uint8_t* q,
                         uint8_t* scales, int64_t scale_cols, void* stream) {
  if (rows < 0 || cols <= 0 || !is_src_dtype(src_dtype) || !is_mx_weight(out_dtype)) return MM_ERR_INVALID_ARG;
  if (cols % 16 != 0) return MM_ERR_UNSUPPORTED;
  if (scale_cols < ceil_div(cols, 32)) return MM_ERR_INVALID_ARG;
  if (rows == 0) return MM_OK;
  if (!src || !q || !scales || !aligned16(src) || !aligned16(q)) return MM_ERR_INVALID_ARG;
  PermuteArgs a = {};
  a.src = src;
  a.src_dtype = src_dtype;
  a.n = rows;
  a.h = cols;
  a.k = 1;
  a.dest = nullptr;
  a.dest_limit = rows;
  a.out_fmt = out_dtype;
  a.out = q;
  a.scales = scales;
  a.scale_cols = scale_cols;
  return cuda_status(launch_permute(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
