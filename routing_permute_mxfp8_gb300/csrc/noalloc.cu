// mm_moe_init_routing_noalloc: the routing + permute of mm_moe_init_routing
// for callers that cannot provide device scratch memory.
//
// Who needs it: a host program or plug-in that talks to this library through
// the plain C interface but has no device allocator of its own to hand out a
// workspace, or that must not call cudaMalloc / cudaFree while it serves
// requests (those calls can synchronise the device and fragment memory).
// Such a caller still owns its inputs and outputs; only the scratch of the
// routing kernels (per-chunk histograms, per-expert offsets and, when the
// caller does not ask for it, the scatter index) comes from a fixed array
// that this file reserves in device memory.
//
// The array is a file-scope __device__ variable of MM_NOALLOC_SCRATCH_BYTES
// (4 MiB): every GPU that loads the library holds it until the process exits.
// Host code cannot use the array's name as a device address, so the first
// call on each device looks the address up with cudaGetSymbolAddress while
// that device is current and keeps it; that first call should therefore come
// before any stream capture.  All calls share the one array, and it keeps
// whatever the last call left in it: two calls whose kernels overlap on the
// GPU (different streams, no ordering between them) race on it.  No part of
// it has to start at zero, because every word the kernels read is written
// earlier in the same call.
#include <mutex>

#include "mm_route.cuh"

namespace {

constexpr size_t kNoallocScratchBytes = MM_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (set up once per
// device), or nullptr if the lookup failed.
void* noalloc_scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> g(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    g_noalloc_ptr[dev] = p;
  }
  return g_noalloc_ptr[dev];
}

size_t piece(int64_t bytes) { return (size_t)mm::round_up(bytes, 256); }

}  // namespace

extern "C" mm_status mm_moe_init_routing_noalloc(const void* x, int x_dtype, const int32_t* expert_idx,
                                                 int64_t num_rows, int64_t h, int64_t k, int64_t expert_num,
                                                 int quant_mode, int expert_tokens_num_type, void* expanded_x,
                                                 uint8_t* expanded_scale, int32_t* expanded_row_idx,
                                                 int32_t* sorted_row_idx, int64_t* expert_tokens,
                                                 int32_t* dev_err, void* stream) {
  using namespace mm;
  if (num_rows < 0 || k <= 0 || expert_num <= 0 || expert_num > 10240 || h <= 0) return MM_ERR_INVALID_ARG;
  if (num_rows * k >= 16777215) return MM_ERR_INVALID_ARG;
  if (x_dtype != MM_DT_BFLOAT16 && x_dtype != MM_DT_FLOAT16 && x_dtype != MM_DT_FLOAT32) return MM_ERR_INVALID_ARG;
  if (quant_mode != MM_QUANT_NONE && quant_mode != MM_QUANT_MXFP8_E5M2 && quant_mode != MM_QUANT_MXFP8_E4M3FN)
    return MM_ERR_UNSUPPORTED;
  if (expert_tokens_num_type != 0 && expert_tokens_num_type != 1) return MM_ERR_UNSUPPORTED;
  const bool quant = quant_mode != MM_QUANT_NONE;
  const int esz = x_dtype == MM_DT_FLOAT32 ? 4 : 2;
  if (quant ? (h % 16 != 0) : ((h * esz) % 16 != 0)) return MM_ERR_UNSUPPORTED;
  const int64_t rows = num_rows * k;
  if (rows == 0) {  // no rows: every expert's count (and the cumsum) is 0
    if (expert_tokens &&
        cudaMemsetAsync(expert_tokens, 0, (size_t)expert_num * sizeof(int64_t), static_cast<cudaStream_t>(stream)) !=
            cudaSuccess)
      return MM_ERR_CUDA;
    return MM_OK;
  }
  if (!x || !expert_idx || !expanded_x || (quant && !expanded_scale)) return MM_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(expanded_x) & 15))
    return MM_ERR_INVALID_ARG;

  // scratch: per-chunk histograms, offsets, scatter index (unless the caller's)
  const RoutePlan plan = route_plan(rows, (int)expert_num);
  const size_t hist_b = piece((int64_t)plan.num_experts * plan.units * 4);
  const size_t off_b = piece((2 * expert_num + 1) * 4);
  const size_t idx_b = expanded_row_idx ? 0 : piece(rows * 4);
  if (hist_b + off_b + idx_b > kNoallocScratchBytes) return MM_ERR_WORKSPACE;  // problem too large
  uint8_t* base = static_cast<uint8_t*>(noalloc_scratch_address());
  if (!base) return MM_ERR_CUDA;
  int32_t* hist = reinterpret_cast<int32_t*>(base);
  int32_t* offsets = reinterpret_cast<int32_t*>(base + hist_b);
  int32_t* exp_idx = expanded_row_idx ? expanded_row_idx : reinterpret_cast<int32_t*>(base + hist_b + off_b);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RouteOutputs o;
  o.expanded_row_idx = exp_idx;
  o.sorted_row_idx = sorted_row_idx;
  o.expert_tokens = expert_tokens;
  o.tokens_cumsum = expert_tokens_num_type == 0;
  if (launch_route(plan, expert_idx, false, hist, offsets, o, dev_err, st) != cudaSuccess) return MM_ERR_CUDA;
  PermuteArgs a = {};
  a.src = x;
  a.src_dtype = x_dtype;
  a.n = num_rows;
  a.h = h;
  a.k = (int)k;
  a.dest = exp_idx;
  a.dest_limit = rows;
  a.out_fmt = quant_mode == MM_QUANT_MXFP8_E5M2 ? MM_DT_FP8_E5M2 : (quant ? MM_DT_FP8_E4M3FN : -1);
  a.out = expanded_x;
  a.scales = expanded_scale;
  a.scale_cols = round_up(ceil_div(h, 32), 2);
  a.dev_err = dev_err;
  return launch_permute(a, st) == cudaSuccess ? MM_OK : MM_ERR_CUDA;
}
