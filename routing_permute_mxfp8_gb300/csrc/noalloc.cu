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
// GPU (different streams, no ordering between them) race on it.  The one
// word that has to start at zero, the routing launch's grid-barrier counter,
// is cleared on the stream by every call before its routing kernel runs;
// every other word the kernels read is written earlier in the same call.
// Capacity: the histogram takes 4 * E * min(ceil(R / 256), 512) bytes, the
// offsets about 8 * E bytes, and the scatter index 4 * R bytes only when the
// caller passes no expanded_row_idx (each piece rounded up to 256 bytes).
// At E = 256 that leaves room for any R < 16777215 with a caller index, and
// for R up to 916,928 without one; from E = 2041 up, problems of 131,072 ids
// or more do not fit either way.
// The calls are counted and timed by mm_timing_read like mm_moe_init_routing.
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
  // the same argument checks as mm_moe_init_routing
  mm_status s = validate_init_routing(x, x_dtype, expert_idx, num_rows, h, k, expert_num, quant_mode,
                                      expert_tokens_num_type, expanded_x, expanded_scale);
  if (s != MM_OK) return s;
  const int64_t rows = num_rows * k;
  if (rows == 0) {  // no rows: every expert's count (and the cumsum) is 0
    if (expert_tokens &&
        cudaMemsetAsync(expert_tokens, 0, (size_t)expert_num * sizeof(int64_t), static_cast<cudaStream_t>(stream)) !=
            cudaSuccess)
      return MM_ERR_CUDA;
    return MM_OK;
  }

  // scratch: per-chunk histograms, offsets (with the grid-barrier counter),
  // and the scatter index unless the caller passes expanded_row_idx
  const RoutePlan plan = route_plan(rows, (int)expert_num);
  const size_t hist_b = piece((int64_t)plan.num_experts * plan.units * 4);
  const size_t off_b = piece(route_offsets_words(plan.num_experts) * 4);
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
  StageScope sr(MM_STAGE_ROUTE, st);
  int nl = 0;
  cudaError_t e = launch_route(plan, expert_idx, false, hist, offsets, o, dev_err, st, &nl);
  sr.finish(nl);
  if (e != cudaSuccess) return MM_ERR_CUDA;
  PermuteArgs a = {};
  a.src = x;
  a.src_dtype = x_dtype;
  a.n = num_rows;
  a.h = h;
  a.k = (int)k;
  a.dest = exp_idx;
  a.dest_limit = rows;
  a.out_fmt = init_routing_out_fmt(quant_mode);
  a.out = expanded_x;
  a.scales = expanded_scale;
  a.scale_cols = round_up(ceil_div(h, 32), 2);
  a.dev_err = dev_err;
  StageScope sd(MM_STAGE_DISPATCH, st);
  e = launch_permute(a, st);
  sd.finish(1);
  return e == cudaSuccess ? MM_OK : MM_ERR_CUDA;
}
