// Routing: stable counting sort of the flattened expert ids.
//
// MoeInitRoutingV3 (moe/moe_init_routing_v3), formula steps 1-3:
//   sortedExpertIdx, sortedRowIdx = keyValueSort(expertIdx, rowIdx)
//   expandedRowIdx[sortedRowIdx[i]] = i
//   expertTokensCountOrCumsum = Histogram(sortedExpertIdx)
// The keys are expert ids in [0, E) (or their place in an active expert
// range, activeExpertRangeOptional and step 6; or the destination rank of
// expert parallelism), so one counting pass replaces the two sorts the
// permute article describes (sort, then argsort of the result):
//   1. k_route_hist     each warp counts the ids of its contiguous chunk
//   2. k_route_scan_experts   one warp per expert scans its per-chunk counts
//                       (exclusive prefix over chunks, in place) and totals
//   3. k_route_scan_offsets   one block scans the totals: per-expert offsets,
//                       counts / cumsum outputs, and the 128-row tile table
//                       the grouped GEMMs use
//   4. k_route_scatter  each warp walks its chunk in index order and gives
//                       every id the next slot of its expert (warp ballots
//                       + popc for ties inside a 32-wide step), which is the
//                       stable order; it writes the inverse map and the
//                       gather index directly.
// Three implementations of the same sort, chosen per call:
//   k_route_cluster  up to 131072 ids: the phases inside one thread-block
//                    cluster (per-CTA counts exchanged through distributed
//                    shared memory, two hardware cluster barriers);
//   k_route_fused    larger problems: the four phases in one cooperative
//                    launch with a grid-wide barrier between phases;
//   the four kernels when the cooperative grid cannot be resident, or under
//                    stream capture.
// No global atomics on the data; the result is deterministic and identical
// on every path.
#include <atomic>
#include <type_traits>
#include <mutex>

#include "mm_route.cuh"

namespace mm {

constexpr int kIdBatch = 8;  // 32-id steps whose loads a warp issues together

// ids j0 + 32 b + lane (b < kIdBatch) of [.., end) into v (0 past the end)
template <typename IdT>
__device__ __forceinline__ void route_load_ids(const IdT* __restrict__ ids, int64_t j0, int64_t end, IdT* v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int b = 0; b < kIdBatch; ++b) {
    const int64_t j = j0 + 32 * b + lane;
    v[b] = j < end ? ids[j] : IdT(0);
  }
}

// Phase 1, one warp per chunk: counts of each expert in chunk `unit`
// (cnt: this warp's [E] shared-memory counters).
// Keys (KeyMap): the sort key of id is (id - off) / div (div 1: the expert
// itself, or its place in an active expert range starting at off; div = the
// experts per rank: the destination rank of expert parallelism); ids without
// a key in [0, num_experts) are left out, and those outside [0, limit) are
// errors.
template <typename IdT>
__device__ __forceinline__ void route_count_warp(const IdT* __restrict__ ids, int64_t rows, int num_experts,
                                                 KeyMap km, int chunk, int unit, int32_t* cnt, int32_t* dev_err,
                                                 IdT* v, bool preloaded = false) {
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < num_experts; e += 32) cnt[e] = 0;
  __syncwarp();
  const int64_t start = (int64_t)unit * chunk;
  const int64_t end = start + chunk < rows ? start + chunk : rows;
  bool bad = false;
  const int64_t id_end = (int64_t)num_experts * km.div;
  // the key is the id itself, and every id without a key is an error
  const bool plain = km.div == 1 && km.off == 0 && km.limit == num_experts;
  // kIdBatch 32-id steps per round: their loads are all in flight before
  // the first is counted (preloaded: the caller has loaded the first round)
  for (int64_t j0 = start; j0 < end; j0 += 32 * kIdBatch) {
    if (!(preloaded && j0 == start)) route_load_ids(ids, j0, end, v);
#pragma unroll
    for (int b = 0; b < kIdBatch; ++b) {
      if (j0 + 32 * b + lane >= end) break;
      if (plain) {
        using UIdT = typename std::make_unsigned<IdT>::type;
        if ((UIdT)v[b] < (UIdT)num_experts)
          atomicAdd(&cnt[(int)v[b]], 1);
        else
          bad = true;
      } else {
        const int64_t id = (int64_t)v[b];
        const int64_t kk = id - km.off;
        if (kk >= 0 && kk < id_end)
          atomicAdd(&cnt[kk / km.div], 1);
        else if (id < 0 || id >= km.limit)
          bad = true;
      }
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) raise_err(dev_err, MM_DEVERR_EXPERT_RANGE);
  __syncwarp();
}

// ... and the counts stored to the global [E][units] table
template <typename IdT>
__device__ __forceinline__ void route_hist_warp(const IdT* __restrict__ ids, int64_t rows, int num_experts,
                                                KeyMap km, int chunk, int units, int unit, int32_t* cnt,
                                                int32_t* __restrict__ hist, int32_t* dev_err) {
  const int lane = threadIdx.x & 31;
  if (unit >= units) return;
  IdT v[kIdBatch];
  route_count_warp(ids, rows, num_experts, km, chunk, unit, cnt, dev_err, v);
  for (int e = lane; e < num_experts; e += 32) hist[(int64_t)e * units + unit] = cnt[e];
}

template <typename IdT>
__global__ void k_route_hist(const IdT* __restrict__ ids, int64_t rows, int num_experts, KeyMap km, int chunk,
                             int units, int32_t* __restrict__ hist, int32_t* dev_err) {
  extern __shared__ int32_t sh_cnt[];  // [warps][E]
  const int warp = threadIdx.x >> 5;
  route_hist_warp(ids, rows, num_experts, km, chunk, units, blockIdx.x * (blockDim.x >> 5) + warp,
                  sh_cnt + warp * num_experts, hist, dev_err);
}

// Exclusive scan of one value per thread across the block (<= 1024 threads).
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t* sh_warp, int64_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int64_t y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  if (lane == 31) sh_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t w = lane < (int)(blockDim.x >> 5) ? sh_warp[lane] : 0;
    int64_t s = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      int64_t y = __shfl_up_sync(0xffffffffu, s, d);
      if (lane >= d) s += y;
    }
    sh_warp[lane] = s - w;  // exclusive warp base
    if (lane == 31) sh_warp[32] = s;
  }
  __syncthreads();
  int64_t r = sh_warp[warp] + x - v;
  total = sh_warp[32];
  __syncthreads();
  return r;
}

constexpr int kMaxUnits = 512;  // chunks per call (route_plan keeps units <= kMaxUnits)

// Phase 2, one warp per expert: exclusive prefix of its per-chunk counts,
// in place, and the expert's total.
__device__ __forceinline__ void route_scan_expert_warp(int32_t* __restrict__ hist, int units, int e,
                                                       int32_t* __restrict__ totals) {
  const int lane = threadIdx.x & 31;
  int32_t* row = hist + (int64_t)e * units;
  constexpr int kPer = kMaxUnits / 32;
  int32_t v[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int u = i * 32 + lane;
    v[i] = u < units ? row[u] : 0;
  }
  int32_t run = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    if (i * 32 >= units) break;
    int32_t x = v[i];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x += y;
    }
    const int u = i * 32 + lane;
    if (u < units) row[u] = run + x - v[i];
    run += __shfl_sync(0xffffffffu, x, 31);
  }
  if (lane == 0) totals[e] = run;
}

// The same with one thread per expert, for few chunks (units <= 32).
__device__ __forceinline__ void route_scan_expert_thread(int32_t* __restrict__ hist, int units, int e,
                                                         int32_t* __restrict__ totals) {
  int32_t* row = hist + (int64_t)e * units;
  int32_t v[32];
#pragma unroll
  for (int u = 0; u < 32; ++u) v[u] = u < units ? row[u] : 0;
  int32_t run = 0;
#pragma unroll
  for (int u = 0; u < 32; ++u) {
    if (u >= units) break;
    row[u] = run;
    run += v[u];
  }
  totals[e] = run;
}

__global__ void __launch_bounds__(1024) k_route_scan_experts(int32_t* __restrict__ hist, int num_experts, int units,
                                                             int32_t* __restrict__ totals) {
  const int e = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (e < num_experts) route_scan_expert_warp(hist, units, e, totals);
}

// Phase 3, one block: expert offsets, count / cumsum outputs, GEMM segment
// table.
__device__ __forceinline__ void route_scan_offsets_block(const RouteScanArgs& a, int64_t* sh_warp) {
  const int nt = blockDim.x;
  const int E = a.num_experts;
  // 1. exclusive scan of the expert totals -> offsets
  {
    const int per = (E + nt - 1) / nt;
    const int lo = threadIdx.x * per;
    const int hi = lo + per < E ? lo + per : E;
    int64_t s = 0;
    for (int e = lo; e < hi; ++e) s += a.totals[e];
    int64_t total;
    int64_t base = block_exclusive_scan(s, sh_warp, total);
    for (int e = lo; e < hi; ++e) {
      const int32_t c = a.totals[e];
      a.offsets[e] = (int32_t)base;
      if (a.expert_tokens) a.expert_tokens[e] = a.tokens_cumsum ? base + c : (int64_t)c;
      if (a.expert_token_nums) a.expert_token_nums[e] = c;
      base += c;
    }
    if (threadIdx.x == 0) a.offsets[E] = (int32_t)total;
    // rows whose id was out of range are left out: pad the gather index
    if (a.sorted_row_idx)
      for (int64_t d = total + threadIdx.x; d < a.rows; d += nt) a.sorted_row_idx[d] = -1;
  }
  // 2. segment table of the grouped GEMMs: routed experts, then shared
  //    experts (shared_rows rows each); 128-row tiles, prefix in tiles.
  if (a.seg_mprefix) {
    const int nseg = E + a.n_shared;
    const int per = (nseg + nt - 1) / nt;
    const int lo = threadIdx.x * per;
    const int hi = lo + per < nseg ? lo + per : nseg;
    int64_t t = 0;
    for (int sg = lo; sg < hi; ++sg) {
      const int64_t rows_s = sg < E ? a.totals[sg] : a.shared_rows;
      t += (rows_s + kBM - 1) / kBM;
    }
    int64_t tot2;
    int64_t b2 = block_exclusive_scan(t, sh_warp, tot2);
    for (int sg = lo; sg < hi; ++sg) {
      const int64_t rows_s = sg < E ? a.totals[sg] : a.shared_rows;
      a.seg_rows[sg] = (int32_t)rows_s;
      a.seg_mprefix[sg] = (int32_t)b2;
      b2 += (rows_s + kBM - 1) / kBM;
    }
    if (threadIdx.x == 0) a.seg_mprefix[nseg] = (int32_t)tot2;
  }
}

__global__ void __launch_bounds__(1024) k_route_scan_offsets(RouteScanArgs a) {
  __shared__ int64_t sh_warp[33];
  route_scan_offsets_block(a, sh_warp);
}

// Phase 4, one warp per chunk, in index order: every id of [start, end)
// takes the next slot of its key (next: this warp's [E] shared-memory slots,
// initialised to the chunk's first slot of each key); ties inside a 32-id
// step are ranked by lane (the lanes with an equal key from ballots of the
// key's bits, then popc), so the order is stable.
// offsets / seg_mprefix: per-key first slot and GEMM tile prefix (pad_row).
template <typename IdT>
__device__ __forceinline__ void route_scatter_walk(const IdT* __restrict__ ids, int64_t start, int64_t end,
                                                   int num_experts, KeyMap km, int32_t* next,
                                                   const int32_t* offsets, const int32_t* seg_mprefix,
                                                   int32_t* __restrict__ expanded_row_idx,
                                                   int32_t* __restrict__ sorted_row_idx, int32_t* __restrict__ pad_row,
                                                   int32_t* __restrict__ sorted_rem, int64_t rows_total,
                                                   int64_t pad_limit, int32_t* dev_err, IdT* v,
                                                   bool preloaded = false) {
  const int lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  const int key_bits = 32 - __clz(num_experts);  // bits of the largest key + 1
  using UIdT = typename std::make_unsigned<IdT>::type;
  const int64_t id_end = (int64_t)num_experts * km.div;
  // the key is the id itself, and every id without a key is an error
  const bool plain = km.div == 1 && km.off == 0 && km.limit == num_experts;
  for (int64_t j0 = start; j0 < end; j0 += 32 * kIdBatch) {
    // the next kIdBatch steps' ids, loaded together (preloaded: the caller
    // has loaded the first round)
    if (!(preloaded && j0 == start)) route_load_ids(ids, j0, end, v);
#pragma unroll
    for (int b = 0; b < kIdBatch; ++b) {
      const int64_t jb = j0 + 32 * b;
      if (jb >= end) break;  // uniform across the warp
      const int64_t j = jb + lane;
      const bool in = j < end;
      int key = -1, rem = 0;
      if (in) {
        if (plain) {
          if ((UIdT)v[b] < (UIdT)num_experts) key = (int)v[b];
        } else {
          const int64_t kk = (int64_t)v[b] - km.off;
          if (kk >= 0 && kk < id_end) {
            key = (int)(kk / km.div);
            rem = (int)(kk - (int64_t)key * km.div);
          }
        }
      }
      // lanes holding the same key: one ballot per bit of key + 1 (the
      // invalid key -1 becomes 0), all bits equal
      const uint32_t kk = (uint32_t)(key + 1);
      unsigned peers = 0xffffffffu;
      for (int bit = 0; bit < key_bits; ++bit) {
        const unsigned m = __ballot_sync(0xffffffffu, (kk >> bit) & 1u);
        peers &= ((kk >> bit) & 1u) ? m : ~m;
      }
      const unsigned below = peers & lt;
      int32_t dest = -1;
      if (key >= 0) dest = next[key] + __popc(below);
      __syncwarp();
      if (key >= 0 && below == 0) next[key] += __popc(peers);
      __syncwarp();
      if (in) {
        if (expanded_row_idx) expanded_row_idx[j] = dest;
        if (key >= 0) {
          if (in_bounds(dest < rows_total, dev_err)) {
            if (sorted_row_idx) sorted_row_idx[dest] = (int32_t)j;
            if (sorted_rem) sorted_rem[dest] = rem;
          }
          if (pad_row) {
            const int32_t pr = seg_mprefix[key] * kBM + (dest - offsets[key]);
            pad_row[j] = in_bounds(pr >= 0 && pr < pad_limit, dev_err) ? pr : -1;
          }
        } else if (pad_row) {
          pad_row[j] = -1;
        }
      }
    }
  }
}

template <typename IdT>
__device__ __forceinline__ void route_scatter_warp(const IdT* __restrict__ ids, int64_t rows, int num_experts,
                                                   KeyMap km, int chunk, int units, int unit, int32_t* next,
                                                   const int32_t* __restrict__ bases,
                                                   const int32_t* __restrict__ offsets,
                                                   const int32_t* __restrict__ seg_mprefix,
                                                   int32_t* __restrict__ expanded_row_idx,
                                                   int32_t* __restrict__ sorted_row_idx, int32_t* __restrict__ pad_row,
                                                   int32_t* __restrict__ sorted_rem, int64_t pad_limit,
                                                   int32_t* dev_err) {
  const int lane = threadIdx.x & 31;
  for (int e = lane; e < num_experts; e += 32) next[e] = offsets[e] + bases[(int64_t)e * units + unit];
  __syncwarp();
  const int64_t start = (int64_t)unit * chunk;
  const int64_t end = start + chunk < rows ? start + chunk : rows;
  IdT v[kIdBatch];
  route_scatter_walk(ids, start, end, num_experts, km, next, offsets, seg_mprefix, expanded_row_idx,
                     sorted_row_idx, pad_row, sorted_rem, rows, pad_limit, dev_err, v);
}

template <typename IdT>
__global__ void k_route_scatter(const IdT* __restrict__ ids, int64_t rows, int num_experts, KeyMap km, int chunk,
                                int units, const int32_t* __restrict__ bases,
                                const int32_t* __restrict__ offsets, const int32_t* __restrict__ seg_mprefix,
                                int32_t* __restrict__ expanded_row_idx, int32_t* __restrict__ sorted_row_idx,
                                int32_t* __restrict__ pad_row, int32_t* __restrict__ sorted_rem, int64_t pad_limit,
                                int32_t* dev_err) {
  extern __shared__ int32_t sh_next[];  // [warps][E]: next free slot per expert
  const int warp = threadIdx.x >> 5;
  const int unit = blockIdx.x * (blockDim.x >> 5) + warp;
  if (unit >= units) return;
  route_scatter_warp(ids, rows, num_experts, km, chunk, units, unit, sh_next + warp * num_experts, bases,
                     offsets, seg_mprefix, expanded_row_idx, sorted_row_idx, pad_row, sorted_rem, pad_limit, dev_err);
}

// Grid-wide barrier of a cooperative launch (every block is resident) on a
// counter that is zero when the launch starts: barrier number b (1, 2, ...)
// opens when the counter reaches b * gridDim.x.  The wait is bounded: after
// kWaitNs the block raises MM_DEVERR_TIMEOUT and the caller stops (the
// other blocks then time out at their next barrier, so the launch ends).
__device__ __forceinline__ bool grid_barrier_bounded(uint32_t* count, uint32_t b, int32_t* dev_err, int* sh_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();  // this block's writes before its arrival
    atomicAdd(count, 1u);
    const uint32_t target = b * gridDim.x;
    int ok = 1;
    if (ld_acquire_u32(count) < target) {
      const uint64_t t0 = globaltimer();
      while (ld_acquire_u32(count) < target) {
        if (globaltimer() - t0 > kWaitNs) {
          ok = 0;
          raise_err(dev_err, MM_DEVERR_TIMEOUT);
          break;
        }
      }
    }
    __threadfence();
    *sh_ok = ok;
  }
  __syncthreads();
  return *sh_ok != 0;
}

// All four phases in one cooperative launch (every block resident), with
// grid-wide barriers between them: one launch instead of four.
template <typename IdT>
__global__ void k_route_fused(const IdT* __restrict__ ids, int64_t rows, int num_experts, KeyMap km, int chunk,
                              int units, int32_t* __restrict__ hist, RouteScanArgs sa,
                              int32_t* __restrict__ expanded_row_idx, int32_t* __restrict__ pad_row,
                              int32_t* __restrict__ sorted_rem, int64_t pad_limit, uint32_t* __restrict__ barrier,
                              int32_t* dev_err) {
  extern __shared__ int32_t sh_route[];  // [warps][E]
  __shared__ int64_t sh_warp[33];
  __shared__ int sh_ok;
  const int warp = threadIdx.x >> 5, wpb = blockDim.x >> 5;
  const int unit = blockIdx.x * wpb + warp;
  int32_t* mine = sh_route + warp * num_experts;
  if (unit < units) route_hist_warp(ids, rows, num_experts, km, chunk, units, unit, mine, hist, dev_err);
  if (!grid_barrier_bounded(barrier, 1, dev_err, &sh_ok)) return;
  if (units <= 32) {
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < num_experts; e += gridDim.x * blockDim.x)
      route_scan_expert_thread(hist, units, e, sa.totals);
  } else {
    for (int e = unit; e < num_experts; e += gridDim.x * wpb) route_scan_expert_warp(hist, units, e, sa.totals);
  }
  if (!grid_barrier_bounded(barrier, 2, dev_err, &sh_ok)) return;
  if (blockIdx.x == 0) route_scan_offsets_block(sa, sh_warp);
  if (!grid_barrier_bounded(barrier, 3, dev_err, &sh_ok)) return;
  if (unit < units)
    route_scatter_warp(ids, rows, num_experts, km, chunk, units, unit, mine, hist, sa.offsets, sa.seg_mprefix,
                       expanded_row_idx, sa.sorted_row_idx, pad_row, sorted_rem, pad_limit, dev_err);
}

// ---------------------------------------------------------------------------
// Problems of up to kClusterMaxRows ids: the whole routing in one
// thread-block cluster of up to 16 CTAs (one per 2048 ids), which exchange
// their per-expert counts through distributed shared memory, with two
// hardware cluster barriers instead of three grid-wide barriers on global
// memory.
//   1. each warp counts its chunk (CTA c owns the chunks c*W .. c*W+W-1, in
//      index order; chunks of up to kIdBatch 32-id steps stay in registers
//      for step 3), then each CTA scans its warps' counts per expert
//      (exclusive, in place) and keeps its own per-expert total;
//   -- cluster barrier: every CTA's totals are visible --
//   2. every CTA reads all CTAs' totals (the prefix over the CTAs before it,
//      and the expert totals) and scans the totals into the expert offsets
//      and the GEMM segment table in shared memory (CTA 0 also writes the
//      outputs);
//   -- arrival: this CTA no longer reads the others' shared memory --
//   3. each warp walks its chunk as in k_route_scatter;
//   -- wait: no CTA leaves while another may still read its totals --
// The cluster's CTAs are co-scheduled by the hardware, so the barriers have
// the standing of __syncthreads: every thread reaches both.
constexpr int kClusterMaxCtas = 16;
constexpr int64_t kClusterRowsPerCta = 2048;
constexpr int64_t kClusterMinWarpIds = 128;
constexpr int64_t kClusterMaxRows = 131072;
constexpr int kClusterMaxExperts = 4096;
constexpr int kClusterCntWords = 32768;  // per-warp counters: warps * E <= this

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the int32 at the same shared-memory offset in CTA `cta` of the cluster
__device__ __forceinline__ int32_t ld_cluster_peer(const int32_t* local, uint32_t cta) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(local);
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(cta));
  int32_t v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(ra) : "memory");
  return v;
}

template <typename IdT>
__global__ void __launch_bounds__(1024) k_route_cluster(const IdT* __restrict__ ids, int64_t rows, int num_experts,
                                                        KeyMap km, int chunk, RouteScanArgs sa,
                                                        int32_t* __restrict__ expanded_row_idx,
                                                        int32_t* __restrict__ pad_row,
                                                        int32_t* __restrict__ sorted_rem, int64_t pad_limit,
                                                        int32_t* dev_err) {
  extern __shared__ int32_t sh_cl[];
  __shared__ int64_t sh_warp[33];
  const int E = num_experts, nt = blockDim.x, W = nt >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t c = cluster_ctarank(), ncta = cluster_nctarank();
  const int nseg = E + sa.n_shared;
  int32_t* cnt = sh_cl;           // [W][E] counts, then each warp's next slots
  int32_t* ctot = cnt + W * E;    // [E] this CTA's per-expert total (read by the others)
  int32_t* cpre = ctot + E;       // [E] the CTAs before this one: their per-expert total
  int32_t* etot = cpre + E;       // [E] expert totals
  int32_t* eoff = etot + E;       // [E + 1] expert offsets
  int32_t* mpre = eoff + E + 1;   // [nseg + 1] tile prefix of the GEMM segments
  const int unit = (int)c * W + warp;
  int32_t* mine = cnt + warp * E;
  pdl_wait();
  pdl_trigger();
  const int64_t start = (int64_t)unit * chunk;
  const int64_t end = start + chunk < rows ? start + chunk : rows;
  const bool resident = chunk <= 32 * kIdBatch;  // the whole chunk fits one round of loads
  IdT v[kIdBatch];
  route_load_ids(ids, start, end, v);

  route_count_warp(ids, rows, E, km, chunk, unit, mine, dev_err, v, true);
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += nt) {
    int32_t run = 0;
    for (int w = 0; w < W; ++w) {
      const int32_t x = cnt[w * E + e];
      cnt[w * E + e] = run;
      run += x;
    }
    ctot[e] = run;
  }
  cluster_arrive_release();
  cluster_wait_acquire();

  for (int e = threadIdx.x; e < E; e += nt) {
    int32_t pre = 0, tot = 0;
    for (uint32_t q0 = 0; q0 < ncta; q0 += 4) {
      int32_t x[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) x[u] = q0 + u < ncta ? ld_cluster_peer(ctot + e, q0 + u) : 0;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (q0 + u < c) pre += x[u];
        tot += x[u];
      }
    }
    cpre[e] = pre;
    etot[e] = tot;
  }
  cluster_arrive_release();
  __syncthreads();

  // expert offsets, counts / cumsum, gather-index tail and the GEMM segment
  // table from one scan over the segments (routed experts, then the shared
  // ones): an entry packs its rows counted in the expert offsets (high word)
  // and its 128-row tiles (low word); neither sum reaches 2^32
  {
    const int nsc = sa.seg_mprefix ? nseg : E;
    const int per = (nsc + nt - 1) / nt;
    const int lo = min(nsc, (int)threadIdx.x * per), hi = min(nsc, lo + per);
    auto pack = [&](int sg) -> int64_t {
      const int64_t r = sg < E ? etot[sg] : sa.shared_rows;
      return ((sg < E ? r : 0) << 32) | ((r + kBM - 1) / kBM);
    };
    int64_t sum = 0;
    for (int sg = lo; sg < hi; ++sg) sum += pack(sg);
    int64_t total;
    int64_t base = block_exclusive_scan(sum, sh_warp, total);
    for (int sg = lo; sg < hi; ++sg) {
      const int32_t off = (int32_t)(base >> 32), tiles = (int32_t)(base & 0xffffffff);
      if (sg < E) {
        const int32_t ce = etot[sg];
        eoff[sg] = off;
        if (c == 0) {
          sa.offsets[sg] = off;
          sa.totals[sg] = ce;
          if (sa.expert_tokens) sa.expert_tokens[sg] = sa.tokens_cumsum ? (int64_t)off + ce : (int64_t)ce;
          if (sa.expert_token_nums) sa.expert_token_nums[sg] = ce;
        }
      }
      if (sa.seg_mprefix) {
        mpre[sg] = tiles;
        if (c == 0) {
          sa.seg_rows[sg] = sg < E ? etot[sg] : sa.shared_rows;
          sa.seg_mprefix[sg] = tiles;
        }
      }
      base += pack(sg);
    }
    const int64_t routed = total >> 32;
    if (threadIdx.x == 0) {
      eoff[E] = (int32_t)routed;
      if (c == 0) sa.offsets[E] = (int32_t)routed;
      if (sa.seg_mprefix) {
        mpre[nseg] = (int32_t)(total & 0xffffffff);
        if (c == 0) sa.seg_mprefix[nseg] = (int32_t)(total & 0xffffffff);
      }
    }
    // rows whose id was out of range are left out: pad the gather index
    if (sa.sorted_row_idx)
      for (int64_t d = routed + (int64_t)c * nt + threadIdx.x; d < rows; d += (int64_t)ncta * nt)
        sa.sorted_row_idx[d] = -1;
  }
  __syncthreads();

  for (int e = lane; e < E; e += 32) mine[e] += eoff[e] + cpre[e];
  __syncwarp();
  route_scatter_walk(ids, start, end, E, km, mine, eoff, mpre, expanded_row_idx, sa.sorted_row_idx, pad_row,
                     sorted_rem, rows, pad_limit, dev_err, v, resident);
  cluster_wait_acquire();
}

// ---------------------------------------------------------------------------
// key_value counts: one block; the non-zero counts are compacted in
// ascending expert order by a block-wide scan of their flags, 1024 experts
// at a time, after the output has been zeroed.
__global__ void __launch_bounds__(1024) k_key_value_counts(const int64_t* __restrict__ counts, int n, int64_t first,
                                                           int64_t out_rows, int64_t* __restrict__ out) {
  __shared__ int warp_tot[32];
  __shared__ int base;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int64_t i = threadIdx.x; i < 2 * out_rows; i += blockDim.x) out[i] = 0;
  if (threadIdx.x == 0) base = 0;
  __syncthreads();
  for (int e0 = 0; e0 < n; e0 += blockDim.x) {
    const int e = e0 + (int)threadIdx.x;
    const int64_t c = e < n ? counts[e] : 0;
    const unsigned m = __ballot_sync(0xffffffffu, c != 0);
    if (lane == 0) warp_tot[w] = __popc(m);
    __syncthreads();
    int before = base;
    for (int i = 0; i < w; ++i) before += warp_tot[i];
    const int pos = before + __popc(m & ((1u << lane) - 1u));
    if (c != 0 && pos < out_rows) {
      out[2 * (int64_t)pos] = first + e;
      out[2 * (int64_t)pos + 1] = c;
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) base = pos + (c != 0 ? 1 : 0);
    __syncthreads();
  }
}

RoutePlan route_plan(int64_t rows, int num_experts) {
  RoutePlan p;
  p.rows = rows;
  p.num_experts = num_experts;
  // chunk: multiple of 32, at least 256 ids, at most kMaxUnits chunks
  int64_t c = (rows + kMaxUnits - 1) / kMaxUnits;
  c = round_up(c < 256 ? 256 : c, 32);
  p.chunk = (int)c;
  p.units = (int)((rows + c - 1) / c);
  if (p.units < 1) p.units = 1;
  int wpb = (int)(40960 / (4 * (int64_t)num_experts));
  p.warps_per_block = wpb < 1 ? 1 : (wpb > 8 ? 8 : wpb);
  return p;
}

int64_t route_offsets_words(int num_experts) {
  // offsets [E + 1], totals [E], then the grid-barrier counter on its own
  // 8-byte boundary
  return round_up(2 * (int64_t)num_experts + 1, 2) + 2;
}

size_t route_workspace_bytes(const RoutePlan& p) {
  return (size_t)round_up((int64_t)p.num_experts * p.units * 4, 256) +
         (size_t)round_up(route_offsets_words(p.num_experts) * 4, 256);
}

namespace {

// Blocks of k_route_fused with `wpb` warps that can be resident at once on
// the current device (0: no cooperative launch).  Queried once per device
// and block size with the largest shared-memory table route_plan allows
// (40 KB), so it never overestimates.
constexpr int kMaxDevices = 64;

template <typename IdT>
int fused_capacity(int wpb) {
  static std::mutex mu;
  static int cap[kMaxDevices][9];
  static bool init[kMaxDevices] = {false};
  int dev = 0;
  if (wpb < 1 || wpb > 8 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> g(mu);
  if (!init[dev]) {
    for (int w = 0; w < 9; ++w) cap[dev][w] = -1;
    init[dev] = true;
  }
  if (cap[dev][wpb] < 0) {
    int coop = 0, per_sm = 0;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess) coop = 0;
    int c = 0;
    if (coop && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_route_fused<IdT>, wpb * 32, 40960) ==
                    cudaSuccess)
      c = per_sm * num_sms();
    cudaGetLastError();
    cap[dev][wpb] = c;
  }
  return cap[dev][wpb];
}

// Path selection for tests and measurements (mm_set_routing_path):
// 0 automatic, 1 cluster, 2 cooperative grid, 3 four kernels.
std::atomic<int> g_route_path{0};

// Warps per CTA of k_route_cluster for E experts, and its shared memory.
int cluster_warps(int num_experts) {
  const int w = kClusterCntWords / (num_experts < 1 ? 1 : num_experts);
  return w < 1 ? 1 : (w > 32 ? 32 : w);
}
size_t cluster_smem(int wpb, int num_experts, int nseg) {
  return 4 * ((size_t)wpb * num_experts + 4 * (size_t)num_experts + 1 + (size_t)nseg + 1);
}
// the largest cluster_smem of any accepted problem (E <= kClusterMaxExperts,
// at most 4 shared segments)
constexpr size_t kClusterMaxSmem = 4 * ((size_t)kClusterCntWords + 5 * (size_t)kClusterMaxExperts + 8);

// launch configuration of one cluster of k_route_cluster (attr: room for
// two attributes; pdl adds the programmatic dependent launch)
cudaLaunchConfig_t cluster_config(int ncta, int wpb, size_t smem, cudaStream_t st, cudaLaunchAttribute* attr,
                                  bool pdl = false) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ncta;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(ncta);
  cfg.blockDim = dim3(wpb * 32);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cfg;
}

// The largest cluster (16, else 8 CTAs; 0: none) of k_route_cluster with
// `wpb` warps per CTA and the largest shared-memory size that fits on the
// current device (queried once per device and block size).
template <typename IdT>
int cluster_max_ctas(int wpb) {
  static std::mutex mu;
  static int fits[kMaxDevices][33];
  static bool init[kMaxDevices] = {false};
  int dev = 0;
  if (wpb < 1 || wpb > 32 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> g(mu);
  if (!init[dev]) {
    for (int w = 0; w < 33; ++w) fits[dev][w] = -1;
    init[dev] = true;
  }
  if (fits[dev][wpb] < 0) {
    int best = 0;
    if (cudaFuncSetAttribute(k_route_cluster<IdT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kClusterMaxSmem) == cudaSuccess) {
      const bool big = cudaFuncSetAttribute(k_route_cluster<IdT>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                            1) == cudaSuccess;
      for (int n : {kClusterMaxCtas, 8}) {
        if (n > 8 && !big) continue;
        cudaLaunchAttribute attr[2];
        cudaLaunchConfig_t cfg = cluster_config(n, wpb, kClusterMaxSmem, nullptr, attr);
        int active = 0;
        if (cudaOccupancyMaxActiveClusters(&active, k_route_cluster<IdT>, &cfg) == cudaSuccess && active >= 1) {
          best = n;
          break;
        }
      }
    }
    cudaGetLastError();
    fits[dev][wpb] = best;
  }
  return fits[dev][wpb];
}

KeyMap key_map(const RouteOutputs& o, int num_experts) {
  KeyMap k;
  k.div = o.key_div;
  k.off = o.key_off;
  k.limit = o.id_limit > 0 ? o.id_limit : (int64_t)num_experts * o.key_div;
  return k;
}

template <typename IdT>
bool launch_route_cluster(const RoutePlan& p, const IdT* ids, RouteScanArgs a, const RouteOutputs& o,
                          int32_t* dev_err, cudaStream_t st) {
  if (p.num_experts > kClusterMaxExperts || a.n_shared > 4 || (o.pad_row && !o.seg_mprefix)) return false;
  // one CTA per kClusterRowsPerCta ids (at most 16); warps of at least
  // kClusterMinWarpIds ids (at least 4, at most what the counters allow)
  int64_t ncta = (p.rows + kClusterRowsPerCta - 1) / kClusterRowsPerCta;
  ncta = ncta < 1 ? 1 : (ncta > kClusterMaxCtas ? kClusterMaxCtas : ncta);
  const int64_t per_cta = (p.rows + ncta - 1) / ncta;
  int64_t w = (per_cta + kClusterMinWarpIds - 1) / kClusterMinWarpIds;
  const int wmax = cluster_warps(p.num_experts);
  w = w < 4 ? 4 : w;
  const int wpb = (int)(w > wmax ? wmax : w);
  const int max_ctas = cluster_max_ctas<IdT>(wpb);
  if (max_ctas < 1) return false;
  if (ncta > max_ctas) ncta = max_ctas;
  int64_t per = (p.rows + ncta * wpb - 1) / (ncta * wpb);
  per = round_up(per < 32 ? 32 : per, 32);
  if (per > INT32_MAX) return false;
  const int64_t rows = p.rows;
  const int ne = p.num_experts, chunk = (int)per;
  const KeyMap km = key_map(o, ne);
  int32_t* exp_idx = o.expanded_row_idx;
  int32_t* pad = o.pad_row;
  int32_t* rem = o.sorted_rem;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = cluster_config((int)ncta, wpb, cluster_smem(wpb, ne, ne + a.n_shared), st, attr, true);
  const int64_t plim = o.pad_limit;
  if (cudaLaunchKernelEx(&cfg, k_route_cluster<IdT>, ids, rows, ne, km, chunk, a, exp_idx, pad, rem, plim, dev_err) ==
      cudaSuccess)
    return true;
  cudaGetLastError();
  return false;
}

template <typename IdT>
cudaError_t launch_route_typed(const RoutePlan& p, const IdT* ids, int32_t* hist, RouteScanArgs a,
                               const RouteOutputs& o, int32_t* dev_err, cudaStream_t st, int& launches) {
  const int path = g_route_path.load();
  if ((path == 1 || (path == 0 && p.rows <= kClusterMaxRows)) && launch_route_cluster(p, ids, a, o, dev_err, st)) {
    launches = 1;
    return cudaSuccess;
  }
  const int wpb = p.warps_per_block;
  const int blocks = (p.units + wpb - 1) / wpb;
  const size_t sh = (size_t)wpb * p.num_experts * sizeof(int32_t);
  // under stream capture the four ordinary launches are used: a refused
  // cooperative launch there would invalidate the caller's capture
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
    cudaGetLastError();
    cap = cudaStreamCaptureStatusActive;
  }
  if (path != 3 && cap == cudaStreamCaptureStatusNone && blocks <= fused_capacity<IdT>(wpb)) {
    int64_t rows = p.rows;
    int ne = p.num_experts, chunk = p.chunk, units = p.units;
    KeyMap km = key_map(o, ne);
    int32_t* exp_idx = o.expanded_row_idx;
    int32_t* pad = o.pad_row;
    int32_t* rem = o.sorted_rem;
    int64_t plim = o.pad_limit;
    // the barrier counter (workspace, after the offsets and totals) starts at 0
    uint32_t* barrier = reinterpret_cast<uint32_t*>(a.offsets + route_offsets_words(p.num_experts) - 2);
    void* args[] = {(void*)&ids, &rows, &ne, &km, &chunk, &units, &hist, &a, &exp_idx, &pad, &rem, &plim, &barrier,
                    &dev_err};
    if (cudaMemsetAsync(barrier, 0, sizeof(uint32_t), st) != cudaSuccess) return cudaGetLastError();
    if (cudaLaunchCooperativeKernel((const void*)k_route_fused<IdT>, dim3(blocks), dim3(wpb * 32), args, sh, st) ==
        cudaSuccess) {
      launches = 1;
      return cudaSuccess;
    }
    cudaGetLastError();  // not launched (e.g. no cooperative launch here): the four kernels below
  }
  k_route_hist<IdT><<<blocks, wpb * 32, sh, st>>>(ids, p.rows, p.num_experts, key_map(o, p.num_experts), p.chunk,
                                                  p.units, hist,
                                                  dev_err);
  k_route_scan_experts<<<(p.num_experts + 31) / 32, 1024, 0, st>>>(hist, p.num_experts, p.units, a.totals);
  k_route_scan_offsets<<<1, 1024, 0, st>>>(a);
  k_route_scatter<IdT><<<blocks, wpb * 32, sh, st>>>(ids, p.rows, p.num_experts, key_map(o, p.num_experts), p.chunk,
                                                     p.units, hist,
                                                     a.offsets, o.seg_mprefix, o.expanded_row_idx,
                                                     o.sorted_row_idx, o.pad_row, o.sorted_rem, o.pad_limit, dev_err);
  launches = 4;
  return cudaGetLastError();
}

}  // namespace

void set_route_path(int path) { g_route_path.store(path); }

cudaError_t launch_key_value_counts(const int64_t* counts, int n, int64_t first, int64_t out_rows, int64_t* out,
                                    cudaStream_t st) {
  k_key_value_counts<<<1, 1024, 0, st>>>(counts, n, first, out_rows, out);
  return cudaGetLastError();
}

cudaError_t launch_route(const RoutePlan& p, const void* ids, bool ids64, int32_t* hist, int32_t* offsets,
                         RouteOutputs o, int32_t* dev_err, cudaStream_t st, int* launches) {
  int n = 0;
  RouteScanArgs a;
  a.hist = hist;
  // per-expert totals live right after the E + 1 offsets (the offsets
  // buffer holds 2 * E + 1 entries)
  a.totals = offsets + p.num_experts + 1;
  a.num_experts = p.num_experts;
  a.units = p.units;
  a.rows = p.rows;
  a.offsets = offsets;
  a.sorted_row_idx = o.sorted_row_idx;
  a.expert_tokens = o.expert_tokens;
  a.tokens_cumsum = o.tokens_cumsum;
  a.expert_token_nums = o.expert_token_nums;
  a.seg_rows = o.seg_rows;
  a.seg_mprefix = o.seg_mprefix;
  a.n_shared = o.n_shared;
  a.shared_rows = o.shared_rows;
  const cudaError_t e = ids64 ? launch_route_typed(p, static_cast<const int64_t*>(ids), hist, a, o, dev_err, st, n)
                              : launch_route_typed(p, static_cast<const int32_t*>(ids), hist, a, o, dev_err, st, n);
  if (launches) *launches = n;
  return e;
}

}  // namespace mm
