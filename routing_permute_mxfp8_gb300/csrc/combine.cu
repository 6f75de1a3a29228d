// Combine (MegaMoE README, A8W8-FP stage 4; at epWorldSize = 1 and, on the
// source rank, with expert parallelism):
//   Y[i] = sum_k W[i,k] * O[pi(i,k)] + sum_s O_s^shared[i]
// One block per token.  The expert rows are gathered with 16-byte loads
// (eight rows in flight per thread), accumulated in fp32 in the order
// k = 0..K-1 then the shared experts, and rounded to bf16 once.  No atomics,
// so the result is deterministic.
#include "mm_route.cuh"

namespace mm {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxTerms = 36;  // top-K <= 32 plus up to 4 shared experts
constexpr int kBatch = 8;      // expert rows gathered per round

// 8 FP8 codes (E4M3 / E5M2) -> fp32 times the group's scale 2^(s - 127)
// (E8M0 code s; 0 is 2^-127, a subnormal): DQ_MX of the combine exchange.
template <int kFmt>
__device__ __forceinline__ void fp8x8_dq(uint2 q, uint32_t s, float* f) {
  const float sc = s ? __uint_as_float(s << 23) : __uint_as_float(0x00400000u);
  const uint32_t w[2] = {q.x, q.y};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_fp8x2_storage_t p = (__nv_fp8x2_storage_t)((w[i >> 1] >> (16 * (i & 1))) & 0xffffu);
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(p, kFmt == MM_DT_FP8_E5M2 ? __NV_E5M2 : __NV_E4M3);
    const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&hr));
    f[2 * i] = v.x * sc;
    f[2 * i + 1] = v.y * sc;
  }
}

// The rows of token i's terms and their weights in shared memory: routed
// terms from pad_row, then the shared experts' rows (weight 1).
template <bool kSep>
__device__ __forceinline__ void combine_terms(const CombineArgs& a, int64_t i, int32_t* rows, float* w) {
  const int nterm = a.k + a.n_shared;
  if (threadIdx.x < a.k) {
    const int64_t j = i * a.k + threadIdx.x;
    const int32_t r = a.pad_row[j];
    rows[threadIdx.x] = in_bounds(r < a.rows_cap, a.dev_err) ? r : -1;
    w[threadIdx.x] = a.gate_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.gate)[j])
                                 : static_cast<const float*>(a.gate)[j];
  } else if (threadIdx.x < nterm) {
    const int s = threadIdx.x - a.k;
    if (kSep) {
      rows[threadIdx.x] = (int32_t)((int64_t)s * a.n + i);  // the caller's [n_shared, n, h] rows
    } else {
      const int64_t r = (int64_t)a.seg_mprefix[a.n_routed + s] * kBM + i;
      rows[threadIdx.x] = in_bounds(r >= 0 && r < a.rows_cap, a.dev_err) ? (int32_t)r : -1;
    }
    w[threadIdx.x] = 1.0f;
  }
}

// kSep: the shared experts' rows come from the caller's o_sh, not from o
template <bool kSep>
__global__ void __launch_bounds__(kThreads) k_combine(CombineArgs a) {
  __shared__ int32_t rows[kMaxTerms];
  __shared__ float w[kMaxTerms];
  const int64_t i = blockIdx.x;
  const int nterm = a.k + a.n_shared;
  pdl_wait();
  pdl_trigger();
  combine_terms<kSep>(a, i, rows, w);
  __syncthreads();
  for (int64_t c = (int64_t)threadIdx.x * 8; c < a.h; c += kThreads * 8) {
    float acc[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) acc[u] = 0.f;
    // gather up to kBatch rows before accumulating any (all their loads in
    // flight at once), then add them in term order
    for (int t0 = 0; t0 < nterm; t0 += kBatch) {
      uint4 v[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int32_t r = t0 + b < nterm ? rows[t0 + b] : -1;
        const __nv_bfloat16* src = kSep && t0 + b >= a.k ? a.o_sh : a.o;
        v[b] = r >= 0 ? __ldg(reinterpret_cast<const uint4*>(src + (int64_t)r * a.h + c)) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (t0 + b >= nterm || rows[t0 + b] < 0) continue;
        float f[8];
        bf16x8_to_f32(v[b], f);
        const float wt = w[t0 + b];
#pragma unroll
        for (int u = 0; u < 8; ++u) acc[u] = fmaf(wt, f[u], acc[u]);
      }
    }
    uint4 o;
    __nv_bfloat162 p0 = __floats2bfloat162_rn(acc[0], acc[1]);
    __nv_bfloat162 p1 = __floats2bfloat162_rn(acc[2], acc[3]);
    __nv_bfloat162 p2 = __floats2bfloat162_rn(acc[4], acc[5]);
    __nv_bfloat162 p3 = __floats2bfloat162_rn(acc[6], acc[7]);
    o.x = *reinterpret_cast<uint32_t*>(&p0);
    o.y = *reinterpret_cast<uint32_t*>(&p1);
    o.z = *reinterpret_cast<uint32_t*>(&p2);
    o.w = *reinterpret_cast<uint32_t*>(&p3);
    *reinterpret_cast<uint4*>(a.y + i * a.h + c) = o;
  }
}

// The routed rows as MXFP8 codes of type kQ with E8M0 scales (oq, oq_sf;
// the combine exchange under combineQuantMode 3 / 4): 16 codes per thread
// (one 16-byte load a row, within one 32-element group), DQ_MX in fp32,
// the same fp32 sum in term order and the one bf16 rounding; the shared
// experts' rows stay bf16.
template <bool kSep, int kQ>
__global__ void __launch_bounds__(kThreads) k_combine_q(CombineArgs a) {
  __shared__ int32_t rows[kMaxTerms];
  __shared__ float w[kMaxTerms];
  const int64_t i = blockIdx.x;
  pdl_wait();
  pdl_trigger();
  combine_terms<kSep>(a, i, rows, w);
  __syncthreads();
  for (int64_t c = (int64_t)threadIdx.x * 16; c < a.h; c += kThreads * 16) {
    float acc[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) acc[u] = 0.f;
    for (int t0 = 0; t0 < a.k; t0 += kBatch) {
      uint4 v[kBatch];
      uint32_t qs[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int32_t r = t0 + b < a.k ? rows[t0 + b] : -1;
        v[b] = r >= 0 ? __ldg(reinterpret_cast<const uint4*>(a.oq + (int64_t)r * a.h + c)) : make_uint4(0u, 0u, 0u, 0u);
        qs[b] = r >= 0 ? (uint32_t)__ldg(a.oq_sf + (int64_t)r * (a.h / 32) + c / 32) : 0u;
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (t0 + b >= a.k || rows[t0 + b] < 0) continue;
        float f[16];
        fp8x8_dq<kQ>(make_uint2(v[b].x, v[b].y), qs[b], f);
        fp8x8_dq<kQ>(make_uint2(v[b].z, v[b].w), qs[b], f + 8);
        const float wt = w[t0 + b];
#pragma unroll
        for (int u = 0; u < 16; ++u) acc[u] = fmaf(wt, f[u], acc[u]);
      }
    }
    for (int t = a.k; t < a.k + a.n_shared; ++t) {
      const int32_t r = rows[t];
      if (r < 0) continue;
      const __nv_bfloat16* src = (kSep ? a.o_sh : a.o) + (int64_t)r * a.h + c;
      float f[16];
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(src)), f);
      bf16x8_to_f32(__ldg(reinterpret_cast<const uint4*>(src + 8)), f + 8);
#pragma unroll
      for (int u = 0; u < 16; ++u) acc[u] = fmaf(1.0f, f[u], acc[u]);
    }
    uint4 o[2];
#pragma unroll
    for (int hlf = 0; hlf < 2; ++hlf) {
      __nv_bfloat162 p0 = __floats2bfloat162_rn(acc[8 * hlf + 0], acc[8 * hlf + 1]);
      __nv_bfloat162 p1 = __floats2bfloat162_rn(acc[8 * hlf + 2], acc[8 * hlf + 3]);
      __nv_bfloat162 p2 = __floats2bfloat162_rn(acc[8 * hlf + 4], acc[8 * hlf + 5]);
      __nv_bfloat162 p3 = __floats2bfloat162_rn(acc[8 * hlf + 6], acc[8 * hlf + 7]);
      o[hlf].x = *reinterpret_cast<uint32_t*>(&p0);
      o[hlf].y = *reinterpret_cast<uint32_t*>(&p1);
      o[hlf].z = *reinterpret_cast<uint32_t*>(&p2);
      o[hlf].w = *reinterpret_cast<uint32_t*>(&p3);
    }
    *reinterpret_cast<uint4*>(a.y + i * a.h + c) = o[0];
    *reinterpret_cast<uint4*>(a.y + i * a.h + c + 8) = o[1];
  }
}

}  // namespace

cudaError_t launch_combine_rows(const __nv_bfloat16* rows, const int32_t* row_idx, const void* gate, int gate_bf16,
                                int64_t n, int64_t h, int k, const __nv_bfloat16* shared_rows, int n_shared,
                                __nv_bfloat16* y, cudaStream_t st, const uint8_t* rows_q, const uint8_t* rows_sf,
                                int rows_fmt) {
  CombineArgs a = {};
  a.o = rows;
  a.oq = rows_q;
  a.oq_sf = rows_sf;
  a.oq_fmt = rows_q ? rows_fmt : 0;
  a.o_sh = n_shared > 0 ? shared_rows : nullptr;
  a.pad_row = row_idx;
  a.gate = gate;
  a.gate_bf16 = gate_bf16;
  a.n_shared = n_shared;
  a.seg_mprefix = nullptr;
  a.n_routed = 0;
  a.n = n;
  a.h = h;
  a.k = k;
  a.y = y;
  a.rows_cap = INT64_MAX;  // the caller's row buffer: its size is not known here
  a.dev_err = nullptr;
  return launch_combine(a, st);
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
  if (a.n <= 0) return cudaSuccess;
  const dim3 g((unsigned)a.n), b(kThreads);
  const bool sep = a.o_sh && a.n_shared > 0;
  if (a.oq_fmt == MM_DT_FP8_E5M2 || a.oq_fmt == MM_DT_FP8_E4M3FN) {
    if (a.h % 32 != 0) return cudaErrorInvalidValue;
    if (a.oq_fmt == MM_DT_FP8_E5M2)
      return sep ? launch_pdl(k_combine_q<true, MM_DT_FP8_E5M2>, g, b, 0, st, a)
                 : launch_pdl(k_combine_q<false, MM_DT_FP8_E5M2>, g, b, 0, st, a);
    return sep ? launch_pdl(k_combine_q<true, MM_DT_FP8_E4M3FN>, g, b, 0, st, a)
               : launch_pdl(k_combine_q<false, MM_DT_FP8_E4M3FN>, g, b, 0, st, a);
  }
  if (sep) return launch_pdl(k_combine<true>, g, b, 0, st, a);
  return launch_pdl(k_combine<false>, g, b, 0, st, a);
}

}  // namespace mm
