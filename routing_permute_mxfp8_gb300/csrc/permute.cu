// Token permute fused with MX quantisation (dispatch), and weight-scale
// preparation.
//
// moe_token_permute article, 功能说明 / 返回值说明, and MoeInitRoutingV3
// step 5: output row d takes the source token of its flattened index; in
// the MX modes every group of 32 consecutive elements shares one E8M0
// exponent (MegaMoE README, A8W8-FP stage 1, Q_MX), with FP8 E4M3 / E5M2
// codes or packed FP4 E2M1 codes (A4W4-FP stage 1, quant_mode 9).
//
// The gather is turned around: one warp owns one source token (or a span of
// its 512-column slices, when tokens are too few to fill the GPU), reads
// its row once, quantises it once and stores the result at each of its K
// destinations (16-byte stores; one lane holds 16 consecutive elements, so
// a 32-element group is two lanes and its amax takes one shuffle).
#include "mm_route.cuh"

namespace mm {

namespace {

constexpr int kWarpsPerBlock = 8;

// The raw 16-byte vectors of 16 consecutive elements (zeros past the row),
// and their conversion to fp32: split so that a slice's loads can be issued
// before the previous slice is quantised and stored.
template <int kSrc>
struct Raw16 {
  static constexpr int kN = kSrc == MM_DT_FLOAT32 ? 4 : 2;
  uint4 u[kN];
};

template <int kSrc>
__device__ __forceinline__ void load_raw16(const char* row, int64_t col, int64_t h, Raw16<kSrc>& r) {
  constexpr int esz = kSrc == MM_DT_FLOAT32 ? 4 : 2;
  const uint4* p = reinterpret_cast<const uint4*>(row + col * esz);
#pragma unroll
  for (int i = 0; i < Raw16<kSrc>::kN; ++i) r.u[i] = col < h ? __ldg(p + i) : make_uint4(0u, 0u, 0u, 0u);
}

template <int kSrc>
__device__ __forceinline__ void raw16_to_f32(const Raw16<kSrc>& r, float* v) {
  if (kSrc == MM_DT_FLOAT32) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[4 * i] = __uint_as_float(r.u[i].x);
      v[4 * i + 1] = __uint_as_float(r.u[i].y);
      v[4 * i + 2] = __uint_as_float(r.u[i].z);
      v[4 * i + 3] = __uint_as_float(r.u[i].w);
    }
  } else if (kSrc == MM_DT_BFLOAT16) {
    bf16x8_to_f32(r.u[0], v);
    bf16x8_to_f32(r.u[1], v + 8);
  } else {
    f16x8_to_f32(r.u[0], v);
    f16x8_to_f32(r.u[1], v + 8);
  }
}

// Destination t (0 <= t < ndest) of the current row; d0 holds t = lane,
// d1 holds t = lane + 32.  Uniform across the warp.
__device__ __forceinline__ int32_t dest_at(int t, int32_t d0, int32_t d1) {
  int32_t a = __shfl_sync(0xffffffffu, d0, t & 31);
  int32_t b = __shfl_sync(0xffffffffu, d1, t & 31);
  return t < 32 ? a : b;
}

__device__ __forceinline__ void load_dests(const PermuteArgs& a, int64_t row, int lane, int32_t& d0,
                                           int32_t& d1, int& ndest) {
  ndest = a.k + a.n_extra;
  d0 = -1;
  d1 = -1;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int t = lane + 32 * h;
    int32_t d = -1;
    if (t < a.k) {
      d = a.dest ? a.dest[row * a.k + t] : (int32_t)row;
      if (d >= a.dest_limit) d = -1;
    } else if (t < ndest) {
      const int64_t de = (int64_t)a.extra_base[t - a.k] * kBM + row;
      d = in_bounds(de >= 0 && de < a.dest_limit, a.dev_err) ? (int32_t)de : -1;
    }
    if (h == 0) d0 = d; else d1 = d;
  }
  if (a.ids) {  // MegaMoE: the K experts of a token must be distinct
    const int id = lane < a.k ? a.ids[row * a.k + lane] : (int)(0x80000000u + (unsigned)lane);
    const unsigned peers = __match_any_sync(0xffffffffu, id);
    if (lane < a.k && __popc(peers) > 1) raise_err(a.dev_err, MM_DEVERR_DUPLICATE_ID);
  }
}

// wpt warps share a row when rows are few: warp `part` covers columns
// [part * span, +span) (span a multiple of 512).
template <int kSrc, int kFmt, bool kTiled>
// (6 blocks per SM for 2-byte sources: 40 registers; fp32 sources hold
// twice the raw vectors and are left at 5)
__global__ void __launch_bounds__(kWarpsPerBlock * 32, kSrc == MM_DT_FLOAT32 ? 5 : 6)
    k_permute_mx(PermuteArgs a, int wpt, int64_t span) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = (int)blockIdx.x * kWarpsPerBlock + warp;  // n * wpt < 2^31 (checked at launch)
  const int row = wpt == 1 ? gw : gw / wpt;
  const int part = gw - row * wpt;
  pdl_wait();
  pdl_trigger();
  if (row >= a.n) return;
  int32_t d0, d1;
  int ndest;
  load_dests(a, row, lane, d0, d1, ndest);
  if (a.dest_inv && part == 0 && lane < a.k && d0 >= 0) a.dest_inv[d0] = (int32_t)((int64_t)row * a.k + lane);
  constexpr int esz = kSrc == MM_DT_FLOAT32 ? 4 : 2;
  const char* src_row = static_cast<const char*>(a.src) + row * a.h * esz;
  uint8_t* out = static_cast<uint8_t*>(a.out);
  const int64_t groups = (a.h + 31) / 32;
  const int64_t groups4 = a.h / 128;
  const int64_t ostride = a.out_stride ? a.out_stride : (kFmt == MM_DT_FP4_E2M1 ? a.h / 2 : a.h);
  // slice c0 = 512 columns (16 per lane); the next slice's loads are in
  // flight while this one is quantised and written to the K destinations
  const int64_t cbeg = (int64_t)part * span;
  const int64_t cend = cbeg + span < a.h ? cbeg + span : a.h;
  Raw16<kSrc> cur;
  load_raw16<kSrc>(src_row, cbeg + lane * 16, a.h, cur);
  Raw16<kSrc> nxt = cur;
  for (int64_t c0 = cbeg; c0 < cend; c0 += 512) {
    const int64_t col = c0 + lane * 16;
    const bool act = col < a.h;
    if (c0 + 512 < cend) load_raw16<kSrc>(src_row, col + 512, a.h, nxt);
    float v[16];
    raw16_to_f32<kSrc>(cur, v);
    cur = nxt;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    float inv;
    const uint32_t code = mx_scale(amax, fmt_emax<kFmt>(), inv);
    // 16 codes of this lane: 16 FP8 bytes, or 8 bytes of packed FP4
    uint4 packed;
    if (kFmt == MM_DT_FP4_E2M1) {
      const uint2 p4 = pack16_fp4(v, inv);
      packed = make_uint4(p4.x, p4.y, 0u, 0u);
    } else {
      const uint2 lo = pack8_fp8<kFmt>(v, inv);
      const uint2 hi = pack8_fp8<kFmt>(v + 8, inv);
      packed = make_uint4(lo.x, lo.y, hi.x, hi.y);
    }
    // tile layout: lanes 8m..8m+7 hold groups 4m'..4m'+3; lane 8m packs them
    uint32_t word = 0;
    if (kTiled) {
      const uint32_t c1 = __shfl_down_sync(0xffffffffu, code, 2);
      const uint32_t c2 = __shfl_down_sync(0xffffffffu, code, 4);
      const uint32_t c3 = __shfl_down_sync(0xffffffffu, code, 6);
      word = code | (c1 << 8) | (c2 << 16) | (c3 << 24);
    }
    const int64_t g = col / 32;
    for (int t = 0; t < ndest; ++t) {
      const int32_t d = dest_at(t, d0, d1);
      if (d < 0 || !act) continue;
      if (kFmt == MM_DT_FP4_E2M1)
        *reinterpret_cast<uint2*>(out + (int64_t)d * ostride + col / 2) = make_uint2(packed.x, packed.y);
      else
        *reinterpret_cast<uint4*>(out + (int64_t)d * ostride + col) = packed;
      if (kTiled) {
        if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(a.scales + sf_tile_offset(d, g, groups4)) = word;
      } else if ((lane & 1) == 0) {
        a.scales[(int64_t)d * a.scale_cols + g] = (uint8_t)code;
      }
    }
  }
  if (!kTiled && groups < a.scale_cols && part == wpt - 1) {  // zero padding columns of the row layout
    for (int t = 0; t < ndest; ++t) {
      const int32_t d = dest_at(t, d0, d1);
      if (d < 0) continue;
      for (int64_t gg = groups + lane; gg < a.scale_cols; gg += 32) a.scales[(int64_t)d * a.scale_cols + gg] = 0;
    }
  }
}

// Copy mode: 16-byte vectors of the row to each destination; like
// k_permute_mx, wpt warps may share a row (bytes [part * span, +span)) and
// the next 512-byte slice is loaded before the current one is stored.
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    k_permute_copy(PermuteArgs a, int esz, int wpt, int64_t span) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gw = (int)blockIdx.x * kWarpsPerBlock + warp;  // n * wpt < 2^31 (checked at launch)
  const int row = wpt == 1 ? gw : gw / wpt;
  const int part = gw - row * wpt;
  pdl_wait();
  pdl_trigger();
  if (row >= a.n) return;
  int32_t d0, d1;
  int ndest;
  load_dests(a, row, lane, d0, d1, ndest);
  const int64_t rb = a.h * esz;
  const char* src = static_cast<const char*>(a.src) + row * rb;
  char* out = static_cast<char*>(a.out);
  const int64_t bbeg = (int64_t)part * span;
  const int64_t bend = bbeg + span < rb ? bbeg + span : rb;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  uint4 cur = bbeg + lane * 16 < rb ? __ldg(reinterpret_cast<const uint4*>(src + bbeg + lane * 16)) : zero;
  uint4 nxt = cur;
  for (int64_t off0 = bbeg; off0 < bend; off0 += 512) {
    const int64_t off = off0 + lane * 16;
    const bool act = off < rb;
    if (off0 + 512 < bend) nxt = off + 512 < rb ? __ldg(reinterpret_cast<const uint4*>(src + off + 512)) : zero;
    for (int t = 0; t < ndest; ++t) {
      const int32_t d = dest_at(t, d0, d1);
      if (d >= 0 && act) *reinterpret_cast<uint4*>(out + (int64_t)d * rb + off) = cur;
    }
    cur = nxt;
  }
}

// One thread per 4-byte word of the tile layout [E][pair][k-block][2][128
// words]: word wi of a tile holds the 4 scales (k 0-127) of row
// (wi % 4) * 32 + wi / 4 of its 128-row block, the order in which the
// 32x128b scale copy spreads them over TMEM lanes.  Rows past n_out read 0.
__global__ void k_prepare_wscales(const uint8_t* __restrict__ src, int64_t experts, int64_t n_out,
                                  int64_t k_red, int64_t npairs, int which, uint8_t* __restrict__ dst) {
  const int64_t kc_n = k_red / 128;
  const int64_t words = experts * npairs * kc_n * 2 * 128;
  const int64_t sc = k_red / 32;  // source row stride (2 * ceil(K/64) with K % 128 == 0)
  for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < words;
       w += (int64_t)gridDim.x * blockDim.x) {
    const int64_t wi = w & 127;
    const int64_t tile = w >> 7;  // ((e * npairs + pair) * kc_n + kc) * 2 + half
    const int64_t half = tile & 1;
    const int64_t kc = (tile >> 1) % kc_n;
    const int64_t pair = ((tile >> 1) / kc_n) % npairs;
    const int64_t e = (tile >> 1) / (kc_n * npairs);
    // GEMM1 pairs gate block p with up block I/128 + p; GEMM2 pairs 2p, 2p+1
    const int64_t blk = which == 1 ? half * npairs + pair : 2 * pair + half;
    const int64_t r = blk * 128 + (wi & 3) * 32 + (wi >> 2);
    uint32_t v = 0;
    if (r < n_out) v = __ldg(reinterpret_cast<const uint32_t*>(src + (e * n_out + r) * sc + kc * 4));
    reinterpret_cast<uint32_t*>(dst)[w] = v;
  }
}

__global__ void k_unpad(UnpadArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t j = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;
  if (j >= a.rows) return;
  const int32_t d = a.expanded_row_idx[j], p = a.pad_row[j];
  if (d < 0 || p < 0 || !in_bounds(d < a.rows && p < a.rows_cap, a.dev_err)) return;
  const int64_t ss = a.src_stride ? a.src_stride : a.qbytes;
  for (int64_t c = lane * 16; c < a.qbytes; c += 512)
    *reinterpret_cast<uint4*>(a.dst_q + (int64_t)d * a.qbytes + c) =
        *reinterpret_cast<const uint4*>(a.src_q + (int64_t)p * ss + c);
  const int64_t groups = a.cols / 32;
  for (int64_t g = lane; g < groups; g += 32)
    a.dst_sf[(int64_t)d * groups + g] = a.src_sf[sf_tile_offset(p, g, a.cols / 128)];
}

// Pre-quantised pass-through (MegaMoE dispatchQuantMode = 0): the source
// rows already hold FP8 codes (h bytes) or packed FP4 E2M1 codes (h / 2
// bytes) and src_scales their E8M0 scales, [n, h/32]; each row is copied to
// its destinations and its scales rewritten in the GEMM tile layout.  Warp
// per row, 16 bytes per lane, one 4-group scale word per lane and step.
__global__ void __launch_bounds__(kWarpsPerBlock * 32) k_permute_prequant(PermuteArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + warp;
  pdl_wait();
  pdl_trigger();
  if (row >= a.n) return;
  int32_t d0, d1;
  int ndest;
  load_dests(a, row, lane, d0, d1, ndest);
  if (a.dest_inv && lane < a.k && d0 >= 0) a.dest_inv[d0] = (int32_t)(row * a.k + lane);
  const int64_t rb = a.out_fmt == MM_DT_FP4_E2M1 ? a.h / 2 : a.h;
  const int64_t ostride = a.out_stride ? a.out_stride : rb;
  const uint8_t* src_row = static_cast<const uint8_t*>(a.src) + row * rb;
  const uint8_t* src_sf = a.src_scales + row * (a.h / 32);
  uint8_t* out = static_cast<uint8_t*>(a.out);
  const int64_t groups4 = a.h / 128;
  // destinations are read by warp shuffles: every lane runs the t loop
  for (int t = 0; t < ndest; ++t) {
    const int32_t d = dest_at(t, d0, d1);
    if (d < 0) continue;  // uniform across the warp
    for (int64_t col = lane * 16; col < rb; col += 512)
      *reinterpret_cast<uint4*>(out + (int64_t)d * ostride + col) = *reinterpret_cast<const uint4*>(src_row + col);
    for (int64_t w = lane; w < groups4; w += 32)
      *reinterpret_cast<uint32_t*>(a.scales + sf_tile_offset(d, 4 * w, groups4)) =
          *reinterpret_cast<const uint32_t*>(src_sf + 4 * w);
  }
}

template <int kSrc, int kFmt>
cudaError_t launch_mx_variant(const PermuteArgs& a, int, cudaStream_t st) {
  // split each row's 512-column slices over several warps until there are
  // about 2304 warps per SM (many waves of short warps balance better than
  // one wave of whole rows); packed FP4 writes half the bytes a slice, so
  // its warps keep at least two slices to amortise the per-warp
  // destination loads
  const int64_t slices = (a.h + 511) / 512;
  const int64_t max_wpt = kFmt == MM_DT_FP4_E2M1 ? (slices + 1) / 2 : slices;
  int64_t wpt = (int64_t)num_sms() * 2304 / a.n;
  if (wpt < 1) wpt = 1;
  if (wpt > max_wpt) wpt = max_wpt;
  const int64_t span = ceil_div(slices, wpt) * 512;
  wpt = ceil_div(a.h, span);
  if (a.n * wpt > 0x7fffffff - kWarpsPerBlock) return cudaErrorInvalidValue;
  const int64_t blocks = ceil_div(a.n * wpt, kWarpsPerBlock);
  if (a.scale_cols == 0)
    return launch_pdl(k_permute_mx<kSrc, kFmt, true>, dim3((unsigned)blocks), dim3(kWarpsPerBlock * 32), 0, st, a,
                      (int)wpt, span);
  return launch_pdl(k_permute_mx<kSrc, kFmt, false>, dim3((unsigned)blocks), dim3(kWarpsPerBlock * 32), 0, st, a,
                    (int)wpt, span);
}

template <int kSrc>
cudaError_t launch_mx_src(const PermuteArgs& a, int blocks, cudaStream_t st) {
  if (a.out_fmt == MM_DT_FP8_E5M2) return launch_mx_variant<kSrc, MM_DT_FP8_E5M2>(a, blocks, st);
  if (a.out_fmt == MM_DT_FP4_E2M1) return launch_mx_variant<kSrc, MM_DT_FP4_E2M1>(a, blocks, st);
  return launch_mx_variant<kSrc, MM_DT_FP8_E4M3FN>(a, blocks, st);
}

}  // namespace

cudaError_t launch_permute(const PermuteArgs& a, cudaStream_t st) {
  if (a.n <= 0) return cudaSuccess;
  const int64_t blocks64 = (a.n + kWarpsPerBlock - 1) / kWarpsPerBlock;
  if (blocks64 > 0x7fffffff) return cudaErrorInvalidValue;
  const int blocks = (int)blocks64;
  if (a.src_scales) {  // pre-quantised rows into the tile layout
    if (a.scale_cols != 0 || a.h % 128 != 0) return cudaErrorInvalidValue;
    return launch_pdl(k_permute_prequant, dim3(blocks), dim3(kWarpsPerBlock * 32), 0, st, a);
  }
  if (a.out_fmt < 0) {
    const int esz = a.src_dtype == MM_DT_FLOAT32 ? 4 : 2;
    const int64_t rb = a.h * esz, slices = (rb + 511) / 512;
    int64_t wpt = (int64_t)num_sms() * 2304 / a.n;  // as in launch_mx_variant (FP8 outputs)
    if (wpt < 1) wpt = 1;
    if (wpt > slices) wpt = slices;
    const int64_t span = ceil_div(slices, wpt) * 512;
    wpt = ceil_div(rb, span);
    if (a.n * wpt > 0x7fffffff - kWarpsPerBlock) return cudaErrorInvalidValue;
    return launch_pdl(k_permute_copy, dim3((unsigned)ceil_div(a.n * wpt, kWarpsPerBlock)), dim3(kWarpsPerBlock * 32),
                      0, st, a, esz, (int)wpt, span);
  }
  if (a.src_dtype == MM_DT_BFLOAT16) return launch_mx_src<MM_DT_BFLOAT16>(a, blocks, st);
  if (a.src_dtype == MM_DT_FLOAT16) return launch_mx_src<MM_DT_FLOAT16>(a, blocks, st);
  return launch_mx_src<MM_DT_FLOAT32>(a, blocks, st);
}

int64_t prepared_npairs(int64_t n_out, int which) { return which == 1 ? n_out / 256 : ceil_div(n_out, 256); }

cudaError_t launch_prepare_wscales(const uint8_t* src, int64_t experts, int64_t n_out, int64_t k_red, int which,
                                   uint8_t* dst, cudaStream_t st) {
  const int64_t npairs = prepared_npairs(n_out, which);
  const int64_t words = experts * npairs * (k_red / 128) * 2 * 128;
  if (words == 0) return cudaSuccess;
  int64_t blocks = ceil_div(words, 256);
  if (blocks > 65535 * 16) blocks = 65535 * 16;
  k_prepare_wscales<<<(unsigned)blocks, 256, 0, st>>>(src, experts, n_out, k_red, npairs, which, dst);
  return cudaGetLastError();
}

cudaError_t launch_unpad(const UnpadArgs& a, cudaStream_t st) {
  if (a.rows <= 0) return cudaSuccess;
  k_unpad<<<(unsigned)ceil_div(a.rows, 8), 256, 0, st>>>(a);
  return cudaGetLastError();
}

}  // namespace mm
