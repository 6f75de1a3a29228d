// Grouped block-scaled FP8 / FP4 GEMMs of the expert FFN on tcgen05 (sm_103a).
//
// MegaMoE README, A8W8-FP scenario:
//   stage 2  G_e, U_e = DQ_MX(X_hat_e) . DQ_MX(W1_e^(G|U))   then
//            A_e = SiLU(G_e) * U_e (swiglu, or another activation of
//            "Activation function formulas"; gelu acts on all 2I columns),
//            A_hat_e, S_A,e = Q_MX(A_e) in the dispatch FP8 type
//   stage 3  O_e = DQ_MX(A_hat_e) . DQ_MX(W2_e)
// DQ_MX happens inside the MMA: tcgen05.mma kind::mxf8f6f4 with one E8M0
// scale per 32 k for every row of A and of B (scale_vec::1X).  Weights are
// FP8 (A8W8-FP) or packed FP4 E2M1 (A8W4-FP), which TMA expands on load;
// in the A4W4-FP scenario GEMM1's A (the dispatched tokens) is packed FP4
// too and A_hat is MXFP8 E4M3.  Shared segments may have their own A type
// and A_hat type (the shared experts' own input quantisation type): their
// tiles use a second A tensor map, instruction descriptor and quantiser.
//
// Layout.  The expanded rows of every expert (and of each shared expert,
// which sees all tokens) form a segment padded to a multiple of 128 rows,
// so an M tile never straddles two experts.  One persistent kernel walks a
// flat tile list.  Segments with at least `big_mt` m tiles reuse each
// weight strip from L2 across their m tiles (tensor-bound tiles); smaller
// ones stream a weight strip from HBM for one tile (HBM-bound tiles).
// Each kind forms its own list (segment, n tile, m tile), ordered
// expert-major and n-major inside an expert, so the m tiles that share a
// weight strip run on neighbouring CTAs at the same time and the strip
// comes from HBM once; the two lists are then merged in proportion
// (Bresenham), so every wave of CTAs mixes both kinds and the tensor
// cores and HBM stay busy together instead of taking turns.
//
// CTA = 10 warps: warp 0 issues TMA (A tile 128x128 B, B tile 256x128 B,
// 128B swizzle) and bulk copies of the scale tiles into a 4-stage ring;
// warp 1 copies the scales to TMEM (tcgen05.cp) and issues the MMAs
// (M=128, N=256, K=32, four per k-block) into a 256-column fp32 TMEM
// accumulator; warps 2-9 drain the accumulator (tcgen05.ld, one row per
// thread, two warps per row quarter) and run the epilogue:
//   GEMM1: columns [0,128) are gate, [128,256) up, for the same 128
//          intermediate columns -> swiglu -> one MX group per 32 columns,
//          entirely within a thread; writes A_hat (FP8) and its scales
//          directly in GEMM2's operand layouts (the tile layout of the E8M0
//          scales that the 32x128b scale copy reads).
//   GEMM2: fp32 -> bf16 rows of O.
// Output stores: each warp stages a 32-row x 64-byte block (GEMM1: 64
// A_hat codes, GEMM2: 32 bf16) in shared memory (64B swizzle, no bank
// conflicts) and one TMA store writes it; blocks with padding rows, and
// launches whose segment table leaves no room for the staging buffers,
// store rows directly from registers.
// Every wait is bounded; a timeout sets MM_DEVERR_TIMEOUT and the CTA
// drains its own copies and MMAs, frees TMEM and returns.
#include <mutex>

#include "mm_route.cuh"

namespace mm {
namespace {

constexpr int kStages = 4;
constexpr int kEpiWarps = 8;                 // two warps per TMEM lane quarter
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr uint32_t kABytes = kBM * kBK;   // 16 KB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kOStageBytes = 32 * 64;  // one 32 x 32 bf16 block of O
constexpr int kTileN = 256;                  // output columns per tile (GEMM1: 128 gate + 128 up)
#ifndef MM_BIG_MTILES
#define MM_BIG_MTILES 2
#endif
constexpr int kBigMtiles = MM_BIG_MTILES;    // m tiles from which a segment's tiles count as tensor-bound

// Waits for the phase with `parity` of an mbarrier, giving up after
// limit_ns of %globaltimer time (false: the caller raises MM_DEVERR_TIMEOUT).
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns = kWaitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// Self-test of the failure path: one thread waits on a barrier that nothing
// arrives at, with the same bounded wait as the GEMM's pipeline.
__global__ void k_selftest_wait_timeout(uint64_t limit_ns, int32_t* dev_err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  if (!wait_bounded(&bar, 0, limit_ns)) raise_err(dev_err, MM_DEVERR_TIMEOUT);
}

struct GemmArgs {
  const uint8_t* sfa;
  const uint8_t* sfb;
  const uint8_t* sfb_sh;
  const int32_t* seg_rows;
  const int32_t* seg_mprefix;
  int nseg, n_routed;
  int K, N;
  int n_tiles;
  int big_mt;     // segments with >= big_mt m tiles form the tensor-bound list
  int npairs;     // 1 KB scale-tile pairs per expert and k-block in the prepared B scales
  uint32_t idesc, idesc_sh;
  int inter;
  uint8_t* act_q;
  uint8_t* act_sf;
  __nv_bfloat16* out;
  int32_t* dev_err;
  int o_stage;    // stage output blocks (A_hat / O) in shared memory for TMA stores
  int b_fp4, b_fp4_sh;  // routed / shared weights are packed FP4 E2M1
  int a_fp4, a_fp4_sh;  // routed / shared rows of A are packed FP4 E2M1 (GEMM1 of A4W4-FP)
  // mode 1: activation (MM_ACT_*), its parameters, and the width of A_hat
  int act;
  float act_c, act_alpha, act_beta, act_rbeta, act_beta_lin, act_rbeta_lin, act_gelu_k;
  int aw;
  int mtiles_cap;  // 128-row tiles of the A / output buffers (checked build)
  // mode 2, optional: padded row r goes to output row out_row[r] (rows of the
  // output: out_rows), stored from registers
  const int32_t* out_row;
  int64_t out_rows;
};

struct TileInfo {
  int seg, mt, nt;
};

// Checked build: the tile's rows lie inside its segment and inside the
// buffers (every role skips a tile that fails; the producer reports it).
__device__ __forceinline__ bool tile_fits(const GemmArgs& g, const int32_t* mpre, const TileInfo& ti) {
  if (!kChecked) return true;
  const int am = mpre[ti.seg] + ti.mt;
  const int rows_s = g.seg_rows[ti.seg];
  return ti.seg >= 0 && ti.seg < g.nseg && am >= 0 && am < g.mtiles_cap && rows_s >= 0 &&
         rows_s <= (mpre[ti.seg + 1] - mpre[ti.seg]) * kBM;
}

__device__ __forceinline__ TileInfo decode_tile(int t, const int32_t* mpre, int nseg, int n_tiles) {
  int lo = 0, hi = nseg;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (mpre[mid] * n_tiles <= t)
      lo = mid;
    else
      hi = mid;
  }
  TileInfo ti;
  ti.seg = lo;
  const int local = t - mpre[lo] * n_tiles;
  const int mts = mpre[lo + 1] - mpre[lo];
  ti.nt = local / mts;
  ti.mt = local - ti.nt * mts;
  return ti;
}

// Tile t of the merged order.  bpre / spre: prefixes of the m tiles of the
// big / small segments (a segment of the other kind adds 0).  The first t
// tiles hold floor(t * TB / T) big ones, so tile t is big when that count
// steps at t; each list keeps its own order.
__device__ __forceinline__ TileInfo decode_merged(int t, const int32_t* bpre, const int32_t* spre, int nseg,
                                                  int n_tiles) {
  const int64_t tb = (int64_t)bpre[nseg] * n_tiles;
  const int64_t tt = tb + (int64_t)spre[nseg] * n_tiles;
  const int cb = (int)((int64_t)t * tb / tt);
  const int cb1 = (int)((int64_t)(t + 1) * tb / tt);
  return cb1 > cb ? decode_tile(cb, bpre, nseg, n_tiles) : decode_tile(t - cb, spre, nseg, n_tiles);
}

// The MegaMoE activations ("Activation function formulas") on one 32-column
// chunk: sigma(z) = 1 / (1 + e^-z); clamp c (+inf when disabled), G_c =
// min(G, c), U_c = clip(U, -c, c).
//   swiglu      SiLU(G_c) U_c              swiglustep  min(SiLU(G), c) U_c
//   swigluoai   G_c sigma(alpha G_c) (U_c + beta)
//   situglu     beta tanh(G / beta) sigma(G) L(U), L(U) = U or beta_lin tanh(U / beta_lin)
//   gelu        Z sigma(sqrt(8/pi) (Z + 0.044715 Z^3)), element-wise (gv = Z)
// (CUDA's fast intrinsics __expf and __fdividef; the epilogue's arithmetic
// competes with the MMA issue and the loads for the SM's issue slots, so
// its instruction count shows in the GEMM's time on short-K shapes)
__device__ __forceinline__ float sigmoid_f(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

__device__ __forceinline__ void act_chunk(const GemmArgs& g, const uint32_t* gv, const uint32_t* uv, bool gelu,
                                          float* a) {
  const float c = g.act_c;
  if (gelu) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float z = __uint_as_float(gv[j]);
      a[j] = z * sigmoid_f(g.act_gelu_k * (z + 0.044715f * z * z * z));
    }
    return;
  }
  switch (g.act) {
    case MM_ACT_SWIGLUSTEP:
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float gf = __uint_as_float(gv[j]), uf = __uint_as_float(uv[j]);
        a[j] = fminf(gf * sigmoid_f(gf), c) * fminf(fmaxf(uf, -c), c);
      }
      break;
    case MM_ACT_SWIGLUOAI:
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float gc = fminf(__uint_as_float(gv[j]), c), uf = __uint_as_float(uv[j]);
        a[j] = gc * sigmoid_f(g.act_alpha * gc) * (fminf(fmaxf(uf, -c), c) + g.act_beta);
      }
      break;
    case MM_ACT_SITUGLU:
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float gf = __uint_as_float(gv[j]), uf = __uint_as_float(uv[j]);
        const float l = g.act_beta_lin > 0.f ? g.act_beta_lin * tanhf(uf * g.act_rbeta_lin) : uf;
        a[j] = g.act_beta * tanhf(gf * g.act_rbeta) * sigmoid_f(gf) * l;
      }
      break;
    default:  // swiglu
      if (c == INFINITY) {  // no clamp: SiLU(G) U = G / (1 + e^-G) * U
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float gf = __uint_as_float(gv[j]), uf = __uint_as_float(uv[j]);
          a[j] = __fdividef(gf, 1.0f + __expf(-gf)) * uf;
        }
        break;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float gc = fminf(__uint_as_float(gv[j]), c), uf = __uint_as_float(uv[j]);
        // SiLU(G_c) U_c = G_c * (1 / (1 + e^-G_c)) * U_c
        a[j] = gc * sigmoid_f(gc) * fminf(fmaxf(uf, -c), c);
      }
  }
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo, uint32_t hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<uint32_t*>(&v);
}

// kBN: tile width (B rows per tile); kAcc: accumulator buffers in TMEM (2
// lets the MMAs of the next tile run while the epilogue drains this one;
// kBN * kAcc plus 16 scale columns per stage must fit the 512 columns).
// The 32 codes of one MX group in FP8 type kF (inv = 2^-scale) as two 16-byte vectors.
template <int kF>
__device__ __forceinline__ void q_pack32(const float* a, float inv, uint4& lo, uint4& hi) {
  const uint2 p0 = pack8_fp8<kF>(a, inv), p1 = pack8_fp8<kF>(a + 8, inv);
  const uint2 p2 = pack8_fp8<kF>(a + 16, inv), p3 = pack8_fp8<kF>(a + 24, inv);
  lo = make_uint4(p0.x, p0.y, p1.x, p1.y);
  hi = make_uint4(p2.x, p2.y, p3.x, p3.y);
}

// kAlt: the shared segments' A_hat takes the other FP8 type (a separate
// instantiation, so the usual kernels carry no second quantiser)
template <int kMode, int kActFmt, int kBN, int kAcc, bool kAlt = false>
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_mx(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmAs,
              const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmBs,
              const __grid_constant__ CUtensorMap tmO, const GemmArgs g) {
  constexpr int kAltFmt = kActFmt == MM_DT_FP8_E5M2 ? MM_DT_FP8_E4M3FN : MM_DT_FP8_E5M2;
  constexpr uint32_t kBBytes = kBN * kBK;
  constexpr uint32_t kStageTx = kABytes + kBBytes + 512 + 1024;
  constexpr uint32_t kAccCols = kBN * kAcc;
  static_assert(kAccCols + 16 * kStages <= kTmemCols, "TMEM columns");
  static_assert(kMode == 2 || (kBN == 256 && kAcc == 1), "GEMM1 tiles are 128 gate + 128 up columns");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* smA = base;
  uint8_t* smB = smA + kStages * kABytes;
  uint8_t* smSFA = smB + kStages * kBBytes;
  uint8_t* smSFB = smSFA + kStages * 512;
  uint8_t* smO = smSFB + kStages * 1024;  // [kEpiWarps][32 x 64 B] when g.o_stage
  uint64_t* full = reinterpret_cast<uint64_t*>(smO + (g.o_stage ? kEpiWarps * kOStageBytes : 0));
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;      // [kAcc]
  uint64_t* acc_empty = acc_full + kAcc;     // [kAcc]
  uint64_t* drain = acc_empty + kAcc;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drain + 1);
  int32_t* mpre = reinterpret_cast<int32_t*>(tmem_holder + 4);
  int32_t* bpre = mpre + (g.nseg + 1);
  int32_t* spre = bpre + (g.nseg + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nseg = g.nseg;
  // set-up that reads nothing an earlier kernel wrote, before the wait for it
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < kAcc; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 32 * kEpiWarps);
    }
    mbar_init(drain, 1);
    fence_barrier_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    if (nseg > g.n_routed) {
      prefetch_tensormap(&tmAs);
      prefetch_tensormap(&tmBs);
    }
  }
  if (warp == 1) tmem_alloc(tmem_holder, kTmemCols);
  pdl_wait();
  pdl_trigger();
  for (int i = threadIdx.x; i <= nseg; i += kThreads) mpre[i] = g.seg_mprefix[i];
  __syncthreads();
  if (warp == 2) {
    // split the m-tile prefix into the big and the small segments' prefixes:
    // lane l scans segments [l*per, (l+1)*per), then a warp scan
    const int per = (nseg + 31) / 32;
    const int s0 = min(nseg, lane * per), s1 = min(nseg, s0 + per);
    int nb = 0, ns = 0;
    for (int sg = s0; sg < s1; ++sg) {
      const int m = mpre[sg + 1] - mpre[sg];
      if (m >= g.big_mt) nb += m; else ns += m;
    }
    int ib = nb, is = ns;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ub = __shfl_up_sync(0xffffffffu, ib, o), us = __shfl_up_sync(0xffffffffu, is, o);
      if (lane >= o) {
        ib += ub;
        is += us;
      }
    }
    int pb = ib - nb, ps = is - ns;
    for (int sg = s0; sg < s1; ++sg) {
      bpre[sg] = pb;
      spre[sg] = ps;
      const int m = mpre[sg + 1] - mpre[sg];
      if (m >= g.big_mt) pb += m; else ps += m;
    }
    if (lane == 31) {
      bpre[nseg] = ib;
      spre[nseg] = is;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int total = mpre[nseg] * g.n_tiles;
  const int kblocks = g.K / kBK;

  // E8M0 scale tiles of a stage -> its 16 TMEM columns (A, B rows 0-127, B rows 128-255)
  auto copy_sf = [&](uint32_t s) {
    const uint32_t c = tmem + kAccCols + s * 16;
    tc_cp_32x128b_warpx4(c, smem_desc(smem_u32(smSFA + s * 512), 0, 128, 0));
    tc_cp_32x128b_warpx4(c + 4, smem_desc(smem_u32(smSFB + s * 1024), 0, 128, 0));
    tc_cp_32x128b_warpx4(c + 8, smem_desc(smem_u32(smSFB + s * 1024 + 512), 0, 128, 0));
  };

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      uint32_t stage = 0, phase = 0, armed = 0, arm_par = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileInfo ti = decode_merged(t, bpre, spre, nseg, g.n_tiles);
        if (!in_bounds(tile_fits(g, mpre, ti), g.dev_err)) continue;
        const bool sh = ti.seg >= g.n_routed;
        const int e = sh ? ti.seg - g.n_routed : ti.seg;
        const CUtensorMap* mb = sh ? &tmBs : &tmB;
        const uint8_t* sfb = (sh ? g.sfb_sh : g.sfb) + (int64_t)e * g.npairs * kblocks * 1024;
        const int am = mpre[ti.seg] + ti.mt;
        // gated GEMM1: one 4-D box = gate rows nt*128.. and up rows I + nt*128..,
        // whose scale tiles are prepared as one pair; otherwise 256 consecutive
        // rows.  Under gelu, W1's scales are paired gate/up all the same, so the
        // two 128-row blocks 2nt, 2nt+1 come from two pairs.
        const bool gelu1 = kMode == 1 && g.act == MM_ACT_GELU;
        const int p0 = gelu1 ? (2 * ti.nt) % g.npairs : ti.nt;
        const int h0 = gelu1 ? (2 * ti.nt) / g.npairs : 0;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bounded(&empty[stage], phase ^ 1)) {
            ok = false;
            break;
          }
          // packed FP4 operands count their global (packed) bytes
          mbar_arrive_expect_tx(&full[stage], kStageTx - ((sh ? g.b_fp4_sh : g.b_fp4) ? kBBytes / 2 : 0) -
                                                  ((sh ? g.a_fp4_sh : g.a_fp4) ? kABytes / 2 : 0));
          armed |= 1u << stage;
          arm_par = (arm_par & ~(1u << stage)) | (phase << stage);
          tma_load_2d(smA + stage * kABytes, sh ? &tmAs : &tmA, &full[stage], kb * kBK, am * kBM);
          if (kMode == 1 && !gelu1)
            tma_load_4d(smB + stage * kBBytes, mb, &full[stage], kb * kBK, ti.nt * 128, 0, e);
          else
            tma_load_3d(smB + stage * kBBytes, mb, &full[stage], kb * kBK, ti.nt * 256, e);
          bulk_load(smSFA + stage * 512, g.sfa + ((int64_t)am * kblocks + kb) * 512, 512, &full[stage]);
          if (!gelu1) {
            bulk_load(smSFB + stage * 1024, sfb + ((int64_t)ti.nt * kblocks + kb) * 1024, 1024, &full[stage]);
          } else {
            // blocks 2nt and 2nt+1 are in consecutive pairs (same half), or
            // straddle from the last gate pair into the first up pair
            const int p1 = (2 * ti.nt + 1) % g.npairs, h1 = (2 * ti.nt + 1) / g.npairs;
            bulk_load(smSFB + stage * 1024, sfb + (((int64_t)p0 * kblocks + kb) * 2 + h0) * 512, 512, &full[stage]);
            bulk_load(smSFB + stage * 1024 + 512, sfb + (((int64_t)p1 * kblocks + kb) * 2 + h1) * 512, 512,
                      &full[stage]);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok) raise_err(g.dev_err, MM_DEVERR_TIMEOUT);
      // every copy this thread started must land before the CTA exits
      for (int s = 0; s < kStages; ++s)
        if ((armed >> s) & 1u) wait_bounded(&full[s], (arm_par >> s) & 1u);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      uint32_t stage = 0, phase = 0, tcount = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileInfo ti = decode_merged(t, bpre, spre, nseg, g.n_tiles);
        if (!tile_fits(g, mpre, ti)) continue;
        const uint32_t idb = ti.seg >= g.n_routed ? g.idesc_sh : g.idesc;
        const uint32_t buf = tcount % kAcc, use = tcount / kAcc;
        if (!wait_bounded(&acc_empty[buf], (use & 1) ^ 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t dacc = tmem + buf * kBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait_bounded(&full[stage], phase)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // the scale copies serialise with the MMAs in the tensor pipe
          // (one copy instruction costs about a sixth of this k-block's MMAs)
          copy_sf(stage);
          const uint32_t sfc = tmem + kAccCols + stage * 16;
          const uint32_t a0 = smem_u32(smA + stage * kABytes);
          const uint32_t b0 = smem_u32(smB + stage * kBBytes);
#pragma unroll
          for (int k = 0; k < kBK / 32; ++k) {
            tc_mma_mxf8(dacc, smem_desc(a0 + 32 * k, 0, 1024, 2), smem_desc(b0 + 32 * k, 0, 1024, 2),
                        idesc_with_sf(idb, (uint32_t)k), sfc, sfc + 4, (kb | k) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
        ++tcount;
      }
      if (!ok) raise_err(g.dev_err, MM_DEVERR_TIMEOUT);
      tc_commit(drain);  // all MMAs / copies of this thread complete before TMEM is freed
      wait_bounded(drain, 0);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    // Warp w reads TMEM lanes [32*(w%4), +32) (its lane quarter); the two
    // warps of a quarter split the columns.  Each thread loads its whole
    // share of the accumulator first and releases TMEM before doing the
    // math and the global stores, so the next tile's MMAs start early.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    uint32_t tcount = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const TileInfo ti = decode_merged(t, bpre, spre, nseg, g.n_tiles);
      if (!tile_fits(g, mpre, ti)) continue;
      const uint32_t buf = tcount % kAcc, use = tcount / kAcc;
      if (!wait_bounded(&acc_full[buf], use & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t trow = tmem + buf * kBN + ((uint32_t)(q * 32) << 16);
      const bool valid = r < g.seg_rows[ti.seg] - ti.mt * kBM;
      const int64_t grow = (int64_t)(mpre[ti.seg] + ti.mt) * kBM + r;
      if (kMode == 1) {
        // gated activations: output columns [nt*128 + 64*half, +64) from the
        //   gate accumulator columns c*32 and the up columns 128 + c*32 for
        //   the chunks c = 2*half, 2*half+1 (v[0..1] gate, v[2..3] up);
        // gelu: output columns [nt*256 + 128*half, +128) from the accumulator
        //   chunks 4*half .. 4*half+3 (v[0..3]), element-wise
        const bool gelu = g.act == MM_ACT_GELU;
        uint32_t v[4][32];
        if (gelu) {
#pragma unroll
          for (int i = 0; i < 4; ++i) tmem_ld_32x32b_x32(trow + (4 * half + i) * 32, v[i]);
        } else {
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int c = 2 * half + i;
            tmem_ld_32x32b_x32(trow + c * 32, v[i]);
            tmem_ld_32x32b_x32(trow + 128 + c * 32, v[2 + i]);
          }
        }
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
        const int nout = gelu ? 4 : 2;  // 32-column output chunks of this thread
        // A_hat of a shared segment in the shared experts' activation type when it differs
        const bool alt = kAlt && ti.seg >= g.n_routed;
        const int ocol0 = gelu ? ti.nt * 256 + 128 * half : ti.nt * 128 + 64 * half;
        // TMA stores of the warp's 32 x 64 FP8 blocks when all its rows are real
        const bool staged = g.o_stage && g.seg_rows[ti.seg] - ti.mt * kBM >= (q + 1) * 32;
        uint8_t* stg = smO + (warp - 2) * kOStageBytes;
        uint32_t sfw = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (i >= nout) break;
          if (staged && (i & 1) == 0) {
            if (lane == 0) bulk_wait_read();  // the previous block has left the buffer
            __syncwarp();
          }
          float a[32];
          act_chunk(g, v[i], v[(2 + i) & 3], gelu, a);  // up chunk unused under gelu
          float amax = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(a[j]));
          float inv;
          const uint32_t code = alt ? mx_scale(amax, fmt_emax<kAltFmt>(), inv) : mx_scale(amax, fmt_emax<kActFmt>(), inv);
          sfw |= code << (8 * i);
          if (staged || valid) {
            uint4 lo, hi;
            if (alt)
              q_pack32<kAltFmt>(a, inv, lo, hi);
            else
              q_pack32<kActFmt>(a, inv, lo, hi);
            if (staged) {
              const int sw = (lane >> 1) & 3;  // 64B swizzle of row `lane`
              *reinterpret_cast<uint4*>(stg + lane * 64 + (((2 * (i & 1)) ^ sw) << 4)) = lo;
              *reinterpret_cast<uint4*>(stg + lane * 64 + (((2 * (i & 1) + 1) ^ sw) << 4)) = hi;
            } else {
              uint8_t* dst = g.act_q + grow * g.aw + ocol0 + i * 32;
              *reinterpret_cast<uint4*>(dst) = lo;
              *reinterpret_cast<uint4*>(dst + 16) = hi;
            }
          }
          if (staged && (i & 1) == 1) {
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmO, stg, ocol0 + (i - 1) * 32, (int)((grow - r) + q * 32));
              bulk_commit();
            }
          }
        }
        if (valid) {
          uint8_t* sfp = g.act_sf + sf_tile_offset(grow, ocol0 / 32, g.aw / 128);
          if (gelu)
            *reinterpret_cast<uint32_t*>(sfp) = sfw;
          else
            *reinterpret_cast<uint16_t*>(sfp) = (uint16_t)sfw;
        }
      } else {
        // output columns [nt*kBN + 128*half, +128) (the last chunks of a
        // tile narrower than 256 columns: half 1 has fewer)
        constexpr int kChunks = kBN / 32;
        uint32_t v[4][32];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (4 * half + i < kChunks) tmem_ld_32x32b_x32(trow + (4 * half + i) * 32, v[i]);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
        // TMA store when all 32 rows of this lane quarter are real rows
        const bool staged = g.o_stage && g.seg_rows[ti.seg] - ti.mt * kBM >= (q + 1) * 32;
        int64_t orow = grow;
        if (g.out_row && valid) {
          const int64_t m = g.out_row[grow];
          orow = in_bounds(m >= 0 && m < g.out_rows, g.dev_err) ? m : -1;
        }
        uint8_t* stg = smO + (warp - 2) * kOStageBytes;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int64_t col = (int64_t)ti.nt * kBN + (4 * half + i) * 32;
          if (staged && 4 * half + i < kChunks && col < g.N) {
            if (lane == 0) bulk_wait_read();  // the previous block has left the buffer
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 4; ++u)
              *reinterpret_cast<uint4*>(stg + lane * 64 + ((u ^ ((lane >> 1) & 3)) << 4)) =
                  make_uint4(pack_bf16x2(v[i][8 * u], v[i][8 * u + 1]), pack_bf16x2(v[i][8 * u + 2], v[i][8 * u + 3]),
                             pack_bf16x2(v[i][8 * u + 4], v[i][8 * u + 5]),
                             pack_bf16x2(v[i][8 * u + 6], v[i][8 * u + 7]));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmO, stg, (int)col, (int)((grow - r) + q * 32));
              bulk_commit();
            }
          } else if (4 * half + i < kChunks && valid && col < g.N && orow >= 0) {
            uint4* dst = reinterpret_cast<uint4*>(g.out + orow * g.N + col);
#pragma unroll
            for (int u = 0; u < 4; ++u)
              dst[u] = make_uint4(pack_bf16x2(v[i][8 * u], v[i][8 * u + 1]), pack_bf16x2(v[i][8 * u + 2], v[i][8 * u + 3]),
                                  pack_bf16x2(v[i][8 * u + 4], v[i][8 * u + 5]),
                                  pack_bf16x2(v[i][8 * u + 6], v[i][8 * u + 7]));
          }
        }
      }
      ++tcount;
    }
    if (g.o_stage && lane == 0) bulk_wait_all();
    if (!ok) raise_err(g.dev_err, MM_DEVERR_TIMEOUT);
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// FP8 byte matrix [outer][inner] (inner contiguous), box inner 128 codes,
// 128B swizzle; or packed FP4 E2M1 (inner / 2 bytes a row), expanded by TMA
// like the FP4 weights below.
bool map_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_outer, bool fp4 = false,
            uint64_t stride = 0) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {stride ? stride : (fp4 ? inner / 2 : inner)};
  cuuint32_t box[2] = {(cuuint32_t)kBK, box_outer};
  cuuint32_t es[2] = {1, 1};
  EncodeTiledFn f = encode_fn();
  return f && f(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                const_cast<void*>(ptr), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Stacked weights [E][N][K]: FP8 bytes, or FP4 E2M1 packed two per byte,
// which TMA expands into the 16-byte-aligned groups of 16 codes that the
// kind::mxf8f6f4 MMA reads (a box row of 128 codes fills 128 smem bytes,
// like FP8, so the stage layout does not change).
bool map_3d(CUtensorMap* m, const void* ptr, uint64_t k, uint64_t n, uint64_t e, uint32_t box_rows,
            bool fp4 = false) {
  cuuint64_t dims[3] = {k, n, e};
  const uint64_t row_bytes = fp4 ? k / 2 : k;
  cuuint64_t strides[2] = {row_bytes, n * row_bytes};
  cuuint32_t box[3] = {(cuuint32_t)kBK, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  EncodeTiledFn f = encode_fn();
  return f && f(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 3,
                const_cast<void*>(ptr), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Gated weight1 [E][2I][K] viewed as {K, I, 2, E}: one box of 2 x 128 rows
// brings a tile's gate rows and the matching up rows (I further down) to
// consecutive 16 KB halves of the stage.
bool map_4d_pair(CUtensorMap* m, const void* ptr, uint64_t k, uint64_t inter, uint64_t e, bool fp4) {
  cuuint64_t dims[4] = {k, inter, 2, e};
  const uint64_t row_bytes = fp4 ? k / 2 : k;
  cuuint64_t strides[3] = {row_bytes, inter * row_bytes, 2 * inter * row_bytes};
  cuuint32_t box[4] = {(cuuint32_t)kBK, 128, 2, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  EncodeTiledFn f = encode_fn();
  return f && f(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 4,
                const_cast<void*>(ptr), dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output matrix [rows][cols] (cols contiguous) of bf16 (GEMM2's O) or FP8
// bytes (GEMM1's A_hat), box 64 bytes x 32 rows, 64B swizzle: the blocks
// that the epilogue stages in shared memory.
bool map_out(CUtensorMap* m, const void* ptr, bool bf16, uint64_t cols, uint64_t rows) {
  const uint64_t esz = bf16 ? 2 : 1;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * esz};
  cuuint32_t box[2] = {(cuuint32_t)(64 / esz), 32};
  cuuint32_t es[2] = {1, 1};
  EncodeTiledFn f = encode_fn();
  return f && f(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr),
                dims, strides, box, es,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// instruction-descriptor format code (kind::mxf8f6f4): E4M3 0, E5M2 1, E2M1 5
int fmt_code(int dt) { return dt == MM_DT_FP8_E5M2 ? 1 : (dt == MM_DT_FP4_E2M1 ? 5 : 0); }

template <int kMode, int kActFmt, int kBN, int kAcc, bool kAlt = false>
cudaError_t run(const GemmLaunch& L, const CUtensorMap& ma, const CUtensorMap& mas, const CUtensorMap& mb,
                const CUtensorMap& mbs, const CUtensorMap& mo, GemmArgs g, int grid, cudaStream_t st) {
  auto kern = k_gemm_mx<kMode, kActFmt, kBN, kAcc, kAlt>;
  const size_t base = 1024 + (size_t)kStages * (kABytes + kBN * kBK + 512 + 1024) +
                      8 * (2 * kStages + 2 * kAcc + 1) + 16 + 12 * (size_t)(g.nseg + 1);
  constexpr size_t kMaxSmem = 232448;
  // output staging buffers only where the segment table leaves room for them
  g.o_stage = (base + kEpiWarps * kOStageBytes <= kMaxSmem && !g.out_row) ? 1 : 0;
  const size_t smem = base + (g.o_stage ? kEpiWarps * kOStageBytes : 0);
  if (smem > kMaxSmem) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, st, ma, mas, mb, mbs, mo, g);
}

}  // namespace


cudaError_t launch_selftest_wait_timeout(uint64_t limit_ns, int32_t* dev_err, cudaStream_t st) {
  k_selftest_wait_timeout<<<1, 32, 0, st>>>(limit_ns, dev_err);
  return cudaGetLastError();
}

int num_sms() {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static int n[kMaxDevices] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  std::lock_guard<std::mutex> g(mu);
  if (n[dev] == 0) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 1;
    n[dev] = v;
  }
  return n[dev];
}

cudaError_t launch_gemm(const GemmLaunch& L, cudaStream_t st) {
  const int nseg = L.n_routed + L.n_shared;
  const int bn = kTileN;
  const bool pair_map = L.mode == 1 && L.act != MM_ACT_GELU;
  auto map_b = [&](CUtensorMap* m, const void* p, int64_t experts, int fmt) {
    const bool fp4 = fmt == MM_DT_FP4_E2M1;
    return pair_map ? map_4d_pair(m, p, (uint64_t)L.K, (uint64_t)L.inter, (uint64_t)experts, fp4)
                    : map_3d(m, p, (uint64_t)L.K, (uint64_t)L.N, (uint64_t)experts, (uint32_t)bn, fp4);
  };
  CUtensorMap ma, mas, mb, mbs;
  if (!map_2d(&ma, L.a, (uint64_t)L.K, (uint64_t)L.rows_cap, kBM, L.a_fmt == MM_DT_FP4_E2M1, (uint64_t)L.a_stride))
    return cudaErrorInvalidValue;
  if (L.n_shared > 0 && L.a_fmt_sh != L.a_fmt) {
    if (!map_2d(&mas, L.a, (uint64_t)L.K, (uint64_t)L.rows_cap, kBM, L.a_fmt_sh == MM_DT_FP4_E2M1,
                (uint64_t)L.a_stride))
      return cudaErrorInvalidValue;
  } else {
    mas = ma;
  }
  if (!map_b(&mb, L.b, L.n_routed, L.b_fmt)) return cudaErrorInvalidValue;
  if (L.n_shared > 0) {
    if (!map_b(&mbs, L.b_sh, L.n_shared, L.b_fmt_sh)) return cudaErrorInvalidValue;
  } else {
    mbs = mb;
  }
  CUtensorMap mo;
  if (L.mode == 2) {
    if (!map_out(&mo, L.out, true, (uint64_t)L.N, (uint64_t)L.rows_cap)) return cudaErrorInvalidValue;
  } else {
    const int64_t aw = L.act == MM_ACT_GELU ? 2 * L.inter : L.inter;
    if (!map_out(&mo, L.act_q, false, (uint64_t)aw, (uint64_t)L.rows_cap)) return cudaErrorInvalidValue;
  }
  GemmArgs g;
  g.sfa = L.sfa;
  g.sfb = L.sfb;
  g.sfb_sh = L.n_shared > 0 ? L.sfb_sh : L.sfb;
  g.seg_rows = L.seg_rows;
  g.seg_mprefix = L.seg_mprefix;
  g.nseg = nseg;
  g.n_routed = L.n_routed;
  g.K = (int)L.K;
  g.N = (int)L.N;
  g.n_tiles = L.mode == 1 ? (int)(L.act == MM_ACT_GELU ? L.N / 256 : L.inter / 128) : (int)ceil_div(L.N, bn);
  g.big_mt = kBigMtiles;
  g.npairs = (int)prepared_npairs(L.N, L.mode);
  g.b_fp4 = L.b_fmt == MM_DT_FP4_E2M1;
  g.a_fp4 = L.a_fmt == MM_DT_FP4_E2M1;
  g.a_fp4_sh = (L.n_shared > 0 ? L.a_fmt_sh : L.a_fmt) == MM_DT_FP4_E2M1;
  const bool alt = L.mode == 1 && L.n_shared > 0 && L.act_fmt_sh != L.act_fmt;
  g.act = L.act;
  g.act_c = L.act_c;
  g.act_alpha = L.act_alpha;
  g.act_beta = L.act_beta;
  g.act_rbeta = L.act_beta != 0.f ? 1.0f / L.act_beta : 0.f;
  g.act_beta_lin = L.act_beta_lin;
  g.act_rbeta_lin = L.act_beta_lin > 0.f ? 1.0f / L.act_beta_lin : 0.f;
  g.act_gelu_k = (float)sqrt(8.0 / acos(-1.0));
  g.aw = L.mode == 1 ? (L.act == MM_ACT_GELU ? 2 * L.inter : L.inter) : 0;
  g.b_fp4_sh = (L.n_shared > 0 ? L.b_fmt_sh : L.b_fmt) == MM_DT_FP4_E2M1;
  g.idesc = idesc_mxf8(fmt_code(L.a_fmt), fmt_code(L.b_fmt), kBM, bn);
  g.idesc_sh = idesc_mxf8(fmt_code(L.n_shared > 0 ? L.a_fmt_sh : L.a_fmt),
                          fmt_code(L.n_shared > 0 ? L.b_fmt_sh : L.b_fmt), kBM, bn);
  g.inter = L.inter;
  g.act_q = L.act_q;
  g.act_sf = L.act_sf;
  g.out = L.out;
  g.dev_err = L.dev_err;
  g.mtiles_cap = (int)(L.rows_cap / kBM);
  g.out_row = L.mode == 2 ? L.out_row : nullptr;
  g.out_rows = L.out_rows;
  // upper bound of the tile count decides how many persistent CTAs to start
  const int64_t max_mtiles = L.rows_cap / kBM;
  int64_t grid = max_mtiles * g.n_tiles;
  if (grid > num_sms()) grid = num_sms();
  if (grid < 1) grid = 1;
  if (L.mode == 1) {  // the template argument is A_hat's type
    if (L.act_fmt != MM_DT_FP8_E5M2 && L.act_fmt != MM_DT_FP8_E4M3FN) return cudaErrorInvalidValue;
    if (alt && L.act_fmt_sh != MM_DT_FP8_E5M2 && L.act_fmt_sh != MM_DT_FP8_E4M3FN) return cudaErrorInvalidValue;
    if (L.act_fmt == MM_DT_FP8_E5M2)
      return alt ? run<1, MM_DT_FP8_E5M2, 256, 1, true>(L, ma, mas, mb, mbs, mo, g, (int)grid, st)
                 : run<1, MM_DT_FP8_E5M2, 256, 1>(L, ma, mas, mb, mbs, mo, g, (int)grid, st);
    return alt ? run<1, MM_DT_FP8_E4M3FN, 256, 1, true>(L, ma, mas, mb, mbs, mo, g, (int)grid, st)
               : run<1, MM_DT_FP8_E4M3FN, 256, 1>(L, ma, mas, mb, mbs, mo, g, (int)grid, st);
  }
  return run<2, MM_DT_FP8_E4M3FN, 256, 1>(L, ma, mas, mb, mbs, mo, g, (int)grid, st);
}

}  // namespace mm
