// Shared device helpers of libmm_moe: MX quantisation of 32-element groups,
// mbarrier / TMA / tcgen05 wrappers (inline PTX for sm_103a), launch
// descriptors passed between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mm_moe.h"

namespace mm {

constexpr int kGroup = 32;            // MX group size
constexpr int kBM = 128;              // GEMM tile rows (expanded rows)
constexpr int kBK = 128;              // GEMM k-block (FP8 bytes = one 128B swizzle row)
constexpr int kSfChunk = 512;         // E8M0 bytes of one (128 rows x 128 k) scale tile

// MegaMoE activations (the ABI takes their names)
constexpr int MM_ACT_SWIGLU = 0;
constexpr int MM_ACT_SWIGLUSTEP = 1;
constexpr int MM_ACT_SWIGLUOAI = 2;
constexpr int MM_ACT_SITUGLU = 3;
constexpr int MM_ACT_GELU = 4;

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Byte offset of scale (row r, k-group g) inside the GEMM scale-tile layout:
// tiles of 128 rows x 4 groups (512 B), tile (r/128, g/4) at
// ((r/128) * groups4 + g/4) * 512, inside a tile (r%32)*16 + ((r%128)/32)*4 + g%4.
// This is the smem image that tcgen05.cp .32x128b.warpx4 spreads over the
// four TMEM sub-partitions for the block-scaled MMA.
__host__ __device__ inline int64_t sf_tile_offset(int64_t r, int64_t g, int64_t groups4) {
  return ((r >> 7) * groups4 + (g >> 2)) * kSfChunk + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (g & 3);
}

// ---------------------------------------------------------------------------
// MX scale of a group from its amax (finite, >= 0).  s = floor(log2 amax) -
// emax, clamped to [-127, 127]; amax = 0 or fp32-subnormal gives s = -127.
// Returns the E8M0 code and sets inv = 2^-s (exact; s <= 119 for fp32 data).
__device__ __forceinline__ uint32_t mx_scale(float amax, int emax, float& inv) {
  int eb = (int)(__float_as_uint(amax) >> 23);
  int s = eb == 0 ? -127 : eb - 127 - emax;
  s = s < -127 ? -127 : (s > 127 ? 127 : s);
  inv = __uint_as_float((uint32_t)(127 - s) << 23);
  return (uint32_t)(s + 127);
}

template <int kFmt>
__device__ __forceinline__ uint16_t cvt_fp8x2(float lo, float hi) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE,
                                            kFmt == MM_DT_FP8_E5M2 ? __NV_E5M2 : __NV_E4M3);
}

template <int kFmt>
__host__ __device__ constexpr int fmt_emax() {
  return kFmt == MM_DT_FP8_E5M2 ? 15 : (kFmt == MM_DT_FP4_E2M1 ? 2 : 8);
}

// Sixteen fp32 values scaled by inv -> 16 E2M1 codes, two per byte (element
// 2i in bits 0-3), nearest-even, saturated to +-6 (8 bytes in a uint2).
__device__ __forceinline__ uint2 pack16_fp4(const float* v, float inv) {
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t b = (uint32_t)__nv_cvt_float2_to_fp4x2(make_float2(v[2 * i] * inv, v[2 * i + 1] * inv),
                                                          __NV_E2M1, cudaRoundNearest);
    w[i >> 2] |= (b & 0xFFu) << (8 * (i & 3));
  }
  return make_uint2(w[0], w[1]);
}

// Eight fp32 values scaled by inv -> 8 FP8 bytes (little-endian in a uint2).
template <int kFmt>
__device__ __forceinline__ uint2 pack8_fp8(const float* v, float inv) {
  uint32_t w0 = (uint32_t)cvt_fp8x2<kFmt>(v[0] * inv, v[1] * inv) |
                ((uint32_t)cvt_fp8x2<kFmt>(v[2] * inv, v[3] * inv) << 16);
  uint32_t w1 = (uint32_t)cvt_fp8x2<kFmt>(v[4] * inv, v[5] * inv) |
                ((uint32_t)cvt_fp8x2<kFmt>(v[6] * inv, v[7] * inv) << 16);
  return make_uint2(w0, w1);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ void f16x8_to_f32(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
    float2 t = __half22float2(h);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ void raise_err(int32_t* dev_err, int bit) {
  if (dev_err) atomicOr(dev_err, bit);
}

// Checked build (compiled with MM_CHECK): in_bounds(ok, dev_err) reports a
// failed index test as MM_DEVERR_BOUNDS and returns it, so the caller skips
// the access; in the normal build it is `true` and the test compiles away.
#ifdef MM_CHECK
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif
__device__ __forceinline__ bool in_bounds(bool ok, int32_t* dev_err) {
  if (!kChecked) return true;
  if (!ok) raise_err(dev_err, MM_DEVERR_BOUNDS);
  return ok;
}

// Programmatic dependent launch.  A kernel started by launch_pdl may begin
// while the kernel before it on the stream is still finishing; it calls
// pdl_wait() before it reads anything an earlier kernel wrote (the wait
// returns once the previous grid has completed and its writes are visible;
// it is a no-op in a kernel launched without the attribute), and
// pdl_trigger() lets the next kernel begin launching once every CTA of this
// one has called it.  What a kernel does before pdl_wait() touches only its
// own shared memory, barriers and tensor memory.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Limit of every wait inside a kernel (a mbarrier phase, a grid barrier):
// past it the kernel raises MM_DEVERR_TIMEOUT and stops instead of hanging.
constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// Shared-memory addresses, mbarriers, TMA (inline PTX).
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0,
                                            int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"((uint64_t)map), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// Tiled store shared -> global of one box (bulk async group of this thread).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"((uint64_t)map),
               "r"(smem_u32(src)), "r"(c0), "r"(c1)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... and have completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Plain bulk copy global -> shared (16-byte aligned addresses, size % 16 == 0).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"((uint64_t)src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)map) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05 (5th-generation tensor core, tensor memory).
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on an mbarrier when every prior tcgen05 op of this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Copy a 32-row x 16-byte smem matrix into TMEM columns [taddr, taddr+4),
// replicated into all four 32-lane sub-partitions.
__device__ __forceinline__ void tc_cp_32x128b_warpx4(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// D[tmem] (+)= (A[smem] * SFA) x (B[smem] * SFB)^T, FP8 x FP8, E8M0 scale per 32 k.
__device__ __forceinline__ void tc_mma_mxf8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// 32 lanes x 32 columns of 32-bit TMEM -> 32 registers per thread (thread = lane).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
      "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]),
        "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor (tcgen05): start >> 4 at [0,14), leading
// byte offset >> 4 at [16,30), stride byte offset >> 4 at [32,46), version 1
// at [46,48), swizzle mode at [61,64) (0 none, 2 = 128-byte).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}

// Instruction descriptor of kind::mxf8f6f4 with E8M0 block scales:
// B scale id [4,6), A format [7,10), B format [10,13) (0 E4M3, 1 E5M2),
// K-major A and B (bits 15, 16 clear), N >> 3 at [17,23), scale type E8M0
// (bit 23), M >> 4 at [24,29), A scale id [29,31).
__host__ __device__ inline uint32_t idesc_mxf8(int a_fmt, int b_fmt, int m, int n) {
  return ((uint32_t)a_fmt << 7) | ((uint32_t)b_fmt << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
         ((uint32_t)(m >> 4) << 24);
}
__device__ __forceinline__ uint32_t idesc_with_sf(uint32_t base, uint32_t sf_id) {
  return base | (sf_id << 4) | (sf_id << 29);
}

}  // namespace mm
