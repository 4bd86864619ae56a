// mp_device.cuh — device-side building blocks of libmpnum (sm_103a).
//
// Number-format conversions use the hardware cvt instructions (RNE, and
// .satfinite where a cast saturates); every floating-point operation whose
// rounding matters is written with an explicit _rn intrinsic so that the
// compiler cannot fuse it into an FMA.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mp {

// ---------------------------------------------------------------------------
// Streaming memory access.  Each element of the hot path is touched once, so
// loads and stores carry the evict-first (.cs) hint.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 ld_cs(const void* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }
__device__ __forceinline__ float4 ld_cs_f4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st_cs(void* p, uint4 v) { __stcs(reinterpret_cast<uint4*>(p), v); }
__device__ __forceinline__ void st_cs_f4(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }
__device__ __forceinline__ uint4 ld_plain(const void* p) { return *reinterpret_cast<const uint4*>(p); }

// ---------------------------------------------------------------------------
// 16-bit <-> 32-bit.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float f16lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu))); }
__device__ __forceinline__ float f16hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// Two floats to packed 16-bit, round to nearest even; NaN -> 0x7FFF.
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  uint32_t r = *reinterpret_cast<uint32_t*>(&h);
  if (__builtin_expect((lo != lo) | (hi != hi), 0)) {
    if (lo != lo) r = (r & 0xFFFF0000u) | 0x7FFFu;
    if (hi != hi) r = (r & 0x0000FFFFu) | 0x7FFF0000u;
  }
  return r;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  uint32_t r = *reinterpret_cast<uint32_t*>(&h);
  if (__builtin_expect((lo != lo) | (hi != hi), 0)) {
    if (lo != lo) r = (r & 0xFFFF0000u) | 0x7FFFu;
    if (hi != hi) r = (r & 0x0000FFFFu) | 0x7FFF0000u;
  }
  return r;
}

// ---------------------------------------------------------------------------
// FP8 / FP4 conversions (first cvt source lands in the high part).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t cvt_e5m2x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Packed E2M1 pair, round to nearest even, saturating at 6: lo -> bits 0..3.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  unsigned short r;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u16.u8 %0, t; }" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Packed FP6 pair (one 6-bit code per byte, upper two bits zero), round to
// nearest even, saturating at the largest finite value: lo -> bits 0..7.
__device__ __forceinline__ uint32_t cvt_e2m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e2m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ uint32_t cvt_e3m2x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e3m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// Non-negative finite E4M3 byte (0x00..0x7E) -> float, exact.  Normal codes
// rebias the exponent field (7 -> 127); subnormals are m * 2^-9.
__device__ __forceinline__ float e4m3_pos_to_f32(uint32_t code) {
  const uint32_t c = code & 0x7Fu;
  return (c >= 8u) ? __uint_as_float((c << 20) + (120u << 23)) : __fmul_rn((float)c, 0.001953125f);
}
// E2M1 magnitude table (times 2) packed in nibbles: 0,1,2,3,4,6,8,12.
__device__ __forceinline__ float e2m1_to_f32(uint32_t code) {
  uint32_t twice = (0xC8643210u >> ((code & 7u) * 4u)) & 0xFu;
  float v = __fmul_rn((float)twice, 0.5f);
  return (code & 8u) ? -v : v;
}

// NaN-propagating max of |a| into acc (PTX max.NaN).
__device__ __forceinline__ float max_abs_nan(float acc, float a) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(acc), "f"(fabsf(a)));
  return r;
}
// NaN-propagating max of the magnitudes of a packed 16-bit pair w into the
// packed magnitudes acc (PTX max.NaN on bf16x2 / f16x2; a NaN lane becomes the
// canonical NaN of its half).
template <bool BF16>
__device__ __forceinline__ uint32_t max_abs_nan_x2(uint32_t acc, uint32_t w) {
  uint32_t r;
  const uint32_t a = w & 0x7FFF7FFFu;
  if constexpr (BF16)
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(a));
  else
    asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(r) : "r"(acc), "r"(a));
  return r;
}
// Non-negative float or NaN -> ordered bits, NaN canonical (0x7FC00000).
__device__ __forceinline__ uint32_t amax_bits(float a) {
  return (a != a) ? 0x7FC00000u : __float_as_uint(a);
}

// ---------------------------------------------------------------------------
// Block-wide reductions (blockDim.x a multiple of 32, <= 1024).
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* smem32) {
  v = __reduce_max_sync(0xFFFFFFFFu, v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) smem32[warp] = v;
  __syncthreads();
  uint32_t r = 0;
  if (warp == 0) {
    r = (lane < (int)(blockDim.x >> 5)) ? smem32[lane] : 0u;
    r = __reduce_max_sync(0xFFFFFFFFu, r);
  }
  return r;  // valid in warp 0
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11).
// ---------------------------------------------------------------------------
struct u32x4 {
  uint32_t x, y, z, w;
};
__device__ __forceinline__ u32x4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                               uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return u32x4{c0, c1, c2, c3};
}

// ---------------------------------------------------------------------------
// Random signs of the Hadamard transform, applied to packed BF16 pairs: word
// k of a 16-element tile holds elements 2k (low half) and 2k+1 (high half);
// bit j of `mask` set negates element j.
// ---------------------------------------------------------------------------
struct SignWords {
  uint32_t w[8];
};
__device__ __forceinline__ SignWords sign_words(uint32_t mask) {
  SignWords s;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    s.w[k] = (((mask >> (2 * k)) & 1u) << 15) | (((mask >> (2 * k + 1)) & 1u) << 31);
  return s;
}
__device__ __forceinline__ void apply_signs(uint4& a, uint4& b, const SignWords& s) {
  a.x ^= s.w[0]; a.y ^= s.w[1]; a.z ^= s.w[2]; a.w ^= s.w[3];
  b.x ^= s.w[4]; b.y ^= s.w[5]; b.z ^= s.w[6]; b.w ^= s.w[7];
}

// ---------------------------------------------------------------------------
// Bulk asynchronous copies (TMA engine, cp.async.bulk) and mbarriers.
// Every wait is bounded: at most kWaitLimit polls, each suspending for at
// most kWaitSuspendNs, so a wait gives up after about two seconds and the
// caller reports an error instead of spinning on.
// ---------------------------------------------------------------------------
constexpr uint32_t kWaitLimit = 1u << 20;
constexpr uint32_t kWaitSuspendNs = 2000;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kWaitSuspendNs)
      : "memory");
  return ok != 0;
}
// Waits for the phase of `parity` to complete; false after kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (uint32_t i = 0; i < kWaitLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
// Global -> shared bulk copy completing `bytes` of transaction on `bar`.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 16-byte global load with an L2 eviction-priority policy.
__device__ __forceinline__ uint4 ld_hint(const void* p, uint64_t policy) {
  uint4 r;
  asm("ld.global.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
      : "l"(p), "l"(policy));
  return r;
}
// 2-D tiled tensor copy (TMA) of the box at element coordinates (x, y), x the
// innermost, into dst, completing its bytes on `bar`.  The map lives in
// kernel-parameter space (__grid_constant__).  x * element size must be a
// multiple of 16 bytes; parts of the box outside the tensor read as zero.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, int32_t x, int32_t y, uint64_t* bar,
                                           uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void prefetch_tensor_map(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
// Barrier `id` (1..15) over `threads` threads (a multiple of 32).
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

}  // namespace mp
