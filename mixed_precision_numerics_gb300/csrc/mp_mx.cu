// mp_mx.cu — MX block formats: one power-of-two scale per 32 elements.
//
// [MPT-ko] itwiki "혼합 정밀도 학습", "FP8 혼합 정밀도" (microscaling: a
// power-of-two scale for every 32 elements, MXFP8 / MXFP6 / MXFP4; FP6 codes
// are kept one per byte, as the hardware conversion produces them); [NVFP4]
// gist.science "Pretraining Large Language Models with NVFP4", §2.1 (MXFP4:
// 32-element blocks, UE8M0 scale byte).  The scale exponent follows the OCP
// microscaling rule, e = floor(log2 amax) - emax_elem, so the block maximum
// lands in the top binade of the element format.
//
// A 32-element block is 64 B of BF16/F16 (128 B of FP32) and one thread owns
// it end to end: the block amax, the scale byte and every code come from
// registers, with no shuffles.  Threads of a warp own consecutive blocks, so
// the warp reads one contiguous 2 KB (4 KB) span, writes one contiguous run of
// codes and a 32-byte run of scale bytes.  Two blocks (one for FP32) are in
// flight per thread: 128 B of loads.
#include "mp_chain.cuh"
#include "mp_device.cuh"
#include "mp_internal.h"

namespace mp {
namespace {

constexpr int kThreads = 256;
constexpr int kBlock = 32;

enum { XF32 = 0, XF16 = 1, XBF16 = 2 };
enum { EE4M3 = 0, EE5M2 = 1, EE2M1 = 2, EE2M3 = 3, EE3M2 = 4 };

template <int XT>
__host__ __device__ constexpr int words_of() { return XT == XF32 ? 8 : 4; }  // uint4 per block
template <int XT>
__host__ __device__ constexpr int unroll_of() { return XT == XF32 ? 1 : 2; }
template <int EF>
__host__ __device__ constexpr uint32_t emax_of() {
  return EF == EE4M3 ? 8u : EF == EE5M2 ? 15u : EF == EE3M2 ? 4u : 2u;  // E2M1 and E2M3: 2
}

// Element pair k (elements 2k, 2k+1) of a block held as raw 16-byte words.
template <int XT>
__device__ __forceinline__ float2 pair_at(const uint4* r, int k) {
  if constexpr (XT == XF32) {
    const uint4 q = r[k >> 1];
    return (k & 1) ? make_float2(__uint_as_float(q.z), __uint_as_float(q.w))
                   : make_float2(__uint_as_float(q.x), __uint_as_float(q.y));
  } else {
    const uint4 q = r[k >> 2];
    const uint32_t w = (k & 3) == 0 ? q.x : (k & 3) == 1 ? q.y : (k & 3) == 2 ? q.z : q.w;
    return XT == XBF16 ? make_float2(bf16lo(w), bf16hi(w)) : make_float2(f16lo(w), f16hi(w));
  }
}

// Exact value of an element code.  E5M2 is the upper byte of a binary16;
// E4M3 rebiases (sign applied separately); E2M1 reads its magnitude table;
// FP6 (sign at bit 5) is mantissa-with-hidden-bit times a power of two.
template <int EF>
__device__ __forceinline__ float code_value(uint32_t c) {
  if constexpr (EF == EE2M3 || EF == EE3M2) {
    constexpr uint32_t kM = EF == EE2M3 ? 3u : 2u;           // mantissa bits
    constexpr int kBias = EF == EE2M3 ? 1 : 3;
    const uint32_t e = (c & 0x1Fu) >> kM, m = c & ((1u << kM) - 1u);
    // subnormal: m * 2^(1 - bias - M); normal: (2^M + m) * 2^(e - bias - M)
    const float sig = (float)(e ? (m | (1u << kM)) : m);
    const int ex = (e ? (int)e : 1) - kBias - (int)kM;
    const float v = __fmul_rn(sig, __uint_as_float((uint32_t)(127 + ex) << 23));
    return (c & 0x20u) ? -v : v;
  } else if constexpr (EF == EE5M2) {
    return __half2float(__ushort_as_half((unsigned short)(c << 8)));
  } else if constexpr (EF == EE4M3) {
    const float v = e4m3_pos_to_f32(c & 0x7Fu);
    return (c & 0x80u) ? -v : v;
  } else {
    return e2m1_to_f32(c);
  }
}

// Saturating RNE code pair of two scaled finite values; FP8 and FP6 pairs
// occupy 16 bits (element 2k in the low byte), E2M1 pairs 8 bits (element 2k
// in the low nibble).
template <int EF>
__device__ __forceinline__ uint32_t encode_pair(float a, float b) {
  if constexpr (EF == EE2M1) {
    return cvt_e2m1x2(a, b);
  } else if constexpr (EF == EE2M3) {
    return cvt_e2m3x2(a, b);
  } else if constexpr (EF == EE3M2) {
    return cvt_e3m2x2(a, b);
  } else {
    // The block is finite and scaled so its maximum is below twice the
    // format's largest value: the conversion's satfinite mode takes anything
    // beyond that largest value to it, as a clamp would.
    return EF == EE5M2 ? cvt_e5m2x2(a, b) : cvt_e4m3x2(a, b);
  }
}

template <int XT, int EF>
__device__ __forceinline__ void mx_block(const uint4* raw, int64_t blk, uint8_t* __restrict__ codes,
                                         uint8_t* __restrict__ scales, uint16_t* __restrict__ dq) {
  float a = 0.0f;
#pragma unroll
  for (int k = 0; k < kBlock / 2; ++k) {
    const float2 f = pair_at<XT>(raw, k);
    a = max_abs_nan(a, f.x);
    a = max_abs_nan(a, f.y);
  }
  // a is NaN, +inf or a finite non-negative value.  Its biased exponent E
  // gives floor(log2 a) = E - 127 for a normal a; e = E - 127 - emax, and the
  // clamp at -127 covers zero and subnormal maxima (E = 0).  Scale byte:
  // e + 127 = max(E - emax, 0); 0xFF marks a non-finite block.
  const bool bad = !(a <= 3.402823466e38f);
  const uint32_t E = __float_as_uint(a) >> 23;
  constexpr uint32_t emax = emax_of<EF>();
  const uint32_t sb = bad ? 0xFFu : (E > emax ? E - emax : 0u);
  const float mul = __uint_as_float((254u - (bad ? 0u : sb)) << 23);  // 2^-e, a normal binary32
  uint32_t w[8];  // FP8 / FP6: 8 words of 4 one-byte codes; E2M1: 4 words of 8 codes
#pragma unroll
  for (int k = 0; k < kBlock / 2; ++k) {
    const float2 f = pair_at<XT>(raw, k);
    const uint32_t p = bad ? 0u : encode_pair<EF>(__fmul_rn(f.x, mul), __fmul_rn(f.y, mul));
    if constexpr (EF == EE2M1) {
      if ((k & 3) == 0) w[k >> 2] = 0u;
      w[k >> 2] += p << (8 * (k & 3));  // disjoint fields: + is |
    } else {
      if ((k & 1) == 0) w[k >> 1] = 0u;
      w[k >> 1] += p << (16 * (k & 1));
    }
  }
  if constexpr (EF == EE2M1) {
    st_cs(codes + blk * 16, make_uint4(w[0], w[1], w[2], w[3]));
  } else {
    st_cs(codes + blk * 32, make_uint4(w[0], w[1], w[2], w[3]));
    st_cs(codes + blk * 32 + 16, make_uint4(w[4], w[5], w[6], w[7]));
  }
  scales[blk] = (uint8_t)sb;
  if (dq == nullptr) return;
  // value(code) * 2^e is exact in binary32 (at most 4 significant bits, and
  // the smallest product, 2^-16 * 2^-127, is above the subnormal step).
  const float dsc = __uint_as_float(sb == 0u ? 0x00400000u : (sb << 23));
  uint32_t d[16];
#pragma unroll
  for (int k = 0; k < kBlock / 2; ++k) {
    float v0 = 0.0f, v1 = 0.0f;
    if (!bad) {
      if constexpr (EF == EE2M1) {
        const uint32_t byte = w[k >> 2] >> (8 * (k & 3));
        v0 = __fmul_rn(code_value<EF>(byte & 0xFu), dsc);
        v1 = __fmul_rn(code_value<EF>((byte >> 4) & 0xFu), dsc);
      } else {
        const uint32_t half = w[k >> 1] >> (16 * (k & 1));
        v0 = __fmul_rn(code_value<EF>(half & 0xFFu), dsc);
        v1 = __fmul_rn(code_value<EF>((half >> 8) & 0xFFu), dsc);
      }
    }
    d[k] = pack_bf16x2(v0, v1);
  }
  uint8_t* dp = reinterpret_cast<uint8_t*>(dq + blk * kBlock);
#pragma unroll
  for (int j = 0; j < 4; ++j) st_cs(dp + 16 * j, make_uint4(d[4 * j], d[4 * j + 1], d[4 * j + 2], d[4 * j + 3]));
}

// CTA c, iteration i owns blocks (i * gridDim.x + c) * kThreads * U + k * kThreads + t.
template <int XT, int EF>
__global__ __launch_bounds__(kThreads) void k_mx_quantize(const void* __restrict__ x, int64_t nblk,
                                                          uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                          uint16_t* __restrict__ dq) {
  chain_wait();  // the previous kernel in the stream has finished and its writes are visible
  chain_release();
  constexpr int U = unroll_of<XT>(), W = words_of<XT>();
  const uint4* xv = static_cast<const uint4*>(x);
  for (int64_t base = (int64_t)blockIdx.x * kThreads * U; base < nblk; base += (int64_t)gridDim.x * kThreads * U) {
    uint4 raw[U][W];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int64_t blk = base + k * kThreads + threadIdx.x;
      if (blk < nblk) {
#pragma unroll
        for (int j = 0; j < W; ++j) raw[k][j] = __ldcs(xv + blk * W + j);
      }
    }
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int64_t blk = base + k * kThreads + threadIdx.x;
      if (blk < nblk) mx_block<XT, EF>(raw[k], blk, codes, scales, dq);
    }
  }
}

template <int XT, int EF>
mp_status launch(const void* x, int64_t nblk, uint8_t* codes, uint8_t* scales, uint16_t* dq, cudaStream_t s) {
  constexpr int U = unroll_of<XT>();
  const int64_t ctas = (nblk + (int64_t)kThreads * U - 1) / ((int64_t)kThreads * U);
  launch_chained(k_mx_quantize<XT, EF>, dim3(full_grid(ctas)), dim3(kThreads), 0, s, x, nblk, codes, scales, dq);
  note_launches(1);
  return launch_status();
}

template <int XT>
mp_status launch_x(int32_t elem, const void* x, int64_t nblk, uint8_t* codes, uint8_t* scales, uint16_t* dq,
                   cudaStream_t s) {
  switch (elem) {
    case MP_E4M3: return launch<XT, EE4M3>(x, nblk, codes, scales, dq, s);
    case MP_E5M2: return launch<XT, EE5M2>(x, nblk, codes, scales, dq, s);
    case MP_E2M3: return launch<XT, EE2M3>(x, nblk, codes, scales, dq, s);
    case MP_E3M2: return launch<XT, EE3M2>(x, nblk, codes, scales, dq, s);
    default: return launch<XT, EE2M1>(x, nblk, codes, scales, dq, s);
  }
}

}  // namespace
}  // namespace mp

extern "C" MP_API mp_status mx_quantize(const void* x, mp_dtype x_dtype, int64_t rows, int64_t cols,
                                        mp_dtype elem_dtype, void* codes, uint8_t* scales, void* dequant_bf16,
                                        void* stream) {
  using namespace mp;
  if (rows < 0 || cols < 0) return MP_EINVAL;
  if (x_dtype != MP_F32 && x_dtype != MP_F16 && x_dtype != MP_BF16) return MP_EINVAL;
  if (elem_dtype != MP_E4M3 && elem_dtype != MP_E5M2 && elem_dtype != MP_E2M1 && elem_dtype != MP_E2M3 &&
      elem_dtype != MP_E3M2)
    return MP_EINVAL;
  const int64_t n = rows * cols;
  if (n > 0 && (!x || !codes || !scales)) return MP_EINVAL;
  if (cols % kBlock != 0) return MP_ESHAPE;
  if (n > 0 && (!aligned16(x) || !aligned16(codes) || (dequant_bf16 && !aligned16(dequant_bf16)))) return MP_EALIGN;
  if (n == 0) return MP_OK;
  const int64_t nblk = n / kBlock;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* cb = static_cast<uint8_t*>(codes);
  uint16_t* dq = static_cast<uint16_t*>(dequant_bf16);
  switch (x_dtype) {
    case MP_F32: return launch_x<XF32>(elem_dtype, x, nblk, cb, scales, dq, s);
    case MP_F16: return launch_x<XF16>(elem_dtype, x, nblk, cb, scales, dq, s);
    default: return launch_x<XBF16>(elem_dtype, x, nblk, cb, scales, dq, s);
  }
}
