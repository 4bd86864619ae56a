// mp_nvfp4.cu — NVFP4 quantisation and the 16-point random Hadamard transform.
//
// [NVFP4] gist.science "Pretraining Large Language Models with NVFP4":
//   §2.1 "NVFP4 포맷의 특징": 16-element blocks, E4M3 block scale, FP32 tensor
//        scale (two-level scaling), FP4 (E2M1) elements;
//   §2.2 item 2: 16x16 random Hadamard transform of weight-gradient inputs;
//   §2.2 item 3: 16x16 2D block scaling for weights, 1x16 for the rest;
//   §2.2 item 4: stochastic rounding for gradients.
//
// Two passes, because the tensor scale needs the amax of the whole tensor
// before any element can be encoded:
//   k_nvfp4_amax    reads x (2 B/elem), applies the transform when asked,
//                   folds max |x'| with one atomicMax per CTA; the last CTA
//                   (ticket, no waiting) writes s_t = amax / 2688.
//   k_nvfp4_1x16 /  read x again, recompute x', form block scales, encode,
//   k_nvfp4_2d      pack two codes per byte (0.5 B/elem) and one scale byte
//                   per block.
// For 1x16 the amax pass loads the last half-L2's worth of x with the L2
// evict-last policy and the encode pass walks x from the end, so that part
// of the second read is served by L2; a 16x16 input that fits in half the L2
// is kept whole.  The 16x16 encode gives each warp a 16-row strip (a block is
// a lane pair), with no CTA barrier.  The transform is evaluated on CUDA
// cores by the butterfly in binary32, three of its stages as packed FP32x2
// operations, so that its additions happen in the documented order.  Both
// passes are chained launches (mp_chain.cuh).
#include <mutex>

#include "mp_chain.cuh"
#include "mp_device.cuh"
#include "mp_internal.h"

namespace mp {
namespace {

constexpr int kThreads = 256;
constexpr float kTensorDiv = 2688.0f;  // 6 (largest E2M1) * 448 (largest E4M3)

struct Ws {
  uint32_t amax_bits;
  uint32_t ticket;
};

// The 16-point Walsh-Hadamard butterfly, v <- H16 v with H16[i][j] =
// (-1)^popcount(i & j): stages of distance h = 1, 2, 4, 8, each replacing
// (v[i], v[i + h]) for i with bit h clear by (a + b, a - b), every operation a
// binary32 add rounded to nearest even.  Here in packed arithmetic: the tile
// is held as eight pairs p[i] = (v[i], v[i + 8]); the stages of distance 1, 2
// and 4 pair element i with i + h in both halves at once, so one packed add
// gives both sums and one packed fma(b, -1, a) both differences (the product
// by -1 is exact, so the fma rounds a - b once, as the subtraction does); the
// stage of distance 8 works inside each pair.
__device__ __forceinline__ void fwht16_first3(float2 (&p)[8]) {
  const float2 m1 = make_float2(-1.0f, -1.0f);
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i & h) continue;
      const float2 a = p[i], b = p[i + h];
      p[i] = __fadd2_rn(a, b);
      p[i + h] = __ffma2_rn(b, m1, a);
    }
  }
}
__device__ __forceinline__ void fwht16_last(float2 (&p)[8]) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float a = p[i].x, b = p[i].y;
    p[i] = make_float2(__fadd_rn(a, b), __fsub_rn(a, b));
  }
}
__device__ __forceinline__ void fwht16_packed(float2 (&p)[8]) {
  fwht16_first3(p);
  fwht16_last(p);
}

// x' of one 16-element BF16 tile (two 16-byte words) as the pairs
// (x'[i], x'[i + 8]); `quarter` applies the transform's 1/4 (the amax pass
// applies it once to the maximum instead).
template <bool RHT, bool QUARTER = true>
__device__ __forceinline__ void tile_pairs(uint4 a, uint4 b, const SignWords& sw, float2 (&p)[8]) {
  if (RHT) apply_signs(a, b, sw);
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float lo = (i & 1) ? bf16hi(w[i >> 1]) : bf16lo(w[i >> 1]);
    const float hi = (i & 1) ? bf16hi(w[4 + (i >> 1)]) : bf16lo(w[4 + (i >> 1)]);
    p[i] = make_float2(lo, hi);
  }
  if (RHT) {
    fwht16_packed(p);
    if (QUARTER) {
#pragma unroll
      for (int i = 0; i < 8; ++i) p[i] = __fmul2_rn(p[i], make_float2(0.25f, 0.25f));
    }
  }
}

template <bool RHT>
__global__ __launch_bounds__(kThreads) void k_nvfp4_amax(const uint16_t* __restrict__ x, int64_t ntiles,
                                                         uint32_t mask, Ws* ws, float* tensor_scale,
                                                         int32_t* nonfinite, int64_t keep_from) {
  chain_wait();  // the previous kernel in the stream has finished and its writes are visible
  chain_release();
  __shared__ uint32_t red[32];
  __shared__ int is_last;
  const SignWords sw = sign_words(mask);
  float acc = 0.0f;
  uint32_t pm = 0u;            // without the transform: max |x| of BF16 pairs, packed
  constexpr int U = RHT ? 2 : 4;  // 32-byte tiles in flight per thread
  const uint64_t keep = policy_evict_last();
  const int64_t step = (int64_t)gridDim.x * kThreads * U;
  for (int64_t t0 = (int64_t)blockIdx.x * kThreads * U + threadIdx.x; t0 < ntiles; t0 += step) {
    uint4 a[U], b[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t t = t0 + (int64_t)u * kThreads;
      if (t < ntiles) {
        if (t >= keep_from) {
          a[u] = ld_hint(x + t * 16, keep);
          b[u] = ld_hint(x + t * 16 + 8, keep);
        } else {
          a[u] = ld_plain(x + t * 16);
          b[u] = ld_plain(x + t * 16 + 8);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t t = t0 + (int64_t)u * kThreads;
      if (t >= ntiles) continue;
      if (RHT) {
        // The last butterfly stage maps each pair (a, b) to a + b and a - b,
        // the larger magnitude being RN(|a| + |b|); so the first three stages
        // and one add per pair give the tile's max |v| (the 1/4 is applied
        // once to the maximum below).  Only infinite a and b together make a
        // NaN output where that sum is infinite: such a tile takes the last
        // stage in full.
        float2 p[8];
        apply_signs(a[u], b[u], sw);
        const uint32_t w[8] = {a[u].x, a[u].y, a[u].z, a[u].w, b[u].x, b[u].y, b[u].z, b[u].w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float lo = (i & 1) ? bf16hi(w[i >> 1]) : bf16lo(w[i >> 1]);
          const float hi = (i & 1) ? bf16hi(w[4 + (i >> 1)]) : bf16lo(w[4 + (i >> 1)]);
          p[i] = make_float2(lo, hi);
        }
        fwht16_first3(p);
        float m = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) m = max_abs_nan(m, __fadd_rn(fabsf(p[j].x), fabsf(p[j].y)));
        if (__builtin_expect(isinf(m), 0)) {
          fwht16_last(p);
#pragma unroll
          for (int j = 0; j < 8; ++j) m = max_abs_nan(max_abs_nan(m, p[j].x), p[j].y);
        }
        acc = max_abs_nan(acc, m);
      } else {
        const uint32_t w[8] = {a[u].x, a[u].y, a[u].z, a[u].w, b[u].x, b[u].y, b[u].z, b[u].w};
#pragma unroll
        for (int k = 0; k < 8; ++k) pm = max_abs_nan_x2<true>(pm, w[k]);
      }
    }
  }
  if (!RHT) acc = max_abs_nan(max_abs_nan(acc, bf16lo(pm)), bf16hi(pm));
  const uint32_t cta = block_max_u32(amax_bits(acc), red);
  if (threadIdx.x == 0) {
    atomicMax(&ws->amax_bits, cta);
    __threadfence();
    is_last = atomicAdd(&ws->ticket, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!is_last || threadIdx.x != 0) return;
  __threadfence();
  const uint32_t ab = atomicExch(&ws->amax_bits, 0u);
  ws->ticket = 0;
  // Rounding is monotonic, so max(round(|v| / 4)) == round(max|v| / 4).
  float amax = __uint_as_float(ab);
  if (RHT) amax = __fmul_rn(amax, 0.25f);
  if (amax != amax) {
    *tensor_scale = __uint_as_float(0x7FC00000u);
    *nonfinite = 1;
  } else if (isinf(amax)) {
    *tensor_scale = amax;
    *nonfinite = 1;
  } else {
    *tensor_scale = __fdiv_rn(amax, kTensorDiv);
    *nonfinite = 0;
  }
}

struct BlockScale {
  uint32_t code;
  float d, r;
};

// sb = E4M3(RNE((bamax / 6) / s_t)) saturating; d = value(sb) * s_t; r = 1/d.
__device__ __forceinline__ BlockScale block_scale(float bamax, float s_t) {
  BlockScale bs;
  const float q = fminf(__fdiv_rn(__fdiv_rn(bamax, 6.0f), s_t), 448.0f);
  bs.code = cvt_e4m3x2(q, 0.0f) & 0xFFu;
  bs.d = __fmul_rn(e4m3_pos_to_f32(bs.code), s_t);
  bs.r = 0.0f;
  if (bs.d != 0.0f) {
    const float inv = __fdiv_rn(1.0f, bs.d);
    if (isfinite(inv)) bs.r = inv;
  }
  return bs;
}

// prmt.b32: result byte i is byte (sel nibble i & 7) of {b, a}; a nibble with
// bit 3 set gives that byte's top bit copied into all eight bits.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Stochastic E2M1 codes of two values in one hardware conversion.
// cvt.rs.satfinite.e2m1x4.f32 d, {a, b, c, e}, rbits puts the codes of a, b,
// c, e in nibbles 3, 2, 1, 0 of d and rounds each magnitude away from zero
// iff floor(frac * 2^16) + r16 >= 2^16, frac its position between its grid
// neighbours; magnitudes from 6 up give code 7; the sign is kept (-0 gives
// 0x8).  b takes r16 = (rbits byte 3 << 8) | byte 1 and e takes
// (byte 2 << 8) | byte 0; a and c take those same 16 bits in reverse bit
// order, so they would not be independent of b and e and carry zeros here
// (code 0 whatever the bits).  This rounding and lane layout were checked
// against that rule over every value k * 2^-10 in (-7, 7), the values one
// ulp either side of each 1/256 of every grid gap, with every byte pattern,
// and 10^6 random values and bit patterns: identical for every finite or
// infinite input.  (A NaN converts to +6, not the rule's 6 with the NaN's
// sign; no NaN reaches the encode, whose tensors are finite or all zero.)
// lo gets nibble 0 and r16 = (byte 2 << 8) | byte 0; hi gets nibble 2 and
// r16 = (byte 3 << 8) | byte 1.
__device__ __forceinline__ uint32_t cvt_rs_e2m1_pair(float lo, float hi, uint32_t rbits) {
  unsigned short d;
  asm("cvt.rs.satfinite.e2m1x4.f32 %0, {%1, %2, %3, %4}, %5;"
      : "=h"(d)
      : "f"(0.0f), "f"(hi), "f"(0.0f), "f"(lo), "r"(rbits));
  return d;
}

// Stochastic E2M1 codes of 8 values y[j] and the four 32-bit words w0..w3 of
// one Philox call (element j takes 16-bit half j mod 2 of word j / 2);
// element j goes to nibble j.  Elements j and j + 2 share a conversion: a byte
// permute of two Philox words lines up their 16-bit halves with the
// conversion's random-bit bytes, and the results, codes at nibbles 0 and 2,
// interleave with a shift and an add.
__device__ __forceinline__ uint32_t sr_group(const float (&y)[8], u32x4 R) {
  const uint32_t c02 = cvt_rs_e2m1_pair(y[0], y[2], prmt(R.x, R.y, 0x5140u));  // low halves of w0, w1
  const uint32_t c13 = cvt_rs_e2m1_pair(y[1], y[3], prmt(R.x, R.y, 0x7362u));  // high halves of w0, w1
  const uint32_t c46 = cvt_rs_e2m1_pair(y[4], y[6], prmt(R.z, R.w, 0x5140u));
  const uint32_t c57 = cvt_rs_e2m1_pair(y[5], y[7], prmt(R.z, R.w, 0x7362u));
  return (c02 + (c13 << 4)) | ((c46 + (c57 << 4)) << 16);
}

// BF16 RNE of value(code) * d for the 16 codes in (lo, hi).
__device__ __forceinline__ void dequant16(uint2 q, float d, uint16_t* out) {
  uint32_t w[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const uint32_t byte = ((k < 4 ? q.x : q.y) >> (8 * (k & 3))) & 0xFFu;
    w[k] = pack_bf16x2(__fmul_rn(e2m1_to_f32(byte & 0xFu), d), __fmul_rn(e2m1_to_f32(byte >> 4), d));
  }
  st_cs(out, make_uint4(w[0], w[1], w[2], w[3]));
  st_cs(out + 8, make_uint4(w[4], w[5], w[6], w[7]));
}

// Per-CTA table, one entry per E4M3 block-scale code c: d = value(c) * s_t and
// the multiplier that turns the tile's values into y = x' * r, r = 1/d (0 when
// d is 0 or 1/d is not finite).  With the transform the multiplier applies to
// the butterfly's output before its 1/4, so it is r/4: an exact scaling while
// 2^-90 <= s_t <= 2^110 (r between 2^-119 and 2^99), and the product equals
// the oracle's two-step one except for elements below 2^-124, whose codes are
// zero either way (|y| < 2^-27, below any rounding step or random carry).
template <bool RHT>
__device__ __forceinline__ void fill_scale_table(float2* tab, float s_t) {
  for (int c = threadIdx.x; c < 128; c += kThreads) {
    const float d = __fmul_rn(e4m3_pos_to_f32((uint32_t)c), s_t);
    float r = 0.0f;
    if (d != 0.0f) {
      const float inv = __fdiv_rn(1.0f, d);
      if (isfinite(inv)) r = inv;
    }
    if (RHT) r = __fmul_rn(r, 0.25f);
    tab[c] = make_float2(d, r);
  }
}

// Tile of 16 BF16 values (two 16-byte words) as the pairs (x[i], x[i + 8]),
// with the random signs of the transform applied: the low half of a word
// becomes w * 2^16 plus the sign (adding 2^31 flips the top bit), the high
// half (w ^ sign word) with the low half cleared.
template <bool RHT>
__device__ __forceinline__ void unpack_tile(uint4 a, uint4 b, const SignWords& sw, const uint32_t (&slo)[8],
                                            float2 (&p)[8]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float v[16];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    v[2 * k] = __uint_as_float(RHT ? w[k] * 65536u + slo[k] : w[k] << 16);
    v[2 * k + 1] = __uint_as_float((RHT ? (w[k] ^ sw.w[k]) : w[k]) & 0xFFFF0000u);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) p[i] = make_float2(v[i], v[i + 8]);
}

// One 16-element block per thread per step.  Block scale: q~ = bamax * K with
// K = RN(RN(1/6) * RN(1/s_t)) lies within 6.01 units of 2^-24 (relative) of
// q = RN(RN(bamax / 6) / s_t) when everything is normal, so if the E4M3
// conversions of q~ * (1 - 2^-21) and q~ * (1 + 2^-21) agree, that code is
// the code of q (conversion is monotonic); tiny or non-normal cases, and the
// rare disagreement, take the exact divisions.  The code then indexes the
// per-CTA table for d and the multiplier.
template <bool RHT, bool SR, bool DEQ>
__global__ __launch_bounds__(kThreads) void k_nvfp4_1x16(const uint16_t* __restrict__ x, int64_t nblocks,
                                                         uint32_t mask, uint64_t seed,
                                                         const float* __restrict__ tensor_scale,
                                                         const int32_t* __restrict__ nonfinite,
                                                         uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                         uint16_t* __restrict__ deq) {
  __shared__ float2 tab[128];
  chain_wait();  // the previous kernel in the stream has finished and its writes are visible
  chain_release();
  const float s_t = *tensor_scale;
  const bool zero = (*nonfinite != 0) || s_t == 0.0f;
  fill_scale_table<RHT>(tab, s_t);
  __syncthreads();
  const bool fast = s_t >= 0x1p-90f && s_t <= 0x1p110f;
  const float K = __fmul_rn(__fdiv_rn(1.0f, 6.0f), __fdiv_rn(1.0f, s_t));
  const SignWords sw = sign_words(mask);
  uint32_t slo[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) slo[k] = sw.w[k] << 16;
  const uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  const uint64_t last_use = policy_evict_first();  // this pass is the last reader of x
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < nblocks; i += stride) {
    // Last block first: the amax pass marked the tail of x to stay in L2.
    const int64_t blk = nblocks - 1 - i;
    if (zero) {
      *reinterpret_cast<uint2*>(codes + blk * 8) = make_uint2(0u, 0u);
      scales[blk] = 0;
      if (DEQ) {
        st_cs(deq + blk * 16, make_uint4(0u, 0u, 0u, 0u));
        st_cs(deq + blk * 16 + 8, make_uint4(0u, 0u, 0u, 0u));
      }
      continue;
    }
    const uint4 ca = ld_hint(x + blk * 16, last_use), cb = ld_hint(x + blk * 16 + 8, last_use);
    float2 p[8];
    unpack_tile<RHT>(ca, cb, sw, slo, p);
    float bamax;
    if (RHT) {
      // The last butterfly stage turns each pair (a, b) into a + b and a - b,
      // the larger in magnitude being RN(|a| + |b|) (rounding is monotonic and
      // symmetric), so the block's max |v| is the max of those eight sums; and
      // max |x'| = RN(max |v| / 4).
      fwht16_first3(p);
      float m[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) m[j] = __fadd_rn(fabsf(p[j].x), fabsf(p[j].y));
      fwht16_last(p);
      bamax = __fmul_rn(fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])), fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7]))),
                        0.25f);
    } else {
      // max |x| on the packed BF16 words (exact)
      const uint32_t w[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
      uint32_t m = 0u;
#pragma unroll
      for (int k = 0; k < 8; ++k) m = max_abs_nan_x2<true>(m, w[k]);
      bamax = fmaxf(bf16lo(m), bf16hi(m));
    }
    uint32_t code = 0;
    bool ok = fast && (bamax >= 0x1p-120f || bamax == 0.0f);
    if (ok) {
      const float qt = __fmul_rn(bamax, K);
      const uint32_t c2 = cvt_e4m3x2(__fmul_rn(qt, 1.0f - 0x1p-21f), __fmul_rn(qt, 1.0f + 0x1p-21f));
      code = c2 & 0xFFu;
      ok = code == (c2 >> 8);
    }
    float d;
    float2 y[8];
    if (ok) {
      const float2 e = tab[code];
      d = e.x;
#pragma unroll
      for (int j = 0; j < 8; ++j) y[j] = __fmul2_rn(p[j], make_float2(e.y, e.y));
    } else {
      const BlockScale bs = block_scale(bamax, s_t);
      code = bs.code;
      d = bs.d;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float2 xq = RHT ? __fmul2_rn(p[j], make_float2(0.25f, 0.25f)) : p[j];
        y[j] = __fmul2_rn(xq, make_float2(bs.r, bs.r));
      }
    }
    uint2 q;
    if (SR) {
      const uint64_t g = (uint64_t)blk * 2;  // counter of elements 16 blk .. 16 blk + 7
      const u32x4 R0 = philox4x32_10((uint32_t)g, (uint32_t)(g >> 32), 0u, 0u, k0, k1);
      const u32x4 R1 = philox4x32_10((uint32_t)(g + 1), (uint32_t)((g + 1) >> 32), 0u, 0u, k0, k1);
      float g0[8], g1[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        g0[j] = y[j].x;
        g1[j] = y[j].y;
      }
      q = make_uint2(sr_group(g0, R0), sr_group(g1, R1));
    } else {
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        lo |= cvt_e2m1x2(y[2 * k].x, y[2 * k + 1].x) << (8 * k);
        hi |= cvt_e2m1x2(y[2 * k].y, y[2 * k + 1].y) << (8 * k);
      }
      q = make_uint2(lo, hi);
    }
    __stcs(reinterpret_cast<uint2*>(codes + blk * 8), q);
    scales[blk] = (uint8_t)code;
    if (DEQ) dequant16(q, d, deq + blk * 16);
  }
}

// Encode 8 values of x' (half a 1x16 tile, flat index `flat` a multiple of 8)
// with block reciprocal r; returns 8 codes, element j in nibble j.  Stochastic
// rounding takes the 8 random halves of the one Philox call for counter
// flat / 8, as the 1x16 encode does for each half of its tile.
template <bool SR>
__device__ __forceinline__ uint32_t encode8(const float (&v)[8], float r, uint64_t flat, uint32_t k0, uint32_t k1) {
  uint32_t q = 0;
  if (SR) {
    const uint64_t g = flat >> 3;
    const u32x4 R = philox4x32_10((uint32_t)g, (uint32_t)(g >> 32), 0u, 0u, k0, k1);
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) y[j] = __fmul_rn(v[j], r);
    q = sr_group(y, R);
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) q |= cvt_e2m1x2(__fmul_rn(v[2 * k], r), __fmul_rn(v[2 * k + 1], r)) << (8 * k);
  }
  return q;
}

// The 16-point transform of a tile split over a lane pair: the even lane
// holds elements 0-7, the odd lane 8-15.  The stages of distance 1, 2 and 4
// stay within a lane; the stage of distance 8 pairs element i of the even
// lane (a) with element i of the odd lane (b): a + b on the even lane, a - b
// on the odd one -- the butterfly's additions, in its order.  Then the 1/4.
__device__ __forceinline__ void fwht16_pair(float (&v)[8], bool odd) {
#pragma unroll
  for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i & h) continue;
      const float a = v[i], b = v[i + h];
      v[i] = __fadd_rn(a, b);
      v[i + h] = __fsub_rn(a, b);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float o = __shfl_xor_sync(0xFFFFFFFFu, v[i], 1);
    v[i] = odd ? __fsub_rn(o, v[i]) : __fadd_rn(v[i], o);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], 0.25f);
}

// x' of a lane's 8 elements (one 16-byte word of BF16).  With the transform
// every lane of the warp must take part (the pair exchanges values).
template <bool RHT>
__device__ __forceinline__ void half_tile_values(uint4 w, uint32_t s0, uint32_t s1, uint32_t s2, uint32_t s3,
                                                 bool odd, float (&v)[8]) {
  if (RHT) {
    w.x ^= s0;
    w.y ^= s1;
    w.z ^= s2;
    w.w ^= s3;
  }
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[2 * k] = bf16lo(ws[k]);
    v[2 * k + 1] = bf16hi(ws[k]);
  }
  if (RHT) fwht16_pair(v, odd);
}

// 16x16 blocks: a warp takes a strip of 16 rows x 256 columns (16 blocks) at a
// time; lane l holds columns 8l .. 8l + 7 of all 16 rows (sixteen 16-byte
// loads in flight, each row read as 512 consecutive bytes by the warp), so a
// block is the lane pair (2b, 2b + 1) and its amax takes one shuffle; no CTA
// barrier.  Each row's 8 codes go out as one 4-byte store (128 bytes per row
// per warp).  Without the transform the block amax comes from the packed BF16
// words; with it the values are transformed once for the amax and again for
// the encode, keeping only the raw words in registers.
template <bool RHT, bool SR, bool DEQ>
__global__ __launch_bounds__(kThreads) void k_nvfp4_2d(const uint16_t* __restrict__ x, int64_t rows, int64_t cols,
                                                       uint32_t mask, uint64_t seed,
                                                       const float* __restrict__ tensor_scale,
                                                       const int32_t* __restrict__ nonfinite,
                                                       uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
                                                       uint16_t* __restrict__ deq) {
  chain_wait();  // the previous kernel in the stream has finished and its writes are visible
  chain_release();
  const float s_t = *tensor_scale;
  const bool zero = (*nonfinite != 0) || s_t == 0.0f;
  const SignWords sw = sign_words(mask);
  const uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
  const int lane = threadIdx.x & 31;
  const bool odd = lane & 1;
  const uint64_t last_use = policy_evict_first();  // this pass is the last reader of x
  const uint32_t s0 = odd ? sw.w[4] : sw.w[0], s1 = odd ? sw.w[5] : sw.w[1];
  const uint32_t s2 = odd ? sw.w[6] : sw.w[2], s3 = odd ? sw.w[7] : sw.w[3];
  const int64_t ncc = (cols + 255) / 256;
  const int64_t nitems = (rows / 16) * ncc;
  const int64_t nb = cols / 16;
  const int64_t warps = (int64_t)gridDim.x * (kThreads / 32);
  for (int64_t item = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); item < nitems; item += warps) {
    const int64_t tr = item / ncc, cc = item % ncc;
    const int64_t col = cc * 256 + lane * 8;
    const bool active = col < cols;  // cols % 16 == 0: both lanes of a pair agree
    const int64_t base = tr * 16 * cols + col;
    if (zero) {
      if (!active) continue;
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        *reinterpret_cast<uint32_t*>(codes + (base + r * cols) / 2) = 0u;
        if (DEQ) st_cs(deq + base + r * cols, make_uint4(0u, 0u, 0u, 0u));
      }
      if (!odd) scales[tr * nb + col / 16] = 0;
      continue;
    }
    uint4 raw[16];
#pragma unroll
    for (int r = 0; r < 16; ++r)
      raw[r] = active ? ld_hint(x + base + r * cols, last_use) : make_uint4(0u, 0u, 0u, 0u);
    float m;
    if (!RHT) {
      uint32_t acc[4] = {0u, 0u, 0u, 0u};
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        acc[0] = max_abs_nan_x2<true>(acc[0], raw[r].x);
        acc[1] = max_abs_nan_x2<true>(acc[1], raw[r].y);
        acc[2] = max_abs_nan_x2<true>(acc[2], raw[r].z);
        acc[3] = max_abs_nan_x2<true>(acc[3], raw[r].w);
      }
      const uint32_t p = max_abs_nan_x2<true>(max_abs_nan_x2<true>(acc[0], acc[1]), max_abs_nan_x2<true>(acc[2], acc[3]));
      m = fmaxf(bf16lo(p), bf16hi(p));
    } else {
      m = 0.0f;
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float v[8];
        half_tile_values<true>(raw[r], s0, s1, s2, s3, odd, v);
#pragma unroll
        for (int j = 0; j < 8; ++j) m = fmaxf(m, fabsf(v[j]));
      }
    }
    const float bamax = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    const BlockScale bs = block_scale(bamax, s_t);
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float v[8];
      half_tile_values<RHT>(raw[r], s0, s1, s2, s3, odd, v);
      if (!active) continue;
      const uint64_t flat = (uint64_t)(base + r * cols);
      const uint32_t q = encode8<SR>(v, bs.r, flat, k0, k1);
      __stcs(reinterpret_cast<uint32_t*>(codes + flat / 2), q);
      if (DEQ) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t byte = (q >> (8 * k)) & 0xFFu;
          w[k] = pack_bf16x2(__fmul_rn(e2m1_to_f32(byte & 0xFu), bs.d), __fmul_rn(e2m1_to_f32(byte >> 4), bs.d));
        }
        st_cs(deq + flat, make_uint4(w[0], w[1], w[2], w[3]));
      }
    }
    if (active && !odd) scales[tr * nb + col / 16] = (uint8_t)bs.code;
  }
}

// Stochastic E2M1 codes of y with caller-supplied random bits (element i
// takes r16[i]), two elements a thread through the same conversion as the
// encode; codes two per byte, element 2j in the low nibble.  A NaN takes code
// 7 with its sign bit, as the rule's comparison (|NaN| < 6 is false) gives,
// where the conversion alone would give +6.
__global__ __launch_bounds__(kThreads) void k_e2m1_sr(const float* __restrict__ y, const uint16_t* __restrict__ r16,
                                                      int64_t n, uint8_t* __restrict__ codes) {
  chain_wait();  // the previous kernel in the stream has finished and its writes are visible
  chain_release();
  const int64_t npairs = (n + 1) / 2, stride = (int64_t)gridDim.x * kThreads;
  for (int64_t j = (int64_t)blockIdx.x * kThreads + threadIdx.x; j < npairs; j += stride) {
    const int64_t i = 2 * j;
    const float lo = y[i];
    const uint32_t rlo = r16[i];
    float hi = 0.0f;
    uint32_t rhi = 0u;
    if (i + 1 < n) {
      hi = y[i + 1];
      rhi = r16[i + 1];
    }
    // rbits bytes 2:0 = rlo (lane e, lo), bytes 3:1 = rhi (lane b, hi)
    const uint32_t d = cvt_rs_e2m1_pair(lo, hi, prmt(rlo | (rhi << 16), 0u, 0x3120u));
    uint32_t q = (d | (d >> 4)) & 0xFFu;
    if (lo != lo) q = (q & 0xF0u) | 7u | ((__float_as_uint(lo) >> 28) & 8u);
    if (hi != hi) q = (q & 0x0Fu) | 0x70u | ((__float_as_uint(hi) >> 24) & 0x80u);
    codes[j] = (uint8_t)q;
  }
}

template <bool F32OUT>
__global__ __launch_bounds__(kThreads) void k_rht16(const uint16_t* __restrict__ x, int64_t ntiles, uint32_t mask,
                                                    void* __restrict__ y) {
  chain_wait();  // the previous kernel in the stream has finished and its writes are visible
  chain_release();
  const SignWords sw = sign_words(mask);
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t t = (int64_t)blockIdx.x * kThreads + threadIdx.x; t < ntiles; t += stride) {
    float2 p[8];  // (x'[i], x'[i + 8])
    tile_pairs<true>(ld_plain(x + t * 16), ld_plain(x + t * 16 + 8), sw, p);
    if (F32OUT) {
      float* o = static_cast<float*>(y) + t * 16;
      st_cs_f4(o, make_float4(p[0].x, p[1].x, p[2].x, p[3].x));
      st_cs_f4(o + 4, make_float4(p[4].x, p[5].x, p[6].x, p[7].x));
      st_cs_f4(o + 8, make_float4(p[0].y, p[1].y, p[2].y, p[3].y));
      st_cs_f4(o + 12, make_float4(p[4].y, p[5].y, p[6].y, p[7].y));
    } else {
      uint16_t* o = static_cast<uint16_t*>(y) + t * 16;
      st_cs(o, make_uint4(pack_bf16x2(p[0].x, p[1].x), pack_bf16x2(p[2].x, p[3].x), pack_bf16x2(p[4].x, p[5].x),
                          pack_bf16x2(p[6].x, p[7].x)));
      st_cs(o + 8, make_uint4(pack_bf16x2(p[0].y, p[1].y), pack_bf16x2(p[2].y, p[3].y),
                              pack_bf16x2(p[4].y, p[5].y), pack_bf16x2(p[6].y, p[7].y)));
    }
  }
}

template <typename K>
int occ_of(K kernel) {
  int o = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, kThreads, 0) != cudaSuccess || o < 1) o = 1;
  return o;
}

template <bool RHT>
void launch_amax(const uint16_t* x, int64_t ntiles, uint32_t mask, Ws* ws, float* ts, int32_t* nf, int64_t keep_from,
                 cudaStream_t s) {
  static const int occ = occ_of(k_nvfp4_amax<RHT>);
  const int64_t ctas = (ntiles + 2 * kThreads - 1) / (2 * kThreads);
  launch_chained(k_nvfp4_amax<RHT>, dim3(grid_for(ctas, occ)), dim3(kThreads), 0, s, x, ntiles, mask, ws, ts, nf,
                 keep_from);
}

// First tile (32 B each) that the amax pass loads with the L2 evict-last
// policy, so that the encode pass (which reads with evict-first, releasing the
// lines) finds it in L2.  1x16: the last half-L2's worth of x, which the
// encode pass reads first.  16x16: the whole tensor when it fits in half the
// L2 (a weight matrix usually does), else nothing, since that pass reads x in
// the same order as the amax pass.  The L2 size is read once per process.
int64_t keep_from_of(int64_t ntiles, bool block_2d) {
  static const int64_t l2 = [] {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
      v = 0;
    return (int64_t)v;
  }();
  const int64_t keep = l2 / 2 / 32;
  if (block_2d) return ntiles <= keep ? 0 : ntiles;
  return ntiles > keep ? ntiles - keep : 0;
}

template <bool RHT, bool SR, bool DEQ>
void launch_encode(bool block_2d, const uint16_t* x, int64_t rows, int64_t cols, uint32_t mask, uint64_t seed,
                   const float* ts, const int32_t* nf, uint8_t* codes, uint8_t* scales, uint16_t* deq,
                   cudaStream_t s) {
  if (block_2d) {
    static const int occ = occ_of(k_nvfp4_2d<RHT, SR, DEQ>);
    const int64_t items = (rows / 16) * ((cols + 255) / 256);  // one warp each
    const int64_t ctas = (items + kThreads / 32 - 1) / (kThreads / 32);
    // twice as many CTAs as fit at once (measured faster than 1x and 4x)
    launch_chained(k_nvfp4_2d<RHT, SR, DEQ>, dim3(grid_for(ctas, occ * 2)), dim3(kThreads), 0, s, x, rows, cols, mask, seed,
                   ts, nf, codes, scales, deq);
  } else {
    // Four times as many CTAs as fit at once: a CTA that finishes early takes
    // another, so the last wave ends nearly together (measured: 4x beat 1x, 2x,
    // 8x and 16x; a CTA's table costs 128 divisions, so not more).
    static const int occ = occ_of(k_nvfp4_1x16<RHT, SR, DEQ>);
    const int64_t nblocks = rows * (cols / 16);
    const int64_t ctas = (nblocks + kThreads - 1) / kThreads;
    launch_chained(k_nvfp4_1x16<RHT, SR, DEQ>, dim3(grid_for(ctas, occ * 4)), dim3(kThreads), 0, s, x, nblocks, mask,
                   seed, ts, nf, codes, scales, deq);
  }
}

template <bool RHT, bool SR>
void dispatch_deq(bool deq, bool block_2d, const uint16_t* x, int64_t rows, int64_t cols, uint32_t mask,
                  uint64_t seed, const float* ts, const int32_t* nf, uint8_t* codes, uint8_t* scales,
                  uint16_t* dq, cudaStream_t s) {
  if (deq) launch_encode<RHT, SR, true>(block_2d, x, rows, cols, mask, seed, ts, nf, codes, scales, dq, s);
  else launch_encode<RHT, SR, false>(block_2d, x, rows, cols, mask, seed, ts, nf, codes, scales, dq, s);
}

}  // namespace
}  // namespace mp

namespace mp {
namespace {

constexpr size_t kNvfp4WorkspaceBytes = 256;

// The argument checks of both quantiser entry points, run before a call
// enqueues anything.  need_ws: the caller passes a workspace to be checked
// (nvfp4_quantize); the no-alloc entry point has its own scratch.
mp_status nvfp4_check_args(const void* x_bf16, int64_t rows, int64_t cols, int32_t block_2d, const uint8_t* codes,
                           const uint8_t* block_scales, const float* d_tensor_scale, const int32_t* d_nonfinite,
                           const void* dequant_bf16, bool need_ws, const void* d_workspace, size_t workspace_bytes) {
  if (rows < 0 || cols < 0 || !d_tensor_scale || !d_nonfinite) return MP_EINVAL;
  const int64_t n = rows * cols;
  if (n > 0 && (!x_bf16 || !codes || !block_scales)) return MP_EINVAL;
  if (cols % 16 != 0 || (block_2d && rows % 16 != 0)) return MP_ESHAPE;
  if (need_ws && (!d_workspace || workspace_bytes < kNvfp4WorkspaceBytes)) return MP_EWORKSPACE;
  if ((n > 0 && (!aligned16(x_bf16) || !aligned16(codes))) || (dequant_bf16 && !aligned16(dequant_bf16)) ||
      (reinterpret_cast<uintptr_t>(d_tensor_scale) & 3u) || (reinterpret_cast<uintptr_t>(d_nonfinite) & 3u) ||
      (need_ws && (reinterpret_cast<uintptr_t>(d_workspace) & 7u)))
    return MP_EALIGN;
  return MP_OK;
}

}  // namespace
}  // namespace mp

extern "C" {

MP_API size_t nvfp4_workspace_size(void) { return mp::kNvfp4WorkspaceBytes; }

MP_API mp_status nvfp4_quantize(const void* x_bf16, int64_t rows, int64_t cols, int32_t block_2d,
                                int32_t stochastic, uint64_t seed, int32_t apply_rht, uint16_t rht_sign_mask,
                                uint8_t* codes, uint8_t* block_scales, float* d_tensor_scale,
                                int32_t* d_nonfinite, void* dequant_bf16, void* d_workspace,
                                size_t workspace_bytes, void* stream) {
  using namespace mp;
  const mp_status bad = nvfp4_check_args(x_bf16, rows, cols, block_2d, codes, block_scales, d_tensor_scale,
                                         d_nonfinite, dequant_bf16, true, d_workspace, workspace_bytes);
  if (bad != MP_OK) return bad;
  const int64_t n = rows * cols;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
  Ws* ws = static_cast<Ws*>(d_workspace);
  uint16_t* dq = static_cast<uint16_t*>(dequant_bf16);
  const uint32_t mask = rht_sign_mask;
  const bool b2 = block_2d != 0, deq = dq != nullptr;
  const int64_t kf = keep_from_of(n / 16, block_2d != 0);
  if (apply_rht) launch_amax<true>(x, n / 16, mask, ws, d_tensor_scale, d_nonfinite, kf, s);
  else launch_amax<false>(x, n / 16, mask, ws, d_tensor_scale, d_nonfinite, kf, s);
  if (apply_rht && stochastic)
    dispatch_deq<true, true>(deq, b2, x, rows, cols, mask, seed, d_tensor_scale, d_nonfinite, codes, block_scales, dq, s);
  else if (apply_rht)
    dispatch_deq<true, false>(deq, b2, x, rows, cols, mask, seed, d_tensor_scale, d_nonfinite, codes, block_scales, dq, s);
  else if (stochastic)
    dispatch_deq<false, true>(deq, b2, x, rows, cols, mask, seed, d_tensor_scale, d_nonfinite, codes, block_scales, dq, s);
  else
    dispatch_deq<false, false>(deq, b2, x, rows, cols, mask, seed, d_tensor_scale, d_nonfinite, codes, block_scales, dq, s);
  note_launches(2);
  return launch_status();
}

MP_API mp_status e2m1_stochastic_round(const float* y, const uint16_t* r16, int64_t n, uint8_t* codes,
                                       void* stream) {
  using namespace mp;
  if (n < 0) return MP_EINVAL;
  if (n > 0 && (!y || !r16 || !codes)) return MP_EINVAL;
  if (n > 0 && (!aligned16(y) || !aligned16(r16) || !aligned16(codes))) return MP_EALIGN;
  if (n == 0) return MP_OK;
  const int64_t ctas = ((n + 1) / 2 + kThreads - 1) / kThreads;
  launch_chained(k_e2m1_sr, dim3(full_grid(ctas)), dim3(kThreads), 0, static_cast<cudaStream_t>(stream), y, r16, n,
                 codes);
  note_launches(1);
  return launch_status();
}

MP_API mp_status rht16(const void* x_bf16, int64_t rows, int64_t cols, uint16_t sign_mask, void* y,
                       mp_dtype y_dtype, void* stream) {
  using namespace mp;
  if (rows < 0 || cols < 0) return MP_EINVAL;
  const int64_t n = rows * cols;
  if (n > 0 && (!x_bf16 || !y)) return MP_EINVAL;
  if (y_dtype != MP_F32 && y_dtype != MP_BF16) return MP_EINVAL;
  if (cols % 16 != 0) return MP_ESHAPE;
  if (n > 0 && (!aligned16(x_bf16) || !aligned16(y))) return MP_EALIGN;
  if (n == 0) return MP_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t ntiles = n / 16;
  const int64_t ctas = (ntiles + kThreads - 1) / kThreads;
  const uint16_t* x = static_cast<const uint16_t*>(x_bf16);
  if (y_dtype == MP_F32)
    launch_chained(k_rht16<true>, dim3(full_grid(ctas)), dim3(kThreads), 0, s, x, ntiles, (uint32_t)sign_mask, y);
  else
    launch_chained(k_rht16<false>, dim3(full_grid(ctas)), dim3(kThreads), 0, s, x, ntiles, (uint32_t)sign_mask, y);
  note_launches(1);
  return launch_status();
}

}  // extern "C"

// ---------------------------------------------------------------------------
// nvfp4_quantize_noalloc: the same quantiser for callers that cannot hand the
// library a workspace.  Its scratch is this file-scope device array, created
// when the library is loaded on each device and kept until the process exits.
// Host code may not take the array's address directly (the name is a host-side
// stand-in); the device address is looked up with cudaGetSymbolAddress the
// first time each CUDA context calls, with that context current, and kept by
// the context's id, so a device reset (a new context, where the module and
// its array may sit elsewhere) looks it up again.
// ---------------------------------------------------------------------------
namespace mp {
namespace {

constexpr size_t kNoAllocScratchBytes = 256;
__device__ __align__(256) unsigned char g_nvfp4_noalloc_scratch[kNoAllocScratchBytes];

static_assert(kNvfp4WorkspaceBytes <= kNoAllocScratchBytes, "the scratch array holds one call's workspace");

// The driver's id of the current context, reached through the runtime (no
// link against the driver library).  Ids are unique for the life of the
// process, so a context destroyed and created again (cudaDeviceReset) gets a
// new one even where its handle is reused.
bool current_context_id(unsigned long long* id) {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static std::atomic<void*> get_current{nullptr}, get_id{nullptr};
  void* gc = get_current.load(std::memory_order_acquire);
  void* gi = get_id.load(std::memory_order_acquire);
  if (!gc || !gi) {
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &gc, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !gc)
      return false;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &gi, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !gi)
      return false;
    get_current.store(gc, std::memory_order_release);
    get_id.store(gi, std::memory_order_release);
  }
  CUcontext ctx = nullptr;
  if (reinterpret_cast<GetCurrent>(gc)(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return reinterpret_cast<GetId>(gi)(ctx, id) == CUDA_SUCCESS;
}

// The array's device address in the current context, looked up with
// cudaGetSymbolAddress the first time a context calls and kept per context id.
constexpr int kMaxContexts = 64;
std::mutex g_scratch_mu;
struct ScratchEntry {
  unsigned long long ctx_id;
  void* addr;
};
ScratchEntry g_scratch[kMaxContexts] = {};
int g_scratch_used = 0;

mp_status noalloc_scratch_for_current_context(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MP_ECUDA;
  unsigned long long id = 0;
  if (!current_context_id(&id)) {
    // No context is current on this thread yet: the runtime would use the
    // device's primary context, which cudaSetDevice makes current.
    if (cudaSetDevice(dev) != cudaSuccess || !current_context_id(&id)) return MP_ECUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  for (int i = 0; i < g_scratch_used; ++i)
    if (g_scratch[i].ctx_id == id) {
      *out = g_scratch[i].addr;
      return MP_OK;
    }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_nvfp4_noalloc_scratch) != cudaSuccess || !p) return MP_ECUDA;
  const int slot = g_scratch_used < kMaxContexts ? g_scratch_used++ : (int)(id % kMaxContexts);
  g_scratch[slot] = ScratchEntry{id, p};
  *out = p;
  return MP_OK;
}

}  // namespace
}  // namespace mp

extern "C" MP_API size_t nvfp4_noalloc_scratch_bytes(void) { return mp::kNoAllocScratchBytes; }

extern "C" MP_API mp_status nvfp4_quantize_noalloc(const void* x_bf16, int64_t rows, int64_t cols,
                                                   int32_t block_2d, int32_t stochastic, uint64_t seed,
                                                   int32_t apply_rht, uint16_t rht_sign_mask, uint8_t* codes,
                                                   uint8_t* block_scales, float* d_tensor_scale,
                                                   int32_t* d_nonfinite, void* dequant_bf16, void* stream) {
  using namespace mp;
  // Every argument is checked before anything is enqueued or looked up.
  const mp_status bad = nvfp4_check_args(x_bf16, rows, cols, block_2d, codes, block_scales, d_tensor_scale,
                                         d_nonfinite, dequant_bf16, false, nullptr, 0);
  if (bad != MP_OK) return bad;
  // A call needs nvfp4_workspace_size() bytes of scratch; the fixed array
  // must hold that much.
  if (nvfp4_workspace_size() > kNoAllocScratchBytes) return MP_EWORKSPACE;
  void* scratch = nullptr;
  const mp_status rc = noalloc_scratch_for_current_context(&scratch);
  if (rc != MP_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The accumulator and ticket must start at zero; clear them in stream order.
  if (cudaMemsetAsync(scratch, 0, sizeof(Ws), s) != cudaSuccess) return MP_ECUDA;
  return nvfp4_quantize(x_bf16, rows, cols, block_2d, stochastic, seed, apply_rht, rht_sign_mask, codes,
                        block_scales, d_tensor_scale, d_nonfinite, dequant_bf16, scratch, kNoAllocScratchBytes,
                        stream);
}
