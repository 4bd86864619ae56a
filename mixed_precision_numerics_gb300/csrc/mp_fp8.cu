// mp_fp8.cu — FP8 delayed-scaling cast, one read of the input.
//
// [FP8-TE] llm-wiki "FP8 혼합 정밀도 LLM 학습 ...": "Delayed Scaling 동작 원리"
// (amax history ring; scale = fp8_max / (margin * max(history)); the tensor is
// read once because the scale comes from earlier steps), "FP8이 어려운 이유"
// (x_fp8 = clip(x/s, -448, 448)), "E4M3 vs E5M2" (E4M3 forward, E5M2 grads).
//
// k_fp8_cast: every thread streams 16 input elements per vector (32 B of
// BF16/F16, 64 B of F32), 128 B of input in flight, and writes 16 output bytes
// per vector, keeping a running NaN-propagating max |x| in a register.  CTAs
// fold their amax into the meta word with one atomicMax each; CTA 0 folds the
// history entries the call does not overwrite while the stream runs; the last
// CTA to finish (atomic ticket, no waiting) writes the ring slot and derives
// the next scale from the two maxima.
#include "mp_device.cuh"
#include "mp_internal.h"

namespace mp {
namespace {

constexpr int kThreads = 256;
constexpr int kElems = 16;  // elements per vector

enum { XF32 = 0, XF16 = 1, XBF16 = 2 };

// Vectors in flight per thread: 128 bytes of input either way.
template <int XT>
__host__ __device__ constexpr int unroll_of() { return XT == XF32 ? 2 : 4; }

// Raw 16-element vector: two 16-byte words of 16-bit values, or four of FP32.
template <int XT>
__device__ __forceinline__ void load_raw(const void* x, int64_t vec, uint4 (&r)[4]) {
  if constexpr (XT == XF32) {
    const uint4* p = static_cast<const uint4*>(x) + vec * 4;
#pragma unroll
    for (int k = 0; k < 4; ++k) r[k] = __ldcs(p + k);
  } else {
    const uint4* p = static_cast<const uint4*>(x) + vec * 2;
    r[0] = __ldcs(p);
    r[1] = __ldcs(p + 1);
  }
}

// Element pair k (elements 2k, 2k+1) of a raw vector as floats.
template <int XT>
__device__ __forceinline__ float2 pair_of(const uint4 (&r)[4], int k) {
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

template <int XT>
__device__ __forceinline__ float load1(const void* x, int64_t i) {
  if constexpr (XT == XF32) return static_cast<const float*>(x)[i];
  const uint32_t h = static_cast<const uint16_t*>(x)[i];
  return XT == XBF16 ? bf16lo(h) : f16lo(h);
}

// Saturating RNE cast of a product pair: clamp to +-max first (infinities
// included; NaN is handled by the caller), then the hardware cvt.
template <bool E5M2>
__device__ __forceinline__ uint32_t cast_pair(float p0, float p1) {
  constexpr float fmax = E5M2 ? 57344.0f : 448.0f;
  p0 = fminf(fmaxf(p0, -fmax), fmax);
  p1 = fminf(fmaxf(p1, -fmax), fmax);
  return E5M2 ? cvt_e5m2x2(p0, p1) : cvt_e4m3x2(p0, p1);
}

// Ordered key of a history entry: NaN above everything, non-positive as 0.
__device__ __forceinline__ uint32_t hist_key(float h) {
  return (h != h) ? 0x7FC00000u : (h > 0.0f ? __float_as_uint(h) : 0u);
}

template <int XT, bool E5M2>
__global__ __launch_bounds__(kThreads) void k_fp8_cast(const void* __restrict__ x, int64_t n,
                                                       uint8_t* __restrict__ y, mp_fp8_meta* meta,
                                                       float* hist, int32_t hist_len, float margin) {
  constexpr int U = unroll_of<XT>();
  __shared__ uint32_t red[32];
  __shared__ int is_last;
  const float scale = meta->scale;
  const int32_t slot = ((meta->pos % hist_len) + hist_len) % hist_len;  // slot taken modulo the ring length

  // CTA 0 folds the history entries this call does not overwrite while the
  // stream runs, so the last CTA only has to combine them with this amax.
  if (blockIdx.x == 0) {
    uint32_t hm = 0;
    for (int i = threadIdx.x; i < hist_len; i += kThreads)
      if (i != slot) hm = max(hm, hist_key(hist[i]));
    hm = block_max_u32(hm, red);
    if (threadIdx.x == 0) meta->internal_hrest = hm;
    __syncthreads();  // red is reused below
  }

  float acc = 0.0f;
  const int64_t nvec = n / kElems;
  const int64_t step = (int64_t)gridDim.x * kThreads * U;
  for (int64_t v0 = (int64_t)blockIdx.x * kThreads * U + threadIdx.x; v0 < nvec; v0 += step) {
    uint4 raw[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t vec = v0 + (int64_t)u * kThreads;
      if (vec < nvec) load_raw<XT>(x, vec, raw[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t vec = v0 + (int64_t)u * kThreads;
      if (vec >= nvec) continue;
      float vmax = 0.0f;
      uint32_t h[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float2 f = pair_of<XT>(raw[u], k);
        vmax = max_abs_nan(vmax, f.x);
        vmax = max_abs_nan(vmax, f.y);
        h[k] = cast_pair<E5M2>(__fmul_rn(f.x, scale), __fmul_rn(f.y, scale));
      }
      uint4 o = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
      if (__builtin_expect(vmax != vmax, 0)) {  // a NaN input: its byte is 0x7F
        uint8_t* ob = reinterpret_cast<uint8_t*>(&o);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float2 f = pair_of<XT>(raw[u], k);
          if (f.x != f.x) ob[2 * k] = 0x7F;
          if (f.y != f.y) ob[2 * k + 1] = 0x7F;
        }
      }
      st_cs(y + vec * kElems, o);
      acc = max_abs_nan(acc, vmax);
    }
  }
  // Tail elements (n % 16) go to the first CTA.
  if (blockIdx.x == 0) {
    const int64_t i = nvec * kElems + threadIdx.x;
    if (i < n) {
      const float a = load1<XT>(x, i);
      acc = max_abs_nan(acc, a);
      uint32_t b = cast_pair<E5M2>(__fmul_rn(a, scale), 0.0f) & 0xFFu;
      if (a != a) b = 0x7F;
      y[i] = (uint8_t)b;
    }
  }

  const uint32_t cta = block_max_u32(amax_bits(acc), red);
  if (threadIdx.x == 0) {
    atomicMax(&meta->internal_amax, cta);
    __threadfence();
    is_last = atomicAdd(&meta->internal_ticket, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!is_last || threadIdx.x != 0) return;

  // Last CTA: record this step's amax and derive the next scale.
  __threadfence();
  const uint32_t ab = atomicExch(&meta->internal_amax, 0u);
  const uint32_t hm = max(*reinterpret_cast<volatile uint32_t*>(&meta->internal_hrest), ab);
  meta->internal_ticket = 0;
  const float amax = __uint_as_float(ab);
  meta->amax = amax;
  hist[slot] = amax;
  meta->pos = (slot + 1) % hist_len;
  const float H = __uint_as_float(hm);
  if (isfinite(H) && H > 0.0f) {
    const float denom = __fmul_rn(margin, H);
    if (isfinite(denom) && denom > 0.0f) {
      const float ns = __fdiv_rn(E5M2 ? 57344.0f : 448.0f, denom);
      if (isfinite(ns) && ns > 0.0f) {
        meta->scale = ns;
        meta->scale_inv = __fdiv_rn(1.0f, ns);
      }
    }
  }
}

template <int XT, bool E5M2>
mp_status launch(const void* x, int64_t n, uint8_t* y, mp_fp8_meta* meta, float* hist, int32_t len,
                 float margin, cudaStream_t s) {
  static int occ = 0;
  if (occ == 0) {
    int o = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, k_fp8_cast<XT, E5M2>, kThreads, 0) != cudaSuccess || o < 1)
      o = 1;
    occ = o;
  }
  const int64_t nvec = n / kElems;
  constexpr int U = unroll_of<XT>();
  const int64_t ctas = (nvec + (int64_t)kThreads * U - 1) / ((int64_t)kThreads * U);
  k_fp8_cast<XT, E5M2><<<grid_for(ctas, occ), kThreads, 0, s>>>(x, n, y, meta, hist, len, margin);
  note_launches(1);
  return launch_status();
}

}  // namespace
}  // namespace mp

extern "C" MP_API mp_status fp8_cast_delayed(const void* x, mp_dtype x_dtype, int64_t n, void* y,
                                             mp_dtype fp8_dtype, mp_fp8_meta* d_meta, float* d_history,
                                             int32_t history_len, float margin, void* stream) {
  using namespace mp;
  if (n < 0 || !d_meta || !d_history || history_len < 1 || history_len > 65536) return MP_EINVAL;
  if (n > 0 && (!x || !y)) return MP_EINVAL;
  if (x_dtype != MP_F32 && x_dtype != MP_F16 && x_dtype != MP_BF16) return MP_EINVAL;
  if (fp8_dtype != MP_E4M3 && fp8_dtype != MP_E5M2) return MP_EINVAL;
  if (!(margin > 0.0f) || !(margin - margin == 0.0f)) return MP_EINVAL;
  if ((n > 0 && (!aligned16(x) || !aligned16(y))) || (reinterpret_cast<uintptr_t>(d_meta) & 15u) ||
      (reinterpret_cast<uintptr_t>(d_history) & 3u))
    return MP_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* yb = static_cast<uint8_t*>(y);
  const bool e5 = fp8_dtype == MP_E5M2;
  switch (x_dtype) {
    case MP_F32:
      return e5 ? launch<XF32, true>(x, n, yb, d_meta, d_history, history_len, margin, s)
                : launch<XF32, false>(x, n, yb, d_meta, d_history, history_len, margin, s);
    case MP_F16:
      return e5 ? launch<XF16, true>(x, n, yb, d_meta, d_history, history_len, margin, s)
                : launch<XF16, false>(x, n, yb, d_meta, d_history, history_len, margin, s);
    default:
      return e5 ? launch<XBF16, true>(x, n, yb, d_meta, d_history, history_len, margin, s)
                : launch<XBF16, false>(x, n, yb, d_meta, d_history, history_len, margin, s);
  }
}
