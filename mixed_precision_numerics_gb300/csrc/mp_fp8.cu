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
// fold their amax into the meta word with one atomicMax each; every CTA first
// folds a small slice of the history entries the call does not overwrite into
// a second word; the last CTA to finish (atomic ticket, no waiting) writes the
// ring slot and derives the next scale from the two maxima.
//
// The 2-D tile casts -- the cast with a transposed copy (k_fp8_cast_t_tma)
// and the fine-grained cast with 128x128 block scales (k_fp8_block_tma) --
// read 128 x 128 boxes through 2-D tensor copies into a shared-memory ring
// that one producer lane keeps full, consumed by groups of eight warps; each
// wait is bounded and a wait that gives up is counted for mp_wait_failures.
// The cast with 1x128 tile scales (k_fp8_rows128) reads into registers, four
// lanes per tile, with every CTA the tensor needs launched at once.
#include <string.h>

#include "mp_chain.cuh"
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

// Sign bits of element pair k of a raw vector, as 0x80 or 0 per element.  Read
// from the stored bits: the FP16 -> FP32 conversion does not keep a NaN's sign.
template <int XT>
__device__ __forceinline__ uint2 signs_of(const uint4 (&r)[4], int k) {
  if constexpr (XT == XF32) {
    const uint4 q = r[k >> 1];
    const uint32_t a = (k & 1) ? q.z : q.x, b = (k & 1) ? q.w : q.y;
    return make_uint2((a >> 24) & 0x80u, (b >> 24) & 0x80u);
  } else {
    const uint4 q = r[k >> 2];
    const uint32_t w = (k & 3) == 0 ? q.x : (k & 3) == 1 ? q.y : (k & 3) == 2 ? q.z : q.w;
    return make_uint2((w >> 8) & 0x80u, (w >> 24) & 0x80u);
  }
}

template <int XT>
__device__ __forceinline__ uint32_t sign1(const void* x, int64_t i) {
  if constexpr (XT == XF32) return (static_cast<const uint32_t*>(x)[i] >> 24) & 0x80u;
  return (static_cast<const uint16_t*>(x)[i] >> 8) & 0x80u;
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

// At the start of a history-max cast every CTA folds a strided slice of the
// history entries this call does not overwrite (entries blockIdx.x + k *
// gridDim.x) into meta->internal_hrest: the keys of a warp are reduced in
// registers and its lane 0 issues one atomicMax, so no barrier and few
// atomics; the last CTA reads and clears the word.  Called by whole warps.
__device__ __forceinline__ void fold_history_slice(mp_fp8_meta* meta, const float* hist, int32_t hist_len,
                                                   int32_t slot) {
  uint32_t k = 0;
  for (int64_t i = blockIdx.x + (int64_t)threadIdx.x * gridDim.x; i < hist_len;
       i += (int64_t)blockDim.x * gridDim.x)
    if (i != slot) k = max(k, hist_key(hist[i]));
  k = __reduce_max_sync(0xFFFFFFFFu, k);
  if ((threadIdx.x & 31) == 0 && k) atomicMax(&meta->internal_hrest, k);
}

// End of every CTA: fold its amax into the meta word; the last CTA (atomic
// ticket, no waiting) writes the ring slot and derives the next scale from
// max(history) (algo 0) or from this amax alone (algo 1).
// The part run by one thread of each CTA, with the CTA's amax bits.
template <bool E5M2>
__device__ __forceinline__ void fp8_finish_one(mp_fp8_meta* meta, float* hist, int32_t hist_len, int32_t slot,
                                               float margin, int32_t algo, uint32_t cta) {
  atomicMax(&meta->internal_amax, cta);
  __threadfence();
  if (atomicAdd(&meta->internal_ticket, 1u) != gridDim.x - 1) return;
  __threadfence();
  const uint32_t ab = atomicExch(&meta->internal_amax, 0u);
  const uint32_t hm = algo == 1 ? ab : max(atomicExch(&meta->internal_hrest, 0u), ab);
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

template <bool E5M2>
__device__ __forceinline__ void fp8_finish(mp_fp8_meta* meta, float* hist, int32_t hist_len, int32_t slot,
                                           float margin, int32_t algo, float acc, uint32_t* red) {
  const uint32_t cta = block_max_u32(amax_bits(acc), red);
  if (threadIdx.x == 0) fp8_finish_one<E5M2>(meta, hist, hist_len, slot, margin, algo, cta);
}

// FP8 byte of a NaN product: S.1111111 with the input element's sign bit.
__device__ __forceinline__ uint8_t nan_byte(uint32_t sign80) { return (uint8_t)(0x7Fu | sign80); }

// Saturating RNE conversion of a product pair with no clamp: the conversion's
// satfinite mode takes every magnitude beyond fp8_max, infinities included,
// to fp8_max with its sign.  NaN is handled by the caller.
template <bool E5M2>
__device__ __forceinline__ uint32_t cvt_pair_sat(float p0, float p1) {
  return E5M2 ? cvt_e5m2x2(p0, p1) : cvt_e4m3x2(p0, p1);
}

// True if x * scale can be NaN only where x is NaN.
__device__ __forceinline__ bool scale_keeps_numbers(float scale) { return scale > 0.0f && scale < INFINITY; }

// Casts one raw 16-element vector with multiplier `scale`; returns the 16
// output bytes and the vector's NaN-propagating max |x| in *vmax.  A NaN
// product (a NaN input, or an infinite input times a zero multiplier) gives
// 0x7F with the input element's sign bit (0xFF when negative).  With a
// finite positive multiplier only a NaN input makes a NaN product, so the
// vector's own max tells whether the products need checking; otherwise they
// are checked one by one.  The sign is read from the input.
template <int XT, bool E5M2>
__device__ __forceinline__ uint4 cast16(const uint4 (&raw)[4], float scale, float* vmax_out,
                                        uint32_t* saturated = nullptr) {
  constexpr float fmax = E5M2 ? 57344.0f : 448.0f;
  float vmax = 0.0f;
  uint32_t h[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 f = pair_of<XT>(raw, k);
    vmax = max_abs_nan(vmax, f.x);
    vmax = max_abs_nan(vmax, f.y);
    const float p0 = __fmul_rn(f.x, scale), p1 = __fmul_rn(f.y, scale);
    if (saturated) *saturated += (fabsf(p0) > fmax) + (fabsf(p1) > fmax);  // NaN compares false
    h[k] = cvt_pair_sat<E5M2>(p0, p1);
  }
  uint4 o = make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
  if (__builtin_expect((vmax != vmax) || !scale_keeps_numbers(scale), 0)) {
    uint8_t* ob = reinterpret_cast<uint8_t*>(&o);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float2 f = pair_of<XT>(raw, k);
      const uint2 sg = signs_of<XT>(raw, k);
      if (__fmul_rn(f.x, scale) != __fmul_rn(f.x, scale)) ob[2 * k] = nan_byte(sg.x);
      if (__fmul_rn(f.y, scale) != __fmul_rn(f.y, scale)) ob[2 * k + 1] = nan_byte(sg.y);
    }
  }
  *vmax_out = vmax;
  return o;
}

template <int XT, bool E5M2, bool COUNT>
__global__ __launch_bounds__(kThreads) void k_fp8_cast(const void* __restrict__ x, int64_t n,
                                                       uint8_t* __restrict__ y, mp_fp8_meta* meta,
                                                       float* hist, int32_t hist_len, float margin, int32_t algo,
                                                       unsigned long long* saturated_out) {
  chain_wait();  // the previous kernel in the stream has finished and its writes are visible
  chain_release();
  constexpr int U = unroll_of<XT>();
  __shared__ uint32_t red[32];
  const float scale = meta->scale;
  const int32_t slot = ((meta->pos % hist_len) + hist_len) % hist_len;  // slot taken modulo the ring length
  // This thread's share of the history fold (fold_history_slice's entries):
  // the first entry is loaded now and folded after the stream, by when it has
  // arrived, so no thread waits on it before issuing its input loads.  Entries beyond the first (only when the ring has more
  // entries than the grid has threads) are read at the fold.
  const int64_t h0 = blockIdx.x + (int64_t)threadIdx.x * gridDim.x;
  const float hv = (algo == 0 && h0 < hist_len && h0 != slot) ? hist[h0] : 0.0f;
  bool folded = algo != 0;
  auto fold = [&]() {  // called by whole warps: one atomic per warp
    uint32_t k = hist_key(hv);
    for (int64_t i = h0 + (int64_t)blockDim.x * gridDim.x; i < hist_len; i += (int64_t)blockDim.x * gridDim.x)
      if (i != slot) k = max(k, hist_key(hist[i]));
    k = __reduce_max_sync(0xFFFFFFFFu, k);
    if ((threadIdx.x & 31) == 0 && k) atomicMax(&meta->internal_hrest, k);
    folded = true;
  };

  float acc = 0.0f;
  uint32_t sat = 0;  // saturated elements (COUNT only)
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
      float vmax;
      st_cs(y + vec * kElems, cast16<XT, E5M2>(raw[u], scale, &vmax, COUNT ? &sat : nullptr));
      acc = max_abs_nan(acc, vmax);
    }
  }
  if (!folded) fold();
  // Tail elements (n % 16) go to the first CTA.
  if (blockIdx.x == 0) {
    const int64_t i = nvec * kElems + threadIdx.x;
    if (i < n) {
      const float a = load1<XT>(x, i);
      acc = max_abs_nan(acc, a);
      const float p = __fmul_rn(a, scale);
      uint32_t b = cast_pair<E5M2>(p, 0.0f) & 0xFFu;
      if (p != p) b = nan_byte(sign1<XT>(x, i));
      y[i] = (uint8_t)b;
      if (COUNT) sat += fabsf(p) > (E5M2 ? 57344.0f : 448.0f);
    }
  }
  if (COUNT) {
#pragma unroll
    for (int h = 16; h >= 1; h >>= 1) sat += __shfl_xor_sync(0xFFFFFFFFu, sat, h);
    if ((threadIdx.x & 31) == 0 && sat) atomicAdd(saturated_out, (unsigned long long)sat);
  }
  fp8_finish<E5M2>(meta, hist, hist_len, slot, margin, algo, acc, red);
}

// 4 x 4 byte transpose: w[i] holds row i (byte j = column j); returns in
// c[j] the column j (byte i = row i).
__device__ __forceinline__ void transpose4x4(const uint32_t (&w)[4], uint32_t (&c)[4]) {
  const uint32_t a0 = __byte_perm(w[0], w[1], 0x5140), a1 = __byte_perm(w[0], w[1], 0x7362);
  const uint32_t a2 = __byte_perm(w[2], w[3], 0x5140), a3 = __byte_perm(w[2], w[3], 0x7362);
  c[0] = __byte_perm(a0, a2, 0x5410);
  c[1] = __byte_perm(a0, a2, 0x7632);
  c[2] = __byte_perm(a1, a3, 0x5410);
  c[3] = __byte_perm(a1, a3, 0x7632);
}

// ---------------------------------------------------------------------------
// Fine-grained FP8 with online block scales ([FP8-TE] "DeepSeek-V3 FP8 학습
// 사례"; [MPT-ko] "FP8 혼합 정밀도"): each 1x128 tile or 128x128 block is read
// once, its amax reduced on chip, s = amax / fp8_max stored, and its elements
// cast with r = fp8_max / amax (0 if amax is zero or not finite).
// ---------------------------------------------------------------------------
template <bool E5M2>
__device__ __forceinline__ void block_scale_of(float amax, float* s, float* r) {
  constexpr float fmax = E5M2 ? 57344.0f : 448.0f;
  *s = (amax != amax) ? __uint_as_float(0x7FC00000u) : __fdiv_rn(amax, fmax);  // NaN block: quiet NaN
  *r = (isfinite(amax) && amax > 0.0f) ? __fdiv_rn(fmax, amax) : 0.0f;
}

// ---------------------------------------------------------------------------
// 128 x 128 blocks through the tensor-copy engine.  One persistent CTA per SM:
// a producer warp (one lane) issues one 2-D TMA copy per block into a ring of
// shared-memory stages (six 32 KB stages for 16-bit input, two 64 KB for
// FP32).  The consumers are kGroups groups of eight warps; group g
// takes the CTA's rounds g, g + kGroups, ..., so several blocks are reduced
// and cast at once.  A consumer thread reads its 16-byte groups (8 or 4
// elements) of the stage into registers and releases the stage at once, so
// the next copy starts while the block is reduced (four independent maxima,
// packed for 16-bit input, a warp reduction, then one named barrier per
// group, the partial maxima double-buffered by round) and cast from
// registers.  Warp w of a group takes rows 2w + 16k, k = 0..7 (16-bit; FP32
// rows w + 8k, k = 0..15), whole row segments,
// so shared-memory reads cover 512 consecutive bytes per instruction and
// every store writes whole row segments.  Parts of an edge block outside the
// tensor arrive as zeros, which leave the amax unchanged, and are not stored.
// ---------------------------------------------------------------------------
constexpr int kGroupWarps = 8;
constexpr int kGroupThreads = 32 * kGroupWarps;
constexpr int kRingBytes = 192 * 1024;

__device__ unsigned int g_wait_failures;  // bounded waits that gave up (read by mp_wait_failures)

// Ring stage s is filled for the CTA's rounds s, s + kStages, ...; group g
// takes rounds g, g + kGroups, ...  With kStages a multiple of kGroups every
// stage belongs to one group, which waits for the stage's fills in order, so a
// parity wait can never match a phase two fills old.  (A stage shared by two
// groups would let one group run a fill ahead of the other, see the previous
// fill's parity and read stale bytes, and its early arrivals would let the
// producer re-arm a barrier whose phase has not completed.)
template <int XT>
struct BlkGeom {
  static constexpr int kEs = XT == XF32 ? 4 : 2;                 // input element bytes
  static constexpr int kG = 16 / kEs;                             // elements per 16-byte group
  static constexpr int kStage = 128 * 128 * kEs;                  // one block
  static constexpr int kGroups = XT == XF32 ? 2 : 3;              // consumer groups (register budget)
  static constexpr int kStages = XT == XF32 ? 2 : 6;              // 128 KB or 192 KB of ring
  static constexpr int kGpt = 128 * 128 / kG / kGroupThreads;     // 16-byte groups per consumer thread: 8 or 16
  static constexpr int kThreads = kGroups * kGroupThreads + 32;   // + the producer warp
  static constexpr size_t kSmem = (size_t)kStages * kStage + 2 * kStages * sizeof(uint64_t) +
                                  (size_t)kGroups * 2 * kGroupWarps * sizeof(uint32_t);
  static_assert(kStages % kGroups == 0, "every ring stage must belong to one consumer group");
  static_assert(kStages * kStage <= kRingBytes, "ring larger than its budget");
};

// One 16-byte group of raw input (8 16-bit or 4 FP32 elements) cast with
// multiplier r: 8 (or 4) output bytes, element 0 in the lowest byte.  NaN
// products take S.1111111 with the input element's sign.
template <int XT, bool E5M2>
__device__ __forceinline__ uint2 cast_group(const uint4 q, float r) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  if constexpr (XT == XF32) {
    float p[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = __fmul_rn(__uint_as_float(w[i]), r);
    uint32_t o = cast_pair<E5M2>(p[0], p[1]) | (cast_pair<E5M2>(p[2], p[3]) << 16);
    if (__builtin_expect((p[0] != p[0]) | (p[1] != p[1]) | (p[2] != p[2]) | (p[3] != p[3]), 0)) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (p[i] != p[i]) o = (o & ~(0xFFu << (8 * i))) | ((uint32_t)nan_byte((w[i] >> 24) & 0x80u) << (8 * i));
    }
    return make_uint2(o, 0u);
  } else {
    float p[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo = XT == XBF16 ? bf16lo(w[k]) : f16lo(w[k]);
      const float hi = XT == XBF16 ? bf16hi(w[k]) : f16hi(w[k]);
      p[2 * k] = __fmul_rn(lo, r);
      p[2 * k + 1] = __fmul_rn(hi, r);
    }
    uint32_t o[2];
#pragma unroll
    for (int h = 0; h < 2; ++h)
      o[h] = cast_pair<E5M2>(p[4 * h], p[4 * h + 1]) | (cast_pair<E5M2>(p[4 * h + 2], p[4 * h + 3]) << 16);
    bool any = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) any |= p[i] != p[i];
    if (__builtin_expect(any, 0)) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t sg = (w[i >> 1] >> ((i & 1) ? 24 : 8)) & 0x80u;
        if (p[i] != p[i]) o[i >> 2] = (o[i >> 2] & ~(0xFFu << (8 * (i & 3)))) | ((uint32_t)nan_byte(sg) << (8 * (i & 3)));
      }
    }
    return make_uint2(o[0], o[1]);
  }
}

// NaN-propagating max magnitude of a group, word j into accumulator j: FP32
// words as floats, 16-bit pairs packed (the two halves are folded at the end).
template <int XT>
__device__ __forceinline__ void group_max(const uint4 q, uint32_t (&acc)[4]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if constexpr (XT == XF32)
      acc[j] = __float_as_uint(max_abs_nan(__uint_as_float(acc[j]), __uint_as_float(w[j])));
    else
      acc[j] = max_abs_nan_x2<XT == XBF16>(acc[j], w[j]);
  }
}

// The four accumulators of group_max folded to one float (NaN if any is NaN).
template <int XT>
__device__ __forceinline__ float fold_max(const uint32_t (&acc)[4]) {
  if constexpr (XT == XF32) {
    return max_abs_nan(max_abs_nan(__uint_as_float(acc[0]), __uint_as_float(acc[1])),
                       max_abs_nan(__uint_as_float(acc[2]), __uint_as_float(acc[3])));
  } else {
    const uint32_t m = max_abs_nan_x2<XT == XBF16>(max_abs_nan_x2<XT == XBF16>(acc[0], acc[1]),
                                                   max_abs_nan_x2<XT == XBF16>(acc[2], acc[3]));
    const float lo = XT == XBF16 ? bf16lo(m) : f16lo(m), hi = XT == XBF16 ? bf16hi(m) : f16hi(m);
    return max_abs_nan(lo, hi);
  }
}

// cast_group for products known not to be NaN (a block whose amax is finite,
// or a NaN-free group under a finite positive scale): the conversion's
// satfinite mode saturates every larger magnitude, infinities included, so
// neither the clamp nor the NaN repair is needed.
template <int XT, bool E5M2>
__device__ __forceinline__ uint2 cast_group_finite(const uint4 q, float r) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint32_t h[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    float a, b;
    if constexpr (XT == XF32) {
      if (k >= 2) break;
      a = __uint_as_float(w[2 * k]);
      b = __uint_as_float(w[2 * k + 1]);
    } else {
      a = XT == XBF16 ? bf16lo(w[k]) : f16lo(w[k]);
      b = XT == XBF16 ? bf16hi(w[k]) : f16hi(w[k]);
    }
    const float p0 = __fmul_rn(a, r), p1 = __fmul_rn(b, r);
    h[k] = cvt_pair_sat<E5M2>(p0, p1);
  }
  if constexpr (XT == XF32) return make_uint2(h[0] | (h[1] << 16), 0u);
  return make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
}

// One scale per 128 x 128 box (block).
template <int XT, bool E5M2>
__global__ __launch_bounds__(BlkGeom<XT>::kThreads, 1) void k_fp8_block_tma(
    const __grid_constant__ CUtensorMap map, int64_t rows, int64_t cols, uint8_t* __restrict__ y,
    float* __restrict__ scales) {
  chain_wait();  // the previous kernel in the stream has finished and its writes are visible
  chain_release();
  using Gm = BlkGeom<XT>;
  constexpr int kS = Gm::kStages, kSB = Gm::kStage, kG = Gm::kG, kGpr = 128 / kG;  // groups per row
  constexpr int kNG = Gm::kGroups;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kS * kSB);
  uint64_t* empty = full + kS;
  uint32_t* red = reinterpret_cast<uint32_t*>(empty + kS);  // [kGroups][2][kGroupWarps]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nbc = (cols + 127) / 128, nb = ((rows + 127) / 128) * nbc;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kGroupWarps);  // the eight warps of the group that reads the stage
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kNG * kGroupWarps) {
    // Producer: one lane issues the block copies.
    if (lane != 0) return;
    prefetch_tensor_map(&map);
    const uint64_t policy = policy_evict_first();
    int issued = 0;
    bool ok = true;
    for (int64_t b = blockIdx.x; b < nb; b += gridDim.x, ++issued) {
      const int sidx = issued % kS;
      if (!mbar_wait_bounded(&empty[sidx], ((issued / kS) & 1) ^ 1)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(&full[sidx], kSB);
      tma_load_2d(smem + sidx * kSB, &map, (int32_t)((b % nbc) * 128), (int32_t)((b / nbc) * 128), &full[sidx],
                  policy);
    }
    if (!ok) {
      atomicAdd(&g_wait_failures, 1u);
      // Let the copies already issued land before the block's shared memory goes away.
      for (int k = issued - kS < 0 ? 0 : issued - kS; k < issued; ++k)
        (void)mbar_wait_bounded(&full[k % kS], (k / kS) & 1);
    }
    return;
  }

  // Consumers.  A warp whose wait gave up stops reading and storing but keeps
  // meeting its group's named barrier every round, so the group never blocks on it.
  const int grp = warp / kGroupWarps, gw = warp % kGroupWarps, t = threadIdx.x % kGroupThreads;
  constexpr int kRowStep = kGroupThreads / kGpr;  // rows between a thread's groups: 16 or 8
  uint32_t* gred = red + grp * 2 * kGroupWarps;
  bool ok = true;
  int it = grp, round = 0;
  for (int64_t b = blockIdx.x + (int64_t)grp * gridDim.x; b < nb; b += (int64_t)kNG * gridDim.x, it += kNG, ++round) {
    const int sidx = it % kS;
    if (ok) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&full[sidx], (it / kS) & 1));
      if (!ok && lane == 0) atomicAdd(&g_wait_failures, 1u);
    }
    uint4 raw[Gm::kGpt];
    uint32_t acc[4] = {0u, 0u, 0u, 0u};
    if (ok) {
      const uint4* st = reinterpret_cast<const uint4*>(smem + sidx * kSB);
#pragma unroll
      for (int k = 0; k < Gm::kGpt; ++k) raw[k] = st[t + kGroupThreads * k];
#pragma unroll
      for (int k = 0; k < Gm::kGpt; ++k) group_max<XT>(raw[k], acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[sidx]);  // the stage's bytes are all in registers
    }
    const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, amax_bits(fold_max<XT>(acc)));
    if (lane == 0) gred[(round & 1) * kGroupWarps + gw] = m;
    named_barrier(1 + grp, kGroupThreads);
    if (!ok) continue;
    uint32_t mb = 0;
#pragma unroll
    for (int w = 0; w < kGroupWarps; ++w) mb = max(mb, gred[(round & 1) * kGroupWarps + w]);
    const float amax = __uint_as_float(mb);
    float sc, r;
    block_scale_of<E5M2>(amax, &sc, &r);
    const int64_t row0 = (b / nbc) * 128 + t / kGpr, col = (b % nbc) * 128 + (t % kGpr) * kG;
    uint8_t* yp = y + row0 * cols + col;
    const int64_t rows_left = rows - row0;  // this thread's rows k * kRowStep < rows_left exist
    if (col < cols) {
      if (isfinite(amax)) {
#pragma unroll
        for (int k = 0; k < Gm::kGpt; ++k) {
          if (k * kRowStep >= rows_left) break;
          const uint2 o = cast_group_finite<XT, E5M2>(raw[k], r);
          if constexpr (XT == XF32)
            __stcs(reinterpret_cast<uint32_t*>(yp + (int64_t)k * kRowStep * cols), o.x);
          else
            __stcs(reinterpret_cast<uint2*>(yp + (int64_t)k * kRowStep * cols), o);
        }
      } else {
#pragma unroll
        for (int k = 0; k < Gm::kGpt; ++k) {
          if (k * kRowStep >= rows_left) break;
          const uint2 o = cast_group<XT, E5M2>(raw[k], r);
          if constexpr (XT == XF32)
            __stcs(reinterpret_cast<uint32_t*>(yp + (int64_t)k * kRowStep * cols), o.x);
          else
            __stcs(reinterpret_cast<uint2*>(yp + (int64_t)k * kRowStep * cols), o);
        }
      }
    }
    if (t == 0) scales[b] = sc;
  }
}

// ---------------------------------------------------------------------------
// 1x128 tiles from registers.  Four lanes per tile, each holding a quarter of
// it (32 elements: 64 B of 16-bit input, 128 B of FP32), one quarter per
// thread, every CTA the tensor needs launched at once.  At 40 registers six
// CTAs share an SM, and that occupancy keeps DRAM busier than a TMA-fed ring
// of 32 x 256 boxes did (16.7 against 19.3 us on [8192 x 4096] BF16; two or
// four quarters per thread, or eight lanes per tile, were slower; the launch
// bound holds the 16-bit forms at 40 registers).  The tile
// max takes two shuffles within the lane quartet; every lane forms the scale
// (the same value), casts its quarter and stores its 32 output bytes, and the
// quartet's first lane stores the scale.  Quarter q is part q % 4 of tile
// q / 4; tile t covers row t / tpr, columns (t % tpr) * 128 .. + 127, with
// tpr = ceil(cols / 128); past a row's end a partial tile reads zeros, which
// leave the max unchanged, and stores nothing.
// ---------------------------------------------------------------------------
template <int XT, bool E5M2>
__global__ __launch_bounds__(kThreads, XT == XF32 ? 4 : 6) void k_fp8_rows128(const void* __restrict__ x, int64_t rows, int64_t cols,
                                                          uint8_t* __restrict__ y, float* __restrict__ scales) {
  chain_wait();  // the previous kernel in the stream has finished and its writes are visible
  chain_release();
  constexpr int kEs = XT == XF32 ? 4 : 2, kG = 16 / kEs, kQG = 32 / kG;  // 16-byte groups per quarter: 4 or 8
  const int64_t tpr = (cols + 127) / 128, nq = rows * tpr * 4;
  const int64_t q = (int64_t)blockIdx.x * kThreads + threadIdx.x, t = q >> 2;
  const int64_t row = t / tpr, col0 = (t % tpr) * 128 + (q & 3) * 32;
  const bool valid = q < nq;  // whole quartets: nq is a multiple of 4
  const unsigned char* xr = static_cast<const unsigned char*>(x) + row * cols * kEs;
  uint4 raw[kQG];
#pragma unroll
  for (int k = 0; k < kQG; ++k) {
    const int64_t c = col0 + k * kG;
    raw[k] = (valid && c < cols) ? __ldcs(reinterpret_cast<const uint4*>(xr + c * kEs)) : make_uint4(0u, 0u, 0u, 0u);
  }
  uint32_t acc[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int k = 0; k < kQG; ++k) group_max<XT>(raw[k], acc);
  uint32_t m = amax_bits(fold_max<XT>(acc));  // ordered bits, NaN above inf
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
  float sc, r;
  block_scale_of<E5M2>(__uint_as_float(m), &sc, &r);
  if (!valid) return;
  if ((q & 3) == 0) scales[row * tpr + col0 / 128] = sc;
  uint8_t* yp = y + row * cols + col0;
  constexpr int kPer = 16 / kG;  // groups per 16 output bytes
#pragma unroll
  for (int k = 0; k < kQG; k += kPer) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const uint2 o = r > 0.0f ? cast_group_finite<XT, E5M2>(raw[k + j], r) : cast_group<XT, E5M2>(raw[k + j], r);
      if constexpr (XT == XF32) {
        w[j] = o.x;
      } else {
        w[2 * j] = o.x;
        w[2 * j + 1] = o.y;
      }
    }
    if (col0 + k * kG < cols) st_cs(yp + k * kG, make_uint4(w[0], w[1], w[2], w[3]));  // cols % 16 == 0
  }
}

// ---------------------------------------------------------------------------
// Cast + transposed copy through the tensor-copy engine: the same producer and
// 128 x 128 boxes as above, a ring of one stage per consumer group (three
// 32 KB stages, or two 64 KB for FP32) and kGroups groups on alternate boxes.  A group casts its box
// from registers with the delayed scale, writes y directly and the same bytes
// row-major into its own 16 KB shared tile (two per group, alternating by
// round, so one named barrier per round suffices), then reads the tile back a
// row of 32 words per instruction, transposes 4 x 4 byte blocks with byte
// permutes and stores 16-byte row segments of y_t.  The tensor amax is kept
// per thread and reduced once per CTA at the end.
// ---------------------------------------------------------------------------
template <int XT>
struct TrGeom {
  static constexpr int kEs = XT == XF32 ? 4 : 2;
  static constexpr int kG = 16 / kEs;
  static constexpr int kStage = 128 * 128 * kEs;
  static constexpr int kGroups = XT == XF32 ? 2 : 3;
  static constexpr int kStages = XT == XF32 ? 2 : 3;              // one stage per group (see BlkGeom)
  static constexpr int kGpt = 128 * 128 / kG / kGroupThreads;     // 8 or 16
  static constexpr int kThreads = kGroups * kGroupThreads + 32;
  static constexpr int kTile = 128 * 128;                         // cast bytes of one box
  static constexpr size_t kSmem = (size_t)kStages * kStage + (size_t)kGroups * 2 * kTile +
                                  2 * kStages * sizeof(uint64_t) + (size_t)kGroups * kGroupWarps * sizeof(uint32_t);
  static_assert(kStages % kGroups == 0, "every ring stage must belong to one consumer group");
  static_assert(kSmem <= 227 * 1024, "shared memory beyond the per-CTA limit");
};

template <int XT, bool E5M2>
__global__ __launch_bounds__(TrGeom<XT>::kThreads, 1) void k_fp8_cast_t_tma(
    const __grid_constant__ CUtensorMap map, int64_t rows, int64_t cols, uint8_t* __restrict__ y,
    uint8_t* __restrict__ y_t, mp_fp8_meta* meta, float* hist, int32_t hist_len, float margin, int32_t algo) {
  chain_wait();  // the previous kernel in the stream has finished and its writes are visible
  chain_release();
  using Gm = TrGeom<XT>;
  constexpr int kS = Gm::kStages, kSB = Gm::kStage, kG = Gm::kG, kGpr = 128 / kG, kNG = Gm::kGroups;
  constexpr int kRowStep = kGroupThreads / kGpr;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* tiles = smem + kS * kSB;  // [kGroups][2][128][128]
  uint64_t* full = reinterpret_cast<uint64_t*>(tiles + kNG * 2 * Gm::kTile);
  uint64_t* empty = full + kS;
  uint32_t* red = reinterpret_cast<uint32_t*>(empty + kS);  // [kGroups * kGroupWarps]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nbc = (cols + 127) / 128, nb = ((rows + 127) / 128) * nbc;
  const float scale = meta->scale;
  const int32_t slot = ((meta->pos % hist_len) + hist_len) % hist_len;  // slot taken modulo the ring length
  if (algo == 0) fold_history_slice(meta, hist, hist_len, slot);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kGroupWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kNG * kGroupWarps) {
    if (lane != 0 || blockIdx.x >= nb) return;
    prefetch_tensor_map(&map);
    const uint64_t policy = policy_evict_first();
    int issued = 0;
    bool ok = true;
    for (int64_t b = blockIdx.x; b < nb; b += gridDim.x, ++issued) {
      const int sidx = issued % kS;
      if (!mbar_wait_bounded(&empty[sidx], ((issued / kS) & 1) ^ 1)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(&full[sidx], kSB);
      tma_load_2d(smem + sidx * kSB, &map, (int32_t)((b % nbc) * 128), (int32_t)((b / nbc) * 128), &full[sidx],
                  policy);
    }
    if (!ok) {
      atomicAdd(&g_wait_failures, 1u);
      for (int k = issued - kS < 0 ? 0 : issued - kS; k < issued; ++k)
        (void)mbar_wait_bounded(&full[k % kS], (k / kS) & 1);
    }
    return;
  }

  const int grp = warp / kGroupWarps, t = threadIdx.x % kGroupThreads;
  const int rs = (t & 7) * 16, cg = t >> 3;  // transposed side: 16-row run, 4-column group
  const bool scale_ok = scale_keeps_numbers(scale);
  uint32_t acc = 0u;  // ordered bits of this thread's running max |x|
  bool ok = true;
  int it = grp, round = 0;
  for (int64_t b = blockIdx.x + (int64_t)grp * gridDim.x; b < nb; b += (int64_t)kNG * gridDim.x, it += kNG, ++round) {
    const int sidx = it % kS;
    if (ok) {
      ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&full[sidx], (it / kS) & 1));
      if (!ok && lane == 0) atomicAdd(&g_wait_failures, 1u);
    }
    const int64_t r0 = (b / nbc) * 128, c0 = (b % nbc) * 128;
    unsigned char* tile = tiles + (grp * 2 + (round & 1)) * Gm::kTile;
    if (ok) {
      uint4 raw[Gm::kGpt];
      uint32_t racc[4] = {0u, 0u, 0u, 0u};
      const uint4* st = reinterpret_cast<const uint4*>(smem + sidx * kSB);
#pragma unroll
      for (int k = 0; k < Gm::kGpt; ++k) raw[k] = st[t + kGroupThreads * k];
#pragma unroll
      for (int k = 0; k < Gm::kGpt; ++k) group_max<XT>(raw[k], racc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[sidx]);
      const float rmax = fold_max<XT>(racc);
      acc = max(acc, amax_bits(rmax));
      const bool clean = scale_ok && rmax == rmax;  // no NaN product possible in this thread's groups
      const int rin = t / kGpr, cin = (t % kGpr) * kG;
      const int64_t row0 = r0 + rin, col = c0 + cin;
      uint8_t* yp = y + row0 * cols + col;
#pragma unroll
      for (int k = 0; k < Gm::kGpt; ++k) {
        const uint2 o = clean ? cast_group_finite<XT, E5M2>(raw[k], scale) : cast_group<XT, E5M2>(raw[k], scale);
        const int trw = rin + k * kRowStep;
        unsigned char* tp = tile + trw * 128 + (cin ^ (((trw >> 4) & 7) << 4));  // 16-byte granules XOR-swizzled
        if constexpr (XT == XF32)
          *reinterpret_cast<uint32_t*>(tp) = o.x;
        else
          *reinterpret_cast<uint2*>(tp) = o;
        if (col < cols && row0 + k * kRowStep < rows) {
          if constexpr (XT == XF32)
            __stcs(reinterpret_cast<uint32_t*>(yp + (int64_t)k * kRowStep * cols), o.x);
          else
            __stcs(reinterpret_cast<uint2*>(yp + (int64_t)k * kRowStep * cols), o);
        }
      }
    }
    named_barrier(1 + grp, kGroupThreads);
    if (!ok) continue;
    // Eight consecutive threads cover one column's 128 rows: every store
    // instruction writes four whole 128-byte lines of y_t.  Rows rs .. rs + 15
    // share the swizzle (rs / 16), which spreads the eight row runs of a
    // column group over distinct banks.
    const int64_t tcol = c0 + 4 * cg, trow = r0 + rs;
    if (tcol < cols && trow < rows) {  // rows and cols are multiples of 16: the 4 columns and 16 rows are all in
      const int sw = (4 * cg) ^ ((rs >> 4) << 4);
      uint32_t out[4][4];  // out[j][m]: column j, rows rs + 4m .. + 3
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        uint32_t w[4], c[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = *reinterpret_cast<const uint32_t*>(tile + (rs + 4 * m + i) * 128 + sw);
        transpose4x4(w, c);
#pragma unroll
        for (int j = 0; j < 4; ++j) out[j][m] = c[j];
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        st_cs(y_t + (tcol + j) * rows + trow, make_uint4(out[j][0], out[j][1], out[j][2], out[j][3]));
    }
  }
  // Tensor amax: warp, then the CTA's consumer warps (one named barrier), then
  // one thread folds it in and the last CTA finishes the history.
  const uint32_t m = __reduce_max_sync(0xFFFFFFFFu, acc);
  if (lane == 0) red[warp] = m;
  named_barrier(1 + kNG, kNG * kGroupThreads);
  if (threadIdx.x == 0) {
    uint32_t cta = 0;
    for (int w = 0; w < kNG * kGroupWarps; ++w) cta = max(cta, red[w]);
    fp8_finish_one<E5M2>(meta, hist, hist_len, slot, margin, algo, cta);
  }
}

template <typename K>
int occ_of(K kernel) {
  int o = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, kThreads, 0) != cudaSuccess || o < 1) o = 1;
  return o;
}

template <int XT, bool E5M2, bool COUNT>
mp_status launch(const void* x, int64_t n, uint8_t* y, mp_fp8_meta* meta, float* hist, int32_t len,
                 float margin, int32_t algo, unsigned long long* saturated, cudaStream_t s) {
  static const int occ = occ_of(k_fp8_cast<XT, E5M2, COUNT>);
  const int64_t nvec = n / kElems;
  constexpr int U = unroll_of<XT>();
  const int64_t ctas = (nvec + (int64_t)kThreads * U - 1) / ((int64_t)kThreads * U);
  launch_chained(k_fp8_cast<XT, E5M2, COUNT>, dim3(grid_for(ctas, occ)), dim3(kThreads), 0, s, x, n, y, meta, hist, len,
                 margin, algo, saturated);
  note_launches(1);
  return launch_status();
}


template <int XT, bool E5M2>
mp_status launch_t(const void* x, int64_t rows, int64_t cols, uint8_t* y, uint8_t* y_t, mp_fp8_meta* meta,
                   float* hist, int32_t len, float margin, int32_t algo, cudaStream_t s) {
  using Gm = TrGeom<XT>;
  CUtensorMap map;
  memset(&map, 0, sizeof(map));  // an empty tensor still runs one CTA (the history is updated); no copy is issued
  if (rows > 0 && cols > 0 && !encode_tile_map_2d(&map, x, Gm::kEs, rows, cols, 128, 128)) return MP_ECUDA;
  static std::atomic<uint64_t> smem_done{0};
  if (!smem_opt_in(k_fp8_cast_t_tma<XT, E5M2>, (int)Gm::kSmem, smem_done)) return MP_ECUDA;
  const int64_t boxes = ((rows + 127) / 128) * ((cols + 127) / 128);
  launch_chained(k_fp8_cast_t_tma<XT, E5M2>, dim3(grid_for(boxes, 1)), dim3(Gm::kThreads), Gm::kSmem, s, map, rows, cols,
                 y, y_t, meta, hist, len, margin, algo);
  note_launches(1);
  return launch_status();
}

template <int XT, bool E5M2>
mp_status launch_blockwise(const void* x, int64_t rows, int64_t cols, bool square, uint8_t* y, float* scales,
                           cudaStream_t s) {
  if (square) {
    using Gm = BlkGeom<XT>;
    CUtensorMap map;
    if (!encode_tile_map_2d(&map, x, Gm::kEs, rows, cols, 128, 128)) return MP_ECUDA;
    const int64_t boxes = ((rows + 127) / 128) * ((cols + 127) / 128);
    static std::atomic<uint64_t> smem_done{0};
    if (!smem_opt_in(k_fp8_block_tma<XT, E5M2>, (int)Gm::kSmem, smem_done)) return MP_ECUDA;
    launch_chained(k_fp8_block_tma<XT, E5M2>, dim3(grid_for(boxes, 1)), dim3(Gm::kThreads), Gm::kSmem, s, map,
                   rows, cols, y, scales);
  } else {
    const int64_t quarters = rows * ((cols + 127) / 128) * 4;
    launch_chained(k_fp8_rows128<XT, E5M2>, dim3(full_grid((quarters + kThreads - 1) / kThreads)), dim3(kThreads), 0,
                   s, x, rows, cols, y, scales);
  }
  note_launches(1);
  return launch_status();
}

mp_status check_common(mp_dtype x_dtype, mp_dtype fp8_dtype, const mp_fp8_meta* d_meta, const float* d_history,
                       int32_t history_len, float margin, int32_t amax_algo) {
  if (!d_meta || !d_history || history_len < 1 || history_len > 65536) return MP_EINVAL;
  if (x_dtype != MP_F32 && x_dtype != MP_F16 && x_dtype != MP_BF16) return MP_EINVAL;
  if (fp8_dtype != MP_E4M3 && fp8_dtype != MP_E5M2) return MP_EINVAL;
  if (amax_algo != 0 && amax_algo != 1) return MP_EINVAL;
  if (!(margin > 0.0f) || !(margin - margin == 0.0f)) return MP_EINVAL;
  if ((reinterpret_cast<uintptr_t>(d_meta) & 15u) || (reinterpret_cast<uintptr_t>(d_history) & 3u)) return MP_EALIGN;
  return MP_OK;
}

template <bool COUNT>
mp_status cast_entry(const void* x, mp_dtype x_dtype, int64_t n, void* y, mp_dtype fp8_dtype, mp_fp8_meta* d_meta,
                     float* d_history, int32_t history_len, float margin, int32_t amax_algo,
                     unsigned long long* saturated, void* stream) {
  if (n < 0 || (n > 0 && (!x || !y))) return MP_EINVAL;
  const mp_status rc = check_common(x_dtype, fp8_dtype, d_meta, d_history, history_len, margin, amax_algo);
  if (rc != MP_OK) return rc;
  if (n > 0 && (!aligned16(x) || !aligned16(y))) return MP_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* yb = static_cast<uint8_t*>(y);
  const bool e5 = fp8_dtype == MP_E5M2;
  switch (x_dtype) {
    case MP_F32:
      return e5 ? launch<XF32, true, COUNT>(x, n, yb, d_meta, d_history, history_len, margin, amax_algo, saturated, s)
                : launch<XF32, false, COUNT>(x, n, yb, d_meta, d_history, history_len, margin, amax_algo, saturated, s);
    case MP_F16:
      return e5 ? launch<XF16, true, COUNT>(x, n, yb, d_meta, d_history, history_len, margin, amax_algo, saturated, s)
                : launch<XF16, false, COUNT>(x, n, yb, d_meta, d_history, history_len, margin, amax_algo, saturated, s);
    default:
      return e5 ? launch<XBF16, true, COUNT>(x, n, yb, d_meta, d_history, history_len, margin, amax_algo, saturated, s)
                : launch<XBF16, false, COUNT>(x, n, yb, d_meta, d_history, history_len, margin, amax_algo, saturated,
                                              s);
  }
}

}  // namespace

uint32_t fp8_wait_failures() {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_wait_failures, sizeof(v)) != cudaSuccess) return 0xFFFFFFFFu;
  return v;
}

}  // namespace mp

extern "C" MP_API mp_status fp8_cast_delayed(const void* x, mp_dtype x_dtype, int64_t n, void* y,
                                             mp_dtype fp8_dtype, mp_fp8_meta* d_meta, float* d_history,
                                             int32_t history_len, float margin, int32_t amax_algo, void* stream) {
  return mp::cast_entry<false>(x, x_dtype, n, y, fp8_dtype, d_meta, d_history, history_len, margin, amax_algo,
                               nullptr, stream);
}

extern "C" MP_API mp_status fp8_cast_delayed_count(const void* x, mp_dtype x_dtype, int64_t n, void* y,
                                                   mp_dtype fp8_dtype, mp_fp8_meta* d_meta, float* d_history,
                                                   int32_t history_len, float margin, int32_t amax_algo,
                                                   unsigned long long* d_saturated, void* stream) {
  if (!d_saturated || (reinterpret_cast<uintptr_t>(d_saturated) & 7u)) return d_saturated ? MP_EALIGN : MP_EINVAL;
  return mp::cast_entry<true>(x, x_dtype, n, y, fp8_dtype, d_meta, d_history, history_len, margin, amax_algo,
                              d_saturated, stream);
}

extern "C" MP_API mp_status fp8_cast_transpose_delayed(const void* x, mp_dtype x_dtype, int64_t rows, int64_t cols,
                                                       void* y, void* y_t, mp_dtype fp8_dtype, mp_fp8_meta* d_meta,
                                                       float* d_history, int32_t history_len, float margin,
                                                       int32_t amax_algo, void* stream) {
  using namespace mp;
  if (rows < 0 || cols < 0) return MP_EINVAL;
  const int64_t n = rows * cols;
  if (n > 0 && (!x || !y || !y_t)) return MP_EINVAL;
  const mp_status rc = check_common(x_dtype, fp8_dtype, d_meta, d_history, history_len, margin, amax_algo);
  if (rc != MP_OK) return rc;
  if (rows % 16 != 0 || cols % 16 != 0) return MP_ESHAPE;
  if (rows >= (1ll << 31) || cols >= (1ll << 31)) return MP_ESHAPE;  // 32-bit tile coordinates
  if (n > 0 && (!aligned16(x) || !aligned16(y) || !aligned16(y_t))) return MP_EALIGN;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t *yb = static_cast<uint8_t*>(y), *ytb = static_cast<uint8_t*>(y_t);
  const bool e5 = fp8_dtype == MP_E5M2;
  switch (x_dtype) {
    case MP_F32:
      return e5 ? launch_t<XF32, true>(x, rows, cols, yb, ytb, d_meta, d_history, history_len, margin, amax_algo, s)
                : launch_t<XF32, false>(x, rows, cols, yb, ytb, d_meta, d_history, history_len, margin, amax_algo, s);
    case MP_F16:
      return e5 ? launch_t<XF16, true>(x, rows, cols, yb, ytb, d_meta, d_history, history_len, margin, amax_algo, s)
                : launch_t<XF16, false>(x, rows, cols, yb, ytb, d_meta, d_history, history_len, margin, amax_algo, s);
    default:
      return e5 ? launch_t<XBF16, true>(x, rows, cols, yb, ytb, d_meta, d_history, history_len, margin, amax_algo, s)
                : launch_t<XBF16, false>(x, rows, cols, yb, ytb, d_meta, d_history, history_len, margin, amax_algo,
                                         s);
  }
}

extern "C" MP_API mp_status fp8_quantize_blockwise(const void* x, mp_dtype x_dtype, int64_t rows, int64_t cols,
                                                   int32_t block_rows, int32_t block_cols, void* y,
                                                   mp_dtype fp8_dtype, float* scales, void* stream) {
  using namespace mp;
  if (rows < 0 || cols < 0) return MP_EINVAL;
  const int64_t n = rows * cols;
  if (n > 0 && (!x || !y || !scales)) return MP_EINVAL;
  if (x_dtype != MP_F32 && x_dtype != MP_F16 && x_dtype != MP_BF16) return MP_EINVAL;
  if (fp8_dtype != MP_E4M3 && fp8_dtype != MP_E5M2) return MP_EINVAL;
  const bool square = block_rows == 128 && block_cols == 128;
  if (!square && !(block_rows == 1 && block_cols == 128)) return MP_ESHAPE;
  if (cols % 16 != 0) return MP_ESHAPE;
  if (rows >= (1ll << 31) || cols >= (1ll << 31)) return MP_ESHAPE;  // 32-bit tile coordinates
  if (n > 0 && (!aligned16(x) || !aligned16(y) || (reinterpret_cast<uintptr_t>(scales) & 3u))) return MP_EALIGN;
  if (n == 0) return MP_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* yb = static_cast<uint8_t*>(y);
  const bool e5 = fp8_dtype == MP_E5M2;
  switch (x_dtype) {
    case MP_F32:
      return e5 ? launch_blockwise<XF32, true>(x, rows, cols, square, yb, scales, s)
                : launch_blockwise<XF32, false>(x, rows, cols, square, yb, scales, s);
    case MP_F16:
      return e5 ? launch_blockwise<XF16, true>(x, rows, cols, square, yb, scales, s)
                : launch_blockwise<XF16, false>(x, rows, cols, square, yb, scales, s);
    default:
      return e5 ? launch_blockwise<XBF16, true>(x, rows, cols, square, yb, scales, s)
                : launch_blockwise<XBF16, false>(x, rows, cols, square, yb, scales, s);
  }
}
