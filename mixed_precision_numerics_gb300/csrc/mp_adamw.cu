// mp_adamw.cu — fused mixed-precision optimizer step and loss-scale update.
//
// [MPT-ko] itwiki "혼합 정밀도 학습": "FP32 마스터 가중치" (update the FP32
// master, re-round the 16-bit copy), "손실 스케일링" (unscale by 1/S in FP32;
// skip the step on inf/NaN; dynamic schedule), "FP16 학습 루프" (AdamW).
// [MPT-es] marovi.ai "Mixed Precision Training/es": "La receta de precisión
// mixta", "Escalado dinámico de pérdida".
//
// A step is two stream-ordered kernels over one multi-tensor table:
//   k_check_finite  reads every grad once (2 B/param), 8 x 16 B in flight per
//                   thread.  Its last CTA to finish (atomic ticket, no
//                   waiting) publishes found_inf, advances the step count and
//                   beta powers when the step is applied, and forms the
//                   per-step scalars in binary64.
//   k_adamw_update  returns at once when found_inf is set; otherwise streams
//                   g, w, m, v in and w, m, v, w16 out (28 B/param).  One
//                   producer warp moves 2816-element chunks of g, w, m, v into
//                   a 3-stage shared-memory ring with bulk asynchronous copies
//                   (cp.async.bulk, completion counted on an mbarrier); eleven
//                   consumer warps compute from shared memory and store
//                   straight to global memory, then hand the stage back.  One
//                   CTA per SM keeps about 115 KB of loads in flight; in
//                   measurements on the full Llama-3-8B list, larger or
//                   smaller amounts in flight, and power-of-two chunk sizes,
//                   were slower.
// With gradient-norm clipping the check pass is k_check_finite_clip, which
// also writes one binary32 sum of the squared unscaled grads per 16384-element
// tile, and k_clip_finish folds those sums in binary64 (32 one-warp CTAs and a
// last-CTA fold) into the norm and the clip factor the update multiplies by.
// The table of tensors travels as a __grid_constant__ kernel parameter (up to
// 512 tensors per launch), so no device-side copy or allocation is needed.
#include <new>

#include "mp_device.cuh"
#include "mp_internal.h"

namespace mp {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8;  // elements per 16-byte grad vector
constexpr int kUnroll = 8;
constexpr int64_t kTile = (int64_t)kThreads * kVec * kUnroll;  // elements per check-pass CTA iteration
constexpr int kBigCap = 512;
constexpr int kSmallCap = 8;

// Update pass: chunk of kChunk elements per pipeline stage, kStages stages,
// kConsumerWarps warps computing, one more warp issuing the copies.
constexpr int kChunk = 2816;
constexpr int kStages = 3;
constexpr int kConsumerWarps = 11;
constexpr int kUpdateThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageBytes = kChunk * 14;  // g 2 + w 4 + m 4 + v 4 bytes per element
constexpr int kUpdateSmem = kStages * kStageBytes + 2 * kStages * 8;
static_assert(kChunk == kConsumerWarps * 32 * 8, "each consumer thread owns 8 elements of a chunk");

struct TensorDesc {
  float* w;
  float* m;
  float* v;
  const uint16_t* g;
  uint16_t* w16;
  int64_t n;
};

template <int CAP>
struct Table {
  int32_t count;
  int32_t pad;
  int64_t tile_start[CAP + 1];  // prefix sums of per-tensor tile counts
  TensorDesc t[CAP];
};

// Largest i with tile_start[i] <= tile (every listed tensor is non-empty).
template <int CAP>
__device__ __forceinline__ int find_tensor(const Table<CAP>& T, int64_t tile) {
  int lo = 0, hi = T.count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (T.tile_start[mid] <= tile) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Step scalars stored in mp_scaler_state::internal_scalars.
enum { S_INV_SCALE = 0, S_STEP_SIZE, S_BC2_SQRT, S_DECAY, S_OMB1, S_OMB2 };

// Runs on one thread of the last CTA of the check pass.
__device__ void finish_check(mp_scaler_state* st, const mp_adamw_hparams hp, bool found) {
  st->found_inf = found ? 1 : 0;
  const double b1 = (double)hp.beta1, b2 = (double)hp.beta2;
  double b1p = st->beta1_pow, b2p = st->beta2_pow;
  if (!found) {
    b1p = __dmul_rn(b1p, b1);
    b2p = __dmul_rn(b2p, b2);
    st->beta1_pow = b1p;
    st->beta2_pow = b2p;
    st->step += 1;
  }
  const double bc1 = __dsub_rn(1.0, b1p), bc2 = __dsub_rn(1.0, b2p);
  float* s = st->internal_scalars;
  s[S_INV_SCALE] = __double2float_rn(__ddiv_rn(1.0, (double)st->scale));
  s[S_STEP_SIZE] = __double2float_rn(__ddiv_rn((double)hp.lr, bc1));
  s[S_BC2_SQRT] = __double2float_rn(__dsqrt_rn(bc2));
  s[S_DECAY] = __double2float_rn(__dsub_rn(1.0, __dmul_rn((double)hp.lr, (double)hp.weight_decay)));
  s[S_OMB1] = __double2float_rn(__dsub_rn(1.0, b1));
  s[S_OMB2] = __double2float_rn(__dsub_rn(1.0, b2));
  st->grad_norm = -1.0f;  // replaced by k_clip_finish when clipping
  st->clip_coef = 1.0f;
}

// A 16-bit word pair has an all-ones exponent (inf/NaN) in a half iff adding
// one unit of that half's exponent field carries into its top bit.
template <bool GBF16>
__device__ __forceinline__ uint32_t nonfinite_bits(uint32_t w) {
  constexpr uint32_t em = GBF16 ? 0x7F807F80u : 0x7C007C00u;
  constexpr uint32_t one = GBF16 ? 0x00800080u : 0x04000400u;
  return (w & em) + one;
}

template <bool BF16>
__device__ __forceinline__ float g_lo(uint32_t w) { return BF16 ? bf16lo(w) : f16lo(w); }
template <bool BF16>
__device__ __forceinline__ float g_hi(uint32_t w) { return BF16 ? bf16hi(w) : f16hi(w); }

constexpr int kClipCtasPerSm = 4;  // register cap of the clipping check pass: 4 x 32 KB tiles in flight per SM

// Thread 0: fold the 8 warp sums of a tile as w[i] += w[i + h], h = 4, 2, 1.
__device__ __forceinline__ float fold_warp_sums(const float* ws) {
  float w[kThreads / 32];
#pragma unroll
  for (int i = 0; i < kThreads / 32; ++i) w[i] = ws[i];
#pragma unroll
  for (int h = kThreads / 64; h >= 1; h >>= 1)
#pragma unroll
    for (int i = 0; i < h; ++i) w[i] = __fadd_rn(w[i], w[i + h]);
  return w[0];
}

// With CLIP, every tile of kTile elements also yields the binary32 sum of
// g*g, g = fp32(grad) * inv_scale, in one fixed order: lane t sums its 8
// vectors (u = 0..7) element by element; each warp folds its 32 lane sums by
// v[l] += v[l ^ h], h = 16..1; the 8 warp sums fold as w[i] += w[i + h],
// h = 4, 2, 1.  The sum goes to tile_sums[tile_base + tile].  The warp sums of
// a tile are folded one iteration later, after the next tile's loads are in
// flight, so the CTA's one barrier per tile never holds back a load.
template <int CAP, bool GBF16, bool CLIP>
__device__ __forceinline__ void check_body(const Table<CAP>& T, mp_scaler_state* st, const mp_adamw_hparams& hp,
                                           int finalize, float* __restrict__ tile_sums, int64_t tile_base) {
  __shared__ float warp_sum[2][kThreads / 32];
  uint32_t bad = 0;
  const float inv_scale = CLIP ? __double2float_rn(__ddiv_rn(1.0, (double)st->scale)) : 0.0f;
  const int64_t total = T.tile_start[T.count];
  int par = 0;
  int64_t prev = -1;  // tile whose warp sums wait in warp_sum[par ^ 1]
  for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
    const int ti = find_tensor(T, tile);
    const TensorDesc& d = T.t[ti];
    const int64_t base = (tile - T.tile_start[ti]) * kTile;
    const bool whole = base + kTile <= d.n;  // every vector of the tile is in the tensor
    uint4 g[kUnroll];
    if (whole) {
      const uint4* gp = reinterpret_cast<const uint4*>(d.g + base) + threadIdx.x;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) g[u] = __ldcs(gp + u * kThreads);
    } else {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t e = base + ((int64_t)u * kThreads + threadIdx.x) * kVec;
        if (e + kVec <= d.n) g[u] = ld_cs(d.g + e);
      }
    }
    if (CLIP) {
      // Every warp wrote its sums of tile `prev` before issuing this tile's
      // loads; thread 0 reads them before it reaches the next barrier, so the
      // slot is free again when it is rewritten two tiles later.
      __syncthreads();
      if (threadIdx.x == 0 && prev >= 0) tile_sums[tile_base + prev] = fold_warp_sums(warp_sum[par ^ 1]);
    }
    float lane = 0.0f;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t e = base + ((int64_t)u * kThreads + threadIdx.x) * kVec;
      if (whole || e + kVec <= d.n) {
        bad |= nonfinite_bits<GBF16>(g[u].x) | nonfinite_bits<GBF16>(g[u].y) |
               nonfinite_bits<GBF16>(g[u].z) | nonfinite_bits<GBF16>(g[u].w);
        if (CLIP) {
          const uint32_t gw[4] = {g[u].x, g[u].y, g[u].z, g[u].w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float a = __fmul_rn(g_lo<GBF16>(gw[k]), inv_scale);
            lane = __fadd_rn(lane, __fmul_rn(a, a));
            const float b = __fmul_rn(g_hi<GBF16>(gw[k]), inv_scale);
            lane = __fadd_rn(lane, __fmul_rn(b, b));
          }
        }
      } else {
        for (int64_t i = e; i < d.n; ++i) {
          const uint32_t h = d.g[i];
          bad |= nonfinite_bits<GBF16>(h) & 0x8000u;
          if (CLIP) {
            const float a = __fmul_rn(g_lo<GBF16>(h), inv_scale);
            lane = __fadd_rn(lane, __fmul_rn(a, a));
          }
        }
      }
    }
    if (CLIP) {
#pragma unroll
      for (int h = 16; h >= 1; h >>= 1) lane = __fadd_rn(lane, __shfl_xor_sync(0xFFFFFFFFu, lane, h));
      if ((threadIdx.x & 31) == 0) warp_sum[par][threadIdx.x >> 5] = lane;
      prev = tile;
      par ^= 1;
    }
  }
  if (CLIP) {
    __syncthreads();
    if (threadIdx.x == 0 && prev >= 0) tile_sums[tile_base + prev] = fold_warp_sums(warp_sum[par ^ 1]);
  }
  const int any = __syncthreads_or((bad & 0x80008000u) != 0);
  if (threadIdx.x == 0) {
    if (any) atomicOr(&st->internal_found, 1u);
    if (finalize) {
      __threadfence();
      const uint32_t ticket = atomicAdd(&st->internal_ticket, 1u);
      if (ticket == gridDim.x - 1) {
        __threadfence();
        const uint32_t found = atomicExch(&st->internal_found, 0u);
        st->internal_ticket = 0;
        finish_check(st, hp, found != 0);
      }
    }
  }
}

template <int CAP, bool GBF16>
__global__ __launch_bounds__(kThreads) void k_check_finite(const __grid_constant__ Table<CAP> T, mp_scaler_state* st,
                                                           const mp_adamw_hparams hp, int finalize) {
  check_body<CAP, GBF16, false>(T, st, hp, finalize, nullptr, 0);
}

template <int CAP, bool GBF16>
__global__ __launch_bounds__(kThreads, kClipCtasPerSm) void k_check_finite_clip(
    const __grid_constant__ Table<CAP> T, mp_scaler_state* st, const mp_adamw_hparams hp, int finalize,
    float* __restrict__ tile_sums, int64_t tile_base) {
  check_body<CAP, GBF16, true>(T, st, hp, finalize, tile_sums, tile_base);
}

// Folds the tile sums in binary64 in one fixed order: lane t of kFoldLanes
// adds tiles t, t + kFoldLanes, t + 2 kFoldLanes, ... in that order; each warp
// folds its lanes by v[l] += v[l ^ h], h = 16..1; the warp sums fold as
// w[i] += w[i + h], h = 16..1; then norm = sqrt(total) and
// clip = min(1, max_norm / (norm + 1e-6)).  One warp per CTA, one CTA per
// warp of lanes, so the binary64 additions spread over 32 SMs; loads are
// batched kFoldBatch deep and added in lane order.  The last CTA (atomic
// ticket on st->internal_ticket, which the check pass leaves at zero; no
// waiting) folds the warp sums.
constexpr int kFoldLanes = 1024;
constexpr int kFoldCtas = kFoldLanes / 32;
constexpr int kFoldBatch = 32;
constexpr size_t kFoldBytes = kFoldCtas * sizeof(double);  // warp sums at the start of the workspace
__global__ __launch_bounds__(32) void k_clip_finish(const float* __restrict__ tile_sums, int64_t ntiles,
                                                    double* __restrict__ warp_sums, mp_scaler_state* st,
                                                    float max_norm) {
  const int64_t t = (int64_t)blockIdx.x * 32 + threadIdx.x;
  double lane = 0.0;
  for (int64_t i0 = t; i0 < ntiles; i0 += (int64_t)kFoldLanes * kFoldBatch) {
    float v[kFoldBatch];
#pragma unroll
    for (int j = 0; j < kFoldBatch; ++j) {
      const int64_t i = i0 + (int64_t)j * kFoldLanes;
      v[j] = i < ntiles ? __ldcg(tile_sums + i) : 0.0f;
    }
#pragma unroll
    for (int j = 0; j < kFoldBatch; ++j)
      if (i0 + (int64_t)j * kFoldLanes < ntiles) lane = __dadd_rn(lane, (double)v[j]);
  }
#pragma unroll
  for (int h = 16; h >= 1; h >>= 1) lane = __dadd_rn(lane, __shfl_xor_sync(0xFFFFFFFFu, lane, h));
  if (threadIdx.x != 0) return;
  warp_sums[blockIdx.x] = lane;
  __threadfence();
  if (atomicAdd(&st->internal_ticket, 1u) != gridDim.x - 1) return;
  __threadfence();
  st->internal_ticket = 0;
  double w[kFoldCtas];
#pragma unroll
  for (int i = 0; i < kFoldCtas; ++i) w[i] = __ldcg(warp_sums + i);
#pragma unroll
  for (int h = kFoldCtas / 2; h >= 1; h >>= 1)
#pragma unroll
    for (int i = 0; i < h; ++i) w[i] = __dadd_rn(w[i], w[i + h]);
  const double norm = __dsqrt_rn(w[0]);
  double c = __ddiv_rn((double)max_norm, __dadd_rn(norm, 1e-6));
  if (c > 1.0) c = 1.0;
  st->grad_norm = __double2float_rn(norm);
  st->clip_coef = __double2float_rn(c);
}

struct Scalars {
  float inv_scale, step_size, bc2s, decay, omb1, omb2, beta1, beta2, eps, clip;
};

// One element, binary32, in the order of the documented update.
__device__ __forceinline__ void adamw_elem(float graw, float& w, float& m, float& v, const Scalars& s) {
  const float g = __fmul_rn(__fmul_rn(graw, s.inv_scale), s.clip);  // unscale, then clip
  const float wd = __fmul_rn(w, s.decay);
  m = __fadd_rn(__fmul_rn(m, s.beta1), __fmul_rn(g, s.omb1));
  v = __fadd_rn(__fmul_rn(v, s.beta2), __fmul_rn(__fmul_rn(g, g), s.omb2));
  const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.bc2s), s.eps);
  w = __fsub_rn(wd, __fmul_rn(s.step_size, __fdiv_rn(m, den)));
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  return BF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}

// Elements of a chunk owned by consumer thread t: two runs of four,
// [4t, 4t + 4) and [kChunk/2 + 4t, kChunk/2 + 4t + 4): 16-byte shared-memory
// reads without bank conflicts and 16-byte coalesced global stores.
template <bool GBF16, bool WBF16>
__device__ __forceinline__ void update_run4(const unsigned char* stage, int e, const TensorDesc& d, int64_t off,
                                            const Scalars& s) {
  const uint2 gq = *reinterpret_cast<const uint2*>(stage + 2 * e);
  float4 w = *reinterpret_cast<const float4*>(stage + kChunk * 2 + 4 * e);
  float4 m = *reinterpret_cast<const float4*>(stage + kChunk * 6 + 4 * e);
  float4 v = *reinterpret_cast<const float4*>(stage + kChunk * 10 + 4 * e);
  adamw_elem(g_lo<GBF16>(gq.x), w.x, m.x, v.x, s);
  adamw_elem(g_hi<GBF16>(gq.x), w.y, m.y, v.y, s);
  adamw_elem(g_lo<GBF16>(gq.y), w.z, m.z, v.z, s);
  adamw_elem(g_hi<GBF16>(gq.y), w.w, m.w, v.w, s);
  const int64_t i = off + e;
  st_cs_f4(d.w + i, w);
  st_cs_f4(d.m + i, m);
  st_cs_f4(d.v + i, v);
  __stcs(reinterpret_cast<uint2*>(d.w16 + i), make_uint2(pack16<WBF16>(w.x, w.y), pack16<WBF16>(w.z, w.w)));
}

template <int CAP, bool GBF16, bool WBF16>
__global__ __launch_bounds__(kUpdateThreads) void k_adamw_update(const __grid_constant__ Table<CAP> T,
                                                                 mp_scaler_state* st, float beta1, float beta2,
                                                                 float eps) {
  if (st->found_inf) return;  // skipped step: write nothing
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t total = T.tile_start[T.count];

  if (warp == kConsumerWarps) {
    // Producer: one lane issues the bulk copies of each chunk into its stage.
    if (lane != 0) return;
    const uint64_t policy = policy_evict_first();
    int issued = 0;
    bool ok = true;
    for (int64_t c = blockIdx.x; c < total; c += gridDim.x, ++issued) {
      const int sidx = issued % kStages;
      if (!mbar_wait_bounded(&empty[sidx], ((issued / kStages) & 1) ^ 1)) {
        ok = false;
        break;
      }
      const int ti = find_tensor(T, c);
      const TensorDesc& d = T.t[ti];
      const int64_t off = (c - T.tile_start[ti]) * kChunk;
      const int64_t len = d.n - off < kChunk ? d.n - off : kChunk;
      const uint32_t nb = (uint32_t)(len & ~7ll);  // whole 8-element groups go by bulk copy
      unsigned char* stage = smem + sidx * kStageBytes;
      mbar_arrive_expect_tx(&full[sidx], nb * 14u);
      if (nb) {
        bulk_g2s(stage, d.g + off, nb * 2u, &full[sidx], policy);
        bulk_g2s(stage + kChunk * 2, d.w + off, nb * 4u, &full[sidx], policy);
        bulk_g2s(stage + kChunk * 6, d.m + off, nb * 4u, &full[sidx], policy);
        bulk_g2s(stage + kChunk * 10, d.v + off, nb * 4u, &full[sidx], policy);
      }
    }
    if (!ok) {
      atomicOr(reinterpret_cast<uint32_t*>(&st->error_flags), 1u);
      // Let the copies already issued land before the block's shared memory goes away.
      for (int k = issued - kStages < 0 ? 0 : issued - kStages; k < issued; ++k)
        (void)mbar_wait_bounded(&full[k % kStages], (k / kStages) & 1);
    }
    return;
  }

  // Consumers.
  Scalars s;
  s.inv_scale = st->internal_scalars[S_INV_SCALE];
  s.step_size = st->internal_scalars[S_STEP_SIZE];
  s.bc2s = st->internal_scalars[S_BC2_SQRT];
  s.decay = st->internal_scalars[S_DECAY];
  s.omb1 = st->internal_scalars[S_OMB1];
  s.omb2 = st->internal_scalars[S_OMB2];
  s.beta1 = beta1;
  s.beta2 = beta2;
  s.eps = eps;
  s.clip = st->clip_coef;
  const int t = threadIdx.x;
  int it = 0;
  for (int64_t c = blockIdx.x; c < total; c += gridDim.x, ++it) {
    const int sidx = it % kStages;
    if (!mbar_wait_bounded(&full[sidx], (it / kStages) & 1)) {
      atomicOr(reinterpret_cast<uint32_t*>(&st->error_flags), 2u);
      return;
    }
    const int ti = find_tensor(T, c);
    const TensorDesc& d = T.t[ti];
    const int64_t off = (c - T.tile_start[ti]) * kChunk;
    const int64_t len = d.n - off < kChunk ? d.n - off : kChunk;
    const int nb = (int)(len & ~7ll);
    const unsigned char* stage = smem + sidx * kStageBytes;
    const int e0 = 4 * t, e1 = kChunk / 2 + 4 * t;
    if (e0 + 4 <= nb) update_run4<GBF16, WBF16>(stage, e0, d, off, s);
    if (e1 + 4 <= nb) update_run4<GBF16, WBF16>(stage, e1, d, off, s);
    if (t < len - nb) {  // the last (< 8) elements of a tensor, straight from global memory
      const int64_t i = off + nb + t;
      float wi = d.w[i], mi = d.m[i], vi = d.v[i];
      adamw_elem(g_lo<GBF16>(d.g[i]), wi, mi, vi, s);
      d.w[i] = wi;
      d.m[i] = mi;
      d.v[i] = vi;
      d.w16[i] = (uint16_t)(pack16<WBF16>(wi, 0.0f) & 0xFFFFu);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[sidx]);
  }
}

__global__ void k_loss_scale_update(mp_scaler_state* st, const mp_scaler_cfg cfg) {
  if (st->found_inf) {
    st->scale = __fmul_rn(st->scale, cfg.backoff_factor);
    st->growth_tracker = 0;
    st->skipped += 1;
    return;
  }
  int32_t t = st->growth_tracker + 1;
  if (t >= cfg.growth_interval) {
    const float grown = __fmul_rn(st->scale, cfg.growth_factor);
    if (isfinite(grown)) st->scale = grown;
    t = 0;
  }
  st->growth_tracker = t;
}

template <typename K>
int occupancy(K kernel, int threads, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) n = 1;
  return n;
}

struct Group {
  int first, count;  // indices into the non-empty list
};

template <int CAP>
void fill_table(Table<CAP>& T, const mp_param* const* list, int count, int64_t tile) {
  T.count = count;
  T.pad = 0;
  int64_t acc = 0;
  for (int i = 0; i < count; ++i) {
    const mp_param& p = *list[i];
    T.tile_start[i] = acc;
    T.t[i] = TensorDesc{p.master, p.exp_avg, p.exp_avg_sq, static_cast<const uint16_t*>(p.grad),
                        static_cast<uint16_t*>(p.working), p.numel};
    acc += (p.numel + tile - 1) / tile;
  }
  T.tile_start[count] = acc;
}

struct ClipArgs {
  bool on;
  double* warp_sums;  // kFoldCtas binary64 partial sums (start of the workspace)
  float* tile_sums;   // one binary32 sum per tile (after them)
  float max_norm;
};

template <int CAP, bool GBF16, bool WBF16>
mp_status launch_group(const mp_param* const* list, int count, bool finalize, bool update,
                       const mp_adamw_hparams& hp, mp_scaler_state* st, const ClipArgs& clip, int64_t tile_base,
                       int64_t* tiles_out, cudaStream_t s) {
  Table<CAP> Tl;  // copied by value into the launch's parameter buffer
  if (!update) {
    fill_table(Tl, list, count, kTile);
    *tiles_out = Tl.tile_start[count];
    if (clip.on) {
      static const int occ = occupancy(k_check_finite_clip<CAP, GBF16>, kThreads, 0);
      k_check_finite_clip<CAP, GBF16><<<grid_for(Tl.tile_start[count], occ), kThreads, 0, s>>>(
          Tl, st, hp, finalize ? 1 : 0, clip.tile_sums, tile_base);
    } else {
      static const int occ = occupancy(k_check_finite<CAP, GBF16>, kThreads, 0);
      k_check_finite<CAP, GBF16><<<grid_for(Tl.tile_start[count], occ), kThreads, 0, s>>>(Tl, st, hp,
                                                                                           finalize ? 1 : 0);
    }
  } else {
    fill_table(Tl, list, count, kChunk);
    static std::atomic<uint64_t> smem_done{0};
    if (!smem_opt_in(k_adamw_update<CAP, GBF16, WBF16>, kUpdateSmem, smem_done)) return MP_ECUDA;
    static const int occ = occupancy(k_adamw_update<CAP, GBF16, WBF16>, kUpdateThreads, kUpdateSmem);
    k_adamw_update<CAP, GBF16, WBF16><<<grid_for(Tl.tile_start[count], occ), kUpdateThreads, kUpdateSmem, s>>>(
        Tl, st, hp.beta1, hp.beta2, hp.eps);
  }
  note_launches(1);
  return launch_status();
}

// pass 0: check (only the last group finalises; then the norm when clipping);
// pass 1: update.
template <bool GBF16, bool WBF16>
mp_status run_pass(int pass, const mp_param* const* list, int n, const mp_adamw_hparams& hp, mp_scaler_state* st,
                   const ClipArgs& clip, cudaStream_t s) {
  int first = 0;
  int64_t tile_base = 0;
  do {
    const int count = (n - first) < kBigCap ? (n - first) : kBigCap;
    const bool last = first + count >= n;
    int64_t tiles = 0;
    const mp_status rc =
        (count <= kSmallCap)
            ? launch_group<kSmallCap, GBF16, WBF16>(list + first, count, last, pass == 1, hp, st, clip, tile_base,
                                                    &tiles, s)
            : launch_group<kBigCap, GBF16, WBF16>(list + first, count, last, pass == 1, hp, st, clip, tile_base,
                                                  &tiles, s);
    if (rc != MP_OK) return rc;
    tile_base += tiles;
    first += count;
  } while (first < n);
  if (pass == 0 && clip.on) {
    k_clip_finish<<<kFoldCtas, 32, 0, s>>>(clip.tile_sums, tile_base, clip.warp_sums, st, clip.max_norm);
    note_launches(1);
    return launch_status();
  }
  return MP_OK;
}

mp_status dispatch_pass(int pass, const mp_param* const* list, int n, mp_dtype gdt, mp_dtype wdt,
                        const mp_adamw_hparams& hp, mp_scaler_state* st, const ClipArgs& clip, cudaStream_t s) {
  const bool gb = gdt == MP_BF16, wb = wdt == MP_BF16;
  if (!gb && !wb) return run_pass<false, false>(pass, list, n, hp, st, clip, s);
  if (!gb && wb) return run_pass<false, true>(pass, list, n, hp, st, clip, s);
  if (gb && !wb) return run_pass<true, false>(pass, list, n, hp, st, clip, s);
  return run_pass<true, true>(pass, list, n, hp, st, clip, s);
}

int64_t clip_tiles(const mp_param* params, int32_t n_params) {
  int64_t t = 0;
  for (int i = 0; i < n_params; ++i)
    if (params[i].numel > 0) t += (params[i].numel + kTile - 1) / kTile;
  return t;
}

size_t clip_workspace_bytes(const mp_param* params, int32_t n_params) {
  return kFoldBytes + (size_t)clip_tiles(params, n_params) * sizeof(float);
}

bool finite_f(float x) { return x == x && x - x == 0.0f; }

}  // namespace
}  // namespace mp

namespace mp {
namespace {

// Validates the arguments and lists the non-empty tensors; runs the passes
// in `passes` (bit 0: check, bit 1: update).
mp_status adamw_entry(int passes, const mp_param* params, int32_t n_params, mp_dtype grad_dtype,
                      mp_dtype working_dtype, const mp_adamw_hparams* hp, mp_scaler_state* d_state,
                      void* d_workspace, size_t workspace_bytes, void* stream) {
  if (n_params < 0 || (n_params > 0 && !params) || !hp || !d_state) return MP_EINVAL;
  if ((reinterpret_cast<uintptr_t>(d_state) & 7u) != 0) return MP_EALIGN;
  if ((grad_dtype != MP_F16 && grad_dtype != MP_BF16) || (working_dtype != MP_F16 && working_dtype != MP_BF16))
    return MP_EINVAL;
  if (!finite_f(hp->lr) || !finite_f(hp->weight_decay) || !finite_f(hp->eps) || hp->eps < 0.0f ||
      !(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f) ||
      !finite_f(hp->max_grad_norm) || hp->max_grad_norm < 0.0f)
    return MP_EINVAL;
  unsigned char* ws = static_cast<unsigned char*>(d_workspace);
  ClipArgs clip{(passes & 1) && hp->max_grad_norm > 0.0f, reinterpret_cast<double*>(ws),
                reinterpret_cast<float*>(ws + kFoldBytes), hp->max_grad_norm};
  if (clip.on) {
    if (!d_workspace || workspace_bytes < clip_workspace_bytes(params, n_params)) return MP_EWORKSPACE;
    if (reinterpret_cast<uintptr_t>(d_workspace) & 7u) return MP_EALIGN;
  }
  const mp_param* small[64];
  const mp_param** heap = nullptr;
  const mp_param** list = small;
  if (n_params > 64) {
    heap = new (std::nothrow) const mp_param*[n_params];
    if (!heap) return MP_EINVAL;
    list = heap;
  }
  int n = 0;
  mp_status rc = MP_OK;
  for (int i = 0; i < n_params && rc == MP_OK; ++i) {
    const mp_param& p = params[i];
    if (p.numel < 0) rc = MP_EINVAL;
    else if (p.numel == 0) continue;
    else if (!p.master || !p.exp_avg || !p.exp_avg_sq || !p.grad || !p.working) rc = MP_EINVAL;
    else if (!aligned16(p.master) || !aligned16(p.exp_avg) || !aligned16(p.exp_avg_sq) || !aligned16(p.grad) ||
             !aligned16(p.working))
      rc = MP_EALIGN;
    else list[n++] = &p;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (rc == MP_OK && (passes & 1)) rc = dispatch_pass(0, list, n, grad_dtype, working_dtype, *hp, d_state, clip, s);
  if (rc == MP_OK && (passes & 2)) rc = dispatch_pass(1, list, n, grad_dtype, working_dtype, *hp, d_state, clip, s);
  delete[] heap;
  return rc;
}

}  // namespace
}  // namespace mp

extern "C" {

MP_API size_t mp_adamw_workspace_size(const mp_param* params, int32_t n_params) {
  if (n_params > 0 && !params) return 0;
  return mp::clip_workspace_bytes(params, n_params < 0 ? 0 : n_params);
}

MP_API mp_status mp_adamw_step(const mp_param* params, int32_t n_params, mp_dtype grad_dtype,
                               mp_dtype working_dtype, const mp_adamw_hparams* hp,
                               mp_scaler_state* d_state, void* d_workspace, size_t workspace_bytes,
                               void* stream) {
  return mp::adamw_entry(3, params, n_params, grad_dtype, working_dtype, hp, d_state, d_workspace,
                         workspace_bytes, stream);
}

MP_API mp_status mp_adamw_check(const mp_param* params, int32_t n_params, mp_dtype grad_dtype,
                                const mp_adamw_hparams* hp, mp_scaler_state* d_state, void* d_workspace,
                                size_t workspace_bytes, void* stream) {
  return mp::adamw_entry(1, params, n_params, grad_dtype, MP_F16, hp, d_state, d_workspace, workspace_bytes,
                         stream);
}

MP_API mp_status mp_adamw_apply(const mp_param* params, int32_t n_params, mp_dtype grad_dtype,
                                mp_dtype working_dtype, const mp_adamw_hparams* hp,
                                mp_scaler_state* d_state, void* stream) {
  return mp::adamw_entry(2, params, n_params, grad_dtype, working_dtype, hp, d_state, nullptr, 0, stream);
}

MP_API mp_status loss_scale_update(mp_scaler_state* d_state, const mp_scaler_cfg* cfg, void* stream) {
  using namespace mp;
  if (!d_state || !cfg) return MP_EINVAL;
  if ((reinterpret_cast<uintptr_t>(d_state) & 7u) != 0) return MP_EALIGN;
  if (cfg->growth_interval < 1 || !finite_f(cfg->growth_factor) || !finite_f(cfg->backoff_factor) ||
      cfg->growth_factor <= 0.0f || cfg->backoff_factor <= 0.0f)
    return MP_EINVAL;
  if (!cfg->enabled) return MP_OK;
  k_loss_scale_update<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(d_state, *cfg);
  note_launches(1);
  return launch_status();
}

}  // extern "C"
