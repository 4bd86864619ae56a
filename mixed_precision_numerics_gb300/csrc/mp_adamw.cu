// mp_adamw.cu — fused mixed-precision optimizer step and loss-scale update.
//
// [MPT-ko] itwiki "혼합 정밀도 학습": "FP32 마스터 가중치" (update the FP32
// master, re-round the 16-bit copy), "손실 스케일링" (unscale by 1/S in FP32;
// skip the step on inf/NaN; dynamic schedule), "FP16 학습 루프" (AdamW).
// [MPT-es] marovi.ai "Mixed Precision Training/es": "La receta de precisión
// mixta", "Escalado dinámico de pérdida".
//
// A step is two stream-ordered kernels over one multi-tensor table:
//   k_check_finite  reads every grad once (2 B/param).  Its last CTA to finish
//                   (atomic ticket, no waiting) publishes found_inf, advances
//                   the step count and beta powers when the step is applied,
//                   and forms the per-step scalars in binary64.
//   k_adamw_update  returns at once when found_inf is set; otherwise streams
//                   g, w, m, v in and w, m, v, w16 out (28 B/param), 8
//                   elements per 16-byte grad vector.
// The table of tensors travels as a __grid_constant__ kernel parameter (up to
// 512 tensors per launch), so no device-side copy or allocation is needed.
#include <new>

#include "mp_device.cuh"
#include "mp_internal.h"

namespace mp {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 8;  // elements per 16-byte grad vector
constexpr int kUnroll = 2;
constexpr int64_t kTile = (int64_t)kThreads * kVec * kUnroll;  // elements per CTA iteration
constexpr int kBigCap = 512;
constexpr int kSmallCap = 8;

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
}

// A 16-bit word pair has an all-ones exponent (inf/NaN) in a half iff adding
// one unit of that half's exponent field carries into its top bit.
template <bool GBF16>
__device__ __forceinline__ uint32_t nonfinite_bits(uint32_t w) {
  constexpr uint32_t em = GBF16 ? 0x7F807F80u : 0x7C007C00u;
  constexpr uint32_t one = GBF16 ? 0x00800080u : 0x04000400u;
  return (w & em) + one;
}

template <int CAP, bool GBF16>
__global__ __launch_bounds__(kThreads) void k_check_finite(const __grid_constant__ Table<CAP> T,
                                                           mp_scaler_state* st,
                                                           const mp_adamw_hparams hp, int finalize) {
  uint32_t bad = 0;
  const int64_t total = T.tile_start[T.count];
  for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
    const int ti = find_tensor(T, tile);
    const TensorDesc& d = T.t[ti];
    const int64_t base = (tile - T.tile_start[ti]) * kTile;
    uint4 g[kUnroll];
    bool full[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t e = base + ((int64_t)u * kThreads + threadIdx.x) * kVec;
      full[u] = e + kVec <= d.n;
      if (full[u]) g[u] = ld_cs(d.g + e);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (full[u]) {
        bad |= nonfinite_bits<GBF16>(g[u].x) | nonfinite_bits<GBF16>(g[u].y) |
               nonfinite_bits<GBF16>(g[u].z) | nonfinite_bits<GBF16>(g[u].w);
      } else {
        const int64_t e = base + ((int64_t)u * kThreads + threadIdx.x) * kVec;
        for (int64_t i = e; i < d.n; ++i) bad |= nonfinite_bits<GBF16>(d.g[i]) & 0x8000u;
      }
    }
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

struct Scalars {
  float inv_scale, step_size, bc2s, decay, omb1, omb2, beta1, beta2, eps;
};

// One element, binary32, in the order of the documented update.
__device__ __forceinline__ void adamw_elem(float graw, float& w, float& m, float& v, const Scalars& s) {
  const float g = __fmul_rn(graw, s.inv_scale);
  const float wd = __fmul_rn(w, s.decay);
  m = __fadd_rn(__fmul_rn(m, s.beta1), __fmul_rn(g, s.omb1));
  v = __fadd_rn(__fmul_rn(v, s.beta2), __fmul_rn(__fmul_rn(g, g), s.omb2));
  const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.bc2s), s.eps);
  w = __fsub_rn(wd, __fmul_rn(s.step_size, __fdiv_rn(m, den)));
}

template <bool BF16>
__device__ __forceinline__ float g_lo(uint32_t w) { return BF16 ? bf16lo(w) : f16lo(w); }
template <bool BF16>
__device__ __forceinline__ float g_hi(uint32_t w) { return BF16 ? bf16hi(w) : f16hi(w); }
template <bool BF16>
__device__ __forceinline__ uint32_t pack16(float lo, float hi) {
  return BF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}

template <int CAP, bool GBF16, bool WBF16>
__global__ __launch_bounds__(kThreads) void k_adamw_update(const __grid_constant__ Table<CAP> T,
                                                           const mp_scaler_state* st, float beta1,
                                                           float beta2, float eps) {
  if (st->found_inf) return;  // skipped step: write nothing
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

  const int64_t total = T.tile_start[T.count];
  for (int64_t tile = blockIdx.x; tile < total; tile += gridDim.x) {
    const int ti = find_tensor(T, tile);
    const TensorDesc& d = T.t[ti];
    const int64_t base = (tile - T.tile_start[ti]) * kTile;
    uint4 g[kUnroll];
    float4 w[kUnroll][2], m[kUnroll][2], v[kUnroll][2];
    bool full[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t e = base + ((int64_t)u * kThreads + threadIdx.x) * kVec;
      full[u] = e + kVec <= d.n;
      if (full[u]) {
        g[u] = ld_cs(d.g + e);
        w[u][0] = ld_cs_f4(d.w + e);
        w[u][1] = ld_cs_f4(d.w + e + 4);
        m[u][0] = ld_cs_f4(d.m + e);
        m[u][1] = ld_cs_f4(d.m + e + 4);
        v[u][0] = ld_cs_f4(d.v + e);
        v[u][1] = ld_cs_f4(d.v + e + 4);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t e = base + ((int64_t)u * kThreads + threadIdx.x) * kVec;
      if (full[u]) {
        float* wf = reinterpret_cast<float*>(&w[u][0]);
        float* mf = reinterpret_cast<float*>(&m[u][0]);
        float* vf = reinterpret_cast<float*>(&v[u][0]);
        const uint32_t gw[4] = {g[u].x, g[u].y, g[u].z, g[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          adamw_elem(g_lo<GBF16>(gw[k]), wf[2 * k], mf[2 * k], vf[2 * k], s);
          adamw_elem(g_hi<GBF16>(gw[k]), wf[2 * k + 1], mf[2 * k + 1], vf[2 * k + 1], s);
        }
        st_cs_f4(d.w + e, w[u][0]);
        st_cs_f4(d.w + e + 4, w[u][1]);
        st_cs_f4(d.m + e, m[u][0]);
        st_cs_f4(d.m + e + 4, m[u][1]);
        st_cs_f4(d.v + e, v[u][0]);
        st_cs_f4(d.v + e + 4, v[u][1]);
        uint4 o;
        o.x = pack16<WBF16>(wf[0], wf[1]);
        o.y = pack16<WBF16>(wf[2], wf[3]);
        o.z = pack16<WBF16>(wf[4], wf[5]);
        o.w = pack16<WBF16>(wf[6], wf[7]);
        st_cs(d.w16 + e, o);
      } else {
        for (int64_t i = e; i < d.n; ++i) {
          float wi = d.w[i], mi = d.m[i], vi = d.v[i];
          adamw_elem(g_lo<GBF16>(d.g[i]), wi, mi, vi, s);
          d.w[i] = wi;
          d.m[i] = mi;
          d.v[i] = vi;
          d.w16[i] = (uint16_t)(pack16<WBF16>(wi, 0.0f) & 0xFFFFu);
        }
      }
    }
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
int occupancy(K kernel) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kThreads, 0) != cudaSuccess || n < 1) n = 1;
  return n;
}

struct Group {
  int first, count;  // indices into the non-empty list
};

template <int CAP>
void fill_table(Table<CAP>& T, const mp_param* const* list, int count) {
  T.count = count;
  T.pad = 0;
  int64_t acc = 0;
  for (int i = 0; i < count; ++i) {
    const mp_param& p = *list[i];
    T.tile_start[i] = acc;
    T.t[i] = TensorDesc{p.master, p.exp_avg, p.exp_avg_sq, static_cast<const uint16_t*>(p.grad),
                        static_cast<uint16_t*>(p.working), p.numel};
    acc += (p.numel + kTile - 1) / kTile;
  }
  T.tile_start[count] = acc;
}

template <int CAP, bool GBF16, bool WBF16>
mp_status launch_group(const mp_param* const* list, int count, bool finalize, bool update,
                       const mp_adamw_hparams& hp, mp_scaler_state* st, cudaStream_t s) {
  Table<CAP> Tl;  // copied by value into the launch's parameter buffer
  fill_table(Tl, list, count);
  const int64_t tiles = Tl.tile_start[count];
  if (!update) {
    static const int occ = occupancy(k_check_finite<CAP, GBF16>);
    k_check_finite<CAP, GBF16><<<grid_for(tiles, occ), kThreads, 0, s>>>(Tl, st, hp, finalize ? 1 : 0);
  } else {
    static const int occ = occupancy(k_adamw_update<CAP, GBF16, WBF16>);
    k_adamw_update<CAP, GBF16, WBF16><<<grid_for(tiles, occ), kThreads, 0, s>>>(Tl, st, hp.beta1, hp.beta2, hp.eps);
  }
  note_launches(1);
  return launch_status();
}

// pass 0: check (only the last group finalises); pass 1: update.
template <bool GBF16, bool WBF16>
mp_status run_pass(int pass, const mp_param* const* list, int n, const mp_adamw_hparams& hp, mp_scaler_state* st,
                   cudaStream_t s) {
  int first = 0;
  do {
    const int count = (n - first) < kBigCap ? (n - first) : kBigCap;
    const bool last = first + count >= n;
    const mp_status rc =
        (count <= kSmallCap)
            ? launch_group<kSmallCap, GBF16, WBF16>(list + first, count, last, pass == 1, hp, st, s)
            : launch_group<kBigCap, GBF16, WBF16>(list + first, count, last, pass == 1, hp, st, s);
    if (rc != MP_OK) return rc;
    first += count;
  } while (first < n);
  return MP_OK;
}

mp_status dispatch_pass(int pass, const mp_param* const* list, int n, mp_dtype gdt, mp_dtype wdt,
                        const mp_adamw_hparams& hp, mp_scaler_state* st, cudaStream_t s) {
  const bool gb = gdt == MP_BF16, wb = wdt == MP_BF16;
  if (!gb && !wb) return run_pass<false, false>(pass, list, n, hp, st, s);
  if (!gb && wb) return run_pass<false, true>(pass, list, n, hp, st, s);
  if (gb && !wb) return run_pass<true, false>(pass, list, n, hp, st, s);
  return run_pass<true, true>(pass, list, n, hp, st, s);
}

bool finite_f(float x) { return x == x && x - x == 0.0f; }

}  // namespace
}  // namespace mp

extern "C" {

}  // extern "C"

namespace mp {
namespace {

// Validates the arguments and lists the non-empty tensors; runs the passes
// in `passes` (bit 0: check, bit 1: update).
mp_status adamw_entry(int passes, const mp_param* params, int32_t n_params, mp_dtype grad_dtype,
                      mp_dtype working_dtype, const mp_adamw_hparams* hp, mp_scaler_state* d_state,
                      void* stream) {
  if (n_params < 0 || (n_params > 0 && !params) || !hp || !d_state) return MP_EINVAL;
  if ((reinterpret_cast<uintptr_t>(d_state) & 7u) != 0) return MP_EALIGN;
  if ((grad_dtype != MP_F16 && grad_dtype != MP_BF16) || (working_dtype != MP_F16 && working_dtype != MP_BF16))
    return MP_EINVAL;
  if (!finite_f(hp->lr) || !finite_f(hp->weight_decay) || !finite_f(hp->eps) || hp->eps < 0.0f ||
      !(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
    return MP_EINVAL;
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
  if (rc == MP_OK && (passes & 1)) rc = dispatch_pass(0, list, n, grad_dtype, working_dtype, *hp, d_state, s);
  if (rc == MP_OK && (passes & 2)) rc = dispatch_pass(1, list, n, grad_dtype, working_dtype, *hp, d_state, s);
  delete[] heap;
  return rc;
}

}  // namespace
}  // namespace mp

extern "C" {

MP_API mp_status mp_adamw_step(const mp_param* params, int32_t n_params, mp_dtype grad_dtype,
                               mp_dtype working_dtype, const mp_adamw_hparams* hp,
                               mp_scaler_state* d_state, void* stream) {
  return mp::adamw_entry(3, params, n_params, grad_dtype, working_dtype, hp, d_state, stream);
}

MP_API mp_status mp_adamw_check(const mp_param* params, int32_t n_params, mp_dtype grad_dtype,
                                const mp_adamw_hparams* hp, mp_scaler_state* d_state, void* stream) {
  return mp::adamw_entry(1, params, n_params, grad_dtype, MP_F16, hp, d_state, stream);
}

MP_API mp_status mp_adamw_apply(const mp_param* params, int32_t n_params, mp_dtype grad_dtype,
                                mp_dtype working_dtype, const mp_adamw_hparams* hp,
                                mp_scaler_state* d_state, void* stream) {
  return mp::adamw_entry(2, params, n_params, grad_dtype, working_dtype, hp, d_state, stream);
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
