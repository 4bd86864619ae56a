/*
 * oracle.c — plain, scalar CPU oracle for the mixed-precision hot path.
 * TEST INFRASTRUCTURE: see oracle.h for what may load it and how it is pinned.
 *
 * Conversions are written from the bit-field definitions of each format:
 * the magnitude is rounded in binary64 (exact for every binary32 input),
 * then the code is assembled from exponent and mantissa fields.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* ---------------------------------------------------------------------------
 * Generic binary format: M explicit mantissa bits, minimum normal exponent
 * emin, exponent bias.  Ties go to the code whose last mantissa bit is 0,
 * which is the even multiple of the quantum at that exponent.
 * ------------------------------------------------------------------------- */
static double round_mag(double a, int M, int emin) {
  if (a == 0.0) return 0.0;
  int k;
  frexp(a, &k);
  int e = k - 1; /* floor(log2 a) */
  if (e < emin) e = emin;
  double q = ldexp(1.0, e - M);
  double n = a / q; /* exact: q is a power of two */
  double fl = floor(n);
  double rem = n - fl;
  if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
  return fl * q;
}

static uint32_t encode_mag(double r, int M, int emin, int bias) {
  if (r == 0.0) return 0;
  int k;
  frexp(r, &k);
  int e = k - 1;
  if (e < emin) return (uint32_t)(r / ldexp(1.0, emin - M)); /* subnormal */
  uint32_t mant = (uint32_t)(r / ldexp(1.0, e - M)) - (1u << M);
  return ((uint32_t)(e + bias) << M) | mant;
}

static double decode_mag(uint32_t field_e, uint32_t mant, int M, int emin, int bias) {
  if (field_e == 0) return ldexp((double)mant, emin - M);
  return ldexp((double)((1u << M) | mant), (int)field_e - bias - M);
}

/* --- FP16 ([MPT-ko] "왜 그냥 FP16으로는 안 되는가"; [MPT-es] "Formatos") ---- */
uint16_t orc_f32_to_f16(float x) {
  if (isnan(x)) return 0x7FFF; /* reading R-NaN16: the canonical NaN's image */
  uint16_t s = signbit(x) ? 0x8000 : 0;
  double a = fabs((double)x);
  if (isinf(x)) return s | 0x7C00;
  double r = round_mag(a, 10, -14);
  if (r > 65504.0) return s | 0x7C00; /* overflow -> inf */
  return s | (uint16_t)encode_mag(r, 10, -14, 15);
}

float orc_f16_to_f32(uint16_t h) {
  uint32_t e = (h >> 10) & 0x1F, m = h & 0x3FF;
  float sgn = (h & 0x8000) ? -1.0f : 1.0f;
  if (e == 31) return m ? copysignf(NAN, sgn) : sgn * INFINITY; /* a NaN keeps its sign */
  return sgn * (float)decode_mag(e, m, 10, -14, 15);
}

/* --- BF16 ([MPT-es] "Formatos de coma flotante") ------------------------- */
uint16_t orc_f32_to_bf16(float x) {
  if (isnan(x)) return 0x7FFF; /* reading R-NaN16: the canonical NaN's image */
  uint16_t s = signbit(x) ? 0x8000 : 0;
  if (isinf(x)) return s | 0x7F80;
  double a = fabs((double)x);
  double r = round_mag(a, 7, -126);
  double maxv = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
  if (r > maxv) return s | 0x7F80;
  return s | (uint16_t)encode_mag(r, 7, -126, 127);
}

float orc_bf16_to_f32(uint16_t h) {
  uint32_t e = (h >> 7) & 0xFF, m = h & 0x7F;
  float sgn = (h & 0x8000) ? -1.0f : 1.0f;
  if (e == 255) return m ? copysignf(NAN, sgn) : sgn * INFINITY; /* a NaN keeps its sign */
  return sgn * (float)decode_mag(e, m, 7, -126, 127);
}

/* --- FP8 ([MPT-ko] "FP8 혼합 정밀도"; [FP8-TE] "FP8이 어려운 이유", "E4M3 vs E5M2")
 * E4M3: bias 7, no infinity, S.1111.111 is NaN, so the largest finite value
 * is 1.75 * 2^8 = 448 (the range [-448, 448] printed on [FP8-TE]).
 * E5M2: bias 15, exponent 11111 is inf/NaN as in IEEE, so the largest finite
 * value is 1.75 * 2^15 = 57344 (derived from the layout; not printed).
 * The cast clips (x_fp8 = clip(x/s, -448, 448) on [FP8-TE]); reading R1:
 * infinities clip too, and NaN maps to S.1111111 (0x7F / 0xFF) with the sign
 * of the NaN (of the input element when the NaN comes from the product). */
static void fp8_params(int fmt, int* M, int* emin, int* bias, double* maxv) {
  if (fmt == ORC_E4M3) { *M = 3; *emin = -6; *bias = 7; *maxv = 448.0; }
  else { *M = 2; *emin = -14; *bias = 15; *maxv = 57344.0; }
}

uint8_t orc_f32_to_fp8_sat(float x, int fmt) {
  int M, emin, bias;
  double maxv;
  fp8_params(fmt, &M, &emin, &bias, &maxv);
  uint8_t s = signbit(x) ? 0x80 : 0;
  if (isnan(x)) return s | 0x7F;
  double a = isinf(x) ? maxv : fabs((double)x);
  double r = round_mag(a, M, emin);
  if (r > maxv) r = maxv;
  return s | (uint8_t)encode_mag(r, M, emin, bias);
}

float orc_fp8_to_f32(uint8_t c, int fmt) {
  int M, emin, bias;
  double maxv;
  fp8_params(fmt, &M, &emin, &bias, &maxv);
  uint32_t e = (c & 0x7F) >> M, m = c & ((1u << M) - 1);
  float sgn = (c & 0x80) ? -1.0f : 1.0f;
  if (fmt == ORC_E4M3) {
    if (e == 15 && m == 7) return copysignf(NAN, sgn);
  } else if (e == 31) {
    return m ? copysignf(NAN, sgn) : sgn * INFINITY;
  }
  return sgn * (float)decode_mag(e, m, M, emin, bias);
}

/* --- E2M1 ([NVFP4] §2.1 "FP4"; layout reading: 1 sign, 2 exponent bits with
 * bias 1, 1 mantissa bit).  Codes 0..7 are the grid in increasing order. */
static const double kE2M1Grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

uint8_t orc_f32_to_e2m1(float x) {
  uint8_t s = signbit(x) ? 0x8 : 0;
  double a = fabs((double)x);
  if (isinf(x)) a = 6.0;
  double r = round_mag(a, 1, 0);
  if (r > 6.0) r = 6.0;
  return s | (uint8_t)encode_mag(r, 1, 0, 1);
}

/* [NVFP4] §2.2 item 4 "확률적 반올림": unbiased rounding of gradients.
 * Reading R14: 16 random bits per element; round away from zero iff
 * floor(frac * 2^16) + r16 >= 2^16, frac the position of |x| between its
 * neighbours on the grid.  P(up) = floor(frac * 2^16) / 2^16. */
uint8_t orc_f32_to_e2m1_sr(float x, uint32_t r16) {
  uint8_t s = signbit(x) ? 0x8 : 0;
  double a = fabs((double)x);
  if (!(a < 6.0)) return s | 7;
  int j = 0;
  while (j < 7 && kE2M1Grid[j + 1] <= a) ++j;
  double lo = kE2M1Grid[j], hi = kE2M1Grid[j + 1];
  double frac = (a - lo) / (hi - lo); /* exact: power-of-two gap */
  uint32_t f16 = (uint32_t)floor(frac * 65536.0);
  int up = (f16 + (r16 & 0xFFFFu)) >= 65536u;
  return s | (uint8_t)(j + up);
}

float orc_e2m1_to_f32(uint8_t c) {
  uint32_t e = (c >> 1) & 3, m = c & 1;
  float sgn = (c & 0x8) ? -1.0f : 1.0f;
  return sgn * (float)decode_mag(e, m, 1, 0, 1);
}

static void fp6_params(int fmt, int* M, int* emin, int* bias, double* maxv) {
  if (fmt == ORC_E2M3) { *M = 3; *emin = 0; *bias = 1; *maxv = 7.5; }   /* 1.875 * 2^2 */
  else { *M = 2; *emin = -2; *bias = 3; *maxv = 28.0; }                  /* 1.75 * 2^4 */
}

uint8_t orc_f32_to_fp6(float x, int fmt) {
  int M, emin, bias;
  double maxv;
  fp6_params(fmt, &M, &emin, &bias, &maxv);
  uint8_t s = signbit(x) ? 0x20 : 0;
  double a = isinf(x) ? maxv : fabs((double)x);
  double r = round_mag(a, M, emin);
  if (r > maxv) r = maxv;
  return s | (uint8_t)encode_mag(r, M, emin, bias);
}

float orc_fp6_to_f32(uint8_t c, int fmt) {
  int M, emin, bias;
  double maxv;
  fp6_params(fmt, &M, &emin, &bias, &maxv);
  uint32_t e = (c & 0x1F) >> M, m = c & ((1u << M) - 1);
  float sgn = (c & 0x20) ? -1.0f : 1.0f;
  return sgn * (float)decode_mag(e, m, M, emin, bias);
}

static float load_f32(const void* x, int fmt, int64_t i) {
  switch (fmt) {
    case ORC_F32: return ((const float*)x)[i];
    case ORC_F16: return orc_f16_to_f32(((const uint16_t*)x)[i]);
    case ORC_BF16: return orc_bf16_to_f32(((const uint16_t*)x)[i]);
    case ORC_E4M3: return orc_fp8_to_f32(((const uint8_t*)x)[i], ORC_E4M3);
    case ORC_E5M2: return orc_fp8_to_f32(((const uint8_t*)x)[i], ORC_E5M2);
    case ORC_E2M3: return orc_fp6_to_f32(((const uint8_t*)x)[i], ORC_E2M3);
    case ORC_E3M2: return orc_fp6_to_f32(((const uint8_t*)x)[i], ORC_E3M2);
    default: return orc_e2m1_to_f32(((const uint8_t*)x)[i]);
  }
}

void orc_convert(const void* in, int in_fmt, int64_t n, void* out, int out_fmt) {
  for (int64_t i = 0; i < n; ++i) {
    float v = load_f32(in, in_fmt, i);
    switch (out_fmt) {
      case ORC_F32: ((float*)out)[i] = v; break;
      case ORC_F16: ((uint16_t*)out)[i] = orc_f32_to_f16(v); break;
      case ORC_BF16: ((uint16_t*)out)[i] = orc_f32_to_bf16(v); break;
      case ORC_E4M3: ((uint8_t*)out)[i] = orc_f32_to_fp8_sat(v, ORC_E4M3); break;
      case ORC_E5M2: ((uint8_t*)out)[i] = orc_f32_to_fp8_sat(v, ORC_E5M2); break;
      case ORC_E2M3: ((uint8_t*)out)[i] = orc_f32_to_fp6(v, ORC_E2M3); break;
      case ORC_E3M2: ((uint8_t*)out)[i] = orc_f32_to_fp6(v, ORC_E3M2); break;
      default: ((uint8_t*)out)[i] = orc_f32_to_e2m1(v); break;
    }
  }
}

/* max |x|: absolute values compared as numbers, NaN absorbing. */
float orc_amax(const void* x, int fmt, int64_t n) {
  float m = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float v = fabsf(load_f32(x, fmt, i));
    if (isnan(v)) return u2f(0x7FC00000u);
    if (v > m) m = v;
  }
  return m;
}

/* ---------------------------------------------------------------------------
 * Philox4x32-10 (J. Salmon, M. Moraes, R. Dror, D. Shaw, "Parallel Random
 * Numbers: As Easy as 1, 2, 3", SC'11).  Each round multiplies counter words
 * 0 and 2 by the two round multipliers, swaps the halves of the products
 * across the pairs and mixes in the other counter words and the key; the key
 * is advanced by the two Weyl constants between rounds.
 * ------------------------------------------------------------------------- */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t p0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t p1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
    uint32_t n1 = (uint32_t)p1;
    uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
    uint32_t n3 = (uint32_t)p0;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Reading R15: key = (seed lo, seed hi); one Philox call per 8 consecutive
 * elements, counter = (i/8 lo, i/8 hi, 0, 0); element i takes 16-bit half
 * (i mod 2) of output word (i/2 mod 4). */
uint32_t orc_sr_bits(uint64_t seed, uint64_t i) {
  uint64_t g = i >> 3;
  uint32_t ctr[4] = {(uint32_t)g, (uint32_t)(g >> 32), 0u, 0u};
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t out[4];
  orc_philox4x32_10(ctr, key, out);
  return (out[(i >> 1) & 3] >> (16 * (i & 1))) & 0xFFFFu;
}

void orc_e2m1_sr_array(const float* y, int64_t n, uint64_t seed, uint64_t i0, uint8_t* out) {
  for (int64_t k = 0; k < n; ++k) out[k] = orc_f32_to_e2m1_sr(y[k], orc_sr_bits(seed, i0 + (uint64_t)k));
}

void orc_e2m1_sr_bits_array(const float* y, const uint16_t* r16, int64_t n, uint8_t* out) {
  for (int64_t k = 0; k < n; ++k) out[k] = orc_f32_to_e2m1_sr(y[k], r16[k]);
}

/* ---------------------------------------------------------------------------
 * [NVFP4] §2.2 item 2 "랜덤 하다마드 변환": a 16x16 random Hadamard transform
 * spreads outliers before FP4 quantisation.  Reading R16: H16 is the
 * Sylvester matrix, H[i][j] = (-1)^popcount(i & j); the random part is a
 * diagonal of signs; the 1/4 normalisation makes the transform orthogonal.
 * The product with H16 is taken by the fast Walsh-Hadamard butterfly (stages
 * of span 1, 2, 4, 8), whose additions are the ones evaluated here.
 * ------------------------------------------------------------------------- */
void orc_rht16_tile(const float in[16], uint16_t sign_mask, float out[16]) {
  float v[16];
  for (int j = 0; j < 16; ++j) v[j] = ((sign_mask >> j) & 1) ? -in[j] : in[j];
  for (int h = 1; h < 16; h <<= 1) {
    for (int i = 0; i < 16; ++i) {
      if (i & h) continue;
      float a = v[i], b = v[i + h];
      v[i] = a + b;
      v[i + h] = a - b;
    }
  }
  for (int j = 0; j < 16; ++j) out[j] = v[j] * 0.25f;
}

int orc_rht16(const uint16_t* x_bf16, int64_t rows, int64_t cols, uint16_t sign_mask, void* y,
              int y_fmt) {
  if (rows < 0 || cols < 0 || cols % 16) return -1;
  float in[16], out[16];
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t c = 0; c < cols; c += 16) {
      int64_t base = r * cols + c;
      for (int j = 0; j < 16; ++j) in[j] = orc_bf16_to_f32(x_bf16[base + j]);
      orc_rht16_tile(in, sign_mask, out);
      for (int j = 0; j < 16; ++j) {
        if (y_fmt == ORC_F32) ((float*)y)[base + j] = out[j];
        else ((uint16_t*)y)[base + j] = orc_f32_to_bf16(out[j]);
      }
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------------
 * Mixed-precision optimizer step.
 * [MPT-ko] "FP32 마스터 가중치": the update is applied to the FP32 master and
 *   the 16-bit copy is re-rounded from it: w32 <- w32 - eta*fp32(g16),
 *   w16 = round16(w32).
 * [MPT-ko] "손실 스케일링" / [MPT-es] "Escalado de pérdida": g = (1/S) *
 *   fp32(grad of S*L), applied in FP32 before the update.
 * [MPT-ko] "FP16 학습 루프": the optimizer is AdamW (lr 1e-3); its moments
 *   are FP32 ([MPT-es] "Operaciones que permanecen en FP32").  Reading R3:
 *   decoupled weight decay, bias-corrected moments, eps added after the
 *   square root; per-step scalars formed once in binary64 and rounded to
 *   binary32; per-element arithmetic in binary32 in the order written.
 * [MPT-ko] "손실 스케일링" bullets / [MPT-es] "Escalado dinámico de pérdida":
 *   an inf/NaN grad skips the step.  Reading R4: a skipped step writes
 *   nothing and does not advance the step count or the beta powers.
 * ------------------------------------------------------------------------- */
int orc_nonfinite_any(const uint16_t* g, int fmt, int64_t n) {
  uint16_t em = (fmt == ORC_F16) ? 0x7C00 : 0x7F80; /* all-ones exponent */
  for (int64_t i = 0; i < n; ++i)
    if ((g[i] & em) == em) return 1;
  return 0;
}

void orc_adamw_begin(const orc_adamw_hp* hp, orc_scaler_state* st, int found_inf,
                     orc_step_scalars* out) {
  st->found_inf = found_inf ? 1 : 0;
  double b1 = (double)hp->beta1, b2 = (double)hp->beta2;
  double b1p = st->beta1_pow, b2p = st->beta2_pow;
  if (!found_inf) {
    b1p *= b1;
    b2p *= b2;
    st->beta1_pow = b1p;
    st->beta2_pow = b2p;
    st->step += 1;
  }
  double bc1 = 1.0 - b1p, bc2 = 1.0 - b2p;
  out->inv_scale = (float)(1.0 / (double)st->scale);
  out->step_size = (float)((double)hp->lr / bc1);
  out->bc2_sqrt = (float)sqrt(bc2);
  out->decay = (float)(1.0 - (double)hp->lr * (double)hp->weight_decay);
  out->omb1 = (float)(1.0 - b1);
  out->omb2 = (float)(1.0 - b2);
  out->beta1 = hp->beta1;
  out->beta2 = hp->beta2;
  out->eps = hp->eps;
  out->clip = 1.0f;
}

void orc_adamw_apply(const orc_step_scalars* s, float* w, float* m, float* v, const uint16_t* g,
                     int g_fmt, uint16_t* w16, int w16_fmt, int64_t n) {
  for (int64_t i = 0; i < n; ++i) {
    float gf = (g_fmt == ORC_F16) ? orc_f16_to_f32(g[i]) : orc_bf16_to_f32(g[i]);
    float gu = (gf * s->inv_scale) * s->clip;       /* unscale, then clip */
    float wi = w[i] * s->decay;                      /* decoupled decay */
    float mi = m[i] * s->beta1 + gu * s->omb1;       /* first moment */
    float vi = v[i] * s->beta2 + (gu * gu) * s->omb2; /* second moment */
    float den = sqrtf(vi) / s->bc2_sqrt + s->eps;
    wi = wi - s->step_size * (mi / den);
    w[i] = wi;
    m[i] = mi;
    v[i] = vi;
    w16[i] = (w16_fmt == ORC_F16) ? orc_f32_to_f16(wi) : orc_f32_to_bf16(wi);
  }
}

/* Sum of squares of one tensor's unscaled grads, the quantity whose square
 * root over all tensors is the L2 norm that clip_grad_norm_ compares with
 * max_norm ([MPT-ko] "FP16 학습 루프": unscale_ then clip_grad_norm_;
 * [MPT-es] "Operaciones que permanecen en FP32": norms are long reductions
 * kept in high precision).  The unscaled grad is the binary32 value the update
 * uses, gu = fp32(grad) * inv_scale; its square is exact in binary64 (24-bit
 * significands), and the squares are added one after another in element
 * order in binary64. */
double orc_grad_sumsq(const uint16_t* g, int g_fmt, int64_t n, float inv_scale) {
  double total = 0.0;
  for (int64_t i = 0; i < n; ++i) {
    float gf = (g_fmt == ORC_F16) ? orc_f16_to_f32(g[i]) : orc_bf16_to_f32(g[i]);
    double gu = (double)(gf * inv_scale);
    total = total + gu * gu;
  }
  return total;
}

float orc_clip_coef(double norm, float max_norm) {
  double c = (double)max_norm / (norm + 1e-6);
  if (c > 1.0) c = 1.0;
  return (float)c;
}

/* [MPT-ko] "손실 스케일링": start large, on inf/NaN skip and shrink (x0.5),
 * after N clean steps grow (x2); GradScaler defaults 65536 / 2 / 0.5 / 2000.
 * [MPT-es] "Escalado dinámico de pérdida": the same schedule.  Reading R7:
 * growth applies only when the grown scale is finite; no floor on S. */
void orc_loss_scale_update(orc_scaler_state* st, const orc_scaler_cfg* cfg) {
  if (!cfg->enabled) return;
  if (st->found_inf) {
    st->scale = st->scale * cfg->backoff_factor;
    st->growth_tracker = 0;
    st->skipped += 1;
    return;
  }
  int32_t t = st->growth_tracker + 1;
  if (t >= cfg->growth_interval) {
    float grown = st->scale * cfg->growth_factor;
    if (isfinite(grown)) st->scale = grown;
    t = 0;
  }
  st->growth_tracker = t;
}

/* ---------------------------------------------------------------------------
 * FP8 delayed scaling ([FP8-TE] "Delayed Scaling 동작 원리"): each step's
 * amax goes into an amax_history ring; the next scale is
 * fp8_max / (margin * max(history)); the tensor is cast with the scale in
 * force, so the tensor is read once.  Reading R8: the scale multiplies
 * (y = sat(fp32(x) * scale)).  Reading R9: history starts at zero, scale at
 * 1; a history max that is zero or not finite, or a new scale that is not a
 * finite positive number, leaves the scale unchanged.
 * ------------------------------------------------------------------------- */
uint8_t orc_fp8_cast_one(float x, float scale, int fmt) {
  const float p = x * scale;
  /* reading R1: a NaN product (a NaN input, or an infinity times a zero
   * multiplier) takes the input element's sign; the sign of a NaN an
   * operation creates is not fixed across machines */
  if (isnan(p)) return (signbit(x) ? 0x80 : 0) | 0x7F;
  return orc_f32_to_fp8_sat(p, fmt);
}

void orc_fp8_cast_array(const void* x, int x_fmt, int64_t n, uint8_t* y, int fmt, float scale) {
  for (int64_t i = 0; i < n; ++i) y[i] = orc_fp8_cast_one(load_f32(x, x_fmt, i), scale, fmt);
}

int64_t orc_fp8_saturation_count(const void* x, int x_fmt, int64_t n, int fmt, float scale) {
  int M, emin, bias;
  double maxv;
  fp8_params(fmt, &M, &emin, &bias, &maxv);
  int64_t c = 0;
  for (int64_t i = 0; i < n; ++i) {
    float p = load_f32(x, x_fmt, i) * scale;
    if (fabs((double)p) > maxv) ++c; /* false for NaN */
  }
  return c;
}

void orc_fp8_history_update(orc_fp8_meta* meta, float* history, int32_t hist_len, float margin,
                            float amax, int fmt, int amax_algo) {
  meta->amax = amax;
  /* reading R9b: the ring slot is pos taken modulo the ring length */
  int32_t pos = ((meta->pos % hist_len) + hist_len) % hist_len;
  history[pos] = amax;
  meta->pos = (pos + 1) % hist_len;
  float hmax = 0.0f;
  if (amax_algo == 1) {
    hmax = amax > 0.0f || isnan(amax) ? amax : 0.0f;
  } else {
    for (int32_t i = 0; i < hist_len; ++i) {
      if (isnan(history[i])) { hmax = history[i]; break; }
      if (history[i] > hmax) hmax = history[i];
    }
  }
  if (!(isfinite(hmax) && hmax > 0.0f)) return;
  float denom = margin * hmax;
  if (!(isfinite(denom) && denom > 0.0f)) return;
  float fp8_max = (fmt == ORC_E4M3) ? 448.0f : 57344.0f;
  float ns = fp8_max / denom;
  if (!(isfinite(ns) && ns > 0.0f)) return;
  meta->scale = ns;
  meta->scale_inv = 1.0f / ns;
}

void orc_fp8_cast_delayed(const void* x, int x_fmt, int64_t n, uint8_t* y, int fmt,
                          orc_fp8_meta* meta, float* history, int32_t hist_len, float margin,
                          int amax_algo) {
  orc_fp8_cast_array(x, x_fmt, n, y, fmt, meta->scale);
  float amax = orc_amax(x, x_fmt, n);
  orc_fp8_history_update(meta, history, hist_len, margin, amax, fmt, amax_algo);
}

void orc_transpose_u8(const uint8_t* y, int64_t rows, int64_t cols, uint8_t* y_t) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) y_t[c * rows + r] = y[r * cols + c];
}

void orc_fp8_quantize_blockwise(const void* x, int x_fmt, int64_t rows, int64_t cols, int32_t block_rows,
                                int32_t block_cols, int fmt, uint8_t* y, float* scales) {
  float fp8_max = (fmt == ORC_E4M3) ? 448.0f : 57344.0f;
  int64_t nbr = (rows + block_rows - 1) / block_rows, nbc = (cols + block_cols - 1) / block_cols;
  for (int64_t br = 0; br < nbr; ++br) {
    for (int64_t bc = 0; bc < nbc; ++bc) {
      int64_t r1 = (br + 1) * block_rows < rows ? (br + 1) * block_rows : rows;
      int64_t c1 = (bc + 1) * block_cols < cols ? (bc + 1) * block_cols : cols;
      float amax = 0.0f;
      int nan = 0;
      for (int64_t r = br * block_rows; r < r1; ++r)
        for (int64_t c = bc * block_cols; c < c1; ++c) {
          float a = fabsf(load_f32(x, x_fmt, r * cols + c));
          if (isnan(a)) nan = 1;
          else if (a > amax) amax = a;
        }
      if (nan) amax = u2f(0x7FC00000u);
      /* a block holding a NaN stores the quiet NaN 0x7FC00000 as its scale */
      scales[br * nbc + bc] = nan ? amax : amax / fp8_max;
      float rr = (isfinite(amax) && amax > 0.0f) ? fp8_max / amax : 0.0f;
      for (int64_t r = br * block_rows; r < r1; ++r)
        for (int64_t c = bc * block_cols; c < c1; ++c)
          y[r * cols + c] = orc_fp8_cast_one(load_f32(x, x_fmt, r * cols + c), rr, fmt);
    }
  }
}

void orc_mx_quantize(const void* x, int x_fmt, int64_t rows, int64_t cols, int elem_fmt, uint8_t* codes,
                     uint8_t* scales, uint16_t* dequant) {
  int emax = elem_fmt == ORC_E4M3 ? 8 : elem_fmt == ORC_E5M2 ? 15 : elem_fmt == ORC_E3M2 ? 4 : 2;
  int64_t nb = cols / 32;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      int64_t base = r * cols + b * 32;
      float amax = 0.0f;
      int bad = 0;
      for (int j = 0; j < 32; ++j) {
        float a = fabsf(load_f32(x, x_fmt, base + j));
        if (!isfinite(a)) bad = 1;
        else if (a > amax) amax = a;
      }
      int e = -127;
      if (!bad && amax > 0.0f) {
        int k;
        frexp((double)amax, &k); /* amax = f * 2^k, f in [0.5, 1) */
        e = (k - 1) - emax;
        if (e < -127) e = -127;
        if (e > 127) e = 127;
      }
      scales[r * nb + b] = bad ? 0xFF : (uint8_t)(e + 127);
      float mul = (float)ldexp(1.0, -e); /* 2^-e, exact in binary32 for e in [-127, 127] */
      double dq = ldexp(1.0, e);
      for (int j = 0; j < 32; ++j) {
        int64_t i = base + j;
        uint8_t q = 0;
        if (!bad) {
          float y = load_f32(x, x_fmt, i) * mul;
          q = elem_fmt == ORC_E2M1   ? orc_f32_to_e2m1(y)
              : elem_fmt == ORC_E2M3 || elem_fmt == ORC_E3M2 ? orc_f32_to_fp6(y, elem_fmt)
                                                              : orc_f32_to_fp8_sat(y, elem_fmt);
        }
        if (elem_fmt == ORC_E2M1) {
          uint8_t* byte = &codes[i >> 1];
          if (i & 1) *byte = (uint8_t)((*byte & 0x0F) | (q << 4));
          else *byte = (uint8_t)((*byte & 0xF0) | q);
        } else {
          codes[i] = q;
        }
        if (dequant) {
          float v = bad ? 0.0f : load_f32(&q, elem_fmt, 0) * (float)dq;
          dequant[i] = orc_f32_to_bf16(v);
        }
      }
    }
  }
}

/* ---------------------------------------------------------------------------
 * NVFP4 ([NVFP4] §2.1 "NVFP4 포맷의 특징", §2.2): 16-element blocks, one E4M3
 * block scale per block under one FP32 tensor scale (two-level scaling);
 * 16x16 blocks for weights (§2.2 item 3), random Hadamard transform on
 * weight-gradient inputs (item 2), stochastic rounding for gradients
 * (item 4).  Readings: tensor scale amax / (6 * 448) (R-TS); block scale
 * E4M3(RNE((bamax / 6) / s_t)); elements multiplied by the reciprocal of the
 * decoded block scale times s_t (R13); RNE ties to the even code; codes
 * packed two per byte, even element in the low nibble (R18); block scales
 * row-major.  Reading R11/R12: a non-finite amax, or s_t == 0, gives all-zero
 * codes, scales and dequantised values.
 * ------------------------------------------------------------------------- */
int orc_nvfp4_prepare(const uint16_t* x_bf16, int64_t rows, int64_t cols, int apply_rht,
                      uint16_t sign_mask, float* xprime) {
  if (rows < 0 || cols < 0 || cols % 16) return -1;
  if (apply_rht) return orc_rht16(x_bf16, rows, cols, sign_mask, xprime, ORC_F32);
  for (int64_t i = 0; i < rows * cols; ++i) xprime[i] = orc_bf16_to_f32(x_bf16[i]);
  return 0;
}

float orc_nvfp4_tensor_scale(float amax, int32_t* nonfinite) {
  if (!isfinite(amax)) {
    *nonfinite = 1;
    return amax;
  }
  *nonfinite = 0;
  return amax / 2688.0f; /* 6 * 448 */
}

void orc_nvfp4_block_scale(float bamax, float s_t, uint8_t* code, float* d, float* r) {
  float q = (bamax / 6.0f) / s_t;
  uint8_t c = orc_f32_to_fp8_sat(q, ORC_E4M3);
  float dd = orc_fp8_to_f32(c, ORC_E4M3) * s_t;
  float rr = 0.0f;
  if (dd != 0.0f) {
    float inv = 1.0f / dd;
    if (isfinite(inv)) rr = inv;
  }
  *code = c;
  *d = dd;
  *r = rr;
}

static void encode_element(float xp, float r, float d, int stochastic, uint64_t seed,
                           uint64_t flat, uint8_t* codes, uint16_t* dequant) {
  float y = xp * r;
  uint8_t q = stochastic ? orc_f32_to_e2m1_sr(y, orc_sr_bits(seed, flat)) : orc_f32_to_e2m1(y);
  uint8_t* byte = &codes[flat >> 1];
  if (flat & 1) *byte = (uint8_t)((*byte & 0x0F) | (q << 4));
  else *byte = (uint8_t)((*byte & 0xF0) | q);
  if (dequant) dequant[flat] = orc_f32_to_bf16(orc_e2m1_to_f32(q) * d);
}

void orc_nvfp4_encode_rows(const float* xprime, int64_t row0, int64_t nrows, int64_t cols,
                           int block_2d, int stochastic, uint64_t seed, float s_t,
                           int32_t nonfinite, uint8_t* codes, uint8_t* scales,
                           uint16_t* dequant) {
  int64_t nb = cols / 16;
  if (nonfinite || s_t == 0.0f) {
    memset(codes + row0 * cols / 2, 0, (size_t)(nrows * cols / 2));
    if (block_2d) memset(scales + (row0 / 16) * nb, 0, (size_t)((nrows / 16) * nb));
    else memset(scales + row0 * nb, 0, (size_t)(nrows * nb));
    if (dequant) memset(dequant + row0 * cols, 0, (size_t)(nrows * cols) * 2);
    return;
  }
  if (!block_2d) {
    for (int64_t r = 0; r < nrows; ++r) {
      for (int64_t b = 0; b < nb; ++b) {
        const float* blk = xprime + r * cols + b * 16;
        float bamax = 0.0f;
        for (int j = 0; j < 16; ++j)
          if (fabsf(blk[j]) > bamax) bamax = fabsf(blk[j]);
        uint8_t sc;
        float d, rr;
        orc_nvfp4_block_scale(bamax, s_t, &sc, &d, &rr);
        scales[(row0 + r) * nb + b] = sc;
        for (int j = 0; j < 16; ++j) {
          uint64_t flat = (uint64_t)((row0 + r) * cols + b * 16 + j);
          encode_element(blk[j], rr, d, stochastic, seed, flat, codes, dequant);
        }
      }
    }
    return;
  }
  for (int64_t tr = 0; tr < nrows / 16; ++tr) {
    for (int64_t b = 0; b < nb; ++b) {
      float bamax = 0.0f;
      for (int i = 0; i < 16; ++i)
        for (int j = 0; j < 16; ++j) {
          float a = fabsf(xprime[(tr * 16 + i) * cols + b * 16 + j]);
          if (a > bamax) bamax = a;
        }
      uint8_t sc;
      float d, rr;
      orc_nvfp4_block_scale(bamax, s_t, &sc, &d, &rr);
      scales[(row0 / 16 + tr) * nb + b] = sc;
      for (int i = 0; i < 16; ++i)
        for (int j = 0; j < 16; ++j) {
          int64_t lr = tr * 16 + i;
          uint64_t flat = (uint64_t)((row0 + lr) * cols + b * 16 + j);
          encode_element(xprime[lr * cols + b * 16 + j], rr, d, stochastic, seed, flat, codes,
                         dequant);
        }
    }
  }
}

int orc_nvfp4_quantize(const uint16_t* x_bf16, int64_t rows, int64_t cols, int block_2d,
                       int stochastic, uint64_t seed, int apply_rht, uint16_t sign_mask,
                       uint8_t* codes, uint8_t* scales, float* tensor_scale, int32_t* nonfinite,
                       uint16_t* dequant) {
  if (rows < 0 || cols < 0 || cols % 16 || (block_2d && rows % 16)) return -1;
  int64_t n = rows * cols;
  float* xp = (float*)malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
  if (!xp) return -2;
  orc_nvfp4_prepare(x_bf16, rows, cols, apply_rht, sign_mask, xp);
  float amax = orc_amax(xp, ORC_F32, n);
  int32_t nf = 0;
  float s_t = orc_nvfp4_tensor_scale(amax, &nf);
  *tensor_scale = s_t;
  *nonfinite = nf;
  orc_nvfp4_encode_rows(xp, 0, rows, cols, block_2d, stochastic, seed, s_t, nf, codes, scales,
                        dequant);
  free(xp);
  return 0;
}
