/*
 * synth.h — seeded, counter-based synthetic input generator.
 *
 * Every value is a pure function of (seed, stream, index), so any element of
 * any workload tensor can be regenerated on its own, on the host or on the
 * device, with the same bits.  Both builds use only IEEE-754 binary32 add,
 * subtract, multiply, divide and square root (no contraction, no library
 * transcendental), which is what makes host and device agree bit for bit:
 * the host object is built with -ffp-contract=off, and on the device every
 * operation goes through the explicit _rn intrinsics below.
 *
 * This module holds input generation only.  It shares no code with the
 * kernels under test or with the oracle: both sides receive the same bytes.
 *
 * Distributions:
 *   normal     Box-Muller on two 24-bit uniforms, with a logarithm and a
 *              cosine written here as plain series (tails reach ~5.9 sigma).
 *   bernoulli  p compared against a 32-bit hash word.
 *   student-t  nu = 3: Z / sqrt(chi2_3 / 3), chi2_3 a sum of 3 squared normals.
 * Quantisation to 16-bit storage types is round-toward-zero (truncation), a
 * generator convention that is deliberately not any cast under test.
 */
#ifndef SYNTH_H
#define SYNTH_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_FN __host__ __device__ static inline
#else
#define SYNTH_FN static inline
#endif

#if defined(__CUDA_ARCH__)
#define S_ADD(a, b) __fadd_rn((a), (b))
#define S_SUB(a, b) __fsub_rn((a), (b))
#define S_MUL(a, b) __fmul_rn((a), (b))
#define S_DIV(a, b) __fdiv_rn((a), (b))
#define S_SQRT(a) __fsqrt_rn(a)
#define S_F2U(f) __float_as_uint(f)
#define S_U2F(u) __uint_as_float(u)
#else
#include <math.h>
#include <string.h>
#define S_ADD(a, b) ((float)(a) + (float)(b))
#define S_SUB(a, b) ((float)(a) - (float)(b))
#define S_MUL(a, b) ((float)(a) * (float)(b))
#define S_DIV(a, b) ((float)(a) / (float)(b))
#define S_SQRT(a) sqrtf(a)
SYNTH_FN uint32_t s_f2u_host(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
SYNTH_FN float s_u2f_host(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
#define S_F2U(f) s_f2u_host(f)
#define S_U2F(u) s_u2f_host(u)
#endif

/* ---- integer hashing ---------------------------------------------------- */

SYNTH_FN uint64_t synth_mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ULL;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBULL;
  z ^= z >> 31;
  return z;
}

/* One 64-bit word per (seed, stream, index). */
SYNTH_FN uint64_t synth_hash(uint64_t seed, uint64_t stream, uint64_t index) {
  uint64_t k = synth_mix64(seed * 0x9E3779B97F4A7C15ULL + stream * 0xC2B2AE3D27D4EB4FULL + 0x165667B19E3779F9ULL);
  return synth_mix64(k ^ (index * 0xD1B54A32D192ED03ULL + 0x632BE59BD9B4E019ULL));
}

/* Sub-streams used inside one recipe (kept apart from user stream numbers). */
#define SYNTH_SUB_OUTLIER 0x4F55544CULL
#define SYNTH_SUB_T1 0x54310000ULL
#define SYNTH_SUB_T2 0x54320000ULL
#define SYNTH_SUB_T3 0x54330000ULL

/* ---- uniform, log, cos --------------------------------------------------- */

/* 24-bit uniform in (0,1): (k + 0.5) * 2^-24, exact in binary32. */
SYNTH_FN float synth_u24(uint32_t k24) {
  return S_MUL(S_ADD((float)(k24 & 0xFFFFFFu), 0.5f), 5.9604644775390625e-08f);
}

/* Natural log for u in (0, 1], atanh series on the reduced mantissa. */
SYNTH_FN float synth_logf(float u) {
  uint32_t b = S_F2U(u);
  int e = (int)(b >> 23) - 127;
  float m = S_U2F((b & 0x7FFFFFu) | 0x3F800000u); /* [1,2) */
  if (m > 1.41421353816986083984375f) {
    m = S_MUL(m, 0.5f);
    e += 1;
  }
  float s = S_DIV(S_SUB(m, 1.0f), S_ADD(m, 1.0f)); /* |s| < 0.1716 */
  float z = S_MUL(s, s);
  float p = 0.0909090936183929443359375f;               /* 1/11 */
  p = S_ADD(S_MUL(p, z), 0.111111111938953399658203125f); /* 1/9 */
  p = S_ADD(S_MUL(p, z), 0.142857149243354797363281250f); /* 1/7 */
  p = S_ADD(S_MUL(p, z), 0.2000000029802322387695312f);  /* 1/5 */
  p = S_ADD(S_MUL(p, z), 0.3333333432674407958984375f);  /* 1/3 */
  p = S_ADD(S_MUL(p, z), 1.0f);
  float lnm = S_MUL(S_MUL(2.0f, s), p);
  return S_ADD(S_MUL((float)e, 0.693147182464599609375f), lnm);
}

/* sin and cos of phi in [0, pi/2) by Taylor polynomials. */
SYNTH_FN float synth_sin_q(float x) {
  float z = S_MUL(x, x);
  float p = -7.6471637318198164759e-13f;       /* -1/15! */
  p = S_ADD(S_MUL(p, z), 1.6059043836821614599e-10f);  /* 1/13! */
  p = S_ADD(S_MUL(p, z), -2.5052108385441718775e-08f); /* -1/11! */
  p = S_ADD(S_MUL(p, z), 2.7557319223985890653e-06f);  /* 1/9! */
  p = S_ADD(S_MUL(p, z), -1.9841269841269841270e-04f); /* -1/7! */
  p = S_ADD(S_MUL(p, z), 8.3333333333333333333e-03f);  /* 1/5! */
  p = S_ADD(S_MUL(p, z), -1.6666666666666666667e-01f); /* -1/3! */
  p = S_ADD(S_MUL(p, z), 1.0f);
  return S_MUL(x, p);
}
SYNTH_FN float synth_cos_q(float x) {
  float z = S_MUL(x, x);
  float p = 4.7794773323873852974e-14f;        /* 1/16! */
  p = S_ADD(S_MUL(p, z), -1.1470745597729724714e-11f); /* -1/14! */
  p = S_ADD(S_MUL(p, z), 2.0876756987868098979e-09f);  /* 1/12! */
  p = S_ADD(S_MUL(p, z), -2.7557319223985890653e-07f); /* -1/10! */
  p = S_ADD(S_MUL(p, z), 2.4801587301587301587e-05f);  /* 1/8! */
  p = S_ADD(S_MUL(p, z), -1.3888888888888888889e-03f); /* -1/6! */
  p = S_ADD(S_MUL(p, z), 4.1666666666666666667e-02f);  /* 1/4! */
  p = S_ADD(S_MUL(p, z), -0.5f);
  p = S_ADD(S_MUL(p, z), 1.0f);
  return p;
}

/* cos(2*pi*v) for v in [0,1), by quadrant. */
SYNTH_FN float synth_cos2pi(float v) {
  float t = S_MUL(v, 4.0f);
  int q = (int)t; /* 0..3, exact truncation of a value in [0,4) */
  float r = S_SUB(t, (float)q);
  float phi = S_MUL(r, 1.57079637050628662109375f);
  switch (q & 3) {
    case 0: return synth_cos_q(phi);
    case 1: return -synth_sin_q(phi);
    case 2: return -synth_cos_q(phi);
    default: return synth_sin_q(phi);
  }
}

/* ---- distributions -------------------------------------------------------- */

SYNTH_FN float synth_normal(uint64_t seed, uint64_t stream, uint64_t index) {
  uint64_t h = synth_hash(seed, stream, index);
  float u1 = synth_u24((uint32_t)(h >> 40));
  float u2 = synth_u24((uint32_t)(h >> 16));
  float r = S_SQRT(S_MUL(-2.0f, synth_logf(u1)));
  return S_MUL(r, synth_cos2pi(u2));
}

/* 1 with probability thr / 2^32. */
SYNTH_FN int synth_bernoulli(uint64_t seed, uint64_t stream, uint64_t index, uint32_t thr) {
  uint64_t h = synth_hash(seed, stream ^ SYNTH_SUB_OUTLIER, index);
  return (uint32_t)(h >> 32) < thr;
}

/* Student-t with 3 degrees of freedom. */
SYNTH_FN float synth_student_t3(uint64_t seed, uint64_t stream, uint64_t index) {
  float z = synth_normal(seed, stream ^ SYNTH_SUB_T1, index);
  float a = synth_normal(seed, stream ^ SYNTH_SUB_T2, index);
  float b = synth_normal(seed, stream ^ SYNTH_SUB_T3, index);
  float c = synth_normal(seed, stream ^ (SYNTH_SUB_T3 + 1), index);
  float chi = S_ADD(S_ADD(S_MUL(a, a), S_MUL(b, b)), S_MUL(c, c));
  return S_DIV(z, S_SQRT(S_DIV(chi, 3.0f)));
}

/* ---- recipe ---------------------------------------------------------------- */

enum { SYNTH_F32 = 0, SYNTH_F16 = 1, SYNTH_BF16 = 2 };
enum { SYNTH_OUTLIER_NONE = 0, SYNTH_OUTLIER_SCALE = 1, SYNTH_OUTLIER_T3 = 2 };

/* value(i) = sigma * Z_i; at positions drawn with probability
 * outlier_thr / 2^32 either value *= mult (SCALE) or value = sigma * mult * T_i
 * (T3).  Callers set outlier_thr = floor(p * 2^32).  Outlier positions come
 * from (seed, outlier_stream, index), so a sequence of tensors that shares an
 * outlier_stream shares its outlier positions. */
typedef struct {
  uint64_t seed;
  uint64_t stream;
  uint64_t outlier_stream;
  float sigma;
  float outlier_mult;
  uint32_t outlier_thr;
  int32_t outlier_kind;
} synth_recipe;

SYNTH_FN float synth_value(const synth_recipe* r, uint64_t index) {
  float v = S_MUL(r->sigma, synth_normal(r->seed, r->stream, index));
  if (r->outlier_kind != SYNTH_OUTLIER_NONE &&
      synth_bernoulli(r->seed, r->outlier_stream, index, r->outlier_thr)) {
    if (r->outlier_kind == SYNTH_OUTLIER_SCALE)
      v = S_MUL(v, r->outlier_mult);
    else
      v = S_MUL(S_MUL(r->sigma, r->outlier_mult), synth_student_t3(r->seed, r->stream, index));
  }
  return v;
}

/* Round toward zero to bfloat16 storage (drop the low 16 bits). */
SYNTH_FN uint16_t synth_trunc_bf16(float x) { return (uint16_t)(S_F2U(x) >> 16); }

/* Round toward zero to binary16 storage; magnitudes >= 65504 clamp to 65504. */
SYNTH_FN uint16_t synth_trunc_f16(float x) {
  uint32_t u = S_F2U(x);
  uint16_t s = (uint16_t)((u >> 16) & 0x8000u);
  uint32_t a = u & 0x7FFFFFFFu;
  if (a >= 0x477FE000u) return (uint16_t)(s | 0x7BFFu);
  uint32_t e = a >> 23;
  if (e >= 113u) return (uint16_t)(s | ((e - 112u) << 10) | ((a >> 13) & 0x3FFu));
  float sub = S_MUL(S_U2F(a), 16777216.0f); /* |x| * 2^24 < 1024, exact */
  return (uint16_t)(s | (uint16_t)(uint32_t)sub);
}

#endif /* SYNTH_H */
