/*
 * oracle.h — plain, scalar CPU oracle for the mixed-precision hot path.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no source,
 * header, table or helper with the CUDA kernels, and the product never calls
 * it.
 *
 * Build: gcc -O2 -ffp-contract=off (no fast-math, no SIMD intrinsics), so each
 * binary32 operation written below rounds exactly once to nearest-even.
 *
 * Pages cited (title, then section):
 *   [MPT-ko]  itwiki "혼합 정밀도 학습" (mixed precision training)
 *   [FP8-TE]  llm-wiki "FP8 혼합 정밀도 LLM 학습: Transformer Engine과 Delayed Scaling…"
 *   [NVFP4]   gist.science "Pretraining Large Language Models with NVFP4"
 *   [MPT-es]  marovi.ai "Mixed Precision Training/es"
 * Where the pages leave a step open, the reading taken is stated at the
 * function and listed (R-numbers) in the design notes.
 *
 * Parity pins: every function here is pinned by the CPU test suite against
 * values the pages print, closed forms, brute-force searches or independent
 * library routines.  Philox4x32-10 is pinned against an independent library
 * implementation of the same generator.  The FP8 NaN byte (R1) has no page
 * value behind it and is pinned to torch's float8 casts (both signs); the
 * 16-bit NaN pattern (R-NaN16: every NaN becomes 0x7FFF, the image of the
 * canonical binary32 NaN) is pinned to torch's CUDA FP16/BF16 casts of every
 * binary32 NaN pattern and to the CPU libraries' image of 0x7FFFFFFF.
 */
#ifndef MPNUM_ORACLE_H
#define MPNUM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_E4M3 = 3, ORC_E5M2 = 4, ORC_E2M1 = 5, ORC_E2M3 = 6, ORC_E3M2 = 7 };

/* ---- number formats ---------------------------------------------------------
 * [MPT-ko] "왜 그냥 FP16으로는 안 되는가": FP16 = 5 exponent / 10 mantissa bits,
 * max 65504, min normal 2^-14, min subnormal 2^-24.  [MPT-es] "Formatos de
 * coma flotante": BF16 = 8 exponent / 7 mantissa bits.  [MPT-ko] "FP8 혼합
 * 정밀도" and [FP8-TE] "E4M3 vs E5M2": E4M3 (4e3m, range ±448, no infinity),
 * E5M2 (5e2m, IEEE-like inf/NaN).  [NVFP4] §2.1: FP4 elements, read as E2M1
 * (1 sign, 2 exponent, 1 mantissa bit, bias 1) = {0, .5, 1, 1.5, 2, 3, 4, 6}.
 * All roundings are to nearest, ties to the even code. */
uint16_t orc_f32_to_f16(float x);   /* overflow -> inf; NaN -> 0x7FFF */
float orc_f16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16(float x);  /* overflow -> inf; NaN -> 0x7FFF */
float orc_bf16_to_f32(uint16_t h);
/* Saturating FP8: |x| beyond max (inf included) -> ±max; NaN -> 0x7F with
 * the NaN's sign bit (0xFF for a negative NaN). */
uint8_t orc_f32_to_fp8_sat(float x, int fmt);
float orc_fp8_to_f32(uint8_t c, int fmt);
uint8_t orc_f32_to_e2m1(float x); /* finite x; |x| > 6 -> 6; sign kept on zero */
/* Stochastic E2M1: with lo <= |x| < hi adjacent grid values,
 * f16 = floor((|x| - lo) / (hi - lo) * 2^16); result hi iff f16 + r16 >= 2^16. */
uint8_t orc_f32_to_e2m1_sr(float x, uint32_t r16);
float orc_e2m1_to_f32(uint8_t c);
/* FP6 ([MPT-ko] "FP8 혼합 정밀도" names MXFP6; layouts per reading R22):
 * E2M3 = 1 sign, 2 exponent (bias 1), 3 mantissa bits, largest 7.5;
 * E3M2 = 1 sign, 3 exponent (bias 3), 2 mantissa bits, largest 28.  No
 * infinity or NaN.  A code is 6 bits: sign at bit 5.  RNE, saturating (the
 * caller passes finite values). */
uint8_t orc_f32_to_fp6(float x, int fmt);
float orc_fp6_to_f32(uint8_t c, int fmt);
/* Element-wise conversion between any two of the formats above. */
void orc_convert(const void* in, int in_fmt, int64_t n, void* out, int out_fmt);
/* amax = max |x| over n elements; any NaN gives the quiet NaN 0x7FC00000. */
float orc_amax(const void* x, int fmt, int64_t n);

/* ---- Philox4x32-10 (Salmon et al., SC'11) ---------------------------------- */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);
/* 16 stochastic-rounding bits for flat element index i under `seed`. */
uint32_t orc_sr_bits(uint64_t seed, uint64_t i);
/* out[k] = stochastic E2M1 code of y[k] with the bits of index i0 + k. */
void orc_e2m1_sr_array(const float* y, int64_t n, uint64_t seed, uint64_t i0, uint8_t* out);
/* out[k] = stochastic E2M1 code of y[k] with the random bits r16[k]. */
void orc_e2m1_sr_bits_array(const float* y, const uint16_t* r16, int64_t n, uint8_t* out);

/* ---- 16-point random Hadamard transform ([NVFP4] §2.2 item 2) -------------- */
/* out = 1/4 * H16 * diag(s) * in, H16 Sylvester, s_j = -1 iff bit j of mask. */
void orc_rht16_tile(const float in[16], uint16_t sign_mask, float out[16]);
/* Applies the tile transform to every 16 contiguous elements of each row.
 * y_fmt ORC_F32 or ORC_BF16.  Returns 0, or -1 if cols % 16 != 0. */
int orc_rht16(const uint16_t* x_bf16, int64_t rows, int64_t cols, uint16_t sign_mask, void* y,
              int y_fmt);

/* ---- mixed-precision optimizer step ----------------------------------------- */
typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
  float max_grad_norm; /* > 0: clip the unscaled grads to this global L2 norm */
} orc_adamw_hp;

typedef struct {
  float scale;            /* loss scale S in force */
  int32_t growth_tracker; /* consecutive clean steps */
  int32_t found_inf;      /* 1 if the last step saw inf/NaN */
  int32_t pad0;
  int64_t step;           /* applied optimizer steps */
  double beta1_pow;       /* beta1^step */
  double beta2_pow;       /* beta2^step */
  int64_t skipped;        /* skipped steps */
} orc_scaler_state;

typedef struct {
  float growth_factor, backoff_factor;
  int32_t growth_interval, enabled;
} orc_scaler_cfg;

/* Per-step scalars, rounded once from binary64; clip = 1 without clipping. */
typedef struct {
  float inv_scale, step_size, bc2_sqrt, decay, omb1, omb2, beta1, beta2, eps, clip;
} orc_step_scalars;

/* 1 if any of the n 16-bit grads (fmt ORC_F16 / ORC_BF16) is inf or NaN. */
int orc_nonfinite_any(const uint16_t* g, int fmt, int64_t n);
/* Advances step and beta powers unless found_inf; fills the step scalars. */
void orc_adamw_begin(const orc_adamw_hp* hp, orc_scaler_state* st, int found_inf,
                     orc_step_scalars* out);
/* Unscale + AdamW on the FP32 master + rounded 16-bit copy, element-wise. */
void orc_adamw_apply(const orc_step_scalars* s, float* w, float* m, float* v, const uint16_t* g,
                     int g_fmt, uint16_t* w16, int w16_fmt, int64_t n);
/* Gradient-norm clipping ([MPT-ko] "FP16 학습 루프": clip_grad_norm_(max_norm=1.0)
 * after unscale_; [MPT-es] "Operaciones que permanecen en FP32": long
 * reductions such as gradient norms stay in high precision).  The norm is the
 * L2 norm of all unscaled grads g = fp32(grad) * inv_scale (binary32, as the
 * update uses them): orc_grad_sumsq returns one tensor's sum of g*g, squares
 * exact in binary64 and added in element order in binary64; the caller adds
 * the tensors' sums in list order in binary64, norm = sqrt(total).
 * clip = min(1, max_norm / (norm + 1e-6)), binary64, rounded to binary32. */
double orc_grad_sumsq(const uint16_t* g, int g_fmt, int64_t n, float inv_scale);
float orc_clip_coef(double norm, float max_norm);
/* Dynamic loss-scale update from st->found_inf. */
void orc_loss_scale_update(orc_scaler_state* st, const orc_scaler_cfg* cfg);

/* ---- FP8 delayed scaling ---------------------------------------------------- */
typedef struct {
  float scale, scale_inv, amax;
  int32_t pos;
} orc_fp8_meta;

/* One element: saturating RNE cast of fp32(x) * scale. */
uint8_t orc_fp8_cast_one(float x, float scale, int fmt);
/* Casts n elements with meta->scale; does not touch meta. */
void orc_fp8_cast_array(const void* x, int x_fmt, int64_t n, uint8_t* y, int fmt, float scale);
/* Elements the cast saturates ([FP8-TE] "Delayed Scaling 동작 원리": margin is
 * raised when FP8's range is under-used and lowered when casts saturate):
 * the count of i with |fp32(x_i) * scale| (binary32 product) above the
 * format's largest finite value, infinities included, NaN not counted. */
int64_t orc_fp8_saturation_count(const void* x, int x_fmt, int64_t n, int fmt, float scale);
/* Records amax in the ring and derives the next scale from max(history)
 * (amax_algo 0) or from this amax alone (amax_algo 1, "most_recent",
 * [FP8-TE] "도입 체크리스트"). */
void orc_fp8_history_update(orc_fp8_meta* meta, float* history, int32_t hist_len, float margin,
                            float amax, int fmt, int amax_algo);
/* One full iteration: cast with the current scale, amax, ring write, new scale. */
void orc_fp8_cast_delayed(const void* x, int x_fmt, int64_t n, uint8_t* y, int fmt,
                          orc_fp8_meta* meta, float* history, int32_t hist_len, float margin,
                          int amax_algo);
/* y_t[c][r] = y[r][c] for a [rows][cols] byte matrix. */
void orc_transpose_u8(const uint8_t* y, int64_t rows, int64_t cols, uint8_t* y_t);

/* ---- fine-grained FP8 with online block scales ([MPT-ko] "FP8 혼합 정밀도";
 * [FP8-TE] "DeepSeek-V3 FP8 학습 사례"): activations in 1x128 tiles, weights in
 * 128x128 blocks, each block's scale computed from the block itself (no
 * history).  Reading R20: amax = max |x| over the block; the stored scale is
 * s = amax / fp8_max (the quiet NaN 0x7FC00000 for a block holding a NaN);
 * elements are y = sat(RNE(fp32(x) * r)) with
 * r = fp8_max / amax when amax is finite and > 0, else r = 0.  Blocks at the
 * right and bottom edges may be partial.  scales: [ceil(rows/br)][ceil(cols/bc)]. */
void orc_fp8_quantize_blockwise(const void* x, int x_fmt, int64_t rows, int64_t cols, int32_t block_rows,
                                int32_t block_cols, int fmt, uint8_t* y, float* scales);

/* ---- MX block formats ([MPT-ko] "FP8 혼합 정밀도": MXFP8 / MXFP6 / MXFP4, one
 * power-of-two scale per 32 elements; [NVFP4] §2.1: MXFP4 = 32-element blocks
 * with a UE8M0 scale).  Reading R21: for a block of 32 elements along a row,
 * e = floor(log2(amax)) - emax_elem (emax_elem = 8, 15, 2 for E4M3, E5M2,
 * E2M1: the exponent of the format's largest value), clamped to
 * [-127, 127]; amax = 0 gives e = -127.  The scale byte is e + 127 (UE8M0);
 * elements are RNE(fp32(x) * 2^-e) saturating to the element format.  A
 * non-finite amax gives the scale byte 0xFF and all element codes 0.
 * codes: 1 byte per element (E4M3/E5M2) or two E2M1 codes per byte, element
 * 2j in the low nibble; scales [rows][cols / 32]; dequant (optional) is
 * BF16 RNE of value(code) * 2^e.  MXFP6 (E2M3, emax 2; E3M2, emax 4) keeps
 * one 6-bit code per byte (R22). */
void orc_mx_quantize(const void* x, int x_fmt, int64_t rows, int64_t cols, int elem_fmt, uint8_t* codes,
                     uint8_t* scales, uint16_t* dequant);

/* ---- NVFP4 quantisation ([NVFP4] §2.1, §2.2) ---------------------------------- */
/* x' = x or RHT(x), as FP32. */
int orc_nvfp4_prepare(const uint16_t* x_bf16, int64_t rows, int64_t cols, int apply_rht,
                      uint16_t sign_mask, float* xprime);
/* s_t = amax / (6 * 448); non-finite amax -> *nonfinite = 1 and s_t = amax. */
float orc_nvfp4_tensor_scale(float amax, int32_t* nonfinite);
/* Encodes rows [row0, row0 + nrows) of x' (row-major, `cols` wide; x' points
 * at row row0).  Outputs are written at the same row offset.  For 2D blocks
 * row0 and nrows are multiples of 16. */
void orc_nvfp4_encode_rows(const float* xprime, int64_t row0, int64_t nrows, int64_t cols,
                           int block_2d, int stochastic, uint64_t seed, float s_t,
                           int32_t nonfinite, uint8_t* codes, uint8_t* scales,
                           uint16_t* dequant);
/* The whole quantiser.  Returns 0, or -1 on a shape error. */
int orc_nvfp4_quantize(const uint16_t* x_bf16, int64_t rows, int64_t cols, int block_2d,
                       int stochastic, uint64_t seed, int apply_rht, uint16_t sign_mask,
                       uint8_t* codes, uint8_t* scales, float* tensor_scale, int32_t* nonfinite,
                       uint16_t* dequant);
/* Block scale of one block: code, d = value(code) * s_t, r = 1/d (0 if d == 0
 * or 1/d is not finite). */
void orc_nvfp4_block_scale(float bamax, float s_t, uint8_t* code, float* d, float* r);

#ifdef __cplusplus
}
#endif
#endif
