/*
 * mpnum.h — C ABI of libmpnum.so, the GB300 (sm_103a) mixed-precision hot path.
 *
 * Three parts of the precision machinery around the GEMMs of mixed-precision
 * training, each a stream-ordered call on one GPU:
 *   1. the fused optimizer step: unscale, inf/NaN check, AdamW on FP32
 *      masters, rounded 16-bit working copy, and the dynamic loss scale;
 *   2. the FP8 delayed-scaling cast with its amax-history ring;
 *   3. NVFP4 quantisation (E2M1 codes, E4M3 block scales, FP32 tensor scale,
 *      1x16 or 16x16 blocks, optional random Hadamard transform, round to
 *      nearest even or stochastic rounding), plus the standalone transform.
 *
 * Pages cited (title, then section):
 *   [MPT-ko] itwiki "혼합 정밀도 학습" (mixed precision training)
 *   [FP8-TE] llm-wiki "FP8 혼합 정밀도 LLM 학습: Transformer Engine과 Delayed Scaling…"
 *   [NVFP4]  gist.science "Pretraining Large Language Models with NVFP4"
 *   [MPT-es] marovi.ai "Mixed Precision Training/es"
 *
 * Conventions for every entry point:
 *   - Pointers prefixed d_ and all tensor pointers are DEVICE pointers on the
 *     current device; structs passed as `const T*` without the prefix are HOST
 *     pointers read during the call only.  The caller owns every buffer; the
 *     library never allocates, frees or synchronises.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All device work is enqueued on it and runs asynchronously.
 *   - Argument errors are detected on the host and returned before anything
 *     is enqueued.  A failed launch returns MP_ECUDA.  Data conditions
 *     (inf/NaN in the grads, non-finite NVFP4 input) are reported through
 *     device words, never through the return code.
 *   - Tensors are dense, row-major and 16-byte aligned.  Element counts may
 *     be anything >= 0 unless stated.
 *   - Calls that share a state struct, meta struct or workspace must be
 *     ordered on one stream; calls with disjoint state may run concurrently.
 *   - The quantiser kernels (FP8, NVFP4, MX, the transform) are launched with
 *     programmatic stream serialization allowed: their blocks may be
 *     scheduled while the previous kernel in the stream finishes, but each
 *     waits for that kernel to complete (griddepcontrol.wait) before touching
 *     memory, so the stream order seen by memory is unchanged.
 */
#ifndef MPNUM_H
#define MPNUM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MP_API __attribute__((visibility("default")))
#else
#define MP_API
#endif

typedef int32_t mp_status;
enum {
  MP_OK = 0,
  MP_EINVAL = -1,     /* null pointer, negative size, bad enum or hyperparameter */
  MP_EALIGN = -2,     /* a pointer is misaligned (tensors 16-byte; see each call) */
  MP_ESHAPE = -3,     /* a shape the call does not take (see each call) */
  MP_EWORKSPACE = -4, /* workspace missing or smaller than required */
  MP_ECUDA = -5       /* a kernel launch failed */
};

typedef int32_t mp_dtype;
enum { MP_F32 = 0, MP_F16 = 1, MP_BF16 = 2, MP_E4M3 = 3, MP_E5M2 = 4, MP_E2M1 = 5, MP_E2M3 = 6, MP_E3M2 = 7 };

MP_API const char* mp_status_str(mp_status s);
MP_API int32_t mp_version(void);
/* Number of kernels this library has launched in this process (diagnostic). */
MP_API uint64_t mp_launch_count(void);
/* Number of bounded waits on a tile copy that gave up inside this library's
 * FP8 kernels since it was loaded (0 in normal operation).  A kernel whose
 * copy engine stopped answering waits about two seconds per wait, counts the
 * failure here and returns; the outputs of that call are then incomplete.
 * Reads device memory synchronously: call it after synchronising the streams
 * that ran the calls.  *out written; MP_EINVAL if out is NULL. */
MP_API mp_status mp_wait_failures(uint32_t* out);

/* =========================================================================
 * 1. Mixed-precision optimizer step
 * ========================================================================= */

/* One parameter tensor of the step.  master, exp_avg, exp_avg_sq: FP32, read
 * and written.  grad: 16-bit (F16 or BF16), read, holding S * dL/dw.
 * working: 16-bit copy of the master, written.  All numel elements long. */
typedef struct {
  float* master;
  float* exp_avg;
  float* exp_avg_sq;
  const void* grad;
  void* working;
  int64_t numel;
} mp_param;

/* AdamW hyperparameters ([MPT-ko] "FP16 학습 루프": AdamW, lr 1e-3, and
 * clip_grad_norm_(max_norm=1.0) after unscale_).  max_grad_norm > 0 clips the
 * unscaled grads to that global L2 norm; 0 disables clipping. */
typedef struct {
  float lr, beta1, beta2, eps, weight_decay;
  float max_grad_norm;
} mp_adamw_hparams;

/* Device-resident state of the loss scaler and the step counter, 88 bytes.
 * Copying the struct checkpoints it.  Initialise it with
 * mp_scaler_state_init on the host and copy it to the device. */
typedef struct {
  float scale;            /* loss scale S in force for the next step */
  int32_t growth_tracker; /* consecutive clean steps since the last change */
  int32_t found_inf;      /* 1 if the most recent step saw an inf/NaN grad */
  int32_t error_flags;    /* nonzero if a kernel of a step gave up a bounded wait; outputs undefined */
  int64_t step;           /* applied (not skipped) optimizer steps */
  double beta1_pow;       /* beta1^step */
  double beta2_pow;       /* beta2^step */
  int64_t skipped;        /* steps skipped because of inf/NaN */
  float grad_norm;        /* global L2 norm of the unscaled grads (-1 without clipping) */
  float clip_coef;        /* factor applied to the unscaled grads (1 without clipping) */
  /* library-internal: zero after mp_scaler_state_init, left zero between calls */
  uint32_t internal_found;
  uint32_t internal_ticket;
  float internal_scalars[6];
} mp_scaler_state;

/* Loss-scale schedule ([MPT-ko] "손실 스케일링": GradScaler defaults 65536,
 * growth 2, backoff 0.5, interval 2000). */
typedef struct {
  float growth_factor, backoff_factor;
  int32_t growth_interval; /* >= 1 */
  int32_t enabled;         /* 0: loss_scale_update leaves the state unchanged */
} mp_scaler_cfg;

/* Host helper: scale = init_scale, beta powers 1, everything else zero. */
MP_API void mp_scaler_state_init(mp_scaler_state* host_state, float init_scale);

/* mp_adamw_step — one fused mixed-precision optimizer step over n_params
 * tensors ([MPT-ko] "FP32 마스터 가중치", "손실 스케일링", "FP16 학습 루프";
 * [MPT-es] "La receta de precisión mixta", "Escalado dinámico de pérdida").
 *
 * Pass 1 reads every grad once and sets d_state->found_inf to 1 if any grad
 * element is inf or NaN, else 0.  If it is set the step is skipped: no master,
 * moment or working element is written and step / beta powers do not advance
 * ([MPT-ko]: the update of that step is skipped).  Otherwise step += 1, the
 * beta powers advance and every element is updated, in binary32, with
 * scalars formed once per step in binary64 from the float hyperparameters:
 *     g  = (fp32(grad) * (1/S)) * clip             unscale, then clip
 *     w  = w * (1 - lr*wd)                         decoupled weight decay
 *     m  = m*beta1 + g*(1-beta1)
 *     v  = v*beta2 + (g*g)*(1-beta2)
 *     w  = w - (lr/(1-beta1^t)) * (m / (sqrt(v)/sqrt(1-beta2^t) + eps))
 *     working = round-to-nearest-even to the working dtype (NaN -> 0x7FFF)
 * clip = 1 unless hp->max_grad_norm > 0; then pass 1 also forms the global L2
 * norm of the unscaled grads g = fp32(grad) * (1/S) in one fixed order (tiles
 * of 16384 elements per tensor summed in binary32 in a fixed lane/tree order,
 * tile sums folded in binary64 in a fixed order; the oracle states it), writes
 * d_state->grad_norm and clip = min(1, max_grad_norm / (norm + 1e-6)) to
 * d_state->clip_coef ([MPT-ko] "FP16 학습 루프"; [MPT-es] "Operaciones que
 * permanecen en FP32": gradient norms are long reductions kept in FP32).
 * Clipping needs d_workspace of mp_adamw_workspace_size(params, n_params)
 * bytes (device, 8-byte aligned, any contents); without clipping it may be
 * NULL.
 * The host array `params` (n_params >= 0 entries) is read during the call
 * only; its pointers are device pointers, 16-byte aligned.  grad_dtype and
 * working_dtype are MP_F16 or MP_BF16.  The loss scale itself is not changed
 * here: call loss_scale_update after the step.  Launches at most
 * 2 * ceil(n_params / 512) + 1 kernels. */
MP_API size_t mp_adamw_workspace_size(const mp_param* params, int32_t n_params);
MP_API mp_status mp_adamw_step(const mp_param* params, int32_t n_params, mp_dtype grad_dtype,
                               mp_dtype working_dtype, const mp_adamw_hparams* hp,
                               mp_scaler_state* d_state, void* d_workspace, size_t workspace_bytes,
                               void* stream);

/* The two passes of mp_adamw_step as separate calls, mirroring the unscale
 * (inf check) and step calls of [MPT-ko] "FP16 학습 루프", so that work such
 * as gradient-norm clipping can run between them.  mp_adamw_check is pass 1
 * (sets found_inf, advances step / beta powers, forms the step scalars from
 * hp, and the norm and clip coefficient when clipping); mp_adamw_apply is
 * pass 2 and must follow it on the same stream with the same params and hp.
 * mp_adamw_check launches ceil(n_params / 512) kernels (+1 with clipping),
 * mp_adamw_apply ceil(n_params / 512). */
MP_API mp_status mp_adamw_check(const mp_param* params, int32_t n_params, mp_dtype grad_dtype,
                                const mp_adamw_hparams* hp, mp_scaler_state* d_state,
                                void* d_workspace, size_t workspace_bytes, void* stream);
MP_API mp_status mp_adamw_apply(const mp_param* params, int32_t n_params, mp_dtype grad_dtype,
                                mp_dtype working_dtype, const mp_adamw_hparams* hp,
                                mp_scaler_state* d_state, void* stream);

/* loss_scale_update — the dynamic loss-scale schedule ([MPT-ko] "손실 스케일링";
 * [MPT-es] "Escalado dinámico de pérdida"), from d_state->found_inf of the
 * last step: on inf/NaN S *= backoff, tracker = 0, skipped += 1; otherwise
 * tracker += 1 and when it reaches growth_interval S *= growth (kept only if
 * finite) and tracker = 0.  One single-thread kernel. */
MP_API mp_status loss_scale_update(mp_scaler_state* d_state, const mp_scaler_cfg* cfg,
                                   void* stream);

/* =========================================================================
 * 2. FP8 delayed scaling
 * ========================================================================= */

/* Device-resident per-tensor FP8 metadata, 32 bytes. */
typedef struct {
  float scale;     /* scale used by the next cast */
  float scale_inv; /* 1 / scale */
  float amax;      /* amax of the most recent cast's input */
  int32_t pos;     /* next history slot */
  /* library-internal: zero after mp_fp8_meta_init, left zero between calls */
  uint32_t internal_amax;
  uint32_t internal_ticket;
  uint32_t internal_hrest;
  uint32_t reserved;
} mp_fp8_meta;

/* Host helper: scale = scale_inv = 1, amax = 0, pos = 0, internals zero. */
MP_API void mp_fp8_meta_init(mp_fp8_meta* host_meta);

/* amax_algo of the FP8 casts: the next scale comes from the maximum of the
 * history ring (the default of [FP8-TE] "Delayed Scaling 동작 원리"), or from
 * the latest amax alone ([FP8-TE] "도입 체크리스트": most_recent, to follow
 * fast changes). */
enum { MP_AMAX_HISTORY_MAX = 0, MP_AMAX_MOST_RECENT = 1 };

/* fp8_cast_delayed — one delayed-scaling cast ([FP8-TE] "Delayed Scaling 동작
 * 원리", "E4M3 vs E5M2", "FP8이 어려운 이유"; [MPT-ko] "FP8 혼합 정밀도").
 * Reads x once.  For each of the n elements of x (x_dtype MP_F32, MP_F16 or
 * MP_BF16): y = saturate(round-to-nearest-even(fp32(x) * d_meta->scale)) in
 * fp8_dtype (MP_E4M3: max 448; MP_E5M2: max 57344); magnitudes beyond the
 * maximum, infinities included, become the signed maximum; a NaN product
 * becomes 0x7F with the input element's sign bit (0xFF when it is negative).
 * In the same pass amax = max |x| (NaN if any element is NaN).  Then
 * d_meta->amax = amax, d_history[p] = amax with p = pos mod history_len,
 * pos = (p + 1) % history_len, and if H = max(d_history) (amax_algo
 * MP_AMAX_HISTORY_MAX) or H = amax (MP_AMAX_MOST_RECENT) is finite and > 0
 * the next scale is fp8_max / (margin * H) (kept only if finite and > 0),
 * scale_inv = 1/scale.  d_history: history_len FP32 entries (1..65536),
 * zero-initialised by the caller, non-negative.  x and y 16-byte aligned.
 * One kernel launch. */
MP_API mp_status fp8_cast_delayed(const void* x, mp_dtype x_dtype, int64_t n, void* y,
                                  mp_dtype fp8_dtype, mp_fp8_meta* d_meta, float* d_history,
                                  int32_t history_len, float margin, int32_t amax_algo, void* stream);

/* fp8_cast_delayed_count — fp8_cast_delayed that also adds to *d_saturated
 * the number of elements the cast saturates: |fp32(x) * scale| (binary32
 * product) above fp8_max, infinities included, NaN not counted ([FP8-TE]
 * "Delayed Scaling 동작 원리": margin is tuned against saturation).  Same
 * outputs and state updates as fp8_cast_delayed; the counter accumulates over
 * calls (the caller zeroes it); d_saturated is a device pointer, 8-byte
 * aligned.  A separate entry point so that the plain cast pays no atomics.
 * One kernel launch. */
MP_API mp_status fp8_cast_delayed_count(const void* x, mp_dtype x_dtype, int64_t n, void* y,
                                        mp_dtype fp8_dtype, mp_fp8_meta* d_meta, float* d_history,
                                        int32_t history_len, float margin, int32_t amax_algo,
                                        unsigned long long* d_saturated, void* stream);

/* fp8_cast_transpose_delayed — fp8_cast_delayed of a [rows, cols] tensor that
 * also writes y_t [cols, rows] = transpose(y) from the same single read: the
 * backward GEMMs use the transposed operand ([NVFP4] §2.2 item 3 on the
 * transposed tensors of the backward pass).  Same scaling, amax and history
 * semantics; rows % 16 == 0 and cols % 16 == 0, rows and cols < 2^31 (else
 * MP_ESHAPE); x, y, y_t 16-byte aligned.  One kernel launch, reading x
 * through 2-D tensor copies: MP_ECUDA if the driver's tensor-map encoder is
 * unavailable. */
MP_API mp_status fp8_cast_transpose_delayed(const void* x, mp_dtype x_dtype, int64_t rows, int64_t cols,
                                            void* y, void* y_t, mp_dtype fp8_dtype, mp_fp8_meta* d_meta,
                                            float* d_history, int32_t history_len, float margin,
                                            int32_t amax_algo, void* stream);

/* fp8_quantize_blockwise — fine-grained FP8 with scales computed on the fly
 * per block, no history ([FP8-TE] "DeepSeek-V3 FP8 학습 사례": activations in
 * 1x128 tiles, weights in 128x128 blocks, E4M3 throughout; [MPT-ko] "FP8 혼합
 * 정밀도").  For each block (block_rows x block_cols = 1x128 or 128x128;
 * blocks at the right and bottom edges may be partial): amax = max |x| (NaN
 * if any is NaN), scales[block] = amax / fp8_max (the quiet NaN 0x7FC00000
 * for a block holding a NaN; FP32, row-major
 * [ceil(rows/br)][ceil(cols/bc)]), and every element
 * y = saturate(RNE(fp32(x) * r)) with r = fp8_max / amax if amax is finite
 * and > 0, else r = 0 (a NaN product gives 0x7F or, for a negative input
 * element, 0xFF).  Each block is read once.
 * cols % 16 == 0 and rows, cols < 2^31 (else MP_ESHAPE); x, y 16-byte
 * aligned.  One kernel launch; both block shapes read x through 2-D tensor
 * copies of 128 x 128 boxes: MP_ECUDA if the driver's tensor-map encoder is
 * unavailable. */
MP_API mp_status fp8_quantize_blockwise(const void* x, mp_dtype x_dtype, int64_t rows, int64_t cols,
                                        int32_t block_rows, int32_t block_cols, void* y, mp_dtype fp8_dtype,
                                        float* scales, void* stream);

/* =========================================================================
 * 3. NVFP4 quantisation and the random Hadamard transform
 * ========================================================================= */

/* Bytes of workspace nvfp4_quantize needs (zero-filled before first use;
 * every completed call leaves it zero-filled again). */
MP_API size_t nvfp4_workspace_size(void);

/* nvfp4_quantize — two-level NVFP4 quantisation of a BF16 [rows, cols]
 * tensor ([NVFP4] §2.1 "NVFP4 포맷의 특징", §2.2 items 2-4).
 *   x' = x, or with apply_rht the 16-point transform of rht16 applied to
 *        every 16 contiguous elements of each row;
 *   s_t = amax(|x'|) / (6 * 448)                  -> *d_tensor_scale (FP32)
 *   per block (1x16 along a row, or 16x16 when block_2d):
 *        sb = E4M3(round-to-nearest-even((bamax / 6) / s_t)), saturating
 *        d  = value(sb) * s_t,  r = 1/d (0 if d == 0 or 1/d not finite)
 *   per element: q = E2M1(x' * r), saturating at 6, sign kept on zero,
 *        round to nearest even, or with `stochastic` rounded away from zero
 *        iff floor(frac * 2^16) + r16 >= 2^16, where frac is the position of
 *        |x' r| between its grid neighbours and r16 are the 16 bits of
 *        Philox4x32-10 (key = seed, counter = (i/8, 0, 0)) word (i/2)%4,
 *        half i%2, i the flat row-major element index;
 *   dequant (optional, may be NULL) = BF16 RNE of value(q) * d.
 * Outputs: codes [rows, cols/2] (element 2j in the low nibble of byte j),
 * block_scales [rows, cols/16] (1x16) or [rows/16, cols/16] (16x16), E4M3
 * bytes, row-major; d_nonfinite = 1 if amax is not finite, in which case
 * s_t = amax and all codes, scales and dequant values are zero (also when
 * s_t == 0).  Requires cols % 16 == 0, and rows % 16 == 0 when block_2d.
 * Two passes over x (amax, then encode): two kernel launches. */
MP_API mp_status nvfp4_quantize(const void* x_bf16, int64_t rows, int64_t cols, int32_t block_2d,
                                int32_t stochastic, uint64_t seed, int32_t apply_rht,
                                uint16_t rht_sign_mask, uint8_t* codes, uint8_t* block_scales,
                                float* d_tensor_scale, int32_t* d_nonfinite, void* dequant_bf16,
                                void* d_workspace, size_t workspace_bytes, void* stream);

/* nvfp4_quantize_noalloc — nvfp4_quantize without a caller-supplied
 * workspace.  The pages describe nothing like it: it exists for callers that
 * cannot allocate device memory at the point of the call, for example code
 * running inside a framework step whose memory pool must not grow, plugin
 * interfaces that are handed only their inputs and outputs, or host code that
 * must avoid cudaMalloc because it synchronises the device.  Arguments,
 * outputs and results are those of nvfp4_quantize.  The scratch is a
 * file-scope device array of nvfp4_noalloc_scratch_bytes() (256) bytes that
 * every device holds from library load to process exit; a call needs
 * nvfp4_workspace_size() bytes of it and returns MP_EWORKSPACE if that is
 * more than the array holds.  The call allocates and frees nothing.
 * Arguments are checked first, exactly as in nvfp4_quantize, and an argument
 * error returns before anything is enqueued.  The first call in each CUDA
 * context (each device's primary context, and again after cudaDeviceReset
 * makes a new one) looks up the array's device address (cudaGetSymbolAddress)
 * with that context current: make that first call before any stream capture.
 * Each call then clears the words that must start at zero (a stream-ordered
 * memset of the library's own scratch) and enqueues the two kernels.  Every
 * call on a device shares the one array: calls that overlap on the GPU
 * (different streams, no ordering between them) race on it and their results
 * are undefined. */
MP_API size_t nvfp4_noalloc_scratch_bytes(void);
MP_API mp_status nvfp4_quantize_noalloc(const void* x_bf16, int64_t rows, int64_t cols,
                                        int32_t block_2d, int32_t stochastic, uint64_t seed,
                                        int32_t apply_rht, uint16_t rht_sign_mask, uint8_t* codes,
                                        uint8_t* block_scales, float* d_tensor_scale,
                                        int32_t* d_nonfinite, void* dequant_bf16, void* stream);

/* e2m1_stochastic_round — the stochastic rounding of nvfp4_quantize
 * ([NVFP4] §2.2 item 4, "확률적 반올림") on values the caller supplies, with
 * random bits the caller supplies: for i < n, the E2M1 code of y[i] rounded
 * away from zero iff floor(frac * 2^16) + r16[i] >= 2^16, frac the position of
 * |y[i]| between its grid neighbours (0, 0.5, 1, 1.5, 2, 3, 4, 6); magnitudes
 * from 6 up (infinities included) and NaN give 6; the sign bit is kept (-0
 * gives 0x8).  y: FP32 [n], r16: uint16 [n], codes: [(n + 1) / 2] bytes,
 * element 2j in the low nibble of byte j (the high nibble of the last byte is
 * 0 when n is odd); all device pointers, 16-byte aligned (MP_EALIGN), n >= 0
 * (MP_EINVAL).  One kernel launch; the caller owns every buffer. */
MP_API mp_status e2m1_stochastic_round(const float* y, const uint16_t* r16, int64_t n, uint8_t* codes,
                                       void* stream);

/* rht16 — the 16-point random Hadamard transform ([NVFP4] §2.2 item 2):
 * for every 16 contiguous elements t of each row of BF16 x [rows, cols],
 * y_t = 1/4 * H16 * diag(s) * x_t, H16 the Sylvester Hadamard matrix
 * (H[i][j] = (-1)^popcount(i & j)), s_j = -1 iff bit j of sign_mask is set,
 * evaluated in binary32 by the butterfly of span 1, 2, 4, 8.  y_dtype MP_F32
 * or MP_BF16 (round to nearest even).  cols % 16 == 0. */
MP_API mp_status rht16(const void* x_bf16, int64_t rows, int64_t cols, uint16_t sign_mask, void* y,
                       mp_dtype y_dtype, void* stream);

/* =========================================================================
 * 4. MX block formats
 * ========================================================================= */

/* mx_quantize — microscaling quantisation ([MPT-ko] "FP8 혼합 정밀도": one
 * power-of-two scale for every 32 elements, MXFP8 and MXFP4; [NVFP4] §2.1:
 * MXFP4 keeps a UE8M0 scale byte per 32-element block).  x [rows, cols]
 * (x_dtype MP_F32, MP_F16 or MP_BF16, row-major); every run of 32 elements
 * along a row is a block.  elem_dtype MP_E4M3, MP_E5M2 (MXFP8), MP_E2M3,
 * MP_E3M2 (MXFP6: 1 sign, 2 exponent (bias 1), 3 mantissa bits, largest 7.5;
 * 1 sign, 3 exponent (bias 3), 2 mantissa bits, largest 28) or MP_E2M1
 * (MXFP4).  For a block with amax = max |x| finite: e = floor(log2 amax) -
 * emax (emax 8, 15, 2, 4, 2: the exponent of the element format's largest value),
 * clamped below at -127 (so amax = 0 or subnormal gives -127); scales[block]
 * = e + 127 (UE8M0, [rows][cols/32], one byte per block); each element is
 * saturate(RNE(fp32(x) * 2^-e)) in elem_dtype.  A block holding an infinity
 * or NaN gets the scale byte 0xFF (the UE8M0 NaN) and all-zero codes.
 * codes: one byte per element for FP8 and FP6 (an FP6 code in bits 0..5, sign
 * at bit 5, bits 6..7 zero), or two E2M1 codes per byte (element 2j in the
 * low nibble), row-major.  dequant_bf16 (may be NULL): BF16 RNE of
 * value(code) * 2^e, zero for a non-finite block.  cols % 32 == 0 (else
 * MP_ESHAPE); x, codes and dequant_bf16 16-byte aligned.  One kernel launch;
 * rows * cols == 0 launches nothing. */
MP_API mp_status mx_quantize(const void* x, mp_dtype x_dtype, int64_t rows, int64_t cols, mp_dtype elem_dtype,
                             void* codes, uint8_t* scales, void* dequant_bf16, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* MPNUM_H */
