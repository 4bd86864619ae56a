/*
 * synth_host.c — host build of the seeded input generator (see synth.h).
 * Built with -O2 -ffp-contract=off so that every binary32 operation rounds
 * once, exactly like the device build.
 */
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#include "synth.h"

static void fill_range(const synth_recipe* r, int dtype, uint64_t start, int64_t lo, int64_t hi,
                       const int64_t* idx, void* out) {
  for (int64_t i = lo; i < hi; ++i) {
    uint64_t k = idx ? (uint64_t)idx[i] : start + (uint64_t)i;
    float v = synth_value(r, k);
    if (dtype == SYNTH_F32)
      ((float*)out)[i] = v;
    else if (dtype == SYNTH_F16)
      ((uint16_t*)out)[i] = synth_trunc_f16(v);
    else
      ((uint16_t*)out)[i] = synth_trunc_bf16(v);
  }
}

typedef struct {
  const synth_recipe* r;
  int dtype;
  uint64_t start;
  int64_t lo, hi;
  const int64_t* idx;
  void* out;
} job_t;

static void* job_main(void* p) {
  job_t* j = (job_t*)p;
  fill_range(j->r, j->dtype, j->start, j->lo, j->hi, j->idx, j->out);
  return NULL;
}

static void fill_parallel(const synth_recipe* r, int dtype, uint64_t start, int64_t n,
                          const int64_t* idx, void* out, int threads) {
  if (threads <= 1 || n < (1 << 16)) {
    fill_range(r, dtype, start, 0, n, idx, out);
    return;
  }
  if (threads > 64) threads = 64;
  pthread_t tid[64];
  job_t jobs[64];
  int64_t per = (n + threads - 1) / threads;
  int launched = 0;
  for (int t = 0; t < threads; ++t) {
    int64_t lo = (int64_t)t * per, hi = lo + per < n ? lo + per : n;
    if (lo >= hi) break;
    jobs[t] = (job_t){r, dtype, start, lo, hi, idx, out};
    if (pthread_create(&tid[t], NULL, job_main, &jobs[t]) != 0) {
      fill_range(r, dtype, start, lo, hi, idx, out);
      tid[t] = 0;
    }
    launched = t + 1;
  }
  for (int t = 0; t < launched; ++t)
    if (tid[t]) pthread_join(tid[t], NULL);
}

/* out[i] = value(start + i), i in [0, n). */
void synth_fill(const synth_recipe* r, int dtype, uint64_t start, int64_t n, void* out,
                int threads) {
  fill_parallel(r, dtype, start, n, NULL, out, threads);
}

/* out[i] = value(idx[i]), i in [0, n). */
void synth_fill_at(const synth_recipe* r, int dtype, const int64_t* idx, int64_t n, void* out,
                   int threads) {
  fill_parallel(r, dtype, 0, n, idx, out, threads);
}

/* Raw pieces, exposed for the generator's own tests. */
float synth_normal_at(uint64_t seed, uint64_t stream, uint64_t index) {
  return synth_normal(seed, stream, index);
}
float synth_logf_host(float u) { return synth_logf(u); }
float synth_cos2pi_host(float v) { return synth_cos2pi(v); }
uint16_t synth_trunc_f16_host(float x) { return synth_trunc_f16(x); }
uint64_t synth_hash_host(uint64_t seed, uint64_t stream, uint64_t index) {
  return synth_hash(seed, stream, index);
}
