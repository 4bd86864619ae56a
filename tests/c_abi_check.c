/* Plain C99 user of the library: includes only the public header, links
 * libmpnum.so, and exercises the calls that need no GPU (state initialisers,
 * status strings, workspace sizes and argument validation, which returns
 * before anything is launched).  Exit code 0 on success. */
#include <stdio.h>
#include <string.h>

#include "mpnum.h"

#define CHECK(cond)                                          \
  do {                                                       \
    if (!(cond)) {                                           \
      fprintf(stderr, "failed: %s (line %d)\n", #cond, __LINE__); \
      return 1;                                              \
    }                                                        \
  } while (0)

int main(void) {
  mp_scaler_state st;
  mp_fp8_meta meta;
  mp_adamw_hparams hp = {1e-3f, 0.9f, 0.999f, 1e-8f, 0.01f, 0.0f};
  mp_param p;
  CHECK(sizeof(mp_scaler_state) == 88 && sizeof(mp_fp8_meta) == 32 && sizeof(mp_param) == 48);
  mp_scaler_state_init(&st, 65536.0f);
  CHECK(st.scale == 65536.0f && st.step == 0 && st.beta1_pow == 1.0 && st.beta2_pow == 1.0);
  mp_fp8_meta_init(&meta);
  CHECK(meta.scale == 1.0f && meta.scale_inv == 1.0f && meta.pos == 0);
  CHECK(mp_version() > 0);
  CHECK(strlen(mp_status_str(MP_OK)) > 0 && strlen(mp_status_str(MP_ECUDA)) > 0);
  CHECK(nvfp4_workspace_size() >= 8 && nvfp4_noalloc_scratch_bytes() >= nvfp4_workspace_size());

  /* argument errors come back before any launch, with no GPU needed */
  memset(&p, 0, sizeof(p));
  p.numel = 100;
  CHECK(mp_adamw_step(&p, 1, MP_F16, MP_BF16, &hp, (mp_scaler_state*)16, NULL, 0, NULL) == MP_EINVAL);
  CHECK(mp_adamw_step(NULL, 0, MP_E4M3, MP_BF16, &hp, (mp_scaler_state*)16, NULL, 0, NULL) == MP_EINVAL);
  CHECK(fp8_cast_delayed((void*)16, MP_BF16, 64, (void*)16, MP_F16, (mp_fp8_meta*)16, (float*)16, 4, 1.0f,
                         MP_AMAX_HISTORY_MAX, NULL) == MP_EINVAL);
  CHECK(nvfp4_quantize((void*)16, 4, 24, 0, 0, 0, 0, 0, (uint8_t*)16, (uint8_t*)16, (float*)16, (int32_t*)16, NULL,
                       (void*)16, 256, NULL) == MP_ESHAPE);
  CHECK(mx_quantize((void*)16, MP_BF16, 2, 48, MP_E2M1, (void*)16, (uint8_t*)16, NULL, NULL) == MP_ESHAPE);
  CHECK(rht16((void*)16, 2, 40, 0, (void*)16, MP_F32, NULL) == MP_ESHAPE);
  CHECK(mp_wait_failures(NULL) == MP_EINVAL);
  CHECK(mp_launch_count() == 0);
  printf("c abi ok\n");
  return 0;
}
