// mp_common.cu — status strings, version, launch counter, state initialisers.
#include <atomic>
#include <string.h>

#include "mp_internal.h"

namespace mp {

static std::atomic<uint64_t> g_launches{0};
void note_launches(uint64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int sm_count() {
  static std::atomic<int> cached[64];  // zero-initialised (static storage); 0 = not yet read
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
  if (dev < 64) {
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace mp

extern "C" {

MP_API const char* mp_status_str(mp_status s) {
  switch (s) {
    case MP_OK: return "ok";
    case MP_EINVAL: return "invalid argument (null pointer, negative size, bad dtype or hyperparameter)";
    case MP_EALIGN: return "pointer misaligned (tensors 16-byte, clipping workspace 8-byte)";
    case MP_ESHAPE: return "shape not supported by the call (e.g. cols % 16 != 0, or cols % 32 != 0 for MX)";
    case MP_EWORKSPACE: return "workspace missing or too small";
    case MP_ECUDA: return "CUDA launch failed";
    default: return "unknown status";
  }
}

MP_API int32_t mp_version(void) { return 10000; }

MP_API uint64_t mp_launch_count(void) { return mp::g_launches.load(std::memory_order_relaxed); }

MP_API void mp_scaler_state_init(mp_scaler_state* s, float init_scale) {
  if (!s) return;
  memset(s, 0, sizeof(*s));
  s->scale = init_scale;
  s->beta1_pow = 1.0;
  s->beta2_pow = 1.0;
}

MP_API void mp_fp8_meta_init(mp_fp8_meta* m) {
  if (!m) return;
  memset(m, 0, sizeof(*m));
  m->scale = 1.0f;
  m->scale_inv = 1.0f;
}

}  // extern "C"
