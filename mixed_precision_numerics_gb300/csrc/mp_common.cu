// mp_common.cu — status strings, version, launch counter, state initialisers.
#include <cudaTypedefs.h>

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

// The driver's tensor-map encoder, looked up once through the runtime (no
// link against the driver library).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 f = fn.load(std::memory_order_acquire);
  if (f) return f;
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !p)
    return nullptr;
  f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  fn.store(f, std::memory_order_release);
  return f;
}

bool encode_tile_map_2d(CUtensorMap* map, const void* base, int esize, int64_t rows, int64_t cols, int box_rows,
                        int box_cols) {
  if (rows < 1 || cols < 1 || rows >= (1ll << 31) || cols >= (1ll << 31)) return false;  // int32 box coordinates
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || ((cols * esize) & 15)) return false;
  const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const CUtensorMapDataType dt = esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t pitch[1] = {(cuuint64_t)(cols * esize)};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t unit[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void*>(base), dims, pitch, box, unit, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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

MP_API mp_status mp_wait_failures(uint32_t* out) {
  if (!out) return MP_EINVAL;
  *out = mp::fp8_wait_failures();
  return MP_OK;
}

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
