// synth_dev.cu — device build of the seeded input generator (see synth.h).
// Fills device buffers with the same bits the host build produces.
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth.h"

__global__ void synth_fill_kernel(synth_recipe r, int dtype, uint64_t start, int64_t n, void* out) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float v = synth_value(&r, start + (uint64_t)i);
    if (dtype == SYNTH_F32)
      ((float*)out)[i] = v;
    else if (dtype == SYNTH_F16)
      ((uint16_t*)out)[i] = synth_trunc_f16(v);
    else
      ((uint16_t*)out)[i] = synth_trunc_bf16(v);
  }
}

__global__ void synth_fill_at_kernel(synth_recipe r, int dtype, const int64_t* idx, int64_t n,
                                     void* out) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float v = synth_value(&r, (uint64_t)idx[i]);
    if (dtype == SYNTH_F32)
      ((float*)out)[i] = v;
    else if (dtype == SYNTH_F16)
      ((uint16_t*)out)[i] = synth_trunc_f16(v);
    else
      ((uint16_t*)out)[i] = synth_trunc_bf16(v);
  }
}

static int grid_for(int64_t n) {
  int dev = 0, sms = 132;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t want = (n + 255) / 256;
  int64_t cap = (int64_t)sms * 8;
  return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}

extern "C" int synth_fill_dev(const synth_recipe* r, int dtype, uint64_t start, int64_t n,
                              void* d_out, cudaStream_t s) {
  if (n <= 0) return 0;
  synth_fill_kernel<<<grid_for(n), 256, 0, s>>>(*r, dtype, start, n, d_out);
  return (int)cudaGetLastError();
}

extern "C" int synth_fill_at_dev(const synth_recipe* r, int dtype, const int64_t* d_idx,
                                 int64_t n, void* d_out, cudaStream_t s) {
  if (n <= 0) return 0;
  synth_fill_at_kernel<<<grid_for(n), 256, 0, s>>>(*r, dtype, d_idx, n, d_out);
  return (int)cudaGetLastError();
}
