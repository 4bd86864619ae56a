// mp_internal.h — host-side helpers shared by the libmpnum translation units.
#pragma once

#include <cuda.h>  // CUtensorMap (types only; the encoder is reached through the runtime)
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/mpnum.h"

namespace mp {

// Count of kernels launched by this library (diagnostic, process-wide).
void note_launches(uint64_t n);

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Grid size for a grid-stride kernel: enough CTAs to cover `work_ctas`, at
// most `per_sm` resident CTAs on every SM.
inline int grid_for(int64_t work_ctas, int per_sm) {
  int64_t cap = (int64_t)sm_count() * per_sm;
  if (work_ctas < 1) work_ctas = 1;
  return (int)(work_ctas < cap ? work_ctas : cap);
}

// Encodes a 2-D row-major tensor [rows, cols] of `esize`-byte elements at
// `base` as a TMA tile map with box [box_rows, box_cols], no swizzle, zero
// fill outside the tensor.  False if the driver's encoder is unavailable or
// refuses the layout (base not 16-byte aligned, row pitch not a multiple of 16
// bytes, an extent of 2^31 or more: box coordinates are 32-bit signed).
bool encode_tile_map_2d(CUtensorMap* map, const void* base, int esize, int64_t rows, int64_t cols, int box_rows,
                        int box_cols);

// Bounded waits that gave up in this library's kernels since it was loaded.
uint32_t fp8_wait_failures();

// Raises `kernel`'s dynamic shared-memory limit to `bytes` on the current
// device the first time it launches there: the attribute belongs to the
// device, so a process driving several GPUs needs it once on each.  `done` is
// the call site's record, one bit per device (0..63; others set it every call).
template <typename K>
bool smem_opt_in(K kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  if (bit) done.fetch_or(bit, std::memory_order_release);
  return true;
}

// Launches `kernel` on stream `s` with programmatic stream serialization
// allowed: its CTAs may be scheduled before the previous kernel in the stream
// has finished; the kernel itself orders its memory accesses after that kernel
// with chain_wait() (mp_chain.cuh) before touching global memory.
template <typename... P, typename... A>
cudaError_t launch_chained(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, A&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// Grid for a kernel whose threads each take one batch of work: every CTA it
// needs, so the block scheduler hands an SM a new CTA as soon as one finishes
// and the last wave ends nearly together (the kernels keep a grid-stride loop,
// so a smaller grid stays correct).
inline int full_grid(int64_t work_ctas) {
  if (work_ctas < 1) work_ctas = 1;
  return (int)(work_ctas < INT32_MAX ? work_ctas : INT32_MAX);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline mp_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MP_OK : MP_ECUDA;
}

}  // namespace mp
