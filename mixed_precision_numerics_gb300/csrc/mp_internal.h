// mp_internal.h — host-side helpers shared by the libmpnum translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

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

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline mp_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MP_OK : MP_ECUDA;
}

}  // namespace mp
