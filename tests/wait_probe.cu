// wait_probe.cu — a test-only kernel for the bounded mbarrier wait the
// library's pipelines use (mbar_wait_bounded in mp_device.cuh).  One thread
// initialises a shared-memory barrier expecting one arrival, arrives on it or
// not, and waits for its first phase.  Without the arrival nothing can ever
// complete that phase: the wait must give up after its poll limit (about two
// seconds) and report it, leaving the context usable.  No memory is touched
// but the two result words.
#include <cstdint>

#include "mp_device.cuh"

namespace {

__global__ void k_wait_probe(int arrive, uint32_t* ok, unsigned long long* elapsed_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mp::mbar_init(&bar, 1);
  mp::fence_mbar_init();
  if (arrive) mp::mbar_arrive(&bar);
  unsigned long long t0, t1;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  const bool done = mp::mbar_wait_bounded(&bar, 0);
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
  *ok = done ? 1u : 0u;
  *elapsed_ns = t1 - t0;
}

}  // namespace

extern "C" int wait_probe(int arrive, uint32_t* d_ok, unsigned long long* d_elapsed_ns, void* stream) {
  k_wait_probe<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(arrive, d_ok, d_elapsed_ns);
  return cudaGetLastError() == cudaSuccess ? 0 : 1;
}
