// mp_chain.cuh — programmatic dependent launch between consecutive kernels of
// a stream.  The library launches its kernels with programmatic stream
// serialization allowed (launch_chained in mp_internal.h), so a kernel's CTAs
// may be scheduled while the previous kernel in the stream is still finishing.
// Every such kernel calls chain_wait() before it touches global memory: the
// wait returns once the previous grid has completed and its writes are
// visible, exactly the ordering a plain stream launch gives.  chain_release()
// lets the next kernel's launch begin; it carries no memory ordering.
#pragma once

namespace mp {

__device__ __forceinline__ void chain_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void chain_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

}  // namespace mp
