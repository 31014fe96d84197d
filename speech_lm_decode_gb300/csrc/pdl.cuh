// Programmatic dependent launch (device side): a kernel launched with
// launch_pdl (kernels.h) may start while the previous kernel in the stream is
// still running.  pdl_wait() blocks until that kernel has finished and its
// writes are visible, so every such kernel calls it before it touches
// anything; pdl_trigger() lets the next kernel in the stream begin launching
// once every CTA of this one has called it.
#pragma once

namespace q3 {
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
}  // namespace q3
