// ptx_pdl.cuh -- programmatic dependent launch: a kernel launched with the
// programmatic-serialization attribute may start (set up its barriers and
// tensor memory) while the launch before it finishes, and waits for that
// launch before it touches the data it produced.
#pragma once

namespace mha {

// Launches that follow this one on the stream may be scheduled once every
// CTA of this grid has executed this (or exited).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the launches this one depends on have completed and their
// memory operations are visible (returns at once without such launches).
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace mha
