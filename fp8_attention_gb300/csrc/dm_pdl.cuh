// Programmatic dependent launch, device side.
#pragma once

namespace dm {

// The wait returns once every grid this one depends on has completed with its
// writes visible (at once for a kernel launched without the attribute); the
// trigger then lets the next kernel of the stream be scheduled on SMs this
// grid frees, where it runs its own setup and waits here in turn.  A kernel
// touches no global memory before this call.
__device__ __forceinline__ void grid_dependency_sync() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace dm
