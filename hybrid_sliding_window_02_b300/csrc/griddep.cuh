// griddep.cuh -- programmatic dependent launch, device side.
//
// A kernel launched with programmatic stream serialisation may start while
// the kernel before it on the stream is still running.  grid_dep_wait()
// returns once that kernel has completed and its memory operations are
// visible, so every load and store of a buffer it may have written (or may
// still read) comes after the call.  grid_dep_launch() lets the next such
// kernel on the stream be scheduled early; it changes nothing for the
// kernel that calls it.
#pragma once

namespace swa {

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace swa
