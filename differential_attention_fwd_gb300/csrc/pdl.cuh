// pdl.cuh -- programmatic dependent launch between the decode passes.
#pragma once

namespace diffattn {

// The next kernel on the stream, if launched with programmatic stream
// serialisation, may start its blocks once every CTA of this grid has
// executed this (or exited).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the grids this one depends on have completed and their memory
// writes are visible (returns at once without such a dependency).
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace diffattn
