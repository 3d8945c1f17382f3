// Host-side hooks between the C ABI implementation and the profiler.
#pragma once
#include <cuda_runtime.h>

#include "../../include/nanoflow.h"

namespace nf {
// Step metadata plus every attention nano-batch of the plan, on `grid` CTAs.
nf_status attention_on(nf_plan p, const void* q, const void* kp, const void* vp,
                       const int32_t* bt, const int32_t* sl, void* o, int grid,
                       cudaStream_t st);
// Set the calling thread's nf_last_error() text and return `code`.
nf_status set_last_error(nf_status code, const char* msg);
}  // namespace nf
