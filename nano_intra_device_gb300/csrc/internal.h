// Host-side hooks between the C ABI implementation and the profiler.
#pragma once
#include <cuda_runtime.h>

#include <string>
#include <vector>

#include "../../include/nanoflow.h"

namespace nf {
// Step metadata plus every attention nano-batch of the plan, on `grid` CTAs.
nf_status attention_on(nf_plan p, const void* q, const void* kp, const void* vp,
                       const int32_t* bt, const int32_t* sl, void* o, int grid,
                       cudaStream_t st);
// Set the calling thread's nf_last_error() text and return `code`.
nf_status set_last_error(nf_status code, const char* msg);

// One plan of a step profile: the plan, the operations of its traced steps
// (durations averaged over `steps` steps) and its untraced step time.
struct TracedRun {
  nf_plan_opts opts;
  std::vector<nf_trace_entry> ops;
  int steps;
  double step_ms;
};
// Fit the plan search's rates to traced runs of one batch over n_layers
// layers (runs[0] the sequential plan, the rest two-stream plans): the
// interference-free GEMM rate and attention bandwidth, the R -> P table by
// attention SM count, the cost of a cross-stream dependency.  Returns the JSON
// that nf_plan_search reads (empty on invalid input).
std::string fit_step_profile(const nf_model_shape* shape, const nf_batch_desc* batch, int num_sms,
                             int n_layers, const std::vector<TracedRun>& runs);
// The attention nano-batch bounds the plan search generates for n nano-batches
// of this batch (equal token shares, on the 128-token grid from 1024 tokens):
// the plans a step profile measures.
nf_status search_bounds(const nf_model_shape* shape, const nf_batch_desc* batch, int32_t num_sms,
                        int n, int32_t* b);
// The path of the profile registered for this shape (nf_profile_use or
// nf_profile_step), or "".
std::string registered_profile(const nf_model_shape* shape);
}  // namespace nf
