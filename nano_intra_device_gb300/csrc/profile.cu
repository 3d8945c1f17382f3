// Offline profiler of the layer's nano-operations ("NanoFlow: Towards Optimal
// LLM Serving Throughput", "Kernel Profiling and Interference Modeling").
#include "../../include/nanoflow.h"

extern "C" nf_status nf_profile(const nf_model_shape* shape, int32_t max_tokens, int32_t mean_ctx,
                                const char* out_json) {
  (void)shape; (void)max_tokens; (void)mean_ctx; (void)out_json;
  return NF_ERR_UNSUPPORTED;
}
