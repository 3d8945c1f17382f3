// Failure-detection self-test: a bounded device wait that runs out.
//
// Every wait of this library's kernels (TMA and MMA completions, cluster
// exchanges) is bounded by the plan's timeout; a wait that gives up sets the
// timeout bit of the plan's status word, the kernel returns, and nf_plan_poll
// reports NF_ERR_TIMEOUT.  This one-warp kernel waits, through the same
// bounded wait, on a shared-memory barrier that nothing arrives at (or, as
// the control, one that its own thread has arrived at), with no copy in
// flight, so the path from an expired wait to the host runs without any GPU
// fault.
#include "common.cuh"
#include "kernels.h"

namespace nf {
namespace {

__global__ void selftest_wait_kernel(uint32_t* status, unsigned long long timeout_ns, int arrive,
                                     unsigned long long* waited_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  if (arrive) mbar_arrive(&bar);
  const uint64_t t0 = globaltimer_ns();
  const bool got = mbar_wait(&bar, 0, timeout_ns);
  if (waited_ns) *waited_ns = globaltimer_ns() - t0;
  if (!got) raise_status(status, ST_TIMEOUT);
}

}  // namespace

cudaError_t launch_selftest_wait(uint32_t* status, unsigned long long timeout_ns, int arrive,
                                 unsigned long long* waited_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(status, timeout_ns, arrive, waited_ns);
  return cudaGetLastError();
}

}  // namespace nf
