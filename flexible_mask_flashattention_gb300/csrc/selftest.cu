// Self-test of the kernels' failure path: the bounded mbarrier wait.
//
// Every wait in the persistent kernels is bounded (ptx.cuh, mbar_wait): after
// kWaitLimitNs of %globaltimer it records a timeout bit in a status word,
// raises the CTA's abort flag so that the CTA's other waits give up too, and
// returns false, so that the kernel can release what it holds and return.
// This kernel runs that helper on barriers that nothing ever arrives at:
// thread 0 of each block times out, the other threads of the block see the
// abort flag and give up.  No trap, no fault: the context stays usable.
#include "ffa_internal.h"
#include "ptx.cuh"

namespace ffa {
namespace {

__global__ void bounded_wait_selftest_kernel(uint32_t* status, uint32_t* gave_up) {
  __shared__ uint64_t never[2];
  __shared__ int abort;
  if (threadIdx.x == 0) {
    mbar_init(&never[0], 1);
    mbar_init(&never[1], 1);
    abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* ab = &abort;
  // thread 0 waits for phase 0 of a barrier nobody arrives at: it times out
  // after kWaitLimitNs and records kStatusTimeoutOther; every other thread
  // waits on the second such barrier and leaves once the abort flag is up
  const bool ok = threadIdx.x == 0 ? mbar_wait(&never[0], 0, ab, status, kStatusTimeoutOther)
                                   : mbar_wait(&never[1], 0, ab, status, kStatusTimeoutOther);
  if (!ok) atomicAdd(gave_up, 1u);
}

}  // namespace
}  // namespace ffa

using namespace ffa;

extern "C" ffa_status ffa_selftest_bounded_wait(void* stream, uint32_t* status_out, uint32_t* gave_up_out) {
  if (!status_out || !gave_up_out) return FFA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* dev = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&dev), 2 * sizeof(uint32_t), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(dev, 0, 2 * sizeof(uint32_t), s);
  if (e == cudaSuccess) {
    bounded_wait_selftest_kernel<<<1, 64, 0, s>>>(dev, dev + 1);
    e = cudaGetLastError();
  }
  uint32_t host[2] = {0, 0};
  if (e == cudaSuccess) e = cudaMemcpyAsync(host, dev, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (dev) cudaFreeAsync(dev, s);
  *status_out = host[0];
  *gave_up_out = host[1];
  return cuda_status(e);
}
