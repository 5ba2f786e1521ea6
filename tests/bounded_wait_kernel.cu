// bounded_wait_kernel.cu -- test harness for the library's bounded mbarrier
// wait (pkv_device.cuh): one CTA waits on a barrier that nothing arrives on.
// The wait must give up after its time limit, set PKV_DEVERR_WAIT_TIMEOUT in
// the error word and let the kernel return, leaving the context usable.
#include <cuda_runtime.h>

#include "pkv_device.cuh"

namespace {

__global__ void wait_on_silent_barrier(unsigned int* err, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    pkv::mbar_init(&bar, 1);
    pkv::fence_barrier_init();
  }
  __syncthreads();
  const bool ok = pkv::mbar_wait(&bar, 0, err);  // no arrival: phase 0 never completes
  if (threadIdx.x == 0) *status = ok ? 1 : 2;
}

__global__ void wait_on_completed_barrier(unsigned int* err, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    pkv::mbar_init(&bar, 1);
    pkv::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) pkv::mbar_arrive(&bar);
  const bool ok = pkv::mbar_wait(&bar, 0, err);
  if (threadIdx.x == 0) *status = ok ? 1 : 2;
}

}  // namespace

// silent != 0: wait on a barrier nobody arrives on; else on one that completes.
// err and status are device pointers; returns the launch status.
extern "C" __attribute__((visibility("default"))) int bounded_wait_probe(int silent, unsigned int* err, int* status, void* stream) {
  auto s = static_cast<cudaStream_t>(stream);
  if (silent)
    wait_on_silent_barrier<<<1, 64, 0, s>>>(err, status);
  else
    wait_on_completed_barrier<<<1, 64, 0, s>>>(err, status);
  return static_cast<int>(cudaGetLastError());
}
