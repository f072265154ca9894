// wait_timeout_probe.cu -- test support for tests/test_wait_timeout_gpu.py
// (built by that test with nvcc; not part of the library).
//
// Exercises the library's bounded on-chip wait (fm::mbar_wait in
// fm_common.cuh) on an mbarrier that nothing ever arrives on: the wait must
// give up after its time limit, set the timeout bit in the status word it is
// given and return false, and a second waiter of the same CTA must then leave
// too -- so a kernel whose pipeline stalls returns an error status instead of
// hanging the GPU.
#include "fm_common.cuh"

extern "C" __global__ void wait_probe_kernel(unsigned int* status, int* results, unsigned long long* elapsed_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    fm::mbar_init(&bar, 1);  // one arrival expected; none is ever made
    abort_flag = 0;
    fm::fence_mbar_init();
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) {
    const uint64_t t0 = fm::globaltimer();
    const bool ok = fm::mbar_wait(&bar, 0, &abort_flag, status);
    results[threadIdx.x >> 5] = ok ? 1 : 0;
    elapsed_ns[threadIdx.x >> 5] = fm::globaltimer() - t0;
  }
}

extern "C" int launch_wait_probe(unsigned int* status, int* results, unsigned long long* elapsed_ns,
                                 void* stream) {
  wait_probe_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(status, results, elapsed_ns);
  return static_cast<int>(cudaGetLastError());
}
