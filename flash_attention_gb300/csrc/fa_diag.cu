// fa_diag.cu -- diagnostic kernels for the tests: the two exp2 forms of the softmax evaluated on
// an array (so the FMA-pipe polynomial can be checked against CUDA's exp2f on its own), and one
// bounded wait on an mbarrier that nothing ever completes (so the timeout path -- the wait
// giving up, the status word, the host reading it -- is exercised without breaking a kernel).
#include "fa_common.cuh"
#include "fa_launch.h"

namespace fa {

__global__ void __launch_bounds__(256) ex2_probe_kernel(const float* __restrict__ x,
                                                        float* __restrict__ y_poly,
                                                        float* __restrict__ y_mufu,
                                                        float* __restrict__ y_ref, long long n) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (long long)gridDim.x * blockDim.x) {
    const float v = x[i];
    y_poly[i] = ex2_poly(v);
    y_mufu[i] = ex2(v);
    y_ref[i] = exp2f(v);
  }
}

// One warp waits on a barrier with one expected arrival that never comes.
__global__ void __launch_bounds__(32) wait_probe_kernel(int* status, unsigned long long limit_ns,
                                                        unsigned long long* waited_ns) {
  __shared__ uint64_t bar;
  __shared__ WaitCtl wctl;
  if (threadIdx.x == 0) {
    wait_ctl_init(&wctl, limit_ns);
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const uint64_t t0 = globaltimer();
  const bool ok = mbar_wait(&bar, 0, &wctl);
  const uint64_t t1 = globaltimer();
  __syncthreads();
  if (threadIdx.x == 0) {
    if (waited_ns) *waited_ns = ok ? 0ull : (unsigned long long)(t1 - t0);
    report_abort(&wctl, status);
  }
}

cudaError_t launch_ex2_probe(const float* x, float* y_poly, float* y_mufu, float* y_ref,
                             long long n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  long long blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  ex2_probe_kernel<<<(unsigned)blocks, 256, 0, s>>>(x, y_poly, y_mufu, y_ref, n);
  return cudaGetLastError();
}

cudaError_t launch_wait_probe(int* status, uint64_t limit_ns, unsigned long long* waited_ns,
                              cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(status, (unsigned long long)limit_ns, waited_ns);
  return cudaGetLastError();
}

}  // namespace fa
