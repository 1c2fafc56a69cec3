// Self-test of the kernels' failure detection: a bounded wait that runs out.
//
// One CTA initialises an mbarrier that nothing will ever complete and waits on
// it with the same bounded wait the attention kernels use, but with a caller
// chosen limit. The wait gives up, records kErrSelftest in this translation
// unit's error word and the kernel returns; the host then reads the word through
// duo_device_error(). No fault, trap or endless loop is involved.
#include "duo_device.cuh"

namespace duo {
namespace {

__device__ unsigned int g_selftest_err;

__global__ void bounded_wait_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 0;; ++it) {
      if (mbar_try_wait(&bar, 0)) break;  // never true: nothing arrives
      if ((it & 255u) == 255u && global_timer_ns() - t0 > limit_ns) {
        atomicOr(&g_selftest_err, kErrSelftest);
        break;
      }
    }
  }
  __syncthreads();
}

}  // namespace

cudaError_t launch_selftest_wait(uint64_t limit_ns, cudaStream_t stream) {
  bounded_wait_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t selftest_read_clear_error(uint32_t* code) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_selftest_err, sizeof(v));
  if (e != cudaSuccess) return e;
  *code = v;
  if (v) {
    v = 0;
    e = cudaMemcpyToSymbol(g_selftest_err, &v, sizeof(v));
  }
  return e;
}

}  // namespace duo
