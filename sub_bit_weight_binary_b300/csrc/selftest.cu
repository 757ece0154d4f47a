// selftest.cu -- exercises the bounded wait that every kernel of the library
// uses on its mbarriers: one thread waits on a barrier that nothing will
// complete, gives up after the given wall-clock limit, records
// BONSAI_ERR_TIMEOUT in the status word and returns. The GPU context stays
// usable; bonsai_check_async reports and clears the status.
#include "common.cuh"

namespace bonsai {
BONSAI_DEFINE_STATUS(g_status_selftest)

unsigned int read_clear_status_selftest() {
  unsigned int v = 0, z = 0;
  cudaMemcpyFromSymbol(&v, g_status_selftest, sizeof(v));
  cudaMemcpyToSymbol(g_status_selftest, &z, sizeof(z));
  return v;
}

namespace {
__global__ void wait_timeout_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);  // one arrival expected; none will come
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(b, 0, limit_ns)) set_status(BONSAI_ERR_TIMEOUT);
}
}  // namespace

bonsai_status selftest_wait_timeout_launch(uint64_t limit_ns, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>((unsigned long long)limit_ns);
  return cuda_status(cudaGetLastError());
}

}  // namespace bonsai
