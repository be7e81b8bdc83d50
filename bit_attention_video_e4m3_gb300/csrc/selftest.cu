// Failure detection, exercised without a fault: one CTA waits, through the same
// bounded mbarrier wait the attention and prep kernels use, on a barrier that
// nothing arrives on.  The limit expires, the wait raises the CTA's abort flag,
// a second wait sees the flag and returns at once, and the status word of the
// caller's workspace reports a timeout; the context stays usable.
#include "kernels.cuh"
#include "ptx.cuh"

namespace fp8attn {
namespace {

__global__ void __launch_bounds__(64) selftest_wait_kernel(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int ctl[16];
  if (threadIdx.x < 16) ctl[threadIdx.x] = 0;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  const bool first = mbar_wait(smem_u32(&bar), 0, ctl, limit_ns, 0x51u);     // expires
  const bool second = mbar_wait(smem_u32(&bar), 0, ctl, limit_ns, 0x52u);    // sees the abort flag
  __syncthreads();
  if (threadIdx.x == 0 && !first && !second && ctl[0]) {
    atomicExch(status, kStatusTimeout);
    atomicCAS(status + 1, 0, ctl[1]);                                        // where the wait gave up
  }
}

}  // namespace

cudaError_t launch_selftest_wait(int* status, unsigned long long limit_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 64, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace fp8attn
