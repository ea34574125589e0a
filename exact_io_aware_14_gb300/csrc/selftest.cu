// Self-test of the bounded wait every kernel of the library uses (mbar_wait
// in ptx.cuh): one block of two warps waits on mbarrier phases that nothing
// ever completes.  Warp 0 gives up after the caller's limit, sets the
// block's abort flag and records a timeout in the status word the way the
// attention kernels do; warp 1, waiting with the library's full 2 s limit,
// must see that flag and give up at once.  Nothing faults, traps or spins
// without a limit; the kernel returns and the context stays usable.
#include <cuda_runtime.h>

#include "launch.h"
#include "ptx.cuh"

namespace attn {
namespace {

__device__ uint32_t g_selftest_status;

constexpr uint64_t kFullLimitNs = 2000000000ull;

__global__ void __launch_bounds__(64) wait_timeout_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bars[2];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bars + 0, 1);  // one arrival would complete phase 0; none comes
    mbar_init(bars + 1, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  volatile int* abort = &abort_flag;
  bool ok = mbar_wait(bars + warp, 0, abort, warp == 0 ? limit_ns : kFullLimitNs);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok && (threadIdx.x & 31) == 0) atomicCAS(&g_selftest_status, 0u, ((1u + warp) << 8) | kDevTimeout);
}

}  // namespace

cudaError_t launch_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 64, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t fetch_status_selftest(cudaStream_t stream, uint32_t* out) {
  uint32_t zero = 0;
  cudaError_t e =
      cudaMemcpyFromSymbolAsync(out, g_selftest_status, sizeof(uint32_t), 0, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess)
    e = cudaMemcpyToSymbolAsync(g_selftest_status, &zero, sizeof(uint32_t), 0, cudaMemcpyHostToDevice, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  return e;
}

}  // namespace attn
