// Self-tests and a measurement helper.  (1) The software exp2 of
// exp2_poly.cuh evaluated on an array, so that its error can be measured
// against a reference.  (2) A plain streaming read of a buffer, whose
// duration gives the HBM read rate a read-bound kernel is measured against.
// (3) The bounded wait every kernel of the library uses (mbar_wait in
// ptx.cuh): one block of two warps waits on mbarrier phases that nothing
// ever completes.  Warp 0 gives up after the caller's limit, sets the
// block's abort flag and records a timeout in the status word the way the
// attention kernels do; warp 1, waiting with the library's full 2 s limit,
// must see that flag and give up at once.  Nothing faults, traps or spins
// without a limit; the kernel returns and the context stays usable.
#include <cuda_runtime.h>

#include "exp2_poly.cuh"
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

// y = 2^x by the software exp2 of exp2_poly.cuh, one pair per thread (an odd
// last element is paired with 0).
__global__ void __launch_bounds__(256) exp2_poly_kernel(const float* __restrict__ x, float* __restrict__ y,
                                                        long long n) {
  const long long i = 2 * (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const bool two = i + 1 < n;
  const float2 r = exp2_poly2(make_float2(x[i], two ? x[i + 1] : 0.f));
  y[i] = r.x;
  if (two) y[i + 1] = r.y;
}

// Reads n16 16-byte words once, eight loads in flight per thread
// (grid-stride), and folds them into one word per block so that no load can
// be dropped; the folds meet in *sink with one atomic per block.
__global__ void __launch_bounds__(256) read_probe_kernel(const uint4* __restrict__ buf, long long n16,
                                                         unsigned long long* __restrict__ sink) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  uint32_t acc = 0;
  for (; i + 7 * stride < n16; i += 8 * stride) {
    uint4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) v[k] = __ldcs(buf + i + k * stride);
#pragma unroll
    for (int k = 0; k < 8; ++k) acc ^= v[k].x ^ v[k].y ^ v[k].z ^ v[k].w;
  }
  for (; i < n16; i += stride) {
    const uint4 v = __ldcs(buf + i);
    acc ^= v.x ^ v.y ^ v.z ^ v.w;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
  __shared__ uint32_t s_acc[8];
  if ((threadIdx.x & 31) == 0) s_acc[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t a = 0;
    for (int w = 0; w < 8; ++w) a ^= s_acc[w];
    atomicXor(sink, static_cast<unsigned long long>(a));
  }
}

}  // namespace

cudaError_t launch_read_probe(const void* buf, long long n16, unsigned long long* sink, cudaStream_t stream) {
  int dev = 0, n_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  read_probe_kernel<<<n_sm * 8, 256, 0, stream>>>(static_cast<const uint4*>(buf), n16, sink);
  return cudaGetLastError();
}

cudaError_t launch_selftest_exp2_poly(const float* x, float* y, long long n, cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const long long pairs = (n + 1) / 2;
  exp2_poly_kernel<<<static_cast<unsigned>((pairs + 255) / 256), 256, 0, stream>>>(x, y, n);
  return cudaGetLastError();
}

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
