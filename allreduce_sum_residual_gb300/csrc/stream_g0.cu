// Instantiations of the streamed epilogue kernel for n = 1 .. 4 inputs.
#include "stream_epilogue.cuh"

namespace arn {

#define ARN_ROW(N) {&k_stream_epilogue<N, 1>, &k_stream_epilogue<N, 2>, \
                    &k_stream_epilogue<N, 4>, &k_stream_epilogue<N, 8>}

StreamKernel stream_kernel_group0(int n, int vpt_log2) {
  static const StreamKernel table[4][4] = {ARN_ROW(1), ARN_ROW(2), ARN_ROW(3), ARN_ROW(4)};
  return table[n - 1][vpt_log2];
}

}  // namespace arn

namespace arn {

// A wait on an mbarrier that nothing ever completes: it must give up after
// limit_ns and record AR_ERR_TIMEOUT (exercises the bounded-wait path).
__global__ void k_bounded_wait_selftest(uint64_t limit_ns, int *status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  mbar_wait_bounded(&bar, 0, &abort_flag, limit_ns, status);
}

cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, int *status, cudaStream_t s) {
  k_bounded_wait_selftest<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace arn

namespace arn {

// One failing bounds check and nothing else: in the checking build it
// records AR_ERR_BOUNDS, in the normal build the check compiles away.
__global__ void k_bounds_selftest(int *status) { (void)in_bounds(false, status); }

cudaError_t launch_bounds_selftest(int *status, cudaStream_t s) {
  k_bounds_selftest<<<1, 1, 0, s>>>(status);
  return cudaGetLastError();
}

}  // namespace arn
