// Stage 1 of the two-stage path: a flat reduce of every 16-byte pack across
// the n ranks, rounded to bf16 into the temporary buffer.
//
// ROCm/aiter #3817 "perf: optimize fused AllReduce + RMSNorm
// (custom_all_reduce)", Technical Details, 2stage, reduce-scatter: one
// thread owns one 16-byte pack, sums it over the ranks in fp32 in pointer
// order, rounds the sum to bf16 and stores it, with neither shared memory
// nor a block barrier.  Stage-1 launch config: 256-thread blocks.
//
// A launch covers the pack range [begin, end) and stores every sum into
// ndst destinations at the same position.  The two-stage path uses the
// whole range and one destination (this GPU's temporary).  One rank of a
// reduce-scatter uses its slice and one destination per rank -- the page's
// stores straight into each rank's temporary; across GPUs those would be
// peer-mapped buffers.  The grid is a multiple of the SM count and
// strides over the range; each step of a thread handles U packs 256 apart,
// issuing all U*n loads before the first add.  U = 1 ships: on GB300 it
// beat U = 2 and 4 at every measured shape (two-stage 1-12 % faster; the
// most at a few hundred rows, where U = 1 gives twice the CTAs).
#include "epilogue.cuh"

namespace arn {

constexpr int kReduceThreads = 256;

template <int N, int U>
__global__ void __launch_bounds__(kReduceThreads)
k_reduce_flat(const __grid_constant__ ReduceArgs a) {
  // Previous grids first, then let stage 2 be scheduled; stage 2 waits for
  // this grid's results itself (griddepcontrol.wait) before reading them.
  // Before the wait, one thread per partial asks L2 for the CTA's first
  // step of packs (a bulk prefetch), so that the first DRAM round trip
  // overlaps the previous grid's tail.
  // Checking build: a valid destination count and pack range.
  const bool live = in_bounds(a.ndst >= 1 && a.ndst <= AR_MAX_RANKS && a.begin >= 0 &&
                                  a.begin <= a.end,
                              a.status);
  if (live && a.prefetch && threadIdx.x < N) {
    const int64_t b0 = a.begin + static_cast<int64_t>(blockIdx.x) * kReduceThreads * U;
    if (b0 < a.end) {
      const int64_t cnt = a.end - b0 < kReduceThreads * U ? a.end - b0 : kReduceThreads * U;
      prefetch_l2(a.p[threadIdx.x] + b0, static_cast<uint32_t>(cnt) * 16u);
    }
  }
  pdl_wait_prior_grid();
  pdl_launch_dependents();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kReduceThreads * U;
  for (int64_t i0 = a.begin + static_cast<int64_t>(blockIdx.x) * kReduceThreads * U + threadIdx.x;
       live && i0 < a.end; i0 += stride) {
    float acc[U][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t idx = i0 + static_cast<int64_t>(u) * kReduceThreads;
      if (idx < a.end) sum_pack_in_rank_order<N>(a.p, idx, acc[u]);
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t idx = i0 + static_cast<int64_t>(u) * kReduceThreads;
      if (idx < a.end) {
        const uint4 v = pack8(acc[u]);
        for (int d = 0; d < a.ndst; ++d) st_stream(a.dst[d] + idx, v);
      }
    }
  }
}

constexpr int kReduceUnroll = 1;

using ReduceKernel = void (*)(ReduceArgs);

static ReduceKernel reduce_kernel(int n) {
#define ARN_R(N) &k_reduce_flat<N, kReduceUnroll>
  static const ReduceKernel table[AR_MAX_RANKS] = {
      ARN_R(1), ARN_R(2), ARN_R(3), ARN_R(4), ARN_R(5), ARN_R(6), ARN_R(7), ARN_R(8),
      ARN_R(9), ARN_R(10), ARN_R(11), ARN_R(12), ARN_R(13), ARN_R(14), ARN_R(15), ARN_R(16)};
#undef ARN_R
  return table[n - 1];
}

// Launch stage 1 over the pack range of `a`; `sms` is the device's SM count.
cudaError_t launch_reduce_flat(const ReduceArgs &a, int n, int sms, cudaStream_t stream) {
  const int64_t per_block = static_cast<int64_t>(kReduceThreads) * kReduceUnroll;
  int64_t blocks = (a.end - a.begin + per_block - 1) / per_block;
  const int64_t cap = static_cast<int64_t>(sms) * (2048 / kReduceThreads);
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kReduceThreads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, reduce_kernel(n), a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace arn
