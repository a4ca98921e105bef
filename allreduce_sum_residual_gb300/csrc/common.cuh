// Device-side building blocks shared by the ar_rmsnorm kernels (sm_103a).
//
// A "pack" is 16 bytes = 8 bf16: the unit every thread loads and stores, so
// that a warp moves 512 contiguous bytes per instruction.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ar_rmsnorm.h"

// The checking build (nvcc -DAR_CHECK=1, see _build.py) compiles device-side
// bounds checks into the kernels: every index a kernel derives from its
// launch shape (row, pack range, cluster rank, shared-memory slot, rank
// count) is tested against the buffer or array it addresses before use.
#ifndef AR_CHECK
#define AR_CHECK 0
#endif

namespace arn {

// `ok` in the checking build, where a false `ok` also records AR_ERR_BOUNDS
// in the device status word; always true in the normal build (the test
// compiles away).  The caller skips the access that `ok` guards: a thread
// never leaves its kernel early, because the barriers of its CTA (or
// cluster) would then wait for it forever.
__device__ __forceinline__ bool in_bounds(bool ok, int *status) {
#if AR_CHECK
  if (!ok && status != nullptr) atomicExch(status, AR_ERR_BOUNDS);
  return ok;
#else
  (void)ok;
  (void)status;
  return true;
#endif
}

constexpr int kPackElems = 8;            // bf16 per 16-byte pack
constexpr int kMaxClusterCtas = 16;      // widest row split (non-portable cluster)
constexpr int kMaxPacksPerCta = 1024;    // 8192 columns held in registers per CTA

// Kernel parameters of the fused epilogue (one-stage, and stage 2 with n = 1).
struct EpilogueArgs {
  const uint4 *p[AR_MAX_RANKS];  // partial k, [m, H/8] packs, rank order
  const uint4 *res;              // residual [m, H/8]
  const uint4 *w;                // weight [H/8]
  uint4 *out;                    // [m, H/8]
  uint4 *rout;                   // residual_out [m, H/8]
  float4 *sum;                   // optional fp32 sum [m, H/4] float4s, or null
  int64_t m;                     // rows
  int P;                         // packs per row = H / 8
  int per_cta;                   // packs of a row one CTA covers
  float H;                       // columns, as the divisor of the mean
  float eps;
  int early_reads;               // weight and residual may be read before the
                                 // wait on the previous grid (stage 2 only)
  int prefetch_own;              // prefetch this CTA's slice of its row into L2
                                 // before the wait on the previous grid
  int64_t ahead;                 // > 0: after its sums, prefetch the same slice of
                                 // row + ahead into L2 (the row the CTA that takes
                                 // this one's place will read); 0: none
  uint64_t wait_limit_ns;        // bound of the cluster-exchange wait
  int *status;                   // device status word (AR_ERR_TIMEOUT on timeout)
};

// Kernel parameters of stage 1 (flat reduce of every pack across ranks).
// Stage 1 reduces the packs [begin, end) and stores each bf16 sum at the
// same position of every destination dst[0 .. ndst-1] (ndst = 1 for the
// two-stage temporary; one per rank for the all-gather by stores).
struct ReduceArgs {
  const uint4 *p[AR_MAX_RANKS];
  uint4 *dst[AR_MAX_RANKS];
  int ndst;
  int prefetch;   // prefetch each CTA's first packs into L2 before the wait
  int64_t begin;
  int64_t end;
  int *status;    // device status word (checking build: AR_ERR_BOUNDS)
};

// --- bf16 <-> fp32 ----------------------------------------------------------

// Widen the 8 bf16 of a pack: a bf16 is the top half of an fp32.
__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Round 8 fp32 to bf16 (nearest even, one cvt.rn.bf16x2.f32 per pair).
__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t *>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// --- global memory ------------------------------------------------------------

// Read-only 16-byte load through the non-coherent path; the data is never
// written during the kernel, which lets the compiler hoist these freely.
__device__ __forceinline__ uint4 ld_ro(const uint4 *p) { return __ldg(p); }

// Streaming 16-byte store: the outputs are not re-read by this kernel.
__device__ __forceinline__ void st_stream(uint4 *p, const uint4 &v) { __stcs(p, v); }

// Ask L2 to fetch `bytes` of global memory at `p` (both multiples of 16)
// without waiting for it and without touching registers or L1
// (cp.async.bulk.prefetch, the bulk-copy engine's prefetch form).  L2 is
// the point of coherence of this GPU's memory, so a line prefetched before
// another grid writes it is updated by that write: a prefetch may run
// before griddepcontrol.wait.  Only for memory of this GPU.
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// --- reductions -----------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Sum of `v` over the CTA, returned to every thread.  `scratch` holds 33
// floats and is used once per kernel.  Butterfly within each warp, one slot
// per warp; with up to 8 warps every thread then adds the slots itself (one
// barrier), with more warp 0 folds them and publishes the total (two
// barriers, fewer shared-memory reads per thread).  The square-sum order is
// not part of the bit-exact contract.
__device__ __forceinline__ float block_sum(float v, float *scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  if (nwarps <= 8) {
    float t = 0.f;
    for (int i = 0; i < nwarps; ++i) t += scratch[i];
    return t;
  }
  if (warp == 0) {
    float t = lane < nwarps ? scratch[lane] : 0.f;
    t = warp_sum(t);
    if (lane == 0) scratch[32] = t;
  }
  __syncthreads();
  return scratch[32];
}

// --- programmatic dependent launch ---------------------------------------------------
//
// Every kernel of the library is launched with programmatic stream
// serialization, so it may be scheduled before the previous grid in the
// stream has finished.  Each kernel therefore (1) waits for the previous
// grids (griddepcontrol.wait) before it reads or writes global memory --
// which keeps plain stream-order semantics whatever ran before -- and only
// then (2) allows the next kernel to be scheduled.  Because of that order,
// when a kernel starts every grid before its predecessor has completed.

// Let the next kernel in the stream start its prologue while this grid runs.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait until the preceding grids in the stream have completed and their
// writes are visible.  Returns at once when this grid was launched without
// a programmatic dependency.
__device__ __forceinline__ void pdl_wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// --- thread-block clusters --------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// Split cluster barrier.  arrive.release at kernel start (after this CTA
// has initialised what its peers will touch), wait.acquire right before the
// first access to a peer's shared memory -- which must not happen before
// every CTA of the cluster runs.
__device__ __forceinline__ void cluster_arrive_release() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acquire() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// --- mbarriers (PTX) ---------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait until phase `parity` of `bar` completes, for at most limit_ns.  On
// timeout: record AR_ERR_TIMEOUT, raise the CTA's abort flag, return false.
// Also returns false (without waiting) once another thread raised abort.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  volatile int *abort_flag, uint64_t limit_ns,
                                                  int *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1;
      if (status) atomicExch(status, AR_ERR_TIMEOUT);
      return false;
    }
  }
}

// Store a float into the shared memory of CTA `rank` of this cluster, at the
// address that `local_slot` has in this CTA, completing 4 transaction bytes
// on that CTA's mbarrier at the address of `local_bar` (st.async): the
// receiver learns of the value by waiting on its own barrier, without a
// cluster-wide barrier.
__device__ __forceinline__ void st_async_remote_f32(float *local_slot, uint32_t rank, float v,
                                                    uint64_t *local_bar) {
  uint32_t ra, rb;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(smem_addr(local_slot)), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rb) : "r"(smem_addr(local_bar)), "r"(rank));
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];" ::"r"(ra),
               "f"(v), "r"(rb)
               : "memory");
}

}  // namespace arn
