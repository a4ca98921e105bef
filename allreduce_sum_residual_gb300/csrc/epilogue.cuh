// The fused epilogue kernel: rank-order fp32 sum of n partials, residual
// add, RMSNorm.  One-stage uses it with the n partials; stage 2 of the
// two-stage path uses it with n = 1 and the bf16 temporary as the only
// partial (ROCm/aiter #3817 "perf: optimize fused AllReduce + RMSNorm
// (custom_all_reduce)", Technical Details: 1stage decode path, and 2stage
// stage-2 local_device_load_rmsnorm).
//
// Work split.  A row of H columns is P = H/8 packs.  The CTAs of one
// thread-block cluster (S = 1..16 CTAs, consecutive in x) share a row: CTA
// rank q covers packs [q*per_cta, (q+1)*per_cta).  Thread t of a CTA covers
// packs t, t+T, t+2T, ... (VPT of them), so each warp load is 512 contiguous
// bytes.  Every partial element is owned by exactly one thread, which sums
// it over the ranks in order: the sum does not depend on S, T or VPT.
//
// The square sum is reduced warp -> CTA -> cluster.  In the cluster step
// every CTA sends its total into slot q of every peer's shared memory with
// st.async, which completes 4 bytes on the receiver's mbarrier; each CTA
// waits on its own barrier for the S totals (a one-sided wait, no cluster-
// wide barrier) and adds slots 0..S-1 in rank order, so all CTAs of a row
// derive the same scale.  A CTA leaves only after all S totals reached it,
// so no peer writes into an exited CTA.  The wait is bounded: on timeout
// it records AR_ERR_TIMEOUT in the device status word and goes on (the
// outputs of that call are then not valid).
#pragma once

#include "common.cuh"

namespace arn {

// acc = p_0 + p_1 + ... + p_{N-1} for one pack, in fp32, in rank order.
// Used by every path, so one-stage, stage 1 and stage 2 share this exact
// sequence of fp32 adds.
template <int N>
__device__ __forceinline__ void sum_pack_in_rank_order(const uint4 *const (&p)[AR_MAX_RANKS],
                                                       int64_t idx, float (&acc)[8]) {
  uint4 x[N];
#pragma unroll
  for (int k = 0; k < N; ++k) x[k] = ld_ro(p[k] + idx);
  unpack8(x[0], acc);
#pragma unroll
  for (int k = 1; k < N; ++k) {
    float t[8];
    unpack8(x[k], t);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], t[e]);
  }
}

// CL: launched as a thread-block cluster (S > 1 CTAs per row).  A one-CTA-
// per-row launch uses the CL = false instantiation, which has no exchange
// code and so keeps the register count (and the CTAs per SM) of a plain
// row kernel.
// LW (one CTA per row only): load the weight after the sums instead of
// with the inputs.  Its registers are then free while the n partials are
// in flight -- 3 to 11 fewer a thread for n = 4 .. 8 at one pack per
// thread, enough for a second CTA per SM at some row lengths -- at the
// price of one more (L2-resident) load before the output.  The launch plan
// picks whichever is faster for the shape.
template <int N, int VPT, bool CL, bool LW = false>
__global__ void __launch_bounds__(1024 / VPT)
k_fused_epilogue(const __grid_constant__ EpilogueArgs a) {
  static_assert(!(CL && LW), "the late weight load is for one CTA per row");
  __shared__ float red[33];
  __shared__ float cta_totals[kMaxClusterCtas];
  __shared__ uint64_t totals_bar;  // completes when the S cluster totals have arrived
  __shared__ int totals_abort;

  const uint32_t S = CL ? cluster_nctarank() : 1u;
  const uint32_t q = CL ? cluster_ctarank() : 0u;
  const int64_t row = blockIdx.x / S;
  const int c0 = static_cast<int>(q) * a.per_cta;
  const int c1 = min(a.P, c0 + a.per_cta);
  const int64_t base = row * static_cast<int64_t>(a.P);
  const int T = blockDim.x;
  // Checking build: the row exists, this CTA's pack range lies inside the
  // row and its threads cover it, and the cluster rank addresses one of at
  // most kMaxClusterCtas total slots.  Every access below is guarded by it.
  const bool live = in_bounds(row < a.m && c0 >= 0 &&
                                  (c1 <= c0 || (c1 <= a.P && c1 - c0 <= VPT * T)) &&
                                  S <= static_cast<uint32_t>(kMaxClusterCtas) && q < S,
                              a.status);
  if constexpr (CL) {
    if (threadIdx.x == 0) {
      mbar_init(&totals_bar, 1);
      totals_abort = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    cluster_arrive_release();  // this CTA runs and its barrier is ready for its peers
  }

  // Loads first: n partials, the residual and the weight of every pack this
  // thread owns.  Nothing is stored before the last load is issued.  In
  // stage 2 the previous grid is stage 1, and in the one-shot call it is
  // the barrier kernel; neither writes the weight or the residual (and
  // everything before it has completed), so with early_reads those two are
  // read before the wait, the temporary or the partials only after.
  //
  // Before that wait, lanes 0..N of warp 0 ask L2 for this CTA's slice of
  // the n partials and the residual, one bulk prefetch each.  Under
  // programmatic dependent launch this grid's CTAs start while the previous
  // grid still runs, so the DRAM round trip of the first loads overlaps its
  // tail; the loads after the wait then find their lines in L2 (or in
  // flight).  Nothing enters registers or L1 before the wait.
  float r[VPT][8];
  uint4 wv[VPT], rv[VPT];
  if (live && a.prefetch_own && threadIdx.x <= N && c1 > c0) {
    const uint4 *src = threadIdx.x < N ? a.p[threadIdx.x] : a.res;
    prefetch_l2(src + base + c0, static_cast<uint32_t>(c1 - c0) * 16u);
  }
  if (!a.early_reads) pdl_wait_prior_grid();
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = c0 + static_cast<int>(threadIdx.x) + v * T;
    if (live && c < c1) {
      if constexpr (!LW) wv[v] = ld_ro(a.w + c);
      rv[v] = ld_ro(a.res + base + c);
    }
  }
  if (a.early_reads) pdl_wait_prior_grid();
  pdl_launch_dependents();
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = c0 + static_cast<int>(threadIdx.x) + v * T;
    if (live && c < c1) {
      float acc[8], rs[8];
      sum_pack_in_rank_order<N>(a.p, base + c, acc);
      unpack8(rv[v], rs);
      if (a.sum != nullptr) {
        a.sum[2 * (base + c)] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        a.sum[2 * (base + c) + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) r[v][e] = __fadd_rn(acc[e], rs[e]);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) r[v][e] = 0.f;
      wv[v] = make_uint4(0, 0, 0, 0);
    }
  }

  // The row one wave ahead: this CTA's loads have landed, so while it
  // reduces and stores, L2 fetches the slice that the CTA taking its place
  // (a later wave) will read.
  if (live && a.ahead > 0 && threadIdx.x <= N && c1 > c0 && row + a.ahead < a.m) {
    const uint4 *src = threadIdx.x < N ? a.p[threadIdx.x] : a.res;
    prefetch_l2(src + base + a.ahead * a.P + c0, static_cast<uint32_t>(c1 - c0) * 16u);
  }

  // residual_out = bf16(r); square sum of this thread's r.
  float ss = 0.f;
#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = c0 + static_cast<int>(threadIdx.x) + v * T;
    if (live && c < c1) st_stream(a.rout + base + c, pack8(r[v]));
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(r[v][e], r[v][e], ss);
  }

  if constexpr (LW) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = c0 + static_cast<int>(threadIdx.x) + v * T;
      if (live && c < c1) wv[v] = ld_ro(a.w + c);
    }
  }
  float total = block_sum(ss, red);
  if constexpr (CL) {
    cluster_wait_acquire();  // every peer runs and has initialised its barrier
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&totals_bar, S * static_cast<uint32_t>(sizeof(float)));
    if (live && threadIdx.x < S) st_async_remote_f32(&cta_totals[q], threadIdx.x, total, &totals_bar);
    mbar_wait_bounded(&totals_bar, 0, &totals_abort, a.wait_limit_ns, a.status);
    total = 0.f;
    const uint32_t slots = AR_CHECK ? min(S, static_cast<uint32_t>(kMaxClusterCtas)) : S;
    for (uint32_t k = 0; k < slots; ++k) total += cta_totals[k];
  }
  const float inv = rsqrtf(total / a.H + a.eps);

#pragma unroll
  for (int v = 0; v < VPT; ++v) {
    const int c = c0 + static_cast<int>(threadIdx.x) + v * T;
    if (live && c < c1) {
      float w[8], y[8];
      unpack8(wv[v], w);
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] = (r[v][e] * inv) * w[e];
      st_stream(a.out + base + c, pack8(y));
    }
  }
}

// Kernel pointer for (n, vpt, clustered, late weight); n in [1,
// AR_MAX_RANKS], vpt in {1, 2, 4, 8}; late weight only without a cluster.
using EpilogueKernel = void (*)(EpilogueArgs);
EpilogueKernel epilogue_kernel(int n, int vpt, bool clustered, bool late_weight);

}  // namespace arn
