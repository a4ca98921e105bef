// The fused epilogue for many rows: a persistent, warp-specialised kernel
// that streams rows through shared memory with bulk asynchronous copies.
//
// Same arithmetic as k_fused_epilogue (rank-order fp32 sum of n partials,
// residual add, RMSNorm; ROCm/aiter #3817 "perf: optimize fused AllReduce +
// RMSNorm (custom_all_reduce)", Technical Details, 1stage), same ownership of
// every element by one thread, so the sum and residual_out are bit-identical
// to it.  What changes is how bytes reach the SM:
//
//   * one producer warp (lane 0) issues cp.async.bulk copies (the 1-D TMA
//     path) of a row tile of every input -- the n partials and the residual,
//     T_c packs each -- into a ring of S shared-memory slots, completing on
//     the slot's "full" mbarrier with a transaction-byte count;
//   * C consumer warps (T_c = 32*C threads) wait on "full", read their pack
//     of each input from shared memory, keep r = sum + residual in
//     registers, and release the slot on its "empty" mbarrier;
//   * after the last tile of a row the consumers reduce the square sum among
//     themselves (named barrier 1), then store residual_out and out.
//
// The CTA is persistent: CTA b handles rows b, b + G, b + 2G, ...  The
// producer runs up to S tiles ahead, across row boundaries, so the next
// row's loads overlap this row's reduction and stores, and the bytes in
// flight per SM are bounded by shared memory rather than by registers.
//
// Every mbarrier wait is bounded (wait_limit_ns of %globaltimer): on timeout
// the waiting thread records AR_ERR_TIMEOUT in a device status word, raises
// the CTA's abort flag and stops; the producer stops issuing and drains the
// copies it has in flight (again bounded) before the CTA exits.
#pragma once

#include "common.cuh"

namespace arn {

struct StreamArgs {
  const uint4 *src[AR_MAX_RANKS + 1];  // partials in rank order, then the residual
  const uint4 *w;                      // weight [H/8]
  uint4 *out;                          // [m, H/8]
  uint4 *rout;                         // [m, H/8]
  float4 *sum;                         // optional fp32 sum, or null
  int64_t m;
  int P;                               // packs per row
  int tiles;                           // tiles per row: ceil(P / T_c)
  int stages;                          // ring slots
  float H;
  float eps;
  uint64_t wait_limit_ns;              // bound of every mbarrier wait
  int *status;                         // device status word (AR_ERR_TIMEOUT on timeout)
  int prefetch_first;                  // L2 prefetch of the CTA's first row before
                                       // the wait on the previous grid
  int prefetch_next;                   // L2 prefetch of the CTA's next row while it
                                       // streams the current one
  int smem_bytes;                      // dynamic shared memory of the launch
};

// --- bulk copy (PTX) -----------------------------------------------------------

// 1-D bulk copy global -> shared, completing `bytes` on `bar`.  Addresses and
// size are multiples of 16 bytes.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void named_barrier_sync(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// --- the kernel -------------------------------------------------------------------

// Dynamic shared memory: [stages][N + 1][T_c] uint4 slots, then 2*stages
// mbarriers, then the reduction scratch and the abort flag.
constexpr int kStreamMaxConsumers = 512;

template <int N, int VPT>
__global__ void __launch_bounds__(32 + kStreamMaxConsumers, 1)
k_stream_epilogue(const __grid_constant__ StreamArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int Tc = static_cast<int>(blockDim.x) - 32;
  const int S = a.stages;
  uint4 *slots = reinterpret_cast<uint4 *>(smem);
  const size_t slot_packs = static_cast<size_t>(N + 1) * Tc;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(S) * slot_packs * 16);
  uint64_t *empty = full + S;
  float *red = reinterpret_cast<float *>(empty + S);  // [2][32]
  volatile int *abort_flag = reinterpret_cast<volatile int *>(red + 64);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = Tc >> 5;
  // Checking build: the ring, its barriers and the reduction scratch fit
  // the launch's shared memory, the consumers are whole warps (at most
  // kStreamMaxConsumers, one scratch slot each), and the row's tiles fit
  // the template's VPT.  When this fails nothing below touches memory.
  const bool live = in_bounds(
      Tc >= 32 && Tc % 32 == 0 && Tc <= kStreamMaxConsumers && S >= 1 && a.tiles >= 1 &&
          a.tiles <= VPT && static_cast<int64_t>(a.tiles) * Tc >= a.P &&
          static_cast<int64_t>(S) * slot_packs * 16 + 16 * S + 64 * 4 + 4 <= a.smem_bytes,
      a.status);
  if (live && threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int64_t G = gridDim.x;
  const int V = a.tiles;
  // Before the wait: lanes 0..N of the producer warp ask L2 for this CTA's
  // first row of every input.  A CTA that starts while the previous grid's
  // last CTAs still run (on an SM they left) overlaps its first DRAM round
  // trip with their tail.
  if (live && a.prefetch_first && warp == 0 && lane <= N && blockIdx.x < a.m)
    prefetch_l2(a.src[lane] + static_cast<int64_t>(blockIdx.x) * a.P,
                static_cast<uint32_t>(a.P) * 16u);
  pdl_wait_prior_grid();

  if (warp == 0) {
    // ---------------- producer
    if (lane != 0 || !live) return;
    int64_t t = 0;
    for (int64_t row = blockIdx.x; row < a.m; row += G) {
      // The next row of this CTA, one row ahead of the ring's copies.
      if (a.prefetch_next && row + G < a.m) {
#pragma unroll 1
        for (int j = 0; j <= N; ++j)
          prefetch_l2(a.src[j] + (row + G) * a.P, static_cast<uint32_t>(a.P) * 16u);
      }
      for (int v = 0; v < V; ++v, ++t) {
        const int s = static_cast<int>(t % S);
        const int64_t k = t / S;
        if (k > 0 && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>((k - 1) & 1), abort_flag,
                                        a.wait_limit_ns, a.status))
          goto drain;
        if (*abort_flag) goto drain;
        const int c0 = v * Tc;
        const int packs = min(Tc, a.P - c0);
        const uint32_t bytes = static_cast<uint32_t>(packs) * 16u;
        mbar_arrive_expect_tx(&full[s], bytes * (N + 1));
        uint4 *dst = slots + static_cast<size_t>(s) * slot_packs;
        const int64_t off = row * a.P + c0;
#pragma unroll
        for (int j = 0; j <= N; ++j) bulk_g2s(dst + static_cast<size_t>(j) * Tc, a.src[j] + off, bytes, &full[s]);
      }
    }
    // This CTA is near its end: the next grid may be scheduled.  (Released
    // late, so that its CTAs do not sit on these SMs while the ring runs.)
    pdl_launch_dependents();
  drain:
    // Every slot's last issued fill must land before the CTA may exit.
    for (int s = 0; s < S; ++s) {
      if (t > s) {
        const int64_t last = ((t - 1 - s) / S) * S + s;  // last tile issued into slot s
        mbar_wait_bounded(&full[s], static_cast<uint32_t>((last / S) & 1), abort_flag,
                          a.wait_limit_ns, a.status);
      }
    }
    return;
  }

  // ---------------- consumers
  const int tc = static_cast<int>(threadIdx.x) - 32;
  const int cw = warp - 1;
  // The weight is the same for every row: up to 4 tiles it stays in
  // registers for the CTA's lifetime; wider rows re-read it (L1 hits).
  constexpr int kWRegs = VPT <= 4 ? VPT : 1;
  uint4 wv[kWRegs];
#pragma unroll
  for (int v = 0; v < kWRegs; ++v) {
    const int c = v * Tc + tc;
    wv[v] = (live && VPT <= 4 && v < V && c < a.P) ? ld_ro(a.w + c) : make_uint4(0, 0, 0, 0);
  }

  int64_t t = 0;
  int parity_row = 0;
  for (int64_t row = blockIdx.x; live && row < a.m; row += G, parity_row ^= 1) {
    const int64_t base = row * a.P;
    if (row + G >= a.m) pdl_launch_dependents();  // last row of this CTA
    float r[VPT][8];
    float ss = 0.f;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
#pragma unroll
      for (int e = 0; e < 8; ++e) r[v][e] = 0.f;
      if (v < V) {
        const int s = static_cast<int>(t % S);
        // After an abort the consumers keep walking the rows without waiting
        // or touching memory, so that every one of them still reaches each
        // named barrier below.
        const bool ok = mbar_wait_bounded(&full[s], static_cast<uint32_t>((t / S) & 1), abort_flag,
                                          a.wait_limit_ns, a.status);
        const int c = v * Tc + tc;
        if (ok && c < a.P) {
          const uint4 *slot = slots + static_cast<size_t>(s) * slot_packs + tc;
          float acc[8], rs[8];
          unpack8(slot[0], acc);
#pragma unroll
          for (int j = 1; j < N; ++j) {
            float x[8];
            unpack8(slot[static_cast<size_t>(j) * Tc], x);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = __fadd_rn(acc[e], x[e]);
          }
          unpack8(slot[static_cast<size_t>(N) * Tc], rs);
          if (a.sum != nullptr) {
            a.sum[2 * (base + c)] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            a.sum[2 * (base + c) + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) r[v][e] = __fadd_rn(acc[e], rs[e]);
        }
        __syncwarp();
        if (lane == 0 && ok) mbar_arrive(&empty[s]);
        ++t;
      }
    }
    const bool live = !*abort_flag;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = v * Tc + tc;
      if (live && v < V && c < a.P) st_stream(a.rout + base + c, pack8(r[v]));
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(r[v][e], r[v][e], ss);
    }
    ss = warp_sum(ss);
    float *rb = red + 32 * parity_row;
    if (lane == 0) rb[cw] = ss;
    named_barrier_sync(1, static_cast<uint32_t>(Tc));
    float total = 0.f;
    for (int i = 0; i < C; ++i) total += rb[i];
    const float inv = rsqrtf(total / a.H + a.eps);
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
      const int c = v * Tc + tc;
      if (live && v < V && c < a.P) {
        float w[8], y[8];
        unpack8(VPT <= 4 ? wv[v < kWRegs ? v : 0] : ld_ro(a.w + c), w);
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = (r[v][e] * inv) * w[e];
        st_stream(a.out + base + c, pack8(y));
      }
    }
  }
}

using StreamKernel = void (*)(StreamArgs);
StreamKernel stream_kernel(int n, int vpt);

}  // namespace arn
