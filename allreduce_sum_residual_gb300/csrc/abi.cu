// C ABI of libarnorm.so: argument checks, the one-/two-stage choice, launch
// planning, the two-stage workspace and the launches.  Host code only.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "epilogue.cuh"
#include "peer.cuh"
#include "plan_table.cuh"
#include "stream_epilogue.cuh"

// The device status word: AR_OK, or AR_ERR_TIMEOUT after a bounded wait in a
// kernel gave up.  One per device (every device that loads the module holds
// its own copy); kernels receive its address.
__device__ int g_arn_status;

namespace arn {

EpilogueKernel epilogue_kernel_group0(int n, int vpt_log2);
EpilogueKernel epilogue_kernel_group1(int n, int vpt_log2);
EpilogueKernel epilogue_kernel_group2(int n, int vpt_log2);
EpilogueKernel epilogue_kernel_group3(int n, int vpt_log2);
EpilogueKernel epilogue_cluster_kernel_group0(int n, int vpt_log2);
EpilogueKernel epilogue_cluster_kernel_group1(int n, int vpt_log2);
EpilogueKernel epilogue_cluster_kernel_group2(int n, int vpt_log2);
EpilogueKernel epilogue_cluster_kernel_group3(int n, int vpt_log2);
EpilogueKernel epilogue_late_kernel_group0(int n, int vpt_log2);
EpilogueKernel epilogue_late_kernel_group1(int n, int vpt_log2);
EpilogueKernel epilogue_late_kernel_group2(int n, int vpt_log2);
EpilogueKernel epilogue_late_kernel_group3(int n, int vpt_log2);
cudaError_t launch_reduce_flat(const ReduceArgs &a, int n, int sms, cudaStream_t stream);
StreamKernel stream_kernel_group0(int n, int vpt_log2);
StreamKernel stream_kernel_group1(int n, int vpt_log2);
StreamKernel stream_kernel_group2(int n, int vpt_log2);
StreamKernel stream_kernel_group3(int n, int vpt_log2);
cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, int *status, cudaStream_t s);
cudaError_t launch_bounds_selftest(int *status, cudaStream_t s);

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait
constexpr int kAssumedSmemOptin = 232448;         // sm_100-class opt-in per CTA (host-only plans)

static int vpt_log2(int vpt) { return vpt == 1 ? 0 : vpt == 2 ? 1 : vpt == 4 ? 2 : vpt == 8 ? 3 : -1; }

EpilogueKernel epilogue_kernel(int n, int vpt, bool clustered, bool late_weight) {
  const int l = vpt_log2(vpt);
  if (n < 1 || n > AR_MAX_RANKS || l < 0) return nullptr;
  if (clustered && late_weight) return nullptr;
  if (late_weight) switch ((n - 1) / 4) {
      case 0: return epilogue_late_kernel_group0(n, l);
      case 1: return epilogue_late_kernel_group1(n, l);
      case 2: return epilogue_late_kernel_group2(n, l);
      default: return epilogue_late_kernel_group3(n, l);
    }
  if (clustered) switch ((n - 1) / 4) {
      case 0: return epilogue_cluster_kernel_group0(n, l);
      case 1: return epilogue_cluster_kernel_group1(n, l);
      case 2: return epilogue_cluster_kernel_group2(n, l);
      default: return epilogue_cluster_kernel_group3(n, l);
    }
  switch ((n - 1) / 4) {
    case 0: return epilogue_kernel_group0(n, l);
    case 1: return epilogue_kernel_group1(n, l);
    case 2: return epilogue_kernel_group2(n, l);
    default: return epilogue_kernel_group3(n, l);
  }
}

StreamKernel stream_kernel(int n, int vpt) {
  const int l = vpt_log2(vpt);
  if (n < 1 || n > AR_MAX_RANKS || l < 0) return nullptr;
  switch ((n - 1) / 4) {
    case 0: return stream_kernel_group0(n, l);
    case 1: return stream_kernel_group1(n, l);
    case 2: return stream_kernel_group2(n, l);
    default: return stream_kernel_group3(n, l);
  }
}

// ---------------------------------------------------------------- per-device state

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;        // attributes read and kernel attributes set
  int sms = 0;
  int smem_optin = 0;        // largest dynamic shared memory per CTA
  int *status = nullptr;     // this device's g_arn_status
  void *workspace = nullptr; // two-stage bf16 temporary
  int64_t workspace_elems = 0;
};

static std::mutex g_mu;
static DeviceState g_dev[kMaxDevices];

// [device][n - 1][log2 vpt][late weight][threads / 32 - 1]: CTAs per SM of
// the one-CTA register kernels (the driver's occupancy figure), filled when
// a device is made ready; 0 = unknown.
static signed char g_occupancy[kMaxDevices][AR_MAX_RANKS][4][2][32];

// Every one-CTA register kernel at every thread count the plan can give it
// (up to 1024 / vpt), so that planning needs no CUDA call later (it may run
// inside a graph capture).  About 1900 queries, once per device.
static void fill_occupancy(int dev) {
  for (int n = 1; n <= AR_MAX_RANKS; ++n)
    for (int vl = 0; vl < 4; ++vl)
      for (int late = 0; late < 2; ++late) {
        const EpilogueKernel kern = epilogue_kernel(n, 1 << vl, false, late != 0);
        for (int t = 32; t <= 1024 >> vl; t += 32) {
          int k = 0;
          if (kern == nullptr ||
              cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                  &k, reinterpret_cast<const void *>(kern), t, 0) != cudaSuccess ||
              k < 0 || k > 64) {
            cudaGetLastError();
            k = 0;
          }
          g_occupancy[dev][n - 1][vl][late][t / 32 - 1] = static_cast<signed char>(k);
        }
      }
}

// Make the current device ready (SM count, kernel attributes); returns its
// state or null.  Must run outside graph capture the first time.
static DeviceState *current_device(int *status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    *status = AR_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState &d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess ||
        cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_arn_status) != cudaSuccess) {
      cudaGetLastError();
      *status = AR_ERR_CUDA;
      return nullptr;
    }
    for (int n = 1; n <= AR_MAX_RANKS; ++n)
      for (int vpt = 1; vpt <= 8; vpt *= 2) {
        if (cudaFuncSetAttribute(reinterpret_cast<const void *>(stream_kernel(n, vpt)),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, d.smem_optin) !=
            cudaSuccess) {
          cudaGetLastError();
          *status = AR_ERR_CUDA;
          return nullptr;
        }
      }
    // Rows split over up to 16 CTAs need the non-portable cluster size.
    for (int n = 1; n <= AR_MAX_RANKS; ++n)
      for (int vpt = 1; vpt <= 8; vpt *= 2) {
        if (cudaFuncSetAttribute(reinterpret_cast<const void *>(epilogue_kernel(n, vpt, true, false)),
                                 cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
          cudaGetLastError();
          *status = AR_ERR_CUDA;
          return nullptr;
        }
      }
    fill_occupancy(dev);
    d.ready = true;
  }
  *status = AR_OK;
  return &d;
}

// ---------------------------------------------------------------- checks

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};

static bool overlap(const Range &a, const Range &b) { return a.lo < b.hi && b.lo < a.hi; }

static Range range_of(const void *p, int64_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Range{lo, lo + static_cast<uintptr_t>(bytes)};
}

static int check_shape(int n, int64_t m, int64_t H, float eps) {
  if (n < 1 || n > AR_MAX_RANKS || m < 0 || H <= 0) return AR_ERR_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return AR_ERR_ARG;
  if (H % kPackElems != 0) return AR_ERR_ALIGN;
  if (H > AR_MAX_HIDDEN) return AR_ERR_UNSUPPORTED;
  if (m > (int64_t{1} << 40) / H) return AR_ERR_UNSUPPORTED;  // keeps every byte count in range
  return AR_OK;
}

// check_shape for the entry points defined in other translation units.
int check_call_shape(int n, int64_t m, int64_t H, float eps) { return check_shape(n, m, H, eps); }

// Pointers of a full epilogue call: null, alignment, then overlaps.
static int check_buffers(const void *const *partials, int n, const void *residual,
                         const void *weight, int64_t m, int64_t H, const void *out,
                         const void *residual_out, const void *sum_out) {
  if (!partials || !residual || !weight || !out || !residual_out) return AR_ERR_ARG;
  for (int k = 0; k < n; ++k)
    if (!partials[k]) return AR_ERR_ARG;
  for (int k = 0; k < n; ++k)
    if (!aligned16(partials[k])) return AR_ERR_ALIGN;
  if (!aligned16(residual) || !aligned16(weight) || !aligned16(out) || !aligned16(residual_out) ||
      (sum_out && !aligned16(sum_out)))
    return AR_ERR_ALIGN;
  const int64_t bytes = m * H * 2;
  const Range o = range_of(out, bytes), ro = range_of(residual_out, bytes);
  const Range res = range_of(residual, bytes), w = range_of(weight, H * 2);
  if (overlap(o, ro) || overlap(o, res) || overlap(o, w)) return AR_ERR_ALIAS;
  if (overlap(ro, w)) return AR_ERR_ALIAS;
  if (overlap(ro, res) && residual_out != residual) return AR_ERR_ALIAS;
  for (int k = 0; k < n; ++k) {
    const Range p = range_of(partials[k], bytes);
    if (overlap(p, o) || overlap(p, ro)) return AR_ERR_ALIAS;
  }
  if (sum_out) {
    const Range s = range_of(sum_out, m * H * 4);
    if (overlap(s, o) || overlap(s, ro) || overlap(s, res) || overlap(s, w)) return AR_ERR_ALIAS;
    for (int k = 0; k < n; ++k)
      if (overlap(s, range_of(partials[k], bytes))) return AR_ERR_ALIAS;
  }
  return AR_OK;
}

// ---------------------------------------------------------------- policy

// One-stage up to this many rows, two-stage above.  Measured on GB300 with
// both paths at n in {4, 8}, H in {4096, 8192}, m = 1 .. 16384 (the bench's
// sweep mode, cold buffers, graphs of back-to-back calls): one-stage was
// faster at every point -- by 1.6-2.4 us at m <= 64 (two-stage adds a launch)
// and by 1.25-1.7x at m >= 512 (two-stage moves (n+5)/(n+3) of the bytes).
// On one GPU there is no cross-GPU traffic for the two-stage reduce-scatter
// to save, so the threshold is unbounded for every (n, H).  (The pages' rule,
// one-stage for m <= 32 at 4 ranks and m <= 16 at 8, was set on MI355X
// across GPUs: ROCm/aiter #3817, Test Results.)
static int64_t one_stage_max_rows(int n, int64_t H) {
  (void)n;
  (void)H;
  return INT64_MAX;
}

static int select_mode(int n, int64_t m, int64_t H) {
  return m <= one_stage_max_rows(n, H) ? AR_MODE_ONE_STAGE : AR_MODE_TWO_STAGE;
}

// Kernel choice from 64 rows on, for rows up to the table's longest (1024
// packs, H = 8192): the lookup table of plan_table.cuh, measured on GB300.
// For every (inputs, packs per row, rows) of its grid it holds each
// candidate's speed as a percentage of the fastest there: the stream kernel
// and the register kernel with 1, 2, 4 or 8 packs per thread (one-stage,
// cold buffers, CUDA-graph timing; repeated sweeps agreed within 0.5 %).
// No simple rule fits it: which kernel wins turns on how many CTAs of each
// fit an SM (the register counts of each instantiation), whether the rows
// fill a whole number of waves, and how many bytes are then in flight --
// one more wave of a few rows can cost 25 %.  Between grid points the
// percentages of the grid cells that bracket the shape (two columns per
// axis where it falls between two: inputs, packs, rows) are added up and
// the best sum wins, which prefers a candidate that is good on both sides
// of a cliff.  Rows are first scaled to the table's SM count; rows
// shorter than the table's shortest use its column.  Returns the kernel
// and its packs per thread, or kernel 0 where the table does not apply
// (fewer than 64 rows, where the register kernel spreads a row over a
// cluster, or rows longer than the table's longest).
constexpr int64_t kTableMinRows = 64;

// The grid columns around x: [lo, hi] = [i - 1, i] between two columns,
// [i, i] on a column or beyond either end.
template <int K>
static void bracket(const int (&grid)[K], double x, int *lo, int *hi) {
  if (x <= grid[0]) {
    *lo = *hi = 0;
    return;
  }
  for (int i = 0; i < K; ++i) {
    if (x == grid[i]) {
      *lo = *hi = i;
      return;
    }
    if (x < grid[i]) {
      *lo = i - 1;
      *hi = i;
      return;
    }
  }
  *lo = *hi = K - 1;
}

template <int K>
static int last_of(const int (&grid)[K]) {
  return grid[K - 1];
}

struct TableChoice {
  int kernel;  // AR_KERNEL_STREAM, AR_KERNEL_REGISTER or AR_KERNEL_REGISTER_LATE_W; 0: no table
  int vpt;     // register kernels: packs per thread
};

// Candidate c of the table: 0 the stream kernel; 1 .. 4 the register
// kernel with 1, 2, 4, 8 packs per thread; 5 .. 8 the same with the weight
// loaded after the sums.
static TableChoice candidate(int c) {
  if (c == 0) return {AR_KERNEL_STREAM, 0};
  if (c <= 4) return {AR_KERNEL_REGISTER, 1 << (c - 1)};
  return {AR_KERNEL_REGISTER_LATE_W, 1 << (c - 5)};
}

// CTAs of the one-CTA-per-row register kernel (inputs, vpt, late weight)
// with `threads` threads that fit one SM of the current device, from the
// table filled when the device was made ready; 0 where unknown.  No CUDA
// call here, so planning stays safe inside a graph capture.
static int device_register_occupancy(int inputs, int vpt, int late, int threads) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return 0;
  }
  const int vl = vpt_log2(vpt);
  if (vl < 0 || inputs < 1 || inputs > AR_MAX_RANKS || threads < 32 || threads > 1024 ||
      threads % 32 != 0)
    return 0;
  return g_occupancy[dev][inputs - 1][vl][late ? 1 : 0][threads / 32 - 1];
}

using OccupancyFn = ar_occupancy_fn;

// `occupancy` (may be null) makes the rows interpolation wave-aware.  A
// register-kernel candidate runs its rows in waves of (CTAs per SM x SMs);
// where the two bracketing rows columns lie in different wave counts for
// it, only the column with the shape's own wave count is used for that
// candidate: one more, mostly idle wave costs up to 25 %, so the column
// across the wave boundary does not describe the shape.  (Held out against
// the sweep, this lifted the pick from 0.984 to 0.990 of the best candidate
// on average.)  Candidates are compared by their mean percentage.
static TableChoice table_choice(int inputs, int64_t m, int64_t P, int sms,
                                OccupancyFn occupancy) {
  if (m < kTableMinRows || P > last_of(kPlanPacks)) return {0, 0};
  int n0, n1, p0, p1, m0, m1;
  bracket(kPlanInputs, static_cast<double>(inputs), &n0, &n1);
  bracket(kPlanPacks, static_cast<double>(P), &p0, &p1);
  const double rows = static_cast<double>(m) * kPlanTableSms / sms;  // in the table's SMs
  bracket(kPlanRows, rows, &m0, &m1);
  int best = 0;
  double best_mean = -1.0;
  for (int c = 0; c < kPlanCandidates; ++c) {
    int lo = m0, hi = m1;
    const TableChoice k = candidate(c);
    if (occupancy != nullptr && k.kernel != AR_KERNEL_STREAM && m0 != m1 && P <= kMaxPacksPerCta) {
      const int threads = static_cast<int>(((P + k.vpt - 1) / k.vpt + 31) / 32 * 32);
      const int per_sm = occupancy(inputs, k.vpt, k.kernel == AR_KERNEL_REGISTER_LATE_W ? 1 : 0,
                                   threads);
      if (per_sm > 0) {
        const double wave = static_cast<double>(per_sm) * kPlanTableSms;
        const double w = std::ceil(rows / wave);
        const bool at_lo = std::ceil(kPlanRows[m0] / wave) == w;
        const bool at_hi = std::ceil(kPlanRows[m1] / wave) == w;
        if (at_lo && !at_hi) hi = m0;
        if (at_hi && !at_lo) lo = m1;
      }
    }
    int sum = 0, count = 0;
    for (int ni = n0; ni <= n1; ++ni)
      for (int pi = p0; pi <= p1; ++pi)
        for (int mi = lo; mi <= hi; ++mi) {
          sum += kPlanScore[ni][pi][mi][c];
          ++count;
        }
    const double mean = static_cast<double>(sum) / count;
    if (mean > best_mean) {
      best_mean = mean;
      best = c;
    }
  }
  return candidate(best);
}

// Rows of more than 1024 packs (beyond the table): the stream kernel for 4
// inputs from max(4 x SMs, 1024) rows and for 5 or more from 256 rows (at
// H = 8192 the register kernel's 1024-thread CTAs fit once per SM, up to
// 1.4x slower than the stream kernel from 256 rows at n = 8); otherwise the
// register kernel, a row split over a cluster.
static bool long_rows_want_stream(int inputs, int64_t m, int sms) {
  if (inputs < 4) return false;
  const int64_t four_waves = 4 * static_cast<int64_t>(sms);
  return m >= (inputs > 4 ? 256 : (four_waves > 1024 ? four_waves : 1024));
}

// Register kernel: launch shape for m rows of P packs.  Set from the GB300
// launch-shape sweep (the bench's shapes mode: decode n = 8 and mid-size
// n = 4 at H = 7168, every cluster size x packs per thread, hot and cold):
//  * cluster S: the fewest CTAs per row that hold a row slice in registers
//    (<= 1024 packs per CTA); below 64 rows, a row is spread over 8 CTAs
//    (each keeping >= 32 packs) -- 8 matched or beat 16, 4, 2 and 1 at
//    m <= 32 once the cluster exchange became one st.async per CTA pair --
//    while from 64 rows one CTA per row was as fast or faster;
//  * vpt: `table_vpt` where the lookup table gives one; otherwise (below 64
//    rows, or rows of more than 1024 packs) 1 pack per thread, the most
//    loads in flight per CTA, except 2 for 256 .. 1023 rows of more than
//    512 packs a CTA (a CTA of up to 1024 threads fits once per SM and the
//    rows would run in two waves) and for 1024 rows or more with 4 inputs
//    or more, or one input with more than 512 packs a CTA.  Either way a
//    CTA stays within 1024 / vpt threads.
static void plan_register(int64_t m, int64_t P, int inputs, int force_cluster, int force_vpt,
                          int table_vpt, ar_plan_t *pl) {
  int S = 1;
  while (S < kMaxClusterCtas && (P + S - 1) / S > kMaxPacksPerCta) S *= 2;
  if (m < 64)
    while (S < 8 && (P + 2 * S - 1) / (2 * S) >= 32) S *= 2;
  if (force_cluster > 0) S = force_cluster;
  const int64_t per_cta = (P + S - 1) / S;
  int vpt = 1;
  if (table_vpt > 0 && (S == 1 || P > kMaxPacksPerCta))
    vpt = table_vpt;
  else if (m >= 1024)
    vpt = (inputs >= 4 || (inputs == 1 && per_cta > 512)) ? 2 : 1;
  else if (m >= 256 && per_cta > 512)
    vpt = 2;
  while (vpt < 8 && (per_cta + vpt - 1) / vpt > 1024 / vpt) vpt *= 2;
  if (force_vpt > 0) vpt = force_vpt;
  int threads = static_cast<int>((per_cta + vpt - 1) / vpt);
  threads = (threads + 31) / 32 * 32;
  pl->kernel = AR_KERNEL_REGISTER;
  pl->cluster = S;
  pl->vpt = vpt;
  pl->threads = threads;
  pl->stages = 0;
  pl->ctas = m * S;
}

static int64_t stream_smem_bytes(int inputs, int consumers, int stages) {
  return static_cast<int64_t>(stages) * (inputs + 1) * consumers * 16 + 16 * stages + 64 * 4 + 16;
}

// Stream kernel.  A row is split into V tiles of T_c <= 512 packs (about
// 256 where that gives <= 8 tiles).  The ring is sized for about
// kStreamInflightBytes of bulk copies in flight per SM: 2 CTAs per SM while
// two 2-slot rings stay within kStreamTwoCtaMaxBytes (and fit in shared
// memory and the register file), else 1, each with as many slots as the
// target allows (>= 2).  Measured on GB300 (one-stage, m = 8192, n = 4 ..
// 16, H = 4096 .. 8192, repeats within 0.1-0.5 %): about 100-150 KB in
// flight per SM ran at 7.0-7.2 TB/s, filling shared memory (216 KB) at
// 6.3-6.4 TB/s -- deeper queues of outstanding bulk copies are slower; at
// n = 4 three 18 KB slots per CTA beat four by 7 %, and with >= 12 inputs
// one CTA per SM beat two.  A forced plan may set T_c (threads - 32), the
// ring depth and the grid.  False if the shape cannot apply.
constexpr int64_t kStreamInflightBytes = 120 * 1024;
constexpr int64_t kStreamTwoCtaMaxBytes = 160 * 1024;

static bool plan_stream(int64_t m, int64_t P, int inputs, int sms, int smem_optin,
                        const ar_plan_t *force, ar_plan_t *pl) {
  if (P > AR_STREAM_MAX_HIDDEN / kPackElems) return false;
  int64_t V = (P + 255) / 256;
  if (V > 8) V = (P + kStreamMaxConsumers - 1) / kStreamMaxConsumers;
  int Tc = static_cast<int>(((P + V - 1) / V + 31) / 32 * 32);
  if (force && force->threads > 0) {
    Tc = force->threads - 32;
    if (Tc < 32 || Tc > kStreamMaxConsumers || Tc % 32 != 0) return false;
    V = (P + Tc - 1) / Tc;
  }
  if (V > 8) return false;
  const int64_t slot = static_cast<int64_t>(inputs + 1) * Tc * 16;
  // Two CTAs per SM need two 2-slot rings in shared memory and their threads'
  // registers in the register file (<= 96 registers a thread: T_c <= 288).
  const int64_t half_budget = smem_optin / 2 - 1024;
  int64_t per_sm = (stream_smem_bytes(inputs, Tc, 2) <= half_budget && Tc <= 288 &&
                    4 * slot <= kStreamTwoCtaMaxBytes)
                       ? 2
                       : 1;
  int64_t ctas = per_sm * sms;
  int stages = static_cast<int>(kStreamInflightBytes / (per_sm * slot));
  if (force && force->ctas > 0) {
    ctas = force->ctas;
    per_sm = (ctas + sms - 1) / sms;
  }
  if (force && force->stages > 0) stages = force->stages;
  if (stages > 16) stages = 16;
  if (stages < 2) stages = 2;
  const int64_t budget = smem_optin / per_sm - (per_sm > 1 ? 1024 : 0);
  while (stages >= 2 && stream_smem_bytes(inputs, Tc, stages) > budget) --stages;
  if (stages < 2) return false;
  if (ctas > m) ctas = m;
  int vpt = 1;
  while (vpt < V) vpt *= 2;
  pl->kernel = AR_KERNEL_STREAM;
  pl->cluster = 1;
  pl->vpt = vpt;
  pl->threads = 32 + Tc;
  pl->stages = stages;
  pl->ctas = ctas;
  return true;
}

// Rows a register-kernel plan works on at once on the device: its CTAs per
// SM x SMs / CTAs per row; 0 if unknown or a stream-kernel plan.  For a
// row split over a cluster the one-CTA instantiation's occupancy at the
// same thread count stands in for the cluster copy's (only a prefetch
// distance depends on it).
static int64_t resident_rows(const ar_plan_t &pl, int inputs, int sms, OccupancyFn occupancy) {
  if (occupancy == nullptr || pl.kernel == AR_KERNEL_STREAM || pl.cluster < 1) return 0;
  const int per_sm =
      occupancy(inputs, pl.vpt, pl.kernel == AR_KERNEL_REGISTER_LATE_W ? 1 : 0, pl.threads);
  return per_sm > 0 ? static_cast<int64_t>(per_sm) * sms / pl.cluster : 0;
}

// L2 prefetch of the epilogue kernel, measured on GB300 (cold buffers,
// graphs of back-to-back calls).  Every kernel prefetches its first row
// (slice) before it waits for the previous grid: decode m = 1 went from
// 2.05 to 1.74 us per call, n = 4, H = 4096, m = 256 from 3.97 to 2.93 us,
// the stream kernel gained 1-3 % at 512-1024 rows.  A register kernel whose
// rows need more than one wave of CTAs also prefetches the row one wave
// ahead (n = 4, H = 7168, m = 1024: 6.8 -> 7.15 TB/s).  The stream kernel
// does not prefetch ahead: its ring already runs ahead, and an extra row of
// prefetches in flight cost it 10-25 %.
static int plan_prefetch(const ar_plan_t &pl, int64_t m, int inputs, int sms,
                         OccupancyFn occupancy) {
  if (pl.kernel == AR_KERNEL_STREAM) return AR_PREFETCH_ROW;
  const int64_t wave = resident_rows(pl, inputs, sms, occupancy);
  return wave > 0 && m > wave ? AR_PREFETCH_ROW_AHEAD : AR_PREFETCH_ROW;
}

static int make_plan(int n, int64_t m, int64_t H, int mode, int sms, int smem_optin,
                     const ar_plan_t *force, ar_plan_t *pl, OccupancyFn occupancy = nullptr) {
  if (mode != AR_MODE_AUTO && mode != AR_MODE_ONE_STAGE && mode != AR_MODE_TWO_STAGE)
    return AR_ERR_ARG;
  std::memset(pl, 0, sizeof *pl);
  pl->mode = mode == AR_MODE_AUTO ? select_mode(n, m, H) : mode;
  int fk = AR_KERNEL_AUTO, fc = 0, fv = 0;
  if (force) {
    fk = force->kernel;
    fc = force->cluster;
    fv = force->vpt;
    if (fk != AR_KERNEL_AUTO && fk != AR_KERNEL_REGISTER && fk != AR_KERNEL_STREAM &&
        fk != AR_KERNEL_REGISTER_LATE_W)
      return AR_ERR_ARG;
    if (fk == AR_KERNEL_REGISTER_LATE_W && fc > 1) return AR_ERR_ARG;
    if (fc != 0 && fc != 1 && fc != 2 && fc != 4 && fc != 8 && fc != 16) return AR_ERR_ARG;
    if (fv != 0 && vpt_log2(fv) < 0) return AR_ERR_ARG;
    if (fk == AR_KERNEL_STREAM && (fc > 1 || fv != 0)) return AR_ERR_ARG;
    if (fk != AR_KERNEL_STREAM && (force->threads != 0 || force->stages != 0 || force->ctas != 0))
      return AR_ERR_ARG;
    if (force->threads < 0 || force->stages < 0 || force->stages > 16 || force->ctas < 0)
      return AR_ERR_ARG;
    if (force->prefetch < AR_PREFETCH_AUTO || force->prefetch > AR_PREFETCH_ROW_AHEAD)
      return AR_ERR_ARG;
  }
  const int64_t P = H / kPackElems;
  const int inputs = pl->mode == AR_MODE_TWO_STAGE ? 1 : n;
  const bool shape_forced = fc != 0 || fv != 0;
  const TableChoice choice = table_choice(inputs, m, P, sms, occupancy);
  bool want_stream = fk == AR_KERNEL_STREAM;
  if (fk == AR_KERNEL_AUTO && !shape_forced)
    want_stream = choice.kernel ? choice.kernel == AR_KERNEL_STREAM
                                : long_rows_want_stream(inputs, m, sms);
  if (!(want_stream && plan_stream(m, P, inputs, sms, smem_optin,
                                   fk == AR_KERNEL_STREAM ? force : nullptr, pl))) {
    if (fk == AR_KERNEL_STREAM) return AR_ERR_ARG;
    const bool table_register = choice.kernel == AR_KERNEL_REGISTER ||
                                choice.kernel == AR_KERNEL_REGISTER_LATE_W;
    plan_register(m, P, inputs, fc, fv, table_register ? choice.vpt : 0, pl);
    const bool late = fk == AR_KERNEL_REGISTER_LATE_W ||
                      (fk == AR_KERNEL_AUTO && !shape_forced &&
                       choice.kernel == AR_KERNEL_REGISTER_LATE_W);
    if (late && pl->cluster == 1) pl->kernel = AR_KERNEL_REGISTER_LATE_W;
    if (fk == AR_KERNEL_REGISTER_LATE_W && pl->cluster != 1) return AR_ERR_ARG;
    const int64_t per_cta = (P + pl->cluster - 1) / pl->cluster;
    if (per_cta > kMaxPacksPerCta) return AR_ERR_ARG;  // forced shape too small
  }
  if (pl->ctas > INT32_MAX) return AR_ERR_UNSUPPORTED;
  pl->launches = pl->mode == AR_MODE_TWO_STAGE ? 2 : 1;
  pl->prefetch = plan_prefetch(*pl, m, inputs, sms, occupancy);
  if (force && force->prefetch != AR_PREFETCH_AUTO) {
    pl->prefetch = force->prefetch;
  }
  return AR_OK;
}

// Every launch carries programmatic stream serialization: the kernel may be
// scheduled while the previous grid in the stream drains, and waits for it
// (griddepcontrol.wait) before touching global memory.  `after_prior` marks
// stage 2, whose predecessor is stage 1 of the same call: it may read the
// weight and the residual before that wait.
static cudaError_t launch_epilogue(const EpilogueArgs &a, int n, const ar_plan_t &pl,
                                   bool after_prior, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.ctas), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(pl.threads), 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (pl.cluster > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(pl.cluster);
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  cfg.attrs = attr;
  cfg.numAttrs = na;
  EpilogueArgs args = a;
  args.early_reads = after_prior ? 1 : 0;
  // Stage 2 loads its residual and weight before the wait instead; its
  // input (the temporary) is being written by stage 1 until then.
  if (after_prior) args.prefetch_own = 0;
  const cudaError_t e = cudaLaunchKernelEx(
      &cfg, epilogue_kernel(n, pl.vpt, pl.cluster > 1, pl.kernel == AR_KERNEL_REGISTER_LATE_W), args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

static cudaError_t launch_stream(const void *const *inputs, int n, const void *residual,
                                 const void *weight, float eps, int64_t m, int64_t H, void *out,
                                 void *residual_out, float *sum_out, const ar_plan_t &pl,
                                 int *status, bool after_prior, cudaStream_t stream) {
  StreamArgs a;
  std::memset(&a, 0, sizeof a);
  for (int k = 0; k < n; ++k) a.src[k] = static_cast<const uint4 *>(inputs[k]);
  a.src[n] = static_cast<const uint4 *>(residual);
  a.w = static_cast<const uint4 *>(weight);
  a.out = static_cast<uint4 *>(out);
  a.rout = static_cast<uint4 *>(residual_out);
  a.sum = reinterpret_cast<float4 *>(sum_out);
  a.m = m;
  a.P = static_cast<int>(H / kPackElems);
  const int Tc = pl.threads - 32;
  a.tiles = (a.P + Tc - 1) / Tc;
  a.stages = pl.stages;
  a.H = static_cast<float>(H);
  a.eps = eps;
  a.wait_limit_ns = kWaitLimitNs;
  a.status = status;
  // Stage 2 reads the temporary stage 1 is still writing until the wait.
  a.prefetch_first = !after_prior && (pl.prefetch == AR_PREFETCH_ROW ||
                                      pl.prefetch == AR_PREFETCH_ROW_AHEAD);
  a.prefetch_next = pl.prefetch == AR_PREFETCH_ROW_AHEAD;
  a.smem_bytes = static_cast<int>(stream_smem_bytes(n, Tc, pl.stages));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(pl.ctas), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(pl.threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(stream_smem_bytes(n, Tc, pl.stages));
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, stream_kernel(n, pl.vpt), a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

static void fill_epilogue_args(EpilogueArgs *a, const void *const *inputs, int n,
                               const void *residual, const void *weight, float eps, int64_t m,
                               int64_t H, void *out, void *residual_out, float *sum_out,
                               const ar_plan_t &pl, int *status) {
  std::memset(a, 0, sizeof *a);
  for (int k = 0; k < n; ++k) a->p[k] = static_cast<const uint4 *>(inputs[k]);
  a->res = static_cast<const uint4 *>(residual);
  a->w = static_cast<const uint4 *>(weight);
  a->out = static_cast<uint4 *>(out);
  a->rout = static_cast<uint4 *>(residual_out);
  a->sum = reinterpret_cast<float4 *>(sum_out);
  a->m = m;
  a->P = static_cast<int>(H / kPackElems);
  a->per_cta = static_cast<int>((a->P + pl.cluster - 1) / pl.cluster);
  a->H = static_cast<float>(H);
  a->eps = eps;
  a->wait_limit_ns = kWaitLimitNs;
  a->status = status;
  a->prefetch_own = pl.prefetch == AR_PREFETCH_ROW || pl.prefetch == AR_PREFETCH_ROW_AHEAD;
  a->ahead = 0;
  if (pl.prefetch == AR_PREFETCH_ROW_AHEAD) {
    int sms = 0;
    const DeviceState *d = nullptr;
    int dev = -1;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices && g_dev[dev].ready) {
      d = &g_dev[dev];
      sms = d->sms;
    } else {
      cudaGetLastError();
    }
    if (d != nullptr) a->ahead = resident_rows(pl, n, sms, device_register_occupancy);
  }
}

// True if the current device `dev` can use `p` at the same address: its own
// device memory, managed memory, or host memory that is pinned and mapped
// (cudaHostAlloc, cudaHostRegister; with unified addressing the device
// address equals the host address).  Pageable host memory, another device's
// memory and unknown pointers are refused.
static bool device_accessible(const void *p, int dev) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  switch (at.type) {
    case cudaMemoryTypeDevice: {
      if (at.device == dev) return true;  // this device's memory, or another process's (IPC)
      int can = 0;                        // another GPU's memory through a peer mapping
      if (cudaDeviceCanAccessPeer(&can, dev, at.device) != cudaSuccess) {
        cudaGetLastError();
        return false;
      }
      return can != 0;
    }
    case cudaMemoryTypeManaged: return true;
    case cudaMemoryTypeHost: return at.devicePointer == p;
    default: return false;
  }
}

static int check_mapped(const void *const *partials, int n, const void *residual,
                        const void *weight, const void *out, const void *residual_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  for (int k = 0; k < n; ++k)
    if (!device_accessible(partials[k], dev)) return AR_ERR_ARG;
  if (!device_accessible(residual, dev) || !device_accessible(weight, dev) ||
      !device_accessible(out, dev) || !device_accessible(residual_out, dev))
    return AR_ERR_ARG;
  return AR_OK;
}

// `mapped`: any buffer may be pinned host memory (checked per pointer); the
// epilogue then runs on the register kernel, whose plain loads and stores
// reach host memory over the host link.  (The stream kernel's bulk copies
// are kept to device memory.)
static int run(const void *const *partials, int n, const void *residual, const void *weight,
               float eps, int64_t m, int64_t H, void *out, void *residual_out, int mode,
               void *stream, float *sum_out, const ar_plan_t *force, bool mapped = false) {
  int st = check_shape(n, m, H, eps);
  if (st != AR_OK) return st;
  if (mode != AR_MODE_AUTO && mode != AR_MODE_ONE_STAGE && mode != AR_MODE_TWO_STAGE)
    return AR_ERR_ARG;
  if (m == 0) return AR_OK;  // nothing is read or written; pointers may be null
  st = check_buffers(partials, n, residual, weight, m, H, out, residual_out, sum_out);
  if (st != AR_OK) return st;
  ar_plan_t register_only;
  if (mapped) {
    st = check_mapped(partials, n, residual, weight, out, residual_out);
    if (st != AR_OK) return st;
    std::memset(&register_only, 0, sizeof register_only);
    register_only.kernel = AR_KERNEL_REGISTER;
    register_only.prefetch = AR_PREFETCH_NONE;  // bulk prefetches stay on device memory
    force = &register_only;
  }
  DeviceState *d = current_device(&st);
  if (!d) return st;
  ar_plan_t pl;
  st = make_plan(n, m, H, mode, d->sms, d->smem_optin, force, &pl, device_register_occupancy);
  if (st != AR_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The epilogue over `inputs` (the partials, or the two-stage temporary).
  auto epilogue = [&](const void *const *inputs, int count, bool after_prior) -> int {
    cudaError_t e;
    if (pl.kernel == AR_KERNEL_STREAM) {
      e = launch_stream(inputs, count, residual, weight, eps, m, H, out, residual_out, sum_out, pl,
                        d->status, after_prior, s);
    } else {
      EpilogueArgs a;
      fill_epilogue_args(&a, inputs, count, residual, weight, eps, m, H, out, residual_out,
                         sum_out, pl, d->status);
      e = launch_epilogue(a, count, pl, after_prior, s);
    }
    return e == cudaSuccess ? AR_OK : AR_ERR_CUDA;
  };
  if (pl.mode == AR_MODE_ONE_STAGE) return epilogue(partials, n, false);
  // two-stage: stage 1 into the workspace, stage 2 from it
  void *ws;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    if (d->workspace == nullptr || d->workspace_elems < m * H) return AR_ERR_WORKSPACE;
    ws = d->workspace;
  }
  const Range wr = range_of(ws, m * H * 2);
  const int64_t bytes = m * H * 2;
  if (overlap(wr, range_of(out, bytes)) || overlap(wr, range_of(residual_out, bytes)) ||
      overlap(wr, range_of(residual, bytes)) || overlap(wr, range_of(weight, H * 2)) ||
      (sum_out && overlap(wr, range_of(sum_out, m * H * 4))))
    return AR_ERR_ALIAS;
  for (int k = 0; k < n; ++k)
    if (overlap(wr, range_of(partials[k], bytes))) return AR_ERR_ALIAS;
  ReduceArgs ra;
  std::memset(&ra, 0, sizeof ra);
  for (int k = 0; k < n; ++k) ra.p[k] = static_cast<const uint4 *>(partials[k]);
  ra.dst[0] = static_cast<uint4 *>(ws);
  ra.ndst = 1;
  ra.begin = 0;
  ra.end = m * H / kPackElems;
  ra.prefetch = pl.prefetch != AR_PREFETCH_NONE;
  ra.status = d->status;
  if (launch_reduce_flat(ra, n, d->sms, s) != cudaSuccess) return AR_ERR_CUDA;
  const void *temp_in[1] = {ws};
  return epilogue(temp_in, 1, true);
}

// The two-stage path with a temporary the caller supplies (`temp`, room for
// `temp_elems` bf16), instead of the reserved workspace.  Same checks, plan
// and kernels as ar_rmsnorm in AR_MODE_TWO_STAGE; allocates nothing.
int two_stage_with_temp(const void *const *partials, int n, const void *residual,
                        const void *weight, float eps, int64_t m, int64_t H, void *out,
                        void *residual_out, void *temp, int64_t temp_elems, void *stream) {
  int st = check_shape(n, m, H, eps);
  if (st != AR_OK) return st;
  if (m == 0) return AR_OK;
  st = check_buffers(partials, n, residual, weight, m, H, out, residual_out, nullptr);
  if (st != AR_OK) return st;
  if (!temp || !aligned16(temp) || temp_elems < m * H) return AR_ERR_ARG;
  const int64_t bytes = m * H * 2;
  const Range tr = range_of(temp, bytes);
  if (overlap(tr, range_of(out, bytes)) || overlap(tr, range_of(residual_out, bytes)) ||
      overlap(tr, range_of(residual, bytes)) || overlap(tr, range_of(weight, H * 2)))
    return AR_ERR_ALIAS;
  for (int k = 0; k < n; ++k)
    if (overlap(tr, range_of(partials[k], bytes))) return AR_ERR_ALIAS;
  DeviceState *d = current_device(&st);
  if (!d) return st;
  ar_plan_t pl;
  st = make_plan(n, m, H, AR_MODE_TWO_STAGE, d->sms, d->smem_optin, nullptr, &pl,
                 device_register_occupancy);
  if (st != AR_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  ReduceArgs ra;
  std::memset(&ra, 0, sizeof ra);
  for (int k = 0; k < n; ++k) ra.p[k] = static_cast<const uint4 *>(partials[k]);
  ra.dst[0] = static_cast<uint4 *>(temp);
  ra.ndst = 1;
  ra.begin = 0;
  ra.end = m * H / kPackElems;
  ra.prefetch = pl.prefetch != AR_PREFETCH_NONE;
  ra.status = d->status;
  if (launch_reduce_flat(ra, n, d->sms, s) != cudaSuccess) return AR_ERR_CUDA;
  const void *temp_in[1] = {temp};
  cudaError_t e;
  if (pl.kernel == AR_KERNEL_STREAM) {
    e = launch_stream(temp_in, 1, residual, weight, eps, m, H, out, residual_out, nullptr, pl,
                      d->status, true, s);
  } else {
    EpilogueArgs a;
    fill_epilogue_args(&a, temp_in, 1, residual, weight, eps, m, H, out, residual_out, nullptr, pl,
                       d->status);
    e = launch_epilogue(a, 1, pl, true, s);
  }
  return e == cudaSuccess ? AR_OK : AR_ERR_CUDA;
}

}  // namespace arn

using namespace arn;

extern "C" {

int ar_rmsnorm(const void *const *partials, int n, const void *residual, const void *weight,
               float eps, int64_t m, int64_t H, void *out, void *residual_out, int mode,
               void *stream) {
  return run(partials, n, residual, weight, eps, m, H, out, residual_out, mode, stream, nullptr,
             nullptr);
}

int ar_rmsnorm_ex(const void *const *partials, int n, const void *residual, const void *weight,
                  float eps, int64_t m, int64_t H, void *out, void *residual_out, int mode,
                  void *stream, float *sum_out, const ar_plan_t *plan) {
  return run(partials, n, residual, weight, eps, m, H, out, residual_out, mode, stream, sum_out,
             plan);
}

int ar_rmsnorm_mapped(const void *const *partials, int n, const void *residual,
                      const void *weight, float eps, int64_t m, int64_t H, void *out,
                      void *residual_out, int mode, void *stream) {
  return run(partials, n, residual, weight, eps, m, H, out, residual_out, mode, stream, nullptr,
             nullptr, true);
}

int ar_get_plan(int n, int64_t m, int64_t H, int mode, int sm_count, ar_plan_t *plan) {
  if (!plan) return AR_ERR_ARG;
  int st = check_shape(n, m, H, 0.f);
  if (st != AR_OK) return st;
  int smem = kAssumedSmemOptin;
  OccupancyFn occupancy = nullptr;  // pure host logic for a given SM count
  if (sm_count <= 0) {
    DeviceState *d = current_device(&st);
    if (!d) return st;
    sm_count = d->sms;
    smem = d->smem_optin;
    occupancy = device_register_occupancy;
  }
  return make_plan(n, m, H, mode, sm_count, smem, nullptr, plan, occupancy);
}

int ar_register_occupancy(int inputs, int vpt, int late_weight, int threads) {
  return device_register_occupancy(inputs, vpt, late_weight, threads);
}

int ar_get_plan_ex(int n, int64_t m, int64_t H, int mode, int sm_count,
                   ar_occupancy_fn ctas_per_sm, ar_plan_t *plan) {
  if (!plan || sm_count <= 0) return AR_ERR_ARG;
  const int st = check_shape(n, m, H, 0.f);
  if (st != AR_OK) return st;
  return make_plan(n, m, H, mode, sm_count, kAssumedSmemOptin, nullptr, plan, ctas_per_sm);
}

int ar_device_status(int device, int reset) {
  if (device < 0 || device >= kMaxDevices) return AR_ERR_ARG;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  int st = AR_OK, value = AR_OK;
  DeviceState *d = current_device(&st);
  if (d) {
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&value, d->status, sizeof value, cudaMemcpyDeviceToHost) != cudaSuccess) {
      cudaGetLastError();
      st = AR_ERR_CUDA;
    } else if (reset) {
      const int zero = AR_OK;
      if (cudaMemcpy(d->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        st = AR_ERR_CUDA;
      }
    }
  }
  cudaSetDevice(prev);
  return st != AR_OK ? st : value;
}

int ar_selftest_bounded_wait(int device, unsigned limit_us) {
  if (device < 0 || device >= kMaxDevices || limit_us == 0 || limit_us > 10000000u)
    return AR_ERR_ARG;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  int st = AR_OK;
  DeviceState *d = current_device(&st);
  if (d) {
    if (launch_bounded_wait_selftest(static_cast<uint64_t>(limit_us) * 1000u, d->status, nullptr) !=
        cudaSuccess)
      st = AR_ERR_CUDA;
  }
  cudaSetDevice(prev);
  if (st != AR_OK) return st;
  return ar_device_status(device, 1);
}

int ar_selftest_bounds(int device) {
  if (device < 0 || device >= kMaxDevices) return AR_ERR_ARG;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  int st = AR_OK;
  DeviceState *d = current_device(&st);
  if (d && launch_bounds_selftest(d->status, nullptr) != cudaSuccess) st = AR_ERR_CUDA;
  cudaSetDevice(prev);
  if (st != AR_OK) return st;
  return ar_device_status(device, 1);
}

int ar_checks_bounds(void) { return AR_CHECK ? 1 : 0; }

int ar_reduce_scatter_flat(const void *const *partials, int n, int64_t count, void *temp,
                           void *stream) {
  if (n < 1 || n > AR_MAX_RANKS || count < 0) return AR_ERR_ARG;
  if (count % kPackElems != 0) return AR_ERR_ALIGN;
  if (count > (int64_t{1} << 40)) return AR_ERR_UNSUPPORTED;
  if (count == 0) return AR_OK;  // nothing is read or written; pointers may be null
  if (!partials || !temp) return AR_ERR_ARG;
  for (int k = 0; k < n; ++k)
    if (!partials[k]) return AR_ERR_ARG;
  if (!aligned16(temp)) return AR_ERR_ALIGN;
  for (int k = 0; k < n; ++k)
    if (!aligned16(partials[k])) return AR_ERR_ALIGN;
  for (int k = 0; k < n; ++k)
    if (overlap(range_of(partials[k], count * 2), range_of(temp, count * 2))) return AR_ERR_ALIAS;
  int st;
  DeviceState *d = current_device(&st);
  if (!d) return st;
  ReduceArgs ra;
  std::memset(&ra, 0, sizeof ra);
  for (int k = 0; k < n; ++k) ra.p[k] = static_cast<const uint4 *>(partials[k]);
  ra.dst[0] = static_cast<uint4 *>(temp);
  ra.ndst = 1;
  ra.begin = 0;
  ra.end = count / kPackElems;
  ra.prefetch = 1;
  ra.status = d->status;
  return launch_reduce_flat(ra, n, d->sms, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? AR_OK
             : AR_ERR_CUDA;
}

int ar_reduce_scatter_store(const void *const *partials, int n, int64_t count, int rank,
                            int world, void *const *temps, void *stream) {
  if (n < 1 || n > AR_MAX_RANKS || count < 0 || world < 1 || world > AR_MAX_RANKS || rank < 0 ||
      rank >= world)
    return AR_ERR_ARG;
  if (count % kPackElems != 0) return AR_ERR_ALIGN;
  if (count > (int64_t{1} << 40)) return AR_ERR_UNSUPPORTED;
  if (count == 0) return AR_OK;  // nothing is read or written; pointers may be null
  if (!partials || !temps) return AR_ERR_ARG;
  for (int k = 0; k < n; ++k)
    if (!partials[k]) return AR_ERR_ARG;
  for (int d = 0; d < world; ++d)
    if (!temps[d]) return AR_ERR_ARG;
  for (int k = 0; k < n; ++k)
    if (!aligned16(partials[k])) return AR_ERR_ALIGN;
  for (int d = 0; d < world; ++d)
    if (!aligned16(temps[d])) return AR_ERR_ALIGN;
  const int64_t bytes = count * 2;
  for (int d = 0; d < world; ++d) {
    const Range t = range_of(temps[d], bytes);
    for (int k = 0; k < n; ++k)
      if (overlap(t, range_of(partials[k], bytes))) return AR_ERR_ALIAS;
    for (int e = d + 1; e < world; ++e)
      if (overlap(t, range_of(temps[e], bytes))) return AR_ERR_ALIAS;
  }
  const int64_t npacks = count / kPackElems;
  const int64_t per = (npacks + world - 1) / world;
  const int64_t begin = static_cast<int64_t>(rank) * per;
  const int64_t end = begin + per < npacks ? begin + per : npacks;
  if (begin >= end) return AR_OK;  // this rank's slice is empty
  int st;
  DeviceState *d = current_device(&st);
  if (!d) return st;
  ReduceArgs ra;
  std::memset(&ra, 0, sizeof ra);
  for (int k = 0; k < n; ++k) ra.p[k] = static_cast<const uint4 *>(partials[k]);
  for (int e = 0; e < world; ++e) ra.dst[e] = static_cast<uint4 *>(temps[e]);
  ra.ndst = world;
  ra.begin = begin;
  ra.end = end;
  ra.status = d->status;
  return launch_reduce_flat(ra, n, d->sms, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? AR_OK
             : AR_ERR_CUDA;
}

// ---------------------------------------------------------------- cross-rank signals

static int check_pads(void *const *pads, int world, int rank) {
  if (world < 1 || world > AR_MAX_RANKS || rank < 0 || rank >= world || !pads) return AR_ERR_ARG;
  for (int d = 0; d < world; ++d)
    if (!pads[d]) return AR_ERR_ARG;
  for (int d = 0; d < world; ++d)
    if (!aligned16(pads[d])) return AR_ERR_ALIGN;
  return AR_OK;
}

static int signal_call(void *const *pads, const void *mine, int world, int rank, uint32_t epoch,
                       unsigned limit_us, bool post, bool wait, void *stream) {
  if (wait && (limit_us == 0 || limit_us > 10000000u)) return AR_ERR_ARG;
  int st;
  DeviceState *d = current_device(&st);
  if (!d) return st;
  SignalArgs a;
  std::memset(&a, 0, sizeof a);
  if (post)
    for (int k = 0; k < world; ++k) a.pads[k] = static_cast<uint32_t *>(pads[k]);
  a.mine = static_cast<uint32_t *>(const_cast<void *>(mine));
  a.world = world;
  a.rank = rank;
  a.post = post;
  a.wait = wait;
  a.epoch = epoch;
  a.limit_ns = static_cast<uint64_t>(limit_us) * 1000u;
  a.status = d->status;
  return launch_signal(a, static_cast<cudaStream_t>(stream)) == cudaSuccess ? AR_OK : AR_ERR_CUDA;
}

int ar_signal_post(void *const *pads, int world, int rank, uint32_t epoch, void *stream) {
  const int st = check_pads(pads, world, rank);
  if (st != AR_OK) return st;
  return signal_call(pads, pads[rank], world, rank, epoch, 0, true, false, stream);
}

int ar_signal_wait(const void *pad, int world, uint32_t epoch, unsigned limit_us, void *stream) {
  if (!pad || world < 1 || world > AR_MAX_RANKS) return AR_ERR_ARG;
  if (!aligned16(pad)) return AR_ERR_ALIGN;
  return signal_call(nullptr, pad, world, 0, epoch, limit_us, false, true, stream);
}

int ar_barrier(void *const *pads, int world, int rank, uint32_t epoch, unsigned limit_us,
               void *stream) {
  const int st = check_pads(pads, world, rank);
  if (st != AR_OK) return st;
  return signal_call(pads, pads[rank], world, rank, epoch, limit_us, true, true, stream);
}

int ar_selftest_barrier(int device, int world, int rounds, unsigned limit_us, int *mismatches) {
  if (device < 0 || device >= kMaxDevices || world < 1 || world > AR_MAX_RANKS || rounds < 1 ||
      rounds > 1000000 || limit_us == 0 || limit_us > 10000000u || !mismatches)
    return AR_ERR_ARG;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  int st = AR_OK;
  DeviceState *d = current_device(&st);
  int *count = nullptr;
  if (d) {
    if (cudaMalloc(&count, sizeof(int)) != cudaSuccess || cudaMemset(count, 0, sizeof(int)) != cudaSuccess ||
        launch_barrier_selftest(world, rounds, static_cast<uint64_t>(limit_us) * 1000u, d->status,
                                count) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(mismatches, count, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
      cudaGetLastError();
      st = AR_ERR_CUDA;
    }
    if (count) cudaFree(count);
  }
  cudaSetDevice(prev);
  if (st != AR_OK) return st;
  return ar_device_status(device, 1);
}

int ar_rmsnorm_two_shot(const void *const *partials, int n, const void *residual,
                        const void *weight, float eps, int64_t m, int64_t H, void *out,
                        void *residual_out, int rank, int world, void *const *temps,
                        void *const *pads, uint32_t epoch, unsigned limit_us, void *stream) {
  int st = check_shape(n, m, H, eps);
  if (st != AR_OK) return st;
  st = check_pads(pads, world, rank);
  if (st != AR_OK) return st;
  if (limit_us == 0 || limit_us > 10000000u) return AR_ERR_ARG;
  if (m == 0) return AR_OK;
  if (!temps) return AR_ERR_ARG;
  for (int e = 0; e < world; ++e)
    if (!temps[e]) return AR_ERR_ARG;
  for (int e = 0; e < world; ++e)
    if (!aligned16(temps[e])) return AR_ERR_ALIGN;
  st = check_buffers(partials, n, residual, weight, m, H, out, residual_out, nullptr);
  if (st != AR_OK) return st;
  const int64_t bytes = m * H * 2;
  for (int e = 0; e < world; ++e) {
    const Range t = range_of(temps[e], bytes);
    for (int k = 0; k < n; ++k)
      if (overlap(t, range_of(partials[k], bytes))) return AR_ERR_ALIAS;
    for (int f = e + 1; f < world; ++f)
      if (overlap(t, range_of(temps[f], bytes))) return AR_ERR_ALIAS;
  }
  const Range mine = range_of(temps[rank], bytes);
  if (overlap(mine, range_of(out, bytes)) || overlap(mine, range_of(residual_out, bytes)) ||
      overlap(mine, range_of(residual, bytes)) || overlap(mine, range_of(weight, H * 2)))
    return AR_ERR_ALIAS;
  DeviceState *d = current_device(&st);
  if (!d) return st;
  ar_plan_t pl;
  st = make_plan(n, m, H, AR_MODE_TWO_STAGE, d->sms, d->smem_optin, nullptr, &pl,
                 device_register_occupancy);
  if (st != AR_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Stage 1: this rank's slice, stored into every rank's temporary.  The
  // partials and temporaries of other ranks are peer mappings: no bulk
  // prefetch there.
  const int64_t npacks = m * H / kPackElems;
  const int64_t per = (npacks + world - 1) / world;
  const int64_t begin = static_cast<int64_t>(rank) * per;
  const int64_t end = begin + per < npacks ? begin + per : npacks;
  if (begin < end) {
    ReduceArgs ra;
    std::memset(&ra, 0, sizeof ra);
    for (int k = 0; k < n; ++k) ra.p[k] = static_cast<const uint4 *>(partials[k]);
    for (int e = 0; e < world; ++e) ra.dst[e] = static_cast<uint4 *>(temps[e]);
    ra.ndst = world;
    ra.prefetch = 0;
    ra.begin = begin;
    ra.end = end;
    ra.status = d->status;
    if (launch_reduce_flat(ra, n, d->sms, s) != cudaSuccess) return AR_ERR_CUDA;
  }
  // Every rank's stores into this rank's temporary have landed.
  st = signal_call(pads, pads[rank], world, rank, epoch, limit_us, true, true, stream);
  if (st != AR_OK) return st;
  // Stage 2 on this rank's (local) temporary.
  const void *temp_in[1] = {temps[rank]};
  cudaError_t e;
  if (pl.kernel == AR_KERNEL_STREAM) {
    e = launch_stream(temp_in, 1, residual, weight, eps, m, H, out, residual_out, nullptr, pl,
                      d->status, true, s);
  } else {
    EpilogueArgs a;
    fill_epilogue_args(&a, temp_in, 1, residual, weight, eps, m, H, out, residual_out, nullptr, pl,
                       d->status);
    e = launch_epilogue(a, 1, pl, true, s);
  }
  return e == cudaSuccess ? AR_OK : AR_ERR_CUDA;
}

int ar_load_rmsnorm(const void *temp, const void *residual, const void *weight, float eps,
                    int64_t m, int64_t H, void *out, void *residual_out, void *stream) {
  const void *inputs[1] = {temp};
  return run(inputs, 1, residual, weight, eps, m, H, out, residual_out, AR_MODE_ONE_STAGE, stream,
             nullptr, nullptr);
}

int ar_reserve_workspace(int64_t max_elems, int device) {
  if (max_elems < 0 || device < 0 || device >= kMaxDevices) return AR_ERR_ARG;
  if (max_elems > (int64_t{1} << 40)) return AR_ERR_UNSUPPORTED;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  if (cudaSetDevice(device) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  int st;
  DeviceState *d = current_device(&st);
  if (d) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (d->workspace_elems < max_elems) {
      if (d->workspace) {
        cudaDeviceSynchronize();
        cudaFree(d->workspace);
        d->workspace = nullptr;
        d->workspace_elems = 0;
      }
      const int64_t elems = (max_elems + 7) / 8 * 8;
      if (cudaMalloc(&d->workspace, static_cast<size_t>(elems) * 2) != cudaSuccess) {
        cudaGetLastError();
        d->workspace = nullptr;
        st = AR_ERR_CUDA;
      } else {
        d->workspace_elems = elems;
      }
    }
  }
  cudaSetDevice(prev);
  return st;
}

int ar_release_workspace(int device) {
  if (device < 0 || device >= kMaxDevices) return AR_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState &d = g_dev[device];
  if (!d.workspace) return AR_OK;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  cudaDeviceSynchronize();
  const cudaError_t e = cudaFree(d.workspace);
  d.workspace = nullptr;
  d.workspace_elems = 0;
  cudaSetDevice(prev);
  return e == cudaSuccess ? AR_OK : AR_ERR_CUDA;
}

int64_t ar_workspace_elems(int device) {
  if (device < 0 || device >= kMaxDevices) return -1;
  std::lock_guard<std::mutex> lock(g_mu);
  return g_dev[device].workspace_elems;
}

int ar_select_mode(int n, int64_t m, int64_t H) {
  if (n < 1 || n > AR_MAX_RANKS || m < 0 || H <= 0) return -AR_ERR_ARG;
  return select_mode(n, m, H);
}

const char *ar_strerror(int status) {
  switch (status) {
    case AR_OK: return "success";
    case AR_ERR_ARG: return "invalid argument (n, m, H, eps, mode or a null pointer)";
    case AR_ERR_ALIGN: return "misaligned: pointers must be 16-byte aligned and H a multiple of 8";
    case AR_ERR_ALIAS: return "overlapping buffers (only residual_out == residual may alias)";
    case AR_ERR_WORKSPACE: return "two-stage workspace missing or too small: call ar_reserve_workspace";
    case AR_ERR_CUDA: return "CUDA runtime error or launch failure";
    case AR_ERR_TIMEOUT: return "a bounded device-side wait timed out";
    case AR_ERR_UNSUPPORTED: return "unsupported size (H above AR_MAX_HIDDEN or too many rows)";
    case AR_ERR_BOUNDS: return "a device-side bounds check failed (checking build)";
    case AR_ERR_SCRATCH_LIMIT:
      return "m*H exceeds the fixed device scratch of ar_rmsnorm_two_stage_static (AR_STATIC_SCRATCH_ELEMS)";
    default: return "unknown status";
  }
}

int ar_version(void) { return 100; }

}  // extern "C"
