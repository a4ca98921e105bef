// The launch plan: which path (one- or two-stage), which kernel and which
// launch shape a call gets, from the measured table of plan_table.cuh and
// the device's occupancy figures.  Pure host logic (no CUDA call), so it is
// safe inside a graph capture; ar_get_plan / ar_get_plan_ex expose it.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "host.cuh"
#include "plan_table.cuh"

namespace arn {

// ---------------------------------------------------------------- policy

// One-stage up to this many rows, two-stage above.  Measured on GB300 with
// both paths at n in {4, 8}, H in {4096, 8192}, m = 1 .. 16384 (the bench's
// sweep mode, cold buffers, graphs of back-to-back calls): one-stage was
// faster at every point -- by 1.1-1.6 us at m <= 64 (two-stage adds a launch)
// and by 1.09-1.42x at m >= 512 (two-stage moves (n+5)/(n+3) of the bytes).
// On one GPU there is no cross-GPU traffic for the two-stage reduce-scatter
// to save, so the threshold is unbounded for every (n, H).  (The pages' rule,
// one-stage for m <= 32 at 4 ranks and m <= 16 at 8, was set on MI355X
// across GPUs: ROCm/aiter #3817, Test Results.)
static int64_t one_stage_max_rows(int n, int64_t H) {
  (void)n;
  (void)H;
  return INT64_MAX;
}

int select_mode(int n, int64_t m, int64_t H) {
  return m <= one_stage_max_rows(n, H) ? AR_MODE_ONE_STAGE : AR_MODE_TWO_STAGE;
}

// Kernel choice from 64 rows on, for rows up to the table's longest (2048
// packs, H = 16384): the lookup table of plan_table.cuh, measured on GB300.
// For every (inputs, packs per row, rows) of its grid it holds each
// candidate's speed as a percentage of the fastest there: the stream kernel
// and the register kernel with 1, 2, 4 or 8 packs per thread, with the
// weight loaded early or late (one-stage, cold buffers, CUDA-graph timing;
// repeated sweeps agreed within 0.5 %).  Rows of more than 1024 packs are
// split over a 2-CTA cluster, where the late forms do not run.
// No simple rule fits it: which kernel wins turns on how many CTAs of each
// fit an SM (the register counts of each instantiation), whether the rows
// fill a whole number of waves, and how many bytes are then in flight --
// one more wave of a few rows can cost 25 %.  Between grid points the
// percentages of the grid cells that bracket the shape (two columns per
// axis where it falls between two: inputs, packs, rows) are averaged and
// the best mean wins, which prefers a candidate that is good on both sides
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

using OccupancyFn = ar_occupancy_fn;

// `occupancy` (may be null) makes the rows interpolation wave-aware.  A
// register-kernel candidate runs its rows in waves of (CTAs per SM x SMs);
// where the two bracketing rows columns lie in different wave counts for
// it, only the column with the shape's own wave count is used for that
// candidate: one more, mostly idle wave costs up to 25 %, so the column
// across the wave boundary does not describe the shape.  (Held out against
// the sweep, this lifted the pick from 0.984 to 0.990 of the best candidate
// on average.)  Candidates are compared by their mean percentage.
// `no_stream` leaves the stream kernel (candidate 0) out.
static TableChoice table_choice(int inputs, int64_t m, int64_t P, int sms,
                                OccupancyFn occupancy, bool no_stream) {
  if (m < kTableMinRows || P > last_of(kPlanPacks)) return {0, 0};
  int n0, n1, p0, p1, m0, m1;
  bracket(kPlanInputs, static_cast<double>(inputs), &n0, &n1);
  bracket(kPlanPacks, static_cast<double>(P), &p0, &p1);
  const double rows = static_cast<double>(m) * kPlanTableSms / sms;  // in the table's SMs
  bracket(kPlanRows, rows, &m0, &m1);
  const int first = no_stream ? 1 : 0;
  int best = first;
  double best_mean = -1.0;
  for (int c = first; c < kPlanCandidates; ++c) {
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

// Rows beyond the table (more than 2048 packs), and below its shortest
// rows column where the table does not apply: the stream kernel for 4
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
//    rows, or rows beyond the table) 1 pack per thread, the most
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

int64_t stream_smem_bytes(int inputs, int consumers, int stages) {
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
int64_t resident_rows(const ar_plan_t &pl, int inputs, int sms, OccupancyFn occupancy) {
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

int make_plan(int n, int64_t m, int64_t H, int mode, int sms, int smem_optin,
              const ar_plan_t *force, ar_plan_t *pl, OccupancyFn occupancy, bool plain_loads) {
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
    if (plain_loads && fk == AR_KERNEL_STREAM) return AR_ERR_ARG;
  }
  const int64_t P = H / kPackElems;
  const int inputs = pl->mode == AR_MODE_TWO_STAGE ? 1 : n;
  const bool shape_forced = fc != 0 || fv != 0;
  const TableChoice choice = table_choice(inputs, m, P, sms, occupancy, plain_loads);
  bool want_stream = fk == AR_KERNEL_STREAM;
  if (fk == AR_KERNEL_AUTO && !shape_forced && !plain_loads)
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
  if (plain_loads) pl->prefetch = AR_PREFETCH_NONE;
  return AR_OK;
}

}  // namespace arn
