// C ABI of libarnorm.so: per-device state, argument checks, the launches,
// the two-stage workspace and the single-GPU entry points.  Host code only.
// The launch plan is in plan.cu, the cross-rank entry points in peer.cu.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "host.cuh"

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
StreamKernel stream_kernel_group0(int n, int vpt_log2);
StreamKernel stream_kernel_group1(int n, int vpt_log2);
StreamKernel stream_kernel_group2(int n, int vpt_log2);
StreamKernel stream_kernel_group3(int n, int vpt_log2);
cudaError_t launch_bounded_wait_selftest(uint64_t limit_ns, int *status, cudaStream_t s);
cudaError_t launch_bounds_selftest(int *status, cudaStream_t s);

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
DeviceState *current_device(int *status) {
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

// CTAs of the one-CTA-per-row register kernel (inputs, vpt, late weight)
// with `threads` threads that fit one SM of the current device, from the
// table filled when the device was made ready; 0 where unknown.  No CUDA
// call here, so planning stays safe inside a graph capture.
int device_register_occupancy(int inputs, int vpt, int late, int threads) {
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

// ---------------------------------------------------------------- checks

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const Range &a, const Range &b) { return a.lo < b.hi && b.lo < a.hi; }

Range range_of(const void *p, int64_t bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return Range{lo, lo + static_cast<uintptr_t>(bytes)};
}

int check_shape(int n, int64_t m, int64_t H, float eps) {
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
int check_buffers(const void *const *partials, int n, const void *residual,
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

// Every launch carries programmatic stream serialization: the kernel may be
// scheduled while the previous grid in the stream drains, and waits for it
// (griddepcontrol.wait) before touching global memory.  `after_prior` marks
// stage 2, whose predecessor is stage 1 of the same call: it may read the
// weight and the residual before that wait.
cudaError_t launch_epilogue(const EpilogueArgs &a, int n, const ar_plan_t &pl,
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

cudaError_t launch_stream(const void *const *inputs, int n, const void *residual,
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

void fill_epilogue_args(EpilogueArgs *a, const void *const *inputs, int n, const void *residual,
                        const void *weight, float eps, int64_t m, int64_t H, void *out,
                        void *residual_out, float *sum_out, const ar_plan_t &pl,
                        const DeviceState &d) {
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
  a->status = d.status;
  a->prefetch_own = pl.prefetch == AR_PREFETCH_ROW || pl.prefetch == AR_PREFETCH_ROW_AHEAD;
  a->ahead = pl.prefetch == AR_PREFETCH_ROW_AHEAD
                 ? resident_rows(pl, n, d.sms, device_register_occupancy)
                 : 0;
}

// True if the current device `dev` can use `p` at the same address: its own
// device memory, managed memory, or host memory that is pinned and mapped
// (cudaHostAlloc, cudaHostRegister; with unified addressing the device
// address equals the host address).  Pageable host memory, another device's
// memory and unknown pointers are refused.
bool device_accessible(const void *p, int dev) {
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

int check_mapped(const void *const *partials, int n, const void *residual, const void *weight,
                 const void *out, const void *residual_out) {
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
  if (mapped) {
    st = check_mapped(partials, n, residual, weight, out, residual_out);
    if (st != AR_OK) return st;
  }
  DeviceState *d = current_device(&st);
  if (!d) return st;
  ar_plan_t pl;
  st = make_plan(n, m, H, mode, d->sms, d->smem_optin, force, &pl, device_register_occupancy,
                 mapped);
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
                         sum_out, pl, *d);
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
                       *d);
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
  ar_occupancy_fn occupancy = nullptr;  // pure host logic for a given SM count
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
