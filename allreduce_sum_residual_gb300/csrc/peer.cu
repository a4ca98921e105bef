// The cross-rank data plane of the all-reduce: the buffers of every rank
// mapped into each rank's address space (CUDA IPC handles), a bounded flag
// barrier, and the two entry points built on it -- the two-shot path
// (stage 1 into every rank's temporary, barrier, stage 2) and the one-shot
// path (barrier, the epilogue over every rank's partial, barrier).
//
// ROCm/aiter #3817 "perf: optimize fused AllReduce + RMSNorm
// (custom_all_reduce)", Technical Details, 2stage, reduce-scatter: stage 1
// of every rank stores its reduced slice straight into the temporary buffer
// of every rank, so before stage 2 reads its own temporary every rank's
// stores must have landed -- a cross-rank synchronisation the page implies
// but does not describe.  lightseekorg/tokenspeed #968 "perf(comm): add
// opt-in Triton AR+RMSNorm backend" maps the ranks' buffers with HIP IPC
// handles and synchronises through signal flags; its review adds that a
// rank which fails alone must not leave its peers waiting forever.  The
// PyTorch symmetric-memory pages (pytorch #137643 stack) wait on a signal
// pad in the same way.
//
// Here: every rank owns a signal pad of AR_MAX_RANKS 32-bit flags in its
// own device memory, zeroed before first use.  Rank r "posts" epoch e by
// storing e into flag r of every rank's pad (release, system scope, after a
// system-scope fence that orders every write the previous grids made), and
// "waits" for epoch e by spinning on every flag of its own pad until each
// holds e or later (acquire, system scope).  Every wait is bounded by
// %globaltimer: on timeout the kernel records AR_ERR_TIMEOUT in the device
// status word and returns, so a missing peer becomes an error the host can
// read rather than a hang.  No multicast or NVLS object is involved: plain
// loads and stores through peer mappings.
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <string>

#include "common.cuh"
#include "host.cuh"
#include "peer.cuh"

namespace arn {

__device__ __forceinline__ void st_release_sys(uint32_t *p, uint32_t v) {
  asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_sys(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_sys() { asm volatile("fence.acq_rel.sys;" ::: "memory"); }

// Epoch e has been reached by a flag holding f when f - e, as a signed
// 32-bit difference, is not negative (so epochs may wrap around).
__device__ __forceinline__ bool reached(uint32_t f, uint32_t e) {
  return static_cast<int32_t>(f - e) >= 0;
}

// Spin until *flag reaches epoch, for at most limit_ns; false on timeout.
__device__ __forceinline__ bool wait_flag(const uint32_t *flag, uint32_t epoch, uint64_t limit_ns) {
  if (reached(ld_acquire_sys(flag), epoch)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(64);
    if (reached(ld_acquire_sys(flag), epoch)) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Word of a pad holding its owner's epoch counter (after the 16 flags).
constexpr int kCounterWord = AR_MAX_RANKS;

// One warp: lane d posts into rank d's pad, lane j waits for rank j's flag.
__global__ void __launch_bounds__(32) k_signal(const __grid_constant__ SignalArgs a) {
  // Everything the previous grids wrote (stage 1's stores into the peers'
  // temporaries) is complete once this returns; the fence below makes it
  // visible at system scope before the flag says so.
  pdl_wait_prior_grid();
  pdl_launch_dependents();
  const int t = static_cast<int>(threadIdx.x);
  // Checking build: a rank count the pad holds and a slot inside it.
  if (!in_bounds(a.world >= 1 && a.world <= AR_MAX_RANKS && a.rank >= 0 && a.rank < a.world,
                 a.status))
    return;
  // AR_EPOCH_AUTO: the epoch is this rank's counter, kept in its own pad and
  // touched only by its owner's calls (in stream order): a post moves it on.
  uint32_t epoch = a.epoch;
  if (epoch == AR_EPOCH_AUTO) {
    uint32_t c = 0;
    if (t == 0) {
      c = a.mine[kCounterWord];
      if (a.post) {
        c += 1u;
        if (c == AR_EPOCH_AUTO) c = 1u;
        a.mine[kCounterWord] = c;
      }
    }
    epoch = __shfl_sync(0xFFFFFFFFu, c, 0);
  }
  if (a.post && t < a.world) {
    fence_sys();
    st_release_sys(a.pads[t] + a.rank, epoch);
  }
  // In a barrier, lane `rank` has just stored this rank's own flag (mine is
  // pads[rank]); its wait would only re-read its own store, and skipping it
  // took 0.3 us off the one- and two-shot calls at decode size.
  if (a.wait && t < a.world && !(a.post && t == a.rank) &&
      !wait_flag(a.mine + t, epoch, a.limit_ns))
    atomicExch(a.status, AR_ERR_TIMEOUT);
  __syncwarp();
}

cudaError_t launch_signal(const SignalArgs &a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, k_signal, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------- self-test
//
// All ranks of a barrier in one kernel: CTA r plays rank r.  A cooperative
// launch guarantees that the `world` CTAs run at the same time (or the
// launch fails), which ranks that wait on one another need.  Each round e,
// rank r writes a value into its data slot of round parity e, posts epoch
// e, waits for every rank, then reads every rank's slot of that parity: the
// release/acquire pair must make each peer's value of round e visible.
// (With two parities no rank can overwrite a slot before every rank has
// read it: writing it again needs round e + 2, which needs every rank's
// post of round e + 1, which each makes after its reads of round e.)

static __device__ uint32_t g_selftest_pads[AR_MAX_RANKS * AR_MAX_RANKS];
static __device__ uint32_t g_selftest_data[2 * AR_MAX_RANKS];

__global__ void __launch_bounds__(32)
k_barrier_selftest(int world, int rounds, uint64_t limit_ns, int *status, int *mismatches) {
  const int rank = static_cast<int>(blockIdx.x);
  const int t = static_cast<int>(threadIdx.x);
  for (int e = 1; e <= rounds; ++e) {
    const int parity = e & 1;
    if (t == 0) g_selftest_data[parity * AR_MAX_RANKS + rank] = static_cast<uint32_t>(e * 1000 + rank);
    __syncwarp();
    if (t < world) {
      fence_sys();
      st_release_sys(g_selftest_pads + t * AR_MAX_RANKS + rank, static_cast<uint32_t>(e));
    }
    bool ok = true;
    if (t < world) {
      ok = wait_flag(g_selftest_pads + rank * AR_MAX_RANKS + t, static_cast<uint32_t>(e), limit_ns);
      if (!ok) {
        atomicExch(status, AR_ERR_TIMEOUT);
      } else {
        const uint32_t v = *reinterpret_cast<volatile uint32_t *>(
            &g_selftest_data[parity * AR_MAX_RANKS + t]);
        if (v != static_cast<uint32_t>(e * 1000 + t)) atomicAdd(mismatches, 1);
      }
    }
    if (__any_sync(0xFFFFFFFFu, !ok)) return;  // a rank is missing: stop, do not wait again
    __syncwarp();
  }
}

cudaError_t launch_barrier_selftest(int world, int rounds, uint64_t limit_ns, int *status,
                                    int *mismatches) {
  void *pads = nullptr, *data = nullptr;
  if (cudaGetSymbolAddress(&pads, g_selftest_pads) != cudaSuccess ||
      cudaGetSymbolAddress(&data, g_selftest_data) != cudaSuccess)
    return cudaGetLastError();
  cudaError_t e = cudaMemset(pads, 0, sizeof(g_selftest_pads));
  if (e == cudaSuccess) e = cudaMemset(data, 0, sizeof(g_selftest_data));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(world), 1, 1);
  cfg.blockDim = dim3(32, 1, 1);
  cfg.stream = nullptr;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k_barrier_selftest, world, rounds, limit_ns, status, mismatches);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------- IPC handles

namespace {

// cuMemGetAddressRange, looked up from the driver at run time (the library
// links only the runtime): the start of the allocation holding a pointer,
// since an IPC handle names a whole allocation.
using AddressRangeFn = int (*)(unsigned long long *base, size_t *size, unsigned long long ptr);

AddressRangeFn address_range_fn() {
  static std::once_flag once;
  static AddressRangeFn fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<AddressRangeFn>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

// Allocations of other processes opened in this one, by handle: a handle
// may be opened once per process, so repeated opens share the mapping.
struct Opened {
  void *base;
  int refs;
};
std::mutex g_ipc_mu;
std::map<std::string, Opened> g_opened;

std::string key_of(const void *handle) {
  return std::string(static_cast<const char *>(handle), sizeof(cudaIpcMemHandle_t));
}

}  // namespace
}  // namespace arn

using namespace arn;

extern "C" {

int ar_ipc_get_handle(const void *ptr, void *handle, int64_t *offset) {
  if (!ptr || !handle || !offset) return AR_ERR_ARG;
  const AddressRangeFn range = address_range_fn();
  if (!range) return AR_ERR_CUDA;
  unsigned long long base = 0;
  size_t size = 0;
  if (range(&base, &size, reinterpret_cast<unsigned long long>(ptr)) != 0 || base == 0)
    return AR_ERR_ARG;  // not device memory of this process
  cudaIpcMemHandle_t h;
  if (cudaIpcGetMemHandle(&h, reinterpret_cast<void *>(base)) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  std::memcpy(handle, &h, sizeof h);
  *offset = static_cast<int64_t>(reinterpret_cast<unsigned long long>(ptr) - base);
  return AR_OK;
}

int ar_ipc_open(const void *handle, int64_t offset, void **ptr) {
  if (!handle || !ptr || offset < 0) return AR_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_ipc_mu);
  const std::string key = key_of(handle);
  auto it = g_opened.find(key);
  if (it == g_opened.end()) {
    cudaIpcMemHandle_t h;
    std::memcpy(&h, handle, sizeof h);
    void *base = nullptr;
    if (cudaIpcOpenMemHandle(&base, h, cudaIpcMemLazyEnablePeerAccess) != cudaSuccess) {
      cudaGetLastError();
      return AR_ERR_CUDA;
    }
    it = g_opened.emplace(key, Opened{base, 0}).first;
  }
  ++it->second.refs;
  *ptr = static_cast<char *>(it->second.base) + offset;
  return AR_OK;
}

int ar_ipc_close(const void *handle) {
  if (!handle) return AR_ERR_ARG;
  std::lock_guard<std::mutex> lock(g_ipc_mu);
  auto it = g_opened.find(key_of(handle));
  if (it == g_opened.end()) return AR_ERR_ARG;
  if (--it->second.refs > 0) return AR_OK;
  const cudaError_t e = cudaIpcCloseMemHandle(it->second.base);
  g_opened.erase(it);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  return AR_OK;
}

// ---------------------------------------------------------------- signals, barrier, two-shot

static int check_pads(void *const *pads, int world, int rank) {
  if (world < 1 || world > AR_MAX_RANKS || rank < 0 || rank >= world || !pads) return AR_ERR_ARG;
  for (int d = 0; d < world; ++d)
    if (!pads[d]) return AR_ERR_ARG;
  for (int d = 0; d < world; ++d)
    if (!aligned16(pads[d])) return AR_ERR_ALIGN;
  return AR_OK;
}

// The epoch of a call's second barrier: e + 1 (1 where that wraps to 0), or
// AR_EPOCH_AUTO again, which takes the next value of the pad's counter.
static uint32_t next_epoch(uint32_t e) {
  return e == AR_EPOCH_AUTO ? AR_EPOCH_AUTO : (e + 1u == 0u ? 1u : e + 1u);
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
  // Every pointer reachable from this device (its own, IPC or peer memory).
  st = check_mapped(partials, n, residual, weight, out, residual_out);
  if (st != AR_OK) return st;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  for (int e = 0; e < world; ++e)
    if (!device_accessible(temps[e], dev)) return AR_ERR_ARG;
  DeviceState *d = current_device(&st);
  if (!d) return st;
  ar_plan_t pl;
  st = make_plan(n, m, H, AR_MODE_TWO_STAGE, d->sms, d->smem_optin, nullptr, &pl,
                 device_register_occupancy);
  if (st != AR_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Every rank's partial is written: stage 1 reads a slice of each.
  st = signal_call(pads, pads[rank], world, rank, epoch, limit_us, true, true, stream);
  if (st != AR_OK) return st;
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
  st = signal_call(pads, pads[rank], world, rank, next_epoch(epoch), limit_us, true, true, stream);
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
                       *d);
    e = launch_epilogue(a, 1, pl, true, s);
  }
  return e == cudaSuccess ? AR_OK : AR_ERR_CUDA;
}

int ar_rmsnorm_one_shot(const void *const *partials, int n, const void *residual,
                        const void *weight, float eps, int64_t m, int64_t H, void *out,
                        void *residual_out, int rank, int world, void *const *pads,
                        uint32_t epoch, unsigned limit_us, int end_barrier, void *stream) {
  int st = check_shape(n, m, H, eps);
  if (st != AR_OK) return st;
  st = check_pads(pads, world, rank);
  if (st != AR_OK) return st;
  if (limit_us == 0 || limit_us > 10000000u || (end_barrier != 0 && end_barrier != 1))
    return AR_ERR_ARG;
  if (m == 0) return AR_OK;
  st = check_buffers(partials, n, residual, weight, m, H, out, residual_out, nullptr);
  if (st != AR_OK) return st;
  st = check_mapped(partials, n, residual, weight, out, residual_out);
  if (st != AR_OK) return st;
  DeviceState *d = current_device(&st);
  if (!d) return st;
  // The plan of ar_rmsnorm_mapped's one-stage path: the register kernel with
  // plain loads, no bulk prefetch (other ranks' partials are mappings).
  ar_plan_t pl;
  st = make_plan(n, m, H, AR_MODE_ONE_STAGE, d->sms, d->smem_optin, nullptr, &pl,
                 device_register_occupancy, true);
  if (st != AR_OK) return st;
  // Every rank's partial is written.
  st = signal_call(pads, pads[rank], world, rank, epoch, limit_us, true, true, stream);
  if (st != AR_OK) return st;
  // The epilogue over every rank's partial.  Its predecessor is the barrier
  // kernel, which writes only flags, so the residual and weight are read
  // before its wait and the partials after it.
  EpilogueArgs a;
  fill_epilogue_args(&a, partials, n, residual, weight, eps, m, H, out, residual_out, nullptr, pl,
                     *d);
  if (launch_epilogue(a, n, pl, true, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return AR_ERR_CUDA;
  if (!end_barrier) return AR_OK;
  // No rank reads a partial any more: each may overwrite its own.
  return signal_call(pads, pads[rank], world, rank, next_epoch(epoch), limit_us, true, true,
                     stream);
}

}  // extern "C"
