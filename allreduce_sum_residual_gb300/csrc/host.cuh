// Host-side pieces shared by the C ABI's translation units (abi.cu,
// plan.cu, peer.cu): per-device state, argument checks, the launch plan
// and the launches.  Host code only; no kernel includes this.
#pragma once

#include <cstdint>

#include "epilogue.cuh"
#include "stream_epilogue.cuh"

namespace arn {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait
constexpr int kAssumedSmemOptin = 232448;         // sm_100-class opt-in per CTA (host-only plans)
constexpr int kMaxDevices = 64;

inline int vpt_log2(int vpt) { return vpt == 1 ? 0 : vpt == 2 ? 1 : vpt == 4 ? 2 : vpt == 8 ? 3 : -1; }

struct DeviceState {
  bool ready = false;        // attributes read and kernel attributes set
  int sms = 0;
  int smem_optin = 0;        // largest dynamic shared memory per CTA
  int *status = nullptr;     // this device's g_arn_status
  void *workspace = nullptr; // two-stage bf16 temporary
  int64_t workspace_elems = 0;
};

// The current device, made ready (SM count, kernel attributes, occupancy
// table) on first use, which must be outside graph capture; null on error
// (*status set).
DeviceState *current_device(int *status);

// CTAs per SM of the one-CTA register kernel on the current device, from
// the table filled when it was made ready (0 if unknown); no CUDA call
// beyond cudaGetDevice.
int device_register_occupancy(int inputs, int vpt, int late, int threads);

// --- checks (abi.cu)
struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};
bool aligned16(const void *p);
bool overlap(const Range &a, const Range &b);
Range range_of(const void *p, int64_t bytes);
int check_shape(int n, int64_t m, int64_t H, float eps);
int check_buffers(const void *const *partials, int n, const void *residual, const void *weight,
                  int64_t m, int64_t H, const void *out, const void *residual_out,
                  const void *sum_out);
// Every pointer usable by the current device at its own address (its own or
// an IPC allocation, a peer GPU's memory it can reach, managed or mapped
// pinned host memory): AR_OK, else AR_ERR_ARG (AR_ERR_CUDA if the device
// cannot be queried).
int check_mapped(const void *const *partials, int n, const void *residual, const void *weight,
                 const void *out, const void *residual_out);
// One pointer of check_mapped's kinds, for device `dev`.
bool device_accessible(const void *p, int dev);

// --- the launch plan (plan.cu)
int select_mode(int n, int64_t m, int64_t H);
int64_t stream_smem_bytes(int inputs, int consumers, int stages);
int64_t resident_rows(const ar_plan_t &pl, int inputs, int sms, ar_occupancy_fn occupancy);
// `plain_loads`: the plan for buffers that may lie outside this GPU's own
// memory (host, IPC or peer mappings): the best register-kernel candidate
// (the stream kernel's bulk copies are left out) and no bulk L2 prefetch.
int make_plan(int n, int64_t m, int64_t H, int mode, int sms, int smem_optin,
              const ar_plan_t *force, ar_plan_t *pl, ar_occupancy_fn occupancy = nullptr,
              bool plain_loads = false);

// --- launches (abi.cu, reduce_flat.cu)
// The epilogue kernel's arguments for a plan on device `d` (its status
// word; its SM count sets the prefetch distance one wave ahead).
void fill_epilogue_args(EpilogueArgs *a, const void *const *inputs, int n, const void *residual,
                        const void *weight, float eps, int64_t m, int64_t H, void *out,
                        void *residual_out, float *sum_out, const ar_plan_t &pl,
                        const DeviceState &d);
cudaError_t launch_epilogue(const EpilogueArgs &a, int n, const ar_plan_t &pl, bool after_prior,
                            cudaStream_t stream);
cudaError_t launch_stream(const void *const *inputs, int n, const void *residual,
                          const void *weight, float eps, int64_t m, int64_t H, void *out,
                          void *residual_out, float *sum_out, const ar_plan_t &pl, int *status,
                          bool after_prior, cudaStream_t stream);
cudaError_t launch_reduce_flat(const ReduceArgs &a, int n, int sms, cudaStream_t stream);

}  // namespace arn
