// Device side of the cross-rank signal pads: release/acquire flags at system
// scope (other GPUs see them through peer mappings) and a bounded wait.
//
// A rank's pad is AR_SIGNAL_PAD_BYTES of its own device memory: flags
// 0 .. AR_MAX_RANKS-1 (flag d = the last epoch rank d posted here), the
// rank's own epoch counter, and the arrival counter of its fused stage 1.
#pragma once

#include "common.cuh"

namespace arn {

constexpr int kCounterWord = AR_MAX_RANKS;      // epoch counter (AR_EPOCH_AUTO)
constexpr int kArriveWord = AR_MAX_RANKS + 1;   // CTAs of stage 1 that finished

__device__ __forceinline__ void st_release_sys(uint32_t *p, uint32_t v) {
  asm volatile("st.release.sys.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_sys(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_sys() { asm volatile("fence.acq_rel.sys;" ::: "memory"); }

// atomicAdd with acquire-release semantics at GPU scope: the CTAs of one
// grid count their arrivals on a word of their own GPU's memory.
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

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

// The next epoch of a pad's counter (AR_EPOCH_AUTO), skipping 0.
__device__ __forceinline__ uint32_t next_epoch(uint32_t c) {
  c += 1u;
  return c == AR_EPOCH_AUTO ? 1u : c;
}

}  // namespace arn
