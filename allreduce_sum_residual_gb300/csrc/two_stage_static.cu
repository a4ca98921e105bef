// ar_rmsnorm_two_stage_static: the two-stage path with its bf16 temporary in
// a fixed array of device memory compiled into the library, for callers that
// cannot allocate device memory (see include/ar_rmsnorm.h).
#include <cstdint>
#include <mutex>

#include "common.cuh"

// The temporary: AR_STATIC_SCRATCH_ELEMS bf16 (16 MiB), 256-byte aligned.
// Every device that loads the library holds its own copy until exit.
static __device__ __align__(256) uint4 g_two_stage_scratch[AR_STATIC_SCRATCH_ELEMS / 8];

namespace arn {

int two_stage_with_temp(const void *const *partials, int n, const void *residual,
                        const void *weight, float eps, int64_t m, int64_t H, void *out,
                        void *residual_out, void *temp, int64_t temp_elems, void *stream);
int check_call_shape(int n, int64_t m, int64_t H, float eps);

namespace {

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxScratchDevices];  // device address of the array, per device

// Device address of this device's array.  In host code the array's name is
// only a host-side stand-in, so the address comes from the runtime, looked
// up once per device with that device current.
int scratch_address(void **addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_two_stage_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return AR_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return AR_OK;
}

}  // namespace
}  // namespace arn

extern "C" int ar_rmsnorm_two_stage_static(const void *const *partials, int n,
                                           const void *residual, const void *weight, float eps,
                                           int64_t m, int64_t H, void *out, void *residual_out,
                                           void *stream) {
  // The same shape checks, in the same order, as every other entry point
  // (n, m, H, eps; then H's alignment and AR_MAX_HIDDEN); then this entry
  // point's own limit; only then is m == 0 a no-op.
  const int shape = arn::check_call_shape(n, m, H, eps);
  if (shape != AR_OK) return shape;
  if (m > AR_STATIC_SCRATCH_ELEMS / H) return AR_ERR_SCRATCH_LIMIT;
  if (m == 0) return AR_OK;
  void *scratch = nullptr;
  const int st = arn::scratch_address(&scratch);
  if (st != AR_OK) return st;
  return arn::two_stage_with_temp(partials, n, residual, weight, eps, m, H, out, residual_out,
                                  scratch, AR_STATIC_SCRATCH_ELEMS, stream);
}
