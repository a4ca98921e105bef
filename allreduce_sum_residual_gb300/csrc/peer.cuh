// Launch interface of the cross-rank signal kernels (peer.cu).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ar_rmsnorm.h"

namespace arn {

struct SignalArgs {
  uint32_t *pads[AR_MAX_RANKS];  // pads[d]: rank d's pad (post), in rank order
  uint32_t *mine;                // this rank's pad (wait)
  int world;
  int rank;                      // slot this rank posts into
  int post;                      // store the epoch into every rank's pad
  int wait;                      // wait for every rank's epoch in `mine`
  uint32_t epoch;
  uint64_t limit_ns;             // bound of the wait
  int *status;
};

cudaError_t launch_signal(const SignalArgs &a, cudaStream_t stream);
cudaError_t launch_barrier_selftest(int world, int rounds, uint64_t limit_ns, int *status,
                                    int *mismatches);

}  // namespace arn
