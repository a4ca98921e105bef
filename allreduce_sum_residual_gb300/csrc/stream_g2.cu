// Instantiations of the streamed epilogue kernel for n = 9 .. 12 inputs.
#include "stream_epilogue.cuh"

namespace arn {

#define ARN_ROW(N) {&k_stream_epilogue<N, 1>, &k_stream_epilogue<N, 2>, \
                    &k_stream_epilogue<N, 4>, &k_stream_epilogue<N, 8>}

StreamKernel stream_kernel_group2(int n, int vpt_log2) {
  static const StreamKernel table[4][4] = {ARN_ROW(9), ARN_ROW(10), ARN_ROW(11), ARN_ROW(12)};
  return table[n - 9][vpt_log2];
}

}  // namespace arn
