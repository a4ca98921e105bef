// Instantiations of the streamed epilogue kernel for n = 5 .. 8 inputs.
#include "stream_epilogue.cuh"

namespace arn {

#define ARN_ROW(N) {&k_stream_epilogue<N, 1>, &k_stream_epilogue<N, 2>, \
                    &k_stream_epilogue<N, 4>, &k_stream_epilogue<N, 8>}

StreamKernel stream_kernel_group1(int n, int vpt_log2) {
  static const StreamKernel table[4][4] = {ARN_ROW(5), ARN_ROW(6), ARN_ROW(7), ARN_ROW(8)};
  return table[n - 5][vpt_log2];
}

}  // namespace arn
