// Instantiations of the streamed epilogue kernel for n = 13 .. 16 inputs.
#include "stream_epilogue.cuh"

namespace arn {

#define ARN_ROW(N) {&k_stream_epilogue<N, 1>, &k_stream_epilogue<N, 2>, \
                    &k_stream_epilogue<N, 4>, &k_stream_epilogue<N, 8>}

StreamKernel stream_kernel_group3(int n, int vpt_log2) {
  static const StreamKernel table[4][4] = {ARN_ROW(13), ARN_ROW(14), ARN_ROW(15), ARN_ROW(16)};
  return table[n - 13][vpt_log2];
}

}  // namespace arn
