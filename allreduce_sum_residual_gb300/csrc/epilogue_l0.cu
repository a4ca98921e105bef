// Instantiations of the fused epilogue kernel for n = 1 .. 4 partials,
// launched with one CTA per row, the weight loaded after the sums.
// (Split over several translation units so that they compile in parallel.)
#include "epilogue.cuh"

namespace arn {

#define ARN_ROW(N) {&k_fused_epilogue<N, 1, false, true>, &k_fused_epilogue<N, 2, false, true>, \
                    &k_fused_epilogue<N, 4, false, true>, &k_fused_epilogue<N, 8, false, true>}

EpilogueKernel epilogue_late_kernel_group0(int n, int vpt_log2) {
  static const EpilogueKernel table[4][4] = {ARN_ROW(1), ARN_ROW(2), ARN_ROW(3), ARN_ROW(4)};
  return table[n - 1][vpt_log2];
}

}  // namespace arn
