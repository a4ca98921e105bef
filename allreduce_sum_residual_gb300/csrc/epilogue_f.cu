// Instantiations of the fused epilogue kernel for stage 2 of the two-shot
// path: one input, with the wait on the signal pad's flags before the
// temporary is read.
#include "epilogue.cuh"

namespace arn {

#define ARN_ROW(CL, LW) {&k_fused_epilogue<1, 1, CL, LW, true>, &k_fused_epilogue<1, 2, CL, LW, true>, \
                         &k_fused_epilogue<1, 4, CL, LW, true>, &k_fused_epilogue<1, 8, CL, LW, true>}

EpilogueKernel epilogue_flag_kernel(int vpt_log2, bool clustered, bool late_weight) {
  static const EpilogueKernel table[3][4] = {ARN_ROW(false, false), ARN_ROW(false, true),
                                             ARN_ROW(true, false)};
  return table[clustered ? 2 : late_weight ? 1 : 0][vpt_log2];
}

}  // namespace arn
