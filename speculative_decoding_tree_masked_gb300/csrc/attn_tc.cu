// Placeholder until the tcgen05 kernel lands: the bf16 path is not enabled.
#include "common.cuh"
#include "internal.h"

namespace tv {
cudaError_t launch_attn_tc(const AttnProblem&, const SplitPlan&, float*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace tv
