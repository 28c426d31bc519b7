// Shared stage of the beam attention on the tcgen05 tensor cores (placeholder
// until the tensor-core kernel lands; the planner never selects it yet).
#include "internal.h"

namespace bd {
int launch_attn_shared_tc(const AttnArgs&, const AttnPlan&, cudaStream_t) {
  return BEAMDEC_ERR_UNSUPPORTED;
}
}  // namespace bd
