// Tensor-core (tcgen05 / TMEM) verify kernel: not built yet.
#include <cuda_runtime.h>

#include "vmla_internal.h"

namespace vmla {
int launch_tc(const PlanParams&, const RunArgs&, void*) { return VMLA_ERR_DEVICE; }
}  // namespace vmla
