// the decode megakernel compiled for PlanHidden2048 (mk_plans.h)
#include "mk_device.cuh"
#include "mk_launch.h"

namespace mk {
const void *kernel_hidden2048() { return reinterpret_cast<const void *>(&mk_decode_kernel<128, PlanHidden2048>); }
}  // namespace mk
