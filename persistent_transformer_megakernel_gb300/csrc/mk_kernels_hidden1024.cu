// the decode megakernel compiled for PlanHidden1024 (mk_plans.h)
#include "mk_device.cuh"
#include "mk_launch.h"

namespace mk {
const void *kernel_hidden1024() { return reinterpret_cast<const void *>(&mk_decode_kernel<128, PlanHidden1024>); }
}  // namespace mk
