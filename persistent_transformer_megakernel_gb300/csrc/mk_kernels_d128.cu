// head_dim 128 instantiation of the general decode megakernel
#include "mk_device.cuh"
#include "mk_launch.h"

namespace mk {
const void *kernel_d128() { return reinterpret_cast<const void *>(&mk_decode_kernel<128, PlanGeneral>); }
}  // namespace mk
