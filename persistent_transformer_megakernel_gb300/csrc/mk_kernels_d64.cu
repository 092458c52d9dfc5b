// head_dim 64 instantiation of the general decode megakernel
#include "mk_device.cuh"
#include "mk_launch.h"

namespace mk {
const void *kernel_d64() { return reinterpret_cast<const void *>(&mk_decode_kernel<64, PlanGeneral>); }
}  // namespace mk
