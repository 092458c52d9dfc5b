// Host-side handles to the kernel instantiations (one translation unit each).
#pragma once
namespace mk {
const void *kernel_d64();
const void *kernel_d128();
}  // namespace mk
