// Host-side handles to the kernel instantiations (one translation unit each).
#pragma once
namespace mk {
const void *kernel_d64();            // general kernel, head_dim 64
const void *kernel_d128();           // general kernel, head_dim 128
const void *kernel_hidden1024();     // PlanHidden1024 (mk_plans.h)
const void *kernel_hidden2048();     // PlanHidden2048
}  // namespace mk
