// Step kernels with CS_STATE_DYN8 moments (all argument classes, with and without
// master weights); the kernel itself is in step_kernel.cuh.
#include "step_kernel.cuh"

CS_STEP_KERNEL_TU(dyn8, CS_STATE_DYN8)
