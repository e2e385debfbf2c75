// Step kernels with CS_STATE_INT8_UV moments (all argument classes, with and without
// master weights); the kernel itself is in step_kernel.cuh.
#include "step_kernel.cuh"

CS_STEP_KERNEL_TU(int8uv, CS_STATE_INT8_UV)
