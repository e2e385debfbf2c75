// Dispatch of a step launch to the kernels of its state kind (each compiled
// in its own translation unit, step_kernel_<kind>.cu).
#include "adamw_internal.h"

namespace cs {

cudaError_t launch_step_f32(ArgClass, int, const void*, int, cudaStream_t);
cudaError_t launch_step_bf16(ArgClass, int, const void*, int, cudaStream_t);
cudaError_t launch_step_int8(ArgClass, int, const void*, int, cudaStream_t);
cudaError_t launch_step_int8uv(ArgClass, int, const void*, int, cudaStream_t);
cudaError_t launch_step_dyn8(ArgClass, int, const void*, int, cudaStream_t);
cudaError_t step_occupancy_f32(ArgClass, int, int*);
cudaError_t step_occupancy_bf16(ArgClass, int, int*);
cudaError_t step_occupancy_int8(ArgClass, int, int*);
cudaError_t step_occupancy_int8uv(ArgClass, int, int*);
cudaError_t step_occupancy_dyn8(ArgClass, int, int*);

cudaError_t launch_step(int state_kind, ArgClass cls, int variant, const void* args, int grid,
                        cudaStream_t stream) {
  switch (state_kind) {
    case CS_STATE_F32: return launch_step_f32(cls, variant, args, grid, stream);
    case CS_STATE_BF16: return launch_step_bf16(cls, variant, args, grid, stream);
    case CS_STATE_INT8: return launch_step_int8(cls, variant, args, grid, stream);
    case CS_STATE_INT8_UV: return launch_step_int8uv(cls, variant, args, grid, stream);
    case CS_STATE_DYN8: return launch_step_dyn8(cls, variant, args, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t step_kernel_occupancy(int state_kind, ArgClass cls, int variant,
                                  int* blocks_per_sm) {
  switch (state_kind) {
    case CS_STATE_F32: return step_occupancy_f32(cls, variant, blocks_per_sm);
    case CS_STATE_BF16: return step_occupancy_bf16(cls, variant, blocks_per_sm);
    case CS_STATE_INT8: return step_occupancy_int8(cls, variant, blocks_per_sm);
    case CS_STATE_INT8_UV: return step_occupancy_int8uv(cls, variant, blocks_per_sm);
    case CS_STATE_DYN8: return step_occupancy_dyn8(cls, variant, blocks_per_sm);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cs
