// Internal layouts shared by the host plan builder (plan.cu) and the kernels
// (adamw_kernels.cu). Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "compact_state.h"

namespace cs {

constexpr int kThreads = 256;              // threads per CTA of the step kernel
constexpr int kWarps = kThreads / 32;
constexpr int kDefaultUnitElems = 32768;   // elements per work unit
constexpr int kInt8Block = CS_INT8_BLOCK;

// One tensor, as the kernel sees it. 64 bytes, one per tensor.
struct alignas(16) TensorDesc {
  void* param;
  const void* grad;
  void* m;
  void* v;
  float* m_scale;
  float* v_scale;
  int64_t numel;
  int16_t group;
  uint8_t param_dtype;   // CS_DTYPE_*
  uint8_t vec_ok;        // every buffer aligned for 4-element vector access
  int32_t n_units;       // work units of this tensor (commit counter target)
};
static_assert(sizeof(TensorDesc) == 64, "descriptor must stay 64 bytes");

// One work unit: `len` elements of tensor `tensor` starting at `start`.
struct alignas(16) WorkUnit {
  int64_t start;
  int32_t tensor;
  int32_t len;
};
static_assert(sizeof(WorkUnit) == 16, "work unit must stay 16 bytes");

// Per-step kernel arguments, passed by value (__grid_constant__). Three size
// classes keep small launches small; the largest fits the 32 KB parameter
// space of a launch.
template <int MAXG, int MAXW>
struct StepArgs {
  const TensorDesc* descs;
  const WorkUnit* units;
  int32_t* step;             // [n_tensors] per-tensor step counts
  const float* inv_scale;    // may be null (1)
  const float* found_inf;    // may be null (0)
  uint32_t* sched;           // [2]: next unit ticket, CTAs finished
  uint32_t* commit;          // [n_tensors]: units of each tensor started
  int32_t n_units;
  int32_t all_present;       // 1: ignore `present`
  adamw_group_t groups[MAXG];
  uint32_t present[MAXW];
};

constexpr int kSmallGroups = 8, kSmallWords = 128;      // <= 4096 tensors
constexpr int kMidGroups = 64, kMidWords = 1024;        // <= 32768 tensors
constexpr int kLargeGroups = 64, kLargeWords = 7680;    // <= 245760 tensors
static_assert(kLargeWords * 32 == CS_MAX_TENSORS, "tensor limit");
static_assert(sizeof(StepArgs<kLargeGroups, kLargeWords>) <= 32764,
              "kernel parameter space");

enum ArgClass { kClassSmall = 0, kClassMid = 1, kClassLarge = 2 };

// Launch one step. Defined in adamw_kernels.cu.
cudaError_t launch_step(int state_kind, ArgClass cls, const void* args,
                        int grid, cudaStream_t stream);
// Max resident CTAs per SM of the kernel for (state_kind, cls).
cudaError_t step_kernel_occupancy(int state_kind, ArgClass cls, int* blocks_per_sm);

}  // namespace cs
