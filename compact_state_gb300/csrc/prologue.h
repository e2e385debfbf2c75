// Gradient prologue (prologue.cu): launch arguments and entry points shared
// with the plan code. One pass over a plan's gradients computing the
// non-finite flag, the global L2 norm and the clip factor for the step.
#pragma once

#include "adamw_internal.h"

namespace cs {

constexpr int kPrologueThreads = 256;
constexpr int kProloguePiece = 8192;       // elements per work item
constexpr int kPrologueBlocksPerSm = 8;    // register budget: 32 per thread
constexpr int kPrologueMaxBlocks = 2048;   // partial sums held in the plan's scratch

template <int MAXW>
struct PrologueArgs {
  const TensorDesc* descs;
  const WorkUnit* units;
  const float* inv_scale;    // may be null (1)
  float* found_inf_out;      // device fp32
  float* norm_out;           // device fp32, may be null
  float* scale_out;          // device fp32
  double* partial;           // [gridDim.x] per-block sums of squares
  uint32_t* words;           // [0] blocks finished, [1] non-finite seen
  float max_norm;            // <= 0: no clipping
  int32_t n_units;
  int32_t pieces_per_unit;
  int32_t all_present;
  uint32_t present[MAXW];
};
cudaError_t launch_prologue(ArgClass cls, const void* args, int grid, cudaStream_t stream);
// Resident prologue blocks per SM for an argument class (the grid is one wave).
cudaError_t prologue_occupancy(ArgClass cls, int* blocks_per_sm);

}  // namespace cs
