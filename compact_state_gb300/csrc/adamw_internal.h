// Internal layouts shared by the host plan builder (plan.cu) and the kernels
// (step_kernel.cuh). Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "compact_state.h"

namespace cs {

#ifndef CS_WARPS_ELEMENTWISE
#define CS_WARPS_ELEMENTWISE 24   // compute warps per CTA, fp32 moments
#endif
#ifndef CS_WARPS_BF16
#define CS_WARPS_BF16 12          // compute warps per CTA, bf16 moments
#endif
#ifndef CS_WARPS_INT8
#define CS_WARPS_INT8 16          // compute warps per CTA, 8-bit moments
#endif

constexpr int kDefaultUnitElems = CS_NOALLOC_UNIT;     // elements per work unit
constexpr int kInt8Block = CS_INT8_BLOCK;
constexpr int kProducerWarps = 2;                      // tile publisher + unit fetcher
constexpr int kStageBudget = 216 * 1024;               // dynamic shared memory for stages
constexpr uint64_t kDefaultWaitNs = 2000000000ull;     // 2 s bound on every wait

// The 8-bit state kinds share one kernel shape (whole 256-element blocks per
// compute warp, one byte per moment element).
constexpr bool is_8bit(int state_kind) {
  return state_kind == CS_STATE_INT8 || state_kind == CS_STATE_INT8_UV ||
         state_kind == CS_STATE_DYN8;
}

// Kernel variants of one state kind, chosen per plan:
//   kVarPlain     -- every param dtype, no master weights;
//   kVarExtended  -- also tensors with fp32 master weights or, in an 8-bit
//                    plan, tensors kept in fp32 moments (extra per-tile cases
//                    that cost the plain paths up to 5% when always built in);
//   kVarP16       -- 8-bit kinds only, every param and grad 16-bit and none of
//                    the extended cases: the stage holds 2-byte params, so a
//                    stage of the same shared memory holds twice the tile, and
//                    each compute warp takes two blocks of it with their code
//                    interleaved (twice the independent work per warp, the
//                    per-tile wait and dispatch paid once per two blocks);
//   kVarP16Pack   -- kVarP16 for lists with small units (kPackMax elements or
//                    fewer), which it packs several to a stage;
//   kVarPlainPack -- kVarPlain for lists with small units, packing them (every
//                    kind but the codebook one, whose tables leave no shared
//                    memory for the segment table).
// The packing kernels are kernels of their own: packing code inside kVarP16
// cost the Llama-3-8B list with int8 moments 0.4-1% of its rate, inside the
// bf16-moment kVarPlain 1.5%, through code generation alone (lists without
// small units never pack).
enum Variant : int {
  kVarPlain = 0, kVarExtended = 1, kVarP16 = 2, kVarP16Pack = 3, kVarPlainPack = 4
};
constexpr int kVariants = 5;
constexpr bool is_p16(int variant) { return variant == kVarP16 || variant == kVarP16Pack; }
// Units of at most this many elements are packed (packing kernels only).
constexpr int kPackMax = 1536;

// bf16 moments move the fewest bytes per element of the elementwise kinds,
// so their tiles come fastest; with 12 warps each thread takes two 4-element
// groups per tile and the per-tile overhead (wait, metadata, dispatch) is
// paid half as often (measured: 320 -> 289 us on 8 x 4096^2 bf16/bf16).
constexpr int consumer_warps(int state_kind) {
  return is_8bit(state_kind)                ? CS_WARPS_INT8
         : state_kind == CS_STATE_BF16      ? CS_WARPS_BF16
                                            : CS_WARPS_ELEMENTWISE;
}
constexpr int block_threads(int state_kind) {
  return 32 * (kProducerWarps + consumer_warps(state_kind));
}
// 256-element blocks per compute warp per tile (8-bit kinds).
constexpr int blocks_per_warp(int variant) { return is_p16(variant) ? 2 : 1; }
// Elements per pipeline stage: 3072 for fp32/bf16 moments (one 4-element
// group per compute thread with fp32 moments, two with bf16); for the 8-bit
// kinds one 256-element block per compute warp, two with kVarP16.
constexpr int kElementwiseTile = 3072;
constexpr int tile_elems(int state_kind, int variant = kVarPlain) {
  return is_8bit(state_kind) ? consumer_warps(state_kind) * blocks_per_warp(variant) * kInt8Block
                             : kElementwiseTile;
}
// Bytes of one pipeline stage: params sized for fp32 (the widest param type,
// since it varies per tensor), or for 16-bit params in kVarP16.
constexpr int stage_bytes(int state_kind, int variant = kVarPlain) {
  return state_kind == CS_STATE_F32    ? tile_elems(state_kind) * 16
         : state_kind == CS_STATE_BF16 ? tile_elems(state_kind) * 12
                                       : tile_elems(state_kind, variant) *
                                                 (is_p16(variant) ? 6 : 10) +
                                             2 * (tile_elems(state_kind, variant) / kInt8Block) * 4;
}
constexpr int stages_for(int state_kind, int variant = kVarPlain) {
  return kStageBudget / ((stage_bytes(state_kind, variant) + 127) / 128 * 128) > 16
             ? 16
             : kStageBudget / ((stage_bytes(state_kind, variant) + 127) / 128 * 128);
}
static_assert(tile_elems(CS_STATE_INT8) % 1024 == 0 && tile_elems(CS_STATE_F32) % 1024 == 0 &&
                  tile_elems(CS_STATE_INT8, kVarP16) % 1024 == 0,
              "tiles hold whole int8 blocks in 16-byte scale groups");
static_assert(stages_for(CS_STATE_INT8, kVarP16) >= 4 && stages_for(CS_STATE_INT8) >= 5,
              "stage rings of the 8-bit kinds");
static_assert(block_threads(CS_STATE_F32) <= 1024 && block_threads(CS_STATE_INT8) <= 1024,
              "threads per CTA");
static_assert(kElementwiseTile % (4 * 32 * CS_WARPS_ELEMENTWISE) == 0 &&
                  kElementwiseTile % (4 * 32 * CS_WARPS_BF16) == 0,
              "elementwise tiles hold whole 4-element groups for every compute thread");
static_assert(kDefaultUnitElems % kInt8Block == 0, "units hold whole int8 blocks");

// Error bits the kernel sets in the plan's error word (never traps).
enum : uint32_t {
  kErrConsumerWait = 1u,   // a compute warp gave up waiting for a tile
  kErrProducerWait = 2u,   // the producer gave up waiting for a tile's compute
  kErrDrainWait = 4u,      // the producer gave up waiting for its own loads
  kErrFetchWait = 8u,      // the unit fetcher gave up waiting for the publisher
};
// Debug flags (test hook; 0 in normal use).
enum : uint32_t {
  kDebugSkipFirstTile = 1u,   // the first tile of the queue's first unit is never signalled
};

// One tensor, as the kernel sees it. 64 bytes, one per tensor.
struct alignas(16) TensorDesc {
  void* param;
  const void* grad;
  void* m;
  void* v;
  float* m_scale;
  float* v_scale;
  float* master;         // fp32 master weights of a 16-bit param, or null
  int16_t group;
  uint8_t param_dtype;   // CS_DTYPE_* of param and grad
  uint8_t flags;         // kVec | kBulk | kBulkScale | kMaster
  int32_t n_units;       // work units of this tensor (commit counter target)
};
static_assert(sizeof(TensorDesc) == 64, "descriptor must stay 64 bytes");
enum : uint8_t {
  kVec = 1,    // every buffer aligned to four elements: vector loads
  kBulk = 2,   // every buffer 16-byte aligned: bulk (TMA) copies
  kBulkScale = 4,  // int8 scale arrays 16-byte aligned
  kMaster = 8,     // theta lives in `master` (fp32); param is its 16-bit copy
  kStateF32 = 16,  // 8-bit plan: this tensor keeps fp32 moments (direct path)
};
// How a tile reads and writes theta: the param dtype, or an fp32 master with
// a 16-bit copy (kThetaMasterBF16 / kThetaMasterF16 = dtype + 2).
enum : int32_t { kThetaMasterBF16 = 3, kThetaMasterF16 = 4 };

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
  uint32_t* err;             // error bits (kErr*)
  uint64_t wait_ns;          // bound on every wait
  uint32_t debug;            // kDebug* flags
  int32_t n_units;
  int32_t all_present;       // 1: ignore `present`
  int32_t pad_;
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

// Host-side validation shared by the entry points (defined in plan.cu).
namespace host {
int elem_bytes(int32_t dtype);
int state_elem_bytes(int32_t kind);
int check_tensor(const adamw_tensor_t& t, int32_t state_kind, uint8_t* flags);
uint8_t access_flags(const adamw_tensor_t& t, int32_t state_kind);
// The device descriptor of a checked tensor (n_units left 0).
TensorDesc make_desc(const adamw_tensor_t& t, int32_t state_kind, uint8_t flags);
int check_group(const adamw_group_t& g);
}  // namespace host

// The kernel variant a tensor list needs (Variant above): `extended` when
// some tensor has fp32 master weights or (8-bit kinds) fp32 moments;
// `all16` when every tensor with elements has 16-bit params; `small` when
// some work unit has at most kPackMax elements.
constexpr int pick_variant(int state_kind, bool extended, bool all16, bool small) {
  return extended                          ? kVarExtended
         : (is_8bit(state_kind) && all16) ? (small ? kVarP16Pack : kVarP16)
         : (small && state_kind != CS_STATE_DYN8) ? kVarPlainPack
                                                   : kVarPlain;
}
// Whether the kernel of (state_kind, variant) is built.
constexpr bool variant_built(int state_kind, int variant) {
  return is_p16(variant) ? is_8bit(state_kind)
                         : variant != kVarPlainPack || state_kind != CS_STATE_DYN8;
}

// Launch one step with the kernel of (state_kind, cls, variant). Defined in
// step_launch.cu.
cudaError_t launch_step(int state_kind, ArgClass cls, int variant, const void* args, int grid,
                        cudaStream_t stream);
// Max resident CTAs per SM of that kernel; also sets its dynamic shared
// memory limit.
cudaError_t step_kernel_occupancy(int state_kind, ArgClass cls, int variant,
                                  int* blocks_per_sm);

}  // namespace cs
