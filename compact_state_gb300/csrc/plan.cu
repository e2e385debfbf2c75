// Host side of the C ABI: validation, the work-unit table, the device-resident
// descriptor tables, and the per-step launch.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include "adamw_internal.h"
#include "prologue.h"

using cs::TensorDesc;
using cs::WorkUnit;

struct adamw_plan {
  int device = 0;
  int32_t n_tensors = 0;
  int32_t state_kind = 0;
  int32_t unit_elems = 0;
  int32_t max_group = 0;
  int32_t sm_count = 0;
  bool any_master = false;         // some tensor has fp32 masters or fp32 moments in an 8-bit plan
  bool all16 = true;               // every tensor with elements has 16-bit params
  int variant = 0;                 // kernel variant (cs::Variant)
  int64_t n_units = 0;
  int64_t total_numel = 0;
  int64_t device_bytes = 0;
  int grid[3] = {0, 0, 0};        // persistent grid per argument class
  int pgrid[3] = {0, 0, 0};       // gradient prologue: one wave of resident blocks
  void* dev = nullptr;            // one allocation: descs | units | commit | sched | prologue
  TensorDesc* d_descs = nullptr;
  WorkUnit* d_units = nullptr;
  uint32_t* d_commit = nullptr;
  uint32_t* d_sched = nullptr;     // [0] next unit, [1] CTAs done, [2] error bits
  double* d_partial = nullptr;     // gradient prologue: per-block sums of squares
  uint32_t* d_pwords = nullptr;    // gradient prologue: [0] blocks done, [1] non-finite
  uint64_t wait_ns = cs::kDefaultWaitNs;
  uint32_t debug = 0;
  std::vector<TensorDesc> h_descs;
  std::vector<int64_t> h_numel;
  TensorDesc* h_staging = nullptr;   // pinned, for adamw_plan_set_grads
  cudaEvent_t staging_done = nullptr;
  bool staging_pending = false;
};

namespace cs {
namespace host {

int elem_bytes(int32_t dtype) {
  switch (dtype) {
    case CS_DTYPE_F32: return 4;
    case CS_DTYPE_BF16: return 2;
    case CS_DTYPE_F16: return 2;
    default: return 0;
  }
}

int state_elem_bytes(int32_t kind) {
  switch (kind) {
    case CS_STATE_F32: return 4;
    case CS_STATE_BF16: return 2;
    case CS_STATE_INT8: return 1;
    case CS_STATE_INT8_UV: return 1;
    case CS_STATE_DYN8: return 1;
    default: return 0;
  }
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Vector access needs every buffer aligned to four of its elements, bulk
// copies 16-byte alignment of everything they load (theta comes from the
// master when there is one; param is then only stored, four at a time).
uint8_t access_flags(const adamw_tensor_t& t, int32_t state_kind) {
  const int pb = elem_bytes(t.param_dtype);
  const bool f32_state = (t.flags & CS_TENSOR_STATE_F32) != 0;
  const bool coded = cs::is_8bit(state_kind) && !f32_state;
  const int sb = f32_state ? 4 : state_elem_bytes(state_kind);
  const bool vec_core = aligned(t.param, 4 * pb) && aligned(t.grad, 4 * pb) &&
                        aligned(t.m, 4 * sb) && aligned(t.v, 4 * sb);
  const bool bulk_core = aligned(t.grad, 16) && aligned(t.m, 16) && aligned(t.v, 16);
  uint8_t f = 0;
  if (t.master) {
    f |= cs::kMaster;
    if (vec_core && aligned(t.master, 16)) f |= cs::kVec;
    if (bulk_core && aligned(t.master, 16) && aligned(t.param, 4 * pb)) f |= cs::kBulk;
  } else {
    if (vec_core) f |= cs::kVec;
    if (bulk_core && aligned(t.param, 16)) f |= cs::kBulk;
  }
  if (coded && aligned(t.m_scale, 16) && aligned(t.v_scale, 16)) f |= cs::kBulkScale;
  if (f32_state) f |= cs::kStateF32;
  return f;
}

// Validates one tensor; sets *flags to its access flags.
int check_tensor(const adamw_tensor_t& t, int32_t state_kind, uint8_t* flags) {
  if (t.numel < 0 || t.group < 0) return CS_ERR_INVALID_ARGUMENT;
  const int pb = elem_bytes(t.param_dtype);
  if (pb == 0) return CS_ERR_UNSUPPORTED;
  if (t.group >= CS_MAX_GROUPS) return CS_ERR_LIMIT;
  if (t.master && t.param_dtype == CS_DTYPE_F32) return CS_ERR_INVALID_ARGUMENT;
  if (t.flags & ~CS_TENSOR_STATE_F32) return CS_ERR_INVALID_ARGUMENT;
  const bool f32_state = (t.flags & CS_TENSOR_STATE_F32) != 0;
  if (f32_state && !cs::is_8bit(state_kind)) return CS_ERR_INVALID_ARGUMENT;
  *flags = static_cast<uint8_t>((t.master ? cs::kMaster : 0) | (f32_state ? cs::kStateF32 : 0));
  if (t.numel == 0) return CS_OK;
  if (t.numel > (int64_t(1) << 40)) return CS_ERR_LIMIT;
  const int sb = f32_state ? 4 : state_elem_bytes(state_kind);
  if (!t.param || !t.grad || !t.m || !t.v) return CS_ERR_INVALID_ARGUMENT;
  if (!aligned(t.param, pb) || !aligned(t.grad, pb) || !aligned(t.m, sb) || !aligned(t.v, sb))
    return CS_ERR_MISALIGNED;
  if (t.master && !aligned(t.master, 4)) return CS_ERR_MISALIGNED;
  if (cs::is_8bit(state_kind) && !f32_state) {
    if (!t.m_scale || !t.v_scale) return CS_ERR_INVALID_ARGUMENT;
    if (!aligned(t.m_scale, 4) || !aligned(t.v_scale, 4)) return CS_ERR_MISALIGNED;
  }
  *flags = access_flags(t, state_kind);
  return CS_OK;
}

TensorDesc make_desc(const adamw_tensor_t& t, int32_t state_kind, uint8_t flags) {
  TensorDesc d;
  std::memset(&d, 0, sizeof(d));
  d.param = t.param;
  d.grad = t.grad;
  d.m = t.m;
  d.v = t.v;
  const bool coded = cs::is_8bit(state_kind) && !(t.flags & CS_TENSOR_STATE_F32);
  d.m_scale = coded ? t.m_scale : nullptr;
  d.v_scale = coded ? t.v_scale : nullptr;
  d.master = t.master;
  d.group = static_cast<int16_t>(t.group);
  d.param_dtype = static_cast<uint8_t>(t.param_dtype);
  d.flags = flags;
  return d;
}

int check_unit_elems(int32_t unit_elems, int32_t* out) {
  if (unit_elems == 0) unit_elems = cs::kDefaultUnitElems;
  if (unit_elems < 0 || unit_elems % cs::kInt8Block != 0 || unit_elems > (1 << 30))
    return CS_ERR_INVALID_ARGUMENT;
  *out = unit_elems;
  return CS_OK;
}

// Units of every tensor: starts at multiples of unit_elems; the longest first
// (ties keep tensor order), so a dynamic queue ends on its smallest units. A
// tensor with no elements gets one empty unit, which only commits its step.
void build_units(const int64_t* numels, int32_t n, int32_t unit_elems,
                 std::vector<WorkUnit>* units, std::vector<int32_t>* per_tensor) {
  units->clear();
  per_tensor->assign(n, 0);
  for (int32_t i = 0; i < n; ++i) {
    const int64_t ne = numels[i];
    int32_t k = 0;
    for (int64_t s = 0; s < ne; s += unit_elems, ++k) {
      WorkUnit w;
      w.start = s;
      w.tensor = i;
      w.len = static_cast<int32_t>(std::min<int64_t>(unit_elems, ne - s));
      units->push_back(w);
    }
    if (ne == 0) {            // an empty tensor still counts its steps
      units->push_back(WorkUnit{0, i, 0});
      k = 1;
    }
    (*per_tensor)[i] = k;
  }
  std::stable_sort(units->begin(), units->end(),
                   [](const WorkUnit& a, const WorkUnit& b) { return a.len > b.len; });
}

// Finer units at the end of the queue. CTAs take units dynamically, so they
// finish up to one unit apart; with 49152-element units that is ~15 us of one
// CTA's bandwidth, a large part of a short step. The units holding the last
// `waves` x `ctas` full units' worth of elements are re-cut into pieces of
// `piece` elements (a multiple of the tile, so of the 256-element block) and
// kept longest first. Recounts the units of each tensor.
void split_tail(std::vector<WorkUnit>* units, std::vector<int32_t>* per_tensor, int64_t ctas,
                int32_t unit_elems, int32_t piece, int waves) {
  const int64_t tail_elems = static_cast<int64_t>(waves) * ctas * unit_elems;
  size_t first = units->size();
  int64_t acc = 0;
  while (first > 0 && acc < tail_elems) acc += (*units)[--first].len;
  std::vector<WorkUnit> tail;
  for (size_t k = first; k < units->size(); ++k) {
    const WorkUnit& w = (*units)[k];
    if (w.len <= piece) {
      tail.push_back(w);
      continue;
    }
    for (int32_t off = 0; off < w.len; off += piece)
      tail.push_back(WorkUnit{w.start + off, w.tensor, std::min(piece, w.len - off)});
  }
  std::stable_sort(tail.begin(), tail.end(),
                   [](const WorkUnit& a, const WorkUnit& b) { return a.len > b.len; });
  units->resize(first);
  units->insert(units->end(), tail.begin(), tail.end());
  std::fill(per_tensor->begin(), per_tensor->end(), 0);
  for (const WorkUnit& w : *units) ++(*per_tensor)[w.tensor];
}

// The queue a plan uses: the unit cut, then the last two waves re-cut into
// pieces of four tiles; for the 8-bit kinds the last `ctas` of those are cut
// again into two-tile pieces, which CTAs take one per trip (measured on the
// LoRA set: 69.5 -> 68.5 us with int8 moments; with bf16 moments the same cut
// cost 0.7 us, and single-tile pieces were slower for every kind: a one-tile
// trip is shorter than the fetch that has to hide behind it).
void build_queue(const int64_t* numels, int32_t n, int32_t state_kind, int32_t unit_elems,
                 int64_t ctas, std::vector<WorkUnit>* units, std::vector<int32_t>* per_tensor) {
  build_units(numels, n, unit_elems, units, per_tensor);
  const int32_t tile = cs::tile_elems(state_kind);
  const int32_t piece = std::min(unit_elems, 4 * tile);
  split_tail(units, per_tensor, ctas, unit_elems, piece, 2);
  if (cs::is_8bit(state_kind) && piece > 2 * tile)
    split_tail(units, per_tensor, ctas, piece, 2 * tile, 1);
}

}  // namespace host
}  // namespace cs

using namespace cs::host;

namespace {

bool finite_f(float x) { return std::isfinite(x); }

}  // namespace

namespace cs {
namespace host {

int check_group(const adamw_group_t& g) {
  if (!finite_f(g.lr) || !finite_f(g.eps) || !finite_f(g.weight_decay)) return CS_ERR_HYPERPARAM;
  if (!(g.beta1 >= 0.0f && g.beta1 < 1.0f)) return CS_ERR_HYPERPARAM;
  if (!(g.beta2 >= 0.0f && g.beta2 < 1.0f)) return CS_ERR_HYPERPARAM;
  // eps keeps the denominator sqrt(v_hat) + eps away from zero: a moment that
  // is zero, or flushed to zero from a subnormal, would otherwise divide 0/0
  if (!(g.eps > 0.0f)) return CS_ERR_HYPERPARAM;
  return CS_OK;
}

}  // namespace host
}  // namespace cs

namespace {

template <int G, int W>
int launch_class(adamw_plan* p, cs::ArgClass cls, const adamw_group_t* groups,
                 int32_t n_groups, const uint32_t* present, int32_t* step,
                 const float* inv_scale, const float* found_inf, cudaStream_t stream) {
  cs::StepArgs<G, W> a;
  std::memset(&a, 0, sizeof(a));
  a.descs = p->d_descs;
  a.units = p->d_units;
  a.step = step;
  a.inv_scale = inv_scale;
  a.found_inf = found_inf;
  a.sched = p->d_sched;
  a.commit = p->d_commit;
  a.err = p->d_sched + 2;
  a.wait_ns = p->wait_ns;
  a.debug = p->debug;
  a.n_units = static_cast<int32_t>(p->n_units);
  std::memcpy(a.groups, groups, sizeof(adamw_group_t) * n_groups);
  if (present) {
    a.all_present = 0;
    std::memcpy(a.present, present, sizeof(uint32_t) * ((p->n_tensors + 31) / 32));
  } else {
    a.all_present = 1;
  }
  const cudaError_t e =
      cs::launch_step(p->state_kind, cls, p->variant, &a, p->grid[cls], stream);
  return e == cudaSuccess ? CS_OK : CS_ERR_CUDA;
}

}  // namespace

namespace {

template <int W>
int launch_prologue_class(adamw_plan* p, cs::ArgClass cls, const uint32_t* present,
                          const float* inv_scale, float max_norm, float* found_inf_out,
                          float* norm_out, float* scale_out, cudaStream_t stream) {
  cs::PrologueArgs<W> a;
  std::memset(&a, 0, sizeof(a));
  a.descs = p->d_descs;
  a.units = p->d_units;
  a.inv_scale = inv_scale;
  a.found_inf_out = found_inf_out;
  a.norm_out = norm_out;
  a.scale_out = scale_out;
  a.partial = p->d_partial;
  a.words = p->d_pwords;
  a.max_norm = max_norm;
  a.n_units = static_cast<int32_t>(p->n_units);
  a.pieces_per_unit = (p->unit_elems + cs::kProloguePiece - 1) / cs::kProloguePiece;
  if (present) {
    a.all_present = 0;
    std::memcpy(a.present, present, sizeof(uint32_t) * ((p->n_tensors + 31) / 32));
  } else {
    a.all_present = 1;
  }
  const int64_t items = static_cast<int64_t>(a.n_units) * a.pieces_per_unit;
  const int grid = static_cast<int>(std::max<int64_t>(
      1, std::min<int64_t>(items, p->pgrid[cls])));
  return cs::launch_prologue(cls, &a, grid, stream) == cudaSuccess ? CS_OK : CS_ERR_CUDA;
}

// Host-only unit tables for adamw_build_units (state_kind < 0: the plain cut)
// and adamw_build_queue (the plan's queue for `ctas` CTAs).
int write_units(const int64_t* numels, int32_t n_tensors, int32_t state_kind,
                int32_t unit_elems, int32_t ctas, int32_t* tensor_out, int64_t* start_out,
                int32_t* len_out, int64_t cap, int64_t* n_units_out) {
  if (!n_units_out || n_tensors < 0 || (n_tensors > 0 && !numels) || cap < 0)
    return CS_ERR_INVALID_ARGUMENT;
  int32_t ue = 0;
  int rc = check_unit_elems(unit_elems, &ue);
  if (rc) return rc;
  for (int32_t i = 0; i < n_tensors; ++i)
    if (numels[i] < 0) return CS_ERR_INVALID_ARGUMENT;
  try {
    std::vector<WorkUnit> units;
    std::vector<int32_t> per;
    if (state_kind < 0) {
      build_units(numels, n_tensors, ue, &units, &per);
    } else {
      build_queue(numels, n_tensors, state_kind, ue, ctas, &units, &per);
    }
    *n_units_out = static_cast<int64_t>(units.size());
    if (static_cast<int64_t>(units.size()) > cap) return cap == 0 ? CS_OK : CS_ERR_LIMIT;
    if (!tensor_out || !start_out || !len_out) return CS_ERR_INVALID_ARGUMENT;
    for (size_t k = 0; k < units.size(); ++k) {
      tensor_out[k] = units[k].tensor;
      start_out[k] = units[k].start;
      len_out[k] = units[k].len;
    }
  } catch (const std::bad_alloc&) {
    return CS_ERR_OUT_OF_MEMORY;
  }
  return CS_OK;
}

}  // namespace

extern "C" {

const char* adamw_strerror(int status) {
  switch (status) {
    case CS_OK: return "success";
    case CS_ERR_INVALID_ARGUMENT: return "invalid argument";
    case CS_ERR_UNSUPPORTED: return "unsupported dtype or state kind";
    case CS_ERR_MISALIGNED: return "pointer not aligned to its element size";
    case CS_ERR_LIMIT: return "size limit exceeded (tensors, groups, elements or capacity)";
    case CS_ERR_CUDA: return "CUDA runtime error";
    case CS_ERR_OUT_OF_MEMORY: return "out of memory";
    case CS_ERR_HYPERPARAM: return "invalid hyper-parameter (beta outside [0,1), eps not positive or non-finite value)";
    case CS_ERR_WRONG_DEVICE: return "current CUDA device is not the plan's device";
    default: return "unknown status";
  }
}

int adamw_state_bytes(const int64_t* numels, const int32_t* flags, int32_t n_tensors,
                      int32_t state_kind, int64_t* out_bytes) {
  if (!out_bytes || n_tensors < 0 || (n_tensors > 0 && !numels)) return CS_ERR_INVALID_ARGUMENT;
  const int sb = state_elem_bytes(state_kind);
  if (sb == 0) return CS_ERR_UNSUPPORTED;
  int64_t total = 0;
  for (int32_t i = 0; i < n_tensors; ++i) {
    const int64_t n = numels[i];
    const int32_t f = flags ? flags[i] : 0;
    if (n < 0 || (f & ~CS_TENSOR_STATE_F32)) return CS_ERR_INVALID_ARGUMENT;
    const bool f32 = (f & CS_TENSOR_STATE_F32) != 0;
    if (f32 && !cs::is_8bit(state_kind)) return CS_ERR_INVALID_ARGUMENT;
    // two moments (fp32 for a tensor kept in fp32) + a 4-byte step counter
    total += 2 * (f32 ? 4 : sb) * n + 4;
    if (cs::is_8bit(state_kind) && !f32)
      total += 2 * 4 * ((n + cs::kInt8Block - 1) / cs::kInt8Block);
  }
  *out_bytes = total;
  return CS_OK;
}

int adamw_build_units(const int64_t* numels, int32_t n_tensors, int32_t unit_elems,
                      int32_t* tensor_out, int64_t* start_out, int32_t* len_out,
                      int64_t cap, int64_t* n_units_out) {
  return write_units(numels, n_tensors, -1, unit_elems, 0, tensor_out, start_out, len_out, cap,
                     n_units_out);
}

int adamw_build_queue(const int64_t* numels, int32_t n_tensors, int32_t state_kind,
                      int32_t unit_elems, int32_t ctas, int32_t* tensor_out, int64_t* start_out,
                      int32_t* len_out, int64_t cap, int64_t* n_units_out) {
  if (state_elem_bytes(state_kind) == 0) return CS_ERR_UNSUPPORTED;
  if (ctas < 1) return CS_ERR_INVALID_ARGUMENT;
  return write_units(numels, n_tensors, state_kind, unit_elems, ctas, tensor_out, start_out,
                     len_out, cap, n_units_out);
}

int adamw_shard_ranges(const int64_t* numels, int32_t n_tensors, int32_t world, int32_t rank,
                       int64_t* lo_out, int64_t* hi_out, int64_t* offset_out,
                       int64_t* shard_elems_out) {
  if (n_tensors < 0 || (n_tensors > 0 && (!numels || !lo_out || !hi_out)))
    return CS_ERR_INVALID_ARGUMENT;
  if (world < 1 || rank < 0 || rank >= world) return CS_ERR_INVALID_ARGUMENT;
  const int64_t B = cs::kInt8Block;
  // flat layout: every tensor padded to whole 256-element blocks, end to end
  int64_t flat = 0;
  for (int32_t i = 0; i < n_tensors; ++i) {
    if (numels[i] < 0) return CS_ERR_INVALID_ARGUMENT;
    if (numels[i] > (int64_t(1) << 40)) return CS_ERR_LIMIT;
    flat += (numels[i] + B - 1) / B * B;
  }
  // equal shards of whole blocks: world * shard covers the flat buffer
  const int64_t blocks = flat / B;
  const int64_t shard = (blocks + world - 1) / world * B;
  const int64_t r0 = static_cast<int64_t>(rank) * shard, r1 = r0 + shard;
  int64_t off = 0;
  for (int32_t i = 0; i < n_tensors; ++i) {
    const int64_t n = numels[i];
    int64_t lo = std::min(std::max<int64_t>(r0 - off, 0), n);
    int64_t hi = std::min(std::max<int64_t>(r1 - off, 0), n);
    if (hi <= lo) lo = hi = 0;
    lo_out[i] = lo;
    hi_out[i] = hi;
    if (offset_out) offset_out[i] = off;
    off += (n + B - 1) / B * B;
  }
  if (shard_elems_out) *shard_elems_out = shard;
  return CS_OK;
}

int adamw_plan_create(const adamw_tensor_t* tensors, int32_t n_tensors, int32_t state_kind,
                      int32_t unit_elems, adamw_plan_t** out_plan) {
  if (!out_plan) return CS_ERR_INVALID_ARGUMENT;
  *out_plan = nullptr;
  if (!tensors || n_tensors <= 0) return CS_ERR_INVALID_ARGUMENT;
  if (n_tensors > CS_MAX_TENSORS) return CS_ERR_LIMIT;
  if (state_elem_bytes(state_kind) == 0) return CS_ERR_UNSUPPORTED;
  int32_t ue = 0;
  int rc = check_unit_elems(unit_elems, &ue);
  if (rc) return rc;

  adamw_plan* p = nullptr;
  try {
    p = new adamw_plan();
    p->n_tensors = n_tensors;
    p->state_kind = state_kind;
    p->unit_elems = ue;
    p->h_descs.resize(n_tensors);
    std::vector<int64_t> numels(n_tensors);
    for (int32_t i = 0; i < n_tensors; ++i) {
      const adamw_tensor_t& t = tensors[i];
      uint8_t vec = 0;
      rc = check_tensor(t, state_kind, &vec);
      if (rc) { delete p; return rc; }
      p->h_descs[i] = make_desc(t, state_kind, vec);
      p->any_master = p->any_master || t.master != nullptr || (vec & cs::kStateF32) != 0;
      p->all16 = p->all16 && (t.numel == 0 || t.param_dtype != CS_DTYPE_F32);
      numels[i] = t.numel;
      p->total_numel += t.numel;
      p->max_group = std::max(p->max_group, t.group);
    }
    if (cudaGetDevice(&p->device) != cudaSuccess) { delete p; return CS_ERR_CUDA; }
    if (cudaDeviceGetAttribute(&p->sm_count, cudaDevAttrMultiProcessorCount, p->device) != cudaSuccess) {
      delete p; return CS_ERR_CUDA;
    }
    std::vector<WorkUnit> units;
    std::vector<int32_t> per;
    build_queue(numels.data(), n_tensors, state_kind, ue, p->sm_count, &units, &per);
    bool small = false;
    for (const WorkUnit& w : units) small = small || (w.len > 0 && w.len <= cs::kPackMax);
    p->variant = cs::pick_variant(state_kind, p->any_master, p->all16, small);
    p->h_numel = numels;
    if (units.size() >= (size_t(1) << 31) - (size_t(1) << 20)) { delete p; return CS_ERR_LIMIT; }
    for (int32_t i = 0; i < n_tensors; ++i) p->h_descs[i].n_units = per[i];
    p->n_units = static_cast<int64_t>(units.size());

    for (int c = 0; c < 3; ++c) {
      int per_sm = 0;
      if (cs::step_kernel_occupancy(state_kind, static_cast<cs::ArgClass>(c), p->variant,
                                    &per_sm) != cudaSuccess ||
          per_sm <= 0) {
        delete p; return CS_ERR_CUDA;
      }
      const int64_t want = static_cast<int64_t>(per_sm) * p->sm_count;
      // never more CTAs than units (at least one)
      p->grid[c] = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(want, p->n_units)));
      if (cs::prologue_occupancy(static_cast<cs::ArgClass>(c), &per_sm) != cudaSuccess || per_sm <= 0) {
        delete p; return CS_ERR_CUDA;
      }
      p->pgrid[c] = static_cast<int>(
          std::min<int64_t>(static_cast<int64_t>(per_sm) * p->sm_count, cs::kPrologueMaxBlocks));
    }

    const size_t b_desc = sizeof(TensorDesc) * n_tensors;
    const size_t b_units = sizeof(WorkUnit) * std::max<size_t>(units.size(), 1);
    const size_t b_commit = ((sizeof(uint32_t) * n_tensors + 255) / 256) * 256;
    const size_t b_sched = 256;
    const size_t b_pro = sizeof(double) * cs::kPrologueMaxBlocks + 256;
    const size_t total = b_desc + b_units + b_commit + b_sched + b_pro;
    if (cudaMalloc(&p->dev, total) != cudaSuccess) {
      cudaGetLastError();
      delete p;
      return CS_ERR_OUT_OF_MEMORY;
    }
    p->device_bytes = static_cast<int64_t>(total);
    char* base = static_cast<char*>(p->dev);
    p->d_descs = reinterpret_cast<TensorDesc*>(base);
    p->d_units = reinterpret_cast<WorkUnit*>(base + b_desc);
    p->d_commit = reinterpret_cast<uint32_t*>(base + b_desc + b_units);
    p->d_sched = reinterpret_cast<uint32_t*>(base + b_desc + b_units + b_commit);
    p->d_partial = reinterpret_cast<double*>(base + b_desc + b_units + b_commit + b_sched);
    p->d_pwords = reinterpret_cast<uint32_t*>(base + b_desc + b_units + b_commit + b_sched +
                                              sizeof(double) * cs::kPrologueMaxBlocks);
    bool ok = cudaMemcpy(p->d_descs, p->h_descs.data(), b_desc, cudaMemcpyHostToDevice) == cudaSuccess;
    if (ok && !units.empty())
      ok = cudaMemcpy(p->d_units, units.data(), sizeof(WorkUnit) * units.size(),
                      cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && cudaMemset(p->d_commit, 0, b_commit + b_sched + b_pro) == cudaSuccess;
    ok = ok && cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) {
      cudaFree(p->dev);
      delete p;
      return CS_ERR_CUDA;
    }
  } catch (const std::bad_alloc&) {
    if (p) {
      if (p->dev) cudaFree(p->dev);
      delete p;
    }
    return CS_ERR_OUT_OF_MEMORY;
  }
  *out_plan = p;
  return CS_OK;
}

int adamw_step(adamw_plan_t* p, const adamw_group_t* groups, int32_t n_groups,
               const uint32_t* grad_present, int32_t* step, const float* inv_scale,
               const float* found_inf, struct CUstream_st* stream) {
  if (!p || !groups || !step) return CS_ERR_INVALID_ARGUMENT;
  if (n_groups <= 0) return CS_ERR_INVALID_ARGUMENT;
  if (n_groups > CS_MAX_GROUPS) return CS_ERR_LIMIT;
  if (p->max_group >= n_groups) return CS_ERR_INVALID_ARGUMENT;
  for (int32_t g = 0; g < n_groups; ++g) {
    const int rc = check_group(groups[g]);
    if (rc) return rc;
  }
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CS_ERR_CUDA;
  if (dev != p->device) return CS_ERR_WRONG_DEVICE;

  cs::ArgClass cls;
  const int32_t need_tensors = grad_present ? p->n_tensors : 0;
  if (n_groups <= cs::kSmallGroups && need_tensors <= cs::kSmallWords * 32) cls = cs::kClassSmall;
  else if (need_tensors <= cs::kMidWords * 32) cls = cs::kClassMid;
  else cls = cs::kClassLarge;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (cls) {
    case cs::kClassSmall:
      return launch_class<cs::kSmallGroups, cs::kSmallWords>(p, cls, groups, n_groups, grad_present,
                                                             step, inv_scale, found_inf, s);
    case cs::kClassMid:
      return launch_class<cs::kMidGroups, cs::kMidWords>(p, cls, groups, n_groups, grad_present,
                                                         step, inv_scale, found_inf, s);
    default:
      return launch_class<cs::kLargeGroups, cs::kLargeWords>(p, cls, groups, n_groups, grad_present,
                                                             step, inv_scale, found_inf, s);
  }
}

int adamw_grad_prologue(adamw_plan_t* p, const uint32_t* grad_present, const float* inv_scale,
                        float max_norm, float* found_inf_out, float* grad_norm_out,
                        float* scale_out, struct CUstream_st* stream) {
  if (!p || !found_inf_out || !scale_out) return CS_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(max_norm)) return CS_ERR_HYPERPARAM;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CS_ERR_CUDA;
  if (dev != p->device) return CS_ERR_WRONG_DEVICE;
  const int32_t need = grad_present ? p->n_tensors : 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (need <= cs::kSmallWords * 32)
    return launch_prologue_class<cs::kSmallWords>(p, cs::kClassSmall, grad_present, inv_scale,
                                                  max_norm, found_inf_out, grad_norm_out,
                                                  scale_out, s);
  if (need <= cs::kMidWords * 32)
    return launch_prologue_class<cs::kMidWords>(p, cs::kClassMid, grad_present, inv_scale,
                                                max_norm, found_inf_out, grad_norm_out,
                                                scale_out, s);
  return launch_prologue_class<cs::kLargeWords>(p, cs::kClassLarge, grad_present, inv_scale,
                                                max_norm, found_inf_out, grad_norm_out, scale_out,
                                                s);
}

int adamw_plan_set_grads(adamw_plan_t* p, const void* const* grads, struct CUstream_st* stream) {
  if (!p || !grads) return CS_ERR_INVALID_ARGUMENT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CS_ERR_CUDA;
  if (dev != p->device) return CS_ERR_WRONG_DEVICE;
  // validate first: nothing changes on error
  for (int32_t i = 0; i < p->n_tensors; ++i) {
    const TensorDesc& d = p->h_descs[i];
    if (p->h_numel[i] == 0) continue;
    const int pb = elem_bytes(d.param_dtype);
    if (!grads[i]) return CS_ERR_INVALID_ARGUMENT;
    if (!aligned(grads[i], pb)) return CS_ERR_MISALIGNED;
  }
  const size_t bytes = sizeof(TensorDesc) * p->n_tensors;
  if (!p->h_staging) {
    if (cudaMallocHost(reinterpret_cast<void**>(&p->h_staging), bytes) != cudaSuccess) {
      cudaGetLastError();
      p->h_staging = nullptr;
      return CS_ERR_OUT_OF_MEMORY;
    }
    if (cudaEventCreateWithFlags(&p->staging_done, cudaEventDisableTiming) != cudaSuccess)
      return CS_ERR_CUDA;
  }
  if (p->staging_pending && cudaEventSynchronize(p->staging_done) != cudaSuccess) return CS_ERR_CUDA;
  for (int32_t i = 0; i < p->n_tensors; ++i) {
    TensorDesc& d = p->h_descs[i];
    if (p->h_numel[i] == 0) continue;
    d.grad = grads[i];
    adamw_tensor_t t{};
    t.param = d.param;
    t.grad = d.grad;
    t.m = d.m;
    t.v = d.v;
    t.m_scale = d.m_scale;
    t.v_scale = d.v_scale;
    t.master = d.master;
    t.param_dtype = d.param_dtype;
    t.flags = (d.flags & cs::kStateF32) ? CS_TENSOR_STATE_F32 : 0;
    d.flags = access_flags(t, p->state_kind);
  }
  std::memcpy(p->h_staging, p->h_descs.data(), bytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(p->d_descs, p->h_staging, bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return CS_ERR_CUDA;
  if (cudaEventRecord(p->staging_done, s) != cudaSuccess) return CS_ERR_CUDA;
  p->staging_pending = true;
  return CS_OK;
}

int adamw_plan_error(adamw_plan_t* p, uint32_t* out_flags) {
  if (!p || !out_flags) return CS_ERR_INVALID_ARGUMENT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CS_ERR_CUDA;
  if (dev != p->device) return CS_ERR_WRONG_DEVICE;
  uint32_t v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return CS_ERR_CUDA;
  if (cudaMemcpy(&v, p->d_sched + 2, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CS_ERR_CUDA;
  if (v != 0) {
    // a step that gave up may leave queue words and commit tickets behind:
    // clear them together with the error word
    const size_t bytes = reinterpret_cast<char*>(p->d_sched) + 256 -
                         reinterpret_cast<char*>(p->d_commit);
    if (cudaMemset(p->d_commit, 0, bytes) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
      return CS_ERR_CUDA;
  }
  *out_flags = v;
  return CS_OK;
}

int adamw_plan_set_debug(adamw_plan_t* p, uint64_t wait_ns, uint32_t flags) {
  if (!p) return CS_ERR_INVALID_ARGUMENT;
  if (wait_ns == 0) wait_ns = cs::kDefaultWaitNs;
  if (wait_ns > 60ull * 1000000000ull || (flags & ~uint32_t(cs::kDebugSkipFirstTile)))
    return CS_ERR_INVALID_ARGUMENT;
  p->wait_ns = wait_ns;
  p->debug = flags;
  return CS_OK;
}

int adamw_plan_info(const adamw_plan_t* p, adamw_plan_info_t* out) {
  if (!p || !out) return CS_ERR_INVALID_ARGUMENT;
  out->n_units = p->n_units;
  out->total_numel = p->total_numel;
  out->device_bytes = p->device_bytes;
  out->n_tensors = p->n_tensors;
  out->state_kind = p->state_kind;
  out->unit_elems = p->unit_elems;
  out->grid_blocks = p->grid[cs::kClassSmall];
  out->block_threads = cs::block_threads(p->state_kind);
  out->device = p->device;
  return CS_OK;
}

int adamw_plan_destroy(adamw_plan_t* p) {
  if (!p) return CS_OK;
  int rc = CS_OK;
  int prev = -1;
  cudaGetDevice(&prev);
  if (prev != p->device) cudaSetDevice(p->device);
  if (cudaDeviceSynchronize() != cudaSuccess) rc = CS_ERR_CUDA;
  if (p->dev && cudaFree(p->dev) != cudaSuccess) rc = CS_ERR_CUDA;
  if (p->staging_done) cudaEventDestroy(p->staging_done);
  if (p->h_staging) cudaFreeHost(p->h_staging);
  if (prev >= 0 && prev != p->device) cudaSetDevice(prev);
  delete p;
  return rc;
}

}  // extern "C"
