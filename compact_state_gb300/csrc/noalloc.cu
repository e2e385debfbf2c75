// Step entry point that allocates nothing: adamw_step_noalloc().
//
// Some callers of this library cannot call cudaMalloc. An allocator or
// memory-pool implementation that runs the optimizer step from inside its own
// callbacks must not re-enter the device allocator, and runtimes that hand
// all of the GPU's memory to their own pool at start-up leave nothing for a
// plan to allocate. For them this entry point keeps the step kernel's scratch
// (tensor descriptors, work units, commit tickets, scheduler and error words)
// in one file-scope __device__ array of fixed size, so a step needs no device
// allocation. The caller still owns and passes every input and output.
//
// The array is shared by every call on a device and keeps the last call's
// contents: each call rewrites the tables and clears the words that must start
// at zero before it launches, so calls that overlap on the GPU race with each
// other and must be ordered by the caller (one stream, or events). The error
// word is the exception: it collects the bits of every call until
// adamw_noalloc_error() reads and clears it.
//
// A call copies its tables from host staging arrays that the next call
// rewrites, so a captured call would replay with another call's tables; a
// call on a stream that is being captured is refused.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "adamw_internal.h"

namespace cs {
namespace {

constexpr int kNaMaxTensors = CS_NOALLOC_MAX_TENSORS;
constexpr int kNaMaxUnits = CS_NOALLOC_MAX_UNITS;
constexpr size_t kNaDescBytes = sizeof(TensorDesc) * kNaMaxTensors;
constexpr size_t kNaUnitBytes = sizeof(WorkUnit) * kNaMaxUnits;
constexpr size_t kNaCommitBytes = ((sizeof(uint32_t) * kNaMaxTensors + 255) / 256) * 256;
constexpr size_t kNaSchedBytes = 256;   // [0] next unit, [1] CTAs done, [2] error bits
constexpr size_t kNaScratchBytes = kNaDescBytes + kNaUnitBytes + kNaCommitBytes + kNaSchedBytes;
static_assert(kNaMaxTensors <= kSmallWords * 32, "fits the small argument class");

// The scratch. In host code this name only stands for the symbol; its device
// address comes from cudaGetSymbolAddress in setup_device().
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaScratchBytes];

constexpr int kNaMaxDevices = 64;
struct NaDevice {
  bool ready;
  unsigned char* scratch;   // device address of g_noalloc_scratch on this device
  int grid[5][kVariants][3];  // persistent grid per [state kind][variant][argument class]
};
NaDevice g_dev[kNaMaxDevices];
std::mutex g_mu;                              // guards set-up, staging and the hook
TensorDesc g_stage_descs[kNaMaxTensors];      // host staging of this call's tables
WorkUnit g_stage_units[kNaMaxUnits];
uint64_t g_wait_ns = kDefaultWaitNs;          // test hook (adamw_noalloc_set_debug)
uint32_t g_debug = 0;

// Once per device, with that device current: the array's device address and
// the persistent grid of every kernel variant.
int setup_device(int dev, NaDevice** out) {
  if (dev < 0 || dev >= kNaMaxDevices) return CS_ERR_LIMIT;
  NaDevice& d = g_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return CS_ERR_CUDA;
    }
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return CS_ERR_CUDA;
    for (int sk = 0; sk < 5; ++sk)
      for (int var = 0; var < kVariants; ++var)
        for (int c = 0; c < 3; ++c) {
          d.grid[sk][var][c] = 0;
          if (!variant_built(sk, var)) continue;
          int per_sm = 0;
          if (step_kernel_occupancy(sk, static_cast<ArgClass>(c), var, &per_sm) != cudaSuccess ||
              per_sm <= 0)
            return CS_ERR_CUDA;
          d.grid[sk][var][c] = per_sm * sms;
        }
    d.scratch = static_cast<unsigned char*>(p);
    d.ready = true;
  }
  *out = &d;
  return CS_OK;
}

template <int G, int W>
int launch_args(const TensorDesc* descs, const WorkUnit* units, uint32_t* commit,
                uint32_t* sched, int32_t n_units, int32_t n_tensors, int state_kind,
                ArgClass cls, int grid, const adamw_group_t* groups, int32_t n_groups,
                const uint32_t* present, int32_t* step, const float* inv_scale,
                const float* found_inf, int variant, cudaStream_t stream) {
  StepArgs<G, W> a;
  std::memset(&a, 0, sizeof(a));
  a.descs = descs;
  a.units = units;
  a.step = step;
  a.inv_scale = inv_scale;
  a.found_inf = found_inf;
  a.sched = sched;
  a.commit = commit;
  a.err = sched + 2;
  a.wait_ns = g_wait_ns;
  a.debug = g_debug;
  a.n_units = n_units;
  std::memcpy(a.groups, groups, sizeof(adamw_group_t) * n_groups);
  if (present) {
    a.all_present = 0;
    std::memcpy(a.present, present, sizeof(uint32_t) * ((n_tensors + 31) / 32));
  } else {
    a.all_present = 1;
  }
  return launch_step(state_kind, cls, variant, &a, std::min(grid, n_units), stream) == cudaSuccess
             ? CS_OK
             : CS_ERR_CUDA;
}

}  // namespace
}  // namespace cs

extern "C" int adamw_step_noalloc(const adamw_tensor_t* tensors, int32_t n_tensors,
                                  int32_t state_kind, const adamw_group_t* groups,
                                  int32_t n_groups, const uint32_t* grad_present, int32_t* step,
                                  const float* inv_scale, const float* found_inf,
                                  struct CUstream_st* stream) {
  using namespace cs;
  if (!tensors || !groups || !step || n_tensors <= 0 || n_groups <= 0)
    return CS_ERR_INVALID_ARGUMENT;
  if (n_tensors > kNaMaxTensors || n_groups > CS_MAX_GROUPS) return CS_ERR_LIMIT;
  if (host::state_elem_bytes(state_kind) == 0) return CS_ERR_UNSUPPORTED;
  for (int32_t g = 0; g < n_groups; ++g) {
    const int rc = host::check_group(groups[g]);
    if (rc) return rc;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
    cudaGetLastError();
    return CS_ERR_CUDA;
  }
  if (cap != cudaStreamCaptureStatusNone) return CS_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> lock(g_mu);
  // this call's descriptors and work units, in host staging (no allocation)
  int64_t nu = 0;
  bool any_master = false;
  bool all16 = true;
  for (int32_t i = 0; i < n_tensors; ++i) {
    const adamw_tensor_t& t = tensors[i];
    uint8_t flags = 0;
    const int rc = host::check_tensor(t, state_kind, &flags);
    if (rc) return rc;
    if (t.group >= n_groups) return CS_ERR_INVALID_ARGUMENT;
    const int64_t units =
        t.numel == 0 ? 1 : (t.numel + kDefaultUnitElems - 1) / kDefaultUnitElems;
    if (nu + units > kNaMaxUnits) return CS_ERR_LIMIT;
    TensorDesc& d = g_stage_descs[i];
    d = host::make_desc(t, state_kind, flags);
    any_master = any_master || t.master != nullptr || (flags & kStateF32) != 0;
    all16 = all16 && (t.numel == 0 || t.param_dtype != CS_DTYPE_F32);
    d.n_units = static_cast<int32_t>(units);
    for (int64_t k = 0; k < units; ++k) {
      WorkUnit& w = g_stage_units[nu + k];
      w.start = k * kDefaultUnitElems;
      w.tensor = i;
      w.len = static_cast<int32_t>(std::min<int64_t>(kDefaultUnitElems, t.numel - w.start));
    }
    nu += units;
  }
  // longest first, then tensor and start: the same queue order as a plan's
  std::sort(g_stage_units, g_stage_units + nu, [](const WorkUnit& a, const WorkUnit& b) {
    if (a.len != b.len) return a.len > b.len;
    if (a.tensor != b.tensor) return a.tensor < b.tensor;
    return a.start < b.start;
  });
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CS_ERR_CUDA;
  NaDevice* nd = nullptr;
  const int rc = setup_device(dev, &nd);
  if (rc) return rc;
  unsigned char* base = nd->scratch;
  TensorDesc* d_descs = reinterpret_cast<TensorDesc*>(base);
  WorkUnit* d_units = reinterpret_cast<WorkUnit*>(base + kNaDescBytes);
  uint32_t* d_commit = reinterpret_cast<uint32_t*>(base + kNaDescBytes + kNaUnitBytes);
  uint32_t* d_sched =
      reinterpret_cast<uint32_t*>(base + kNaDescBytes + kNaUnitBytes + kNaCommitBytes);
  // tables of this call (pageable host source: staged by the runtime before
  // the copy returns), then zeroed tickets and scheduler words; the error
  // word (sched[2]) keeps its bits for adamw_noalloc_error
  if (cudaMemcpyAsync(d_descs, g_stage_descs, sizeof(TensorDesc) * n_tensors,
                      cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(d_units, g_stage_units, sizeof(WorkUnit) * nu, cudaMemcpyHostToDevice,
                      s) != cudaSuccess ||
      cudaMemsetAsync(d_commit, 0, kNaCommitBytes + 2 * sizeof(uint32_t), s) != cudaSuccess)
    return CS_ERR_CUDA;
  const int32_t n_units = static_cast<int32_t>(nu);
  bool small = false;
  for (int64_t k = 0; k < nu; ++k) small = small || (g_stage_units[k].len > 0 &&
                                                     g_stage_units[k].len <= kPackMax);
  const int var = pick_variant(state_kind, any_master, all16, small);
  if (n_groups <= kSmallGroups)
    return launch_args<kSmallGroups, kSmallWords>(
        d_descs, d_units, d_commit, d_sched, n_units, n_tensors, state_kind, kClassSmall,
        nd->grid[state_kind][var][kClassSmall], groups, n_groups, grad_present, step, inv_scale,
        found_inf, var, s);
  return launch_args<kMidGroups, kMidWords>(d_descs, d_units, d_commit, d_sched, n_units,
                                            n_tensors, state_kind, kClassMid,
                                            nd->grid[state_kind][var][kClassMid], groups,
                                            n_groups, grad_present, step, inv_scale, found_inf,
                                            var, s);
}

extern "C" int adamw_noalloc_error(uint32_t* out_flags) {
  using namespace cs;
  if (!out_flags) return CS_ERR_INVALID_ARGUMENT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return CS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  NaDevice* nd = nullptr;
  const int rc = setup_device(dev, &nd);
  if (rc) return rc;
  uint32_t* err = reinterpret_cast<uint32_t*>(nd->scratch + kNaDescBytes + kNaUnitBytes +
                                              kNaCommitBytes) + 2;
  uint32_t v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return CS_ERR_CUDA;
  if (v != 0 && (cudaMemset(err, 0, sizeof(v)) != cudaSuccess ||
                 cudaDeviceSynchronize() != cudaSuccess))
    return CS_ERR_CUDA;
  *out_flags = v;
  return CS_OK;
}

extern "C" int adamw_noalloc_set_debug(uint64_t wait_ns, uint32_t flags) {
  using namespace cs;
  if (wait_ns == 0) wait_ns = kDefaultWaitNs;
  if (wait_ns > 60ull * 1000000000ull || (flags & ~uint32_t(kDebugSkipFirstTile)))
    return CS_ERR_INVALID_ARGUMENT;
  std::lock_guard<std::mutex> lock(g_mu);
  g_wait_ns = wait_ns;
  g_debug = flags;
  return CS_OK;
}
