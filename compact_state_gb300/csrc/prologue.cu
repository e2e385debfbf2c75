// Gradient prologue for sm_103a: one pass over every present gradient before
// the AdamW step, computing the non-finite flag, the global L2 norm of the
// unscaled gradients, and the factor the step should scale gradients by.
//
// "Fused Optimizers and State Precision", section 06: mixed-precision training
// unscales the gradients, checks them for non-finite values and clips them,
// and only then updates; a step skipped by the check leaves everything
// untouched. The Apex fused-optimizers guide does the check (FusedAdam
// capturable path, section 4.3) and the global gradient norm (FusedLAMB,
// section 5.3) on the device, so nothing syncs the host. Here:
//   found_inf = 1 if any g*inv_scale (fp32) of a present tensor is NaN/inf;
//   norm      = sqrt(sum (g*inv_scale)^2) over present tensors;
//   scale     = inv_scale * min(1, max_norm / (norm + 1e-6))   (max_norm > 0),
//               inv_scale otherwise or when found_inf is set.
// found_inf and scale are then adamw_step's found_inf and inv_scale: unscale,
// check, clip and update happen in that order, all on the device.
//
// Work: the plan's work units cut into 8192-element items, assigned to blocks
// round-robin (items of one size class, so blocks stay balanced without a
// queue). Each thread squares its elements in fp32, sums four at a time and
// adds the group sums with Kahan compensation; blocks combine in fp64; the
// last block to finish adds the per-block sums in block order (so the result
// does not depend on timing), writes the outputs and rewinds its counters.
// Squares are fp32: a single unscaled value above ~1.8e19 makes the norm
// infinite (clip factor 0) although the value itself is finite.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cmath>
#include <cstdint>

#include "prologue.h"

namespace cs {
namespace {

__device__ __forceinline__ bool nonfinite(float x) {
  return (__float_as_uint(x) & 0x7f800000u) == 0x7f800000u;
}

// Kahan-compensated running sum (s - c is the sum).
struct Kahan {
  float s = 0.0f, c = 0.0f;
  __device__ __forceinline__ void add(float x) {
    const float y = x - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
};

__device__ __forceinline__ void group4(float a, float b, float c, float d, float inv, Kahan& k,
                                       bool& bad) {
  a *= inv; b *= inv; c *= inv; d *= inv;
  bad |= nonfinite(a) | nonfinite(b) | nonfinite(c) | nonfinite(d);
  k.add(fmaf(a, a, b * b) + fmaf(c, c, d * d));
}

__device__ __forceinline__ float to_f32_bf16(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}
__device__ __forceinline__ float to_f32_f16(uint16_t h) {
  return __half2float(*reinterpret_cast<const __half*>(&h));
}

// Bulk L2 prefetch of the 16-byte-aligned part of [p, p + bytes): a hint with
// no completion to wait for.
__device__ __forceinline__ void prefetch_l2(const void* p, int64_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  const uintptr_t lo = (a + 15) & ~uintptr_t(15);
  const uintptr_t hi = (a + static_cast<uintptr_t>(bytes)) & ~uintptr_t(15);
  if (hi > lo) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                 :: "l"(lo), "r"(static_cast<uint32_t>(hi - lo)) : "memory");
  }
}

// Four consecutive gradient elements starting at e (16-byte or 8-byte aligned).
template <int DT>
__device__ __forceinline__ void load4(const void* grad, int64_t e, float (&x)[4]) {
  if constexpr (DT == CS_DTYPE_F32) {
    const float4 r = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(grad) + e));
    x[0] = r.x; x[1] = r.y; x[2] = r.z; x[3] = r.w;
  } else {
    const uint2 r = __ldcs(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(grad) + e));
    if constexpr (DT == CS_DTYPE_BF16) {
      x[0] = __uint_as_float(r.x << 16);
      x[1] = __uint_as_float(r.x & 0xffff0000u);
      x[2] = __uint_as_float(r.y << 16);
      x[3] = __uint_as_float(r.y & 0xffff0000u);
    } else {
      const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&r.x));
      const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&r.y));
      x[0] = lo.x; x[1] = lo.y; x[2] = hi.x; x[3] = hi.y;
    }
  }
}

// Sum of squares of elements [s0, s0+len) of one gradient, dtype DT.
template <int DT>
__device__ __forceinline__ void accumulate(const void* grad, int64_t s0, int len, bool vec,
                                           float inv, Kahan& k, bool& bad) {
  int done = 0;
  if (vec) {
    // Full passes: kU independent 4-element groups per thread, all loads
    // issued before any arithmetic; then the remaining groups one at a time.
    constexpr int kU = 8;
    constexpr int kPass = kPrologueThreads * kU;
    const int ng = len >> 2;
    const int full = ng - ng % kPass;
    for (int base = threadIdx.x; base < full; base += kPass) {
      float x[kU][4];
#pragma unroll
      for (int u = 0; u < kU; ++u) load4<DT>(grad, s0 + 4 * int64_t(base + u * kPrologueThreads), x[u]);
#pragma unroll
      for (int u = 0; u < kU; ++u) group4(x[u][0], x[u][1], x[u][2], x[u][3], inv, k, bad);
    }
    for (int gi = full + threadIdx.x; gi < ng; gi += kPrologueThreads) {
      float x[4];
      load4<DT>(grad, s0 + 4 * int64_t(gi), x);
      group4(x[0], x[1], x[2], x[3], inv, k, bad);
    }
    done = ng << 2;
  }
  for (int i = done + threadIdx.x; i < len; i += kPrologueThreads) {
    const int64_t e = s0 + i;
    float x;
    if constexpr (DT == CS_DTYPE_F32) {
      x = __ldcs(static_cast<const float*>(grad) + e);
    } else {
      const uint16_t h = __ldcs(reinterpret_cast<const unsigned short*>(grad) + e);
      x = DT == CS_DTYPE_BF16 ? to_f32_bf16(h) : to_f32_f16(h);
    }
    x *= inv;
    bad |= nonfinite(x);
    k.add(x * x);
  }
}

// Sum of one fp64 value per thread over the block, in a fixed order; the
// result is valid in thread 0. Ends with the block synchronised.
__device__ __forceinline__ double block_sum(double x) {
  __shared__ double warp_sums[kPrologueThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  __syncthreads();   // warp_sums may still be read by an earlier call
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = x;
  __syncthreads();
  double b = 0.0;
  if (threadIdx.x == 0) {
    for (int w = 0; w < kPrologueThreads / 32; ++w) b += warp_sums[w];
  }
  return b;
}

template <int MAXW>
__global__ void __launch_bounds__(kPrologueThreads, kPrologueBlocksPerSm)
grad_prologue_kernel(const __grid_constant__ PrologueArgs<MAXW> a) {
  // Programmatic dependent launch, as in the step kernel: the step launched
  // next may place its CTAs as this grid's CTAs leave; this grid touches
  // global memory only once the grids it depends on have completed.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const float inv = (a.inv_scale != nullptr) ? *a.inv_scale : 1.0f;
  Kahan k;
  bool bad = false;
  const int64_t n_items = static_cast<int64_t>(a.n_units) * a.pieces_per_unit;
  // The next item's unit record and gradient descriptor are read while the
  // current item streams, and one thread asks L2 to prefetch the next item's
  // gradient bytes: registers hold only about one vector load per thread in
  // flight, and the prefetch keeps HBM busy beyond that.
  struct Item {
    const void* grad;
    int64_t s0;
    int32_t len;     // 0: nothing to do (past the unit's end or tensor absent)
    int32_t dtype, flags;
  };
  // item = unit * pieces_per_unit + piece, stepped by gridDim.x without division
  const int32_t ppu = a.pieces_per_unit;
  const int64_t step_u = gridDim.x / ppu;
  const int32_t step_p = static_cast<int32_t>(gridDim.x % ppu);
  int64_t nu = blockIdx.x / ppu;            // unit and piece of the next item
  int32_t np = static_cast<int32_t>(blockIdx.x % ppu);
  auto fetch = [&]() {
    Item it{};
    const WorkUnit w = a.units[nu];
    const int32_t off = np * kProloguePiece;
    nu += step_u;
    np += step_p;
    if (np >= ppu) { np -= ppu; ++nu; }
    const int ti = w.tensor;
    if (off >= w.len || (!a.all_present && !((a.present[ti >> 5] >> (ti & 31)) & 1u))) return it;
    const TensorDesc& d = a.descs[ti];
    it.grad = d.grad;
    it.dtype = d.param_dtype;
    it.flags = d.flags;
    it.s0 = w.start + off;
    it.len = min(kProloguePiece, w.len - off);
    if (threadIdx.x == 0) {
      const int es = it.dtype == CS_DTYPE_F32 ? 4 : 2;
      prefetch_l2(static_cast<const char*>(it.grad) + it.s0 * es, int64_t(it.len) * es);
    }
    return it;
  };
  Item next{};
  if (blockIdx.x < n_items) next = fetch();
  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const Item cur = next;
    if (item + gridDim.x < n_items) next = fetch();
    if (cur.len == 0) continue;
    const bool vec = (cur.flags & kVec) != 0;
    switch (cur.dtype) {
      case CS_DTYPE_F32: accumulate<CS_DTYPE_F32>(cur.grad, cur.s0, cur.len, vec, inv, k, bad); break;
      case CS_DTYPE_BF16: accumulate<CS_DTYPE_BF16>(cur.grad, cur.s0, cur.len, vec, inv, k, bad); break;
      default: accumulate<CS_DTYPE_F16>(cur.grad, cur.s0, cur.len, vec, inv, k, bad); break;
    }
  }
  // block sum in fp64
  double sum = static_cast<double>(k.s) - static_cast<double>(k.c);
  sum = block_sum(sum);
  __shared__ bool last;
  const int any_bad = __syncthreads_or(bad ? 1 : 0);
  if (threadIdx.x == 0) {
    a.partial[blockIdx.x] = sum;
    if (any_bad) atomicOr(a.words + 1, 1u);
    __threadfence();
    last = atomicAdd(a.words, 1u) + 1u == gridDim.x;
  }
  __syncthreads();
  if (!last) return;
  // The last block: every thread adds a fixed, strided subset of the per-block
  // sums, then the block combines them in a fixed tree, so the total does not
  // depend on which block finished last.
  __threadfence();
  double t = 0.0;
  for (unsigned b = threadIdx.x; b < gridDim.x; b += kPrologueThreads) t += __ldcg(a.partial + b);
  const double total = block_sum(t);
  if (threadIdx.x != 0) return;
  const bool found = atomicAdd(a.words + 1, 0u) != 0u;
  float scale = inv;
  float norm = NAN;
  if (!found) {
    const double nd = sqrt(total);
    norm = static_cast<float>(nd);
    if (a.max_norm > 0.0f) {
      const double coef = fmin(1.0, static_cast<double>(a.max_norm) / (nd + 1e-6));
      scale = static_cast<float>(static_cast<double>(inv) * coef);
    }
  }
  *a.found_inf_out = found ? 1.0f : 0.0f;
  *a.scale_out = scale;
  if (a.norm_out != nullptr) *a.norm_out = norm;
  a.words[0] = 0u;
  a.words[1] = 0u;
}

template <int W>
cudaError_t occupancy_w(int* blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, grad_prologue_kernel<W>,
                                                       kPrologueThreads, 0);
}

template <int W>
cudaError_t launch_w(const void* args, int grid, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kPrologueThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, grad_prologue_kernel<W>,
                            *static_cast<const PrologueArgs<W>*>(args));
}

}  // namespace

cudaError_t prologue_occupancy(ArgClass cls, int* blocks_per_sm) {
  switch (cls) {
    case kClassSmall: return occupancy_w<kSmallWords>(blocks_per_sm);
    case kClassMid: return occupancy_w<kMidWords>(blocks_per_sm);
    default: return occupancy_w<kLargeWords>(blocks_per_sm);
  }
}

cudaError_t launch_prologue(ArgClass cls, const void* args, int grid, cudaStream_t stream) {
  switch (cls) {
    case kClassSmall: return launch_w<kSmallWords>(args, grid, stream);
    case kClassMid: return launch_w<kMidWords>(args, grid, stream);
    default: return launch_w<kLargeWords>(args, grid, stream);
  }
}

}  // namespace cs
