// Shared device helpers of the W4A16 decode kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace bm {

using bf16 = __nv_bfloat16;

constexpr int kWarp = 32;

// Device-side index check: an out-of-range slot, token or expert id is
// skipped and recorded here; the host reads it in bm_engine_sync.
struct DevCheck {
  int* flag;  // may be null
  __device__ __forceinline__ void fail(int code) const {
    if (flag) atomicExch(flag, code);
  }
};

// Programmatic dependent launch.  A kernel launched with launch_k(pdl=true)
// may start while the previous kernel of the stream is finishing: it calls
// pdl_wait() before touching anything that kernel (or any earlier one)
// writes, and pdl_trigger() to let the next kernel start early.  Both are
// no-ops when the kernel was launched the ordinary way.  Every kernel of a
// PDL chain calls pdl_wait() before it writes memory or exits, so the chain
// stays ordered end to end.  Only kernels whose whole grid is resident at
// once trigger, right after their own wait: their dependents' CTAs then fill
// the free slots and run their weight loads (which no kernel writes) before
// their own wait, without holding slots the triggering grid still needs.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_k(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

__device__ __forceinline__ float bf2f(bf16 v) { return __bfloat162float(v); }
__device__ __forceinline__ bf16 f2bf(float v) { return __float2bfloat16_rn(v); }
// Round an fp32 value to the nearest bf16 value and return it as fp32.
__device__ __forceinline__ float round_bf16(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// Low / high bf16 of a packed pair, as fp32 (exact).
__device__ __forceinline__ float bf_lo(uint32_t p) { return __uint_as_float(p << 16); }
__device__ __forceinline__ float bf_hi(uint32_t p) { return __uint_as_float(p & 0xFFFF0000u); }

// The int4 code at nibble `p` (0..7) of a packed word, as the exact fp32 value
// q = u - 8.  0x4B000000 | u is the float 2^23 + u; subtracting 2^23 + 8 is exact.
template <int P>
__device__ __forceinline__ float nib_q(uint32_t w) {
  const uint32_t u = (w >> (4 * P)) & 0xFu;
  return __uint_as_float(0x4B000000u | u) - 8388616.0f;
}

template <typename T>
__device__ __forceinline__ T warp_sum(T v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Sum over the groups of `Width` consecutive lanes, fixed butterfly order.
template <int Width>
__device__ __forceinline__ float group_sum(float v) {
#pragma unroll
  for (int o = Width / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// 1 / sqrt(S / n + eps), S = the CTA-wide sum of the threads' partials ss,
// added in a fixed order (each warp's butterfly, then the warps in ascending
// order).  Every thread returns the same value.  red: >= 32 floats of shared
// memory, not reused by the caller until the next __syncthreads.
__device__ __forceinline__ float block_rms_inv(float ss, int n, float eps, float* red) {
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) tot += red[w];
  return 1.0f / sqrtf(tot / (float)n + eps);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

}  // namespace bm
