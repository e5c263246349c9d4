// Timing probe of the tcgen05 MMA on this GPU, for the measurement tools
// (bench.py --tc-probe): one CTA issues `iters` stages of four kind::f16 MMAs
// of M 128 x N x K 16 into one TMEM accumulator, and the issuing thread's
// clock gives the SM cycles per MMA, to issue the run and to see it complete
// (its commit's mbarrier).  Variants: A from tensor memory or from shared
// memory; the shared-memory operands in the no-swizzle core-matrix layout
// (8 rows x 16 bytes per core matrix) or the 128-byte-swizzled K-major layout
// (rows of 128 bytes, 16-byte chunks permuted within each 8-row atom).  The
// operands are zero: only time is measured, and every address stays inside
// the CTA's tiles.
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace bm {

namespace {

constexpr int kProbeATile = 128 * 128;   // A: 128 rows x 64 fp16
constexpr int kProbeBTile = 256 * 128;   // B: up to 256 rows x 64 fp16
constexpr int kProbeSmem = kProbeATile + kProbeBTile + 1024;   // + alignment slack

// K-major, 128-byte swizzle: 8-row atoms of 1024 bytes (SBO), LBO unused
// (encoded 1), layout type 2; the start address moves by 32 bytes per K 16.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}

// roundtrip = 1: commit and wait after every stage of four MMAs, so the
// cycles per MMA include the commit-to-mbarrier latency of each stage.
__global__ void __launch_bounds__(128, 1) k_tc_probe(int n, int a_tmem, int swz, int iters, int roundtrip,
                                                     unsigned long long* out) {
  extern __shared__ unsigned char raw[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tslot;
  const uint32_t base0 = tc::smem_u32(raw);
  const uint32_t pad = (1024u - (base0 & 1023u)) & 1023u;   // 1024-byte aligned tiles
  unsigned char* sm = raw + pad;
  for (int i = threadIdx.x; i < (kProbeATile + kProbeBTile) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x < 32) {
    tc::tmem_alloc(tc::smem_u32(&tslot), 512);
    tc::tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    tc::mbar_init(tc::smem_u32(&bar), 1);
    tc::fence_mbar_init();
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tslot;
  if (threadIdx.x == 0) {
    const uint32_t a_base = tc::smem_u32(sm), b_base = a_base + kProbeATile;
    const uint32_t idesc = tc::idesc_f16_f32(128, n);
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint64_t bd = swz ? smem_desc_sw128(b_base + 32u * q) : tc::smem_desc_noswizzle(b_base + 256u * q, 128u, 1024u);
        const uint32_t acc = (uint32_t)(it > 0 || q > 0);
        if (a_tmem) {
          tc::mma_f16_tmem_a(tmem, tmem + 256 + q * 8, bd, idesc, acc);
        } else {
          const uint64_t ad = swz ? smem_desc_sw128(a_base + 32u * q) : tc::smem_desc_noswizzle(a_base + 256u * q, 128u, 1024u);
          tc::mma_f16_ss(tmem, ad, bd, idesc, acc);
        }
      }
      if (roundtrip) {
        tc::mma_commit(tc::smem_u32(&bar));
        if (!tc::mbar_wait(tc::smem_u32(&bar), (uint32_t)(it & 1), 1u << 18)) break;
      }
    }
    const long long t1 = clock64();
    tc::mma_commit(tc::smem_u32(&bar));
    const bool ok = tc::mbar_wait(tc::smem_u32(&bar), roundtrip ? (uint32_t)(iters & 1) : 0u, 1u << 18);
    const long long t2 = clock64();
    out[0] = (unsigned long long)(t1 - t0);
    out[1] = (unsigned long long)(t2 - t0);
    out[2] = ok ? 1ull : 0ull;
  }
  tc::fence_before_sync();
  __syncthreads();
  if (threadIdx.x < 32) tc::tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_tc_probe(int n, int a_tmem, int swz, int iters, int roundtrip, unsigned long long* out,
                            cudaStream_t st) {
  if (n < 16 || n > 256 || n % 16 || iters < 1 || iters > 4096) return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_tc_probe, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  k_tc_probe<<<1, 128, kProbeSmem, st>>>(n, a_tmem, swz, iters, roundtrip, out);
  return cudaGetLastError();
}

}  // namespace bm

#include "errors.h"

extern "C" bm_status bm_probe_tcgen05_mma(int n, int a_in_tmem, int swizzle128, int iters, int roundtrip,
                                          double* issue_cycles, double* complete_cycles) {
  if (!issue_cycles || !complete_cycles) return bm::set_error(BM_ERR_INVALID_ARG, "bm_probe_tcgen05_mma: null argument");
  unsigned long long* d = nullptr;
  cudaError_t e = cudaMalloc(&d, 3 * sizeof(unsigned long long));
  if (e == cudaSuccess) e = bm::launch_tc_probe(n, a_in_tmem, swizzle128, iters, roundtrip, d, nullptr);
  unsigned long long h[3] = {0, 0, 0};
  if (e == cudaSuccess) e = cudaMemcpy(h, d, sizeof(h), cudaMemcpyDeviceToHost);
  if (d) cudaFree(d);
  if (e == cudaErrorInvalidValue)
    return bm::set_error(BM_ERR_INVALID_ARG, "bm_probe_tcgen05_mma: need n a multiple of 16 in [16, 256], iters in [1, 4096]");
  if (e != cudaSuccess) return bm::set_error(BM_ERR_CUDA, std::string("bm_probe_tcgen05_mma: ") + cudaGetErrorString(e));
  if (!h[2]) return bm::set_error(BM_ERR_DEVICE_CHECK, "bm_probe_tcgen05_mma: the completion wait timed out");
  *issue_cycles = (double)h[0] / (4.0 * iters);
  *complete_cycles = (double)h[1] / (4.0 * iters);
  return bm::ok();
}
