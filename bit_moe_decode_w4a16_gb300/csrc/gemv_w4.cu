// Dense W4A16 projection on CUDA cores: Y = X · Wᵀ (+ R), optionally with
// the RMSNorm of X fused into the activation staging.
//
// Every packed weight byte is read from HBM once per launch, whatever M is
// (the batched 4-bit GEMM of the batched-serving page, §1: one read of each
// packed dense weight serves all B rows); the weights of a warp's
// rows stay in registers while the CTA walks the activation rows in tiles
// of up to four.
#include "kernels.cuh"
#include "w4_simt.cuh"

namespace bm {

namespace {

template <int LPR, int CPL>
__global__ void __launch_bounds__(kSimtThreads) k_w4_gemv(GemvArgs a) {
  extern __shared__ float xs[];
  __shared__ const bf16* rows[kMaxTile];
  __shared__ float rinv_s[kMaxTile];
  constexpr int R = 2;
  constexpr int kGroups = kWarp / LPR;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPR, gl = lane % LPR;
  const int n0 = blockIdx.x * (kSimtWarps * kGroups * R) + (warp * kGroups + grp) * R;
  const uint8_t* wrow[R];
  const __half* srow[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const bool ok = n0 + r < a.N;
    wrow[r] = ok ? a.W + (size_t)(n0 + r) * (a.K >> 1) : nullptr;
    srow[r] = ok ? a.S + (size_t)(n0 + r) * (a.K / a.g) : nullptr;
  }
  uint4 w[R][CPL];
  float s[R][CPL];
  load_w4<LPR, CPL, R>(wrow, srow, a.g, gl, w, s);
  const int nch = a.K >> 5;
  for (int m0 = 0; m0 < a.M; m0 += kMaxTile) {
    const int mc = min(kMaxTile, a.M - m0);
    __syncthreads();
    if (threadIdx.x < mc) rows[threadIdx.x] = a.X + (size_t)(m0 + threadIdx.x) * a.ldx;
    __syncthreads();
    stage_rows(xs, rows, mc, a.K, a.do_norm != 0, a.norm_w, a.eps, rinv_s);
    __syncthreads();
    dot_tile<LPR, CPL, R>(w, s, xs, nch, gl, mc, [&](int r, int m, float v) {
      if (wrow[r] && gl == ((r * kMaxTile + m) % LPR)) {
        const size_t mm = m0 + m, n = n0 + r;
        if (a.Res) v += bf2f(a.Res[mm * a.ldr + n]);
        a.Y[mm * a.ldy + n] = f2bf(v);
      }
    });
  }
}

template <int LPR, int CPL>
cudaError_t run(const GemvArgs& a, cudaStream_t st) {
  constexpr int rows_per_cta = kSimtWarps * (kWarp / LPR) * 2;
  const int grid = (a.N + rows_per_cta - 1) / rows_per_cta;
  const size_t smem = (size_t)min(a.M, kMaxTile) * a.K * sizeof(float);
  k_w4_gemv<LPR, CPL><<<grid, kSimtThreads, smem, st>>>(a);
  return cudaGetLastError();
}

template <int LPR, int CPL>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(k_w4_gemv<LPR, CPL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              kMaxTile * LPR * CPL * 32 * (int)sizeof(float));
}

}  // namespace

// (LPR, CPL) by number of 32-element chunks; LPR * CPL == K / 32.
#define BM_SIMT_SHAPES(X) X(32, 1) X(32, 2) X(32, 3) X(32, 4) X(16, 1) X(16, 3) X(8, 1) X(8, 3)

bool simt_supports_k(int K) {
  if (K <= 0 || K % 32 != 0) return false;
  const int nch = K / 32;
#define BM_CASE(L, C) if (nch == (L) * (C)) return true;
  BM_SIMT_SHAPES(BM_CASE)
#undef BM_CASE
  return false;
}

cudaError_t launch_w4_gemv(const GemvArgs& a, cudaStream_t st) {
  const int nch = a.K / 32;
#define BM_CASE(L, C) if (nch == (L) * (C)) return run<L, C>(a, st);
  BM_SIMT_SHAPES(BM_CASE)
#undef BM_CASE
  return cudaErrorInvalidValue;
}

cudaError_t init_gemv_attributes() {
  cudaError_t e = cudaSuccess;
#define BM_CASE(L, C) if (e == cudaSuccess) e = set_attr<L, C>();
  BM_SIMT_SHAPES(BM_CASE)
#undef BM_CASE
  return e;
}

}  // namespace bm
