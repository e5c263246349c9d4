// CUDA-core W4A16 dot-product core shared by the dense GEMV and the grouped
// expert kernels.
//
// Work split: a warp is divided into groups of LPR lanes; each group owns R
// weight rows at a time and each lane of a group owns CPL chunks of 32
// consecutive K elements (16 packed bytes, one 128-bit load).  Lane l of a
// group reads chunks c = l, l + LPR, ..., so a group's loads of one row are
// contiguous and coalesced.  Activations are staged once per CTA in shared
// memory as fp32, laid out [m][quad][chunk] (a quad = 4 consecutive K
// elements) so that the LPR lanes of a group read consecutive 16-byte quads
// without bank conflicts.
//
// Reduction order of one output element (fixed, independent of the number of
// activation rows M and of which other rows share the launch):
//   chunk sum  = sum over the 32 elements of a chunk, ascending k, of q * x
//   lane sum   = sum over the lane's chunks, ascending c, of scale * chunk sum
//   result     = butterfly sum of the LPR lane sums (xor 16, 8, 4, 2, 1)
// LPR and CPL depend on K only, so a stream's bytes do not depend on the
// batch it runs in (each row of the batched GEMM is computed on its own, as
// on the batched-serving page, §3, with one reduction order for solo and
// batched as in the KV-slot isolation page's follow-up update).
#pragma once

#include "common.cuh"

namespace bm {

constexpr int kSimtThreads = 256;
constexpr int kSimtWarps = kSimtThreads / kWarp;

// Shared-memory float index of element k of staged row m.
__device__ __forceinline__ int xs_index(int m, int k, int nch) {
  const int c = k >> 5, e = k & 31;
  return (((m * 8 + (e >> 2)) * nch + c) << 2) + (e & 3);
}

// 1 / sqrt(mean(x^2) + eps) of one bf16 row, computed by one warp (fixed order:
// lane-strided fp32 sums, then the warp butterfly).
__device__ __forceinline__ float row_rinv(const bf16* x, int K, float eps, int lane) {
  float ss = 0.f;
  for (int k = lane * 2; k < K; k += 64) {
    const uint32_t p = *reinterpret_cast<const uint32_t*>(x + k);
    const float a = bf_lo(p), b = bf_hi(p);
    ss = fmaf(a, a, ss);
    ss = fmaf(b, b, ss);
  }
  ss = warp_sum(ss);
  return 1.0f / sqrtf(ss / (float)K + eps);
}

// Stage activation rows 0..mcount-1 into shared memory as fp32.  Row m is
// `rows[m]` (a device pointer).  With `do_norm`, each value becomes
// round_bf16(x * rinv * w) — the RMSNorm of the row, rounded to bf16 exactly
// like a standalone norm kernel's output.  Must be reached by every thread of
// the CTA (it synchronises when normalising).
__device__ __forceinline__ void stage_rows(float* xs, const bf16* const* rows, int mcount, int K,
                                           bool do_norm, const bf16* norm_w, float eps, float* rinv_s) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nch = K >> 5;
  if (do_norm) {
    for (int m = warp; m < mcount; m += kSimtWarps) {
      const float r = row_rinv(rows[m], K, eps, lane);
      if (lane == 0) rinv_s[m] = r;
    }
    __syncthreads();
  }
  for (int m = 0; m < mcount; ++m) {
    const bf16* x = rows[m];
    const float r = do_norm ? rinv_s[m] : 1.f;
    for (int k = tid * 2; k < K; k += kSimtThreads * 2) {
      const uint32_t p = *reinterpret_cast<const uint32_t*>(x + k);
      float a = bf_lo(p), b = bf_hi(p);
      if (do_norm) {
        const float wa = norm_w ? bf2f(norm_w[k]) : 1.f;
        const float wb = norm_w ? bf2f(norm_w[k + 1]) : 1.f;
        a = round_bf16(a * r * wa);
        b = round_bf16(b * r * wb);
      }
      xs[xs_index(m, k, nch)] = a;
      xs[xs_index(m, k + 1, nch)] = b;
    }
  }
}

// Load the packed weights and scales of R rows for this lane's CPL chunks.
// wrow[r] / srow[r] point at the first byte / scale of row r, or are null
// for an absent row (loads skipped, zeros).
template <int LPR, int CPL, int R>
__device__ __forceinline__ void load_w4(const uint8_t* const (&wrow)[R], const __half* const (&srow)[R],
                                        int g, int gl, uint4 (&w)[R][CPL], float (&s)[R][CPL]) {
#pragma unroll
  for (int r = 0; r < R; ++r) {
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
      const int c = gl + LPR * j;
      if (wrow[r]) {
        w[r][j] = ldg_nc_v4(wrow[r] + c * 16);
        s[r][j] = __half2float(srow[r][(c * 32) / g]);
      } else {
        w[r][j] = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
        s[r][j] = 0.f;
      }
    }
  }
}

// acc[r][m] (this lane's partial) for the MT staged rows.
template <int LPR, int CPL, int R, int MT>
__device__ __forceinline__ void dot_w4(const uint4 (&w)[R][CPL], const float (&s)[R][CPL],
                                       const float* xs, int nch, int gl, float (&acc)[R][MT]) {
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[r][m] = 0.f;
  const float4* xq = reinterpret_cast<const float4*>(xs);
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    const int c = gl + LPR * j;
    float part[R][MT];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) part[r][m] = 0.f;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      float q[R][8];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const uint32_t word = (wi == 0) ? w[r][j].x : (wi == 1) ? w[r][j].y : (wi == 2) ? w[r][j].z : w[r][j].w;
        q[r][0] = nib_q<0>(word); q[r][1] = nib_q<1>(word);
        q[r][2] = nib_q<2>(word); q[r][3] = nib_q<3>(word);
        q[r][4] = nib_q<4>(word); q[r][5] = nib_q<5>(word);
        q[r][6] = nib_q<6>(word); q[r][7] = nib_q<7>(word);
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        const float4 x0 = xq[(m * 8 + 2 * wi) * nch + c];
        const float4 x1 = xq[(m * 8 + 2 * wi + 1) * nch + c];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          float p = part[r][m];
          p = fmaf(q[r][0], x0.x, p); p = fmaf(q[r][1], x0.y, p);
          p = fmaf(q[r][2], x0.z, p); p = fmaf(q[r][3], x0.w, p);
          p = fmaf(q[r][4], x1.x, p); p = fmaf(q[r][5], x1.y, p);
          p = fmaf(q[r][6], x1.z, p); p = fmaf(q[r][7], x1.w, p);
          part[r][m] = p;
        }
      }
    }
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[r][m] = fmaf(s[r][j], part[r][m], acc[r][m]);
  }
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[r][m] = group_sum<LPR>(acc[r][m]);
}

constexpr int kMaxTile = 4;   // activation rows staged per pass

// One pass over `mcount` (1..kMaxTile) staged rows; emit(r, m, value) is
// called on every lane with the group's total for weight row r and
// activation row m.  The arithmetic of one (r, m) element is the same for
// every mcount, so a stream's bytes do not depend on how many other rows
// share its pass.
template <int LPR, int CPL, int R, class Emit>
__device__ __forceinline__ void dot_tile(const uint4 (&w)[R][CPL], const float (&s)[R][CPL], const float* xs,
                                         int nch, int gl, int mcount, Emit emit) {
  if (mcount >= 4) {
    float acc[R][4];
    dot_w4<LPR, CPL, R, 4>(w, s, xs, nch, gl, acc);
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < 4; ++m) emit(r, m, acc[r][m]);
  } else if (mcount == 3) {
    float acc[R][3];
    dot_w4<LPR, CPL, R, 3>(w, s, xs, nch, gl, acc);
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < 3; ++m) emit(r, m, acc[r][m]);
  } else if (mcount == 2) {
    float acc[R][2];
    dot_w4<LPR, CPL, R, 2>(w, s, xs, nch, gl, acc);
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int m = 0; m < 2; ++m) emit(r, m, acc[r][m]);
  } else {
    float acc[R][1];
    dot_w4<LPR, CPL, R, 1>(w, s, xs, nch, gl, acc);
#pragma unroll
    for (int r = 0; r < R; ++r) emit(r, 0, acc[r][0]);
  }
}

}  // namespace bm
