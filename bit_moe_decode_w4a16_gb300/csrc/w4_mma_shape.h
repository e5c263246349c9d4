// Work split of the warp-MMA projections (host side).  It depends only on
// the matrix shape: a warp covers 2 x 16 rows and CPW chunks of 64 along K,
// KS = (K / 64) / CPW warps share the rows, and a CTA holds RTP such row
// pairs (KS x RTP <= 16 warps).
#pragma once

#include <cuda_runtime.h>

namespace bm {

struct Shape {
  int cpw = 0, ks = 0, rtp = 0;
};

inline bool mma_shape_ok(int rows, int K, int g) {
  return rows > 0 && rows % 32 == 0 && K >= 128 && K % 128 == 0 && K <= 4096 && (g == 32 || g == 64 || g == 128) &&
         K % g == 0;
}

// rtp is the largest that keeps at least `min_ctas` CTAs in a launch of
// `groups` token groups (it only regroups warps: no sum depends on it).
inline Shape mma_shape(int rows, int K, int /*g*/, int groups = 0, int min_ctas = 0) {
  Shape s;
  const int nc = K / 64;                          // even: K % 128 == 0
  s.cpw = nc % 4 == 0 ? 4 : 2;                    // 256 or 128 of K per warp
  s.ks = nc / s.cpw;                              // <= 16 for K <= 4096
  s.rtp = 1;
  while (s.rtp * 2 * s.ks <= 16 && rows % (32 * s.rtp * 2) == 0 &&
         (long)(rows / (32 * s.rtp * 2)) * groups >= min_ctas)
    s.rtp *= 2;
  return s;
}

cudaError_t init_mma_expert_attributes();

}  // namespace bm
