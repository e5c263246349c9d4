// Warp-MMA W4A16 family: the grouped expert gate/up (SiLU fused) and down
// projections.  Grid x = row block of one expert matrix, y = routing job (one
// active expert and up to 8 of its sorted tokens, in expert order, so the
// CTAs that read an expert's rows run next to each other).
#include "w4_mma.cuh"
#include "w4_mma_shape.h"

namespace bm {

using namespace mma;

namespace {

template <int MODE, int CPW, int G>
cudaError_t run(const MmaArgs& a, const Shape& sh, cudaStream_t st) {
  const dim3 grid(a.rows / (32 * sh.rtp), a.max_jobs);
  const size_t smem = (size_t)sh.ks * sh.rtp * 2 * 4 * 32 * sizeof(float);
  k_w4_mma<MODE, 1, CPW, G><<<grid, 32 * sh.ks * sh.rtp, smem, st>>>(a);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch(MmaArgs a, cudaStream_t st) {
  if (!mma_shape_ok(a.rows, a.K, a.g) || a.max_jobs < 1 || !a.n_jobs || !a.jobs) return cudaErrorInvalidValue;
  const Shape sh = mma_shape(a.rows, a.K, a.g);
  a.ks = sh.ks;
  if (sh.cpw == 4) {
    if (a.g == 32) return run<MODE, 4, 32>(a, sh, st);
    if (a.g == 64) return run<MODE, 4, 64>(a, sh, st);
    return run<MODE, 4, 128>(a, sh, st);
  }
  if (a.g == 32) return run<MODE, 2, 32>(a, sh, st);
  if (a.g == 64) return run<MODE, 2, 64>(a, sh, st);
  return run<MODE, 2, 128>(a, sh, st);
}

}  // namespace

cudaError_t launch_w4_mma_gateup(MmaArgs a, cudaStream_t st) { return launch<GATEUP>(a, st); }
cudaError_t launch_w4_mma_down(MmaArgs a, cudaStream_t st) { return launch<DOWN>(a, st); }

cudaError_t init_mma_expert_attributes() {
  // at most 16 warps x 1 KB of partial sums: within the default 48 KB
  return cudaSuccess;
}

}  // namespace bm
