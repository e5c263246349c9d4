// Warp-MMA W4A16 family: the grouped expert gate/up (SiLU fused) and down
// projections.  The persistent staged kernel (w4_mma_staged.cuh) runs them
// whenever a work item's stage fits in shared memory twice; otherwise
// k_w4_mma does, with grid x = row block of one expert matrix and y = routing
// job (an expert and up to 8 of its sorted tokens), in expert order.  Both
// compute every output with the same arithmetic in the same order.
#include "w4_mma_shape.h"
#include "w4_mma_staged.cuh"

namespace bm {

using namespace mma;

namespace {

constexpr size_t kSmemLimit = 227 * 1024;

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 132;
  return n;
}

// Geometry of the staged kernel for this matrix: items of 32 x rtp rows
// (rtp = the shape's row pairs per CTA), one CTA per SM with as many stages
// as fit (at most kMaxStages); ns = 0 if two do not fit.
StagedGeom staged_geom(const MmaArgs& a, const Shape& sh) {
  StagedGeom g{};
  g.rtp = sh.rtp;
  g.nw = sh.ks * sh.rtp;
  const int rows = 32 * sh.rtp;
  g.nrb = a.rows / rows;
  g.w_bytes = (uint32_t)rows * (uint32_t)(a.K / 2);
  g.s_bytes = (uint32_t)rows * (uint32_t)(a.K / a.g) * 2u;
  g.x_stride = (uint32_t)(a.K + kXPad) * 2u;
  g.stage = (g.w_bytes + g.s_bytes + (uint32_t)kJobTokens * g.x_stride + 127u) & ~127u;
  const size_t red = (size_t)g.nw * 2 * 4 * 32 * sizeof(float);
  const size_t per_cta = kSmemLimit - red - 1024;
  const int ns = (int)(per_cta / g.stage);
  g.ns = ns >= 2 ? (ns > kMaxStages ? kMaxStages : ns) : 0;
  return g;
}

template <int MODE, int CPW, int G>
cudaError_t run_staged(const MmaArgs& a, const StagedGeom& geo, cudaStream_t st) {
  const size_t smem = (size_t)geo.ns * geo.stage + (size_t)geo.nw * 2 * 4 * 32 * sizeof(float);
  const int threads = (geo.nw + 1) * 32;
  static bool attr_set = false;   // per instantiation; the limit is the same on every device
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_w4_mma_staged<MODE, CPW, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(kSmemLimit - 1024));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_w4_mma_staged<MODE, CPW, G>, threads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  const long items = (long)a.max_jobs * geo.nrb;
  const long cap = (long)sm_count() * per_sm;
  const int grid = (int)(items < cap ? items : cap);
  return launch_k(a.pdl != 0, k_w4_mma_staged<MODE, CPW, G>, dim3(grid), dim3(threads), smem, st, a, geo);
}

template <int MODE, int CPW, int G>
cudaError_t run(const MmaArgs& a, const Shape& sh, cudaStream_t st) {
  const StagedGeom geo = staged_geom(a, sh);
  if (geo.ns >= 2) return run_staged<MODE, CPW, G>(a, geo, st);
  const dim3 grid(a.rows / (32 * sh.rtp), a.max_jobs);
  const size_t smem = (size_t)sh.ks * sh.rtp * 2 * 4 * 32 * sizeof(float);
  return launch_k(a.pdl != 0, k_w4_mma<MODE, 1, CPW, G, false>, grid, dim3(32 * sh.ks * sh.rtp), smem, st, a);
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

cudaError_t init_mma_expert_attributes() { return cudaSuccess; }

}  // namespace bm
