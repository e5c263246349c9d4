// Warp-MMA W4A16 family: repack into the mma layout, the dense projection
// launcher and the output projection with the greedy argmax fused in.  The
// projection kernel itself and its layout are described in w4_mma.cuh.
#include "w4_mma.cuh"
#include "w4_mma_shape.h"

namespace bm {

using namespace mma;

namespace {

// Canonical [rows][K/2] + [rows][K/g] -> mma layout (one thread per output
// 16-byte lane word set and per output scale word).  With src2 the output's
// 16-row tile T holds rows 8T..8T+7 of src then the same rows of src2.
__global__ void k_repack_mma(const uint8_t* src, const __half* ssrc, const uint8_t* src2, const __half* ssrc2,
                             int rows, int K, int g, uint8_t* dst, uint32_t* sdst) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int NC = K / kChunkK, NG = K / g;
  auto src_row = [&](int R, const uint8_t* a, const uint8_t* b) -> const uint8_t* {
    if (!b) return a + (size_t)R * (K / 2);
    const int T = R >> 4, rr = R & 15;
    return ((rr < 8) ? a : b) + (size_t)(T * 8 + (rr & 7)) * (K / 2);
  };
  auto code = [](const uint8_t* row, int k) -> uint32_t { return (row[k >> 1] >> ((k & 1) * 4)) & 0xFu; };
  const int64_t nwords = (int64_t)(rows / 16) * NC * 32;
  if (idx < nwords) {
    const int lane = (int)(idx & 31);
    const int64_t tc = idx >> 5;
    const int T = (int)(tc / NC), c = (int)(tc - (int64_t)T * NC);
    const int gq = lane >> 2, t = lane & 3;
    const uint8_t* row0 = src_row(T * 16 + gq, src, src2);
    const uint8_t* row1 = src_row(T * 16 + gq + 8, src, src2);
    uint32_t o[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const int base = c * kChunkK + 32 * (s >> 1) + 8 * t + 4 * (s & 1);
      o[s] = code(row0, base) | code(row1, base) << 4 | code(row0, base + 2) << 8 | code(row1, base + 2) << 12 |
             code(row0, base + 1) << 16 | code(row1, base + 1) << 20 | code(row0, base + 3) << 24 |
             code(row1, base + 3) << 28;
    }
    *reinterpret_cast<uint4*>(dst + (size_t)idx * 16) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  const int64_t nsw = (int64_t)(rows / 16) * NG * 8;
  if (idx < nsw) {
    const int p = (int)(idx & 7);
    const int64_t tg = idx >> 3;
    const int T = (int)(tg / NG), j = (int)(tg - (int64_t)T * NG);
    auto scale = [&](int R) -> uint32_t {
      const __half* s = ssrc + (size_t)R * NG;
      if (ssrc2) {
        const int rr = R & 15;
        s = ((rr < 8) ? ssrc : ssrc2) + (size_t)((R >> 4) * 8 + (rr & 7)) * NG;
      }
      return __half_as_ushort(s[j]);
    };
    sdst[idx] = scale(T * 16 + p) | (scale(T * 16 + p + 8) << 16);
  }
}

template <int MODE, int NT, int CPW, int G>
cudaError_t run(const MmaArgs& a, const Shape& sh, dim3 grid, cudaStream_t st) {
  const int threads = 32 * sh.ks * sh.rtp;
  const size_t smem = (size_t)sh.ks * sh.rtp * 2 * NT * 4 * 32 * sizeof(float);
  if (a.x_bf16) return launch_k(a.pdl != 0, k_w4_mma<MODE, NT, CPW, G, true>, grid, dim3(threads), smem, st, a);
  return launch_k(a.pdl != 0, k_w4_mma<MODE, NT, CPW, G, false>, grid, dim3(threads), smem, st, a);
}

template <int NT>
cudaError_t dense_nt(const MmaArgs& a, const Shape& sh, dim3 grid, cudaStream_t st) {
  if (sh.cpw == 4) {
    if (a.g == 32) return run<DENSE, NT, 4, 32>(a, sh, grid, st);
    if (a.g == 64) return run<DENSE, NT, 4, 64>(a, sh, grid, st);
    return run<DENSE, NT, 4, 128>(a, sh, grid, st);
  }
  if (a.g == 32) return run<DENSE, NT, 2, 32>(a, sh, grid, st);
  if (a.g == 64) return run<DENSE, NT, 2, 64>(a, sh, grid, st);
  return run<DENSE, NT, 2, 128>(a, sh, grid, st);
}

// ---------------------------------------------------------------- output projection

// Order-preserving map of a float to an unsigned key (NaN lowest, -0 = +0).
__device__ __forceinline__ uint32_t ord_key(float v) {
  if (isnan(v)) return 0u;
  if (v == 0.f) v = 0.f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

constexpr int kLmWarps = 8;

// A warp owns RT 16-row tiles of W and the whole K, walking it in chunks of
// 64 with the next chunk's weight loads in flight (two CTAs per SM for the
// wider variants, so enough weight bytes are in flight per SM); the same K permutation as the
// int4 layout lets each lane's A and B fragments of a 32-wide block be 16
// consecutive bytes of a row, so W is read in its plain row-major form.
// Each logit is one fp32 sum over K in a fixed order.
template <int NT, int RT>
__global__ void __launch_bounds__(kLmWarps * 32, NT * RT >= 2 ? 2 : 1) k_lm_mma(LmArgs a) {
  __shared__ unsigned long long best_s[kLmWarps][32];
  __shared__ int last_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, t = lane & 3;
  const int tok0 = blockIdx.y * 8 * NT;
  const int ntok = min(8 * NT, a.B - tok0);
  const int row0 = ((int)blockIdx.x * kLmWarps + warp) * RT * 16;
  const bool active = row0 < a.V;
  const int K = a.K, NC = K / kChunkK;

  float acc[RT][NT][4];
#pragma unroll
  for (int rt = 0; rt < RT; ++rt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[rt][nt][c] = 0.f;

  bool waited = false;
  if (active) {
    const bf16* wr[RT][2];
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
      for (int h = 0; h < 2; ++h) wr[rt][h] = a.W + (size_t)(row0 + rt * 16 + h * 8 + g) * K + 8 * t;
    const bf16* xr[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int tk = nt * 8 + g;
      xr[nt] = tk < ntok ? a.X + (size_t)(tok0 + tk) * K + 8 * t : nullptr;
    }
    // weights: two chunks in flight per warp; activations (the same rows for
    // every warp of the CTA, so mostly L1 hits) are loaded right before use
    uint4 wa[RT][2][2], wb[RT][2][2], xf[NT][2];
    auto loadw = [&](uint4 (&w)[RT][2][2], int c) {
#pragma unroll
      for (int rt = 0; rt < RT; ++rt)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int b = 0; b < 2; ++b) w[rt][h][b] = ldg_nc_v4(wr[rt][h] + c * kChunkK + 32 * b);
    };
    auto loadx = [&](int c) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int b = 0; b < 2; ++b)
          xf[nt][b] = xr[nt] ? *reinterpret_cast<const uint4*>(xr[nt] + c * kChunkK + 32 * b) : make_uint4(0, 0, 0, 0);
    };
    auto compute = [&](const uint4 (&w)[RT][2][2]) {
#pragma unroll
      for (int rt = 0; rt < RT; ++rt)
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          const int b = s >> 1;
          const bool hi = s & 1;
          const uint32_t af[4] = {hi ? w[rt][0][b].z : w[rt][0][b].x, hi ? w[rt][1][b].z : w[rt][1][b].x,
                                  hi ? w[rt][0][b].w : w[rt][0][b].y, hi ? w[rt][1][b].w : w[rt][1][b].y};
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_bf16(acc[rt][nt], af, hi ? xf[nt][b].z : xf[nt][b].x, hi ? xf[nt][b].w : xf[nt][b].y);
        }
    };
    // the first two chunks' weights do not depend on the previous kernel
    loadw(wa, 0);
    if (NC > 1) loadw(wb, 1);
    pdl_wait();
    waited = true;
    for (int c = 0; c < NC; c += 2) {
      loadx(c);
      compute(wa);
      if (c + 2 < NC) loadw(wa, c + 2);
      if (c + 1 < NC) {
        loadx(c + 1);
        compute(wb);
        if (c + 3 < NC) loadw(wb, c + 3);
      }
    }
    // logits: acc[rt][nt][c] is row row0 + 16 rt + g (+8 for c >= 2), token nt * 8 + 2t + (c & 1)
#pragma unroll
    for (int rt = 0; rt < RT; ++rt)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int tk = nt * 8 + 2 * t + (c & 1);
          if (tk < ntok)
            a.logits[(size_t)(tok0 + tk) * a.V + row0 + rt * 16 + g + (c >> 1) * 8] = acc[rt][nt][c];
        }
  }

  if (!waited) pdl_wait();
  // ---- argmax: per token, the largest (value, lowest row) of this warp,
  // then of the CTA, then one atomicMax per token and CTA
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      unsigned long long best = 0ull;
      if (active) {
#pragma unroll
        for (int rt = 0; rt < RT; ++rt)
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t row = row0 + rt * 16 + h * 8 + g;
            const unsigned long long key =
                ((unsigned long long)ord_key(acc[rt][nt][2 * h + j]) << 32) | (0xFFFFFFFFu - row);
            best = key > best ? key : best;
          }
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        const unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
        best = other > best ? other : best;
      }
      if (g == 0) best_s[warp][nt * 8 + 2 * t + j] = best;
    }
  __syncthreads();
  if (threadIdx.x < 8 * NT && (int)threadIdx.x < ntok) {
    unsigned long long best = 0ull;
    for (int w = 0; w < kLmWarps; ++w) best = best_s[w][threadIdx.x] > best ? best_s[w][threadIdx.x] : best;
    atomicMax(a.keys + tok0 + threadIdx.x, best);
  }
  // one thread fences and counts after the barrier that orders the CTA's
  // atomics; the last arrival fences again before releasing the key reads
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned int total = gridDim.x * gridDim.y;
    __threadfence();
    const bool last = atomicAdd(a.counter, 1u) == total - 1;
    if (last) __threadfence();
    last_s = last;
  }
  __syncthreads();
  if (!last_s) return;
  for (int b = threadIdx.x; b < a.B; b += blockDim.x) {
    const unsigned long long key = atomicExch(a.keys + b, 0ull);
    a.next[b] = (int32_t)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull));
    if (a.advance) a.len[a.slots[b]] += a.advance;
  }
  if (threadIdx.x == 0) *a.counter = 0u;
}

template <int NT, int RT>
cudaError_t run_lm(const LmArgs& a, cudaStream_t st) {
  const int rows_per_cta = kLmWarps * RT * 16;
  const dim3 grid((a.V + rows_per_cta - 1) / rows_per_cta, (a.B + 8 * NT - 1) / (8 * NT));
  return launch_k(a.pdl != 0, k_lm_mma<NT, RT>, grid, dim3(kLmWarps * 32), 0, st, a);
}

template <int MODE, int NT, int CPW, int G>
cudaError_t set_attr() {
  const int bytes = kMaxWarps * 2 * NT * 4 * 32 * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k_w4_mma<MODE, NT, CPW, G, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_w4_mma<MODE, NT, CPW, G, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e;
}

}  // namespace

bool mma_supports(int rows, int K, int g) { return mma_shape_ok(rows, K, g); }

bool lm_mma_supports(int V, int K, int B) { return V > 0 && V % 16 == 0 && K > 0 && K % 64 == 0 && B >= 1; }

cudaError_t launch_repack_mma(const uint8_t* W, const __half* S, const uint8_t* W2, const __half* S2, int rows,
                              int K, int g, uint8_t* Wm, uint32_t* Sm, cudaStream_t st) {
  if (!mma_shape_ok(rows, K, g)) return cudaErrorInvalidValue;
  const int64_t nwords = (int64_t)(rows / 16) * (K / kChunkK) * 32;
  const int64_t nsw = (int64_t)(rows / 16) * (K / g) * 8;
  const int64_t n = nwords > nsw ? nwords : nsw;
  k_repack_mma<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(W, S, W2, S2, rows, K, g, Wm, Sm);
  return cudaGetLastError();
}

cudaError_t launch_w4_mma_dense(MmaArgs a, cudaStream_t st) {
  if (!mma_shape_ok(a.rows, a.K, a.g) || a.ntok < 1) return cudaErrorInvalidValue;
  const int NT = a.ntok <= 8 ? 1 : (a.ntok <= 16 ? 2 : 4);
  const int groups = (a.ntok + 8 * NT - 1) / (8 * NT);
  const Shape sh = mma_shape(a.rows, a.K, a.g, groups, 2 * 152);
  a.ks = sh.ks;
  const dim3 grid(a.rows / (32 * sh.rtp), groups);
  if (NT == 1) return dense_nt<1>(a, sh, grid, st);
  if (NT == 2) return dense_nt<2>(a, sh, grid, st);
  return dense_nt<4>(a, sh, grid, st);
}

cudaError_t launch_lm_mma(const LmArgs& a, cudaStream_t st) {
  if (!lm_mma_supports(a.V, a.K, a.B) || !a.keys || !a.counter) return cudaErrorInvalidValue;
  if (a.B <= 8) return a.V % 32 == 0 ? run_lm<1, 2>(a, st) : run_lm<1, 1>(a, st);
  if (a.B <= 16) return a.V % 32 == 0 ? run_lm<2, 2>(a, st) : run_lm<2, 1>(a, st);
  return run_lm<4, 1>(a, st);
}

cudaError_t init_mma_attributes() {
  // the dense kernels with NT = 4 and 16 warps need 64 KB of shared memory
  cudaError_t e = cudaSuccess;
#define BM_MMA_ATTR(CPW, G)                                      \
  if (e == cudaSuccess) e = set_attr<DENSE, 1, CPW, G>();        \
  if (e == cudaSuccess) e = set_attr<DENSE, 2, CPW, G>();        \
  if (e == cudaSuccess) e = set_attr<DENSE, 4, CPW, G>();
  BM_MMA_ATTR(2, 32) BM_MMA_ATTR(2, 64) BM_MMA_ATTR(2, 128) BM_MMA_ATTR(4, 32) BM_MMA_ATTR(4, 64)
  BM_MMA_ATTR(4, 128)
#undef BM_MMA_ATTR
  if (e == cudaSuccess) e = init_mma_expert_attributes();
  return e;
}

}  // namespace bm
