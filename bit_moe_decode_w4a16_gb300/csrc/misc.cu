// Embedding gather, bf16 output projection, greedy argmax, slot-length
// advance and the int4 encoder.
#include <float.h>

#include "kernels.cuh"
#include "w4_simt.cuh"

namespace bm {

namespace {

__global__ void k_embed(const bf16* table, int V, int H, const int32_t* tokens, bf16* x, DevCheck chk) {
  const int b = blockIdx.x;
  const int tok = tokens[b];
  uint4* dst = reinterpret_cast<uint4*>(x + (size_t)b * H);
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) chk.fail(3);
    for (int i = threadIdx.x; i < H / 8; i += blockDim.x) dst[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(table + (size_t)tok * H);
  for (int i = threadIdx.x; i < H / 8; i += blockDim.x) dst[i] = src[i];
}

// One CTA per token: x = the embedding row, xn = bf16(x * rinv * nw).
__global__ void __launch_bounds__(256) k_embed_norm(const bf16* table, int V, int H, const int32_t* tokens, bf16* x,
                                                    const bf16* nw, float eps, __half* xn, DevCheck chk) {
  __shared__ float red[32];
  pdl_wait();
  pdl_trigger();   // one wave: the next projection may start its weight loads
  const int b = blockIdx.x;
  int tok = tokens[b];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) chk.fail(3);
    tok = -1;
  }
  float ss = 0.f;
  for (int h = threadIdx.x; h < H; h += blockDim.x) {
    const bf16 v = tok >= 0 ? table[(size_t)tok * H + h] : f2bf(0.f);
    x[(size_t)b * H + h] = v;
    ss = fmaf(bf2f(v), bf2f(v), ss);
  }
  const float r = block_rms_inv(ss, H, eps, red);
  for (int h = threadIdx.x; h < H; h += blockDim.x)
    xn[(size_t)b * H + h] = __float2half_rn(round_bf16(bf2f(x[(size_t)b * H + h]) * r * (nw ? bf2f(nw[h]) : 1.f)));
}

// logits[m][v] = sum_k xn[m][k] * W[v][k]; a lane group of LPR lanes owns two
// vocab rows; each lane owns CPL chunks of 32 consecutive k (64 bytes).
// Order per element: ascending k within a chunk, ascending chunk per lane,
// butterfly over the group.
template <int LPR, int CPL>
__global__ void __launch_bounds__(kSimtThreads) k_lm_head(const bf16* W, int V, int H, const bf16* x,
                                                          const bf16* norm_w, float eps, float* logits, int B) {
  extern __shared__ float xs[];
  __shared__ const bf16* rows[kMaxTile];
  __shared__ float rinv_s[kMaxTile];
  constexpr int R = 2, kGroups = kWarp / LPR;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPR, gl = lane % LPR;
  const int v0 = blockIdx.x * (kSimtWarps * kGroups * R) + (warp * kGroups + grp) * R;
  uint4 w[R][CPL][4];
#pragma unroll
  for (int r = 0; r < R; ++r)
#pragma unroll
    for (int j = 0; j < CPL; ++j)
#pragma unroll
      for (int u = 0; u < 4; ++u)
        w[r][j][u] = (v0 + r < V) ? ldg_nc_v4(W + (size_t)(v0 + r) * H + (gl + LPR * j) * 32 + u * 8)
                                  : make_uint4(0, 0, 0, 0);
  const int nch = H >> 5;
  const float4* xq = reinterpret_cast<const float4*>(xs);
  for (int m0 = 0; m0 < B; m0 += kMaxTile) {
    const int mc = min(kMaxTile, B - m0);
    __syncthreads();
    if (threadIdx.x < mc) rows[threadIdx.x] = x + (size_t)(m0 + threadIdx.x) * H;
    __syncthreads();
    stage_rows(xs, rows, mc, H, true, norm_w, eps, rinv_s);
    __syncthreads();
    for (int m = 0; m < mc; ++m) {
      float acc[R] = {0.f, 0.f};
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        const int c = gl + LPR * j;
        float part[R] = {0.f, 0.f};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float4 x0 = xq[(m * 8 + 2 * u) * nch + c];
          const float4 x1 = xq[(m * 8 + 2 * u + 1) * nch + c];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const uint4 q = w[r][j][u];
            float p = part[r];
            p = fmaf(bf_lo(q.x), x0.x, p); p = fmaf(bf_hi(q.x), x0.y, p);
            p = fmaf(bf_lo(q.y), x0.z, p); p = fmaf(bf_hi(q.y), x0.w, p);
            p = fmaf(bf_lo(q.z), x1.x, p); p = fmaf(bf_hi(q.z), x1.y, p);
            p = fmaf(bf_lo(q.w), x1.z, p); p = fmaf(bf_hi(q.w), x1.w, p);
            part[r] = p;
          }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) acc[r] += part[r];
      }
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float tot = group_sum<LPR>(acc[r]);
        if (v0 + r < V && gl == r) logits[(size_t)(m0 + m) * V + v0 + r] = tot;
      }
    }
  }
}

__global__ void __launch_bounds__(1024) k_argmax(const float* logits, int V, int32_t* next, int32_t* len,
                                                 const int32_t* slots, int advance) {
  __shared__ float sv[32];
  __shared__ int si[32];
  const int b = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const float* lg = logits + (size_t)b * V;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int v = t; v < V; v += blockDim.x) {
    const float x = lg[v];
    if (x > bv) { bv = x; bi = v; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
  }
  if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
  __syncthreads();
  if (warp == 0) {
    bv = lane < (int)(blockDim.x >> 5) ? sv[lane] : -INFINITY;
    bi = lane < (int)(blockDim.x >> 5) ? si[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) {
      next[b] = bi == 0x7fffffff ? 0 : bi;
      if (advance) len[slots[b]] += 1;
    }
  }
}

__global__ void k_advance(int32_t* len, const int32_t* slots, int B, int by) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) len[slots[b]] += by;
}

// One thread per (row, group of g).
__global__ void k_quantize(const float* W, int N, int K, int g, uint8_t* packed, __half* scales) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int ng = K / g;
  if (gid >= (int64_t)N * ng) return;
  const int64_t n = gid / ng;
  const int j = (int)(gid - n * ng);
  const float* w = W + n * K + (int64_t)j * g;
  float amax = 0.f;
  for (int i = 0; i < g; ++i) amax = fmaxf(amax, fabsf(w[i]));
  const __half s = __float2half_rn(amax / 7.0f);
  const float sf = __half2float(s);
  scales[gid] = s;
  uint8_t* out = packed + n * (K / 2) + (int64_t)j * (g / 2);
  for (int i = 0; i < g; i += 2) {
    int u[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float r = sf > 0.f ? w[i + h] / sf : 0.f;
      if (!isfinite(r)) r = 0.f;
      const float q = fminf(fmaxf(rintf(r), -8.f), 7.f);
      u[h] = (int)q + 8;
    }
    out[i / 2] = (uint8_t)(u[0] | (u[1] << 4));
  }
}

template <int LPR, int CPL>
cudaError_t run_lm(const bf16* W, int V, int H, const bf16* x, const bf16* nw, float eps, float* logits, int B,
                   cudaStream_t st) {
  constexpr int rows = kSimtWarps * (kWarp / LPR) * 2;
  const int grid = (V + rows - 1) / rows;
  const size_t smem = (size_t)min(B, kMaxTile) * H * sizeof(float);
  k_lm_head<LPR, CPL><<<grid, kSimtThreads, smem, st>>>(W, V, H, x, nw, eps, logits, B);
  return cudaGetLastError();
}

#define BM_LM_SHAPES(X) X(32, 1) X(32, 2) X(32, 4) X(16, 1) X(8, 1)

}  // namespace

cudaError_t launch_embed(const bf16* table, int V, int H, const int32_t* tokens, bf16* x, int B, DevCheck chk,
                         cudaStream_t st) {
  k_embed<<<B, 256, 0, st>>>(table, V, H, tokens, x, chk);
  return cudaGetLastError();
}

cudaError_t launch_embed_norm(const bf16* table, int V, int H, const int32_t* tokens, bf16* x, const bf16* nw,
                              float eps, __half* xn, int B, DevCheck chk, cudaStream_t st, bool pdl) {
  return launch_k(pdl, k_embed_norm, dim3(B), dim3(256), 0, st, table, V, H, tokens, x, nw, eps, xn, chk);
}

cudaError_t launch_lm_head(const bf16* W, int V, int H, const bf16* x, const bf16* norm_w, float eps,
                           float* logits, int B, cudaStream_t st) {
  const int nch = H / 32;
#define BM_CASE(L, C) if (nch == (L) * (C)) return run_lm<L, C>(W, V, H, x, norm_w, eps, logits, B, st);
  BM_LM_SHAPES(BM_CASE)
#undef BM_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_argmax(const float* logits, int V, int B, int32_t* next, int32_t* len, const int32_t* slots,
                          int advance, cudaStream_t st) {
  k_argmax<<<B, 1024, 0, st>>>(logits, V, next, len, slots, advance);
  return cudaGetLastError();
}

cudaError_t launch_advance(int32_t* len, const int32_t* slots, int B, cudaStream_t st, int by) {
  k_advance<<<(B + 127) / 128, 128, 0, st>>>(len, slots, B, by);
  return cudaGetLastError();
}

cudaError_t launch_quantize(const float* W, int N, int K, int g, uint8_t* packed, __half* scales,
                            cudaStream_t st) {
  const int64_t groups = (int64_t)N * (K / g);
  const int64_t blocks = (groups + 255) / 256;
  k_quantize<<<(unsigned)blocks, 256, 0, st>>>(W, N, K, g, packed, scales);
  return cudaGetLastError();
}

cudaError_t init_misc_attributes() {
  cudaError_t e = cudaSuccess;
#define BM_CASE(L, C)                                                                        \
  if (e == cudaSuccess)                                                                      \
    e = cudaFuncSetAttribute(k_lm_head<L, C>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             kMaxTile * L * C * 32 * (int)sizeof(float));
  BM_LM_SHAPES(BM_CASE)
#undef BM_CASE
  return e;
}

}  // namespace bm
