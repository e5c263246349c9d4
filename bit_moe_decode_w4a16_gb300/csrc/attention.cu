// Slot-indexed decode attention over the fixed KV arena.
//
// The arena is [layer][slot][kv head][position][d] bf16 for K and for V; a
// stream's K/V live in its stable slot and nothing here reads or writes any
// other slot (the KV-slot isolation page, §1: the batched arena is indexed by
// a stable per-stream slot and never wiped on a batch-composition change).
//
//   k_rope_append  RoPE (rotate-half) of q and k at pos = len[slot]; q to a
//                  query buffer, k and v to the arena at pos
//   k_kv_append    the same append for k, v that are already rotated
//   k_attn_part    split-K: one CTA per (128-position chunk, kv head, stream)
//                  computes, for the q heads of that kv head, the chunk's
//                  running max, exp-sum and unnormalised p·V
//   k_attn_combine merges a stream's chunks in ascending order
// The chunk grid depends only on a stream's own length, so its output does
// not depend on the other streams of the batch.
#include <float.h>

#include "kernels.cuh"

namespace bm {

namespace {

constexpr int kMaxGroup = 8;   // q heads per kv head handled by one CTA

__global__ void k_rope_append(AttnArena ar, int layer, const int32_t* slots, const bf16* qkv, int ld_qkv,
                              int qh, const float2* rope, bf16* qout, DevCheck chk) {
  extern __shared__ float cs[];   // [d/2] cos, [d/2] sin
  pdl_wait();
  const int b = blockIdx.x;
  const int slot = slots[b];
  if (slot < 0 || slot >= ar.S) { if (threadIdx.x == 0) chk.fail(1); return; }
  const int pos = ar.len[slot];
  if (pos < 0 || pos >= ar.cap) { if (threadIdx.x == 0) chk.fail(2); return; }
  const int d = ar.d, half = d / 2;
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const float2 v = rope[(size_t)pos * half + i];
    cs[i] = v.x;
    cs[half + i] = v.y;
  }
  __syncthreads();
  const bf16* row = qkv + (size_t)b * ld_qkv;
  const int heads = qh + ar.kvh;
  for (int idx = threadIdx.x; idx < heads * half; idx += blockDim.x) {
    const int h = idx / half, i = idx - h * half;
    const bf16* src = row + (size_t)h * d;
    const float x0 = bf2f(src[i]), x1 = bf2f(src[i + half]);
    const float c = cs[i], s = cs[half + i];
    const bf16 y0 = f2bf(x0 * c - x1 * s);
    const bf16 y1 = f2bf(x1 * c + x0 * s);
    if (h < qh) {
      bf16* dst = qout + ((size_t)b * qh + h) * d;
      dst[i] = y0;
      dst[i + half] = y1;
    } else {
      const int kh = h - qh;
      bf16* dst = ar.K + layer * ar.layer_stride() + slot * ar.slot_stride() + ((size_t)kh * ar.cap + pos) * d;
      dst[i] = y0;
      dst[i + half] = y1;
    }
  }
  const bf16* vsrc = row + (size_t)(qh + ar.kvh) * d;
  for (int idx = threadIdx.x; idx < ar.kvh * d; idx += blockDim.x) {
    const int kh = idx / d, i = idx - kh * d;
    ar.V[layer * ar.layer_stride() + slot * ar.slot_stride() + ((size_t)kh * ar.cap + pos) * d + i] = vsrc[idx];
  }
}

__global__ void k_kv_append(AttnArena ar, int layer, const int32_t* slots, const bf16* k, const bf16* v,
                            DevCheck chk) {
  const int b = blockIdx.x;
  const int slot = slots[b];
  if (slot < 0 || slot >= ar.S) { if (threadIdx.x == 0) chk.fail(1); return; }
  const int pos = ar.len[slot];
  if (pos < 0 || pos >= ar.cap) { if (threadIdx.x == 0) chk.fail(2); return; }
  for (int idx = threadIdx.x; idx < ar.kvh * ar.d; idx += blockDim.x) {
    const int kh = idx / ar.d, i = idx - kh * ar.d;
    const size_t o = layer * ar.layer_stride() + slot * ar.slot_stride() + ((size_t)kh * ar.cap + pos) * ar.d + i;
    ar.K[o] = k[(size_t)b * ar.kvh * ar.d + idx];
    ar.V[o] = v[(size_t)b * ar.kvh * ar.d + idx];
  }
}

// Partials layout: [B][qh][max_chunks] records of (d floats o, m, l).
__device__ __forceinline__ size_t part_index(int b, int h, int c, int qh, int max_chunks, int d) {
  return (((size_t)b * qh + h) * max_chunks + c) * (size_t)(d + 2);
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// blockDim.x == kAttnChunk == 128 threads; D = head_dim (64 or 128).  Grid
// (kv head, stream, chunk): the chunks past a stream's length exit at once
// and sit at the end of the launch order.
// The chunk's V rows are copied to shared memory asynchronously while the
// scores are computed.  Scores: thread t takes position j0 + t, its whole K
// row loaded up front.  p.V: thread t takes dimension t of every q head of
// the group, positions in ascending order.
template <int D>
__global__ void __launch_bounds__(kAttnChunk) k_attn_part(AttnArena ar, int layer, const int32_t* slots,
                                                          const bf16* q, int qh, float* part, int max_chunks,
                                                          DevCheck chk) {
  __shared__ float qs[kMaxGroup][D];
  __shared__ float ps[kMaxGroup][kAttnChunk];
  __shared__ float red[kMaxGroup][kAttnChunk / 32];
  __shared__ float stat[kMaxGroup][2];
  __shared__ __align__(16) bf16 vs[kAttnChunk][D];
  pdl_wait();
  const int kh = blockIdx.x, b = blockIdx.y, c = blockIdx.z;
  const int slot = slots[b];
  if (slot < 0 || slot >= ar.S) { if (c == 0 && kh == 0 && threadIdx.x == 0) chk.fail(1); return; }
  const int L = ar.len[slot] + 1;   // committed prefix + this step's position
  if (L < 1 || L > ar.cap) { if (c == 0 && kh == 0 && threadIdx.x == 0) chk.fail(2); return; }
  const int j0 = c * kAttnChunk;
  if (j0 >= L) return;
  const int n = min(kAttnChunk, L - j0);
  const int G = qh / ar.kvh, t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const float scale = 1.0f / sqrtf((float)D);
  const size_t base = layer * ar.layer_stride() + slot * ar.slot_stride() + (size_t)kh * ar.cap * D;
  const bf16* Kb = ar.K + base;
  const bf16* Vb = ar.V + base;
  constexpr int kVecs = D / 8;
  for (int i = t; i < n * kVecs; i += kAttnChunk) {
    const int r = i / kVecs, v8 = i - r * kVecs;
    cp_async16(&vs[r][v8 * 8], Vb + (size_t)(j0 + r) * D + v8 * 8);
  }
  cp_async_commit();
  for (int idx = t; idx < G * D; idx += blockDim.x) {
    const int g = idx / D, i = idx - g * D;
    qs[g][i] = bf2f(q[((size_t)b * qh + kh * G + g) * D + i]);
  }
  const int j = j0 + t;
  uint4 kr[kVecs];
  if (j < L) {
    const uint4* src = reinterpret_cast<const uint4*>(Kb + (size_t)j * D);
#pragma unroll
    for (int i = 0; i < kVecs; ++i) kr[i] = src[i];
  }
  __syncthreads();
  float sc[kMaxGroup];
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) sc[g] = 0.f;
  if (j < L) {
#pragma unroll
    for (int i = 0; i < kVecs; ++i) {
      const float k0 = bf_lo(kr[i].x), k1 = bf_hi(kr[i].x), k2 = bf_lo(kr[i].y), k3 = bf_hi(kr[i].y);
      const float k4 = bf_lo(kr[i].z), k5 = bf_hi(kr[i].z), k6 = bf_lo(kr[i].w), k7 = bf_hi(kr[i].w);
#pragma unroll
      for (int g = 0; g < kMaxGroup; ++g) {
        if (g < G) {
          const float* qq = &qs[g][i * 8];
          float acc = sc[g];
          acc = fmaf(qq[0], k0, acc); acc = fmaf(qq[1], k1, acc); acc = fmaf(qq[2], k2, acc);
          acc = fmaf(qq[3], k3, acc); acc = fmaf(qq[4], k4, acc); acc = fmaf(qq[5], k5, acc);
          acc = fmaf(qq[6], k6, acc); acc = fmaf(qq[7], k7, acc);
          sc[g] = acc;
        }
      }
    }
  }
  // chunk max per head
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    if (g >= G) break;
    const float s = (j < L) ? sc[g] * scale : -FLT_MAX;
    sc[g] = s;
    const float m = warp_max(s);
    if (lane == 0) red[g][warp] = m;
  }
  __syncthreads();
  if (t < G) {
    float m = red[t][0];
    for (int w = 1; w < kAttnChunk / 32; ++w) m = fmaxf(m, red[t][w]);
    stat[t][0] = m;
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    if (g >= G) break;
    const float p = (j < L) ? expf(sc[g] - stat[g][0]) : 0.f;
    ps[g][t] = p;
    const float sum = warp_sum(p);
    if (lane == 0) red[g][warp] = sum;
  }
  cp_async_wait_all();
  __syncthreads();
  if (t < G) {
    float l = 0.f;
    for (int w = 0; w < kAttnChunk / 32; ++w) l += red[t][w];
    stat[t][1] = l;
  }
  __syncthreads();
  if (t < D) {
    float o[kMaxGroup];
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g) o[g] = 0.f;
    for (int jj = 0; jj < n; ++jj) {
      const float vv = bf2f(vs[jj][t]);
#pragma unroll
      for (int g = 0; g < kMaxGroup; ++g)
        if (g < G) o[g] = fmaf(ps[g][jj], vv, o[g]);
    }
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g) {
      if (g >= G) break;
      float* rec = part + part_index(b, kh * G + g, c, qh, max_chunks, D);
      rec[t] = o[g];
      if (t == 0) {
        rec[D] = stat[g][0];
        rec[D + 1] = stat[g][1];
      }
    }
  }
}

// One CTA per (q head, stream): the chunks' (m, l) go to shared memory in
// parallel, then thread t merges dimension t over the chunks in ascending
// order with eight chunks' loads in flight at a time.
constexpr int kMaxChunksSmem = 1024;

__global__ void k_attn_combine(AttnArena ar, const int32_t* slots, const float* part, int qh, int max_chunks,
                               void* out, int out_f16) {
  __shared__ float ml_s[kMaxChunksSmem][2];
  __shared__ float M_s;
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y, t = threadIdx.x, d = ar.d;
  const int slot = slots[b];
  if (slot < 0 || slot >= ar.S) return;
  const int L = ar.len[slot] + 1;
  if (L < 1 || L > ar.cap) return;
  const int nc = (L + kAttnChunk - 1) / kAttnChunk;
  for (int c = t; c < nc; c += blockDim.x) {
    const float* rec = part + part_index(b, h, c, qh, max_chunks, d);
    ml_s[c][0] = rec[d];
    ml_s[c][1] = rec[d + 1];
  }
  __syncthreads();
  if (t == 0) {
    float M = -FLT_MAX;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, ml_s[c][0]);
    M_s = M;
  }
  __syncthreads();
  const float M = M_s;
  float den = 0.f, acc = 0.f;
  for (int c0 = 0; c0 < nc; c0 += 8) {
    float o[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      o[u] = (t < d && c0 + u < nc) ? part[part_index(b, h, c0 + u, qh, max_chunks, d) + t] : 0.f;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (c0 + u < nc) {
        const float w = expf(ml_s[c0 + u][0] - M);
        den = fmaf(ml_s[c0 + u][1], w, den);
        acc = fmaf(o[u], w, acc);
      }
    }
  }
  if (t < d) {
    const size_t o = ((size_t)b * qh + h) * d + t;
    if (out_f16) static_cast<__half*>(out)[o] = __float2half_rn(round_bf16(acc / den));
    else static_cast<bf16*>(out)[o] = f2bf(acc / den);
  }
}

__global__ void k_set_len(int32_t* len, int slot, int value) { len[slot] = value; }

}  // namespace

size_t attn_partial_floats(int B, int qh, int cap, int d) {
  const int max_chunks = (cap + kAttnChunk - 1) / kAttnChunk;
  return (size_t)B * qh * max_chunks * (d + 2);
}

cudaError_t launch_rope_append(const AttnArena& ar, int layer, const int32_t* slots, const bf16* qkv, int ld_qkv,
                               int qh, const float2* rope, bf16* qout, int B, DevCheck chk, cudaStream_t st,
                               bool pdl) {
  return launch_k(pdl, k_rope_append, dim3(B), dim3(256), sizeof(float) * ar.d, st, ar, layer, slots, qkv, ld_qkv, qh,
                  rope, qout, chk);
}

cudaError_t launch_kv_append(const AttnArena& ar, int layer, const int32_t* slots, const bf16* k, const bf16* v,
                             int B, DevCheck chk, cudaStream_t st) {
  k_kv_append<<<B, 256, 0, st>>>(ar, layer, slots, k, v, chk);
  return cudaGetLastError();
}

cudaError_t launch_attention(const AttnArena& ar, int layer, const int32_t* slots, const bf16* q, void* out,
                             int qh, int B, float* partials, DevCheck chk, cudaStream_t st, int* launches,
                             const Marker& mark, int out_f16, bool pdl) {
  if (ar.d > 128 || ar.d % 8 != 0 || qh % ar.kvh != 0 || qh / ar.kvh > kMaxGroup) return cudaErrorInvalidValue;
  const int max_chunks = (ar.cap + kAttnChunk - 1) / kAttnChunk;
  if (max_chunks > kMaxChunksSmem) return cudaErrorInvalidValue;
  dim3 g1(ar.kvh, B, max_chunks);
  cudaError_t e;
  if (ar.d == 128)
    e = launch_k(pdl, k_attn_part<128>, g1, dim3(kAttnChunk), 0, st, ar, layer, slots, q, qh, partials, max_chunks, chk);
  else if (ar.d == 64)
    e = launch_k(pdl, k_attn_part<64>, g1, dim3(kAttnChunk), 0, st, ar, layer, slots, q, qh, partials, max_chunks, chk);
  else
    return cudaErrorInvalidValue;
  if (e != cudaSuccess) return e;
  mark(KT_ATTN_PART);
  dim3 g2(qh, B);
  if ((e = launch_k(pdl, k_attn_combine, g2, dim3(128), 0, st, ar, slots, (const float*)partials, qh, max_chunks, out,
                    out_f16)) != cudaSuccess)
    return e;
  mark(KT_ATTN_COMBINE);
  if (launches) *launches += 2;
  return cudaSuccess;
}

cudaError_t launch_set_len(int32_t* len, int slot, int value, cudaStream_t st) {
  k_set_len<<<1, 1, 0, st>>>(len, slot, value);
  return cudaGetLastError();
}

}  // namespace bm
