// Device code of the decode routing (router logits with the RMSNorm fused,
// softmax top-k), shared by the routing kernels (moe.cu) and by the
// persistent decode step: both run the same instructions, so they leave the
// same bits.
#pragma once

#include <float.h>

#include "kernels.cuh"

namespace bm {
namespace routedev {

constexpr int kRouterWarps = 8;

// Router logits.  Grid (ceil(E / kRouterExperts), B): a CTA takes one token
// and kRouterExperts experts, two per warp.  Each warp issues the loads of
// its first router row before anything else (the router weights do not
// depend on the previous kernel, so they go out before the dependency wait),
// then the CTA normalises the token's row itself (every CTA of the token
// computes the same bf16 values in the same order; the CTAs of expert block 0
// also write them out for the expert GEMMs) and keeps it in shared memory as
// fp32.  A warp's dot product takes the row in 128-float strips, lane l
// holding elements 4l..4l+3 of each strip, in a fixed order.
constexpr int kRouterExperts = 2 * kRouterWarps;
constexpr int kRouterStrips = 16;   // 16 x 128 = 2048 floats of a router row per pass

__device__ __forceinline__ void router_load(const float* wr, int H, int k0, float4 (&w4)[kRouterStrips]) {
#pragma unroll
  for (int i = 0; i < kRouterStrips; ++i)
    if (k0 + 128 * i < H) w4[i] = __ldg(reinterpret_cast<const float4*>(wr + k0 + 128 * i));
}

__device__ __forceinline__ float router_fma(const float* xs, int H, int k0, const float4 (&w4)[kRouterStrips],
                                            float acc) {
#pragma unroll
  for (int i = 0; i < kRouterStrips; ++i) {
    const int k = k0 + 128 * i;
    if (k < H) {
      const float4 x = *reinterpret_cast<const float4*>(xs + k);
      acc = fmaf(x.x, w4[i].x, acc); acc = fmaf(x.y, w4[i].y, acc);
      acc = fmaf(x.z, w4[i].z, acc); acc = fmaf(x.w, w4[i].w, acc);
    }
  }
  return acc;
}

// The router logits of one token and kRouterExperts experts (one CTA); the
// dependency wait of a programmatic launch is taken inside, after the
// weight prefetch.
// EPC = experts per CTA: 16 (two per warp) or 8 (one per warp, for small
// batches: twice the CTAs and no second router row on the dependency chain).
// A logit's arithmetic does not depend on EPC.
// The logits of token `tkn` and experts [EPC eb, EPC (eb + 1)), by threads
// 0..255 of the caller (synchronised by `sync`); `red` holds kRouterWarps
// floats of shared memory.
// `trigger`: the launch is one wave, so its dependents may launch once this
// CTA has taken its dependency wait.
template <int EPC, class Sync>
__device__ __forceinline__ void router_cta(const MoeArgs& a, const MoeBufs& b, float* xs, float* red, int eb, int tkn,
                                           Sync sync, bool trigger = false) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = a.H;
  float4 w4[kRouterStrips];
  const int e_first = eb * EPC + warp;
  if (e_first < a.E) router_load(a.wr + (size_t)e_first * H, H, lane * 4, w4);
  pdl_wait();
  if (trigger) pdl_trigger();
  const bf16* x = a.x + (size_t)tkn * H;
  float ss = 0.f;
  for (int k = threadIdx.x * 8; k < H; k += 256 * 8) {
    const uint4 p = *reinterpret_cast<const uint4*>(x + k);
    const uint32_t w[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float v0 = bf_lo(w[q]), v1 = bf_hi(w[q]);
      xs[k + 2 * q] = v0;
      xs[k + 2 * q + 1] = v1;
      ss = fmaf(v0, v0, ss);
      ss = fmaf(v1, v1, ss);
    }
  }
  if (a.do_norm) {
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    sync();
    float tot = 0.f;
    for (int w = 0; w < kRouterWarps; ++w) tot += red[w];
    const float r = 1.0f / sqrtf(tot / (float)H + a.eps);
    // the thread's own 8 elements: one 16-byte load of the norm weights and
    // one 16-byte store of the normed values
    for (int k = threadIdx.x * 8; k < H; k += 256 * 8) {
      uint4 nwv = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);   // bf16 ones
      if (a.norm_w) nwv = *reinterpret_cast<const uint4*>(a.norm_w + k);
      const uint32_t nw[4] = {nwv.x, nwv.y, nwv.z, nwv.w};
      uint32_t hw[4], bw[4];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float w = (q & 1) ? bf_hi(nw[q >> 1]) : bf_lo(nw[q >> 1]);
        const bf16 v = f2bf(xs[k + q] * r * w);
        xs[k + q] = bf2f(v);
        const uint32_t hb = (uint32_t)__half_as_ushort(__float2half_rn(bf2f(v)));
        const uint32_t bb = (uint32_t)__bfloat16_as_ushort(v);
        hw[q >> 1] = (q & 1) ? (hw[q >> 1] | (hb << 16)) : hb;
        bw[q >> 1] = (q & 1) ? (bw[q >> 1] | (bb << 16)) : bb;
      }
      if (eb == 0) {
        const uint4 out = a.xn_f16 ? make_uint4(hw[0], hw[1], hw[2], hw[3]) : make_uint4(bw[0], bw[1], bw[2], bw[3]);
        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(b.xn) + (size_t)tkn * H + k) = out;
      }
    }
  }
  sync();
  for (int ei = warp; ei < EPC; ei += kRouterWarps) {
    const int e = eb * EPC + ei;
    if (e >= a.E) break;
    const float* wr = a.wr + (size_t)e * H;
    float acc = 0.f;
    for (int k0 = lane * 4; k0 < H; k0 += kRouterStrips * 128) {
      if (ei != warp || k0 != lane * 4) router_load(wr, H, k0, w4);
      acc = router_fma(xs, H, k0, w4, acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) b.logits[(size_t)tkn * a.E + e] = acc;
  }
}

// Softmax top-k of token t by one warp (ties: lower expert id; a NaN logit
// ranks as -inf, and every token still gets k distinct valid ids); writes
// topk_ids / topk_w of the token and, if ids_out, the ids there too.  With
// `cg` the logits are read through L2 (they were written by other CTAs of the
// same launch).
// topk_core: the same for the logits row `lg` of one token, writing its k
// ids and weights to ids[0..k) and w[0..k) (shared or global memory), and the
// ids to ids2 too if it is not null.
__device__ __forceinline__ void topk_core(const float* lg, int E, int k, int renorm, bool cg, int* ids, float* wts,
                                          int* ids2) {
  const int lane = threadIdx.x & 31;
  float v[8];
  bool taken[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    const float x = e < E ? (cg ? __ldcg(lg + e) : lg[e]) : -INFINITY;
    v[i] = isnan(x) ? -INFINITY : x;
    taken[i] = e >= E;
  }
  float lmax = -INFINITY;
#pragma unroll
  for (int i = 0; i < 8; ++i) lmax = fmaxf(lmax, v[i]);
  lmax = warp_max(lmax);
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) z += taken[i] ? 0.f : expf(v[i] - lmax);
  z = warp_sum(z);
  float sel_v[16];
  int sel_e[16];
  for (int r = 0; r < k; ++r) {
    // the lane's best untaken (value, lowest id), then the warp's: the
    // largest order key of the value, and among the lanes holding it the
    // lowest id (-0 and +0 share a key, so they tie, as under ==)
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      if (!taken[i] && (v[i] > bv || (v[i] == bv && e < be))) { bv = v[i]; be = e; }
    }
    const uint32_t u = __float_as_uint(bv == 0.f ? 0.f : bv);
    const uint32_t key = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
    be = (int)__reduce_min_sync(0xffffffffu, key == kmax ? (uint32_t)be : 0x7fffffffu);
    bv = __shfl_sync(0xffffffffu, bv, be & 31);
    sel_v[r] = bv;
    sel_e[r] = be;   // k <= E, so an untaken id always exists
    if ((be & 31) == lane) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (i == (be >> 5)) taken[i] = true;
    }
  }
  if (lane == 0) {
    float ex[16], sum = 0.f;
    for (int r = 0; r < k; ++r) { ex[r] = expf(sel_v[r] - lmax); sum += ex[r]; }
    const float den = renorm ? sum : z;
    for (int r = 0; r < k; ++r) {
      ids[r] = sel_e[r];
      wts[r] = ex[r] / den;
      if (ids2) ids2[r] = sel_e[r];
    }
  }
}

__device__ __forceinline__ void topk_warp(const MoeArgs& a, const MoeBufs& b, int t, bool cg, int* ids_out) {
  topk_core(b.logits + (size_t)t * a.E, a.E, a.k, a.renorm, cg, b.topk_ids + t * a.k, b.topk_w + t * a.k,
            ids_out ? ids_out + t * a.k : nullptr);
}

struct CtaSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

}  // namespace routedev
}  // namespace bm
