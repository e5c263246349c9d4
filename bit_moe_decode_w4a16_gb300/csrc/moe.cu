// Grouped int4 expert op of B tokens (the batched-serving page, §1: the
// experts chosen for all B streams run as one grouped operation over the
// expert bank that stays resident on the device).
//
//   1. k_router      fp32 router logits of every token (RMSNorm fused; CTA 0
//                    also writes the normed input for the experts)
//   2. k_topk_sort   softmax top-k per token (ties: lower expert id), weights,
//                    then a stable counting sort of the B*k (token, rank)
//                    pairs by expert and the list of active experts
//   3. k_gateup      per active expert and tile of F: SiLU(x W_g) * (x W_u)
//                    for all of its tokens; each packed byte read once
//   4. k_down        per active expert and tile of H: the down projection of
//                    its tokens, fp32 out
//   5. k_combine     y_b = res_b + sum_r w_{b,r} out_{b,r}, rank order
//
// Sorting by expert reads every active expert's weights once however many
// streams picked it, which is what the pages' de-dup pass tried to achieve;
// no separate compaction step exists.  Every reduction has a fixed order and
// no floating-point atomics are used, so a token's result does not depend on
// which other tokens share the launch.
#include <float.h>

#include <algorithm>

#include "kernels.cuh"
#include "route_dev.cuh"
#include "w4_simt.cuh"

namespace bm {

namespace {

constexpr int kMaxPairs = 1024;   // B * k handled by the single-CTA sort

using namespace routedev;

__global__ void __launch_bounds__(256) k_router(MoeArgs a, MoeBufs b) {
  extern __shared__ __align__(16) float xs[];   // [H] normalised row
  __shared__ float red[kRouterWarps];
  router_cta<kRouterExperts>(a, b, xs, red, blockIdx.x, blockIdx.y, CtaSync{});
}

// Stable counting sort of the P = B k (token, rank) pairs by expert, the
// list of active experts and the job list, by the whole CTA from ids_s
// (shared memory, pair p = b k + r).  Warp 0 walks the pairs 32 at a time in
// order: lanes holding the same expert find each other (match), a pair's
// rank among its expert's pairs is the expert's running count plus the
// same-expert lanes below it, and the group's lowest lane adds the group to
// the running count.  Then exclusive scans over the experts give the
// offsets.  Every result is a count, so it does not depend on timing.
__device__ __forceinline__ void group_pairs(const MoeArgs& a, const MoeBufs& b, const int* ids_s, int* cnt_s,
                                            int* off_s, int* rank_s) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, k = a.k, P = a.B * a.k;
  for (int e = threadIdx.x; e < E; e += blockDim.x) cnt_s[e] = 0;
  __syncthreads();
  if (warp == 0) {
    const unsigned lt = (1u << lane) - 1u;
    for (int p0 = 0; p0 < P; p0 += 32) {
      const int p = p0 + lane;
      const int e = p < P ? ids_s[p] : -1 - lane;   // past the end: a value no other lane holds
      const unsigned same = __match_any_sync(0xffffffffu, e);
      const int before = p < P ? cnt_s[e] : 0;
      __syncwarp();   // every lane has read its expert's count before any is updated
      if (p < P) {
        rank_s[p] = before + __popc(same & lt);
        if ((same & lt) == 0u) cnt_s[e] = before + __popc(same);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // warp 0: exclusive scans over the experts (ascending id) of the pair
  // counts, the active flags and the job counts, 32 experts at a time
  if (warp == 0) {
    int run_off = 0, run_u = 0, run_j = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? cnt_s[e] : 0, act = c > 0, nj = (c + kJobTokens - 1) / kJobTokens;
      // one inclusive scan of the three counts packed in a word: over 32
      // experts the pair count stays below 2^11, the active count below
      // 2^6 and the job count below 2^8, so the fields never carry
      uint32_t packed = (uint32_t)c | ((uint32_t)act << 11) | ((uint32_t)nj << 17);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t p2 = __shfl_up_sync(0xffffffffu, packed, o);
        if (lane >= o) packed += p2;
      }
      const int ic = (int)(packed & 0x7FFu), ia = (int)((packed >> 11) & 0x3Fu), ij = (int)(packed >> 17);
      if (e < E) {
        const int off = run_off + ic - c, u = run_u + ia - act, j0 = run_j + ij - nj;
        off_s[e] = off;
        if (act) {
          b.active_e[u] = e;
          b.active_off[u] = off;
          // one self-contained word per job: expert | first pair << 9 | tokens << 21
          for (int g = 0; g < nj; ++g) {
            const int n = min(kJobTokens, c - g * kJobTokens);
            b.jobs[j0 + g] = e | ((off + g * kJobTokens) << 9) | (n << 21);
          }
        }
      }
      run_off += __shfl_sync(0xffffffffu, ic, 31);
      run_u += __shfl_sync(0xffffffffu, ia, 31);
      run_j += __shfl_sync(0xffffffffu, ij, 31);
    }
    if (lane == 0) {
      off_s[E] = run_off;
      b.active_off[run_u] = run_off;
      *b.n_active = run_u;
      *b.n_jobs = run_j;
      if (a.u_log) *a.u_log = run_u;
    }
  }
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int pos = off_s[ids_s[p]] + rank_s[p];
    b.pair_token[pos] = p / k;
    b.pos_of[p] = pos;
  }
}

__global__ void __launch_bounds__(1024) k_topk_sort(MoeArgs a, MoeBufs b) {
  __shared__ int ids_s[kMaxPairs];
  __shared__ int rank_s[kMaxPairs];
  __shared__ int cnt_s[256];
  __shared__ int off_s[257];
  const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int t = warp; t < a.B; t += nwarps) topk_warp(a, b, t, false, ids_s);
  __syncthreads();
  group_pairs(a, b, ids_s, cnt_s, off_s, rank_s);
}

// Router, top-k and grouping in one launch.  Every CTA computes its
// experts' logits for one token; the CTA that finishes a token last (per-token
// arrival counter) runs the token's top-k; the CTA that finishes the last
// token (a second counter) sorts the pairs and writes the job list.  Stores
// are made visible with __threadfence before each arrival, and the late
// readers load through L2.  The counters are zero before the launch and are
// left zero.  The result is the same as k_router + k_topk_sort.
template <int EPC>
__global__ void __launch_bounds__(256) k_route_fused(MoeArgs a, MoeBufs b, unsigned int* tok_cnt,
                                                     unsigned int* all_cnt, int trigger) {
  extern __shared__ __align__(16) float xs[];   // [H] normalised row
  __shared__ int ids_s[kMaxPairs];
  __shared__ int rank_s[kMaxPairs];
  __shared__ int cnt_s[256];
  __shared__ int off_s[257];
  __shared__ int flag_s;
  __shared__ float red[kRouterWarps];
  const int tkn = blockIdx.y, warp = threadIdx.x >> 5;
  // takes the dependency wait after its weight prefetch (and triggers the
  // expert launch, whose CTAs then set up as this launch's SMs free up)
  router_cta<EPC>(a, b, xs, red, blockIdx.x, tkn, CtaSync{}, trigger != 0);
  // Arrivals are one thread's: after the CTA barrier that orders the other
  // threads' stores, thread 0 fences and counts, and the last arrival fences
  // again before the barrier that releases the reads of the others' results.
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const bool last = atomicAdd(&tok_cnt[tkn], 1u) == gridDim.x - 1;
    if (last) __threadfence();
    flag_s = last;
  }
  __syncthreads();
  if (!flag_s) return;
  if (warp == 0) topk_warp(a, b, tkn, true, nullptr);   // its results are thread 0's stores
  __syncthreads();   // every thread has read flag_s
  if (threadIdx.x == 0) {
    tok_cnt[tkn] = 0u;
    __threadfence();
    const bool last = atomicAdd(all_cnt, 1u) == gridDim.y - 1;
    if (last) __threadfence();
    flag_s = last;
  }
  __syncthreads();
  if (!flag_s) return;
  const int P = a.B * a.k;
  for (int p = threadIdx.x; p < P; p += blockDim.x) ids_s[p] = __ldcg(b.topk_ids + p);
  __syncthreads();
  group_pairs(a, b, ids_s, cnt_s, off_s, rank_s);
  if (threadIdx.x == 0) *all_cnt = 0u;
}

// ---- routing of a prompt block (hundreds of rows, up to kMaxPairsWide
// pairs): k_router, then one warp per row for its top-k, then one CTA groups
// the pairs by expert.  The same top-k as the decode step; the grouping
// computes the same offsets, ranks and active list with plain scans (no job
// list: the prompt-length expert GEMMs take an expert's rows directly).
constexpr int kMaxPairsWide = 4096;

__global__ void __launch_bounds__(256) k_topk_rows(MoeArgs a, MoeBufs b) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t < a.B) topk_warp(a, b, t, false, nullptr);
}

// The grouping of up to kMaxPairsWide pairs by 32 warps: warp w ranks the
// pairs of its block [w * per, (w + 1) * per) within their experts (32 at a
// time, as group_pairs), the blocks' counts are scanned per expert in warp
// order, then the experts' offsets in ascending id; the ranks are the stable
// ones of the serial grouping (pair order within an expert).
__global__ void __launch_bounds__(1024) k_group_wide(MoeArgs a, MoeBufs b) {
  __shared__ short rank_s[kMaxPairsWide];
  __shared__ unsigned char ids_s[kMaxPairsWide];
  __shared__ short cnt_w[32][256];   // per warp block and expert: pairs, then the exclusive base
  __shared__ int off_s[257];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = a.E, k = a.k, P = a.B * a.k;
  const int per = ((P + 31) / 32 + 31) & ~31;   // pairs per warp block, a multiple of 32
  for (int p = threadIdx.x; p < P; p += blockDim.x) ids_s[p] = (unsigned char)b.topk_ids[p];
  for (int i = threadIdx.x; i < 32 * 256; i += blockDim.x) (&cnt_w[0][0])[i] = 0;
  __syncthreads();
  {
    const unsigned lt = (1u << lane) - 1u;
    const int p_end = min(P, (warp + 1) * per);
    for (int p0 = warp * per; p0 < p_end; p0 += 32) {
      const int p = p0 + lane;
      const int e = p < p_end ? (int)ids_s[p] : -1 - lane;
      const unsigned same = __match_any_sync(0xffffffffu, e);
      const int before = p < p_end ? cnt_w[warp][e] : 0;
      __syncwarp();
      if (p < p_end) {
        rank_s[p] = (short)(before + __popc(same & lt));
        if ((same & lt) == 0u) cnt_w[warp][e] = (short)(before + __popc(same));
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // per expert: the blocks' counts -> exclusive bases in warp order, and the total
  if (threadIdx.x < E) {
    const int e = threadIdx.x;
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int c = cnt_w[w][e];
      cnt_w[w][e] = (short)run;
      run += c;
    }
    off_s[e] = run;   // the count, scanned below
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive scans over the experts of the counts, the active flags and
    // the prompt GEMM jobs (tiles of kPromptTileRows rows); each active
    // expert writes its jobs u | t << 16
    int run_off = 0, run_u = 0, run_j = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? off_s[e] : 0, act = c > 0, nj = (c + kPromptTileRows - 1) / kPromptTileRows;
      int ic = c, ia = act, ij = nj;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int c2 = __shfl_up_sync(0xffffffffu, ic, o), a2 = __shfl_up_sync(0xffffffffu, ia, o);
        const int j2 = __shfl_up_sync(0xffffffffu, ij, o);
        if (lane >= o) { ic += c2; ia += a2; ij += j2; }
      }
      __syncwarp();
      if (e < E) {
        const int off = run_off + ic - c, u = run_u + ia - act, j0 = run_j + ij - nj;
        off_s[e] = off;
        if (act) {
          b.active_e[u] = e;
          b.active_off[u] = off;
          for (int t = 0; t < nj; ++t) b.jobs[j0 + t] = u | (t << 16);
        }
      }
      run_off += __shfl_sync(0xffffffffu, ic, 31);
      run_u += __shfl_sync(0xffffffffu, ia, 31);
      run_j += __shfl_sync(0xffffffffu, ij, 31);
    }
    if (lane == 0) {
      off_s[E] = run_off;
      b.active_off[run_u] = run_off;
      *b.n_active = run_u;
      *b.n_jobs = run_j;
      if (a.u_log) *a.u_log = run_u;
    }
  }
  __syncthreads();
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int e = ids_s[p];
    const int pos = off_s[e] + cnt_w[p / per][e] + rank_s[p];
    b.pair_token[pos] = p / k;
    b.pos_of[p] = pos;
  }
}

// RMSNorm of prompt rows for the router and the experts, a CTA per row:
// router_cta's arithmetic (thread t sums the squares of elements 8t .. 8t + 7,
// each warp's butterfly, then the 8 warps in order; each element bf16(x rinv
// w)), so a prompt row's normed row is the bits a decode step gives it.
// Written to xn as fp16 (xn_f16) or bf16; either holds the bf16 values
// exactly.  H <= 2048, H % 8 == 0.
__global__ void __launch_bounds__(256) k_norm_rows(MoeArgs a, MoeBufs b) {
  __shared__ float red[kRouterWarps];
  const int t = blockIdx.x, H = a.H, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kk = threadIdx.x * 8;
  const bool has = kk < H;
  const uint4 pv = has ? *reinterpret_cast<const uint4*>(a.x + (size_t)t * H + kk) : make_uint4(0, 0, 0, 0);
  const uint32_t w[4] = {pv.x, pv.y, pv.z, pv.w};
  float ss = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float v0 = bf_lo(w[q]), v1 = bf_hi(w[q]);
    ss = fmaf(v0, v0, ss);
    ss = fmaf(v1, v1, ss);
  }
  ss = warp_sum(ss);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  float tot = 0.f;
  for (int i = 0; i < kRouterWarps; ++i) tot += red[i];
  const float ri = 1.0f / sqrtf(tot / (float)H + a.eps);
  if (!has) return;
  uint4 nwv = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);   // bf16 ones
  if (a.norm_w) nwv = *reinterpret_cast<const uint4*>(a.norm_w + kk);
  const uint32_t nw[4] = {nwv.x, nwv.y, nwv.z, nwv.w};
  uint32_t hw[4], bw[4];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float x = (q & 1) ? bf_hi(w[q >> 1]) : bf_lo(w[q >> 1]);
    const float g = (q & 1) ? bf_hi(nw[q >> 1]) : bf_lo(nw[q >> 1]);
    const bf16 v = f2bf(x * ri * g);
    const uint32_t hb = (uint32_t)__half_as_ushort(__float2half_rn(bf2f(v)));
    const uint32_t bb = (uint32_t)__bfloat16_as_ushort(v);
    hw[q >> 1] = (q & 1) ? (hw[q >> 1] | (hb << 16)) : hb;
    bw[q >> 1] = (q & 1) ? (bw[q >> 1] | (bb << 16)) : bb;
  }
  const uint4 out = a.xn_f16 ? make_uint4(hw[0], hw[1], hw[2], hw[3]) : make_uint4(bw[0], bw[1], bw[2], bw[3]);
  *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(b.xn) + (size_t)t * H + kk) = out;
}

// Router logits of prompt rows: a CTA takes kRowsR normed rows (k_norm_rows)
// and 8 experts (one per warp); each logit is router_cta's dot product (the
// warp's 128-float strips, lane l holding 4l .. 4l + 3, then the butterfly),
// so a prompt row's logits are the bits a decode step gives it.  The rows
// stay 16-bit in shared memory (xn's bf16 values, as fp16 or bf16; both
// convert to fp32 exactly), so a strip of a row is one 8-byte load.
constexpr int kRowsR = 8;

template <bool F16>
__device__ __forceinline__ float4 x4_of(uint2 p) {
  if (F16) {
    const float2 lo = __half22float2(*reinterpret_cast<const __half2*>(&p.x));
    const float2 hi = __half22float2(*reinterpret_cast<const __half2*>(&p.y));
    return make_float4(lo.x, lo.y, hi.x, hi.y);
  }
  return make_float4(bf_lo(p.x), bf_hi(p.x), bf_lo(p.y), bf_hi(p.y));
}

template <bool F16>
__global__ void __launch_bounds__(256) k_router_rows(MoeArgs a, MoeBufs b) {
  extern __shared__ __align__(16) uint16_t xs16[];   // [2][kRowsR][H]: two row blocks
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, H = a.H;
  const int eb = blockIdx.x, e = eb * 8 + warp;
  const int nrb = (a.B + kRowsR - 1) / kRowsR;
  // the warp's router row stays in registers while the CTA walks row blocks
  // blockIdx.y, + gridDim.y, ..., each block's copies in flight during the
  // previous block's logits
  float4 w4[kRouterStrips];
  if (e < a.E) router_load(a.wr + (size_t)e * H, H, lane * 4, w4);
  const int kk = threadIdx.x * 8;
  auto issue = [&](int rbk, int buf) {
    if (kk >= H) return;
    for (int j = 0; j < kRowsR; ++j) {
      const int r = rbk * kRowsR + j;
      if (r >= a.B) break;
      const uint32_t dst = (uint32_t)__cvta_generic_to_shared(xs16 + ((size_t)buf * kRowsR + j) * H + kk);
      const void* src = reinterpret_cast<const uint16_t*>(b.xn) + (size_t)r * H + kk;
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
    }
  };
  int buf = 0;
  if ((int)blockIdx.y < nrb) issue(blockIdx.y, 0);
  asm volatile("cp.async.commit_group;" ::: "memory");
  for (int rbk = blockIdx.y; rbk < nrb; rbk += gridDim.y, buf ^= 1) {
    const int nxt = rbk + (int)gridDim.y;
    if (nxt < nrb) issue(nxt, buf ^ 1);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_group 1;" ::: "memory");   // this block's rows have landed
    __syncthreads();
    const int r0 = rbk * kRowsR, rows = min(kRowsR, a.B - r0);
    const uint16_t* xb = xs16 + (size_t)buf * kRowsR * H;
    if (e < a.E) {
      // all of the block's rows at once: independent fmaf chains (each logit's
      // own order is router_cta's); rows past the last read a valid row and
      // are not stored
      float acc[kRowsR];
#pragma unroll
      for (int j = 0; j < kRowsR; ++j) acc[j] = 0.f;
#pragma unroll
      for (int i = 0; i < kRouterStrips; ++i) {
        const int k = lane * 4 + 128 * i;
        if (k < H) {
#pragma unroll
          for (int j = 0; j < kRowsR; ++j) {
            const float4 x = x4_of<F16>(*reinterpret_cast<const uint2*>(xb + (size_t)(j < rows ? j : 0) * H + k));
            acc[j] = fmaf(x.x, w4[i].x, acc[j]); acc[j] = fmaf(x.y, w4[i].y, acc[j]);
            acc[j] = fmaf(x.z, w4[i].z, acc[j]); acc[j] = fmaf(x.w, w4[i].w, acc[j]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kRowsR; ++j) {
        const float v = warp_sum(acc[j]);
        if (lane == 0 && j < rows) b.logits[(size_t)(r0 + j) * a.E + e] = v;
      }
    }
    __syncthreads();   // every warp is done with this buffer before it is refilled
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// Gate/up: a lane group computes rows f of W_g[e] and W_u[e] together.
template <int LPR, int CPL>
__global__ void __launch_bounds__(kSimtThreads) k_gateup(MoeArgs a, MoeBufs b, const bf16* xin) {
  extern __shared__ float xs[];
  __shared__ const bf16* rows[kMaxTile];
  __shared__ float rinv_unused[kMaxTile];
  const int u = blockIdx.y;
  if (u >= *b.n_active) return;
  const int e = b.active_e[u], off = b.active_off[u], cnt = b.active_off[u + 1] - off;
  constexpr int kGroups = kWarp / LPR;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPR, gl = lane % LPR;
  const int f = blockIdx.x * (kSimtWarps * kGroups) + warp * kGroups + grp;
  const bool ok = f < a.F;
  const size_t row = (size_t)e * a.F + f;
  const uint8_t* wrow[2] = {ok ? a.wg + row * (a.H >> 1) : nullptr, ok ? a.wu + row * (a.H >> 1) : nullptr};
  const __half* srow[2] = {ok ? a.wg_s + row * (a.H / a.g) : nullptr, ok ? a.wu_s + row * (a.H / a.g) : nullptr};
  uint4 w[2][CPL];
  float s[2][CPL];
  load_w4<LPR, CPL, 2>(wrow, srow, a.g, gl, w, s);
  const int nch = a.H >> 5;
  for (int t0 = 0; t0 < cnt; t0 += kMaxTile) {
    const int mc = min(kMaxTile, cnt - t0);
    __syncthreads();
    if (threadIdx.x < mc) rows[threadIdx.x] = xin + (size_t)b.pair_token[off + t0 + threadIdx.x] * a.H;
    __syncthreads();
    stage_rows(xs, rows, mc, a.H, false, nullptr, 0.f, rinv_unused);
    __syncthreads();
    float gate[kMaxTile];
    dot_tile<LPR, CPL, 2>(w, s, xs, nch, gl, mc, [&](int r, int m, float v) {
      if (r == 0) {
        gate[m] = v;
      } else if (ok && gl == (m % LPR)) {
        const float gv = gate[m];
        const float sv = gv / (1.f + expf(-gv));
        b.act[(size_t)(off + t0 + m) * a.F + f] = f2bf(sv * v);
      }
    });
  }
}

template <int LPR, int CPL>
__global__ void __launch_bounds__(kSimtThreads) k_down(MoeArgs a, MoeBufs b) {
  extern __shared__ float xs[];
  __shared__ const bf16* rows[kMaxTile];
  __shared__ float rinv_unused[kMaxTile];
  const int u = blockIdx.y;
  if (u >= *b.n_active) return;
  const int e = b.active_e[u], off = b.active_off[u], cnt = b.active_off[u + 1] - off;
  constexpr int kGroups = kWarp / LPR;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = lane / LPR, gl = lane % LPR;
  const int h0 = blockIdx.x * (kSimtWarps * kGroups * 2) + (warp * kGroups + grp) * 2;
  const uint8_t* wrow[2];
  const __half* srow[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const bool ok = h0 + r < a.H;
    const size_t row = (size_t)e * a.H + h0 + r;
    wrow[r] = ok ? a.wd + row * (a.F >> 1) : nullptr;
    srow[r] = ok ? a.wd_s + row * (a.F / a.g) : nullptr;
  }
  uint4 w[2][CPL];
  float s[2][CPL];
  load_w4<LPR, CPL, 2>(wrow, srow, a.g, gl, w, s);
  const int nch = a.F >> 5;
  for (int t0 = 0; t0 < cnt; t0 += kMaxTile) {
    const int mc = min(kMaxTile, cnt - t0);
    __syncthreads();
    if (threadIdx.x < mc) rows[threadIdx.x] = b.act + (size_t)(off + t0 + threadIdx.x) * a.F;
    __syncthreads();
    stage_rows(xs, rows, mc, a.F, false, nullptr, 0.f, rinv_unused);
    __syncthreads();
    dot_tile<LPR, CPL, 2>(w, s, xs, nch, gl, mc, [&](int r, int m, float v) {
      if (wrow[r] && gl == ((r * kMaxTile + m) % LPR))
        b.out[(size_t)(off + t0 + m) * a.H + h0 + r] = v;
    });
  }
}

__global__ void __launch_bounds__(256) k_combine(MoeArgs a, MoeBufs b) {
  __shared__ float w_s[16];
  __shared__ int pos_s[16];
  const int t = blockIdx.x;
  if (threadIdx.x < a.k) {
    w_s[threadIdx.x] = b.topk_w[t * a.k + threadIdx.x];
    pos_s[threadIdx.x] = b.pos_of[t * a.k + threadIdx.x];
  }
  __syncthreads();
  for (int h = threadIdx.x; h < a.H; h += blockDim.x) {
    float ov[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) ov[r] = r < a.k ? b.out[(size_t)pos_s[r] * a.H + h] : 0.f;
    float acc = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r)
      if (r < a.k) acc = fmaf(w_s[r], ov[r], acc);
    const float res = a.res ? bf2f(a.res[(size_t)t * a.H + h]) : 0.f;
    a.y[(size_t)t * a.H + h] = f2bf(res + acc);
  }
}

// The combine followed by the next RMSNorm of the same row: y as in
// k_combine, then xn = bf16(y * rinv * nw) with rinv from the bf16 values of
// y.  One CTA of kCombineThreads per token (H <= kCombineMaxH, the row kept
// in shared memory); each thread issues the k loads of an element at once.
constexpr int kCombineThreads = 1024, kCombineMaxH = 8192;

__global__ void __launch_bounds__(kCombineThreads) k_combine_norm(MoeArgs a, MoeBufs b, const bf16* __restrict__ nw,
                                                                  void* __restrict__ xn, int xn_f16) {
  __shared__ float red[32];
  __shared__ float w_s[16];
  __shared__ int pos_s[16];
  __shared__ float ys[kCombineMaxH];
  const int t = blockIdx.x, H = a.H;
  // Everything but the expert outputs is loaded before the dependency wait:
  // the routing weights and positions and the residual row were written
  // before the down projection took its own wait (this launch starts only
  // once the down projection has triggered or completed, and it never
  // triggers before that wait), and the norm weights are constant.  These
  // are the first pass's elements h and h + kCombineThreads (all of them
  // while H <= 2 kCombineThreads).
  if (threadIdx.x < a.k) {
    w_s[threadIdx.x] = b.topk_w[t * a.k + threadIdx.x];
    pos_s[threadIdx.x] = b.pos_of[t * a.k + threadIdx.x];
  }
  float res_pre[2] = {0.f, 0.f}, nw_pre[2] = {1.f, 1.f};
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int h = threadIdx.x + j * kCombineThreads;
    if (h < H) {
      if (a.res) res_pre[j] = bf2f(a.res[(size_t)t * H + h]);
      if (nw) nw_pre[j] = bf2f(nw[h]);
    }
  }
  pdl_wait();
  pdl_trigger();   // one wave (a CTA per token): the next projection may start its weight loads
  __syncthreads();
  const float* __restrict__ outp = b.out;
  const int kk = a.k;
  float ss = 0.f;
  // two elements per thread at a time (H <= 2048 in one pass), every expert
  // output of both loaded before either sum; the sums and the squares run in
  // the same order as one element at a time
  for (int h = threadIdx.x; h < H; h += 2 * kCombineThreads) {
    const int h2 = h + kCombineThreads;
    const bool two = h2 < H, first = h == (int)threadIdx.x;
    float ov[2][8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      ov[0][r] = r < kk ? __ldg(outp + (size_t)pos_s[r] * H + h) : 0.f;
      ov[1][r] = r < kk && two ? __ldg(outp + (size_t)pos_s[r] * H + h2) : 0.f;
    }
    const float res0 = first ? res_pre[0] : a.res ? bf2f(a.res[(size_t)t * H + h]) : 0.f;
    const float res1 = first ? res_pre[1] : a.res && two ? bf2f(a.res[(size_t)t * H + h2]) : 0.f;
#pragma unroll
    for (int e2 = 0; e2 < 2; ++e2) {
      const int he = e2 ? h2 : h;
      if (e2 && !two) break;
      float acc = 0.f;
#pragma unroll
      for (int r = 0; r < 8; ++r)
        if (r < kk) acc = fmaf(w_s[r], ov[e2][r], acc);
      for (int r = 8; r < kk; ++r) acc = fmaf(w_s[r], __ldg(outp + (size_t)pos_s[r] * H + he), acc);
      const bf16 y = f2bf((e2 ? res1 : res0) + acc);
      a.y[(size_t)t * H + he] = y;
      ys[he] = bf2f(y);
      ss = fmaf(ys[he], ys[he], ss);
    }
  }
  const float r = block_rms_inv(ss, H, a.eps, red);
  for (int h = threadIdx.x, j = 0; h < H; h += kCombineThreads, ++j) {
    const float v = round_bf16(ys[h] * r * (j < 2 ? nw_pre[j] : nw ? bf2f(nw[h]) : 1.f));
    if (xn_f16) static_cast<__half*>(xn)[(size_t)t * H + h] = __float2half_rn(v);
    else static_cast<bf16*>(xn)[(size_t)t * H + h] = f2bf(v);
  }
}

// The same for the rows of a prompt, many at once: one CTA of kRowThreads
// per row and 8 consecutive elements per thread, every expert output of its
// elements loaded at once (16-byte loads).  Each element is the same fmaf
// chain over the row's experts as in k_combine_norm; only the order in which
// the squares meet for the norm differs (a row's result still depends on
// nothing but the row).  k <= 8, H % 8 == 0, H <= 8 x kRowThreads x 2.
constexpr int kRowThreads = 256, kRowMaxK = 8, kRowVecs = 2;

__global__ void __launch_bounds__(kRowThreads) k_combine_norm_rows(MoeArgs a, MoeBufs b, const bf16* __restrict__ nw,
                                                                   void* __restrict__ xn, int xn_f16) {
  __shared__ float red[kRowThreads / 32];
  __shared__ float w_s[kRowMaxK];
  __shared__ int pos_s[kRowMaxK];
  const int t = blockIdx.x, H = a.H, kk = a.k;
  if (threadIdx.x < kk) {
    w_s[threadIdx.x] = b.topk_w[t * kk + threadIdx.x];
    pos_s[threadIdx.x] = b.pos_of[t * kk + threadIdx.x];
  }
  __syncthreads();
  float ss = 0.f;
  for (int vi = 0; vi < kRowVecs; ++vi) {
    const int h0 = (vi * kRowThreads + (int)threadIdx.x) * 8;
    if (h0 >= H) break;
    float4 ov[kRowMaxK][2];
#pragma unroll
    for (int r = 0; r < kRowMaxK; ++r) {
      if (r < kk) {
        const float4* src = reinterpret_cast<const float4*>(b.out + (size_t)pos_s[r] * H + h0);
        ov[r][0] = __ldg(src);
        ov[r][1] = __ldg(src + 1);
      }
    }
    uint4 rv = make_uint4(0u, 0u, 0u, 0u);
    if (a.res) rv = *reinterpret_cast<const uint4*>(a.res + (size_t)t * H + h0);
    const uint32_t rw[4] = {rv.x, rv.y, rv.z, rv.w};
    uint32_t yw[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float acc = 0.f;
#pragma unroll
      for (int r = 0; r < kRowMaxK; ++r) {
        if (r < kk) {
          const float4 q = ov[r][i >> 2];
          const float o = (i & 3) == 0 ? q.x : (i & 3) == 1 ? q.y : (i & 3) == 2 ? q.z : q.w;
          acc = fmaf(w_s[r], o, acc);
        }
      }
      const float res = a.res ? ((i & 1) ? bf_hi(rw[i >> 1]) : bf_lo(rw[i >> 1])) : 0.f;
      const bf16 y = f2bf(res + acc);
      const uint32_t yb = (uint32_t)__bfloat16_as_ushort(y);
      yw[i >> 1] = (i & 1) ? (yw[i >> 1] | (yb << 16)) : yb;
      const float yf = bf2f(y);
      ss = fmaf(yf, yf, ss);
    }
    *reinterpret_cast<uint4*>(a.y + (size_t)t * H + h0) = make_uint4(yw[0], yw[1], yw[2], yw[3]);
  }
  const float rinv = block_rms_inv(ss, H, a.eps, red);
  for (int vi = 0; vi < kRowVecs; ++vi) {
    const int h0 = (vi * kRowThreads + (int)threadIdx.x) * 8;
    if (h0 >= H) break;
    // this thread's own y values, just written
    const uint4 yv = *reinterpret_cast<const uint4*>(a.y + (size_t)t * H + h0);
    const uint32_t yr[4] = {yv.x, yv.y, yv.z, yv.w};
    uint32_t ow[4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float yf = (i & 1) ? bf_hi(yr[i >> 1]) : bf_lo(yr[i >> 1]);
      const float v = round_bf16(yf * rinv * (nw ? bf2f(nw[h0 + i]) : 1.f));
      const uint32_t bits =
          xn_f16 ? (uint32_t)__half_as_ushort(__float2half_rn(v)) : (uint32_t)__bfloat16_as_ushort(f2bf(v));
      ow[i >> 1] = (i & 1) ? (ow[i >> 1] | (bits << 16)) : bits;
    }
    uint16_t* dst = static_cast<uint16_t*>(xn) + (size_t)t * H + h0;
    *reinterpret_cast<uint4*>(dst) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
  }
}

template <int LPR, int CPL>
cudaError_t run_gateup(const MoeArgs& a, const MoeBufs& b, const bf16* xin, int max_u, cudaStream_t st) {
  constexpr int kGroups = kWarp / LPR;
  dim3 grid((a.F + kSimtWarps * kGroups - 1) / (kSimtWarps * kGroups), max_u);
  const size_t smem = (size_t)min(a.B, kMaxTile) * a.H * sizeof(float);
  k_gateup<LPR, CPL><<<grid, kSimtThreads, smem, st>>>(a, b, xin);
  return cudaGetLastError();
}

template <int LPR, int CPL>
cudaError_t run_down(const MoeArgs& a, const MoeBufs& b, int max_u, cudaStream_t st) {
  constexpr int rows = kSimtWarps * (kWarp / LPR) * 2;
  dim3 grid((a.H + rows - 1) / rows, max_u);
  const size_t smem = (size_t)min(a.B, kMaxTile) * a.F * sizeof(float);
  k_down<LPR, CPL><<<grid, kSimtThreads, smem, st>>>(a, b);
  return cudaGetLastError();
}

#define BM_EXPERT_SHAPES(X) X(32, 1) X(32, 2) X(32, 3) X(32, 4) X(16, 1) X(16, 3) X(8, 1) X(8, 3)

cudaError_t dispatch_gateup(const MoeArgs& a, const MoeBufs& b, const bf16* xin, int max_u, cudaStream_t st) {
  const int nch = a.H / 32;
#define BM_CASE(L, C) if (nch == (L) * (C)) return run_gateup<L, C>(a, b, xin, max_u, st);
  BM_EXPERT_SHAPES(BM_CASE)
#undef BM_CASE
  return cudaErrorInvalidValue;
}

cudaError_t dispatch_down(const MoeArgs& a, const MoeBufs& b, int max_u, cudaStream_t st) {
  const int nch = a.F / 32;
#define BM_CASE(L, C) if (nch == (L) * (C)) return run_down<L, C>(a, b, max_u, st);
  BM_EXPERT_SHAPES(BM_CASE)
#undef BM_CASE
  return cudaErrorInvalidValue;
}

template <int L, int C>
cudaError_t set_attr_pair() {
  const int bytes = kMaxTile * L * C * 32 * (int)sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(k_gateup<L, C>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(k_down<L, C>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e;
}

size_t align_up(size_t v) { return (v + 255) & ~size_t(255); }

}  // namespace

size_t moe_scratch_bytes(int B, int E, int k, int H, int F) {
  const size_t P = (size_t)B * k;
  return align_up(sizeof(float) * B * E) + align_up(sizeof(int32_t) * P) + align_up(sizeof(float) * P) +
         align_up(sizeof(bf16) * B * H) + align_up(sizeof(int32_t)) + align_up(sizeof(int32_t) * E) +
         align_up(sizeof(int32_t) * (E + 1)) + align_up(sizeof(int32_t) * P) + align_up(sizeof(int32_t) * P) +
         align_up(sizeof(int32_t)) + align_up(sizeof(int32_t) * moe_max_jobs(B, E, k)) +
         align_up(sizeof(bf16) * P * F) + align_up(sizeof(float) * P * H);
}

int moe_max_jobs(int B, int E, int k) {
  const int P = B * k;
  return (P < E ? P : E) + P / kJobTokens;
}

MoeBufs moe_carve(void* ws, int B, int E, int k, int H, int F) {
  char* p = static_cast<char*>(ws);
  const size_t P = (size_t)B * k;
  auto take = [&](size_t bytes) { char* r = p; p += align_up(bytes); return r; };
  MoeBufs b;
  b.logits = reinterpret_cast<float*>(take(sizeof(float) * B * E));
  b.topk_ids = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * P));
  b.topk_w = reinterpret_cast<float*>(take(sizeof(float) * P));
  b.xn = reinterpret_cast<bf16*>(take(sizeof(bf16) * B * H));
  b.n_active = reinterpret_cast<int32_t*>(take(sizeof(int32_t)));
  b.active_e = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * E));
  b.active_off = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (E + 1)));
  b.pair_token = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * P));
  b.pos_of = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * P));
  b.n_jobs = reinterpret_cast<int32_t*>(take(sizeof(int32_t)));
  b.jobs = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * moe_max_jobs(B, E, k)));
  b.act = reinterpret_cast<bf16*>(take(sizeof(bf16) * P * F));
  b.out = reinterpret_cast<float*>(take(sizeof(float) * P * H));
  return b;
}

cudaError_t launch_moe_combine_norm(const MoeArgs& a, const MoeBufs& b, const bf16* nw, void* xn, int xn_f16,
                                    cudaStream_t st, const Marker& mark, bool pdl) {
  if (a.H > kCombineMaxH || a.k > 16) return cudaErrorInvalidValue;
  cudaError_t err = launch_k(pdl, k_combine_norm, dim3(a.B), dim3(kCombineThreads), 0, st, a, b, nw, xn, xn_f16);
  if (err == cudaSuccess) mark(KT_COMBINE);
  return err;
}

cudaError_t launch_moe_combine_norm_rows(const MoeArgs& a, const MoeBufs& b, const bf16* nw, void* xn, int xn_f16,
                                         cudaStream_t st) {
  if (a.k > kRowMaxK || a.H % 8 || a.H > 8 * kRowThreads * kRowVecs) return launch_moe_combine_norm(a, b, nw, xn, xn_f16, st, Marker(), false);
  k_combine_norm_rows<<<a.B, kRowThreads, 0, st>>>(a, b, nw, xn, xn_f16);
  return cudaGetLastError();
}

cudaError_t launch_moe(const MoeArgs& a, const MoeBufs& b, cudaStream_t st, int* launches, const Marker& mark) {
  if (a.B * a.k > kMaxPairs || a.E > 256 || a.k > 16) return cudaErrorInvalidValue;
  const dim3 rgrid((a.E + kRouterExperts - 1) / kRouterExperts, a.B);
  k_router<<<rgrid, 256, sizeof(float) * a.H, st>>>(a, b);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  mark(KT_ROUTER);
  k_topk_sort<<<1, 1024, 0, st>>>(a, b);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  mark(KT_TOPK_SORT);
  const bf16* xin = a.do_norm ? b.xn : a.x;
  const int max_u = a.B * a.k < a.E ? a.B * a.k : a.E;
  // A token routes to k distinct experts, so no expert has more than B
  // tokens and the staging buffer needs min(B, 4) rows.
  if ((err = dispatch_gateup(a, b, xin, max_u, st)) != cudaSuccess) return err;
  mark(KT_GATEUP);
  if ((err = dispatch_down(a, b, max_u, st)) != cudaSuccess) return err;
  mark(KT_DOWN);
  k_combine<<<a.B, 256, 0, st>>>(a, b);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  mark(KT_COMBINE);
  if (launches) *launches += 5;
  return cudaSuccess;
}

cudaError_t launch_moe_route(const MoeArgs& a, const MoeBufs& b, cudaStream_t st, const Marker& mark) {
  if (a.B * a.k > kMaxPairs || a.E > 256 || a.k > 16) return cudaErrorInvalidValue;
  const dim3 rgrid((a.E + kRouterExperts - 1) / kRouterExperts, a.B);
  k_router<<<rgrid, 256, sizeof(float) * a.H, st>>>(a, b);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  mark(KT_ROUTER);
  k_topk_sort<<<1, 1024, 0, st>>>(a, b);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  mark(KT_TOPK_SORT);
  return cudaSuccess;
}

cudaError_t launch_moe_route_fused(const MoeArgs& a, const MoeBufs& b, unsigned int* tok_cnt, unsigned int* all_cnt,
                                  cudaStream_t st, const Marker& mark, bool pdl) {
  if (a.B * a.k > kMaxPairs || a.E > 256 || a.k > 16 || !tok_cnt || !all_cnt) return cudaErrorInvalidValue;
  // up to 16 rows: one expert per warp, so that the grid covers more SMs and
  // each warp has a single router row to fetch
  cudaError_t err;
  const size_t smem = sizeof(float) * a.H;
  // one wave (every CTA resident at once): the launch may trigger its
  // dependents without their CTAs taking slots it still needs
  auto one_wave = [&](auto kern, const dim3& grid) {
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem) != cudaSuccess)
      return 0;
    return (long)grid.x * grid.y <= (long)sms * per_sm ? 1 : 0;
  };
  if (a.B <= 16) {
    const dim3 rgrid((a.E + kRouterWarps - 1) / kRouterWarps, a.B);
    const int trig = pdl ? one_wave(k_route_fused<kRouterWarps>, rgrid) : 0;
    err = launch_k(pdl, k_route_fused<kRouterWarps>, rgrid, dim3(256), smem, st, a, b, tok_cnt, all_cnt, trig);
  } else {
    const dim3 rgrid((a.E + kRouterExperts - 1) / kRouterExperts, a.B);
    const int trig = pdl ? one_wave(k_route_fused<kRouterExperts>, rgrid) : 0;
    err = launch_k(pdl, k_route_fused<kRouterExperts>, rgrid, dim3(256), smem, st, a, b, tok_cnt, all_cnt, trig);
  }
  if (err == cudaSuccess) mark(KT_ROUTER);
  return err;
}

cudaError_t launch_moe_route_wide(const MoeArgs& a, const MoeBufs& b, cudaStream_t st) {
  if (a.B * a.k > kMaxPairsWide || a.E > 256 || a.k > 16 || a.H > 2048 * kRouterStrips / 16 || a.H % 8)
    return cudaErrorInvalidValue;
  const size_t smem = 2 * (size_t)kRowsR * a.H * sizeof(uint16_t);
  static bool attr = false;
  if (!attr) {
    cudaError_t e0 = cudaFuncSetAttribute(k_router_rows<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e0 == cudaSuccess)
      e0 = cudaFuncSetAttribute(k_router_rows<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    if (e0 != cudaSuccess) return e0;
    attr = true;
  }
  if (smem > 96 * 1024) return cudaErrorInvalidValue;
  k_norm_rows<<<a.B, 256, 0, st>>>(a, b);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  // about two CTAs per SM, each walking its share of the row blocks
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 132;
  }
  const int eblocks = (a.E + 7) / 8, nrb = (a.B + kRowsR - 1) / kRowsR;
  const int gy = std::max(1, std::min(nrb, (2 * sms + eblocks - 1) / eblocks));
  const dim3 rgrid(eblocks, gy);
  if (a.xn_f16) k_router_rows<true><<<rgrid, 256, smem, st>>>(a, b);
  else k_router_rows<false><<<rgrid, 256, smem, st>>>(a, b);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  k_topk_rows<<<(a.B + 7) / 8, 256, 0, st>>>(a, b);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  k_group_wide<<<1, 1024, 0, st>>>(a, b);
  return cudaGetLastError();
}

cudaError_t launch_moe_combine(const MoeArgs& a, const MoeBufs& b, cudaStream_t st, const Marker& mark) {
  k_combine<<<a.B, 256, 0, st>>>(a, b);
  const cudaError_t err = cudaGetLastError();
  if (err == cudaSuccess) mark(KT_COMBINE);
  return err;
}

cudaError_t init_moe_attributes() {
  cudaError_t e = cudaSuccess;
#define BM_CASE(L, C) if (e == cudaSuccess) e = set_attr_pair<L, C>();
  BM_EXPERT_SHAPES(BM_CASE)
#undef BM_CASE
  return e;
}

}  // namespace bm
