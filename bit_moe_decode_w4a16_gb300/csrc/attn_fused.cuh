// Device code of the fused decode attention of the warp-MMA family, shared by
// its own kernel (k_attn_fused, one work item per CTA pass) and by the
// persistent decode step (one item per pass of the CTA's first eight warps):
// both run the same instructions on an item, so they leave the same bits.
// What an item computes is described in attention_mma.cu.
//
// An item is run by kAttnThreads threads numbered by threadIdx.x from 0 and
// synchronised by `sync` (the CTA barrier, or a named barrier of exactly those
// threads).
#pragma once

#include <float.h>

#include "kernels.cuh"
#include "w4_mma.cuh"

namespace bm {
namespace attnf {

constexpr int kWarpsA = 8;   // a warp takes 16 of a chunk's 128 positions
constexpr int kAttnThreads = kWarpsA * 32;
static_assert(kAttnThreads >= 256, "a thread holds at most one element of a head (D <= 256)");
constexpr int kMaxBatch = 128;

__device__ __forceinline__ size_t rec_index(int b, int h, int c, int qh, int max_chunks, int d) {
  return (((size_t)b * qh + h) * max_chunks + c) * (size_t)(d + 2);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

// Rotate-half RoPE of one pair (x0 = x[i], x1 = x[i + d/2]) with explicit
// roundings, so every kernel that rotates k produces the same bits.
__device__ __forceinline__ void rope_pair(float x0, float x1, float c, float s, bf16& y0, bf16& y1) {
  y0 = f2bf(__fmaf_rn(x0, c, -__fmul_rn(x1, s)));
  y1 = f2bf(__fmaf_rn(x1, c, __fmul_rn(x0, s)));
}

// Position of row b: the slot's length, plus b for the rows of a prompt.
__device__ __forceinline__ int row_position(const AttnFusedArgs& a, int b, int slot) {
  return a.ar.len[slot] + (a.prefill ? a.row0 + b : 0);
}

template <int D>
struct AttnSmem {
  static constexpr int kVS = D + 8;   // padded V row: conflict-free ldmatrix
  union {
    bf16 vs[kAttnChunk][kVS];          // V rows of the chunk
    float ored[kWarpsA][8][kVS];       // per-warp partial O (after the V reads); rows padded like
                                       // vs, so a warp's 8 head rows start in 8 bank groups
  } u;
  bf16 qs[8][D];                       // rotated q of the kv group
  bf16 knew[D];                        // rotated k of a decode row's new position
  float red_m[kWarpsA][8], red_l[kWarpsA][8];
  float stat_m[8], stat_l[8];
  float mm[8][kMaxMergeChunks], ll[8][kMaxMergeChunks], ww[8][kMaxMergeChunks];   // merge: m, l, weights
  float mden[8];
  int slot[kMaxBatch], nc[kMaxBatch], pos[kMaxBatch], pre[kMaxBatch + 1];
  int ord[kMaxBatch];                  // the streams in item order
  int last;
  int next;                            // the work queue's claim for this CTA
};

// Slots, positions, chunk counts and the item prefix (chunk-major within a
// stream) of the launch's rows, into sm; returns the number of items.
// `report`: this caller records bad slots and positions in the check flag.
// Streams are in row order unless the launch has more than `slots` items
// (more than its CTAs can take at once): then longest first, ties in row
// order, so the last items handed out belong to the shortest streams, whose
// merges are the cheapest.  The order does not change what an item computes.
template <int D, class Sync>
__device__ __forceinline__ int attn_prologue(const AttnFusedArgs& a, AttnSmem<D>& sm, bool report, Sync sync,
                                             int slots = 0x7fffffff) {
  const AttnArena& ar = a.ar;
  const int tid = threadIdx.x;
  const int kvh = ar.kvh, B = a.B;
  // ---- slots, positions, chunk counts and the item prefix (chunk-major within a stream)
  for (int b = tid; b < B; b += kAttnThreads) {
    const int slot = a.slots[b];
    int nc = 0, pos = 0;
    if (slot < 0 || slot >= ar.S) {
      if (report) a.chk.fail(1);
    } else {
      pos = row_position(a, b, slot);
      if (pos < 0 || pos + 1 > ar.cap) {
        if (report) a.chk.fail(2);
      } else {
        nc = (pos + kAttnChunk) / kAttnChunk;
      }
    }
    sm.slot[b] = slot;
    sm.nc[b] = nc;
    sm.pos[b] = pos;
    sm.ord[b] = b;
  }
  sync();
  if (tid == 0) {
    sm.pre[0] = 0;
    for (int r = 0; r < B; ++r) sm.pre[r + 1] = sm.pre[r] + sm.nc[r] * kvh;
  }
  sync();
  if (sm.pre[B] > slots) {
    for (int b = tid; b < B; b += kAttnThreads) {
      const int nb = sm.nc[b];
      int r = 0;
      for (int o = 0; o < B; ++o) r += sm.nc[o] > nb || (sm.nc[o] == nb && o < b);
      sm.ord[r] = b;
    }
    sync();
    if (tid == 0)
      for (int r = 0; r < B; ++r) sm.pre[r + 1] = sm.pre[r] + sm.nc[sm.ord[r]] * kvh;
    sync();
  }
  return sm.pre[B];
}

// Work item `it` (stream, kv head, chunk) of the launch, after attn_prologue.
template <int D, class Sync>
__device__ __forceinline__ void attn_item(const AttnFusedArgs& a, AttnSmem<D>& sm, int it, Sync sync) {
  constexpr int kBlk = D / 32;
  constexpr int kV8 = D / 8;
  constexpr int kNT = D / 8;
  const AttnArena& ar = a.ar;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int kvh = ar.kvh, G = a.qh / kvh, half = D / 2;
  const float scale = 1.0f / sqrtf((float)D);
  int rank = 0;
  while (sm.pre[rank + 1] <= it) ++rank;
  const int b = sm.ord[rank];
  const int r = it - sm.pre[rank], kh = r % kvh, c = r / kvh;
  const int slot = sm.slot[b], nc = sm.nc[b], pos = sm.pos[b], L = pos + 1;
  const int j0 = c * kAttnChunk, n = min(kAttnChunk, L - j0);
  const bool last_chunk = c == nc - 1;
  // on the chunk that holds a decode row's new position, k and v of that
  // position come from this row's qkv (rotated here), not from the arena
  const bool own_new = last_chunk && !a.prefill;
  const int p_new = own_new ? pos - j0 : -1;
  const bf16* row = a.qkv + (size_t)b * a.ld_qkv;
  const bf16* ksrc = row + (size_t)(a.qh + kh) * D;
  const bf16* vsrc = row + (size_t)(a.qh + kvh + kh) * D;
  const size_t base = (size_t)a.layer * ar.layer_stride() + (size_t)slot * ar.slot_stride() + (size_t)kh * ar.cap * D;
  bf16* Kb = ar.K + base;
  bf16* Vb = ar.V + base;

  // ---- every load of the item at once: V rows (async, to shared memory),
  // the lane's K rows, the rotation table, q and the new k / v
  for (int i = tid; i < kAttnChunk * kV8; i += kAttnThreads) {
    const int rr = i / kV8, v8 = i - rr * kV8;
    if (rr == p_new) cp_async16(&sm.u.vs[rr][v8 * 8], vsrc + v8 * 8);
    else if (rr < n) cp_async16(&sm.u.vs[rr][v8 * 8], Vb + (size_t)(j0 + rr) * D + v8 * 8);
    else *reinterpret_cast<uint4*>(&sm.u.vs[rr][v8 * 8]) = make_uint4(0, 0, 0, 0);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  uint4 kb[2][kBlk];   // this lane's B column of n-tile nt: position 16w + 8nt + g
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int p = 16 * warp + 8 * nt + g;
#pragma unroll
    for (int blk = 0; blk < kBlk; ++blk)
      kb[nt][blk] = p < n && p != p_new
                        ? __ldcg(reinterpret_cast<const uint4*>(Kb + (size_t)(j0 + p) * D + 32 * blk + 8 * t))
                        : make_uint4(0, 0, 0, 0);
  }

  // ---- RoPE of the kv group's q heads (and of the new k, with its append):
  // every load first (the q pairs, the new k pair and v, the rotation
  // table), then the rotations, so the phase waits on one round trip
  const float2* cs = a.rope + (size_t)pos * half;
  constexpr int kQ = (4 * D + kAttnThreads - 1) / kAttnThreads;   // q pairs per thread (8 heads x D / 2)
  float qx0[kQ], qx1[kQ];
  float2 qcs[kQ];
#pragma unroll
  for (int u = 0; u < kQ; ++u) {
    const int idx = tid + u * kAttnThreads, h = idx / half, i = idx - h * half;
    qx0[u] = qx1[u] = 0.f;
    qcs[u] = make_float2(0.f, 0.f);
    if (idx < 8 * half && h < G) {
      const bf16* src = row + (size_t)(kh * G + h) * D;
      qx0[u] = bf2f(src[i]);
      qx1[u] = bf2f(src[i + half]);
      qcs[u] = cs[i];
    }
  }
  // the new position's k pair and v element of this thread (half <= D <= kAttnThreads)
  const bool kt = own_new && tid < half, vt = own_new && tid < D;
  float kx0 = 0.f, kx1 = 0.f;
  float2 kcs = make_float2(0.f, 0.f);
  bf16 vnew = f2bf(0.f);
  if (kt) {
    kx0 = bf2f(ksrc[tid]);
    kx1 = bf2f(ksrc[tid + half]);
    kcs = cs[tid];
  }
  if (vt) vnew = vsrc[tid];
#pragma unroll
  for (int u = 0; u < kQ; ++u) {
    const int idx = tid + u * kAttnThreads, h = idx / half, i = idx - h * half;
    if (idx < 8 * half) {
      bf16 y0 = f2bf(0.f), y1 = f2bf(0.f);
      if (h < G) rope_pair(qx0[u], qx1[u], qcs[u].x, qcs[u].y, y0, y1);
      sm.qs[h][i] = y0;
      sm.qs[h][i + half] = y1;
    }
  }
  if (kt) {
    bf16 y0, y1;
    rope_pair(kx0, kx1, kcs.x, kcs.y, y0, y1);
    sm.knew[tid] = y0;
    sm.knew[tid + half] = y1;
    Kb[(size_t)pos * D + tid] = y0;
    Kb[(size_t)pos * D + tid + half] = y1;
  }
  if (vt) Vb[(size_t)pos * D + tid] = vnew;
  sync();
  if (own_new) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
      if (16 * warp + 8 * nt + g == p_new) {
#pragma unroll
        for (int blk = 0; blk < kBlk; ++blk) kb[nt][blk] = *reinterpret_cast<const uint4*>(&sm.knew[32 * blk + 8 * t]);
      }
  }

  // ---- scores: warp w takes positions [16w, 16w + 16): 2 n-tiles of 8
  uint32_t qa[kBlk][4];
#pragma unroll
  for (int blk = 0; blk < kBlk; ++blk) {
    const uint4 q4 = *reinterpret_cast<const uint4*>(&sm.qs[g][32 * blk + 8 * t]);
    qa[blk][0] = q4.x; qa[blk][1] = q4.y; qa[blk][2] = q4.z; qa[blk][3] = q4.w;
  }
  float s[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int q = 0; q < 4; ++q) s[nt][q] = 0.f;
#pragma unroll
    for (int blk = 0; blk < kBlk; ++blk) {
      const uint32_t a0[4] = {qa[blk][0], 0u, qa[blk][1], 0u};
      const uint32_t a1[4] = {qa[blk][2], 0u, qa[blk][3], 0u};
      mma::mma_bf16(s[nt], a0, kb[nt][blk].x, kb[nt][blk].y);
      mma::mma_bf16(s[nt], a1, kb[nt][blk].z, kb[nt][blk].w);
    }
  }
  // s[nt][0..1] = S[head g][position 16w + 8nt + 2t (+1)]; rows g + 8 (c2, c3) are padding
  float mx = -FLT_MAX;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int p = 16 * warp + 8 * nt + 2 * t + j;
      s[nt][j] = p < n ? s[nt][j] * scale : -FLT_MAX;
      mx = fmaxf(mx, s[nt][j]);
    }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  if (t == 0) sm.red_m[warp][g] = mx;
  sync();
  // every lane takes its head's maximum over the warps itself (a maximum does
  // not depend on the order), so no second barrier waits for one thread's;
  // the record's copy is written by the first 8 threads
  float mrow = sm.red_m[0][g];
  for (int w = 1; w < kWarpsA; ++w) mrow = fmaxf(mrow, sm.red_m[w][g]);
  if (tid < 8) {
    float m = sm.red_m[0][tid];
    for (int w = 1; w < kWarpsA; ++w) m = fmaxf(m, sm.red_m[w][tid]);
    sm.stat_m[tid] = m;
  }
  float ls = 0.f;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int p = 16 * warp + 8 * nt + 2 * t + j;
      s[nt][j] = p < n ? expf(s[nt][j] - mrow) : 0.f;
      ls += s[nt][j];
    }
  ls += __shfl_xor_sync(0xffffffffu, ls, 1);
  ls += __shfl_xor_sync(0xffffffffu, ls, 2);
  if (t == 0) sm.red_l[warp][g] = ls;
  asm volatile("cp.async.wait_all;" ::: "memory");
  sync();
  if (tid < 8) {
    float l = 0.f;
    for (int w = 0; w < kWarpsA; ++w) l += sm.red_l[w][tid];
    sm.stat_l[tid] = l;
  }

  // ---- O = P V over the warp's 16 positions (one k-step)
  float o[kNT][4];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int q = 0; q < 4; ++q) o[nt][q] = 0.f;
  {
    const uint32_t pa[4] = {pack_f16(s[0][0], s[0][1]), 0u, pack_f16(s[1][0], s[1][1]), 0u};
    const int vrow = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int dt = 0; dt < kNT / 2; ++dt) {
      uint32_t vb[4];
      ldsm_x4_trans(vb, static_cast<uint32_t>(__cvta_generic_to_shared(&sm.u.vs[vrow][16 * dt + (lane >> 4) * 8])));
#pragma unroll
      for (int q = 0; q < 4; ++q) vb[q] = mma::bf2_to_h2(vb[q]);   // exact: V is bf16 inside fp16's range
      mma::mma_f16(o[2 * dt], pa, vb[0], vb[1]);
      mma::mma_f16(o[2 * dt + 1], pa, vb[2], vb[3]);
    }
  }
  sync();   // all V reads are done: the union now holds the partial O
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt) {
    *reinterpret_cast<float2*>(&sm.u.ored[warp][g][8 * nt + 2 * t]) = make_float2(o[nt][0], o[nt][1]);
  }
  sync();

  if (nc == 1) {
    // ---- one chunk: its record is the result (the merge of one chunk has
    // weight exp(0) = 1, so o / l is the merge's value bit for bit)
    for (int idx = tid; idx < G * D; idx += kAttnThreads) {
      const int h = idx / D, d = idx - h * D;
      float v = 0.f;
      for (int w = 0; w < kWarpsA; ++w) v += sm.u.ored[w][h][d];
      a.out[((size_t)b * a.qh + kh * G + h) * D + d] = __float2half_rn(round_bf16(v / sm.stat_l[h]));
    }
    sync();
    return;
  }

  // ---- the chunk's record: o (warps added in order), m, l
  for (int idx = tid; idx < G * D; idx += kAttnThreads) {
    const int h = idx / D, d = idx - h * D;
    float v = 0.f;
    for (int w = 0; w < kWarpsA; ++w) v += sm.u.ored[w][h][d];
    a.part[rec_index(b, kh * G + h, c, a.qh, a.max_chunks, D) + d] = v;
  }
  if (tid < G) {
    float* rec = a.part + rec_index(b, kh * G + tid, c, a.qh, a.max_chunks, D);
    rec[D] = sm.stat_m[tid];
    rec[D + 1] = sm.stat_l[tid];
  }
  sync();
  // ---- merges, ascending order throughout.  A stream of at most
  // kAttnMergeBlock chunks: the last arriving chunk merges them all.  A longer
  // one merges in two levels: the last chunk of each block of kAttnMergeBlock
  // merges the block into a block record (over the block's first chunk
  // record: o unnormalised, its m and l), and the last block merges the
  // block records, so no merge reads more than kAttnMergeBlock records.
  // `merge` runs over `count` records c_first, c_first + c_step, ...; `fin`:
  // write the normalised output, else the block record.
  auto merge = [&](int c_first, int c_step, int count, bool fin) {
    // a thread's outputs (at most 8 D / kAttnThreads of the G x D); every
    // record load in flight before the sums
    constexpr int kOut = 8 * D / kAttnThreads;
    float pv[kOut][kAttnMergeBlock];
#pragma unroll
    for (int o = 0; o < kOut; ++o) {
      const int idx = tid + o * kAttnThreads, h = idx / D, d = idx - h * D;
#pragma unroll
      for (int u = 0; u < kAttnMergeBlock; ++u)
        pv[o][u] = idx < G * D && u < count
                       ? __ldcg(a.part + rec_index(b, kh * G + h, c_first + u * c_step, a.qh, a.max_chunks, D) + d)
                       : 0.f;
    }
    for (int idx = tid; idx < G * count; idx += kAttnThreads) {
      const int h = idx / count, cc = idx - h * count;
      const float* rec = a.part + rec_index(b, kh * G + h, c_first + cc * c_step, a.qh, a.max_chunks, D);
      sm.mm[h][cc] = __ldcg(rec + D);
      sm.ll[h][cc] = __ldcg(rec + D + 1);
    }
    sync();
    if (tid < G) {
      float M = -FLT_MAX;
      for (int cc = 0; cc < count; ++cc) M = fmaxf(M, sm.mm[tid][cc]);
      float den = 0.f;
      for (int cc = 0; cc < count; ++cc) {
        const float w = expf(sm.mm[tid][cc] - M);
        sm.ww[tid][cc] = w;
        den = fmaf(sm.ll[tid][cc], w, den);
      }
      sm.mden[tid] = den;
      sm.stat_m[tid] = M;
    }
    sync();
#pragma unroll
    for (int o = 0; o < kOut; ++o) {
      const int idx = tid + o * kAttnThreads, h = idx / D, d = idx - h * D;
      if (idx >= G * D) continue;
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < kAttnMergeBlock; ++u)
        if (u < count) acc = fmaf(pv[o][u], sm.ww[h][u], acc);
      if (fin) {
        a.out[((size_t)b * a.qh + kh * G + h) * D + d] = __float2half_rn(round_bf16(acc / sm.mden[h]));
      } else {
        a.part[rec_index(b, kh * G + h, c_first, a.qh, a.max_chunks, D) + d] = acc;
      }
    }
    if (!fin && tid < G) {
      float* rec = a.part + rec_index(b, kh * G + tid, c_first, a.qh, a.max_chunks, D);
      rec[D] = sm.stat_m[tid];
      rec[D + 1] = sm.mden[tid];
    }
  };
  // Arrival on a counter after a CTA barrier: thread 0 fences (every thread's
  // record stores are ordered before it by the barrier) and counts; the last
  // of n arrivals fences again, so the other CTAs' records are visible to the
  // merge's loads after the next barrier.
  auto arrive = [&](unsigned int* cnt, int n) {
    if (tid == 0) {
      __threadfence();
      const bool last = atomicAdd(cnt, 1u) == (unsigned)(n - 1);
      if (last) __threadfence();
      sm.last = last;
    }
    sync();
    return sm.last != 0;
  };
  unsigned int* scnt = &a.counters[b * kvh + kh];
  if (nc <= kAttnMergeBlock) {
    if (arrive(scnt, nc)) {
      merge(0, 1, nc, true);
      if (tid == 0) *scnt = 0u;
    }
  } else {
    const int blk = c / kAttnMergeBlock, c0b = blk * kAttnMergeBlock, nbk = min(kAttnMergeBlock, nc - c0b);
    const int nblk = (nc + kAttnMergeBlock - 1) / kAttnMergeBlock;
    unsigned int* bcnt = a.counters + (size_t)a.B * kvh + (size_t)(b * kvh + kh) * kAttnMergeBlocks + blk;
    if (arrive(bcnt, nbk)) {
      merge(c0b, 1, nbk, false);
      if (tid == 0) *bcnt = 0u;
      sync();   // the block record is written
      if (arrive(scnt, nblk)) {
        merge(0, kAttnMergeBlock, nblk, true);
        if (tid == 0) *scnt = 0u;
      }
    }
  }
  sync();   // shared memory is reused by the next item
}

struct CtaSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

}  // namespace attnf
}  // namespace bm
