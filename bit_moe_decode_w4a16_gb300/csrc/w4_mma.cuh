// Warp-level tensor-core W4A16 projections (mma.sync m16n8k16, fp16 x fp16
// -> fp32) for the decode step: the dense projections and the grouped expert
// gate/up and down GEMMs.
//
// Operands.  The MMA runs on fp16: every activation this family consumes is
// written as fp16 by the kernel that produces it (a bf16 value converts to
// fp16 exactly inside fp16's range), and each code enters as a biased fp16
// integer from the packed word: the nibbles of rows r0 become (1024 + u)
// (low nibble of a byte, magic 0x6400) and those of rows r1 (64 + u) (high
// nibble, magic 0x5400: 64 has an ulp of 1/16, so the nibble at bits 4-7
// adds exactly u); one HSUB2 each (1032, 72) leaves the exact code q = u - 8.
// That is 5 integer and 4 fp16 ops per 8 codes, on two different pipes.
// Products q x are exact in fp32.
//
// Why this instruction.  A decode projection streams its int4 weights once
// per step against at most a few dozen tokens, so it is bound by HBM, and the
// per-instruction cost of the multiply decides whether the weight stream can
// be kept at the memory rate.  Measured on this GPU, one tcgen05.mma of
// M=128 x N x K=16 costs about 97 SM cycles for every N up to 128, whatever
// its operand sources, so at a decode batch's N a CTA retires ~1 KB of int4
// weights per 97 cycles through it (~3.3 TB/s over the whole GPU before any
// other cost).  mma.sync.m16n8k16 retires at 2 cycles per SM with four or
// more warps issuing, i.e. 128 bytes of int4 weights per instruction per SM
// every 2 cycles: the tensor pipe stops being the limit.
//
// Work split.  A warp owns two 16-row tiles (32 weight rows) and a fixed
// range of K (CPW chunks of 64); the KS warps that share the rows cover the
// whole K.  A CTA is RTP such row pairs x KS K-ranges.  KS and CPW depend
// only on the matrix shape, never on the batch, so each output is the same
// fixed-order sum whatever the batch holds:
//     y = sum over ks (ascending) of [ sum over the warp's scale groups
//         (ascending K) of scale x (exact group sum of q x) ]
// where the group sum is accumulated in fp32 by the MMA.
//
// Int4 layout ("mma layout", written once by the repack kernel): for 16-row
// tile T and 64-wide chunk c, 32 lanes x 16 bytes; lane (g = lane / 4,
// t = lane % 4) holds one 32-bit word per MMA step s = 0..3 of the chunk.
// K is permuted inside each 32-wide block b = s / 2 so that a lane's B
// fragment of a block is the 8 consecutive activations k = 32b + 8t .. +7:
// with base = 64c + 32b + 8t + 4(s % 2), the word's nibbles 0..7 are
//     W[r0][base], W[r1][base], W[r0][base+2], W[r1][base+2],
//     W[r0][base+1], W[r1][base+1], W[r0][base+3], W[r1][base+3]
// (r0 = 16T + g, r1 = r0 + 8): fragment registers a0, a1 are the masks
// 0x000F000F and 0x00F000F0 of the word, a2, a3 the same masks of word >> 8.
// Scales: [T][K/g][8] words, word p = fp16
// scales of rows (16T + p, 16T + p + 8).  Expert gate/up banks interleave
// by 8 inside a tile: rows 0-7 are gate rows 8T..8T+7, rows 8-15 the up
// rows of the same features, so one thread holds both halves of a SiLU pair.
#pragma once

#include "kernels.cuh"

namespace bm {
namespace mma {

constexpr int kChunkK = 64;
constexpr int kMaxWarps = 16;

enum Mode { DENSE = 0, GATEUP = 1, DOWN = 2 };

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A * B, m16n8k16, fp16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (a & MASK) | MAGIC in one LOP3.  Written out because the compiler splits
// the C form into an AND and an OR per pair of codes (measured: 9 integer
// instructions per packed word instead of 5, the kernels' busiest pipe).
template <uint32_t MASK, uint32_t MAGIC>
__device__ __forceinline__ uint32_t and_or(uint32_t a) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(d) : "r"(a), "n"(MASK), "n"(MAGIC));   // (a & b) | c
  return d;
}
__device__ __forceinline__ uint32_t sub_h2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// One packed word -> the four A-fragment registers: fp16 pairs of the exact
// codes q, rows r0 in a0, a2 and rows r1 in a1, a3 (biased codes 1024 + u and
// 64 + u less 1032 and 72).
__device__ __forceinline__ void dq_word(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t w8 = w >> 8;
  a[0] = sub_h2(and_or<0x000F000Fu, 0x64006400u>(w), 0x64086408u);
  a[1] = sub_h2(and_or<0x00F000F0u, 0x54005400u>(w), 0x54805480u);
  a[2] = sub_h2(and_or<0x000F000Fu, 0x64006400u>(w8), 0x64086408u);
  a[3] = sub_h2(and_or<0x00F000F0u, 0x54005400u>(w8), 0x54805480u);
}

// bf16 pair -> fp16 pair (exact inside fp16's range).
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t p) {
  const float lo = __uint_as_float(p << 16), hi = __uint_as_float(p & 0xFFFF0000u);
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint4 bf8_to_h8(uint4 v) {
  return make_uint4(bf2_to_h2(v.x), bf2_to_h2(v.y), bf2_to_h2(v.z), bf2_to_h2(v.w));
}

__device__ __forceinline__ uint32_t ldg_nc_u32(const void* p) {
  uint32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

__device__ __forceinline__ float half_lo(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// The projection kernel.  Grid: x = row block (RTP x 32 rows), y = token
// group (dense, 8 * NT tokens each) or routing job (experts: one expert and
// up to 8 of its sorted tokens).  Block: KS * RTP warps.
template <int MODE, int NT, int CPW, int G, bool XBF = false>
__global__ void __launch_bounds__(kMaxWarps * 32) k_w4_mma(MmaArgs a) {
  extern __shared__ float red[];   // [KS][RTP][2][NT][4][32]
  constexpr int kSpg = G / 16;                           // k-steps per scale group
  constexpr int kSpc = G >= kChunkK ? 1 : kChunkK / G;   // scale words per chunk
  static_assert(G == 32 || G == 64 || G == 128, "group size");
  static_assert(G <= kChunkK * CPW, "a warp's K range holds whole groups");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KS = a.ks, RTP = (blockDim.x >> 5) / KS;
  const int ks = warp % KS, rtp = warp / KS;

  if (MODE != DENSE) pdl_wait();   // the job list comes from the previous kernel
  const uint8_t* W = a.W;
  const uint32_t* S = a.S;
  int ntok, tok0;
  if (MODE == DENSE) {
    tok0 = blockIdx.y * 8 * NT;
    ntok = min(8 * NT, a.ntok - tok0);
  } else {
    static_assert(MODE == DENSE || NT == 1, "expert jobs hold at most 8 tokens");
    const int njobs = *a.n_jobs;
    const int job = a.jobs[blockIdx.y];   // beyond njobs: a stale word, unused
    if ((int)blockIdx.y >= njobs) return;
    const int e = job & 0x1FF;
    tok0 = (job >> 9) & 0xFFF;
    ntok = (job >> 21) & 0x1F;
    W += (size_t)e * a.w_expert_stride;
    S += (size_t)e * a.s_expert_stride;
  }
  if (ntok <= 0) return;   // uniform over the CTA

  const int NC = a.K / kChunkK, NG = a.K / G;
  const int T0 = ((int)blockIdx.x * RTP + rtp) * 2;   // first 16-row tile of this warp
  const int c0 = ks * CPW;

  // ---- all of this warp's weight and scale loads in flight at once
  uint4 wv[CPW][2];
  uint32_t sv[CPW][2][kSpc];
#pragma unroll
  for (int j = 0; j < CPW; ++j)
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
      wv[j][rt] = ldg_nc_v4(W + ((size_t)((T0 + rt) * NC + c0 + j) * 32 + lane) * 16);
#pragma unroll
  for (int j = 0; j < CPW; ++j)
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int q = 0; q < kSpc; ++q) {
        const int grp = G >= kChunkK ? ((c0 + j) * kChunkK) / G : (c0 + j) * kSpc + q;
        sv[j][rt][q] = ldg_nc_u32(S + ((size_t)(T0 + rt) * NG + grp) * 8 + (lane >> 2));
      }

  // dense: the weights above do not depend on the previous kernel
  if (MODE == DENSE) {
    pdl_wait();
    // one token group is one wave (at most two CTAs per SM): the next kernel
    // may start its own weight loads; wider launches keep their slots
    if (gridDim.y == 1) pdl_trigger();
  }

  // dense with a residual: the residual of this thread's first epilogue
  // units, loaded now so its round trip overlaps the MMA loop (a unit's
  // rows and token follow from its index alone)
  constexpr int kResPre = 2;   // the epilogue below selects these two by hand
  float res_pre[kResPre][2];
  if (MODE == DENSE && a.Res) {
#pragma unroll
    for (int u = 0; u < kResPre; ++u) {
      const int uix = (int)threadIdx.x + u * (int)blockDim.x;
      const int l = uix & 31, j = (uix >> 5) & 1, nt = (uix >> 6) % NT, rt = (uix / (64 * NT)) & 1,
                rp = uix / (128 * NT);
      const int token = nt * 8 + 2 * (l & 3) + j;
      res_pre[u][0] = res_pre[u][1] = 0.f;
      if (uix < RTP * NT * 128 && token < ntok) {
        const int tile = ((int)blockIdx.x * RTP + rp) * 2 + rt;
        const int r0 = tile * 16 + (l >> 2);
        const size_t m = (size_t)tok0 + token;
        res_pre[u][0] = bf2f(a.Res[m * a.ldr + r0]);
        res_pre[u][1] = bf2f(a.Res[m * a.ldr + r0 + 8]);
      }
    }
  }

  // ---- activation rows of the lane's B-fragment column (token g of each n-tile)
  const bf16* xr[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int tk = nt * 8 + (lane >> 2);
    const bf16* p = nullptr;
    if (tk < ntok) {
      const int row = MODE == GATEUP ? a.pair_token[tok0 + tk] : tok0 + tk;
      p = reinterpret_cast<const bf16*>(a.X) + (size_t)row * a.ldx + (lane & 3) * 8;
    }
    xr[nt] = p;
  }
  auto load_x = [&](uint4 (&dst)[NT][2], int c) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        uint4 v = xr[nt] ? *reinterpret_cast<const uint4*>(xr[nt] + c * kChunkK + 32 * b) : make_uint4(0, 0, 0, 0);
        if (XBF) v = bf8_to_h8(v);
        dst[nt][b] = v;
      }
  };

  float acc[2][NT][4];
  float tmp[2][NT][4];
#pragma unroll
  for (int rt = 0; rt < 2; ++rt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[rt][nt][c] = 0.f;

  uint4 xb[2][NT][2];
  load_x(xb[0], c0);
#pragma unroll
  for (int j = 0; j < CPW; ++j) {
    if (j + 1 < CPW) load_x(xb[(j + 1) & 1], c0 + j + 1);
#pragma unroll
    for (int rt = 0; rt < 2; ++rt) {
      const uint32_t wwords[4] = {wv[j][rt].x, wv[j][rt].y, wv[j][rt].z, wv[j][rt].w};
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const int gs = j * 4 + s;   // k-step index inside the warp's range
        uint32_t af[4];
        dq_word(wwords[s], af);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          if (gs % kSpg == 0) {
#pragma unroll
            for (int c = 0; c < 4; ++c) tmp[rt][nt][c] = 0.f;
          }
          const uint4& xv = xb[j & 1][nt][s >> 1];
          const uint32_t b0 = (s & 1) ? xv.z : xv.x, b1 = (s & 1) ? xv.w : xv.y;
          mma_f16(tmp[rt][nt], af, b0, b1);
          if ((gs + 1) % kSpg == 0) {
            const uint32_t sw = sv[j][rt][G >= kChunkK ? 0 : (s * 16) / G];
            const float slo = half_lo(sw), shi = half_hi(sw);
            acc[rt][nt][0] = fmaf(slo, tmp[rt][nt][0], acc[rt][nt][0]);
            acc[rt][nt][1] = fmaf(slo, tmp[rt][nt][1], acc[rt][nt][1]);
            acc[rt][nt][2] = fmaf(shi, tmp[rt][nt][2], acc[rt][nt][2]);
            acc[rt][nt][3] = fmaf(shi, tmp[rt][nt][3], acc[rt][nt][3]);
          }
        }
      }
    }
  }

  // ---- the KS partial sums of each output meet in shared memory
#pragma unroll
  for (int rt = 0; rt < 2; ++rt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        red[((((ks * RTP + rtp) * 2 + rt) * NT + nt) * 4 + c) * 32 + lane] = acc[rt][nt][c];
  __syncthreads();

  // ---- epilogue: unit (rtp, rt, nt, j, lane) = rows (g, g + 8) of the tile,
  // token nt * 8 + 2t + j; partials added in ks order
  const int units = RTP * NT * 128;
  for (int uix = threadIdx.x, u = 0; uix < units; uix += blockDim.x, ++u) {
    const int l = uix & 31, j = (uix >> 5) & 1, nt = (uix >> 6) % NT, rt = (uix / (64 * NT)) & 1,
              rp = uix / (128 * NT);
    const int token = nt * 8 + 2 * (l & 3) + j;
    if (token >= ntok) continue;
    float v0 = 0.f, v1 = 0.f;
    for (int k2 = 0; k2 < KS; ++k2) {
      const int base = (((k2 * RTP + rp) * 2 + rt) * NT + nt) * 4;
      v0 += red[(base + j) * 32 + l];
      v1 += red[(base + j + 2) * 32 + l];
    }
    const int tile = ((int)blockIdx.x * RTP + rp) * 2 + rt;
    const int r0 = tile * 16 + (l >> 2), r1 = r0 + 8;
    const size_t m = (size_t)tok0 + token;
    if (MODE == DENSE) {
      float y0 = v0, y1 = v1;
      if (a.Res) {
        // (selects, not an index: the array stays in registers)
        y0 += u == 0 ? res_pre[0][0] : u == 1 ? res_pre[1][0] : bf2f(a.Res[m * a.ldr + r0]);
        y1 += u == 0 ? res_pre[0][1] : u == 1 ? res_pre[1][1] : bf2f(a.Res[m * a.ldr + r1]);
      }
      a.Y[m * a.ldy + r0] = f2bf(y0);
      a.Y[m * a.ldy + r1] = f2bf(y1);
    } else if (MODE == GATEUP) {
      // the activation is rounded to bf16 (the path's 16-bit activations) and
      // stored as the same value in fp16 for the down projection's MMA
      const int f = tile * 8 + (l >> 2);
      const float sv0 = v0 / (1.f + expf(-v0));
      a.act16[m * a.F + f] = __float2half_rn(round_bf16(sv0 * v1));
    } else {
      a.out[m * a.H + r0] = v0;
      a.out[m * a.H + r1] = v1;
    }
  }
}

}  // namespace mma
}  // namespace bm
