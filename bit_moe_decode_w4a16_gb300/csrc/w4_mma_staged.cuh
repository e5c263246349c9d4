// Persistent, warp-specialised form of the warp-MMA expert projections
// (gate/up and down): the same per-output arithmetic and summation order as
// k_w4_mma (w4_mma.cuh), with the operands staged in shared memory.
//
// A work item is one block of 32 x RTP rows of one routing job (an expert and
// up to 8 of its sorted tokens) over the whole K.  In the mma layout the
// block's 16-row tiles are one contiguous slab of the expert's matrix, as are
// their scales, and each token's activation row is contiguous too, so one
// producer warp moves an item into a shared-memory stage with a handful of
// bulk async copies (cp.async.bulk, completion counted in bytes on the
// stage's `full` mbarrier).  NS stages rotate: while the consumer warps
// compute item n, the copies of the next items are in flight, without
// holding them in registers.  A CTA walks a contiguous run of items in job
// order; the producer puts each item's token rows in the stage header.
//
// Consumer warp (rtp, ks) reads its two tiles' A fragments and scales for
// chunks [ks*CPW, +CPW) and the B fragments of the 8 token rows from the
// stage into registers and releases the stage at once (`empty` mbarrier, one
// arrival per consumer warp), so the producer refills it with item n+NS while
// the warps compute; the KS partial sums meet in shared memory and are added
// in ks order, exactly as in k_w4_mma.  Every mbarrier wait is bounded; a wait that gives up sets
// the error flag and the CTA stops consuming (the remaining waits stay
// bounded), so a fault in the pipeline cannot hang the GPU.
#pragma once

#include "tc_ptx.cuh"
#include "w4_mma.cuh"

namespace bm {
namespace mma {

constexpr int kMaxStages = 8;
constexpr uint32_t kStagedWaitLimit = 1u << 18;   // polls of ~3.7 us each: a wait gives up after about a second
constexpr int kXPad = 32;   // 16-bit elements of padding per staged activation row (conflict-free LDS.128)

// Bytes the phase will see, without an arrival (the phase cannot complete
// before the arrival that follows).
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
// Bulk async copy global -> shared, completion counted on `mbar` in bytes.
// dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(mbar)
               : "memory");
}
__device__ __forceinline__ void consumer_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

struct StagedGeom {
  int nw;            // consumer warps = KS * RTP
  int rtp;           // 32-row blocks per item
  int nrb;           // items per expert matrix
  uint32_t w_bytes;  // weight slab of one item
  uint32_t s_bytes;  // scale slab of one item
  uint32_t x_stride; // bytes per staged activation row
  uint32_t stage;    // bytes of one stage (w | s | 8 activation rows), 128-aligned
  int ns;            // stages
};

struct ItemInfo {
  int tok0, ntok, rb;
  int row[kJobTokens];   // activation row of each token
};

template <int MODE, int CPW, int G>
__global__ void __launch_bounds__((kMaxWarps + 1) * 32, 1) k_w4_mma_staged(MmaArgs a, StagedGeom geo) {
  constexpr int kSpg = G / 16;
  constexpr int kSpc = G >= kChunkK ? 1 : kChunkK / G;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ ItemInfo info_s[kMaxStages];
  __shared__ int abort_s;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NW = geo.nw, RTP = geo.rtp, KS = NW / RTP;
  const int NC = a.K / kChunkK, NG = a.K / G;
  // gate/up: the job list comes from the previous kernel; its grid is one
  // wave, and each CTA's producer triggers the dependents when it issues the
  // CTA's last item, so the down projection launches on each SM as that SM's
  // CTA finishes (an earlier trigger measured slower per launch).  down: the
  // job list was written by the routing launch, which completed before the
  // gate/up launch took its own wait, so it is read (through L2) before this
  // launch's wait, and the first stages' weights and scales are on their way
  // while gate/up runs its last items; only the rows it wrote wait.
  if (MODE != DOWN) pdl_wait();
  // this CTA's items: a contiguous, balanced share of (job, row block) in
  // job order, so consecutive items of a CTA read the same activation rows
  const int n_items = (MODE == DOWN ? __ldcg(a.n_jobs) : *a.n_jobs) * geo.nrb;
  const int per = n_items / (int)gridDim.x, extra = n_items % (int)gridDim.x;
  const int first = (int)blockIdx.x * per + min((int)blockIdx.x, extra);
  const int count = per + ((int)blockIdx.x < extra ? 1 : 0);
  float* red = reinterpret_cast<float*>(smem + (size_t)geo.ns * geo.stage);   // [KS][RTP][2][4][32]

  if (threadIdx.x == 0) {
    for (int i = 0; i < geo.ns; ++i) {
      tc::mbar_init(tc::smem_u32(&full_bar[i]), 1);
      tc::mbar_init(tc::smem_u32(&empty_bar[i]), NW);   // one arrival per consumer warp
    }
    tc::fence_mbar_init();
    abort_s = 0;
  }
  __syncthreads();

  if (warp == NW) {
    // ---------------- producer: one lane issues every copy
    if (lane == 0) {
      int cur_j = -1, cur_e = 0, cur_tok0 = 0, cur_ntok = 0, cur_row[kJobTokens];
      const uint32_t x_bytes = (uint32_t)a.K * 2u;
      int n0 = 0;
      if (MODE == DOWN) {
        // the first stages: weights and scales now, the activation rows (and
        // the stage's one arrival) after the wait
        const int pre = min(geo.ns, count);
        for (int n = 0; n < pre; ++n) {
          const int it = first + n, j = it / geo.nrb, rb = it - j * geo.nrb;
          if (j != cur_j) {
            cur_j = j;
            const int job = __ldcg(a.jobs + j);
            cur_e = job & 0x1FF;
            cur_tok0 = (job >> 9) & 0xFFF;
            cur_ntok = (job >> 21) & 0x1F;
            for (int r = 0; r < kJobTokens; ++r) cur_row[r] = r < cur_ntok ? cur_tok0 + r : -1;
          }
          ItemInfo& inf = info_s[n];
          inf.tok0 = cur_tok0;
          inf.ntok = cur_ntok;
          inf.rb = rb;
          for (int r = 0; r < kJobTokens; ++r) inf.row[r] = cur_row[r];
          if (it + 1 == a.drop_item1) continue;
          const uint32_t base = tc::smem_u32(smem + (size_t)n * geo.stage);
          const uint32_t bar = tc::smem_u32(&full_bar[n]);
          mbar_expect_tx(bar, geo.w_bytes + geo.s_bytes);
          const uint8_t* wsrc = a.W + (size_t)cur_e * a.w_expert_stride + (size_t)rb * geo.w_bytes;
          for (uint32_t off = 0; off < geo.w_bytes; off += 16384u) {
            const uint32_t len = min(16384u, geo.w_bytes - off);
            bulk_g2s(base + off, wsrc + off, len, bar);
          }
          const uint32_t* ssrc = a.S + (size_t)cur_e * a.s_expert_stride + (size_t)rb * (geo.s_bytes / 4);
          bulk_g2s(base + geo.w_bytes, ssrc, geo.s_bytes, bar);
        }
        pdl_wait();
        for (int n = 0; n < pre; ++n) {
          if (first + n + 1 == a.drop_item1) continue;
          const ItemInfo& inf = info_s[n];
          const uint32_t base = tc::smem_u32(smem + (size_t)n * geo.stage);
          const uint32_t bar = tc::smem_u32(&full_bar[n]);
          mbar_arrive_expect_tx(bar, (uint32_t)inf.ntok * x_bytes);
          for (int r = 0; r < inf.ntok; ++r)
            bulk_g2s(base + geo.w_bytes + geo.s_bytes + (uint32_t)r * geo.x_stride,
                     static_cast<const uint8_t*>(a.X) + (size_t)inf.row[r] * a.ldx * 2, x_bytes, bar);
        }
        n0 = pre;
      }
      if (MODE == GATEUP && count == 0) pdl_trigger();
      for (int n = n0; n < count; ++n) {
        const int it = first + n, s = n % geo.ns;
        if (MODE == GATEUP && n == count - 1) pdl_trigger();   // the CTA's last item: its dependents may launch
        if (n >= geo.ns) {
          if (!tc::mbar_wait(tc::smem_u32(&empty_bar[s]), ((n / geo.ns) - 1) & 1, kStagedWaitLimit)) {
            if (a.err) atomicExch(a.err, 5);
            break;   // the consumers time out on this stage's full barrier and stop
          }
          tc::fence_proxy_async_smem();
        }
        const int j = it / geo.nrb, rb = it - j * geo.nrb;
        if (j != cur_j) {   // consecutive items of a CTA mostly share their job: decode it once
          cur_j = j;
          const int job = a.jobs[j];
          cur_e = job & 0x1FF;
          cur_tok0 = (job >> 9) & 0xFFF;
          cur_ntok = (job >> 21) & 0x1F;
          for (int r = 0; r < kJobTokens; ++r)
            cur_row[r] = r < cur_ntok ? (MODE == GATEUP ? a.pair_token[cur_tok0 + r] : cur_tok0 + r) : -1;
        }
        const int e = cur_e, tok0 = cur_tok0, ntok = cur_ntok;
        ItemInfo& inf = info_s[s];
        inf.tok0 = tok0;
        inf.ntok = ntok;
        inf.rb = rb;
        for (int r = 0; r < kJobTokens; ++r) inf.row[r] = cur_row[r];
        // failure-detection tests: this item's copies are never issued, so the
        // stage's full barrier never completes and the consumers give up
        if (it + 1 == a.drop_item1) continue;
        const uint32_t base = tc::smem_u32(smem + (size_t)s * geo.stage);
        const uint32_t bar = tc::smem_u32(&full_bar[s]);
        mbar_arrive_expect_tx(bar, geo.w_bytes + geo.s_bytes + (uint32_t)ntok * x_bytes);
        const uint8_t* wsrc = a.W + (size_t)e * a.w_expert_stride + (size_t)rb * geo.w_bytes;
        for (uint32_t off = 0; off < geo.w_bytes; off += 16384u) {
          const uint32_t len = min(16384u, geo.w_bytes - off);
          bulk_g2s(base + off, wsrc + off, len, bar);
        }
        const uint32_t* ssrc = a.S + (size_t)e * a.s_expert_stride + (size_t)rb * (geo.s_bytes / 4);
        bulk_g2s(base + geo.w_bytes, ssrc, geo.s_bytes, bar);
        for (int r = 0; r < ntok; ++r)
          bulk_g2s(base + geo.w_bytes + geo.s_bytes + (uint32_t)r * geo.x_stride,
                   static_cast<const uint8_t*>(a.X) + (size_t)inf.row[r] * a.ldx * 2, x_bytes, bar);
      }
    }
    return;
  }

  if (MODE == DOWN) pdl_wait();   // before any write of this launch (its rows arrive after it anyway)
  // ---------------- consumers: warp (rtp, ks) takes chunks [ks * CPW, +CPW)
  // of tiles 2 rtp and 2 rtp + 1 of the item
  const int ks = warp % KS, rtp = warp / KS;
  const int c0 = ks * CPW;
  // consumer groups: the row pairs rtp = grp, grp + NGRP, ... share a named
  // barrier and their own epilogue, so the groups' compute and epilogue
  // phases drift apart instead of running in lockstep
  const int NGRP = RTP < 8 ? RTP : 8;
  const int grp = rtp % NGRP, per_grp = RTP / NGRP;
  const int gthreads = per_grp * KS * 32;
  const int gtid = ((rtp / NGRP) * KS + ks) * 32 + lane;
  const int bar_id = 1 + grp;
  int n = 0;
  for (; n < count; ++n) {
    const int s = n % geo.ns;
    if (!tc::mbar_wait(tc::smem_u32(&full_bar[s]), (n / geo.ns) & 1, kStagedWaitLimit)) abort_s = 1;
    consumer_sync(bar_id, gthreads);
    if (abort_s) break;
    const int tok0 = info_s[s].tok0, ntok = info_s[s].ntok, rb = info_s[s].rb;
    const unsigned char* st = smem + (size_t)s * geo.stage;
    const uint4* ws = reinterpret_cast<const uint4*>(st);
    const uint32_t* ss = reinterpret_cast<const uint32_t*>(st + geo.w_bytes);
    // rows past ntok hold stale bytes: they only feed MMA columns that are never stored
    const unsigned char* xrow = st + geo.w_bytes + geo.s_bytes + (size_t)(lane >> 2) * geo.x_stride + (lane & 3) * 16;
    // this warp's operands of the item -> registers, then the stage is released
    // at once, so its refill overlaps the warp's MMAs
    uint4 wreg[CPW][2], xreg[CPW][2];
    uint32_t sreg[CPW][2][kSpc];
#pragma unroll
    for (int j = 0; j < CPW; ++j) {
      const int c = c0 + j;
      xreg[j][0] = *reinterpret_cast<const uint4*>(xrow + (size_t)c * kChunkK * 2);
      xreg[j][1] = *reinterpret_cast<const uint4*>(xrow + (size_t)c * kChunkK * 2 + 64);
#pragma unroll
      for (int rt = 0; rt < 2; ++rt) {
        const int lt = rtp * 2 + rt;
        wreg[j][rt] = ws[(lt * NC + c) * 32 + lane];
#pragma unroll
        for (int q = 0; q < kSpc; ++q) {
          const int grp = G >= kChunkK ? (c * kChunkK) / G : c * kSpc + q;
          sreg[j][rt][q] = ss[(lt * NG + grp) * 8 + (lane >> 2)];
        }
      }
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(tc::smem_u32(&empty_bar[s]));
    float acc[2][4], tmp[2][4];
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[rt][c] = 0.f;
#pragma unroll
    for (int j = 0; j < CPW; ++j) {
      const uint4 xv0 = xreg[j][0], xv1 = xreg[j][1];
#pragma unroll
      for (int rt = 0; rt < 2; ++rt) {
        const uint4 wv = wreg[j][rt];
        const uint32_t(&sw)[kSpc] = sreg[j][rt];
        const uint32_t wwords[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
        for (int st4 = 0; st4 < 4; ++st4) {
          const int gs = j * 4 + st4;
          uint32_t af[4];
          dq_word(wwords[st4], af);
          if (gs % kSpg == 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q) tmp[rt][q] = 0.f;
          }
          const uint4& xv = (st4 >> 1) ? xv1 : xv0;
          const uint32_t b0 = (st4 & 1) ? xv.z : xv.x, b1 = (st4 & 1) ? xv.w : xv.y;
          mma_f16(tmp[rt], af, b0, b1);
          if ((gs + 1) % kSpg == 0) {
            const uint32_t w2 = sw[G >= kChunkK ? 0 : (st4 * 16) / G];
            const float slo = half_lo(w2), shi = half_hi(w2);
            acc[rt][0] = fmaf(slo, tmp[rt][0], acc[rt][0]);
            acc[rt][1] = fmaf(slo, tmp[rt][1], acc[rt][1]);
            acc[rt][2] = fmaf(shi, tmp[rt][2], acc[rt][2]);
            acc[rt][3] = fmaf(shi, tmp[rt][3], acc[rt][3]);
          }
        }
      }
    }
#pragma unroll
    for (int rt = 0; rt < 2; ++rt)
#pragma unroll
      for (int c = 0; c < 4; ++c) red[((((ks * RTP + rtp) * 2 + rt) * 4 + c) * 32) + lane] = acc[rt][c];
    consumer_sync(bar_id, gthreads);   // the group's partials are in

    // epilogue of the group's row pairs: unit (rp, rt, j, lane) -> rows
    // (g, g + 8), token 2t + j; partials in ks order
    for (int uix = gtid; uix < per_grp * 128; uix += gthreads) {
      const int l = uix & 31, jj = (uix >> 5) & 1, rt = (uix >> 6) & 1, rp = grp + NGRP * (uix >> 7);
      const int token = 2 * (l & 3) + jj;
      if (token >= ntok) continue;
      float v0 = 0.f, v1 = 0.f;
      for (int k2 = 0; k2 < KS; ++k2) {
        const int b4 = ((k2 * RTP + rp) * 2 + rt) * 4;
        v0 += red[(b4 + jj) * 32 + l];
        v1 += red[(b4 + jj + 2) * 32 + l];
      }
      const int tile = (rb * RTP + rp) * 2 + rt;
      const size_t m = (size_t)tok0 + token;
      if (MODE == GATEUP) {
        const int f = tile * 8 + (l >> 2);
        const float sv0 = v0 / (1.f + expf(-v0));
        a.act16[m * a.F + f] = __float2half_rn(round_bf16(sv0 * v1));
      } else {
        const int r0 = tile * 16 + (l >> 2);
        a.out[m * a.H + r0] = v0;
        a.out[m * a.H + r0 + 8] = v1;
      }
    }
    consumer_sync(bar_id, gthreads);   // the partials are read before the next item overwrites them
  }
  if (abort_s) {
    if (threadIdx.x == 0 && a.err) atomicExch(a.err, 5);
    // let the copies already issued for this CTA land before it exits
    for (int m = n; m < n + geo.ns && m < count; ++m)
      tc::mbar_wait(tc::smem_u32(&full_bar[m % geo.ns]), (m / geo.ns) & 1, kStagedWaitLimit);
  }
}

}  // namespace mma
}  // namespace bm
