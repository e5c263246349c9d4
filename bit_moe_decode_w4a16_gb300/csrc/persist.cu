// The decode step of a small batch (B <= 8 rows) as one persistent,
// cooperative kernel: all layers' QKV projection, attention, output
// projection, routing, expert gate/up and down with the top-k combine run in
// a single launch of one CTA per SM, the phases separated by grid-wide
// barriers instead of kernel boundaries.  This is the solo / small-batch
// path the batched-serving pages keep beside the batched kernels ([KV-slot
// isolation] follow-up update: a lone request through the batched path is a
// few percent slower than the solo kernel).
//
// Same bits as the multi-kernel step.  Every output is computed with the
// arithmetic of the kernel it replaces, in the same order:
//   - projections (dense and expert): the warp-MMA split of w4_mma.cuh — a
//     16-row tile's output is the sum, in ks order, of KS partials, each over
//     CPW = 4 chunks of 64 along K with the per-group scale applied by fmaf
//     (w4_mma_shape.h fixes KS from the shape alone);
//   - attention and routing: the very same device functions as the
//     multi-kernel step (attn_fused.cuh, route_dev.cuh);
//   - the top-k combine and the next RMSNorm: the arithmetic of
//     k_combine_norm, its 1024-thread reduction replayed thread for thread.
// So a stream's bytes do not depend on which path ran its step.
//
// Warp roles.  Warps 0-15 compute; warp 16 is the weight producer: one lane
// streams, in the order the compute warps consume them, weight "items" into a
// byte ring in shared memory with cp.async.bulk.  An item is one tile job, a
// 16-row tile of a matrix over its whole K (contiguous in the mma layout:
// 16 KB of int4 for K = 2048, and its scales), copied with one bulk copy per
// 16 KB and counted in bytes on the item's `full` mbarrier; it is consumed in
// "units" of 256 of K (2 KB) by the compute warps, which copy a unit to
// registers and count it off; the last one releases the item (`empty`
// mbarrier).  Few large copies keep many bytes in flight per SM.  The dense weights do
// not depend on the data, so the producer runs ahead across phases and layers
// (the next layer's QKV and output projection arrive while the experts of
// this one compute); the expert units wait for this CTA's routing (the
// `route` mbarrier, armed by the compute warps after their top-k).
//
// Phases of a layer, each ending in a grid barrier:
//   1. QKV: this CTA's 16-row tiles T = cta, cta + grid, ...; the input rows
//      are RMSNorm(x) (layer 0: the embedding kernel's), staged as fp16;
//   2. attention: work items (stream, kv head, chunk) over the CTAs, warps
//      0-7, chunk records merged by the last arriving CTA;
//   3. output projection + residual;
//   4. router logits: items (8 experts, token), warps 0-7;
//   5. every CTA takes the softmax top-k of all rows and groups the (row,
//      rank) pairs by expert itself (the same integers everywhere), then the
//      gate/up tiles (expert, 16-row tile) = cta, cta + grid, ...;
//   6. down: CTA c takes 16-row output tile c for all active experts, then
//      combines its rows: y = h + sum_r w_r out_r in rank order.
// A grid barrier is one release-add per CTA on a counter that is zero at
// launch and an acquire poll until it reaches (barrier number) x grid; every
// poll loop is bounded (about a second), after which the CTA records error
// code 6 and every CTA leaves at its next barrier.
#include "attn_fused.cuh"
#include "persist.h"
#include "route_dev.cuh"
#include "tc_ptx.cuh"
#include "w4_mma.cuh"

#include <algorithm>

namespace bm {

namespace {

using namespace mma;

constexpr int kPCompute = 16;                 // compute warps
constexpr int kPThreads = (kPCompute + 1) * 32;
constexpr int kPCThreads = kPCompute * 32;
constexpr int kUnitChunks = 4;                // CPW: chunks of 64 along K per unit
constexpr int kUnitW = kUnitChunks * 512;     // weight bytes of a unit
constexpr int kRoundUnits = 32;               // units per reduction round
constexpr int kMaxItems = 64;                 // weight items in flight per CTA
constexpr int kPMaxPairs = 64;
constexpr int kPMaxE = 256;
constexpr int kBarCompute = 1, kBarGroup = 2;
constexpr unsigned long long kPWaitNs = 1000000000ull;   // a bounded wait gives up after about a second
constexpr int kPErr = 6;
constexpr int kGUTiles = 1;                   // gate/up tiles per weight item (one expert's consecutive tiles)
constexpr int kMaxGUJobs = 64;                // gate/up tile jobs of one CTA
constexpr uint32_t kCopyMax = 65536;          // bytes per bulk copy: the per-copy cost is paid per copy, not per byte

struct PSmem {
  uint64_t full[kMaxItems], empty[kMaxItems], route;   // per weight item (descriptor d = item % kMaxItems)
  unsigned long long it_v[kMaxItems];   // producer: virtual ring offset of the item
  uint32_t it_off[kMaxItems];           // ring offset of the item's bytes
  int it_cnt[kMaxItems];                // units of the item consumed so far
  int ids[kPMaxPairs], rank[kPMaxPairs], pos_of[kPMaxPairs], pair_token[kPMaxPairs];
  float w[kPMaxPairs];
  int cnt[kPMaxE], off[kPMaxE + 1];
  int active_e[kPMaxPairs], active_off[kPMaxPairs + 1];
  int n_active;
  float out[kPMaxPairs][16];      // down outputs of this CTA's tile, [sorted pair][row]
  float rnorm[kPMaxRows][32];     // RMSNorm partial sums of the 32 warps of the replayed reduction
  float router_red[routedev::kRouterWarps];
  float hres[kPMaxRows][16];      // the residual rows of this CTA's down tile, for the combine
  short gu_item[kMaxGUJobs], gu_tt[kMaxGUJobs], gu_n[kMaxGUJobs];   // gate/up job -> item, tile in item, tiles
  int gu_items;
  int abort;   // set by any thread of the CTA that gives up
  int stop;    // thread 0's copy of abort at the last grid barrier
};

struct NamedSync {
  int id, n;
  __device__ __forceinline__ void operator()() const { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
};

__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t mbar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(mbar)
               : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void arrive_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}

// Wait for an mbarrier phase; gives up after about a second, or at once when
// the CTA is aborting.
__device__ __forceinline__ bool pwait(uint32_t mbar, uint32_t parity, const volatile int* abort) {
  const unsigned long long t0 = now_ns();
  for (;;) {
    if (tc::mbar_wait(mbar, parity, 64)) return true;
    if (*abort || now_ns() - t0 > kPWaitNs) return false;
  }
}

__device__ __forceinline__ void fail(const PersistArgs& a, PSmem& ps) {
  ps.abort = 1;
  if (a.err) atomicCAS(a.err, 0, kPErr);
}

// Grid barrier of the compute warps (see the file comment).  Returns false if
// the step is being abandoned.
// The decision to go on is taken by thread 0 alone and read by all after the
// second named barrier, so the compute warps never diverge around a barrier.
__device__ __forceinline__ bool grid_barrier(const PersistArgs& a, PSmem& ps, unsigned& nbar) {
  NamedSync{kBarCompute, kPCThreads}();
  ++nbar;
  if (threadIdx.x == 0) {
    if (!*reinterpret_cast<volatile int*>(&ps.abort)) {
      __threadfence();
      red_release_add(a.bar, 1u);
      const unsigned target = nbar * gridDim.x;
      const unsigned long long t0 = now_ns();
      unsigned polls = 0;
      while (ld_acquire(a.bar) < target) {
        if ((++polls & 63u) == 0u &&
            (*reinterpret_cast<volatile int*>(a.err) != 0 || now_ns() - t0 > kPWaitNs)) {
          fail(a, ps);
          break;
        }
      }
    }
    ps.stop = *reinterpret_cast<volatile int*>(&ps.abort);
  }
  NamedSync{kBarCompute, kPCThreads}();
  return !ps.stop;
}

// ---------------------------------------------------------------- units
// A unit is 256 of K of a 16-row tile: 4 chunks of 64 (2 KB of int4 in the
// mma layout) and the scale words of their groups; a tile's units are
// contiguous, and so are its scale words.
template <int G>
__host__ __device__ constexpr uint32_t unit_s_bytes() {
  return (uint32_t)(kUnitChunks * 64 / G) * 32u;
}

// One unit's partial sums by one warp: the operands come from the slot
// (released as soon as they are in registers) and the staged activation row
// of the lane's token column (null: a column that is never stored; zeros).
// The arithmetic is the consumer step of the staged expert kernel
// (w4_mma_staged.cuh), which is that of k_w4_mma.
template <int G>
__device__ __forceinline__ void unit_mma(const unsigned char* wp, const unsigned char* sp, PSmem& ps, int d, int KS,
                                         const __half* xrow, int c0, float (&acc)[4]) {
  constexpr int kSpg = G / 16;
  constexpr int kSpc = G >= kChunkK ? 1 : kChunkK / G;
  const int lane = threadIdx.x & 31;
  uint4 wreg[kUnitChunks], xreg[kUnitChunks][2];
  uint32_t sreg[kUnitChunks][kSpc];
  const uint4* ws = reinterpret_cast<const uint4*>(wp);
  const uint32_t* ss = reinterpret_cast<const uint32_t*>(sp);
#pragma unroll
  for (int j = 0; j < kUnitChunks; ++j) {
    wreg[j] = ws[j * 32 + lane];
#pragma unroll
    for (int q = 0; q < kSpc; ++q) {
      const int grp = G >= kChunkK ? (j * kChunkK) / G : j * kSpc + q;   // within the unit
      sreg[j][q] = ss[grp * 8 + (lane >> 2)];
    }
    if (xrow) {
      const __half* p = xrow + (size_t)(c0 + j) * kChunkK + (lane & 3) * 8;
      xreg[j][0] = *reinterpret_cast<const uint4*>(p);
      xreg[j][1] = *reinterpret_cast<const uint4*>(p + 32);
    } else {
      xreg[j][0] = xreg[j][1] = make_uint4(0, 0, 0, 0);
    }
  }
  __syncwarp();
  if (lane == 0 && atomicAdd(&ps.it_cnt[d], 1) == KS - 1) {   // the item's last unit: release it
    ps.it_cnt[d] = 0;
    tc::mbar_arrive(tc::smem_u32(&ps.empty[d]));
  }
  float tmp[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) acc[c] = 0.f;
#pragma unroll
  for (int j = 0; j < kUnitChunks; ++j) {
    const uint32_t wwords[4] = {wreg[j].x, wreg[j].y, wreg[j].z, wreg[j].w};
#pragma unroll
    for (int st4 = 0; st4 < 4; ++st4) {
      const int gs = j * 4 + st4;
      uint32_t af[4];
      dq_word(wwords[st4], af);
      if (gs % kSpg == 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) tmp[q] = 0.f;
      }
      const uint4& xv = xreg[j][st4 >> 1];
      const uint32_t b0 = (st4 & 1) ? xv.z : xv.x, b1 = (st4 & 1) ? xv.w : xv.y;
      mma_f16(tmp, af, b0, b1);
      if ((gs + 1) % kSpg == 0) {
        const uint32_t w2 = sreg[j][G >= kChunkK ? 0 : (st4 * 16) / G];
        const float slo = half_lo(w2), shi = half_hi(w2);
        acc[0] = fmaf(slo, tmp[0], acc[0]);
        acc[1] = fmaf(slo, tmp[1], acc[1]);
        acc[2] = fmaf(shi, tmp[2], acc[2]);
        acc[3] = fmaf(shi, tmp[3], acc[3]);
      }
    }
  }
}

enum PMode { P_QKV = 0, P_OPROJ = 1, P_GATEUP = 2, P_DOWN = 3 };

// Shared-memory plan (dynamic): ring | reduction buffer | phase union.
struct PPtrs {
  unsigned char* ring;
  float* red;
  unsigned char* uni;
};

// Stage `rows` activation rows of K fp16 values (row stride ld in global,
// xs in shared) with 16-byte loads; rows past `rows` are not touched (their
// columns are never stored).
__device__ __forceinline__ void stage_rows(__half* dst, int xs, const __half* src, int ld, int rows, int K) {
  const int per = K / 8;
  for (int i = threadIdx.x; i < rows * per; i += kPCThreads) {
    const int r = i / per, c = i - r * per;
    *reinterpret_cast<uint4*>(dst + (size_t)r * xs + c * 8) =
        *reinterpret_cast<const uint4*>(src + (size_t)r * ld + c * 8);
  }
}

// RMSNorm of the B rows of the residual stream x, as k_combine_norm computes
// it: 1024 threads, thread t summing y[h]^2 for h = t, t + 1024, ... with
// fmaf, each warp's butterfly, then the 32 warp sums in order; then
// round_bf16(y * rinv * nw).  Compute thread c plays threads c and c + 512.
// The rows are first staged in shared memory (ys, B x H bf16) with all
// loads in flight at once.  xs_dst: fp16 rows to shared memory (stride xs);
// else bf16 rows to global g_dst.
__device__ __forceinline__ void norm_rows(const PersistArgs& a, PSmem& ps, const bf16* nw, bf16* ys,
                                          __half* xs_dst, int xs, bf16* g_dst) {
  const int H = a.H, B = a.B, ct = threadIdx.x, warp = ct >> 5, lane = ct & 31;
  stage_rows(reinterpret_cast<__half*>(ys), H, reinterpret_cast<const __half*>(a.x), H, B, H);
  NamedSync{kBarCompute, kPCThreads}();
  for (int b = 0; b < B; ++b) {
    const bf16* y = ys + (size_t)b * H;
#pragma unroll
    for (int hv = 0; hv < 2; ++hv) {
      const int vt = ct + hv * kPCThreads;   // the replayed thread
      float ss = 0.f;
      for (int h = vt; h < H; h += 2 * kPCThreads) {
        const float v = bf2f(y[h]);
        ss = fmaf(v, v, ss);
      }
      ss = warp_sum(ss);
      if (lane == 0) ps.rnorm[b][warp + hv * kPCompute] = ss;
    }
  }
  NamedSync{kBarCompute, kPCThreads}();
  for (int b = 0; b < B; ++b) {
    float tot = 0.f;
    for (int w = 0; w < 32; ++w) tot += ps.rnorm[b][w];
    const float r = 1.0f / sqrtf(tot / (float)H + a.eps);
    const bf16* y = ys + (size_t)b * H;
    for (int h = ct; h < H; h += kPCThreads) {
      const float v = round_bf16(bf2f(y[h]) * r * (nw ? bf2f(nw[h]) : 1.f));
      if (xs_dst) xs_dst[(size_t)b * xs + h] = __float2half_rn(v);
      else g_dst[(size_t)b * H + h] = f2bf(v);
    }
  }
  NamedSync{kBarCompute, kPCThreads}();
}

}  // namespace

// The kernel.  Template: head dimension D and int4 group size G.
template <int D, int G>
__global__ void __launch_bounds__(kPThreads, 1) k_persist_step(PersistArgs a) {
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ __align__(16) PSmem ps;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x, grid = gridDim.x;
  const PersistGeo& geo = a.geo;
  PPtrs p{dsm + geo.ring_off, reinterpret_cast<float*>(dsm + geo.red_off), dsm + geo.uni_off};
  constexpr uint32_t kSBytes = unit_s_bytes<G>();
  const uint32_t R = geo.ring_bytes;
  const int H = a.H, B = a.B, F = a.F, E = a.E, K = a.k;
  const int KSq = (H / 64) / kUnitChunks, KSo = (a.qd / 64) / kUnitChunks, KSd = (F / 64) / kUnitChunks;
  const int NTq = a.qkv_rows / 16, NTo = H / 16, NTg = 2 * F / 16, NTd = H / 16;
  const int nEB = E / 8;   // router items per token: 8 experts each

  if (threadIdx.x == 0) {
    for (int i = 0; i < kMaxItems; ++i) {
      tc::mbar_init(tc::smem_u32(&ps.full[i]), 1);
      tc::mbar_init(tc::smem_u32(&ps.empty[i]), 1);
      ps.it_cnt[i] = 0;
    }
    tc::mbar_init(tc::smem_u32(&ps.route), 1);
    tc::fence_mbar_init();
    ps.abort = 0;
    ps.stop = 0;
  }
  __syncthreads();

  if (warp == kPCompute) {
    // ================================================================ producer
    if (lane != 0) return;
    unsigned nit = 0, oldest = 0;   // items issued; items seen released
    unsigned long long vhead = 0;    // virtual ring offset: physical = v % R
    bool ok = true;
    // One item: [wb bytes of int4 | sb bytes of scales] at a ring offset
    // where it does not wrap, once the items that held those bytes (and the
    // item's descriptor) are released.
    auto issue = [&](const uint8_t* wsrc, uint32_t wb, const uint32_t* ssrc, uint32_t sb) {
      const uint32_t S = wb + sb;
      unsigned long long v = vhead;
      if (v % R + S > R) v = (v / R + 1) * R;
      while (oldest < nit && (v + S - ps.it_v[oldest % kMaxItems] > R || nit - oldest >= (unsigned)kMaxItems)) {
        if (!pwait(tc::smem_u32(&ps.empty[oldest % kMaxItems]), (oldest / kMaxItems) & 1, &ps.abort)) {
          ok = false;
          return;
        }
        ++oldest;
      }
      tc::fence_proxy_async_smem();
      const int d = (int)(nit % kMaxItems);
      ps.it_v[d] = v;
      vhead = v + S;
      const uint32_t off = (uint32_t)(v % R);
      ps.it_off[d] = off;
      if (++nit == (unsigned)a.drop_unit1) return;   // failure-detection tests: this item never arrives
      const uint32_t dst = tc::smem_u32(p.ring + off);
      const uint32_t bar = tc::smem_u32(&ps.full[d]);
      arrive_expect_tx(bar, S);
      for (uint32_t o = 0; o < wb; o += kCopyMax) bulk_g2s(dst + o, wsrc + o, min(kCopyMax, wb - o), bar);
      bulk_g2s(dst + wb, ssrc, sb, bar);
    };
    const uint32_t wbH = (uint32_t)(H / 64) * 512u, sbH = (uint32_t)(H / G) * 32u;
    const uint32_t wbO = (uint32_t)(a.qd / 64) * 512u, sbO = (uint32_t)(a.qd / G) * 32u;
    const uint32_t wbF = (uint32_t)(F / 64) * 512u, sbF = (uint32_t)(F / G) * 32u;
    for (int l = 0; l < a.layers && ok; ++l) {
      const PersistLayer& Lw = a.L[l];
      for (int T = cta; T < NTq && ok; T += grid)
        issue(Lw.wqkv + (size_t)T * wbH, wbH, Lw.sqkv + (size_t)T * (sbH / 4), sbH);
      for (int T = cta; T < NTo && ok; T += grid)
        issue(Lw.wo + (size_t)T * wbO, wbO, Lw.so + (size_t)T * (sbO / 4), sbO);
      // this CTA's router rows to L2 ahead of the routing phase
      for (int i = cta; i < nEB * B; i += grid) {
        const float* wr = Lw.wr + (size_t)(i % nEB) * 8 * H;
        for (uint32_t off = 0; off < (uint32_t)(8 * H * 4); off += 16384u)
          prefetch_l2(reinterpret_cast<const unsigned char*>(wr) + off, min(16384u, (uint32_t)(8 * H * 4) - off));
      }
      if (!ok) break;
      if (!pwait(tc::smem_u32(&ps.route), (uint32_t)(l & 1), &ps.abort)) { ok = false; break; }
      const int U = ps.n_active;
      // gate/up: this CTA's contiguous range of (expert, tile) jobs, expert
      // major, in items of up to kGUTiles consecutive tiles of one expert
      const int J = U * NTg;
      const int jb = (int)((long long)J * cta / grid), je = (int)((long long)J * (cta + 1) / grid);
      for (int j = jb; j < je && ok;) {
        const int u = j / NTg, T = j - u * NTg, nt = min(min(kGUTiles, je - j), NTg - T);
        const int e = ps.active_e[u];
        issue(Lw.wg + (size_t)e * a.wg_stride + (size_t)T * wbH, (uint32_t)nt * wbH,
              Lw.sg + (size_t)e * a.sg_stride + (size_t)T * (sbH / 4), (uint32_t)nt * sbH);
        j += nt;
      }
      for (int T = cta; T < NTd && ok; T += grid)
        for (int u = 0; u < U && ok; ++u) {
          const int e = ps.active_e[u];
          issue(Lw.wd + (size_t)e * a.wd_stride + (size_t)T * wbF, wbF,
                Lw.sd + (size_t)e * a.sd_stride + (size_t)T * (sbF / 4), sbF);
        }
    }
    if (!ok) fail(a, ps);
    // the copies still in flight land before this thread (and so the CTA) exits
    for (unsigned m = nit > (unsigned)kMaxItems ? nit - kMaxItems : 0u; m < nit; ++m)
      tc::mbar_wait(tc::smem_u32(&ps.full[m % kMaxItems]), (m / kMaxItems) & 1, 1u << 16);
    return;
  }

  // ================================================================ compute warps
  unsigned nit = 0;    // items consumed (the producer's order)
  unsigned nbar = 0;   // grid barriers passed
  __half* xs16 = reinterpret_cast<__half*>(p.uni);

  // One phase of tile jobs: job j (0 <= j < nj) has KS units and sits in
  // weight item place(j) = (item, tile in item, tiles of the item) of the
  // phase's n_items items; rounds of whole jobs (at most kRoundUnits units);
  // col(j, g) = the staged row of token column g of job j (or -1);
  // epi(j, l, jj, v0, v1) stores a result.
  auto run_jobs = [&](int nj, int KS, int n_items, int xstride, auto place, auto col, auto epi) {
    const int per_round = kRoundUnits / KS;
    for (int j0 = 0; j0 < nj; j0 += per_round) {
      const int rj = min(per_round, nj - j0), nu = rj * KS;
      for (int i = warp; i < nu; i += kPCompute) {
        const int jl = i / KS, ks = i - jl * KS;
        const int3 pl = place(j0 + jl);
        const unsigned it = nit + (unsigned)pl.x;
        const int d = (int)(it % kMaxItems);
        float acc[4];
        if (!pwait(tc::smem_u32(&ps.full[d]), (it / kMaxItems) & 1, &ps.abort)) {
          if (lane == 0) fail(a, ps);
          for (int c = 0; c < 4; ++c) acc[c] = 0.f;
        } else {
          const int r = col(j0 + jl, lane >> 2);
          const unsigned char* item = p.ring + ps.it_off[d];
          const int un = pl.y * KS + ks;   // unit within the item
          unit_mma<G>(item + (size_t)un * kUnitW, item + (size_t)pl.z * KS * kUnitW + (size_t)un * kSBytes, ps, d,
                      pl.z * KS, r >= 0 ? xs16 + (size_t)r * xstride : nullptr, ks * kUnitChunks, acc);
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) p.red[(i * 4 + c) * 32 + lane] = acc[c];
      }
      NamedSync{kBarCompute, kPCThreads}();
      for (int idx = threadIdx.x; idx < rj * 64; idx += kPCThreads) {
        const int jl = idx >> 6, jj = (idx >> 5) & 1, l = idx & 31;
        float v0 = 0.f, v1 = 0.f;
        for (int k2 = 0; k2 < KS; ++k2) {
          const int b4 = (jl * KS + k2) * 4;
          v0 += p.red[(b4 + jj) * 32 + l];
          v1 += p.red[(b4 + jj + 2) * 32 + l];
        }
        epi(j0 + jl, l, jj, v0, v1);
      }
      NamedSync{kBarCompute, kPCThreads}();
    }
    nit += (unsigned)n_items;
  };
  auto one = [](int j) { return make_int3(j, 0, 1); };   // one tile per item

  for (int l = 0; l < a.layers; ++l) {
    const PersistLayer& Lw = a.L[l];

    // ---------------- 1. QKV of RMSNorm(x)
    const int xq = H + 32;
    if (l == 0) {
      stage_rows(xs16, xq, a.xn16, H, B, H);
      NamedSync{kBarCompute, kPCThreads}();
    } else {
      norm_rows(a, ps, Lw.attn_nw, reinterpret_cast<bf16*>(xs16 + (size_t)B * xq), xs16, xq, nullptr);
    }
    {
      const int njq = cta < NTq ? (NTq - 1 - cta) / grid + 1 : 0;
      run_jobs(njq, KSq, njq, xq, one, [&](int, int g) { return g < B ? g : -1; },
               [&](int j, int ll, int jj, float v0, float v1) {
                 const int T = cta + j * grid, m = 2 * (ll & 3) + jj;
                 if (m >= B) return;
                 const int r0 = T * 16 + (ll >> 2);
                 a.qkv[(size_t)m * a.qkv_rows + r0] = f2bf(v0);
                 a.qkv[(size_t)m * a.qkv_rows + r0 + 8] = f2bf(v1);
               });
    }
    if (!grid_barrier(a, ps, nbar)) break;

    // ---------------- 2. attention (warps 0-7)
    if (warp < attnf::kWarpsA) {
      AttnFusedArgs at = a.at;
      at.layer = l;
      attnf::AttnSmem<D>& sm = *reinterpret_cast<attnf::AttnSmem<D>*>(p.uni);
      const NamedSync gs{kBarGroup, attnf::kAttnThreads};
      const int total = attnf::attn_prologue<D>(at, sm, cta == 0, gs);
      for (int it = cta; it < total; it += grid) attnf::attn_item<D>(at, sm, it, gs);
    }
    if (!grid_barrier(a, ps, nbar)) break;

    // ---------------- 3. output projection + residual
    const int xo = a.qd + 32;
    stage_rows(xs16, xo, a.attn, a.qd, B, a.qd);
    NamedSync{kBarCompute, kPCThreads}();
    {
      const int njo = cta < NTo ? (NTo - 1 - cta) / grid + 1 : 0;
      run_jobs(njo, KSo, njo, xo, one, [&](int, int g) { return g < B ? g : -1; },
               [&](int j, int ll, int jj, float v0, float v1) {
                 const int T = cta + j * grid, m = 2 * (ll & 3) + jj;
                 if (m >= B) return;
                 const int r0 = T * 16 + (ll >> 2);
                 const size_t o = (size_t)m * H + r0;
                 a.h[o] = f2bf(v0 + bf2f(a.x[o]));
                 a.h[o + 8] = f2bf(v1 + bf2f(a.x[o + 8]));
               });
    }
    if (!grid_barrier(a, ps, nbar)) break;

    // ---------------- 4. router logits (warps 0-7)
    if (warp < routedev::kRouterWarps) {
      MoeArgs ma = a.moe;
      ma.wr = Lw.wr;
      ma.norm_w = Lw.ffn_nw;
      const NamedSync gs{kBarGroup, routedev::kRouterWarps * 32};
      for (int it = cta; it < nEB * B; it += grid) {
        routedev::router_cta<8>(ma, a.mb, reinterpret_cast<float*>(p.uni), ps.router_red, it % nEB, it / nEB, gs);
        gs();
      }
    }
    if (!grid_barrier(a, ps, nbar)) break;

    // ---------------- 5. top-k and grouping (every CTA), then gate/up
    const int P = B * K;
    if (warp < B)
      routedev::topk_core(a.mb.logits + (size_t)warp * E, E, K, a.moe.renorm, true, ps.ids + warp * K,
                          ps.w + warp * K, nullptr);
    for (int e = threadIdx.x; e < E; e += kPCThreads) ps.cnt[e] = 0;
    NamedSync{kBarCompute, kPCThreads}();
    if (warp == 0) {
      // stable ranks of the pairs within their expert, 32 pairs at a time in
      // pair order (as the multi-kernel grouping)
      const unsigned lt = (1u << lane) - 1u;
      for (int p0 = 0; p0 < P; p0 += 32) {
        const int pp = p0 + lane;
        const int e = pp < P ? ps.ids[pp] : -1 - lane;
        const unsigned same = __match_any_sync(0xffffffffu, e);
        const int before = pp < P ? ps.cnt[e] : 0;
        __syncwarp();
        if (pp < P) {
          ps.rank[pp] = before + __popc(same & lt);
          if ((same & lt) == 0u) ps.cnt[e] = before + __popc(same);
        }
        __syncwarp();
      }
      // exclusive scans over the experts of the counts and active flags
      int run_off = 0, run_u = 0;
      for (int base = 0; base < E; base += 32) {
        const int e = base + lane;
        const int c = e < E ? ps.cnt[e] : 0, act = c > 0;
        int ic = c, ia = act;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int c2 = __shfl_up_sync(0xffffffffu, ic, o), a2 = __shfl_up_sync(0xffffffffu, ia, o);
          if (lane >= o) { ic += c2; ia += a2; }
        }
        if (e < E) {
          const int off = run_off + ic - c, u = run_u + ia - act;
          ps.off[e] = off;
          if (act) {
            ps.active_e[u] = e;
            ps.active_off[u] = off;
          }
        }
        run_off += __shfl_sync(0xffffffffu, ic, 31);
        run_u += __shfl_sync(0xffffffffu, ia, 31);
      }
      if (lane == 0) {
        ps.active_off[run_u] = run_off;
        ps.n_active = run_u;
      }
    }
    NamedSync{kBarCompute, kPCThreads}();
    for (int pp = threadIdx.x; pp < P; pp += kPCThreads) {
      const int pos = ps.off[ps.ids[pp]] + ps.rank[pp];
      ps.pos_of[pp] = pos;
      ps.pair_token[pos] = pp / K;
    }
    NamedSync{kBarCompute, kPCThreads}();
    if (threadIdx.x == 0) tc::mbar_arrive(tc::smem_u32(&ps.route));   // the producer may issue the expert units
    const int U = ps.n_active;
    if (cta == 0) {
      // the routing of the step, as the multi-kernel path leaves it
      for (int pp = threadIdx.x; pp < P; pp += kPCThreads) {
        a.mb.topk_ids[pp] = ps.ids[pp];
        a.mb.topk_w[pp] = ps.w[pp];
        a.mb.pos_of[pp] = ps.pos_of[pp];
        a.mb.pair_token[pp] = ps.pair_token[pp];
      }
      for (int u = threadIdx.x; u <= U; u += kPCThreads) {
        if (u < U) a.mb.active_e[u] = ps.active_e[u];
        a.mb.active_off[u] = ps.active_off[u];
      }
      if (threadIdx.x == 0) {
        *a.mb.n_active = U;
        if (a.u_log) a.u_log[l] = U;
      }
    }
    // this CTA's contiguous range of gate/up jobs and their items (the
    // producer's grouping); the residual rows of its down tile
    const int J = U * NTg;
    const int jb = (int)((long long)J * cta / grid), je = (int)((long long)J * (cta + 1) / grid);
    if (threadIdx.x == 0) {
      int ni = 0;
      for (int j = jb; j < je; ++ni) {
        const int u = j / NTg, T = j - u * NTg, nt = min(min(kGUTiles, je - j), NTg - T);
        for (int tt = 0; tt < nt; ++tt) {
          ps.gu_item[j - jb + tt] = (short)ni;
          ps.gu_tt[j - jb + tt] = (short)tt;
          ps.gu_n[j - jb + tt] = (short)nt;
        }
        j += nt;
      }
      ps.gu_items = ni;
    }
    if (cta < NTd)
      for (int idx = threadIdx.x; idx < B * 16; idx += kPCThreads)
        ps.hres[idx >> 4][idx & 15] = bf2f(__ldcg(a.h + (size_t)(idx >> 4) * H + cta * 16 + (idx & 15)));
    const int xg = H + 32;
    stage_rows(xs16, xg, reinterpret_cast<const __half*>(a.mb.xn), H, B, H);
    NamedSync{kBarCompute, kPCThreads}();
    {
      run_jobs(je - jb, KSq, ps.gu_items, xg,
               [&](int j) { return make_int3(ps.gu_item[j], ps.gu_tt[j], ps.gu_n[j]); },
               [&](int j, int g) {
                 const int u = (jb + j) / NTg;
                 const int off = ps.active_off[u], cnt = ps.active_off[u + 1] - off;
                 return g < cnt ? ps.pair_token[off + g] : -1;
               },
               [&](int j, int ll, int jq, float v0, float v1) {
                 const int jj = jb + j, u = jj / NTg, T = jj - u * NTg;
                 const int off = ps.active_off[u], cnt = ps.active_off[u + 1] - off, tk = 2 * (ll & 3) + jq;
                 if (tk >= cnt) return;
                 const int f = T * 8 + (ll >> 2);
                 const float sv0 = v0 / (1.f + expf(-v0));
                 a.mb_act16[(size_t)(off + tk) * F + f] = __float2half_rn(round_bf16(sv0 * v1));
               });
    }
    if (!grid_barrier(a, ps, nbar)) break;

    // ---------------- 6. down and the top-k combine of this CTA's tile
    const int xd = F + 32;
    stage_rows(xs16, xd, a.mb_act16, F, P, F);
    NamedSync{kBarCompute, kPCThreads}();
    for (int T = cta; T < NTd; T += grid) {
      run_jobs(U, KSd, U, xd, one,
               [&](int u, int g) {
                 const int off = ps.active_off[u], cnt = ps.active_off[u + 1] - off;
                 return g < cnt ? off + g : -1;
               },
               [&](int u, int ll, int jq, float v0, float v1) {
                 const int off = ps.active_off[u], cnt = ps.active_off[u + 1] - off, tk = 2 * (ll & 3) + jq;
                 if (tk >= cnt) return;
                 ps.out[off + tk][ll >> 2] = v0;
                 ps.out[off + tk][(ll >> 2) + 8] = v1;
               });
      // y = h + sum_r w_r out_r in rank order (k_combine_norm's arithmetic)
      for (int idx = threadIdx.x; idx < B * 16; idx += kPCThreads) {
        const int b = idx >> 4, rr = idx & 15;
        const size_t o = (size_t)b * H + T * 16 + rr;
        float acc = 0.f;
        for (int r = 0; r < K; ++r) acc = fmaf(ps.w[b * K + r], ps.out[ps.pos_of[b * K + r]][rr], acc);
        const float res = T == cta ? ps.hres[b][rr] : bf2f(__ldcg(a.h + o));
        a.x[o] = f2bf(res + acc);
      }
      NamedSync{kBarCompute, kPCThreads}();
    }
    if (!grid_barrier(a, ps, nbar)) break;
  }
  // the final RMSNorm for the output projection (bf16 rows)
  if (cta == 0 && !ps.stop) norm_rows(a, ps, a.final_nw, reinterpret_cast<bf16*>(xs16), nullptr, 0, a.xn_out);
}

namespace {

template <int D, int G>
cudaError_t launch_dg(const PersistArgs& a, size_t smem, cudaStream_t st) {
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_persist_step<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.geo.grid);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr1[1];
  attr1[0].id = cudaLaunchAttributeCooperative;
  attr1[0].val.cooperative = 1;
  cfg.attrs = attr1;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_persist_step<D, G>, a);
}

size_t dyn_smem(const PersistGeo& g) { return (size_t)g.uni_off + g.uni_bytes; }

}  // namespace

bool persist_plan(int H, int qd, int qkv_rows, int F, int E, int k, int g, int d, int cap, int max_rows,
                  PersistGeo* geo, const char** why) {
  auto no = [&](const char* w) {
    if (why) *why = w;
    return false;
  };
  if (d != 64 && d != 128) return no("head_dim must be 64 or 128");
  if (g != 32 && g != 64 && g != 128) return no("group must be 32, 64 or 128");
  if (H % 256 || qd % 256 || F % 256 || qkv_rows % 32 || (2 * F) % 32 || H % 32)
    return no("H, q_heads x head_dim and F must be multiples of 256");
  if (H / 256 > kRoundUnits || qd / 256 > kRoundUnits || F / 256 > kRoundUnits)
    return no("a reduction length above 8192");
  if (E % 8 || E > kPMaxE) return no("experts must be a multiple of 8, at most 256");
  if (max_rows < 1 || max_rows > kPMaxRows || max_rows * k > kPMaxPairs) return no("rows x top_k above 64");
  if ((cap + kAttnChunk - 1) / kAttnChunk > kMaxMergeChunks) return no("ctx_cap too large for the chunk merge");
  {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 148;
    const long J = (long)std::min(E, max_rows * k) * (2 * F / 16);
    if ((J + sms - 1) / sms > kMaxGUJobs) return no("too many gate/up tiles per SM");
  }
  PersistGeo r{};
  const size_t attn = d == 128 ? sizeof(attnf::AttnSmem<128>) : sizeof(attnf::AttnSmem<64>);
  size_t uni = attn;
  uni = std::max(uni, (size_t)H * 4);                                             // router row
  uni = std::max(uni, (size_t)max_rows * (H + 32) * 2 + (size_t)max_rows * H * 2); // QKV rows + staged residual rows
  uni = std::max(uni, (size_t)max_rows * (qd + 32) * 2);                          // output projection rows
  uni = std::max(uni, (size_t)max_rows * k * (F + 32) * 2);                       // down rows (pairs)
  r.uni_bytes = (uint32_t)((uni + 127) & ~(size_t)127);
  const size_t red = (size_t)kRoundUnits * 4 * 32 * sizeof(float);
  const size_t limit = 227 * 1024 - sizeof(PSmem) - 256;
  // the largest item: one 16-row tile over the longest K, with its scales
  const size_t tileH = (size_t)(H / 64) * 512 + (size_t)(H / g) * 32;
  const size_t item = std::max(std::max((size_t)kGUTiles * tileH, (size_t)(qd / 64) * 512 + (size_t)(qd / g) * 32),
                               (size_t)(F / 64) * 512 + (size_t)(F / g) * 32);
  if (red + r.uni_bytes + 2 * item > limit) return no("shared memory");
  r.ring_bytes = (uint32_t)((limit - red - r.uni_bytes) & ~(size_t)127);
  r.ring_off = 0;
  r.red_off = r.ring_bytes;
  r.uni_off = r.red_off + (uint32_t)red;
  *geo = r;
  return true;
}

cudaError_t persist_init(const PersistGeo& geo, int d, int g, int* grid) {
  int dev = 0, sms = 0, per = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const size_t smem = dyn_smem(geo);
  auto occ = [&](auto kern) {
    cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (r == cudaSuccess) r = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, kPThreads, smem);
    return r;
  };
  if (d == 128) e = g == 32 ? occ(k_persist_step<128, 32>) : g == 64 ? occ(k_persist_step<128, 64>) : occ(k_persist_step<128, 128>);
  else e = g == 32 ? occ(k_persist_step<64, 32>) : g == 64 ? occ(k_persist_step<64, 64>) : occ(k_persist_step<64, 128>);
  if (e != cudaSuccess) return e;
  if (per < 1) return cudaErrorInvalidConfiguration;
  *grid = sms;   // one CTA per SM: all resident (cooperative launch)
  return cudaSuccess;
}

cudaError_t launch_persist_step(const PersistArgs& a, int d, int g, cudaStream_t st) {
  if (a.B < 1 || a.B > kPMaxRows || a.B * a.k > kPMaxPairs || a.geo.grid < 1) return cudaErrorInvalidValue;
  const size_t smem = dyn_smem(a.geo);
  if (d == 128) {
    if (g == 32) return launch_dg<128, 32>(a, smem, st);
    if (g == 64) return launch_dg<128, 64>(a, smem, st);
    return launch_dg<128, 128>(a, smem, st);
  }
  if (g == 32) return launch_dg<64, 32>(a, smem, st);
  if (g == 64) return launch_dg<64, 64>(a, smem, st);
  return launch_dg<64, 128>(a, smem, st);
}

}  // namespace bm
