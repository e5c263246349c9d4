// Prompt-length W4A16 GEMMs on the 5th-generation tensor cores (tcgen05) for
// prompt ingestion: the dense QKV and output projections over all P rows of
// a prompt, and the grouped expert gate/up (SiLU fused) and down projections
// over each active expert's rows.  At P = hundreds of rows each weight tile
// meets enough rows for the contraction to be compute-dense, which the decode
// kernels (at most a few dozen rows) never see.
//
// The work is a list of items, each a tile of 128 weight rows (MMA M, TMEM
// lanes) against up to 128 rows of activations (MMA N) over the whole K, in
// stages of 64; one CTA per SM loops over the items blockIdx.x, + gridDim.x,
// ..., its stages numbered across items so that the pipeline runs on from one
// item into the next:
//   - sixteen producer warps in four groups; group g makes stages g, g + 4,
//     ... of every item, one weight row per lane of its four warps: the thread
//     reads the row's int4 codes of the stage straight from the warp-MMA
//     layout the engine keeps (64 contiguous bytes: the four lane slots of the
//     row's 8-row group), turns them into the fp16 products q x s with the
//     row's group scale (one rounding: the scale is folded into the weights
//     here, unlike the decode kernels, which scale exact fp32 group sums), and
//     writes them into the stage's TMEM slot as the MMA's A operand;
//   - one lane of a loader warp brings the stage's 128 activation rows (64
//     values of K each) into shared memory by TMA as the B operand, 128-byte
//     swizzled, rows past the tensor's end read as zero;
//   - one elected lane of the MMA warp issues each stage's four MMAs
//     (M 128 x N x K 16, fp16 in, fp32 accumulated in tensor memory), four
//     stages at a time, and commits them to the group's `done` barrier.
// Eight slots rotate; a slot is refilled once the MMAs of the stage that used
// it have completed.  One stage takes a group longer than the MMAs take to
// run it, so the four groups work on four stages at once.  Item m accumulates
// into the TMEM columns 128 (m % 2) ..: after making their stages of item m
// the producers read out item m - 1's accumulator with tcgen05.ld and write
// its epilogue (bf16 output (+ residual), SiLU(gate) x up as bf16-rounded
// fp16, or fp32 expert outputs for the combine) while the MMAs run on item m.
// Every mbarrier wait is bounded; a wait that gives up sets the error flag
// and the kernel runs on to its end (every later wait is bounded too), so
// nothing can hang.
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace bm {

namespace {

constexpr int kPfM = 128;              // weight rows per CTA
constexpr int kPfN = 128;              // activation rows per CTA
constexpr int kPfSlots = 8;            // stages in flight: TMEM A slots and shared-memory B tiles
constexpr int kPfGroups = 4;           // producer groups; group g makes stages g, g + 4, ...
constexpr int kPfProducers = kPfM * kPfGroups;   // a group: 4 warps, one weight row per lane
constexpr int kPfThreads = kPfProducers + 64;   // producers + the MMA warp + the B loader warp
constexpr uint32_t kPfTmemCols = 512;  // two accumulators [0, 256) + 8 A slots of 32 columns
constexpr uint32_t kPfWaitLimit = 1u << 18;   // polls of ~3.7 us: a wait gives up after about a second
constexpr int kPfBTile = kPfN * 128;   // bytes of one stage's B tile (N rows x 64 fp16)
constexpr int kPfMmaGroup = 4;         // stages the MMA lane takes at a time (K % 256 == 0)
constexpr int kPfQS = kPfSlots / kPfMmaGroup;   // groups of slots
static_assert(kPfSlots % kPfMmaGroup == 0, "groups of stages tile the slots");
// dynamic shared memory per CTA: the B tiles of every slot, 1024-byte aligned
// for the 128-byte swizzle (193 KB: one CTA per SM, which also holds all 512
// TMEM columns)
constexpr int kPfSmem = kPfSlots * kPfBTile + 1024;
static_assert(2 * kPfN + kPfSlots * 32 <= (int)kPfTmemCols, "TMEM holds two accumulators and the A slots");

enum PfMode { PF_DENSE = 0, PF_GATEUP = 1, PF_DOWN = 2 };
static_assert(kPfN == kPromptTileRows, "the grouping's job tiles are the GEMM's activation tiles");


// One 2-D TMA tile load (box of the tensor map at column x, row y) into shared
// memory, completion counted in bytes on `mbar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int x, int y, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(mbar)
      : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t mbar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
// K-major operand with the 128-byte swizzle: rows of 128 bytes (64 fp16), 8-row
// atoms of 1024 bytes (SBO), LBO unused (encoded 1), layout type 2; the start
// address moves by 32 bytes per 16 values of K.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) |
         (2ull << 61);
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }

// One item of the launch: weight tile x (rows 128 x .. + 127 of the matrix)
// against activation job j (dense: prompt rows 128 j ..; experts: the job
// list's (active expert, 128-row tile of its sorted pairs)).
struct PfItem {
  int x, n0, ntok;          // weight tile, first activation row, activation rows
  const uint8_t* W;         // the item's matrix (experts: its expert's)
  const uint32_t* S;
};

template <int MODE>
__device__ __forceinline__ PfItem pf_item(const PrefillGemmArgs& a, int tiles, int w) {
  PfItem it;
  const int j = w / tiles;
  it.x = w - j * tiles;
  it.W = a.W;
  it.S = a.S;
  if (MODE == PF_DENSE) {
    it.n0 = j * kPfN;
    it.ntok = min(kPfN, a.ntok - it.n0);
  } else {
    const int job = a.jobs[j], u = job & 0xFFFF, tile = job >> 16;
    const int e = a.active_e[u], off = a.active_off[u], cnt = a.active_off[u + 1] - off;
    it.n0 = off + tile * kPfN;
    it.ntok = min(kPfN, cnt - tile * kPfN);
    it.W += (size_t)e * a.w_expert_stride;
    it.S += (size_t)e * a.s_expert_stride;
  }
  return it;
}
// MMA N of an item: its rows rounded up to a multiple of 16
__device__ __forceinline__ int pf_nmma(int ntok) { return min(kPfN, max(16, (ntok + 15) & ~15)); }

template <int MODE, int G>
__global__ void __launch_bounds__(kPfThreads, 1) k_w4_tc_prefill(PrefillGemmArgs a, const __grid_constant__ TmapBytes tm) {
  extern __shared__ unsigned char smem_raw[];   // kPfSlots B tiles, 1024-byte aligned below
  __shared__ __align__(8) uint64_t full_bar[kPfQS];   // a group of kPfMmaGroup stages is in place
  __shared__ __align__(8) uint64_t done_bar[kPfQS];   // a group's MMAs are done
  __shared__ __align__(8) uint64_t acc_full[2];       // an item's accumulator is complete
  __shared__ __align__(8) uint64_t acc_empty[2];      // an item's accumulator has been read out
  __shared__ uint32_t tmem_slot;
  static_assert(G == 32 || G == 64 || G == 128, "group size");

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int K = a.K, NC = K / 64, NG = K / G;
  const int tiles = a.rows / kPfM;
  const int njobs = MODE == PF_DENSE ? (a.ntok + kPfN - 1) / kPfN : *a.n_jobs;
  // items w = blockIdx.x, + gridDim.x, ... below tiles x njobs (uniform over the CTA)
  const int total = tiles * njobs;
  if ((int)blockIdx.x >= total) return;
  const int n_items = (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1;

  if (warp == 0) {
    tc::tmem_alloc(tc::smem_u32(&tmem_slot), kPfTmemCols);
    tc::tmem_relinquish();
  }
  if (t == 0) {
    // a group of kPfMmaGroup stages completes with one arrival per producer
    // warp of each of its stages and one per stage from the B loader (with
    // the stage's bytes); an accumulator is read out when every producer
    // warp has taken its columns
    for (int i = 0; i < kPfQS; ++i) {
      tc::mbar_init(tc::smem_u32(&full_bar[i]), kPfMmaGroup * (kPfProducers / 32 / kPfGroups + 1));
      tc::mbar_init(tc::smem_u32(&done_bar[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      tc::mbar_init(tc::smem_u32(&acc_full[i]), 1);
      tc::mbar_init(tc::smem_u32(&acc_empty[i]), kPfProducers / 32);
    }
    tc::fence_mbar_init();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  const uint32_t raw_base = tc::smem_u32(smem_raw);
  const uint32_t b_base = raw_base + ((1024u - (raw_base & 1023u)) & 1023u);
  bool ok = true;
  // stage gs of the CTA (counted over all its items) uses slot gs % kPfSlots
  // and the barriers of its group, gs / kPfMmaGroup
  auto group_bar = [&](uint64_t* bars, int gs) { return tc::smem_u32(&bars[(gs / kPfMmaGroup) % kPfQS]); };
  auto group_parity = [](int gs) { return (uint32_t)((gs / kPfSlots) & 1); };

  if (warp == kPfProducers / 32 + 1) {
    // ---------------- B loader: one lane, one TMA tile load per stage into the
    // slot's 128-row B tile, once the MMAs of the stage that used it are done
    if (lane == 0) {
      int gs = 0;
      for (int m = 0; m < n_items; ++m) {
        const PfItem it = pf_item<MODE>(a, tiles, (int)blockIdx.x + m * (int)gridDim.x);
        for (int i = 0; i < NC; ++i, ++gs) {
          const int j = gs - kPfSlots;
          if (j >= 0 && !tc::mbar_wait_spin(group_bar(done_bar, j), group_parity(j), kPfWaitLimit)) ok = false;
          const uint32_t bar = group_bar(full_bar, gs);
          mbar_expect_tx(bar, (uint32_t)kPfBTile);
          tma_load_2d(b_base + (uint32_t)(gs % kPfSlots) * kPfBTile, &tm, i * 64, it.n0, bar);
        }
      }
      // every tile load issued has landed before the CTA may exit (the last
      // groups' barriers complete)
      for (int g0 = gs - kPfSlots > 0 ? gs - kPfSlots : 0; g0 < gs; g0 += kPfMmaGroup)
        if (!tc::mbar_wait(group_bar(full_bar, g0), group_parity(g0), kPfWaitLimit)) ok = false;
    }
    __syncwarp();
  } else if (warp == kPfProducers / 32) {
    // ---------------- MMA warp: one lane issues.  Item m accumulates into
    // TMEM columns 128 (m % 2) ..; it waits until the producers have read out
    // item m - 2 from there.  Stages go in groups of kPfMmaGroup: one wait
    // for the group (the producers run well ahead, so it has mostly completed
    // already), its MMAs back to back, then one commit that releases the
    // group's slots.
    if (lane == 0) {
      int gs = 0;
      for (int m = 0; m < n_items; ++m) {
        const PfItem it = pf_item<MODE>(a, tiles, (int)blockIdx.x + m * (int)gridDim.x);
        const uint32_t idesc = tc::idesc_f16_f32(kPfM, pf_nmma(it.ntok));
        const int b = m & 1;
        if (m >= 2 && !tc::mbar_wait_spin(tc::smem_u32(&acc_empty[b]), (uint32_t)(((m >> 1) - 1) & 1), kPfWaitLimit))
          ok = false;
        tc::fence_after_sync();
        for (int i0 = 0; i0 < NC; i0 += kPfMmaGroup, gs += kPfMmaGroup) {
          if (!tc::mbar_wait_spin(group_bar(full_bar, gs), group_parity(gs), kPfWaitLimit)) ok = false;
          tc::fence_after_sync();
#pragma unroll
          for (int u = 0; u < kPfMmaGroup; ++u) {
            const int s = (gs + u) % kPfSlots;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              // B: the slot's swizzled tile, this MMA's 16 values of K 32 bytes
              // into each 128-byte row; A: the slot's 8 TMEM columns (16 fp16
              // values of K) per MMA
              const uint64_t bd = smem_desc_sw128(b_base + (uint32_t)s * kPfBTile + (uint32_t)q * 32u);
              tc::mma_f16_tmem_a(tmem + b * kPfN, tmem + 2 * kPfN + s * 32 + q * 8, bd, idesc,
                                 (uint32_t)(i0 + u > 0 || q > 0));
            }
          }
          tc::mma_commit(group_bar(done_bar, gs));
        }
        tc::mma_commit(tc::smem_u32(&acc_full[b]));
      }
    }
    __syncwarp();
  } else {
    // ---------------- producers (warps 0-15): group g = w / 4 makes stages g, g + 4,
    // ... of every item; its warp w % 4 takes TMEM lane quarter w % 4 (weight
    // rows 32 (w % 4) + lane of the tile) and all 64 values of K of each of
    // its stages: the 64 bytes of the row's 8-row group's four lane slots in
    // the mma layout.  Four groups keep four stages in the making while the
    // MMA warp works through the earlier ones.  After making its stages of
    // item m the group reads out its columns of item m - 1's accumulator
    // (done by then, the MMAs being on item m) while the MMAs run on.
    const int quarter = warp & 3, group = warp >> 2, lane_row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int gq = lane_row & 7, half = (lane_row >> 3) & 1;
    const uint32_t m_lo = half ? 0x00F000F0u : 0x000F000Fu;
    const uint32_t magic = half ? 0x54005400u : 0x64006400u;
    const __half2 bias = bits_h2(half ? 0x54805480u : 0x64086408u);   // (72, 72) or (1032, 1032)

    // the lane's weight row of an item: its 64 bytes of stage i at + i * 512,
    // its group scales at + group * 8
    auto row_of = [&](const PfItem& it, const uint8_t*& wrow, const uint32_t*& srow) {
      const int T16 = (it.x * kPfM + lane_row) >> 4;
      wrow = it.W + ((size_t)T16 * NC * 32 + gq * 4) * 16;
      srow = it.S + (size_t)T16 * NG * 8 + gq;
    };
    uint4 wreg[4];
    uint32_t sreg[2];
    auto load_a = [&](const uint8_t* wrow, const uint32_t* srow, int i) {
      const uint8_t* p = wrow + (size_t)i * 512;
#pragma unroll
      for (int v = 0; v < 4; ++v) wreg[v] = ldg_nc_v4(p + v * 16);
      const int k0 = i * 64;
      sreg[0] = __ldg(srow + (size_t)(k0 / G) * 8);
      sreg[1] = G == 32 ? __ldg(srow + (size_t)(k0 / G + 1) * 8) : sreg[0];
    };
    // read out item m's accumulator: this group's 8-column chunks (columns
    // 8 group, + 32, ...) of the rows' outputs
    auto epilogue = [&](const PfItem& it, int m) {
      const int b = m & 1;
      if (!tc::mbar_wait(tc::smem_u32(&acc_full[b]), (uint32_t)((m >> 1) & 1), kPfWaitLimit)) ok = false;
      tc::fence_after_sync();
      const int nmma = pf_nmma(it.ntok), ntok = it.ntok, n0 = it.n0;
      const int grow = it.x * kPfM + lane_row;   // weight row within the matrix
      for (int c0 = 8 * group; c0 < nmma; c0 += 8 * kPfGroups) {
        uint32_t d[8];
        tc::tmem_ld8(tmem + lane_base + (uint32_t)(b * kPfN + c0), d);
        tc::tmem_wait_ld();
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int n = c0 + jj;
          float acc = __uint_as_float(d[jj]);
          if (MODE == PF_GATEUP) {
            // rows 8 apart hold the gate and up rows of one feature
            const float up = __shfl_down_sync(0xffffffffu, acc, 8);
            if (half == 0 && n < ntok) {
              const int f = (grow >> 4) * 8 + gq;
              const float sg = acc / (1.f + expf(-acc));
              a.act16[(size_t)(n0 + n) * a.F + f] = __float2half_rn(round_bf16(sg * up));
            }
          } else if (n < ntok) {
            const size_t mrow = (size_t)(n0 + n);
            if (MODE == PF_DENSE) {
              if (a.Res) acc += bf2f(a.Res[mrow * a.ldr + grow]);
              a.Y[mrow * a.ldy + grow] = f2bf(acc);
            } else {
              a.out[mrow * a.H + grow] = acc;
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(tc::smem_u32(&acc_empty[b]));
    };

    PfItem cur = pf_item<MODE>(a, tiles, (int)blockIdx.x), prev = cur;
    const uint8_t* wrow;
    const uint32_t* srow;
    row_of(cur, wrow, srow);
    load_a(wrow, srow, group);
    int gs0 = 0;   // the item's first stage on the CTA's count
    for (int m = 0; m < n_items; ++m) {
      // the next item's row, for the weight load that crosses into it
      const bool more = m + 1 < n_items;
      PfItem nx = cur;
      const uint8_t* wrow_n = wrow;
      const uint32_t* srow_n = srow;
      if (more) {
        nx = pf_item<MODE>(a, tiles, (int)blockIdx.x + (m + 1) * (int)gridDim.x);
        row_of(nx, wrow_n, srow_n);
      }
      for (int i = group; i < NC; i += kPfGroups) {
        const int gs = gs0 + i, s = gs % kPfSlots;
        // the MMAs of stage j = gs - kPfSlots, the last to use this slot, have finished
        const int j = gs - kPfSlots;
        if (j >= 0) {
          if (!tc::mbar_wait_spin(group_bar(done_bar, j), group_parity(j), kPfWaitLimit)) ok = false;
          tc::fence_after_sync();
        }
        // A of stage i: fp16 (q x s) pairs in K order, 32 columns; word
        // (t, ss) of the row's 64 bytes covers K 32 (ss / 2) + 8 t + 4 (ss % 2)
        // .. + 3: columns 16 (ss / 2) + 4 t + 2 (ss % 2) and the next
        uint32_t v[32];
        {
          const __half2 sc0 = bits_h2(half ? (sreg[0] >> 16) * 0x10001u : (sreg[0] & 0xFFFFu) * 0x10001u);
          const __half2 sc1 = bits_h2(half ? (sreg[1] >> 16) * 0x10001u : (sreg[1] & 0xFFFFu) * 0x10001u);
#pragma unroll
          for (int tt = 0; tt < 4; ++tt) {
            const uint32_t wv[4] = {wreg[tt].x, wreg[tt].y, wreg[tt].z, wreg[tt].w};
#pragma unroll
            for (int ss = 0; ss < 4; ++ss) {
              const uint32_t w = wv[ss], w8 = w >> 8;
              const __half2 sc = (ss >> 1) ? sc1 : sc0;   // g = 32: the second half of the stage's K
              const __half2 lo = __hsub2(bits_h2((w & m_lo) | magic), bias);
              const __half2 hi = __hsub2(bits_h2((w8 & m_lo) | magic), bias);
              const int col = 16 * (ss >> 1) + 4 * tt + 2 * (ss & 1);
              v[col] = h2_bits(__hmul2(lo, sc));
              v[col + 1] = h2_bits(__hmul2(hi, sc));
            }
          }
        }
        // the group's next stage: this item's, else the next item's first
        if (i + kPfGroups < NC) {
          load_a(wrow, srow, i + kPfGroups);
        } else if (more) {
          load_a(wrow_n, srow_n, group);
        }
        tc::tmem_st32(tmem + lane_base + (uint32_t)(2 * kPfN + s * 32), v);
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(group_bar(full_bar, gs));
      }
      if (m > 0) epilogue(prev, m - 1);
      prev = cur;
      cur = nx;
      wrow = wrow_n;
      srow = srow_n;
      gs0 += NC;
    }
    epilogue(prev, n_items - 1);
  }
  if (!ok && a.err) atomicExch(a.err, 4);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kPfTmemCols);
}

template <int MODE>
cudaError_t launch_mode(const PrefillGemmArgs& a, const TmapBytes& tm, int max_jobs, cudaStream_t st) {
  // persistent: one CTA per SM (all of its tensor memory), each looping over
  // the items (weight tile, job) blockIdx.x, + gridDim.x, ...
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long items = (long long)(a.rows / kPfM) * max_jobs;
  const dim3 grid((unsigned)(items < sms ? items : sms));
  const size_t smem = kPfSmem;
  if (a.g == 32) {
    k_w4_tc_prefill<MODE, 32><<<grid, kPfThreads, smem, st>>>(a, tm);
  } else if (a.g == 64) {
    k_w4_tc_prefill<MODE, 64><<<grid, kPfThreads, smem, st>>>(a, tm);
  } else {
    k_w4_tc_prefill<MODE, 128><<<grid, kPfThreads, smem, st>>>(a, tm);
  }
  return cudaGetLastError();
}

template <int MODE>
cudaError_t set_attr() {
  const int smem = kPfSmem;
  cudaError_t e = cudaFuncSetAttribute(k_w4_tc_prefill<MODE, 32>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_w4_tc_prefill<MODE, 64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_w4_tc_prefill<MODE, 128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return e;
}

}  // namespace

bool prefill_gemm_supports(int rows, int K, int g) {
  return rows > 0 && rows % kPfM == 0 && K >= 64 * kPfMmaGroup && K % (64 * kPfMmaGroup) == 0 &&
         (g == 32 || g == 64 || g == 128) && K % g == 0;
}

cudaError_t launch_prefill_dense(const PrefillGemmArgs& a, const TmapBytes& tm, cudaStream_t st) {
  if (!prefill_gemm_supports(a.rows, a.K, a.g) || a.ntok < 1) return cudaErrorInvalidValue;
  return launch_mode<PF_DENSE>(a, tm, (a.ntok + kPfN - 1) / kPfN, st);
}

cudaError_t launch_prefill_gateup(const PrefillGemmArgs& a, const TmapBytes& tm, int max_rows_per_expert,
                                  cudaStream_t st) {
  if (!prefill_gemm_supports(a.rows, a.K, a.g) || !a.n_active || !a.n_jobs || a.max_jobs < 1 || max_rows_per_expert < 1)
    return cudaErrorInvalidValue;
  return launch_mode<PF_GATEUP>(a, tm, a.max_jobs, st);
}

cudaError_t launch_prefill_down(const PrefillGemmArgs& a, const TmapBytes& tm, int max_rows_per_expert,
                                cudaStream_t st) {
  if (!prefill_gemm_supports(a.rows, a.K, a.g) || !a.n_active || !a.n_jobs || a.max_jobs < 1 || max_rows_per_expert < 1)
    return cudaErrorInvalidValue;
  return launch_mode<PF_DOWN>(a, tm, a.max_jobs, st);
}

cudaError_t init_prefill_attributes() {
  cudaError_t e = set_attr<PF_DENSE>();
  if (e == cudaSuccess) e = set_attr<PF_GATEUP>();
  if (e == cudaSuccess) e = set_attr<PF_DOWN>();
  return e;
}

}  // namespace bm

namespace bm {

namespace {
__global__ void k_fill_i32(int32_t* p, int32_t value, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = value;
}
}  // namespace

cudaError_t launch_fill_i32(int32_t* p, int32_t value, int n, cudaStream_t st) {
  if (n < 1) return cudaSuccess;
  k_fill_i32<<<(n + 255) / 256, 256, 0, st>>>(p, value, n);
  return cudaGetLastError();
}

}  // namespace bm

#include <cuda.h>   // the tensor-map types; the encoder itself is fetched from the driver at run time

namespace bm {

namespace {

__global__ void k_gather_rows(const __half* __restrict__ src, const int32_t* __restrict__ map, int cols,
                              __half* __restrict__ dst) {
  const int r = blockIdx.x;
  const uint4* s = reinterpret_cast<const uint4*>(src + (size_t)map[r] * cols);
  uint4* d = reinterpret_cast<uint4*>(dst + (size_t)r * cols);
  for (int i = threadIdx.x; i < cols / 8; i += blockDim.x) d[i] = s[i];
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

}  // namespace

cudaError_t encode_rows_tmap(TmapBytes* out, const void* base, int rows, int K, int ld) {
  static_assert(sizeof(CUtensorMap) == sizeof(TmapBytes), "tensor map size");
  EncodeTiledFn fn = encoder();
  if (!fn) return cudaErrorNotSupported;
  if (rows < 1 || K < 64 || K % 64 || ld < K || (ld * 2) % 16 || (reinterpret_cast<uintptr_t>(base) & 15))
    return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)kPfN};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(reinterpret_cast<CUtensorMap*>(out), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base),
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_gather_rows(const __half* src, const int32_t* map, int n, int cols, __half* dst, cudaStream_t st) {
  if (n < 1) return cudaSuccess;
  if (cols % 8) return cudaErrorInvalidValue;
  k_gather_rows<<<n, 256, 0, st>>>(src, map, cols, dst);
  return cudaGetLastError();
}

}  // namespace bm
