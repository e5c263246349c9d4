// Tensor-core (tcgen05) projections of the decode step: the dense W4A16
// projections, the grouped expert gate/up and down GEMMs, and the bf16
// output projection.
//
// A CTA owns a job: a tile of 128 weight rows, up to 16 tokens (M = 128
// weight rows x N = 16 tokens: the large dimension on the MMA's M) and a
// range of K (the whole K, or 1/ksplit of it when there are too few jobs to
// fill the GPU).  Warps 0-3 are producers: thread t streams weight row t and
// writes it with tcgen05.st into TMEM lane t, where it is the MMA's A
// operand — for int4 weights each code becomes the exact fp16 integer q - 8;
// bf16 weights are stored as they are.  Warp 4 issues the MMAs.  The tokens'
// activations sit in shared memory as the B operand (fp16, or bf16 for the
// output projection).
//
// K advances in stages of 64 (32 TMEM columns of A).  An MMA's completion
// reaches its mbarrier about a microsecond after issue, so a CTA keeps
// several stages resident in TMEM: each slot has `full` (the four producer
// warps arrive once its A columns are written) and `done` (tcgen05.commit
// arrives once its MMAs finish); before rewriting a slot the producers wait
// on its `done`.  There is no CTA-wide barrier in the K loop.  For int4
// weights each slot also holds the stage's own fp32 accumulator (one per
// int4 group inside the stage): the products q * x are exact in fp32, and
// the producers apply the fp32 group scale when they drain it, so the
// weights are never rounded.  A row's result is the sum over stages, in
// ascending K, of scale x (exact group sum); with a K split, the CTA that
// arrives last adds the splits' partials in split order.  Nothing depends on
// the other tokens of the tile.
//
// Int4 weight layout ("tc layout", written once by the repack kernel): for
// tile t and 32-wide K chunk c: 128 rows x 16 bytes, row-contiguous, so a
// warp's loads of one chunk are 512 contiguous bytes.  Inside each 32-bit
// word the 8 codes are ordered (k0 k2 k4 k6 k1 k3 k5 k7), so one
// (w >> 4i) & 0x000F000F | 0x64006400 yields the fp16 pair (1024 + u_2i,
// 1024 + u_2i+1) of one TMEM column.  Scales: [tile][K/g][128 rows] fp16.
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace bm {

namespace {

constexpr int kProducers = 256;             // 8 warps: two per TMEM lane quarter
constexpr int kThreads = kProducers + 32;   // + the MMA warp
constexpr int kTokens = 16;                 // MMA N
constexpr int kStageK = 64;                 // K per stage: 32 TMEM columns of A
constexpr uint32_t kTmemCols = 256;
constexpr int kMaxSlots = 6;
constexpr int kLmSlots = 6;                 // output projection: A-only slots, one accumulator
constexpr uint32_t kWaitLimit = 1u << 18;         // polls of ~3.7 us each: a wait gives up after about a second
constexpr int kMaxSplit = 8;

// One packed word (codes ordered k0 k2 k4 k6 k1 k3 k5 k7) -> the four TMEM
// columns of fp16 pairs (q_2i, q_2i+1), q = u - 8, exact.  Nibbles at bits
// 0-3 / 16-19 become 1024 + u (minus 1032 gives q); nibbles at bits 4-7 /
// 20-23 become 1024 + 16u, and (1024 + 16u) / 16 - 72 = u - 8 in one fma.
__device__ __forceinline__ void dq_word(uint32_t w, uint32_t* out) {
  const __half2 k1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
  const __half2 k16th = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));   // 1/16
  const __half2 km72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));    // -72
  const uint32_t w8 = w >> 8;
  uint32_t v0 = (w & 0x000F000Fu) | 0x64006400u, v1 = (w & 0x00F000F0u) | 0x64006400u;
  uint32_t v2 = (w8 & 0x000F000Fu) | 0x64006400u, v3 = (w8 & 0x00F000F0u) | 0x64006400u;
  __half2 h0 = __hsub2(*reinterpret_cast<__half2*>(&v0), k1032);
  __half2 h1 = __hfma2(*reinterpret_cast<__half2*>(&v1), k16th, km72);
  __half2 h2 = __hsub2(*reinterpret_cast<__half2*>(&v2), k1032);
  __half2 h3 = __hfma2(*reinterpret_cast<__half2*>(&v3), k16th, km72);
  out[0] = *reinterpret_cast<uint32_t*>(&h0);
  out[1] = *reinterpret_cast<uint32_t*>(&h1);
  out[2] = *reinterpret_cast<uint32_t*>(&h2);
  out[3] = *reinterpret_cast<uint32_t*>(&h3);
}

__device__ __forceinline__ void dq16(const uint4 w, uint32_t* out) {
  dq_word(w.x, out);
  dq_word(w.y, out + 4);
  dq_word(w.z, out + 8);
  dq_word(w.w, out + 12);
}

enum TcMode { TC_DENSE = 0, TC_GATEUP = 1, TC_DOWN = 2, TC_LM = 3 };

template <int MODE, bool TWO_GROUPS>
__global__ void __launch_bounds__(kThreads, 2) k_w4_tc(TcArgs a) {
  constexpr bool LM = MODE == TC_LM;
  constexpr int kPrefetch = LM ? 4 : 6;   // stages of weights in flight per producer thread
  constexpr int kVec = LM ? 4 : 1;        // 16-byte loads per thread per stage (half a stage)
  constexpr int kHalfTok = kTokens / 2;   // tokens drained by one of a row's two threads
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxSlots];
  __shared__ __align__(8) uint64_t done_bar[kMaxSlots];
  __shared__ __align__(8) uint64_t final_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ float2 scale_s[kMaxSlots][kProducers];   // group scales of the stage in each slot
  __shared__ int flag_s;

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int ksplit = a.ksplit;
  const int tiles = gridDim.x / ksplit;
  const int tile = blockIdx.x / ksplit, ks = blockIdx.x - tile * ksplit;
  const int tg = blockIdx.y;
  const int job = (blockIdx.z * gridDim.y + tg) * tiles + tile;
  const int K = a.K;
  const uint8_t* W = a.W;
  const __half* S = a.S;
  int ntok, row0 = 0;   // tokens of this CTA; first pair / row index
  if (MODE == TC_DENSE || LM) {
    ntok = min(kTokens, a.ntok - tg * kTokens);
    row0 = tg * kTokens;
  } else {
    const int u = blockIdx.z;
    if (u >= *a.n_active) return;
    const int e = a.active_e[u];
    const int off = a.active_off[u], cnt = a.active_off[u + 1] - off;
    ntok = min(kTokens, cnt - tg * kTokens);
    row0 = off + tg * kTokens;
    W += (size_t)e * a.w_expert_stride;
    S += (size_t)e * a.s_expert_stride;
  }
  if (ntok <= 0) return;
  const int nst_all = K / kStageK;
  const int nst = nst_all / ksplit;          // stages of this split
  const int s_begin = ks * nst;
  const int k_begin = s_begin * kStageK, Kc = nst * kStageK;
  // TMEM columns: int4 slots are [A 32 | D 16] (g >= 64) or [A 32 | D 2x16]
  // (g == 32, two groups per stage); the output projection has A-only slots
  // and one accumulator after them.
  constexpr bool two_groups = !LM && TWO_GROUPS;
  constexpr int dcols = LM ? 0 : (two_groups ? 32 : 16);
  constexpr int slot_cols = 32 + dcols;
  constexpr int nslots = LM ? kLmSlots : (two_groups ? 4 : 5);
  constexpr int lm_dcol = kLmSlots * 32;

  // ---- TMEM and barriers
  if (warp == 0) {
    tc::tmem_alloc(tc::smem_u32(&tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  if (t == 0) {
    for (int i = 0; i < nslots; ++i) {
      tc::mbar_init(tc::smem_u32(&full_bar[i]), kProducers / 32);   // one arrive per producer warp
      tc::mbar_init(tc::smem_u32(&done_bar[i]), 1);
    }
    tc::mbar_init(tc::smem_u32(&final_bar), 1);
    tc::fence_mbar_init();
    flag_s = 0;
  }

  // ---- activations (this split's K range) -> shared memory, no-swizzle
  // K-major core matrices of 8 rows x 16 bytes: element (r, k) of the CTA's
  // 16 x Kc tile sits at byte ((r / 8) * Kc / 8 + k / 8) * 128 + (r % 8) * 16
  // + (k % 8) * 2, i.e. 16-byte chunk L = ((r / 8) * Kc / 8 + k / 8) * 8 + r % 8.
  // Thread t fills chunks t, t + kThreads, ... — consecutive threads,
  // consecutive 16 bytes, no bank conflicts.  With the fused RMSNorm each
  // row's mean square comes first (one warp per row, the whole K).
  const bool do_norm = (MODE == TC_DENSE || LM) && a.do_norm;
  const int nk8 = Kc / 8;
  const uint32_t sbo = (uint32_t)nk8 * 128u;   // bytes between the two 8-row groups
  constexpr int kWarps = kThreads / 32;
  __shared__ float rinv_s[kTokens];
  __shared__ const bf16* rowp_s[kTokens];
  if (t < kTokens) {
    const bf16* x = nullptr;
    if (t < ntok) x = (MODE == TC_GATEUP) ? a.X + (size_t)a.pair_token[row0 + t] * a.ldx
                                          : a.X + (size_t)(row0 + t) * a.ldx;
    rowp_s[t] = x;
  }
  __syncthreads();
  if (do_norm) {
    for (int r = warp; r < ntok; r += kWarps) {
      const bf16* x = rowp_s[r];
      float ss = 0.f;
      for (int j0 = lane; j0 < K / 8; j0 += 128) {
        uint4 raw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (j0 + 32 * i < K / 8) raw[i] = *reinterpret_cast<const uint4*>(x + (j0 + 32 * i) * 8);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          if (j0 + 32 * i < K / 8) {
            const uint32_t rw[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float v0 = bf_lo(rw[q]), v1 = bf_hi(rw[q]);
              ss = fmaf(v0, v0, ss);
              ss = fmaf(v1, v1, ss);
            }
          }
        }
      }
      ss = warp_sum(ss);
      if (lane == 0) rinv_s[r] = 1.0f / sqrtf(ss / (float)K + a.eps);
    }
    __syncthreads();
  }
  {
    const int nchunks = kTokens * nk8;
    for (int L0 = t; L0 < nchunks; L0 += 4 * kThreads) {
      uint4 raw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int L = L0 + i * kThreads;
        raw[i] = make_uint4(0, 0, 0, 0);
        if (L < nchunks) {
          const int r = (L / (nk8 * 8)) * 8 + (L & 7), j = (L >> 3) % nk8;
          if (r < ntok) raw[i] = *reinterpret_cast<const uint4*>(rowp_s[r] + k_begin + j * 8);
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int L = L0 + i * kThreads;
        if (L < nchunks) {
          const int r = (L / (nk8 * 8)) * 8 + (L & 7), j = (L >> 3) % nk8;
          uint32_t o[4] = {0u, 0u, 0u, 0u};
          if (r < ntok) {
            const uint32_t rw[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float v0 = bf_lo(rw[q]), v1 = bf_hi(rw[q]);
              if (do_norm) {
                const int k = k_begin + j * 8 + 2 * q;
                const float w0 = a.norm_w ? bf2f(a.norm_w[k]) : 1.f;
                const float w1 = a.norm_w ? bf2f(a.norm_w[k + 1]) : 1.f;
                v0 = round_bf16(v0 * rinv_s[r] * w0);
                v1 = round_bf16(v1 * rinv_s[r] * w1);
              }
              if (LM) {
                o[q] = (__float_as_uint(v0) >> 16) | (__float_as_uint(v1) & 0xFFFF0000u);   // exact: already bf16
              } else {
                __half2 hh = __floats2half2_rn(v0, v1);
                o[q] = *reinterpret_cast<uint32_t*>(&hh);
              }
            }
          }
          *reinterpret_cast<uint4*>(smem + (size_t)L * 16) = make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  bool ok = true;
  float acc[kTokens];
#pragma unroll
  for (int j = 0; j < kTokens; ++j) acc[j] = 0.f;

  if (warp == kProducers / 32) {
    // ---------------- MMA warp: one elected lane issues, the others idle
    if (lane == 0) {
      const uint32_t b_base = tc::smem_u32(smem);
      const uint32_t idesc = LM ? tc::idesc_bf16_f32(128, kTokens) : tc::idesc_f16_f32(128, kTokens);
      int slot = 0;
      uint32_t phase = 0;
      for (int i = 0; i < nst; ++i) {
        if (!tc::mbar_wait(tc::smem_u32(&full_bar[slot]), phase, kWaitLimit)) ok = false;
        tc::fence_after_sync();
        const uint32_t acol = slot * slot_cols;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint64_t bd = tc::smem_desc_noswizzle(b_base + (uint32_t)(i * 4 + q) * 256u, 128u, sbo);
          uint32_t dcol, accum;
          if (LM) {
            dcol = lm_dcol;
            accum = (uint32_t)(i > 0 || q > 0);
          } else if (two_groups) {
            dcol = acol + 32 + (q >> 1) * 16;
            accum = (uint32_t)(q & 1);
          } else {
            dcol = acol + 32;
            accum = (uint32_t)(q > 0);
          }
          tc::mma_f16_tmem_a(tmem + dcol, tmem + acol + q * 8, bd, idesc, accum);
        }
        tc::mma_commit(tc::smem_u32(&done_bar[slot]));
        if (++slot == nslots) {
          slot = 0;
          phase ^= 1u;
        }
      }
      tc::mma_commit(tc::smem_u32(&final_bar));
    }
    __syncwarp();
  } else {
    // ---------------- producers: warps w and w + 4 share TMEM lane quarter
    // w % 4 (weight rows 32 (w % 4) + lane); warp half h = w / 4 writes the
    // h-th 32-wide half of each stage and drains tokens [8h, 8h + 8).
    const int quarter = warp & 3, h = warp >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int ng = LM ? 1 : K / a.g;
    const int gshift = 31 - __clz(a.g);
    const uint8_t* wt = LM ? W + ((size_t)tile * 128 + row) * (size_t)K * 2 + (size_t)(k_begin + 32 * h) * 2
                           : W + ((size_t)tile * (K / 32) + 2 * s_begin + h) * 2048 + (size_t)row * 16;
    const __half* st_ = LM ? nullptr : S + (size_t)tile * ng * 128 + row;
    // The ring holds each stage's weights and scale(s) as loaded: nothing
    // touches a loaded register before the stage comes round (kPrefetch
    // stages later), so no load latency is exposed.
    uint4 ring[kPrefetch][kVec];
    __half slo[kPrefetch], shi[kPrefetch];
    auto load = [&](int i, uint4 (&w)[kVec], __half& lo, __half& hi) {
      if (LM) {
#pragma unroll
        for (int v = 0; v < kVec; ++v) w[v] = ldg_nc_v4(wt + (size_t)i * 128 + v * 16);
      } else {
        w[0] = ldg_nc_v4(wt + (size_t)(2 * i) * 2048);
        const int k0 = (s_begin + i) * kStageK;
        lo = st_[(size_t)(k0 >> gshift) * 128];
        if (two_groups) hi = st_[(size_t)((k0 + 32) >> gshift) * 128];
      }
    };
    // acc[0..8) += scale * D of the stage held in `slot`, for this half's tokens
    auto drain = [&](int slot) {
      const float2 sc = scale_s[slot][t];
      const uint32_t dbase = tmem + lane_base + slot * slot_cols + 32 + h * kHalfTok;
      uint32_t d[8];
      tc::tmem_ld8(dbase, d);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < kHalfTok; ++j) acc[j] = fmaf(sc.x, __uint_as_float(d[j]), acc[j]);
      if (two_groups) {
        tc::tmem_ld8(dbase + 16, d);
        tc::tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < kHalfTok; ++j) acc[j] = fmaf(sc.y, __uint_as_float(d[j]), acc[j]);
      }
    };
#pragma unroll
    for (int p = 0; p < kPrefetch; ++p)
      if (p < nst) load(p, ring[p], slo[p], shi[p]);
    int slot = 0;
    uint32_t phase = 0;   // parity of the `done` phase to wait for at this slot
    for (int i0 = 0; i0 < nst; i0 += kPrefetch) {
#pragma unroll
      for (int p = 0; p < kPrefetch; ++p) {
        const int i = i0 + p;
        if (i < nst) {
          uint32_t v[16];
          float2 sc = make_float2(0.f, 0.f);
          if (LM) {
#pragma unroll
            for (int q = 0; q < kVec; ++q) {
              v[4 * q] = ring[p][q].x; v[4 * q + 1] = ring[p][q].y;
              v[4 * q + 2] = ring[p][q].z; v[4 * q + 3] = ring[p][q].w;
            }
          } else {
            dq16(ring[p][0], v);
            sc.x = __half2float(slo[p]);
            sc.y = two_groups ? __half2float(shi[p]) : sc.x;
          }
          if (i + kPrefetch < nst) load(i + kPrefetch, ring[p], slo[p], shi[p]);
          if (i >= nslots) {
            if (!tc::mbar_wait(tc::smem_u32(&done_bar[slot]), phase, kWaitLimit)) ok = false;
            tc::fence_after_sync();
            if (!LM) drain(slot);   // stage i - nslots, in ascending order
          }
          if (!LM) scale_s[slot][t] = sc;
          tc::tmem_st16(tmem + lane_base + slot * slot_cols + 16 * h, v);
          tc::tmem_wait_st();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(tc::smem_u32(&full_bar[slot]));
          if (++slot == nslots) {
            slot = 0;
            if (i >= nslots) phase ^= 1u;
          }
        }
      }
    }
    if (!tc::mbar_wait(tc::smem_u32(&final_bar), 0u, kWaitLimit)) ok = false;
    tc::fence_after_sync();
    if (LM) {
      uint32_t d[8];
      tc::tmem_ld8(tmem + lane_base + lm_dcol + h * kHalfTok, d);
      tc::tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < kHalfTok; ++j) acc[j] = __uint_as_float(d[j]);
    } else {
      for (int i = (nst > nslots ? nst - nslots : 0); i < nst; ++i) drain(i % nslots);
    }
  }
  if (!ok && a.err) atomicExch(a.err, 4);

  // Producer thread t holds weight row `erow` of the tile and tokens
  // [etok, etok + 8) in acc[0..8).
  const int erow = (warp & 3) * 32 + lane, etok = (warp >> 2) * (kTokens / 2);
  const bool producer = t < kProducers;

  // ---- split-K: every split writes its partial sums; the last to arrive
  // adds them in split order and runs the epilogue
  if (ksplit > 1) {
    float* mine = a.part + ((size_t)job * ksplit + ks) * (kTokens * 128);
    if (producer) {
#pragma unroll
      for (int j = 0; j < kTokens / 2; ++j)
        if (etok + j < ntok) mine[(etok + j) * 128 + erow] = acc[j];
    }
    __threadfence();
    __syncthreads();
    if (t == 0) {
      const int prev = atomicAdd(&a.counters[job], 1);
      flag_s = (prev == ksplit - 1);
    }
    __syncthreads();
    if (!flag_s) {
      tc::fence_before_sync();
      __syncthreads();
      if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
      return;
    }
    __threadfence();
    if (producer) {
      const float* base = a.part + (size_t)job * ksplit * (kTokens * 128);
#pragma unroll
      for (int j = 0; j < kTokens / 2; ++j) {
        if (etok + j < ntok) {
          float s = 0.f;
          for (int k2 = 0; k2 < ksplit; ++k2) s += __ldcg(base + ((size_t)k2 * kTokens + etok + j) * 128 + erow);
          acc[j] = s;
        }
      }
    }
    if (t == 0) a.counters[job] = 0;
  }

  // ---- epilogue
  if (producer) {
    if (MODE == TC_DENSE) {
      const size_t n = (size_t)tile * 128 + erow;
#pragma unroll
      for (int j = 0; j < kTokens / 2; ++j) {
        if (etok + j < ntok) {
          const size_t m = row0 + etok + j;
          float v = acc[j];
          if (a.Res) v += bf2f(a.Res[m * a.ldr + n]);
          a.Y[m * a.ldy + n] = f2bf(v);
        }
      }
    } else if (MODE == TC_GATEUP) {
      // rows interleave (gate f, up f): lanes 2i and 2i+1 hold the pair
      const int f = tile * 64 + (erow >> 1);
#pragma unroll
      for (int j = 0; j < kTokens / 2; ++j) {
        const float other = __shfl_xor_sync(0xffffffffu, acc[j], 1);
        if (etok + j < ntok && (lane & 1) == 0) {
          const float gv = acc[j], uv = other;
          const float sv = gv / (1.f + expf(-gv));
          a.act[(size_t)(row0 + etok + j) * a.F + f] = f2bf(sv * uv);
        }
      }
    } else if (MODE == TC_DOWN) {
      const size_t hh = (size_t)tile * 128 + erow;
#pragma unroll
      for (int j = 0; j < kTokens / 2; ++j)
        if (etok + j < ntok) a.out[(size_t)(row0 + etok + j) * a.H + hh] = acc[j];
    } else {
      const size_t v = (size_t)tile * 128 + erow;
#pragma unroll
      for (int j = 0; j < kTokens / 2; ++j)
        if (etok + j < ntok) a.out[(size_t)(row0 + etok + j) * a.rows + v] = acc[j];
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// Canonical [N][K/2] (+ [N][K/g] scales) -> tc layout.  With `src2`, output
// row 2i is row i of `src` and row 2i+1 is row i of `src2` (gate/up pairs).
__global__ void k_repack_tc(const uint8_t* src, const __half* ssrc, const uint8_t* src2, const __half* ssrc2,
                            int rows, int K, int g, uint8_t* dst, __half* sdst) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int nch = K / 32;
  if (idx < (int64_t)rows * nch) {
    const int R = (int)(idx / nch), c = (int)(idx - (int64_t)R * nch);
    const uint8_t* s = src2 ? ((R & 1) ? src2 : src) + (size_t)(R >> 1) * (K / 2)
                            : src + (size_t)R * (K / 2);
    const uint4 in = *reinterpret_cast<const uint4*>(s + c * 16);
    const uint32_t ws[4] = {in.x, in.y, in.z, in.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t w = ws[q];
      uint32_t r = 0;
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        r |= ((w >> (8 * p)) & 0xFu) << (4 * p);            // element 2p (low nibble of byte p)
        r |= ((w >> (8 * p + 4)) & 0xFu) << (4 * (p + 4));  // element 2p+1 (high nibble)
      }
      o[q] = r;
    }
    const int tile = R >> 7, rr = R & 127;
    uint8_t* d = dst + (((size_t)tile * nch + c) * 128 + rr) * 16;
    *reinterpret_cast<uint4*>(d) = make_uint4(o[0], o[1], o[2], o[3]);
  }
  const int ng = K / g;
  if (idx < (int64_t)rows * ng) {
    const int R = (int)(idx / ng), j = (int)(idx - (int64_t)R * ng);
    const __half* s = ssrc2 ? ((R & 1) ? ssrc2 : ssrc) + (size_t)(R >> 1) * ng : ssrc + (size_t)R * ng;
    sdst[((size_t)(R >> 7) * ng + j) * 128 + (R & 127)] = s[j];
  }
}

template <int MODE>
cudaError_t run_tc(const TcArgs& a, dim3 grid, cudaStream_t st) {
  const bool two = MODE != TC_LM && a.g == 32;
  const int ks = a.ksplit < 1 ? 1 : a.ksplit;
  if ((a.K / kStageK) % ks != 0 || ks > kMaxSplit || (ks > 1 && (!a.part || !a.counters)))
    return cudaErrorInvalidValue;
  grid.x *= ks;
  const size_t smem = (size_t)kTokens * (a.K / ks) * 2;
  if (smem > (size_t)kTokens * 4096 * 2) return cudaErrorInvalidValue;
  if (two) k_w4_tc<MODE, true><<<grid, kThreads, smem, st>>>(a);
  else k_w4_tc<MODE, false><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

int tc_pick_ksplit(int /*jobs*/, int nst) {
  // The split fixes the order in which a row's partial sums are added, so it
  // depends on the reduction length only, never on how many jobs (streams,
  // active experts) share the launch: the largest split <= kMaxSplit that
  // leaves >= 4 stages per split.
  int best = 1;
  for (int ks = 2; ks <= kMaxSplit; ++ks)
    if (nst % ks == 0 && nst / ks >= 4) best = ks;
  return best;
}

size_t tc_part_floats(int jobs, int ksplit) { return (size_t)jobs * ksplit * kTokens * 128; }

bool tc_supports(int rows, int K, int g) {
  return rows > 0 && rows % 128 == 0 && K >= kStageK && K % kStageK == 0 && K <= 4096 &&
         (g == 32 || g == 64 || g == 128) && K % g == 0;
}

cudaError_t launch_repack_tc(const uint8_t* W, const __half* S, const uint8_t* W2, const __half* S2, int rows, int K,
                             int g, uint8_t* Wtc, __half* Stc, cudaStream_t st) {
  const int64_t work = (int64_t)rows * (K / 32 > K / g ? K / 32 : K / g);
  k_repack_tc<<<(unsigned)((work + 255) / 256), 256, 0, st>>>(W, S, W2, S2, rows, K, g, Wtc, Stc);
  return cudaGetLastError();
}

cudaError_t launch_w4_tc_dense(const TcArgs& a, cudaStream_t st) {
  dim3 grid(a.rows / 128, (a.ntok + kTokens - 1) / kTokens, 1);
  return run_tc<TC_DENSE>(a, grid, st);
}

cudaError_t launch_w4_tc_gateup(const TcArgs& a, int max_u, int max_tok, cudaStream_t st) {
  dim3 grid(a.rows / 128, (max_tok + kTokens - 1) / kTokens, max_u);
  return run_tc<TC_GATEUP>(a, grid, st);
}

cudaError_t launch_w4_tc_down(const TcArgs& a, int max_u, int max_tok, cudaStream_t st) {
  dim3 grid(a.rows / 128, (max_tok + kTokens - 1) / kTokens, max_u);
  return run_tc<TC_DOWN>(a, grid, st);
}

cudaError_t launch_lm_tc(const TcArgs& a, cudaStream_t st) {
  if (a.rows % 128 || a.K % kStageK) return cudaErrorInvalidValue;
  dim3 grid(a.rows / 128, (a.ntok + kTokens - 1) / kTokens, 1);
  return run_tc<TC_LM>(a, grid, st);
}

template <int MODE, bool TWO>
cudaError_t set_tc_attrs() {
  cudaError_t e =
      cudaFuncSetAttribute(k_w4_tc<MODE, TWO>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTokens * 4096 * 2);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_w4_tc<MODE, TWO>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
  return e;
}

cudaError_t init_tc_attributes() {
  cudaError_t e = set_tc_attrs<TC_DENSE, false>();
  if (e == cudaSuccess) e = set_tc_attrs<TC_DENSE, true>();
  if (e == cudaSuccess) e = set_tc_attrs<TC_GATEUP, false>();
  if (e == cudaSuccess) e = set_tc_attrs<TC_GATEUP, true>();
  if (e == cudaSuccess) e = set_tc_attrs<TC_DOWN, false>();
  if (e == cudaSuccess) e = set_tc_attrs<TC_DOWN, true>();
  if (e == cudaSuccess) e = set_tc_attrs<TC_LM, false>();
  return e;
}

}  // namespace bm
