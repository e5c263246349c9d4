// Tensor-core (tcgen05) W4A16 projections: dense Y = X·Wᵀ and the grouped
// expert gate/up and down GEMMs.
//
// One CTA of 128 threads owns a tile of 128 weight rows and up to 16 tokens
// (M = 128 weight rows x N = 16 tokens: the large dimension on the MMA's M).
// Thread t streams the packed int4 of row t, turns each code into the exact
// fp16 integer q - 8 in registers and writes it with tcgen05.st into TMEM
// lane t, where it is the MMA's A operand; the tokens' activations (fp16) sit
// in shared memory as the B operand.  Each 64-wide K stage accumulates into
// its own fp32 TMEM region (one per 32-wide half, so every region covers a
// single int4 group when g >= 32): the products q * x are exact in fp32, and
// the threads apply the fp32 group scale when they drain the region, so the
// weights are never rounded.  Three stages rotate through TMEM: before
// rewriting a stage's columns the producers wait on its mbarrier (arrived by
// tcgen05.commit when the MMAs that read it finish) and drain its
// accumulator.  A row's result is the sum over stages in ascending K of
// scale * (exact group sum), whatever the other tokens of the tile are.
//
// Weight layout ("tc layout", written once by the repack kernel): for tile
// t, stage s (64 K) and half h (32 K): 128 rows x 16 bytes, row-contiguous,
// so a warp's loads of one half are 512 contiguous bytes.  Inside each 32-bit
// word the 8 codes are ordered (k0 k2 k4 k6 k1 k3 k5 k7), so one
// (w >> 4i) & 0x000F000F | 0x64006400 yields the fp16 pair (1024 + u_2i,
// 1024 + u_2i+1) of one TMEM column.  Scales: [tile][K/g][128 rows] fp16.
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace bm {

namespace {

constexpr int kThreads = 128;
constexpr int kTokens = 16;            // MMA N
constexpr int kStageK = 64;            // K per stage: A 32 columns, D 2 x 16 columns
constexpr int kStages = 3;             // stages in TMEM
constexpr int kSlotCols = 64;
constexpr uint32_t kTmemCols = 256;
constexpr int kPrefetch = 6;           // stages of weights in flight per thread
constexpr uint32_t kWaitLimit = 1u << 22;

// (u_lo, u_hi) codes of one TMEM column -> the fp16 pair (u_lo - 8, u_hi - 8), exact.
__device__ __forceinline__ uint32_t dq_pair(uint32_t w, int i) {
  const uint32_t v = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;   // (1024 + u_lo, 1024 + u_hi)
  __half2 h = *reinterpret_cast<const __half2*>(&v);
  h = __hsub2(h, __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408)));   // - 1032
  return *reinterpret_cast<uint32_t*>(&h);
}

// 16 packed bytes (32 codes) -> 16 TMEM columns of fp16 pairs.
__device__ __forceinline__ void dq16(const uint4 w, uint32_t* out) {
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int i = 0; i < 4; ++i) out[q * 4 + i] = dq_pair(ws[q], i);
}

enum TcMode { TC_DENSE = 0, TC_GATEUP = 1, TC_DOWN = 2 };

template <int MODE>
__global__ void __launch_bounds__(kThreads) k_w4_tc(TcArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t mbar[kStages + 1];
  __shared__ uint32_t tmem_slot;
  __shared__ float rinv_s[kTokens];
  __shared__ float2 scale_s[kStages][kThreads];   // group scales of the stage in each slot
  __shared__ int abort_s;

  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int tile = blockIdx.x, tg = blockIdx.y;
  const int K = a.K;
  const uint8_t* W = a.W;
  const __half* S = a.S;
  int ntok, row0 = 0;   // tokens of this CTA; first pair / row index
  if (MODE == TC_DENSE) {
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

  // ---- TMEM and barriers
  if (warp == 0) {
    tc::tmem_alloc(tc::smem_u32(&tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  if (t == 0) {
    for (int i = 0; i <= kStages; ++i) tc::mbar_init(tc::smem_u32(&mbar[i]), 1);
    tc::fence_mbar_init();
    abort_s = 0;
  }

  // ---- activations -> shared memory, fp16, no-swizzle K-major core matrices.
  // Warp w stages rows w, w+4, ...; a lane's chunks of a row are loaded
  // together (up to 16 x 16 bytes in flight) before they are used.
  const int nk8 = K / 8;
  const uint32_t sbo = (uint32_t)nk8 * 128u;   // bytes between the two 8-row groups
  for (int r = warp; r < kTokens; r += kThreads / 32) {
    unsigned char* rowp = smem + (r >> 3) * sbo + (r & 7) * 16;
    if (r >= ntok) {
      for (int j = lane; j < nk8; j += 32) *reinterpret_cast<uint4*>(rowp + j * 128) = make_uint4(0, 0, 0, 0);
      continue;
    }
    const bf16* x;
    if (MODE == TC_GATEUP) x = a.X + (size_t)a.pair_token[row0 + r] * a.ldx;
    else x = a.X + (size_t)(row0 + r) * a.ldx;
    constexpr int kMaxChunks = 4096 / 8 / 32;   // K <= 4096
    uint4 raw[kMaxChunks];
#pragma unroll
    for (int i = 0; i < kMaxChunks; ++i)
      if (lane + 32 * i < nk8) raw[i] = *reinterpret_cast<const uint4*>(x + (lane + 32 * i) * 8);
    float rinv = 1.f;
    if (MODE == TC_DENSE && a.do_norm) {
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxChunks; ++i) {
        if (lane + 32 * i < nk8) {
          const uint32_t rw[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float v0 = bf_lo(rw[q]), v1 = bf_hi(rw[q]);
            ss = fmaf(v0, v0, ss);
            ss = fmaf(v1, v1, ss);
          }
        }
      }
      ss = warp_sum(ss);
      rinv = 1.0f / sqrtf(ss / (float)K + a.eps);
    }
#pragma unroll
    for (int i = 0; i < kMaxChunks; ++i) {
      const int j = lane + 32 * i;
      if (j < nk8) {
        const uint32_t rw[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float v0 = bf_lo(rw[q]), v1 = bf_hi(rw[q]);
          if (MODE == TC_DENSE && a.do_norm) {
            const float w0 = a.norm_w ? bf2f(a.norm_w[j * 8 + 2 * q]) : 1.f;
            const float w1 = a.norm_w ? bf2f(a.norm_w[j * 8 + 2 * q + 1]) : 1.f;
            v0 = round_bf16(v0 * rinv * w0);
            v1 = round_bf16(v1 * rinv * w1);
          }
          __half2 h = __floats2half2_rn(v0, v1);
          o[q] = *reinterpret_cast<uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(rowp + j * 128) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t b_base = tc::smem_u32(smem);
  const uint32_t idesc = tc::idesc_f16_f32(128, kTokens);

  // ---- main loop over K stages
  const int nst = K / kStageK;
  const int ng = K / a.g;
  const uint8_t* wt = W + (size_t)tile * nst * 2 * 2048 + (size_t)t * 16;
  const __half* st_ = S + (size_t)tile * ng * 128 + t;
  uint4 ring[kPrefetch][2];
  __half sring[kPrefetch][2];
  auto load = [&](int s, uint4 (&w)[2], __half (&sc)[2]) {
    w[0] = ldg_nc_v4(wt + (size_t)(s * 2) * 2048);
    w[1] = ldg_nc_v4(wt + (size_t)(s * 2 + 1) * 2048);
    sc[0] = st_[(size_t)((s * kStageK) / a.g) * 128];
    sc[1] = st_[(size_t)((s * kStageK + 32) / a.g) * 128];
  };
  float acc[kTokens];
#pragma unroll
  for (int j = 0; j < kTokens; ++j) acc[j] = 0.f;
  // acc += scale_lo * D_lo + scale_hi * D_hi of the stage held in `slot`
  auto drain = [&](int slot) {
    uint32_t d[32];
    tc::tmem_ld32(tmem + lane_base + slot * kSlotCols + 32, d);
    tc::tmem_wait_ld();
    const float2 sc = scale_s[slot][t];
#pragma unroll
    for (int j = 0; j < kTokens; ++j) {
      acc[j] = fmaf(sc.x, __uint_as_float(d[j]), acc[j]);
      acc[j] = fmaf(sc.y, __uint_as_float(d[16 + j]), acc[j]);
    }
  };
#pragma unroll
  for (int p = 0; p < kPrefetch; ++p)
    if (p < nst) load(p, ring[p], sring[p]);
  bool ok = true;
  for (int s0 = 0; s0 < nst; s0 += kPrefetch) {
#pragma unroll
    for (int p = 0; p < kPrefetch; ++p) {
      const int s = s0 + p;
      if (s < nst) {
        const uint4 w0 = ring[p][0], w1 = ring[p][1];
        const float2 sc = make_float2(__half2float(sring[p][0]), __half2float(sring[p][1]));
        if (s + kPrefetch < nst) load(s + kPrefetch, ring[p], sring[p]);
        uint32_t v[32];
        dq16(w0, v);
        dq16(w1, v + 16);
        const int slot = s % kStages;
        if (s >= kStages) {
          if (!abort_s &&
              !tc::mbar_wait(tc::smem_u32(&mbar[slot]), (uint32_t)((s / kStages) - 1) & 1u, kWaitLimit)) {
            abort_s = 1;
            ok = false;
          }
          tc::fence_after_sync();
          drain(slot);   // stage s - kStages, in ascending order
        }
        scale_s[slot][t] = sc;
        tc::tmem_st32(tmem + lane_base + slot * kSlotCols, v);
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncthreads();
        if (t == 0) {
          tc::fence_after_sync();
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint64_t bd = tc::smem_desc_noswizzle(b_base + (uint32_t)(s * 4 + q) * 256u, 128u, sbo);
            const uint32_t dcol = slot * kSlotCols + 32 + (q >> 1) * 16;
            tc::mma_f16_tmem_a(tmem + dcol, tmem + slot * kSlotCols + q * 8, bd, idesc, (uint32_t)(q & 1));
          }
          tc::mma_commit(tc::smem_u32(&mbar[slot]));
          if (s == nst - 1) tc::mma_commit(tc::smem_u32(&mbar[kStages]));
        }
      }
    }
  }

  // ---- drain the last stages, then the epilogue: lane t = weight row t
  if (!tc::mbar_wait(tc::smem_u32(&mbar[kStages]), 0u, kWaitLimit)) ok = false;
  tc::fence_after_sync();
  for (int s = (nst > kStages ? nst - kStages : 0); s < nst; ++s) drain(s % kStages);
  if (!ok && a.err) atomicExch(a.err, 4);
  if (MODE == TC_DENSE) {
    const size_t n = (size_t)tile * 128 + t;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j < ntok) {
        const size_t m = row0 + j;
        float v = acc[j];
        if (a.Res) v += bf2f(a.Res[m * a.ldr + n]);
        a.Y[m * a.ldy + n] = f2bf(v);
      }
    }
  } else if (MODE == TC_GATEUP) {
    // rows interleave (gate f, up f): lanes 2i and 2i+1 hold the pair
    const int f = tile * 64 + (t >> 1);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float other = __shfl_xor_sync(0xffffffffu, acc[j], 1);
      if (j < ntok && (t & 1) == 0) {
        const float gv = acc[j], uv = other;
        const float sv = gv / (1.f + expf(-gv));
        a.act[(size_t)(row0 + j) * a.F + f] = f2bf(sv * uv);
      }
    }
  } else {
    const size_t h = (size_t)tile * 128 + t;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < ntok) a.out[(size_t)(row0 + j) * a.H + h] = acc[j];
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
    const int tile = R >> 7, rr = R & 127, st = c >> 1, h = c & 1;
    uint8_t* d = dst + ((((size_t)tile * (K / kStageK) + st) * 2 + h) * 128 + rr) * 16;
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
  const size_t smem = (size_t)kTokens * a.K * 2;
  k_w4_tc<MODE><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

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

cudaError_t init_tc_attributes() {
  const int bytes = kTokens * 4096 * 2;
  cudaError_t e = cudaFuncSetAttribute(k_w4_tc<TC_DENSE>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_w4_tc<TC_GATEUP>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_w4_tc<TC_DOWN>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  return e;
}

}  // namespace bm
