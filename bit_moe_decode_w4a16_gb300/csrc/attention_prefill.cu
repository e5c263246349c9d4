// Causal attention of a prompt block: P rows of one slot at positions
// len .. len + P - 1 (len = the slot's length before the block), each row
// attending to positions 0 .. its own, over K/V that are all in the slot
// already (the block's rotated k and v are appended first by k_append_rows).
// ([KV-slot isolation] §1: a prompt seeds its slot once, at join.)
//
// The decode kernel (attention_mma.cu) treats every prompt row as its own
// decode query and so reads the slot's K/V once per row and per chunk; here
// a CTA takes one kv head and 16 consecutive rows and streams the K/V it
// needs once, shared by the kv group's q heads and the 16 rows (grouped-query
// attention: 8 heads x 16 rows = 128 queries per K/V tile):
//   - warp w holds q head (kv head x G + w) of the 16 rows as mma.sync A
//     fragments (rotated, rounded to bf16, as every path rotates q);
//   - K/V tiles of 64 positions arrive in shared memory by cp.async, double
//     buffered;
//   - S = Q K^T with mma.sync m16n8k16 (bf16 operands, fp32 accumulators),
//     scaled by 1/sqrt(d), positions after the row's own masked;
//   - a running softmax per row (maximum m, sum l of exp(s - m); earlier
//     partial sums rescaled by exp(m_old - m_new) when the maximum grows);
//   - O += P V with P in fp16 (the probabilities, in [0, 1]) and V converted
//     from bf16 to fp16 (exact inside fp16's range), fp32 accumulators;
//   - out = O / l, rounded to bf16 and stored as fp16 (the form the output
//     projection reads), as the decode kernel stores it.
// The arithmetic differs from the decode kernel's (one running softmax
// instead of 128-position chunks merged afterwards), so a prompt row is not
// bit-identical to the same row decoded; both are exact attention up to fp32
// rounding.
#include <float.h>

#include "attn_fused.cuh"

namespace bm {

namespace {

constexpr int kPaRows = 16;      // prompt rows per CTA
constexpr int kPaWarps = 8;      // one q head of the kv group per warp
constexpr int kPaThreads = kPaWarps * 32;
constexpr int kPaPos = 64;       // positions per K/V tile

template <int D>
struct PaSmem {
  static constexpr int kP = D + 8;   // padded row: conflict-free fragment loads and ldmatrix
  bf16 k[2][kPaPos][kP];
  bf16 v[2][kPaPos][kP];
  bf16 q[kPaWarps][kPaRows][kP];
};

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], const void* p) {
  const uint32_t addr = static_cast<uint32_t>(__cvta_generic_to_shared(p));
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ uint32_t lds32(const bf16* p) { return *reinterpret_cast<const uint32_t*>(p); }

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

template <int D>
__global__ void __launch_bounds__(kPaThreads, 1) k_attn_prefill(AttnFusedArgs a) {
  extern __shared__ __align__(16) unsigned char pa_raw[];
  PaSmem<D>& sm = *reinterpret_cast<PaSmem<D>*>(pa_raw);
  constexpr int kKS = D / 16;   // k-steps of Q K^T
  constexpr int kNT = D / 8;    // n-tiles of O
  const AttnArena& ar = a.ar;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int kh = blockIdx.x, t0 = blockIdx.y * kPaRows;
  const int kvh = ar.kvh, G = a.qh / kvh, half = D / 2;
  const int slot = a.slots[0];
  if (slot < 0 || slot >= ar.S) {
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) a.chk.fail(1);
    return;
  }
  const int len0 = ar.len[slot];
  const int rows = min(kPaRows, a.B - t0);
  const int p_last = len0 + t0 + rows - 1;   // the last position any row of the CTA reads
  if (len0 < 0 || p_last >= ar.cap) {
    if (tid == 0) a.chk.fail(2);
    return;
  }
  const size_t base = (size_t)a.layer * ar.layer_stride() + (size_t)slot * ar.slot_stride() + (size_t)kh * ar.cap * D;
  const bf16* Kb = ar.K + base;
  const bf16* Vb = ar.V + base;
  const int ntiles = p_last / kPaPos + 1;

  auto load_tile = [&](int tile, int buf) {
    const int p0 = tile * kPaPos;
    for (int i = tid; i < kPaPos * (D / 8); i += kPaThreads) {
      const int r = i / (D / 8), c8 = i - r * (D / 8), p = p0 + r;
      if (p <= p_last) {
        cp_async16(&sm.k[buf][r][c8 * 8], Kb + (size_t)p * D + c8 * 8);
        cp_async16(&sm.v[buf][r][c8 * 8], Vb + (size_t)p * D + c8 * 8);
      } else {
        *reinterpret_cast<uint4*>(&sm.k[buf][r][c8 * 8]) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(&sm.v[buf][r][c8 * 8]) = make_uint4(0, 0, 0, 0);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  load_tile(0, 0);

  // ---- q of the kv group's heads for the CTA's rows, rotated at each row's
  // position and rounded to bf16 (rows past the block: zeros, never stored);
  // a thread takes 8 rotation pairs at a time, all its loads before any store
  constexpr int kQ8 = D / 16;                                   // groups of 8 pairs in a head
  constexpr int kQIt = kPaWarps * kPaRows * kQ8 / kPaThreads;   // 4 (d 128) or 2 (d 64)
  static_assert(kQIt * kPaThreads == kPaWarps * kPaRows * kQ8, "q split");
  uint4 x0v[kQIt], x1v[kQIt];
  float4 csv[kQIt][4];
#pragma unroll
  for (int it = 0; it < kQIt; ++it) {
    const int idx = tid + it * kPaThreads, h = idx / (kPaRows * kQ8), rem = idx - h * (kPaRows * kQ8);
    const int r = rem / kQ8, i8 = (rem - r * kQ8) * 8;
    x0v[it] = x1v[it] = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int c = 0; c < 4; ++c) csv[it][c] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (h < G && r < rows) {
      const bf16* src = a.qkv + (size_t)(t0 + r) * a.ld_qkv + (size_t)(kh * G + h) * D;
      x0v[it] = *reinterpret_cast<const uint4*>(src + i8);
      x1v[it] = *reinterpret_cast<const uint4*>(src + half + i8);
      const float4* cs = reinterpret_cast<const float4*>(a.rope + (size_t)(len0 + t0 + r) * half + i8);
#pragma unroll
      for (int c = 0; c < 4; ++c) csv[it][c] = cs[c];
    }
  }
#pragma unroll
  for (int it = 0; it < kQIt; ++it) {
    const int idx = tid + it * kPaThreads, h = idx / (kPaRows * kQ8), rem = idx - h * (kPaRows * kQ8);
    const int r = rem / kQ8, i8 = (rem - r * kQ8) * 8;
    const bf16* x0 = reinterpret_cast<const bf16*>(&x0v[it]);
    const bf16* x1 = reinterpret_cast<const bf16*>(&x1v[it]);
    const float* cs = reinterpret_cast<const float*>(&csv[it][0]);   // (cos, sin) pairs
    bf16 y0[8], y1[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) attnf::rope_pair(bf2f(x0[e]), bf2f(x1[e]), cs[2 * e], cs[2 * e + 1], y0[e], y1[e]);
    *reinterpret_cast<uint4*>(&sm.q[h][r][i8]) = *reinterpret_cast<const uint4*>(y0);
    *reinterpret_cast<uint4*>(&sm.q[h][r][half + i8]) = *reinterpret_cast<const uint4*>(y1);
  }
  __syncthreads();
  uint32_t qa[kKS][4];
#pragma unroll
  for (int ks = 0; ks < kKS; ++ks) {
    qa[ks][0] = lds32(&sm.q[warp][g][16 * ks + 2 * t]);
    qa[ks][1] = lds32(&sm.q[warp][g + 8][16 * ks + 2 * t]);
    qa[ks][2] = lds32(&sm.q[warp][g][16 * ks + 8 + 2 * t]);
    qa[ks][3] = lds32(&sm.q[warp][g + 8][16 * ks + 8 + 2 * t]);
  }

  const float scale = 1.0f / sqrtf((float)D);
  const int pr0 = len0 + t0 + g, pr1 = pr0 + 8;   // positions of the lane's two rows
  float m0 = -FLT_MAX, m1 = -FLT_MAX, l0 = 0.f, l1 = 0.f;
  float o[kNT][4];
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[nt][c] = 0.f;

  for (int tile = 0; tile < ntiles; ++tile) {
    const int buf = tile & 1;
    if (tile + 1 < ntiles) {
      load_tile(tile + 1, buf ^ 1);
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    } else {
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    }
    __syncthreads();
    const int p0 = tile * kPaPos;
    // ---- S = Q K^T over the tile's 64 positions: 8 n-tiles of 8
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int c = 0; c < 4; ++c) s[j][c] = 0.f;
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
        const uint32_t b0 = lds32(&sm.k[buf][8 * j + g][16 * ks + 2 * t]);
        const uint32_t b1 = lds32(&sm.k[buf][8 * j + g][16 * ks + 8 + 2 * t]);
        mma::mma_bf16(s[j], qa[ks], b0, b1);
      }
    }
    // ---- scale, mask, the running softmax of the lane's two rows
    float mx0 = -FLT_MAX, mx1 = -FLT_MAX;
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int p = p0 + 8 * j + 2 * t + c;
        s[j][c] = p <= pr0 ? s[j][c] * scale : -FLT_MAX;
        s[j][c + 2] = p <= pr1 ? s[j][c + 2] * scale : -FLT_MAX;
        mx0 = fmaxf(mx0, s[j][c]);
        mx1 = fmaxf(mx1, s[j][c + 2]);
      }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float c0 = expf(m0 - mn0), c1 = expf(m1 - mn1);   // 0 on the first tile (m = -FLT_MAX)
    m0 = mn0;
    m1 = mn1;
    l0 *= c0;
    l1 *= c1;
#pragma unroll
    for (int nt = 0; nt < kNT; ++nt) {
      o[nt][0] *= c0;
      o[nt][1] *= c0;
      o[nt][2] *= c1;
      o[nt][3] *= c1;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int p = p0 + 8 * j + 2 * t + c;
        s[j][c] = p <= pr0 ? expf(s[j][c] - m0) : 0.f;
        s[j][c + 2] = p <= pr1 ? expf(s[j][c + 2] - m1) : 0.f;
        l0 += s[j][c];
        l1 += s[j][c + 2];
      }
    // ---- O += P V: 4 k-steps of 16 positions; P from the score registers
#pragma unroll
    for (int kp = 0; kp < 4; ++kp) {
      const uint32_t pa[4] = {pack_f16(s[2 * kp][0], s[2 * kp][1]), pack_f16(s[2 * kp][2], s[2 * kp][3]),
                              pack_f16(s[2 * kp + 1][0], s[2 * kp + 1][1]),
                              pack_f16(s[2 * kp + 1][2], s[2 * kp + 1][3])};
      const int vrow = 16 * kp + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int dt = 0; dt < kNT / 2; ++dt) {
        uint32_t vb[4];
        ldsm_x4_trans(vb, &sm.v[buf][vrow][16 * dt + (lane >> 4) * 8]);
#pragma unroll
        for (int q = 0; q < 4; ++q) vb[q] = mma::bf2_to_h2(vb[q]);   // exact: V is bf16 inside fp16's range
        mma::mma_f16(o[2 * dt], pa, vb[0], vb[1]);
        mma::mma_f16(o[2 * dt + 1], pa, vb[2], vb[3]);
      }
    }
    __syncthreads();   // the tile's buffer is refilled next
  }
  // ---- the row sums over the quad, then out = O / l
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  if (warp >= G) return;
  const int h = kh * G + warp;
#pragma unroll
  for (int nt = 0; nt < kNT; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int d = 8 * nt + 2 * t + c;
      if (g < rows)
        a.out[((size_t)(t0 + g) * a.qh + h) * D + d] = __float2half_rn(round_bf16(o[nt][c] / l0));
      if (g + 8 < rows)
        a.out[((size_t)(t0 + g + 8) * a.qh + h) * D + d] = __float2half_rn(round_bf16(o[nt][c + 2] / l1));
    }
}

template <int D>
cudaError_t launch_d(const AttnFusedArgs& a, cudaStream_t st) {
  const size_t smem = sizeof(PaSmem<D>);
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_attn_prefill<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const dim3 grid((unsigned)a.ar.kvh, (unsigned)((a.B + kPaRows - 1) / kPaRows));
  k_attn_prefill<D><<<grid, kPaThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

bool attention_prefill_supports(const AttnArena& ar, int qh) {
  return (ar.d == 64 || ar.d == 128) && qh % ar.kvh == 0 && qh / ar.kvh <= kPaWarps;
}

cudaError_t launch_attention_prefill(const AttnFusedArgs& a, cudaStream_t st) {
  if (!attention_prefill_supports(a.ar, a.qh) || a.B < 1 || a.B > 65535 * kPaRows) return cudaErrorInvalidValue;
  return a.ar.d == 128 ? launch_d<128>(a, st) : launch_d<64>(a, st);
}

}  // namespace bm
