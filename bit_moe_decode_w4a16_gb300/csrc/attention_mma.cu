// Fused decode attention of the warp-MMA family: RoPE of q and of the new k,
// the append of the new k and v to the stream's slot, split-K attention over
// 128-position chunks on the tensor cores, and the ordered merge of a
// stream's chunks, in one persistent launch.
//
// Work items are (stream, kv head, chunk); each CTA reads the slot lengths
// once and enumerates only the chunks that exist, so no CTA is spent on
// positions past a stream's length.  CTA i runs item i; a launch with more
// items than CTAs hands out the rest through a work queue, one item per claim
// by a CTA that has finished its previous one.  For one item the CTA:
//   - issues all of the item's loads before any arithmetic: the chunk's V rows
//     to shared memory (cp.async), the lane's K rows to registers, the
//     rotation table entries, q and the new k / v;
//   - rotates the kv group's G query heads (rotate-half, cos/sin of the
//     position from the table) into shared memory as bf16; on the chunk that
//     holds a decode row's new position it also rotates the new k, writes k
//     and v to the arena at that position, and uses the rotated k (and v
//     straight from the row) for that position instead of the arena, so the
//     chunk never waits for its own append;
//   - computes S = Q K^T with mma.sync m16n8k16 (bf16): the G heads on M
//     (rows past G are zero), 8 positions per n-tile on N, the head dimension
//     on K.  Inside each 32-wide block of d a lane takes the 8 consecutive
//     elements 8t..8t+7 of both q and its K row (the same permutation of the
//     reduction on both operands), so K rows are read straight from memory
//     as 16-byte loads;
//   - takes the chunk's softmax statistics (max m, sum l of exp(s - m)) per
//     head over its 8 warps in a fixed order;
//   - computes O = P V in fp16 (P reused from the score registers as the A
//     operand, V through ldmatrix.trans and converted from bf16 exactly),
//     warp w over its 16 positions, and adds the 8 warps' partials in warp
//     order;
//   - a stream of one chunk writes o / l directly; otherwise the CTA writes
//     the chunk's record (o, m, l) and, if it is the last chunk of its
//     (stream, kv head) to finish (arrival counter), merges all of that
//     stream's chunks in ascending order: M = max m_c, den = sum l_c e^(m_c - M),
//     out = (sum o_c e^(m_c - M)) / den, rounded to bf16 and stored as fp16
//     (with one chunk the weight is e^0 = 1 and both ways give the same bits).
// A stream's result depends only on its own length and data.
//
// Prompt ingestion runs the same kernel over rows that all belong to one
// slot: row b sits at position len + b and attends causally to positions
// 0..len + b.  The rows' rotated k and v are written by k_append_rows first
// (a row reads positions that other rows of the launch produce), and the
// kernel then skips its own append; a row's arithmetic is that of a decode
// step at the same position, so both paths leave the same bytes.
#include "attn_fused.cuh"

namespace bm {

namespace {

using namespace attnf;

template <int D>
__global__ void __launch_bounds__(kWarpsA * 32, 3) k_attn_fused(AttnFusedArgs a) {
  __shared__ __align__(16) AttnSmem<D> sm;
  // The prologue reads only the slot ids (uploaded before the step) and the
  // slot lengths (advanced by the previous step's last launch, which had
  // completed before this launch's predecessor took its own dependency
  // wait), so it runs before this launch's wait; q, k and v come after it.
  const int grid = gridDim.x;
  const int total = attn_prologue<D>(a, sm, blockIdx.x == 0, CtaSync{}, grid);
  pdl_wait();
  pdl_trigger();   // the grid is at most one wave: the output projection may start its weight loads
  // More items than CTAs: after its first item a CTA claims the next one from
  // the launch's queue once it has finished, merges included.  With a fixed
  // stride a CTA that merged started its next item late, was then likely the
  // last arrival of that item's stream again and inherited its merge too; a
  // claim made when the CTA is free gives it the item that the other CTAs
  // free at that moment are also starting.  Which CTA runs an item does not
  // change what the item computes.
  const bool queued = total > grid;
  unsigned int* queue = a.counters + attn_queue_index(a.B, a.ar.kvh);   // [0] claims, [1] CTAs done
  for (int it = blockIdx.x; it < total;) {
    attn_item<D>(a, sm, it, CtaSync{});   // ends with a CTA barrier: every thread has read sm.next
    if (!queued) break;
    if (threadIdx.x == 0) sm.next = grid + (int)atomicAdd(queue, 1u);
    __syncthreads();
    it = sm.next;
  }
  if (queued && threadIdx.x == 0) {
    __threadfence();   // this CTA's last claim is performed before its done count
    if (atomicAdd(queue + 1, 1u) == (unsigned)grid - 1) {
      __threadfence();
      queue[0] = 0u;   // every CTA has made its last claim: leave the queue zero
      queue[1] = 0u;
    }
  }
}

// Rotated k and v of every row to the arena at the row's position: one CTA
// per (row, kv head).
template <int D>
__global__ void __launch_bounds__(64) k_append_rows(AttnFusedArgs a) {
  pdl_wait();
  const AttnArena& ar = a.ar;
  const int b = blockIdx.x, kh = blockIdx.y, half = D / 2;
  const int slot = a.slots[b];
  if (slot < 0 || slot >= ar.S) {
    if (threadIdx.x == 0) a.chk.fail(1);
    return;
  }
  const int pos = row_position(a, b, slot);
  if (pos < 0 || pos >= ar.cap) {
    if (threadIdx.x == 0) a.chk.fail(2);
    return;
  }
  const bf16* row = a.qkv + (size_t)b * a.ld_qkv;
  const bf16* ksrc = row + (size_t)(a.qh + kh) * D;
  const bf16* vsrc = row + (size_t)(a.qh + ar.kvh + kh) * D;
  const size_t base = (size_t)a.layer * ar.layer_stride() + (size_t)slot * ar.slot_stride() +
                      (size_t)kh * ar.cap * D + (size_t)pos * D;
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    const float2 cs = a.rope[(size_t)pos * half + i];
    rope_pair(bf2f(ksrc[i]), bf2f(ksrc[i + half]), cs.x, cs.y, ar.K[base + i], ar.K[base + i + half]);
  }
  for (int i = threadIdx.x; i < D; i += blockDim.x) ar.V[base + i] = vsrc[i];
}

}  // namespace

bool attention_fused_supports(const AttnArena& ar, int qh) {
  return (ar.d == 64 || ar.d == 128) && qh % ar.kvh == 0 && qh / ar.kvh <= 8 &&
         (ar.cap + kAttnChunk - 1) / kAttnChunk <= kMaxMergeChunks;
}

cudaError_t launch_attention_fused(const AttnFusedArgs& a, cudaStream_t st, bool pdl) {
  if (!attention_fused_supports(a.ar, a.qh) || a.B < 1 || a.B > kMaxBatch || !a.counters) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    sms = 132;
  const long items = (long)a.B * a.ar.kvh * a.max_chunks;
  const long cap = (long)sms * 3;   // resident CTAs per SM
  const dim3 grid((unsigned)(items < cap ? items : cap));
  if (a.ar.d == 128) return launch_k(pdl, k_attn_fused<128>, grid, dim3(kWarpsA * 32), 0, st, a);
  return launch_k(pdl, k_attn_fused<64>, grid, dim3(kWarpsA * 32), 0, st, a);
}

cudaError_t launch_append_rows(const AttnFusedArgs& a, cudaStream_t st, bool pdl) {
  if (!attention_fused_supports(a.ar, a.qh) || a.B < 1 || a.B > 65535) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)a.B, (unsigned)a.ar.kvh);
  if (a.ar.d == 128) return launch_k(pdl, k_append_rows<128>, grid, dim3(64), 0, st, a);
  return launch_k(pdl, k_append_rows<64>, grid, dim3(64), 0, st, a);
}

}  // namespace bm
