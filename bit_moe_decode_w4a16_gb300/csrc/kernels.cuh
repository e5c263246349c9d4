// Launchers of the decode-step kernels.  Each returns cudaSuccess or the
// launch error; none synchronises.
#pragma once

#include "common.cuh"

namespace bm {

// Kernel classes of one decode step (for the per-kernel profiler).
enum KernelTag {
  KT_EMBED = 0, KT_QKV, KT_ROPE_APPEND, KT_ATTN_PART, KT_ATTN_COMBINE, KT_OPROJ, KT_ROUTER, KT_TOPK_SORT,
  KT_GATEUP, KT_DOWN, KT_COMBINE, KT_LM_HEAD, KT_ARGMAX, KT_COUNT
};

// Called after each kernel launch with its class; a no-op unless profiling.
struct Marker {
  void (*fn)(void* ctx, int tag) = nullptr;
  void* ctx = nullptr;
  void operator()(int tag) const {
    if (fn) fn(ctx, tag);
  }
};

// ---------------------------------------------------------------- dense
struct GemvArgs {
  const uint8_t* W;   // packed int4 [N][K/2]
  const __half* S;    // fp16 [N][K/g]
  const bf16* X;      // [M][ldx]
  int ldx;
  const bf16* Res;    // [M][ldr] or null
  int ldr;
  bf16* Y;            // [M][ldy]
  int ldy;
  int M, N, K, g;
  int do_norm;        // stage RMSNorm(X) instead of X
  const bf16* norm_w; // [K] or null
  float eps;
};
// True if the CUDA-core W4 kernels handle reduction length K.
bool simt_supports_k(int K);
cudaError_t launch_w4_gemv(const GemvArgs& a, cudaStream_t st);

// ---------------------------------------------------------------- experts
struct MoeBufs {
  // routing
  float* logits;        // [B][E]
  int32_t* topk_ids;    // [B][k]
  float* topk_w;        // [B][k]
  bf16* xn;             // [B][H] normed router / expert input (written when norm is fused)
  // grouping (counting sort of the B*k (token, rank) pairs by expert)
  int32_t* n_active;    // [1]
  int32_t* active_e;    // [E]
  int32_t* active_off;  // [E+1]
  int32_t* pair_token;  // [B*k] token of the p-th pair in expert order
  int32_t* pos_of;      // [B*k] sorted position of pair (b, r) = b*k + r
  // work list of the warp-MMA expert kernels, in expert order: job j =
  // e | first << 9 | n << 21 is the n (<= 8) sorted pairs first.. of expert e
  int32_t* n_jobs;      // [1]
  int32_t* jobs;        // [moe_max_jobs(B, E, k)]
  bf16* act;            // [B*k][F]
  float* out;           // [B*k][H]
};
size_t moe_scratch_bytes(int B, int E, int k, int H, int F);
MoeBufs moe_carve(void* ws, int B, int E, int k, int H, int F);
// Upper bound of the job count: sum over active experts of ceil(count / 8)
// <= min(E, B k) + B k / 8.
int moe_max_jobs(int B, int E, int k);
constexpr int kJobTokens = 8;

struct MoeArgs {
  int B, E, k, H, F, g, renorm;
  const float* wr;                 // [E][H]
  const uint8_t* wg; const __half* wg_s;
  const uint8_t* wu; const __half* wu_s;
  const uint8_t* wd; const __half* wd_s;
  const bf16* x;                   // [B][H] input (raw when do_norm)
  int do_norm;                     // route/experts on RMSNorm(x) (written to bufs.xn)
  const bf16* norm_w;
  float eps;
  const bf16* res;                 // [B][H] residual or null
  bf16* y;                         // [B][H]
  int32_t* u_log;                  // if set, the number of active experts is also written here
  int xn_f16;                      // the router writes bufs.xn as fp16 (warp-MMA experts)
};
// Router logits + top-k + sort, gate/up, down, combine: 5 launches.
cudaError_t launch_moe(const MoeArgs& a, const MoeBufs& b, cudaStream_t st, int* launches,
                       const Marker& mark = Marker());
// The routing half (router logits, top-k + sort: 2 launches) and the
// combine (1 launch) on their own, for the tensor-core expert path.
cudaError_t launch_moe_route(const MoeArgs& a, const MoeBufs& b, cudaStream_t st, const Marker& mark);
cudaError_t launch_moe_combine(const MoeArgs& a, const MoeBufs& b, cudaStream_t st, const Marker& mark);
// Router + top-k + sort in one launch (the same results as launch_moe_route).
// tok_cnt [B] and all_cnt [1] are zero before the launch and left zero.
cudaError_t launch_moe_route_fused(const MoeArgs& a, const MoeBufs& b, unsigned int* tok_cnt, unsigned int* all_cnt,
                                  cudaStream_t st, const Marker& mark, bool pdl = false);
// Routing of a prompt block of up to 4096 (row, rank) pairs: router logits
// with the RMSNorm (bufs.xn written, fp16 with xn_f16), top-k per row, and the
// stable grouping by expert (pair_token, pos_of, n_active, active_e,
// active_off; and the prompt GEMM jobs, see kPromptTileRows).  Three launches.
cudaError_t launch_moe_route_wide(const MoeArgs& a, const MoeBufs& b, cudaStream_t st);
// Rows per expert tile of the prompt-length expert GEMMs: the wide grouping
// lists jobs (active expert u, tile t of kPromptTileRows of its rows) as
// u | t << 16 in bufs.jobs, their number in bufs.n_jobs.
constexpr int kPromptTileRows = 128;
// The combine with the next RMSNorm fused: also xn[b] = RMSNorm(y[b]) * nw
// (nw null = ones; a.eps), rounded to bf16 and stored as fp16 (xn_f16) or
// bf16.  H <= 8192.
cudaError_t launch_moe_combine_norm(const MoeArgs& a, const MoeBufs& b, const bf16* nw, void* xn, int xn_f16,
                                    cudaStream_t st, const Marker& mark, bool pdl = false);
// The same for the rows of a prompt (a.B rows), a CTA per row with 8
// elements per thread: each element's combine is the same; the squares of
// the norm meet in another order.  Falls back to launch_moe_combine_norm
// where k > 8 or H is not a multiple of 8 or above 4096.
cudaError_t launch_moe_combine_norm_rows(const MoeArgs& a, const MoeBufs& b, const bf16* nw, void* xn, int xn_f16,
                                         cudaStream_t st);

// ---------------------------------------------------------------- tensor-core W4A16
struct TcArgs {
  const uint8_t* W;          // tc layout (whole bank for experts)
  const __half* S;           // [tiles][K/g][128]
  int rows, K, g;            // rows of one matrix (one expert for the banks)
  const bf16* X;             // activations: dense rows / expert input rows / act rows
  int ldx;
  int ntok;                  // dense: number of activation rows
  int do_norm;               // dense: RMSNorm of X fused into staging
  const bf16* norm_w;
  float eps;
  const bf16* Res;           // dense: residual [ntok][ldr] or null
  int ldr;
  bf16* Y;                   // dense output [ntok][ldy]
  int ldy;
  const int32_t* n_active;   // experts: routing work list
  const int32_t* active_e;
  const int32_t* active_off;
  const int32_t* pair_token;
  size_t w_expert_stride;    // bytes of one expert's matrix
  size_t s_expert_stride;    // halves of one expert's scales
  bf16* act;                 // gate/up output [pairs][F]
  int F;
  float* out;                // down output [pairs][H]
  int H;
  int* err;                  // device error flag or null
  int ksplit;                // K split across CTAs (1 = none); the last CTA of a job reduces
  float* part;               // split partial sums [jobs][ksplit][16][128]
  int* counters;             // [jobs] arrival counters, zero between launches
};
// Split factor and workspace the launchers below use for `jobs` CTAs-worth
// of (tile, token group, expert) work with `nst` K stages each.
int tc_pick_ksplit(int jobs, int nst);
size_t tc_part_floats(int jobs, int ksplit);
bool tc_supports(int rows, int K, int g);
// Canonical [rows][K/2] (+ scales) -> tc layout; with W2/S2 the output rows
// interleave (row 2i from W, 2i+1 from W2).
cudaError_t launch_repack_tc(const uint8_t* W, const __half* S, const uint8_t* W2, const __half* S2, int rows,
                             int K, int g, uint8_t* Wtc, __half* Stc, cudaStream_t st);
cudaError_t launch_w4_tc_dense(const TcArgs& a, cudaStream_t st);
cudaError_t launch_w4_tc_gateup(const TcArgs& a, int max_u, int max_tok, cudaStream_t st);
cudaError_t launch_w4_tc_down(const TcArgs& a, int max_u, int max_tok, cudaStream_t st);
// Output projection on the tensor cores: W = bf16 [rows][K] row-major (no
// repack), X = final hidden state (RMSNorm fused, bf16), out = fp32 logits
// [ntok][rows].  rows % 128 == 0.
cudaError_t launch_lm_tc(const TcArgs& a, cudaStream_t st);
cudaError_t init_tc_attributes();

// ---------------------------------------------------------------- warp-MMA W4A16
struct MmaArgs {
  const uint8_t* W;          // mma layout (whole bank for experts)
  const uint32_t* S;         // [tiles][K/g][8] fp16 pairs
  int rows, K, g;            // rows of one matrix (one expert for the banks)
  const void* X;             // activations, fp16 (bf16 for the standalone GEMM), normalised where needed
  int ldx;
  int ntok;                  // dense: number of activation rows
  const bf16* Res;           // dense: residual [ntok][ldr] or null
  int ldr;
  bf16* Y;                   // dense output [ntok][ldy]
  int ldy;
  const int32_t* pair_token; // experts: token of each sorted pair
  const int32_t* n_jobs;     // experts: routing work list
  const int32_t* jobs;
  int max_jobs;              // grid bound of the expert launches
  size_t w_expert_stride;    // bytes of one expert's matrix
  size_t s_expert_stride;    // 32-bit words of one expert's scales
  __half* act16;             // gate/up output [pairs][F], bf16-rounded values in fp16
  int F;
  float* out;                // down output [pairs][H]
  int H;
  int* err;                  // device error flag or null
  int x_bf16;                // dense only: X holds bf16 values (converted on load) instead of fp16
  int pdl;                   // launch with programmatic dependent launch
  int ks;                    // set by the launchers
  int drop_item1;            // failure-detection tests only: 1 + the index of a staged expert work item whose
                             // copies the producer does not issue (its consumers' bounded wait runs out); 0 = none
};
// Shape support of the warp-MMA kernels: rows % 32 == 0, K % 128 == 0,
// K <= 4096, g in {32, 64, 128}.
bool mma_supports(int rows, int K, int g);
// Canonical [rows][K/2] (+ scales) -> mma layout; with W2/S2 the 16-row
// tiles hold 8 rows of W then the same 8 rows of W2 (gate/up banks).
cudaError_t launch_repack_mma(const uint8_t* W, const __half* S, const uint8_t* W2, const __half* S2, int rows,
                              int K, int g, uint8_t* Wm, uint32_t* Sm, cudaStream_t st);
cudaError_t launch_w4_mma_dense(MmaArgs a, cudaStream_t st);
cudaError_t launch_w4_mma_gateup(MmaArgs a, cudaStream_t st);
cudaError_t launch_w4_mma_down(MmaArgs a, cudaStream_t st);
// Output projection + greedy argmax: logits[b][v] = x[b] . W[v] (bf16 W
// [V][K] row-major, x already normalised, fp32 out), next[b] = argmax_v
// (ties: lowest v, NaN never wins) and len[slots[b]] += advance, in one
// launch.  keys [B] (u64) and counter [1] are zero before the launch and left
// zero after it.
struct LmArgs {
  const bf16* W;
  int V, K;
  const bf16* X;
  int B;
  float* logits;
  int32_t* next;
  int32_t* len;
  const int32_t* slots;
  int advance;
  unsigned long long* keys;
  unsigned int* counter;
  int pdl;                   // launch with programmatic dependent launch
};
cudaError_t launch_lm_mma(const LmArgs& a, cudaStream_t st);
bool lm_mma_supports(int V, int K, int B);
cudaError_t init_mma_attributes();

// ---------------------------------------------------------------- prompt-length tcgen05 GEMMs
// W4A16 GEMMs over the rows of a prompt block on the tcgen05 tensor cores,
// reading the weights in the warp-MMA layout; fp16 activations; the group
// scale is folded into fp16 weights (one rounding of q x s).  See
// prefill_tc.cu.
struct PrefillGemmArgs {
  const uint8_t* W;          // mma layout (whole bank for the experts)
  const uint32_t* S;         // mma-layout scales
  int rows, K, g;            // rows of one matrix (one expert for the banks); rows % 128 == 0
  const void* X;             // fp16 activation rows [.][ldx]
  int ldx;
  int ntok;                  // dense: rows of X
  const bf16* Res;           // dense: residual [ntok][ldr] or null
  int ldr;
  bf16* Y;                   // dense: output [ntok][ldy]
  int ldy;
  const int32_t* n_active;   // experts: the grouping of the routing kernels
  const int32_t* active_e;
  const int32_t* active_off;
  const int32_t* row_map;    // gate/up: activation row of each sorted pair
  const int32_t* n_jobs;     // experts: (active expert, 128-row tile) jobs, u | tile << 16
  const int32_t* jobs;
  int max_jobs;              // grid bound of the expert launches
  size_t w_expert_stride;    // bytes of one expert's matrix
  size_t s_expert_stride;    // 32-bit scale words of one expert's matrix
  __half* act16;             // gate/up output [pairs][F], bf16-rounded values in fp16
  int F;
  float* out;                // down output [pairs][H]
  int H;
  int* err;                  // device error flag or null
};
// The bytes of a TMA tensor map (CUtensorMap), passed to kernels by value.
struct alignas(64) TmapBytes {
  unsigned char b[128];
};
// A 2-D tensor map over fp16 rows [rows][ld] (K used of each row) with boxes
// of 64 values x 128 rows, 128-byte swizzle, zero fill outside: the B operand
// tiles of the prompt-length GEMMs.  Returns cudaSuccess or the encode error.
cudaError_t encode_rows_tmap(TmapBytes* out, const void* base, int rows, int K, int ld);
bool prefill_gemm_supports(int rows, int K, int g);
// X of the args is the matrix `tm` describes: rows of the B operand in order
// (dense: the M rows; experts: the sorted pairs' rows, gathered beforehand for
// the gate/up projection).
cudaError_t launch_prefill_dense(const PrefillGemmArgs& a, const TmapBytes& tm, cudaStream_t st);
// max_rows_per_expert bounds the grid (an expert has at most one row per token)
cudaError_t launch_prefill_gateup(const PrefillGemmArgs& a, const TmapBytes& tm, int max_rows_per_expert,
                                  cudaStream_t st);
cudaError_t launch_prefill_down(const PrefillGemmArgs& a, const TmapBytes& tm, int max_rows_per_expert,
                                cudaStream_t st);
// dst[r] = src[map[r]] for r < n, rows of `cols` fp16 values (cols % 8 == 0)
cudaError_t launch_gather_rows(const __half* src, const int32_t* map, int n, int cols, __half* dst, cudaStream_t st);
cudaError_t init_prefill_attributes();
// p[0..n) = value
cudaError_t launch_fill_i32(int32_t* p, int32_t value, int n, cudaStream_t st);

// ---------------------------------------------------------------- attention
struct AttnArena {
  bf16* K;        // [layers][S][kvh][cap][d]
  bf16* V;
  int32_t* len;   // [S] committed lengths (device)
  int layers, S, kvh, cap, d;
  __host__ __device__ size_t slot_stride() const { return (size_t)kvh * cap * d; }
  __host__ __device__ size_t layer_stride() const { return (size_t)S * slot_stride(); }
};
constexpr int kAttnChunk = 128;
size_t attn_partial_floats(int B, int qh, int cap, int d);

// RoPE on q and k at pos = len[slot], q -> qout [B][qh][d], k,v -> arena.
cudaError_t launch_rope_append(const AttnArena& ar, int layer, const int32_t* slots, const bf16* qkv,
                               int ld_qkv, int qh, const float2* rope, bf16* qout, int B,
                               DevCheck chk, cudaStream_t st, bool pdl = false);
// Plain append of already-rotated k, v ([B][kvh][d]) at pos = len[slot].
cudaError_t launch_kv_append(const AttnArena& ar, int layer, const int32_t* slots, const bf16* k,
                             const bf16* v, int B, DevCheck chk, cudaStream_t st);
// Split-K attention over positions 0..len[slot] (inclusive) and the combine.
// out is bf16, or fp16 holding the same bf16-rounded values when out_f16.
cudaError_t launch_attention(const AttnArena& ar, int layer, const int32_t* slots, const bf16* q,
                             void* out, int qh, int B, float* partials, DevCheck chk,
                             cudaStream_t st, int* launches, const Marker& mark = Marker(), int out_f16 = 0,
                             bool pdl = false);
cudaError_t launch_set_len(int32_t* len, int slot, int value, cudaStream_t st);

// RoPE + append + attention + merge in one launch (warp-MMA family).  q, k
// and v come straight from the QKV projection's rows; out is fp16 holding
// bf16-rounded values [B][qh][d]; counters [attn_counter_count(B, kvh)] are
// zero before the launch and left zero.  Needs d in {64, 128}, qh / kvh <= 8
// and at most kMaxMergeChunks chunks per stream.  A stream of more than
// kAttnMergeBlock chunks merges in two levels (blocks of kAttnMergeBlock).
constexpr int kMaxMergeChunks = 64;
constexpr int kAttnMergeBlock = 8;
constexpr int kAttnMergeBlocks = kMaxMergeChunks / kAttnMergeBlock;
// Arrival counters of a fused attention launch of B rows: one per (row, kv
// head), then one per (row, kv head, merge block), then the launch's work
// queue (items claimed, CTAs done) when it has more items than CTAs.
__host__ __device__ constexpr size_t attn_queue_index(int B, int kvh) { return (size_t)B * kvh * (1 + kAttnMergeBlocks); }
__host__ __device__ constexpr size_t attn_counter_count(int B, int kvh) { return attn_queue_index(B, kvh) + 2; }
struct AttnFusedArgs {
  AttnArena ar;
  int layer;
  const int32_t* slots;
  const bf16* qkv;
  int ld_qkv, qh;
  const float2* rope;   // [cap][d/2] (cos, sin)
  __half* out;
  float* part;          // chunk records, as attn_partial_floats
  int max_chunks;
  unsigned int* counters;
  int B;
  DevCheck chk;
  int prefill;          // rows of one slot at positions len + row0 + b; k/v appended beforehand
  int row0;             // prefill: position offset of this launch's first row
};
bool attention_fused_supports(const AttnArena& ar, int qh);
// Causal attention of a prompt block (attention_prefill.cu): a.B rows of the
// slot a.slots[0] at positions len + b, their k and v already in the slot;
// out as the fused kernel's.  One launch for the block.
bool attention_prefill_supports(const AttnArena& ar, int qh);
cudaError_t launch_attention_prefill(const AttnFusedArgs& a, cudaStream_t st);
cudaError_t launch_attention_fused(const AttnFusedArgs& a, cudaStream_t st, bool pdl = false);
// Rotated k and v of each row b to the arena at the row's position (len of
// its slot, plus b when a.prefill): the prompt path's append.
cudaError_t launch_append_rows(const AttnFusedArgs& a, cudaStream_t st, bool pdl = false);

// ---------------------------------------------------------------- model glue
cudaError_t launch_embed(const bf16* table, int V, int H, const int32_t* tokens, bf16* x, int B,
                         DevCheck chk, cudaStream_t st);
// The embedding rows and their RMSNorm: xn[b] = bf16(x[b] * rinv * nw),
// stored as fp16.
cudaError_t launch_embed_norm(const bf16* table, int V, int H, const int32_t* tokens, bf16* x, const bf16* nw,
                              float eps, __half* xn, int B, DevCheck chk, cudaStream_t st, bool pdl = false);
// logits[b][v] = RMSNorm(x[b]) . W[v] (bf16 weights, fp32 out).
cudaError_t launch_lm_head(const bf16* W, int V, int H, const bf16* x, const bf16* norm_w, float eps,
                           float* logits, int B, cudaStream_t st);
// next[b] = argmax_v logits[b][v] (ties: lowest v); len[slots[b]] += advance.
cudaError_t launch_argmax(const float* logits, int V, int B, int32_t* next, int32_t* len,
                          const int32_t* slots, int advance, cudaStream_t st);
// len[slots[b]] += by for b < B (slots distinct).
cudaError_t launch_advance(int32_t* len, const int32_t* slots, int B, cudaStream_t st, int by = 1);
cudaError_t launch_quantize(const float* W, int N, int K, int g, uint8_t* packed, __half* scales,
                            cudaStream_t st);

// Kernel attributes (large dynamic shared memory); call once before capture.
cudaError_t init_kernel_attributes();

}  // namespace bm
