/*
 * bitmoe.h — C ABI of the batched W4A16 mixture-of-experts decode step on one
 * GB300 (sm_103a).
 *
 * Pages cited by abbreviated title:
 *   [KV-slot isolation]  "Per-stream KV-slot isolation for parallel low-bit
 *                         decode on Apple Silicon: crash fix with
 *                         byte-identical solo parity and no-regression"
 *   [Crash root cause]   "A falsify-first root cause for a concurrent 4-bit
 *                         decode crash: batch-composition KV-pool wipe trips a
 *                         re-seed precondition"
 *   [Batched serving]    "Batched-concurrent 4-bit serving on Apple Silicon:
 *                         weight-stream amortization with an honest sublinear
 *                         ceiling"
 *
 * Conventions for every call:
 *  - Plain pointers and sizes only.  bf16 and fp16 tensors are passed as
 *    uint16_t bit patterns.  "device" pointers must be CUDA device memory of
 *    the current device; "host" pointers are ordinary host memory.
 *  - Streams are cudaStream_t values passed as void* (NULL = legacy stream).
 *    Every call that takes a stream only enqueues work on it and returns;
 *    outputs are valid once that stream has been synchronised.
 *  - No call throws, traps or aborts.  Errors come back as bm_status; the
 *    calling thread's last error message is available from bm_last_error().
 *    An asynchronous CUDA error surfaces as BM_ERR_CUDA from a later call or
 *    from bm_engine_sync().
 *  - Packed int4 weight layout ("canonical"): row-major [N][K/2] bytes along
 *    K, element 2j in the low nibble of byte j and element 2j+1 in the high
 *    nibble; code u in [0,15] stands for q = u - 8; scales fp16 [N][K/g];
 *    weight = q * scale.  ([Batched serving] §1, §3: packed int4 with
 *    per-group scales; the nibble order and offset are this library's
 *    stated reading, the pages print none.)
 *  - Activations are bf16; every accumulation is fp32; each op rounds its
 *    output to bf16 once.
 */
#ifndef BITMOE_H
#define BITMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum bm_status {
  BM_OK = 0,
  BM_ERR_INVALID_ARG = 1,   /* a size, pointer or layout the call rejects      */
  BM_ERR_CTX_CAP = 2,       /* admission: the stream would exceed the context cap */
  BM_ERR_NO_SLOT = 3,       /* admission: every slot is in use                 */
  BM_ERR_SLOT_FREE = 4,     /* a slot that is not active was used or released  */
  BM_ERR_CUDA = 5,          /* a CUDA runtime call failed                       */
  BM_ERR_OOM = 6,           /* device or pinned host allocation failed         */
  BM_ERR_NOT_READY = 7,     /* decode_step before every layer's weights were set */
  BM_ERR_DEVICE_CHECK = 8,  /* a kernel skipped an out-of-range index, or a bounded
                               pipeline wait inside a kernel gave up              */
  BM_ERR_UNSUPPORTED = 9    /* a shape or option this build does not handle    */
} bm_status;

/* Kernel family of the dense and expert projections.  Chosen once per engine,
 * never per step, so that a stream's bytes never depend on the batch it runs
 * in ([KV-slot isolation] follow-up update: one reduction order for solo and
 * batched).  SIMT = CUDA-core W4A16 GEMV; TC = tcgen05 tensor cores
 * (tensor memory accumulators); MMA = warp-level tensor-core instruction
 * (mma.sync m16n8k16, bf16) with every RMSNorm computed by the kernel that
 * writes its input row and the greedy argmax fused into the output
 * projection.  AUTO picks MMA when the shapes allow it (measured fastest at
 * every decode batch size), else TC, else SIMT. */
typedef enum bm_kernel_policy {
  BM_POLICY_AUTO = 0,
  BM_POLICY_SIMT = 1,
  BM_POLICY_TC = 2,
  BM_POLICY_MMA = 3
} bm_kernel_policy;

/* Model geometry and engine limits. */
typedef struct bm_config {
  int hidden;        /* H                                                     */
  int q_heads;       /* query heads                                           */
  int kv_heads;      /* key/value heads; q_heads % kv_heads == 0              */
  int head_dim;      /* d; 64 or 128                                          */
  int experts;       /* E (<= 256)                                            */
  int top_k;         /* k (<= 16, <= E)                                       */
  int ffn;           /* expert FFN width F                                    */
  int group;         /* int4 group size g along K: 32, 64 or 128             */
  int vocab;         /* V                                                     */
  int layers;        /* decoder layers                                        */
  float rope_base;   /* RoPE base (rotate-half pairing)                       */
  float rms_eps;     /* RMSNorm epsilon                                       */
  int max_streams;   /* slots in the KV arena (<= 64; <= 128 on the MMA family) */
  int ctx_cap;       /* positions per slot                                    */
  int renorm_topk;   /* 1: top-k weights renormalised to sum to one           */
  int kernel_policy; /* bm_kernel_policy                                      */
  int use_graph;     /* 1: decode_step replays one captured CUDA graph per B  */
  int prefill_tc;    /* kv_slot_prefill: 0 = through the decode kernels in blocks
                        of max_streams rows (the bytes of as many decode steps);
                        1 = prompt-length GEMMs on the tcgen05 tensor cores in
                        blocks of up to 512 rows (needs the warp-MMA family)   */
  int persistent_step; /* 1: decode steps of B <= min(8, max_streams, 64 / top_k)
                        rows run every layer in one persistent cooperative
                        kernel (one CTA per SM, grid barriers between the
                        phases), the solo / small-batch path of [KV-slot
                        isolation] (follow-up update).  It computes every
                        value with the multi-kernel step's arithmetic, so the
                        bytes are the same whichever path ran a step.  Needs
                        the warp-MMA family; larger steps use the
                        multi-kernel step.                                     */
} bm_config;

/* One decoder layer's weights, canonical layout, DEVICE pointers.  Borrowed
 * only for the duration of bm_engine_set_layer, which copies them. */
typedef struct bm_layer_weights {
  const uint8_t* wqkv;   const uint16_t* wqkv_s;  /* [(qh+2kvh)d][H/2], [..][H/g]: q rows, then k, then v, head-major */
  const uint8_t* wo;     const uint16_t* wo_s;    /* [H][qh*d/2], [H][qh*d/g]        */
  const float* wr;                                /* router, fp32 [E][H]            */
  const uint8_t* wg;     const uint16_t* wg_s;    /* [E][F][H/2], [E][F][H/g]       */
  const uint8_t* wu;     const uint16_t* wu_s;    /* [E][F][H/2], [E][F][H/g]       */
  const uint8_t* wd;     const uint16_t* wd_s;    /* [E][H][F/2], [E][H][F/g]       */
  const uint16_t* attn_norm;                      /* bf16 [H] or NULL (all ones)    */
  const uint16_t* ffn_norm;                       /* bf16 [H] or NULL (all ones)    */
} bm_layer_weights;

/* Expert bank of one layer for the standalone grouped op, DEVICE pointers,
 * canonical layout as in bm_layer_weights. */
typedef struct bm_moe_weights {
  int experts, top_k, hidden, ffn, group, renorm_topk;
  const float* wr;
  const uint8_t* wg; const uint16_t* wg_s;
  const uint8_t* wu; const uint16_t* wu_s;
  const uint8_t* wd; const uint16_t* wd_s;
} bm_moe_weights;

typedef struct bm_engine bm_engine;
typedef struct bm_slot_map bm_slot_map;

typedef struct bm_stats {
  uint64_t steps;             /* decode_step calls that succeeded            */
  uint64_t tokens;            /* sum of B over those calls                   */
  uint64_t graph_launches;    /* cudaGraphLaunch calls made by decode_step   */
  uint64_t graph_captures;    /* graphs captured (one per distinct B)        */
  uint64_t kernel_launches;   /* kernels enqueued outside graphs + per graph replay */
  uint64_t kernels_per_step;  /* kernels in one decode step (graph nodes)    */
  size_t weight_bytes;        /* device bytes holding the model weights      */
  size_t arena_bytes;         /* device bytes of the KV arena                */
  size_t scratch_bytes;       /* device bytes of activations and partials    */
} bm_stats;

/* Per-kernel-class measurement of one profiled decode step. */
typedef struct bm_kernel_profile {
  char name[24];    /* kernel class, e.g. "expert_gateup"                      */
  int launches;     /* launches of this class in the step                      */
  float ms;         /* summed CUDA-event time of those launches                */
  double bytes;     /* algorithmic HBM bytes of those launches (weights read once,
                       activations, K/V positions actually attended)          */
  double flops;     /* algorithmic flops (2 per multiply-add)                  */
} bm_kernel_profile;

/* ---------------------------------------------------------------- errors */

/* Message of the last failed call on this thread ("" if none).  The pointer
 * stays valid until the next call on this thread. */
const char* bm_last_error(void);

/* ---------------------------------------------------------------- engine */

/* Create an engine on the current CUDA device.  Allocates the weight slab,
 * the fixed KV arena (layers x max_streams x ctx_cap x kv_heads x head_dim x
 * 2 tensors, bf16) and scratch, and writes the standing byte counts to
 * stderr once ([KV-slot isolation] §5: the fixed arena's standing cost is
 * reported at boot).  Errors: BM_ERR_INVALID_ARG (geometry out of range),
 * BM_ERR_UNSUPPORTED, BM_ERR_OOM, BM_ERR_CUDA. */
bm_status bm_engine_create(const bm_config* cfg, bm_engine** out);

/* Free everything the engine owns.  NULL is ignored.  The caller must not
 * have work for this engine in flight. */
void bm_engine_destroy(bm_engine* e);

/* Copy one layer's weights (DEVICE pointers, canonical layout) into the
 * engine, on `stream`.  The source buffers may be freed once the stream has
 * been synchronised.  Errors: BM_ERR_INVALID_ARG (layer out of range or a
 * NULL weight), BM_ERR_CUDA. */
bm_status bm_engine_set_layer(bm_engine* e, int layer, const bm_layer_weights* w, void* stream);

/* Copy the bf16 embedding [V][H], lm_head [V][H] and final norm [H] (NULL =
 * ones), DEVICE pointers.  ([Batched serving] §1: the per-stream output
 * projection is part of the fused step.) */
bm_status bm_engine_set_embeddings(bm_engine* e, const uint16_t* embed, const uint16_t* lm_head,
                                   const uint16_t* final_norm, void* stream);

/* Synchronise `stream` and report device-side checks since the last call
 * (BM_ERR_DEVICE_CHECK; the flag is then cleared).  The message names the
 * code: 1 an out-of-range slot id, 2 an out-of-range position, 3 an
 * out-of-range token id (each skipped by the kernel that met it), 4 a
 * tensor-core projection's pipeline wait that timed out, 5 an expert
 * projection's pipeline wait that timed out (that CTA stopped after waiting
 * for the copies it had issued), 6 a wait of the persistent decode step
 * (persistent_step) that timed out (every CTA left the step at its next grid
 * barrier; the step's outputs are not valid).  No check traps: the context
 * stays usable. */
bm_status bm_engine_sync(bm_engine* e, void* stream);

/* Counters and standing memory. */
bm_status bm_engine_stats(const bm_engine* e, bm_stats* out);

/* The kernel family this engine resolved its policy to (SIMT, TC or MMA). */
int bm_engine_kernel_family(const bm_engine* e);

/* ---------------------------------------------------------------- slots
 * [KV-slot isolation] §1: the batched KV arena is indexed by a stable
 * per-stream slot; a slot is seeded once at join, released at retire (a
 * logical reset, the buffer is reused without a wipe), and a change of batch
 * composition never touches a continuing stream's K/V.  [Crash root cause]
 * §3 is the failure this rules out: pools wiped on a batch-size change and
 * a re-seed that only the host prefix could feed. */

/* Join: take the lowest free slot, copy `len` positions of K and V into it
 * and set its length to `len`.  K, V: bf16 [layers][kv_heads][len][head_dim],
 * host or device memory (NULL allowed when len == 0).  Errors:
 * BM_ERR_CTX_CAP if len >= ctx_cap (no room for one decode token: rejected,
 * never truncated — [KV-slot isolation] §5), BM_ERR_NO_SLOT if every slot
 * is active, BM_ERR_INVALID_ARG for len < 0. */
bm_status kv_slot_seed(bm_engine* e, const uint16_t* K, const uint16_t* V, int len,
                       int* slot_out, void* stream);

/* Write this step's K/V of one layer for B streams at position = each slot's
 * length.  slots: HOST int32 [B]; Knew, Vnew: DEVICE bf16 [B][kv_heads][d]
 * (K already rotated).  The length does not advance (kv_slot_advance does).
 * Errors: BM_ERR_SLOT_FREE, BM_ERR_CTX_CAP (length == ctx_cap),
 * BM_ERR_INVALID_ARG (duplicate slot, layer or B out of range). */
bm_status kv_slot_append(bm_engine* e, int layer, const int32_t* slots, const uint16_t* Knew,
                         const uint16_t* Vnew, int B, void* stream);

/* Decode attention of one layer for B streams: query head h of stream i
 * attends over positions 0..len of slot slots[i] (its committed prefix plus
 * the position this step appended), with KV head h / (q_heads/kv_heads).
 * Reads nothing outside those slots.  slots: HOST int32 [B]; Q: DEVICE bf16
 * [B][q_heads][d] (rotated); O: DEVICE bf16 [B][q_heads][d].  Split-K over
 * fixed 128-position chunks with a fixed-order combine, so a stream's output
 * depends only on its own slot.  Errors as kv_slot_append. */
bm_status kv_slot_attend(bm_engine* e, int layer, const int32_t* slots, const uint16_t* Q,
                         uint16_t* O, int B, void* stream);

/* Commit one appended position for B streams (length += 1).  decode_step
 * does this itself once per step, after all layers. */
bm_status kv_slot_advance(bm_engine* e, const int32_t* slots, int B, void* stream);

/* Retire: mark the slot free and its length 0.  Host only; the slot's K/V
 * bytes are left as they are and overwritten by the next stream.  Errors:
 * BM_ERR_SLOT_FREE on a slot that is not active (double release). */
bm_status kv_slot_release(bm_engine* e, int slot);

/* Committed length of an active slot (host mirror). */
bm_status kv_slot_length(const bm_engine* e, int slot, int* len_out);

/* Copy `count` positions (from 0) of one layer of a slot to DEVICE or HOST
 * buffers K_out, V_out bf16 [kv_heads][count][d].  For tests and checkpoints. */
bm_status kv_slot_read(bm_engine* e, int layer, int slot, int count, uint16_t* K_out,
                       uint16_t* V_out, void* stream);

/* ---------------------------------------------------------------- ops */

/* Batched W4A16 GEMM: Y[m][n] = sum_k X[m][k] * W[n][k] (+ R[m][n]).
 * W: DEVICE packed int4 [N][K/2], S: fp16 [N][K/g]; X: bf16 [M][K];
 * R: bf16 [M][N] or NULL; Y: bf16 [M][N].  All DEVICE, row-major, dense.
 * Each packed weight byte is read from HBM once for all M rows ([Batched
 * serving] §1); a row's result does not depend on M or on the other rows
 * ([Batched serving] §3).  Uses the CUDA-core kernel family.
 * Errors: BM_ERR_INVALID_ARG if M < 1, N < 1, K % 32 != 0, K % g != 0,
 * g not in {32, 64, 128}, or a NULL pointer. */
bm_status w4_gemm_batched(const uint8_t* W, const uint16_t* S, const uint16_t* X, uint16_t* Y,
                          const uint16_t* R, int M, int N, int K, int g, void* stream);

/* Repack canonical int4 weights W [N][K/2] and scales S [N][K/g] (DEVICE)
 * into the tensor-core layout consumed by w4_gemm_batched_tc: Wtc (N*K/2
 * bytes) and Stc (N*K/g fp16), both DEVICE, caller-owned.  The layout: for
 * each tile of 128 rows and each 64-wide K stage, two 32-wide halves of 128
 * rows x 16 bytes; inside each 32-bit word the codes are ordered
 * (k0 k2 k4 k6 k1 k3 k5 k7); scales [N/128][K/g][128].  Errors:
 * BM_ERR_INVALID_ARG unless N % 128 == 0, K % 64 == 0, K <= 4096, g in
 * {32, 64, 128}, K % g == 0. */
bm_status bm_w4_repack_tc(const uint8_t* W, const uint16_t* S, int N, int K, int g, uint8_t* Wtc,
                          uint16_t* Stc, void* stream);

/* The batched W4A16 GEMM of w4_gemm_batched on the tensor cores (tcgen05,
 * fp16 operands, fp32 accumulation in tensor memory), with weights in the
 * layout of bm_w4_repack_tc.  Each int4 code enters the MMA as the exact
 * fp16 integer q - 8 and each activation as fp16(x); the per-stage fp32 sums
 * are multiplied by the fp32 group scale.  Weight bytes are read from HBM
 * once per group of 16 rows of X.  Shapes as bm_w4_repack_tc, M >= 1. */
bm_status w4_gemm_batched_tc(const uint8_t* Wtc, const uint16_t* Stc, const uint16_t* X, uint16_t* Y,
                             const uint16_t* R, int M, int N, int K, int g, void* stream);

/* Repack canonical int4 weights W [N][K/2] and scales S [N][K/g] (DEVICE)
 * into the layout consumed by w4_gemm_batched_mma: Wm (N*K/2 bytes) and Sm
 * (N*K/(2g) 32-bit words), both DEVICE, caller-owned.  Layout: for each tile
 * of 16 rows and each 64-wide K chunk, 32 lane slots of 16 bytes; slot
 * (g = lane / 4, t = lane % 4) holds, for MMA step s = 0..3 of the chunk, the
 * codes of rows 16T+g and 16T+g+8 at k = 64c + 32(s/2) + 8t + 4(s%2) + 0..3
 * (nibbles: r0 k0, r1 k0, r0 k2, r1 k2, r0 k1, r1 k1, r0 k3, r1 k3); scales
 * [N/16][K/g][8] words, word p = the fp16 scales of rows 16T+p and 16T+p+8.
 * Errors: BM_ERR_INVALID_ARG unless N % 32 == 0, K % 128 == 0, K <= 4096,
 * g in {32, 64, 128}, K % g == 0. */
bm_status bm_w4_repack_mma(const uint8_t* W, const uint16_t* S, int N, int K, int g, uint8_t* Wm,
                           uint32_t* Sm, void* stream);

/* The batched W4A16 GEMM of w4_gemm_batched on the warp-level tensor-core
 * instruction (mma.sync m16n8k16, bf16 operands, fp32 accumulation), weights
 * in the layout of bm_w4_repack_mma.  Each int4 code enters the MMA as the
 * exact bf16 integer q - 8 and each activation as itself; the fp32 sum of a
 * scale group is multiplied by the group's fp32 scale.  A weight byte is
 * read from HBM once per group of 32 rows of X.  The summation order of an
 * output depends only on (N, K, g), so a row's result does not depend on M
 * or on the other rows.  Shapes as bm_w4_repack_mma, M >= 1. */
bm_status w4_gemm_batched_mma(const uint8_t* Wm, const uint32_t* Sm, const uint16_t* X, uint16_t* Y,
                              const uint16_t* R, int M, int N, int K, int g, void* stream);

/* The batched W4A16 GEMM at prompt length on the tcgen05 tensor cores (the
 * kernel kv_slot_prefill runs with prefill_tc): Y[m][n] = sum_k X[m][k] *
 * W[n][k] (+ R[m][n]) for M rows at once, weights in the layout of
 * bm_w4_repack_mma.  Work items of 128 weight rows and up to 128 rows of X
 * over the whole K, looped over by one CTA per SM; each weight enters the MMA
 * as the fp16 product q * s (one
 * rounding; the decode kernels instead scale exact fp32 group sums), X as
 * fp16, and the sums are fp32 in tensor memory.  A row's result does not
 * depend on M or on the other rows.  ([Batched serving] §1: a dense
 * projection is one batched GEMM over all rows.)
 * Wm, Sm: DEVICE (bm_w4_repack_mma); X16: DEVICE fp16 [M][K]; R: DEVICE bf16
 * [M][N] or NULL; Y: DEVICE bf16 [M][N].  Errors: BM_ERR_INVALID_ARG unless
 * M >= 1, N % 128 == 0, K % 256 == 0, K <= 4096, g in {32, 64, 128},
 * K % g == 0, or on a NULL pointer. */
bm_status w4_gemm_prompt_tc(const uint8_t* Wm, const uint32_t* Sm, const uint16_t* X16, uint16_t* Y,
                            const uint16_t* R, int M, int N, int K, int g, void* stream);

/* Bytes of DEVICE workspace moe_grouped_w4 needs for B tokens. */
size_t bm_moe_workspace_bytes(int B, int experts, int top_k, int hidden, int ffn);

/* Grouped int4 expert op of B tokens: softmax top-k routing of X, every
 * selected (token, expert) pair sorted by expert, each active expert's
 * gate/up (SiLU) and down projections over its tokens, then
 * Y[b] = Hres[b] + sum_r w[b][r] * out[b][r] in rank order.
 * ([Batched serving] §1: the selected experts of all B streams run as one
 * grouped operation against the resident expert bank.)
 * X: DEVICE bf16 [B][H] (the router and experts' input); Hres: DEVICE bf16
 * [B][H] or NULL (zero); Y: DEVICE bf16 [B][H]; topk_ids: DEVICE int32
 * [B][k] (out, rank order); topk_w: DEVICE fp32 [B][k] (out); ws: DEVICE,
 * at least bm_moe_workspace_bytes(B, ...) bytes, caller-owned.
 * Errors: BM_ERR_INVALID_ARG (bad sizes, NULL, ws too small). */
bm_status moe_grouped_w4(const bm_moe_weights* w, const uint16_t* X, const uint16_t* Hres,
                         uint16_t* Y, int32_t* topk_ids, float* topk_w, int B, void* ws,
                         size_t ws_bytes, void* stream);

/* The grouped expert op for callers that cannot allocate device memory: a
 * plugin inside a host engine that owns the whole device memory pool (an
 * extra cudaMalloc would fail or break the pool's accounting), or code on a
 * latency-critical path where cudaMalloc / cudaFree, which can synchronise
 * the device, are not allowed.  No counterpart on the pages: it exists for
 * those callers only.
 * Same arguments, computation and results as moe_grouped_w4, minus the
 * workspace: the scratch lives in a fixed array of bm_moe_noalloc_max_bytes()
 * (4 MiB) compiled into the library, which every device that loads the
 * library keeps for the life of the process.  The call allocates nothing.
 * Its first call on a device looks up that array's device address and sets
 * kernel attributes for that device; make that first call before any stream
 * capture.  All calls on a device share the one array (no call needs it
 * cleared first): calls whose work overlaps on the GPU — concurrent streams,
 * or host threads without ordering — race on it and must be serialised by the
 * caller.  Errors: as moe_grouped_w4, plus BM_ERR_INVALID_ARG when the sizes
 * need more workspace than the array holds (bm_moe_workspace_bytes(B, ...) >
 * bm_moe_noalloc_max_bytes()), and BM_ERR_CUDA if the array's address cannot
 * be obtained. */
bm_status moe_grouped_w4_noalloc(const bm_moe_weights* w, const uint16_t* X, const uint16_t* Hres,
                                 uint16_t* Y, int32_t* topk_ids, float* topk_w, int B, void* stream);

/* Size of the built-in workspace of moe_grouped_w4_noalloc, in bytes. */
size_t bm_moe_noalloc_max_bytes(void);

/* One batched decode step of B streams through every layer and the output
 * projection ([Batched serving] §1: one fused forward per token for all B
 * streams; the host crosses to the device once per step).
 * slots: HOST int32 [B], distinct active slots, in any order; tokens: int32
 * [B] in HOST or DEVICE memory, token i sits at position length(slots[i]);
 * next_tokens: int32 [B], HOST or DEVICE, greedy argmax (ties: lowest id);
 * logits: DEVICE fp32 [B][V] or NULL.  Row i of every output belongs to
 * slots[i].  Appends each layer's K/V at that position and advances every
 * slot's length by one.  With use_graph, the step is one cudaGraphLaunch of
 * a graph captured on the first step with this B.
 * Errors: BM_ERR_NOT_READY, BM_ERR_SLOT_FREE, BM_ERR_CTX_CAP,
 * BM_ERR_INVALID_ARG (B out of range, duplicate slot), BM_ERR_CUDA. */
bm_status decode_step(bm_engine* e, int B, const int32_t* slots, const int32_t* tokens,
                      int32_t* next_tokens, float* logits, void* stream);

/* Prompt ingestion into an active slot ([KV-slot isolation] §1: a stream's
 * K/V is written once when it joins, then grows one position per decode
 * step): the n_tokens prompt tokens go to positions len .. len + n_tokens - 1
 * of `slot`, each layer's rotated k and v are written there, and the slot's
 * length advances by n_tokens; row j attends causally to positions
 * 0..len + j.  With bm_config.prefill_tc = 0 the prompt runs in blocks of up
 * to max_streams rows through the decode kernels (one CUDA graph per block
 * shape with use_graph), and every row is computed exactly as a decode step
 * at its position, so the arena bytes, logits and next token equal those of
 * n_tokens single-stream decode_step calls fed the same tokens.  With
 * prefill_tc = 1 it runs in blocks of up to 512 rows as prompt-length
 * kernels (the tcgen05 GEMMs of w4_gemm_prompt_tc for the projections and
 * the grouped experts, a causal block attention, the rows' routing with the
 * decode router's per-logit arithmetic); the results are within the
 * tolerance of decoding the prompt, deterministic, and independent of how a
 * prompt is split over calls.
 * tokens: int32 [n_tokens], HOST or DEVICE; next_token: int32 [1], HOST or
 * DEVICE, the greedy argmax after the last prompt token; logits: DEVICE fp32
 * [V] of that position, or NULL.
 * Errors: BM_ERR_INVALID_ARG (NULL, n_tokens < 1, slot out of range),
 * BM_ERR_SLOT_FREE, BM_ERR_CTX_CAP (len + n_tokens > ctx_cap; nothing is
 * written), BM_ERR_NOT_READY, BM_ERR_UNSUPPORTED (an engine not on the
 * warp-MMA kernel family), BM_ERR_CUDA.  The argument errors leave the slot
 * untouched; after BM_ERR_CUDA the slot's contents and length are undefined
 * and the caller releases it. */
bm_status kv_slot_prefill(bm_engine* e, int slot, int n_tokens, const int32_t* tokens,
                          int32_t* next_token, float* logits, void* stream);

/* decode_step run without the graph, with a CUDA event recorded after every
 * kernel launch on `stream`, then synchronised.  Same arguments and the same
 * effect on slots and outputs as decode_step (logits are not returned).  Fills
 * out[0..*n_out) with one entry per kernel class (at most max_out).  Event
 * times include the launch gaps between kernels of an eager launch sequence.
 * Errors as decode_step. */
bm_status bm_engine_profile_step(bm_engine* e, int B, const int32_t* slots, const int32_t* tokens,
                                 int32_t* next_tokens, bm_kernel_profile* out, int max_out, int* n_out,
                                 void* stream);

/* ---------------------------------------------------------------- layer ops of the step
 * The decode step's own kernels on one layer, with the engine's weights (in
 * the layout the step reads) and its scratch, launched exactly as decode_step
 * launches them (same grids, same per-output summation order), so that each
 * block can be checked on its own at any batch size.  The engine must be on
 * the warp-MMA kernel family (BM_ERR_UNSUPPORTED otherwise).  Like every call
 * on an engine they are serialised by the engine and must not overlap with
 * other work on it in flight. */

/* The mixture-of-experts half of decoder layer `layer` for B rows
 * ([Batched serving] §1: the experts selected by all B streams run as one
 * grouped operation against the resident int4 bank): hn = RMSNorm(h) with
 * the layer's ffn norm, fp32 router logits, softmax top-k (ties: lower
 * expert id) with renormalised weights, the (row, rank) pairs grouped by
 * expert, each active expert's gate/up (SiLU) and down projections over its
 * rows, and y = h + sum_r w[r] * out[r] in rank order.  Four launches:
 * routing (router, top-k and grouping in one kernel), gate/up, down, combine.
 * h: DEVICE bf16 [B][H]; y: DEVICE bf16 [B][H] (may not alias h);
 * topk_ids: int32 [B][k] and topk_w: fp32 [B][k], HOST or DEVICE, or NULL.
 * Errors: BM_ERR_INVALID_ARG (NULL h or y, layer or B out of range),
 * BM_ERR_NOT_READY, BM_ERR_UNSUPPORTED, BM_ERR_CUDA.  A pipeline wait that
 * gives up inside the expert kernels is reported by bm_engine_sync
 * (BM_ERR_DEVICE_CHECK, code 5). */
bm_status bm_engine_moe(bm_engine* e, int layer, const uint16_t* h, uint16_t* y, int32_t* topk_ids, float* topk_w,
                        int B, void* stream);

/* The attention block of decoder layer `layer` for B streams in one launch
 * ([KV-slot isolation] §1: each stream's K/V lives in its own slot of the
 * fixed arena): rotate-half RoPE of the q heads and of the new k at position
 * p = length(slots[i]), k and v written to the slot at p, then grouped-query
 * attention of each q head over positions 0..p of that slot (split into
 * 128-position chunks and merged in ascending order), output rounded to bf16.
 * The length does not advance (kv_slot_advance commits the position).
 * slots: HOST int32 [B], distinct active slots; qkv: DEVICE bf16 [B][(q_heads
 * + 2 kv_heads) * head_dim], rows of the QKV projection (q heads, then k,
 * then v, head-major, not rotated); out: DEVICE [B][q_heads][head_dim] fp16
 * bit patterns, each holding a bf16-rounded value (the form the output
 * projection of the step consumes).  Errors as kv_slot_append, plus
 * BM_ERR_UNSUPPORTED. */
bm_status bm_engine_attention(bm_engine* e, int layer, const int32_t* slots, const uint16_t* qkv, uint16_t* out,
                              int B, void* stream);

/* Copy the residual-stream rows left by the last decode_step (the last
 * layer's output, before the final norm), bf16 [B][H], to `out` (HOST or
 * DEVICE).  B <= max_streams.  For tests that check a deep step layer by
 * layer. */
bm_status bm_engine_read_hidden(bm_engine* e, int B, uint16_t* out, void* stream);

/* Failure-detection tests only: make the next bm_engine_moe calls skip the
 * copies of staged expert work item `item` of the gate/up kernel (-1 = none,
 * the default), so that its consumers' bounded wait runs out, the affected
 * CTA stops, and bm_engine_sync reports BM_ERR_DEVICE_CHECK with code 5.
 * Nothing faults: every copy that was issued is waited for before the CTA
 * exits.  decode_step ignores this setting. */
bm_status bm_engine_test_drop_expert_item(bm_engine* e, int item);

/* Switch the persistent small-batch step of an engine created with
 * persistent_step on (enable = 1) or off (0: every decode step runs the
 * multi-kernel step): the solo / batched toggle of [KV-slot isolation]
 * (follow-up update), for measuring both paths on one engine.  Both paths
 * leave the same bytes.  Captured decode graphs are dropped.  Errors:
 * BM_ERR_INVALID_ARG, BM_ERR_UNSUPPORTED (created without persistent_step). */
bm_status bm_engine_set_persistent_step(bm_engine* e, int enable);

/* Failure-detection tests only: make the persistent decode step (engines
 * created with persistent_step) skip the copy of weight item `unit` of its
 * CTAs' producers (the unit-th 16-row tile each producer would stream in a
 * step; -1 = none, the default).  The consumer's bounded wait runs out
 * after about a second, every CTA leaves the step at its next grid barrier,
 * and bm_engine_sync reports BM_ERR_DEVICE_CHECK with code 6.  Nothing
 * faults: every copy that was issued lands before its CTA exits.  Captured
 * decode graphs are dropped so that the next steps use the setting. */
bm_status bm_engine_test_drop_persist_unit(bm_engine* e, int unit);

/* Measurement only: time the tcgen05 MMA on the current GPU.  One CTA issues
 * `iters` stages of four kind::f16 MMAs of M 128 x N n x K 16 (zero operands)
 * into one tensor-memory accumulator, A from tensor memory (a_in_tmem = 1) or
 * shared memory, the shared-memory operands in the no-swizzle core-matrix
 * layout (swizzle128 = 0) or the 128-byte-swizzled K-major layout (1); with
 * roundtrip = 1 each stage is committed and waited for before the next.
 * Writes the SM cycles per MMA to issue the run and to see it complete.  The
 * pages have no counterpart: it measures the instruction the prompt-length
 * GEMMs are built on.  Allocates 24 bytes of device memory and synchronises
 * the device.  Errors: BM_ERR_INVALID_ARG (n not a multiple of 16 in
 * [16, 256], iters outside [1, 4096], NULL outputs), BM_ERR_CUDA,
 * BM_ERR_DEVICE_CHECK (the completion wait gave up). */
bm_status bm_probe_tcgen05_mma(int n, int a_in_tmem, int swizzle128, int iters, int roundtrip,
                               double* issue_cycles, double* complete_cycles);

/* Encode fp32 weights to the canonical int4 layout: per row and group of g,
 * s = fp16(absmax / 7) (fp32 division, round to nearest even), q =
 * clamp(rint(w / s), -8, 7) (fp32 division), u = q + 8; an all-zero group
 * gets s = 0.  W: DEVICE fp32 [N][K]; packed: DEVICE [N][K/2]; scales:
 * DEVICE fp16 [N][K/g].  Errors: BM_ERR_INVALID_ARG. */
bm_status bm_w4_quantize(const float* W, int N, int K, int g, uint8_t* packed, uint16_t* scales,
                         void* stream);

/* ---------------------------------------------------------------- host slot map
 * The engine's slot bookkeeping on its own, with no device involved, for
 * schedulers that want to plan admissions. */

bm_status bm_slot_map_create(int max_streams, int ctx_cap, bm_slot_map** out);
void bm_slot_map_destroy(bm_slot_map* m);
/* Lowest free slot, length = len.  BM_ERR_CTX_CAP if len >= ctx_cap or len < 0
 * is BM_ERR_INVALID_ARG; BM_ERR_NO_SLOT when full. */
bm_status bm_slot_map_acquire(bm_slot_map* m, int len, int* slot_out);
/* BM_ERR_SLOT_FREE on a free slot. */
bm_status bm_slot_map_release(bm_slot_map* m, int slot);
/* Check a batch: slot ids in range, distinct, active, length < ctx_cap. */
bm_status bm_slot_map_check_batch(const bm_slot_map* m, const int32_t* slots, int B);
/* length += 1 for each slot of a checked batch. */
bm_status bm_slot_map_advance(bm_slot_map* m, const int32_t* slots, int B);
bm_status bm_slot_map_length(const bm_slot_map* m, int slot, int* len_out);
int bm_slot_map_active_count(const bm_slot_map* m);

#ifdef __cplusplus
}
#endif

#endif /* BITMOE_H */
