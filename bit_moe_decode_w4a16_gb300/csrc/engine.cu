// Host runtime of the decode step: engine memory, the slot arena, weight
// loading, the per-B CUDA graph cache and the C ABI entry points.
//
// One decode step = one cudaGraphLaunch (the batched-serving page, §1: all
// layers plus the per-stream output projection are folded into one command
// buffer, one submit for the whole batch).  The host crosses to the device
// once per step: a small copy of slot ids and tokens into the graph's static
// input buffers, the launch, and a copy of the next tokens back.
#include <array>
#include <cstdio>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <new>
#include <set>
#include <string>
#include <vector>

#include <cmath>

#include "errors.h"
#include "kernels.cuh"
#include "persist.h"
#include "slot_map.h"

namespace bm {

std::string& last_error_slot() {
  thread_local std::string s;
  return s;
}

cudaError_t init_gemv_attributes();
cudaError_t init_moe_attributes();
cudaError_t init_misc_attributes();

namespace {

#define BM_CUDA(call, what)                                                                     \
  do {                                                                                          \
    cudaError_t _e = (call);                                                                    \
    if (_e != cudaSuccess) return set_error(BM_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(_e)); \
  } while (0)

std::mutex g_attr_mu;
std::set<int> g_attr_devices;

bm_status ensure_attributes() {
  int dev = 0;
  BM_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  std::lock_guard<std::mutex> lk(g_attr_mu);
  if (g_attr_devices.count(dev)) return BM_OK;
  BM_CUDA(init_gemv_attributes(), "kernel attributes (dense)");
  BM_CUDA(init_moe_attributes(), "kernel attributes (experts)");
  BM_CUDA(init_misc_attributes(), "kernel attributes (lm_head)");
  BM_CUDA(init_tc_attributes(), "kernel attributes (tensor-core projections)");
  BM_CUDA(init_mma_attributes(), "kernel attributes (warp-MMA projections)");
  BM_CUDA(init_prefill_attributes(), "kernel attributes (prompt-length tensor-core GEMMs)");
  g_attr_devices.insert(dev);
  return BM_OK;
}

size_t al(size_t v) { return (v + 255) & ~size_t(255); }

bool is_device_ptr(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

struct LayerW {
  uint8_t* wqkv = nullptr; __half* wqkv_s = nullptr;
  uint8_t* wo = nullptr;   __half* wo_s = nullptr;
  float* wr = nullptr;
  uint8_t* wg = nullptr;   __half* wg_s = nullptr;
  uint8_t* wu = nullptr;   __half* wu_s = nullptr;
  uint8_t* wd = nullptr;   __half* wd_s = nullptr;
  bf16* attn_norm_buf = nullptr; bf16* ffn_norm_buf = nullptr;
  bool has_attn_norm = false, has_ffn_norm = false;
  bool set = false;
};

}  // namespace
}  // namespace bm

using namespace bm;

struct bm_engine {
  bm_config cfg{};
  int family = BM_POLICY_SIMT;
  SlotMap slots;
  std::mutex mu;
  int device = 0;
  int qkv_rows = 0;
  // weights
  void* wslab = nullptr;
  size_t wbytes = 0;
  std::vector<LayerW> L;
  bf16* embed = nullptr;
  bf16* lm_head = nullptr;
  bf16* final_norm_buf = nullptr;
  bool has_final_norm = false;
  bool emb_set = false;
  // arena
  AttnArena arena{};
  void* arena_mem = nullptr;
  size_t arena_bytes = 0;
  float2* d_rope = nullptr;   // [ctx_cap][d/2] (cos, sin) of pos * theta_i
  // scratch
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  bf16 *x = nullptr, *qkv = nullptr, *q = nullptr, *attn = nullptr, *h = nullptr;
  bf16* xn = nullptr;                      // RMSNorm of x for the next projection (warp-MMA family)
  unsigned long long* lm_keys = nullptr;   // fused argmax keys [max_streams], zero between launches
  unsigned int* lm_counter = nullptr;
  unsigned int* route_cnt = nullptr;       // fused routing arrival counters [max_streams + 1], zero between launches
  unsigned int* attn_cnt = nullptr;        // fused attention arrival counters [attn_counter_count(max_streams, kv_heads)], zero between launches
  float* attn_part = nullptr;
  void* moe_ws = nullptr;
  float* logits = nullptr;
  int32_t *d_slots = nullptr, *d_tokens = nullptr, *d_next = nullptr, *d_slots_aux = nullptr;
  int* d_err = nullptr;
  // host staging (pinned)
  // A ring of kStageRing staging entries of [2 * max_streams] (slots, tokens)
  // lets the host run up to kStageRing steps ahead of the device.
  static constexpr int kStageRing = 8;
  int32_t* h_stage = nullptr;
  int32_t* h_aux = nullptr;     // [max_streams]: slots of standalone kv calls
  cudaEvent_t ev_ring[kStageRing] = {};
  int ring_pos = 0;
  cudaEvent_t ev_aux = nullptr;
  int32_t* d_u_log = nullptr;   // [layers] active experts of the last step, per layer
  float* tc_part = nullptr;     // split-K partial sums of the tensor-core projections
  int* tc_counters = nullptr;   // split-K arrival counters (zero between launches)
  size_t tc_counter_count = 0;
  std::vector<cudaEvent_t> prof_events;
  cudaStream_t cap_stream = nullptr;
  std::map<int, cudaGraphExec_t> graphs;   // decode graphs by B; prompt blocks under negative keys
  std::map<int, int> graph_kernels;         // kernels in each graph
  int test_drop_item = -1;                  // failure-detection tests: an expert item whose copies are not issued
  int test_drop_unit = -1;                  // failure-detection tests: a persistent-step weight unit not issued
  // prompt ingestion on the tensor cores (prefill_tc): rows per block and its scratch
  int pf_rows = 0;
  void* pf_mem = nullptr;
  bf16 *pf_x = nullptr, *pf_xn = nullptr, *pf_qkv = nullptr, *pf_h = nullptr;
  __half* pf_attn = nullptr;
  void* pf_moe = nullptr;
  float* pf_part = nullptr;
  unsigned int* pf_acnt = nullptr;
  int32_t *pf_slots = nullptr, *pf_tokens = nullptr;
  __half* pf_xg = nullptr;                 // the experts' input rows in sorted-pair order
  TmapBytes tm_xn{}, tm_attn{}, tm_xg{}, tm_act{};   // B operands of the prompt GEMMs
  // persistent small-batch decode step (persistent_step)
  int persist_rows = 0;                    // decode steps of B <= persist_rows rows run persistent; 0 = off
  PersistGeo pgeo{};
  void* pmem = nullptr;
  PersistLayer* d_players = nullptr;       // [layers]
  unsigned int* pst_bar = nullptr;         // grid barrier counter
  std::vector<PersistLayer> h_players;
  bool players_dirty = true;
  bm_stats st{};

  bm_engine(const bm_config& c) : cfg(c), slots(c.max_streams, c.ctx_cap) {}
};

namespace bm {
namespace {

DevCheck chk_of(bm_engine* e) { return DevCheck{e->d_err}; }

// K split of a tensor-core launch of `jobs` (tile, token group, expert) jobs.
void tc_split(bm_engine* e, TcArgs& t, int jobs) {
  t.ksplit = tc_pick_ksplit(jobs, t.K / 64);
  t.part = e->tc_part;
  t.counters = e->tc_counters;
}

// Largest (jobs, jobs * ksplit) over the engine's tensor-core launches.
void tc_workspace(const bm_config& c, int qkv_rows, size_t* max_jobs, size_t* max_part) {
  *max_jobs = 0;
  *max_part = 0;
  const int H = c.hidden, qd = c.q_heads * c.head_dim;
  for (int B = 1; B <= c.max_streams; ++B) {
    const int tg = (B + 15) / 16, max_u = B * c.top_k < c.experts ? B * c.top_k : c.experts;
    const int jobs[4] = {(qkv_rows / 128) * tg, (H / 128) * tg, (2 * c.ffn / 128) * tg * max_u,
                         (H / 128) * tg * max_u};
    const int nst[4] = {H / 64, qd / 64, H / 64, c.ffn / 64};
    for (int i = 0; i < 4; ++i) {
      const size_t j = jobs[i];
      *max_jobs = j > *max_jobs ? j : *max_jobs;
      const size_t p = tc_part_floats(jobs[i], tc_pick_ksplit(jobs[i], nst[i]));
      *max_part = p > *max_part ? p : *max_part;
    }
  }
}

// The step on the warp-MMA family.  Every RMSNorm is computed by the kernel
// that produces its input row (embedding, router, combine), so the
// projections read ready activations: embed+norm, then per layer QKV,
// attention (RoPE, append, chunks and merge in one launch), o_proj+residual,
// routing (router, top-k and sort in one launch), gate/up, down,
// combine+norm; then lm_head with the argmax fused.
// Prompt blocks (`prompt` 1, or 2 for the last block of a prompt) run the
// same kernels over B rows of one slot at positions len .. len + B - 1: the
// rows' k and v go to the arena first, attention takes each row's own
// position, and the length advances by B.  Only the last block's last row
// reaches the output projection.
enum PromptBlock { kDecode = 0, kPromptBlock = 1, kPromptLast = 2 };

cudaError_t enqueue_step_persist(bm_engine* e, int B, cudaStream_t s, int* launches);

cudaError_t enqueue_step_mma(bm_engine* e, int B, cudaStream_t s, int* launches, const Marker& mark,
                             int prompt = kDecode) {
  // small decode batches: one persistent launch for all layers (the same
  // bits); the per-kernel profiler keeps the multi-kernel step
  if (prompt == kDecode && B <= e->persist_rows && !mark.fn) return enqueue_step_persist(e, B, s, launches);
  const bm_config& c = e->cfg;
  const int H = c.hidden, qd = c.q_heads * c.head_dim, F = c.ffn, g = c.group;
  cudaError_t err;
  int n = 0;
  // kernels overlap their launch with the previous kernel's tail, except
  // under the per-kernel profiler, whose events sit between the launches
  const bool pdl = !mark.fn;
  auto attn_nw = [&](int l) -> const bf16* { return e->L[l].has_attn_norm ? e->L[l].attn_norm_buf : nullptr; };
  auto u32 = [](const __half* p) { return reinterpret_cast<const uint32_t*>(p); };
  __half* xn16 = reinterpret_cast<__half*>(e->xn);
  if ((err = launch_embed_norm(e->embed, c.vocab, H, e->d_tokens, e->x, attn_nw(0), c.rms_eps, xn16, B,
                               chk_of(e), s, pdl)) != cudaSuccess)
    return err;
  mark(KT_EMBED);
  ++n;
  for (int l = 0; l < c.layers; ++l) {
    const LayerW& w = e->L[l];
    MmaArgs m1{};
    m1.W = w.wqkv; m1.S = u32(w.wqkv_s); m1.rows = e->qkv_rows; m1.K = H; m1.g = g;
    m1.X = xn16; m1.ldx = H; m1.ntok = B; m1.Y = e->qkv; m1.ldy = e->qkv_rows; m1.pdl = pdl;
    if ((err = launch_w4_mma_dense(m1, s)) != cudaSuccess) return err;
    mark(KT_QKV);
    ++n;
    if (attention_fused_supports(e->arena, c.q_heads)) {
      AttnFusedArgs fa{e->arena, l, e->d_slots, e->qkv, e->qkv_rows, c.q_heads, e->d_rope,
                       reinterpret_cast<__half*>(e->attn), e->attn_part,
                       (c.ctx_cap + kAttnChunk - 1) / kAttnChunk, e->attn_cnt, B, chk_of(e),
                       prompt != kDecode ? 1 : 0};
      if (prompt != kDecode) {
        if ((err = launch_append_rows(fa, s, pdl)) != cudaSuccess) return err;
        mark(KT_ROPE_APPEND);
        ++n;
      }
      if ((err = launch_attention_fused(fa, s, pdl)) != cudaSuccess) return err;
      mark(KT_ATTN_PART);
      ++n;
    } else {
      if (prompt != kDecode) return cudaErrorNotSupported;
      if ((err = launch_rope_append(e->arena, l, e->d_slots, e->qkv, e->qkv_rows, c.q_heads, e->d_rope, e->q, B,
                                    chk_of(e), s, pdl)) != cudaSuccess)
        return err;
      mark(KT_ROPE_APPEND);
      ++n;
      if ((err = launch_attention(e->arena, l, e->d_slots, e->q, e->attn, c.q_heads, B, e->attn_part, chk_of(e), s,
                                  &n, mark, 1, pdl)) != cudaSuccess)
        return err;
    }
    MmaArgs m2{};
    m2.W = w.wo; m2.S = u32(w.wo_s); m2.rows = H; m2.K = qd; m2.g = g;
    m2.X = e->attn; m2.ldx = qd; m2.ntok = B; m2.Res = e->x; m2.ldr = H; m2.Y = e->h; m2.ldy = H; m2.pdl = pdl;
    if ((err = launch_w4_mma_dense(m2, s)) != cudaSuccess) return err;
    mark(KT_OPROJ);
    MoeArgs ma{B, c.experts, c.top_k, H, F, g, c.renorm_topk,
               w.wr, w.wg, w.wg_s, w.wu, w.wu_s, w.wd, w.wd_s,
               e->h, 1, w.has_ffn_norm ? w.ffn_norm_buf : nullptr, c.rms_eps, e->h, e->x, e->d_u_log + l, 1};
    const MoeBufs mb = moe_carve(e->moe_ws, B, c.experts, c.top_k, H, F);
    if ((err = launch_moe_route_fused(ma, mb, e->route_cnt, e->route_cnt + c.max_streams, s, mark, pdl)) !=
        cudaSuccess)
      return err;
    MmaArgs m3{};
    m3.W = w.wg; m3.S = u32(w.wg_s); m3.rows = 2 * F; m3.K = H; m3.g = g; m3.X = mb.xn; m3.ldx = H;
    m3.pair_token = mb.pair_token; m3.n_jobs = mb.n_jobs; m3.jobs = mb.jobs;
    m3.max_jobs = moe_max_jobs(B, c.experts, c.top_k);
    m3.w_expert_stride = (size_t)2 * F * H / 2; m3.s_expert_stride = (size_t)F * (H / g);
    m3.act16 = reinterpret_cast<__half*>(mb.act); m3.F = F; m3.err = e->d_err; m3.pdl = pdl;
    if ((err = launch_w4_mma_gateup(m3, s)) != cudaSuccess) return err;
    mark(KT_GATEUP);
    MmaArgs m4{};
    m4.W = w.wd; m4.S = u32(w.wd_s); m4.rows = H; m4.K = F; m4.g = g; m4.X = mb.act; m4.ldx = F;
    m4.pair_token = mb.pair_token; m4.n_jobs = mb.n_jobs; m4.jobs = mb.jobs; m4.max_jobs = m3.max_jobs;
    m4.w_expert_stride = (size_t)H * F / 2; m4.s_expert_stride = (size_t)H * (F / g) / 2;
    m4.out = mb.out; m4.H = H; m4.err = e->d_err; m4.pdl = pdl;
    if ((err = launch_w4_mma_down(m4, s)) != cudaSuccess) return err;
    mark(KT_DOWN);
    // the next layer's QKV reads fp16; the output projection reads bf16
    const bool last = l + 1 == c.layers;
    const bf16* next_nw = !last ? attn_nw(l + 1) : (e->has_final_norm ? e->final_norm_buf : nullptr);
    if ((err = launch_moe_combine_norm(ma, mb, next_nw, e->xn, last ? 0 : 1, s, mark, pdl)) != cudaSuccess) return err;
    n += 5;   // o_proj, routing, gate/up, down, combine
  }
  if (prompt == kPromptBlock) {
    // the slot's length moves past the block (row 0 of d_slots is the slot)
    if ((err = launch_advance(e->arena.len, e->d_slots, 1, s, B)) != cudaSuccess) return err;
    ++n;
    if (launches) *launches = n;
    return cudaSuccess;
  }
  LmArgs la{};
  la.W = e->lm_head; la.V = c.vocab; la.K = H; la.X = e->xn; la.B = B; la.logits = e->logits;
  la.next = e->d_next; la.len = e->arena.len; la.slots = e->d_slots; la.advance = 1;
  la.keys = e->lm_keys; la.counter = e->lm_counter; la.pdl = pdl;
  if (prompt == kPromptLast) {
    la.X = e->xn + (size_t)(B - 1) * H;
    la.B = 1;
    la.advance = B;
  }
  if ((err = launch_lm_mma(la, s)) != cudaSuccess) return err;
  mark(KT_LM_HEAD);
  ++n;
  if (launches) *launches = n;
  return cudaSuccess;
}

// The decode step of B <= persist_rows rows: the embedding and its RMSNorm,
// one cooperative launch for every layer (persist.cu), then the output
// projection with the fused argmax, as in the multi-kernel step.
cudaError_t enqueue_step_persist(bm_engine* e, int B, cudaStream_t s, int* launches) {
  const bm_config& c = e->cfg;
  const int H = c.hidden, qd = c.q_heads * c.head_dim, F = c.ffn, g = c.group;
  cudaError_t err;
  __half* xn16 = reinterpret_cast<__half*>(e->xn);
  const bf16* nw0 = e->L[0].has_attn_norm ? e->L[0].attn_norm_buf : nullptr;
  if ((err = launch_embed_norm(e->embed, c.vocab, H, e->d_tokens, e->x, nw0, c.rms_eps, xn16, B, chk_of(e), s,
                               false)) != cudaSuccess)
    return err;
  if ((err = cudaMemsetAsync(e->pst_bar, 0, sizeof(unsigned int), s)) != cudaSuccess) return err;
  PersistArgs a{};
  a.L = e->d_players;
  a.layers = c.layers;
  a.B = B;
  a.H = H; a.qd = qd; a.qkv_rows = e->qkv_rows; a.F = F; a.E = c.experts; a.k = c.top_k;
  a.eps = c.rms_eps;
  a.final_nw = e->has_final_norm ? e->final_norm_buf : nullptr;
  a.x = e->x; a.xn16 = xn16; a.xn_out = e->xn; a.qkv = e->qkv;
  a.attn = reinterpret_cast<__half*>(e->attn);
  a.h = e->h;
  a.moe = MoeArgs{B, c.experts, c.top_k, H, F, g, c.renorm_topk, nullptr, nullptr, nullptr, nullptr, nullptr,
                  nullptr, nullptr, e->h, 1, nullptr, c.rms_eps, e->h, e->x, nullptr, 1};
  a.mb = moe_carve(e->moe_ws, B, c.experts, c.top_k, H, F);
  a.mb_act16 = reinterpret_cast<__half*>(a.mb.act);
  a.at = AttnFusedArgs{e->arena, 0, e->d_slots, e->qkv, e->qkv_rows, c.q_heads, e->d_rope,
                       reinterpret_cast<__half*>(e->attn), e->attn_part, (c.ctx_cap + kAttnChunk - 1) / kAttnChunk,
                       e->attn_cnt, B, chk_of(e), 0, 0};
  a.wg_stride = (size_t)2 * F * H / 2; a.sg_stride = (size_t)F * (H / g);
  a.wd_stride = (size_t)H * F / 2;     a.sd_stride = (size_t)H * (F / g) / 2;
  a.u_log = e->d_u_log;
  a.bar = e->pst_bar;
  a.err = e->d_err;
  a.drop_unit1 = e->test_drop_unit >= 0 ? e->test_drop_unit + 1 : 0;
  a.geo = e->pgeo;
  if ((err = launch_persist_step(a, c.head_dim, g, s)) != cudaSuccess) return err;
  LmArgs la{};
  la.W = e->lm_head; la.V = c.vocab; la.K = H; la.X = e->xn; la.B = B; la.logits = e->logits;
  la.next = e->d_next; la.len = e->arena.len; la.slots = e->d_slots; la.advance = 1;
  la.keys = e->lm_keys; la.counter = e->lm_counter; la.pdl = 0;
  if ((err = launch_lm_mma(la, s)) != cudaSuccess) return err;
  if (launches) *launches = 3;
  return cudaSuccess;
}

// Prompt rows on the tensor cores: P rows of one slot (e->pf_slots holds P
// copies of it, e->pf_tokens the tokens) at positions len .. len + P - 1,
// each layer's dense projections and experts as prompt-length tcgen05 GEMMs,
// the rows' k and v appended first, attention in launches of up to 128 rows
// (row j attends to positions 0 .. len + j), the combine with the next
// RMSNorm; then the slot's length moves by P, through the output projection
// of the last row when `last`.
cudaError_t enqueue_prefill_tc(bm_engine* e, int P, bool last, cudaStream_t s, int* launches) {
  const bm_config& c = e->cfg;
  const int H = c.hidden, qd = c.q_heads * c.head_dim, F = c.ffn, g = c.group;
  cudaError_t err;
  int n = 0;
  auto attn_nw = [&](int l) -> const bf16* { return e->L[l].has_attn_norm ? e->L[l].attn_norm_buf : nullptr; };
  auto u32 = [](const __half* p) { return reinterpret_cast<const uint32_t*>(p); };
  __half* xn16 = reinterpret_cast<__half*>(e->pf_xn);
  if ((err = launch_embed_norm(e->embed, c.vocab, H, e->pf_tokens, e->pf_x, attn_nw(0), c.rms_eps, xn16, P, chk_of(e),
                               s, false)) != cudaSuccess)
    return err;
  ++n;
  for (int l = 0; l < c.layers; ++l) {
    const LayerW& w = e->L[l];
    PrefillGemmArgs q{};
    q.W = w.wqkv; q.S = u32(w.wqkv_s); q.rows = e->qkv_rows; q.K = H; q.g = g;
    q.X = xn16; q.ldx = H; q.ntok = P; q.Y = e->pf_qkv; q.ldy = e->qkv_rows; q.err = e->d_err;
    if ((err = launch_prefill_dense(q, e->tm_xn, s)) != cudaSuccess) return err;
    AttnFusedArgs fa{e->arena, l, e->pf_slots, e->pf_qkv, e->qkv_rows, c.q_heads, e->d_rope, e->pf_attn, e->pf_part,
                     (c.ctx_cap + kAttnChunk - 1) / kAttnChunk, e->pf_acnt, P, chk_of(e), 1, 0};
    if ((err = launch_append_rows(fa, s, false)) != cudaSuccess) return err;
    n += 2;
    if ((err = launch_attention_prefill(fa, s)) != cudaSuccess) return err;
    ++n;
    PrefillGemmArgs o{};
    o.W = w.wo; o.S = u32(w.wo_s); o.rows = H; o.K = qd; o.g = g;
    o.X = e->pf_attn; o.ldx = qd; o.ntok = P; o.Res = e->pf_x; o.ldr = H; o.Y = e->pf_h; o.ldy = H; o.err = e->d_err;
    if ((err = launch_prefill_dense(o, e->tm_attn, s)) != cudaSuccess) return err;
    MoeArgs ma{P, c.experts, c.top_k, H, F, g, c.renorm_topk,
               w.wr, w.wg, w.wg_s, w.wu, w.wu_s, w.wd, w.wd_s,
               e->pf_h, 1, w.has_ffn_norm ? w.ffn_norm_buf : nullptr, c.rms_eps, e->pf_h, e->pf_x, nullptr, 1};
    // the carve of the largest block: the tensor maps describe its buffers
    const MoeBufs mb = moe_carve(e->pf_moe, e->pf_rows, c.experts, c.top_k, H, F);
    MoeArgs mw = ma;
    if ((err = launch_moe_route_wide(mw, mb, s)) != cudaSuccess) return err;
    if ((err = launch_gather_rows(reinterpret_cast<const __half*>(mb.xn), mb.pair_token, P * c.top_k, H, e->pf_xg, s)) !=
        cudaSuccess)
      return err;
    PrefillGemmArgs gu{};
    gu.W = w.wg; gu.S = u32(w.wg_s); gu.rows = 2 * F; gu.K = H; gu.g = g; gu.X = e->pf_xg; gu.ldx = H;
    gu.n_active = mb.n_active; gu.active_e = mb.active_e; gu.active_off = mb.active_off; gu.row_map = mb.pair_token;
    gu.n_jobs = mb.n_jobs; gu.jobs = mb.jobs;
    gu.max_jobs = std::min(c.experts, P * c.top_k) + (P * c.top_k + kPromptTileRows - 1) / kPromptTileRows;
    gu.w_expert_stride = (size_t)2 * F * H / 2; gu.s_expert_stride = (size_t)F * (H / g);
    gu.act16 = reinterpret_cast<__half*>(mb.act); gu.F = F; gu.err = e->d_err;
    if ((err = launch_prefill_gateup(gu, e->tm_xg, P, s)) != cudaSuccess) return err;
    PrefillGemmArgs dn{};
    dn.W = w.wd; dn.S = u32(w.wd_s); dn.rows = H; dn.K = F; dn.g = g; dn.X = mb.act; dn.ldx = F;
    dn.n_active = mb.n_active; dn.active_e = mb.active_e; dn.active_off = mb.active_off;
    dn.n_jobs = mb.n_jobs; dn.jobs = mb.jobs; dn.max_jobs = gu.max_jobs;
    dn.w_expert_stride = (size_t)H * F / 2; dn.s_expert_stride = (size_t)H * (F / g) / 2;
    dn.out = mb.out; dn.H = H; dn.err = e->d_err;
    if ((err = launch_prefill_down(dn, e->tm_act, P, s)) != cudaSuccess) return err;
    const bool lastl = l + 1 == c.layers;
    const bf16* next_nw = !lastl ? attn_nw(l + 1) : (e->has_final_norm ? e->final_norm_buf : nullptr);
    if ((err = launch_moe_combine_norm_rows(ma, mb, next_nw, e->pf_xn, lastl ? 0 : 1, s)) != cudaSuccess) return err;
    n += 9;   // o_proj, routing (3), gather, gate/up, down, combine
  }
  if (!last) {
    if ((err = launch_advance(e->arena.len, e->pf_slots, 1, s, P)) != cudaSuccess) return err;
  } else {
    LmArgs la{};
    la.W = e->lm_head; la.V = c.vocab; la.K = H; la.X = e->pf_xn + (size_t)(P - 1) * H; la.B = 1;
    la.logits = e->logits; la.next = e->d_next; la.len = e->arena.len; la.slots = e->pf_slots; la.advance = P;
    la.keys = e->lm_keys; la.counter = e->lm_counter;
    if ((err = launch_lm_mma(la, s)) != cudaSuccess) return err;
  }
  ++n;
  if (launches) *launches = n;
  return cudaSuccess;
}

// Enqueue one decode step for B streams reading e->d_slots / e->d_tokens.
cudaError_t enqueue_step(bm_engine* e, int B, cudaStream_t s, int* launches, const Marker& mark = Marker(),
                         int prompt = kDecode) {
  if (e->family == BM_POLICY_MMA) return enqueue_step_mma(e, B, s, launches, mark, prompt);
  if (prompt != kDecode) return cudaErrorNotSupported;
  const bm_config& c = e->cfg;
  const int H = c.hidden, qd = c.q_heads * c.head_dim;
  const bool tc = e->family == BM_POLICY_TC;
  cudaError_t err;
  int n = 0;
  if ((err = launch_embed(e->embed, c.vocab, H, e->d_tokens, e->x, B, chk_of(e), s)) != cudaSuccess) return err;
  mark(KT_EMBED);
  ++n;
  for (int l = 0; l < c.layers; ++l) {
    const LayerW& w = e->L[l];
    const bf16* attn_nw = w.has_attn_norm ? w.attn_norm_buf : nullptr;
    if (tc) {
      TcArgs t1{};
      t1.W = w.wqkv; t1.S = w.wqkv_s; t1.rows = e->qkv_rows; t1.K = H; t1.g = c.group;
      t1.X = e->x; t1.ldx = H; t1.ntok = B; t1.do_norm = 1; t1.norm_w = attn_nw; t1.eps = c.rms_eps;
      t1.Y = e->qkv; t1.ldy = e->qkv_rows; t1.err = e->d_err;
      tc_split(e, t1, (e->qkv_rows / 128) * ((B + 15) / 16));
      if ((err = launch_w4_tc_dense(t1, s)) != cudaSuccess) return err;
    } else {
      GemvArgs g1{w.wqkv, w.wqkv_s, e->x, H, nullptr, 0, e->qkv, e->qkv_rows, B, e->qkv_rows, H, c.group,
                  1, attn_nw, c.rms_eps};
      if ((err = launch_w4_gemv(g1, s)) != cudaSuccess) return err;
    }
    mark(KT_QKV);
    ++n;
    if ((err = launch_rope_append(e->arena, l, e->d_slots, e->qkv, e->qkv_rows, c.q_heads, e->d_rope, e->q, B,
                                  chk_of(e), s)) != cudaSuccess)
      return err;
    mark(KT_ROPE_APPEND);
    ++n;
    if ((err = launch_attention(e->arena, l, e->d_slots, e->q, e->attn, c.q_heads, B, e->attn_part, chk_of(e), s,
                                &n, mark)) != cudaSuccess)
      return err;
    if (tc) {
      TcArgs t2{};
      t2.W = w.wo; t2.S = w.wo_s; t2.rows = H; t2.K = qd; t2.g = c.group;
      t2.X = e->attn; t2.ldx = qd; t2.ntok = B; t2.Res = e->x; t2.ldr = H; t2.Y = e->h; t2.ldy = H;
      t2.err = e->d_err;
      tc_split(e, t2, (H / 128) * ((B + 15) / 16));
      if ((err = launch_w4_tc_dense(t2, s)) != cudaSuccess) return err;
    } else {
      GemvArgs g2{w.wo, w.wo_s, e->attn, qd, e->x, H, e->h, H, B, H, qd, c.group, 0, nullptr, c.rms_eps};
      if ((err = launch_w4_gemv(g2, s)) != cudaSuccess) return err;
    }
    mark(KT_OPROJ);
    ++n;
    MoeArgs ma{B, c.experts, c.top_k, H, c.ffn, c.group, c.renorm_topk,
               w.wr, w.wg, w.wg_s, w.wu, w.wu_s, w.wd, w.wd_s,
               e->h, 1, w.has_ffn_norm ? w.ffn_norm_buf : nullptr, c.rms_eps, e->h, e->x, e->d_u_log + l};
    const MoeBufs mb = moe_carve(e->moe_ws, B, c.experts, c.top_k, H, c.ffn);
    if (tc) {
      if ((err = launch_moe_route(ma, mb, s, mark)) != cudaSuccess) return err;
      const int max_u = B * c.top_k < c.experts ? B * c.top_k : c.experts;
      TcArgs t3{};
      t3.W = w.wg; t3.S = w.wg_s; t3.rows = 2 * c.ffn; t3.K = H; t3.g = c.group; t3.X = mb.xn; t3.ldx = H;
      t3.n_active = mb.n_active; t3.active_e = mb.active_e; t3.active_off = mb.active_off;
      t3.pair_token = mb.pair_token; t3.w_expert_stride = (size_t)2 * c.ffn * H / 2;
      t3.s_expert_stride = (size_t)2 * c.ffn * (H / c.group); t3.act = mb.act; t3.F = c.ffn; t3.err = e->d_err;
      tc_split(e, t3, (2 * c.ffn / 128) * ((B + 15) / 16) * max_u);
      if ((err = launch_w4_tc_gateup(t3, max_u, B, s)) != cudaSuccess) return err;
      mark(KT_GATEUP);
      TcArgs t4{};
      t4.W = w.wd; t4.S = w.wd_s; t4.rows = H; t4.K = c.ffn; t4.g = c.group; t4.X = mb.act; t4.ldx = c.ffn;
      t4.n_active = mb.n_active; t4.active_e = mb.active_e; t4.active_off = mb.active_off;
      t4.pair_token = mb.pair_token; t4.w_expert_stride = (size_t)H * c.ffn / 2;
      t4.s_expert_stride = (size_t)H * (c.ffn / c.group); t4.out = mb.out; t4.H = H; t4.err = e->d_err;
      tc_split(e, t4, (H / 128) * ((B + 15) / 16) * max_u);
      if ((err = launch_w4_tc_down(t4, max_u, B, s)) != cudaSuccess) return err;
      mark(KT_DOWN);
      if ((err = launch_moe_combine(ma, mb, s, mark)) != cudaSuccess) return err;
      n += 5;
    } else {
      if ((err = launch_moe(ma, mb, s, &n, mark)) != cudaSuccess) return err;
    }
  }
  const bf16* final_nw = e->has_final_norm ? e->final_norm_buf : nullptr;
  if (tc && c.vocab % 128 == 0) {
    TcArgs tl{};
    tl.W = reinterpret_cast<const uint8_t*>(e->lm_head); tl.rows = c.vocab; tl.K = H; tl.g = c.group;
    tl.X = e->x; tl.ldx = H; tl.ntok = B; tl.do_norm = 1; tl.norm_w = final_nw; tl.eps = c.rms_eps;
    tl.out = e->logits; tl.ksplit = 1; tl.err = e->d_err;
    if ((err = launch_lm_tc(tl, s)) != cudaSuccess) return err;
  } else if ((err = launch_lm_head(e->lm_head, c.vocab, H, e->x, final_nw, c.rms_eps, e->logits, B, s)) !=
             cudaSuccess) {
    return err;
  }
  mark(KT_LM_HEAD);
  ++n;
  if ((err = launch_argmax(e->logits, c.vocab, B, e->d_next, e->arena.len, e->d_slots, 1, s)) != cudaSuccess)
    return err;
  mark(KT_ARGMAX);
  ++n;
  if (launches) *launches = n;
  return cudaSuccess;
}

const char* kTagNames[KT_COUNT] = {"embed", "qkv_w4", "rope_append", "attn_partial", "attn_combine", "oproj_w4",
                                   "router", "topk_sort", "expert_gateup", "expert_down", "moe_combine",
                                   "lm_head", "argmax"};

// Algorithmic HBM bytes and flops of one launch of a kernel class for a
// batch of B streams: each weight byte once, each activation once, and the
// K/V positions actually attended (`kv_pos` = sum over streams of len + 1);
// `U` = active experts of the layer.
void algo_cost(const bm_config& c, int qkv_rows, int tag, int B, double U, double kv_pos, double* bytes,
               double* flops) {
  const double H = c.hidden, qd = (double)c.q_heads * c.head_dim, kvd = (double)c.kv_heads * c.head_dim;
  const double g = c.group, E = c.experts, F = c.ffn, V = c.vocab, P = (double)B * c.top_k;
  const double chunks = std::ceil(kv_pos / B / kAttnChunk) * B;
  auto w4 = [&](double rows, double K) { return rows * (K / 2 + K / g * 2); };
  double b = 0, f = 0;
  switch (tag) {
    case KT_EMBED: b = 4.0 * B * H; break;
    case KT_QKV: b = w4(qkv_rows, H) + 2.0 * B * H + 2.0 * B * qkv_rows; f = 2.0 * B * qkv_rows * H; break;
    case KT_ROPE_APPEND: b = 2.0 * B * qkv_rows + 2.0 * B * (qd + 2 * kvd); break;
    case KT_ATTN_PART:
      b = kv_pos * kvd * 2 * 2 + 2.0 * B * qd + chunks * c.q_heads * (c.head_dim + 2) * 4;
      f = kv_pos * c.q_heads * c.head_dim * 4;
      break;
    case KT_ATTN_COMBINE: b = chunks * c.q_heads * (c.head_dim + 2) * 4 + 2.0 * B * qd; break;
    case KT_OPROJ: b = w4(H, qd) + 2.0 * B * qd + 4.0 * B * H; f = 2.0 * B * H * qd; break;
    case KT_ROUTER: b = E * H * 4 + 4.0 * B * H + 4.0 * B * E; f = 2.0 * B * E * H; break;
    case KT_TOPK_SORT: b = 4.0 * B * E + 8.0 * P; break;
    case KT_GATEUP: b = U * w4(2 * F, H) + 2.0 * P * H + 2.0 * P * F; f = 2.0 * P * 2 * F * H; break;
    case KT_DOWN: b = U * w4(H, F) + 2.0 * P * F + 4.0 * P * H; f = 2.0 * P * H * F; break;
    case KT_COMBINE: b = 4.0 * P * H + 4.0 * B * H; break;
    case KT_LM_HEAD: b = 2.0 * V * H + 2.0 * B * H + 4.0 * B * V; f = 2.0 * B * V * H; break;
    case KT_ARGMAX: b = 4.0 * B * V; break;
  }
  *bytes = b;
  *flops = f;
}

bool tc_shapes_ok(const bm_config& c) {
  const int qkv_rows = (c.q_heads + 2 * c.kv_heads) * c.head_dim, qd = c.q_heads * c.head_dim;
  return tc_supports(qkv_rows, c.hidden, c.group) && tc_supports(c.hidden, qd, c.group) &&
         tc_supports(2 * c.ffn, c.hidden, c.group) && tc_supports(c.hidden, c.ffn, c.group);
}

bool mma_shapes_ok(const bm_config& c) {
  const int qkv_rows = (c.q_heads + 2 * c.kv_heads) * c.head_dim, qd = c.q_heads * c.head_dim;
  return mma_supports(qkv_rows, c.hidden, c.group) && mma_supports(c.hidden, qd, c.group) &&
         mma_supports(2 * c.ffn, c.hidden, c.group) && mma_supports(c.hidden, c.ffn, c.group) &&
         c.ffn % 16 == 0 && lm_mma_supports(c.vocab, c.hidden, 1) && c.hidden <= 8192;
}

bm_status check_config(const bm_config& c) {
  auto bad = [](const std::string& m) { return set_error(BM_ERR_INVALID_ARG, "bm_engine_create: " + m); };
  if (c.hidden <= 0 || c.hidden % 32 != 0) return bad("hidden must be a positive multiple of 32");
  if (c.q_heads <= 0 || c.kv_heads <= 0 || c.q_heads % c.kv_heads != 0) return bad("q_heads % kv_heads != 0");
  if (c.q_heads / c.kv_heads > 8) return bad("at most 8 query heads per kv head");
  if (c.head_dim != 64 && c.head_dim != 128) return bad("head_dim must be 64 or 128");
  if (c.experts < 1 || c.experts > 256) return bad("experts must be in [1, 256]");
  if (c.top_k < 1 || c.top_k > 16 || c.top_k > c.experts) return bad("top_k must be in [1, min(16, experts)]");
  if (c.ffn <= 0 || c.ffn % 32 != 0) return bad("ffn must be a positive multiple of 32");
  if (c.group != 32 && c.group != 64 && c.group != 128) return bad("group must be 32, 64 or 128");
  if (c.hidden % c.group || c.ffn % c.group || (c.q_heads * c.head_dim) % c.group)
    return bad("every reduction length must be a multiple of group");
  if (c.vocab < 1 || c.layers < 1) return bad("vocab and layers must be >= 1");
  if (c.max_streams < 1 || c.max_streams > 128) return bad("max_streams must be in [1, 128]");
  if (c.max_streams > 64 && !(c.kernel_policy == BM_POLICY_MMA || (c.kernel_policy == BM_POLICY_AUTO && mma_shapes_ok(c))))
    return bad("max_streams above 64 needs the warp-MMA kernel family");
  if (c.max_streams * c.top_k > 1024) return bad("max_streams * top_k must be <= 1024");
  if (c.ctx_cap < 1 || c.ctx_cap > 131072) return bad("ctx_cap must be in [1, 131072]");
  if (!(c.rope_base > 0.f) || !(c.rms_eps >= 0.f)) return bad("rope_base > 0 and rms_eps >= 0 required");
  if (!simt_supports_k(c.hidden) || !simt_supports_k(c.ffn) || !simt_supports_k(c.q_heads * c.head_dim))
    return set_error(BM_ERR_UNSUPPORTED, "bm_engine_create: a reduction length has no kernel shape in this build");
  if (c.kernel_policy < 0 || c.kernel_policy > 3) return bad("unknown kernel_policy");
  if (c.kernel_policy == BM_POLICY_MMA && !mma_shapes_ok(c))
    return set_error(BM_ERR_UNSUPPORTED, "bm_engine_create: shapes outside the warp-MMA family (rows multiples "
                                         "of 32, reduction lengths multiples of 128 up to 4096, vocab % 16 == 0)");
  if (c.prefill_tc) {
    const int qkv_rows = (c.q_heads + 2 * c.kv_heads) * c.head_dim, qd = c.q_heads * c.head_dim;
    const bool mma_ok = c.kernel_policy == BM_POLICY_MMA || (c.kernel_policy == BM_POLICY_AUTO && mma_shapes_ok(c));
    const AttnArena ar0{nullptr, nullptr, nullptr, c.layers, c.max_streams, c.kv_heads, c.ctx_cap, c.head_dim};
    if (!mma_ok || !attention_prefill_supports(ar0, c.q_heads) || !prefill_gemm_supports(qkv_rows, c.hidden, c.group) ||
        !prefill_gemm_supports(c.hidden, qd, c.group) ||
        !prefill_gemm_supports(2 * c.ffn, c.hidden, c.group) || !prefill_gemm_supports(c.hidden, c.ffn, c.group) ||
        c.top_k > 16 || c.experts > 256)
      return set_error(BM_ERR_UNSUPPORTED, "bm_engine_create: prefill_tc needs the warp-MMA family and rows that are "
                                           "multiples of 128 with reduction lengths multiples of 256");
  }
  if (c.persistent_step) {
    const bool mma_ok = c.kernel_policy == BM_POLICY_MMA || (c.kernel_policy == BM_POLICY_AUTO && mma_shapes_ok(c));
    PersistGeo geo{};
    const char* why = "";
    const int rows = std::min(c.max_streams, kPMaxRows);
    if (!mma_ok)
      return set_error(BM_ERR_UNSUPPORTED, "bm_engine_create: persistent_step needs the warp-MMA kernel family");
    if (!attention_fused_supports(AttnArena{nullptr, nullptr, nullptr, c.layers, c.max_streams, c.kv_heads, c.ctx_cap,
                                            c.head_dim},
                                  c.q_heads) ||
        !persist_plan(c.hidden, c.q_heads * c.head_dim, (c.q_heads + 2 * c.kv_heads) * c.head_dim, c.ffn, c.experts,
                      c.top_k, c.group, c.head_dim, c.ctx_cap, std::min(rows, 64 / c.top_k), &geo, &why))
      return set_error(BM_ERR_UNSUPPORTED, std::string("bm_engine_create: persistent_step: ") + why);
  }
  if (c.kernel_policy == BM_POLICY_TC && !tc_shapes_ok(c))
    return set_error(BM_ERR_UNSUPPORTED, "bm_engine_create: shapes outside the tensor-core family (rows must be "
                                         "multiples of 128, reduction lengths multiples of 64 up to 4096)");
  return BM_OK;
}

void free_engine(bm_engine* e) {
  if (!e) return;
  for (auto& kv : e->graphs) cudaGraphExecDestroy(kv.second);
  if (e->cap_stream) cudaStreamDestroy(e->cap_stream);
  for (cudaEvent_t ev : e->ev_ring)
    if (ev) cudaEventDestroy(ev);
  for (cudaEvent_t ev : e->prof_events) cudaEventDestroy(ev);
  if (e->ev_aux) cudaEventDestroy(e->ev_aux);
  if (e->h_stage) cudaFreeHost(e->h_stage);
  if (e->wslab) cudaFree(e->wslab);
  if (e->arena_mem) cudaFree(e->arena_mem);
  if (e->scratch) cudaFree(e->scratch);
  if (e->pf_mem) cudaFree(e->pf_mem);
  if (e->pmem) cudaFree(e->pmem);
  delete e;
}

// Upload the host slot list of a standalone kv call into d_slots_aux.
bm_status stage_aux_slots(bm_engine* e, const int32_t* slots, int B, cudaStream_t s) {
  BM_CUDA(cudaEventSynchronize(e->ev_aux), "staging event");
  std::memcpy(e->h_aux, slots, sizeof(int32_t) * B);
  BM_CUDA(cudaMemcpyAsync(e->d_slots_aux, e->h_aux, sizeof(int32_t) * B, cudaMemcpyHostToDevice, s), "slot upload");
  BM_CUDA(cudaEventRecord(e->ev_aux, s), "staging event");
  return BM_OK;
}

}  // namespace
}  // namespace bm

// =================================================================== C ABI

extern "C" {

const char* bm_last_error(void) { return bm::last_error_slot().c_str(); }

bm_status bm_engine_create(const bm_config* cfg, bm_engine** out) {
  if (!cfg || !out) return set_error(BM_ERR_INVALID_ARG, "bm_engine_create: null argument");
  *out = nullptr;
  bm_status st = check_config(*cfg);
  if (st != BM_OK) return st;
  if ((st = ensure_attributes()) != BM_OK) return st;
  bm_engine* e = new (std::nothrow) bm_engine(*cfg);
  if (!e) return set_error(BM_ERR_OOM, "bm_engine_create: out of host memory");
  std::unique_ptr<bm_engine, void (*)(bm_engine*)> guard(e, free_engine);
  const bm_config& c = e->cfg;
  cudaGetDevice(&e->device);
  // The family is fixed for the engine's life, never chosen per step, so a
  // stream's bytes never depend on the batch it is decoded in.
  if (c.kernel_policy == BM_POLICY_SIMT) e->family = BM_POLICY_SIMT;
  else if (c.kernel_policy == BM_POLICY_TC) e->family = BM_POLICY_TC;
  else if (mma_shapes_ok(c)) e->family = BM_POLICY_MMA;
  else e->family = tc_shapes_ok(c) ? BM_POLICY_TC : BM_POLICY_SIMT;
  e->qkv_rows = (c.q_heads + 2 * c.kv_heads) * c.head_dim;
  const int H = c.hidden, E = c.experts, F = c.ffn, g = c.group, qd = c.q_heads * c.head_dim;
  const size_t S = c.max_streams;

  // ---- weight slab
  struct Part { size_t off, bytes; };
  size_t off = 0;
  auto take = [&](size_t bytes) { Part p{off, bytes}; off += al(bytes); return p; };
  std::vector<std::array<Part, 13>> lp(c.layers);
  for (int l = 0; l < c.layers; ++l) {
    auto& p = lp[l];
    p[0] = take((size_t)e->qkv_rows * H / 2);
    p[1] = take((size_t)e->qkv_rows * (H / g) * 2);
    p[2] = take((size_t)H * qd / 2);
    p[3] = take((size_t)H * (qd / g) * 2);
    p[4] = take((size_t)E * H * 4);
    // gate and up banks share one region: [wg | wu] (CUDA-core family) or
    // one row-interleaved bank of 2F rows per expert (tensor-core family)
    p[5] = take((size_t)E * 2 * F * H / 2);
    p[6] = take((size_t)E * 2 * F * (H / g) * 2);
    p[7] = take(0);
    p[8] = take(0);
    p[9] = take((size_t)E * H * F / 2);
    p[10] = take((size_t)E * H * (F / g) * 2);
    p[11] = take((size_t)H * 2);
    p[12] = take((size_t)H * 2);
  }
  const Part p_emb = take((size_t)c.vocab * H * 2), p_lm = take((size_t)c.vocab * H * 2), p_fn = take((size_t)H * 2);
  e->wbytes = off;
  BM_CUDA(cudaMalloc(&e->wslab, e->wbytes), "weight slab allocation");
  char* wb = static_cast<char*>(e->wslab);
  e->L.resize(c.layers);
  for (int l = 0; l < c.layers; ++l) {
    auto& p = lp[l];
    LayerW& w = e->L[l];
    w.wqkv = reinterpret_cast<uint8_t*>(wb + p[0].off); w.wqkv_s = reinterpret_cast<__half*>(wb + p[1].off);
    w.wo = reinterpret_cast<uint8_t*>(wb + p[2].off);   w.wo_s = reinterpret_cast<__half*>(wb + p[3].off);
    w.wr = reinterpret_cast<float*>(wb + p[4].off);
    w.wg = reinterpret_cast<uint8_t*>(wb + p[5].off);   w.wg_s = reinterpret_cast<__half*>(wb + p[6].off);
    w.wu = w.wg + (size_t)E * F * H / 2;                w.wu_s = w.wg_s + (size_t)E * F * (H / g);
    w.wd = reinterpret_cast<uint8_t*>(wb + p[9].off);   w.wd_s = reinterpret_cast<__half*>(wb + p[10].off);
    w.attn_norm_buf = reinterpret_cast<bf16*>(wb + p[11].off);
    w.ffn_norm_buf = reinterpret_cast<bf16*>(wb + p[12].off);
  }
  e->embed = reinterpret_cast<bf16*>(wb + p_emb.off);
  e->lm_head = reinterpret_cast<bf16*>(wb + p_lm.off);
  e->final_norm_buf = reinterpret_cast<bf16*>(wb + p_fn.off);

  // ---- KV arena: [layer][slot][kv head][position][d], K then V
  AttnArena& ar = e->arena;
  ar.layers = c.layers; ar.S = c.max_streams; ar.kvh = c.kv_heads; ar.cap = c.ctx_cap; ar.d = c.head_dim;
  const size_t kv_elems = (size_t)c.layers * ar.layer_stride();
  const size_t rope_elems = (size_t)c.ctx_cap * (c.head_dim / 2);
  e->arena_bytes = al(kv_elems * 2) * 2 + al(S * 4) + al(rope_elems * sizeof(float2));
  BM_CUDA(cudaMalloc(&e->arena_mem, e->arena_bytes), "KV arena allocation");
  char* am = static_cast<char*>(e->arena_mem);
  ar.K = reinterpret_cast<bf16*>(am);
  ar.V = reinterpret_cast<bf16*>(am + al(kv_elems * 2));
  ar.len = reinterpret_cast<int32_t*>(am + 2 * al(kv_elems * 2));
  e->d_rope = reinterpret_cast<float2*>(am + 2 * al(kv_elems * 2) + al(S * 4));
  BM_CUDA(cudaMemset(ar.len, 0, S * 4), "arena length reset");
  {
    // cos / sin of pos * theta_i, theta_i = base^(-2i/d), in double, stored as float
    const int half = c.head_dim / 2;
    std::vector<double> theta(half);
    for (int i = 0; i < half; ++i) theta[i] = std::pow((double)c.rope_base, -2.0 * i / c.head_dim);
    std::vector<float2> tab(rope_elems);
    for (int p = 0; p < c.ctx_cap; ++p)
      for (int i = 0; i < half; ++i) {
        const double ang = (double)p * theta[i];
        tab[(size_t)p * half + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
      }
    BM_CUDA(cudaMemcpy(e->d_rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice),
            "rope table upload");
  }

  // ---- scratch
  off = 0;
  const Part s_x = take(S * H * 2), s_qkv = take(S * e->qkv_rows * 2), s_q = take(S * qd * 2),
             s_attn = take(S * qd * 2), s_h = take(S * H * 2),
             s_part = take(attn_partial_floats(c.max_streams, c.q_heads, c.ctx_cap, c.head_dim) * 4),
             s_moe = take(moe_scratch_bytes(c.max_streams, E, c.top_k, H, F)),
             s_log = take(S * (size_t)c.vocab * 4), s_sl = take(S * 4), s_tk = take(S * 4), s_nx = take(S * 4),
             s_sa = take(S * 4), s_err = take(4), s_ulog = take((size_t)c.layers * 4), s_xn = take(S * H * 2),
             s_keys = take(S * 8), s_cnt = take(4), s_rcnt = take((S + 1) * 4), s_acnt = take(attn_counter_count(S, c.kv_heads) * 4);
  size_t tc_jobs = 0, tc_floats = 0;
  if (e->family == BM_POLICY_TC) tc_workspace(c, e->qkv_rows, &tc_jobs, &tc_floats);
  const Part s_tcp = take(tc_floats * 4), s_tcc = take(tc_jobs * 4);
  e->scratch_bytes = off;
  BM_CUDA(cudaMalloc(&e->scratch, e->scratch_bytes), "scratch allocation");
  char* sb = static_cast<char*>(e->scratch);
  e->x = reinterpret_cast<bf16*>(sb + s_x.off);
  e->qkv = reinterpret_cast<bf16*>(sb + s_qkv.off);
  e->q = reinterpret_cast<bf16*>(sb + s_q.off);
  e->attn = reinterpret_cast<bf16*>(sb + s_attn.off);
  e->h = reinterpret_cast<bf16*>(sb + s_h.off);
  e->attn_part = reinterpret_cast<float*>(sb + s_part.off);
  e->moe_ws = sb + s_moe.off;
  e->logits = reinterpret_cast<float*>(sb + s_log.off);
  e->d_slots = reinterpret_cast<int32_t*>(sb + s_sl.off);
  e->d_tokens = reinterpret_cast<int32_t*>(sb + s_tk.off);
  e->d_next = reinterpret_cast<int32_t*>(sb + s_nx.off);
  e->d_slots_aux = reinterpret_cast<int32_t*>(sb + s_sa.off);
  e->d_err = reinterpret_cast<int*>(sb + s_err.off);
  e->d_u_log = reinterpret_cast<int32_t*>(sb + s_ulog.off);
  e->xn = reinterpret_cast<bf16*>(sb + s_xn.off);
  e->lm_keys = reinterpret_cast<unsigned long long*>(sb + s_keys.off);
  e->lm_counter = reinterpret_cast<unsigned int*>(sb + s_cnt.off);
  e->route_cnt = reinterpret_cast<unsigned int*>(sb + s_rcnt.off);
  e->attn_cnt = reinterpret_cast<unsigned int*>(sb + s_acnt.off);

  e->tc_part = tc_floats ? reinterpret_cast<float*>(sb + s_tcp.off) : nullptr;
  e->tc_counters = tc_jobs ? reinterpret_cast<int*>(sb + s_tcc.off) : nullptr;
  e->tc_counter_count = tc_jobs;
  BM_CUDA(cudaMemset(e->scratch, 0, e->scratch_bytes), "scratch reset");

  if (c.prefill_tc) {
    // blocks of up to 512 prompt rows (4096 routed pairs)
    const int P = 4096 / c.top_k < 512 ? 4096 / c.top_k : 512;
    e->pf_rows = P;
    size_t o2 = 0;
    auto take2 = [&](size_t bytes) { size_t r = o2; o2 += al(bytes); return r; };
    const size_t p_x = take2((size_t)P * H * 2), p_xn = take2((size_t)P * H * 2),
                 p_qkv = take2((size_t)P * e->qkv_rows * 2), p_attn = take2((size_t)P * qd * 2),
                 p_h = take2((size_t)P * H * 2), p_moe = take2(moe_scratch_bytes(P, E, c.top_k, H, F)),
                 p_part = take2(attn_partial_floats(128, c.q_heads, c.ctx_cap, c.head_dim) * 4),
                 p_acnt = take2(attn_counter_count(128, c.kv_heads) * 4), p_sl = take2((size_t)P * 4), p_tk = take2((size_t)P * 4),
                 p_xg = take2((size_t)P * c.top_k * H * 2);
    BM_CUDA(cudaMalloc(&e->pf_mem, o2), "prompt scratch allocation");
    char* pb = static_cast<char*>(e->pf_mem);
    e->pf_x = reinterpret_cast<bf16*>(pb + p_x);
    e->pf_xn = reinterpret_cast<bf16*>(pb + p_xn);
    e->pf_qkv = reinterpret_cast<bf16*>(pb + p_qkv);
    e->pf_attn = reinterpret_cast<__half*>(pb + p_attn);
    e->pf_h = reinterpret_cast<bf16*>(pb + p_h);
    e->pf_moe = pb + p_moe;
    e->pf_part = reinterpret_cast<float*>(pb + p_part);
    e->pf_acnt = reinterpret_cast<unsigned int*>(pb + p_acnt);
    e->pf_slots = reinterpret_cast<int32_t*>(pb + p_sl);
    e->pf_tokens = reinterpret_cast<int32_t*>(pb + p_tk);
    e->pf_xg = reinterpret_cast<__half*>(pb + p_xg);
    BM_CUDA(cudaMemset(e->pf_mem, 0, o2), "prompt scratch reset");
    const MoeBufs pmb = moe_carve(e->pf_moe, P, E, c.top_k, H, F);
    BM_CUDA(encode_rows_tmap(&e->tm_xn, e->pf_xn, P, H, H), "prompt tensor map (normed rows)");
    BM_CUDA(encode_rows_tmap(&e->tm_attn, e->pf_attn, P, qd, qd), "prompt tensor map (attention rows)");
    BM_CUDA(encode_rows_tmap(&e->tm_xg, e->pf_xg, P * c.top_k, H, H), "prompt tensor map (expert input rows)");
    BM_CUDA(encode_rows_tmap(&e->tm_act, pmb.act, P * c.top_k, F, F), "prompt tensor map (expert activations)");
    e->scratch_bytes += o2;
  }
  if (c.persistent_step) {
    e->persist_rows = std::min(std::min(c.max_streams, kPMaxRows), 64 / c.top_k);
    const char* why = "";
    if (!persist_plan(H, qd, e->qkv_rows, F, E, c.top_k, g, c.head_dim, c.ctx_cap, e->persist_rows, &e->pgeo, &why))
      return set_error(BM_ERR_UNSUPPORTED, std::string("bm_engine_create: persistent_step: ") + why);
    BM_CUDA(persist_init(e->pgeo, c.head_dim, g, &e->pgeo.grid), "persistent step attributes");
    const size_t lb = al(sizeof(PersistLayer) * c.layers);
    BM_CUDA(cudaMalloc(&e->pmem, lb + 256), "persistent step allocation");
    BM_CUDA(cudaMemset(e->pmem, 0, lb + 256), "persistent step reset");
    e->d_players = static_cast<PersistLayer*>(e->pmem);
    e->pst_bar = reinterpret_cast<unsigned int*>(static_cast<char*>(e->pmem) + lb);
    e->h_players.assign(c.layers, PersistLayer{});
  }
  BM_CUDA(cudaMallocHost(&e->h_stage, sizeof(int32_t) * (2 * bm_engine::kStageRing + 1) * S),
          "pinned staging allocation");
  e->h_aux = e->h_stage + 2 * bm_engine::kStageRing * S;
  for (cudaEvent_t& ev : e->ev_ring) {
    BM_CUDA(cudaEventCreateWithFlags(&ev, cudaEventDisableTiming), "event");
    BM_CUDA(cudaEventRecord(ev, 0), "event");
  }
  BM_CUDA(cudaEventCreateWithFlags(&e->ev_aux, cudaEventDisableTiming), "event");
  BM_CUDA(cudaEventRecord(e->ev_aux, 0), "event");
  BM_CUDA(cudaStreamCreateWithFlags(&e->cap_stream, cudaStreamNonBlocking), "capture stream");
  BM_CUDA(cudaDeviceSynchronize(), "engine setup");

  e->st.weight_bytes = e->wbytes;
  e->st.arena_bytes = e->arena_bytes;
  e->st.scratch_bytes = e->scratch_bytes;
  std::fprintf(stderr,
               "bitmoe: engine on device %d: weights %.3f GB, KV arena %.3f GB (%d layers x %d slots x %d "
               "positions x %d kv heads x %d), scratch %.1f MB, kernel family %s\n",
               e->device, e->wbytes / 1e9, e->arena_bytes / 1e9, c.layers, c.max_streams, c.ctx_cap, c.kv_heads,
               c.head_dim, e->scratch_bytes / 1e6,
               e->family == BM_POLICY_MMA ? "mma" : (e->family == BM_POLICY_TC ? "tc" : "simt"));
  *out = guard.release();
  return bm::ok();
}

void bm_engine_destroy(bm_engine* e) {
  if (!e) return;
  cudaDeviceSynchronize();
  free_engine(e);
}

bm_status bm_engine_set_layer(bm_engine* e, int layer, const bm_layer_weights* w, void* stream) {
  if (!e || !w) return set_error(BM_ERR_INVALID_ARG, "bm_engine_set_layer: null argument");
  std::lock_guard<std::mutex> lk(e->mu);
  const bm_config& c = e->cfg;
  if (layer < 0 || layer >= c.layers) return set_error(BM_ERR_INVALID_ARG, "bm_engine_set_layer: layer out of range");
  if (!w->wqkv || !w->wqkv_s || !w->wo || !w->wo_s || !w->wr || !w->wg || !w->wg_s || !w->wu || !w->wu_s ||
      !w->wd || !w->wd_s)
    return set_error(BM_ERR_INVALID_ARG, "bm_engine_set_layer: a weight pointer is null");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LayerW& d = e->L[layer];
  const int H = c.hidden, E = c.experts, F = c.ffn, g = c.group, qd = c.q_heads * c.head_dim;
  auto cp = [&](void* dst, const void* src, size_t bytes) {
    return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDefault, s);
  };
  if (e->family == BM_POLICY_MMA) {
    // repack into the warp-MMA layout; F % 8 == 0, so tile T of the whole
    // gate/up bank is gate rows 8T..8T+7 then the same up rows, all of one
    // expert, and expert x's tiles start at row 2xF
    auto h = [](const uint16_t* p) { return reinterpret_cast<const __half*>(p); };
    auto u32 = [](__half* p) { return reinterpret_cast<uint32_t*>(p); };
    BM_CUDA(launch_repack_mma(w->wqkv, h(w->wqkv_s), nullptr, nullptr, e->qkv_rows, H, g, d.wqkv, u32(d.wqkv_s), s),
            "set_layer wqkv repack");
    BM_CUDA(launch_repack_mma(w->wo, h(w->wo_s), nullptr, nullptr, H, qd, g, d.wo, u32(d.wo_s), s),
            "set_layer wo repack");
    BM_CUDA(launch_repack_mma(w->wg, h(w->wg_s), w->wu, h(w->wu_s), 2 * E * F, H, g, d.wg, u32(d.wg_s), s),
            "set_layer gate/up repack");
    BM_CUDA(launch_repack_mma(w->wd, h(w->wd_s), nullptr, nullptr, E * H, F, g, d.wd, u32(d.wd_s), s),
            "set_layer down repack");
    BM_CUDA(cp(d.wr, w->wr, (size_t)E * H * 4), "set_layer router");
  } else if (e->family == BM_POLICY_TC) {
    // repack into the tensor-core layout; the gate and up banks interleave
    // row by row (row 2f = gate f, row 2f+1 = up f) so a TMEM lane pair holds
    // both halves of one SiLU(g)*u
    auto h = [](const uint16_t* p) { return reinterpret_cast<const __half*>(p); };
    BM_CUDA(launch_repack_tc(w->wqkv, h(w->wqkv_s), nullptr, nullptr, e->qkv_rows, H, g, d.wqkv, d.wqkv_s, s),
            "set_layer wqkv repack");
    BM_CUDA(launch_repack_tc(w->wo, h(w->wo_s), nullptr, nullptr, H, qd, g, d.wo, d.wo_s, s), "set_layer wo repack");
    BM_CUDA(launch_repack_tc(w->wg, h(w->wg_s), w->wu, h(w->wu_s), 2 * E * F, H, g, d.wg, d.wg_s, s),
            "set_layer gate/up repack");
    BM_CUDA(launch_repack_tc(w->wd, h(w->wd_s), nullptr, nullptr, E * H, F, g, d.wd, d.wd_s, s),
            "set_layer down repack");
    BM_CUDA(cp(d.wr, w->wr, (size_t)E * H * 4), "set_layer router");
  } else {
    BM_CUDA(cp(d.wqkv, w->wqkv, (size_t)e->qkv_rows * H / 2), "set_layer wqkv");
    BM_CUDA(cp(d.wqkv_s, w->wqkv_s, (size_t)e->qkv_rows * (H / g) * 2), "set_layer wqkv scales");
    BM_CUDA(cp(d.wo, w->wo, (size_t)H * qd / 2), "set_layer wo");
    BM_CUDA(cp(d.wo_s, w->wo_s, (size_t)H * (qd / g) * 2), "set_layer wo scales");
    BM_CUDA(cp(d.wr, w->wr, (size_t)E * H * 4), "set_layer router");
    BM_CUDA(cp(d.wg, w->wg, (size_t)E * F * H / 2), "set_layer wg");
    BM_CUDA(cp(d.wg_s, w->wg_s, (size_t)E * F * (H / g) * 2), "set_layer wg scales");
    BM_CUDA(cp(d.wu, w->wu, (size_t)E * F * H / 2), "set_layer wu");
    BM_CUDA(cp(d.wu_s, w->wu_s, (size_t)E * F * (H / g) * 2), "set_layer wu scales");
    BM_CUDA(cp(d.wd, w->wd, (size_t)E * H * F / 2), "set_layer wd");
    BM_CUDA(cp(d.wd_s, w->wd_s, (size_t)E * H * (F / g) * 2), "set_layer wd scales");
  }
  d.has_attn_norm = w->attn_norm != nullptr;
  d.has_ffn_norm = w->ffn_norm != nullptr;
  if (w->attn_norm) BM_CUDA(cp(d.attn_norm_buf, w->attn_norm, (size_t)H * 2), "set_layer attn norm");
  if (w->ffn_norm) BM_CUDA(cp(d.ffn_norm_buf, w->ffn_norm, (size_t)H * 2), "set_layer ffn norm");
  if (e->cfg.persistent_step) {
    auto u32c = [](const __half* p) { return reinterpret_cast<const uint32_t*>(p); };
    e->h_players[layer] = PersistLayer{d.wqkv, u32c(d.wqkv_s), d.wo, u32c(d.wo_s), d.wr, d.wg, u32c(d.wg_s), d.wd,
                                       u32c(d.wd_s), d.has_attn_norm ? d.attn_norm_buf : nullptr,
                                       d.has_ffn_norm ? d.ffn_norm_buf : nullptr};
    e->players_dirty = true;
  }
  d.set = true;
  return bm::ok();
}

bm_status bm_engine_set_embeddings(bm_engine* e, const uint16_t* embed, const uint16_t* lm_head,
                                   const uint16_t* final_norm, void* stream) {
  if (!e || !embed || !lm_head) return set_error(BM_ERR_INVALID_ARG, "bm_engine_set_embeddings: null argument");
  std::lock_guard<std::mutex> lk(e->mu);
  const bm_config& c = e->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t bytes = (size_t)c.vocab * c.hidden * 2;
  BM_CUDA(cudaMemcpyAsync(e->embed, embed, bytes, cudaMemcpyDefault, s), "set_embeddings embed");
  BM_CUDA(cudaMemcpyAsync(e->lm_head, lm_head, bytes, cudaMemcpyDefault, s), "set_embeddings lm_head");
  e->has_final_norm = final_norm != nullptr;
  if (final_norm)
    BM_CUDA(cudaMemcpyAsync(e->final_norm_buf, final_norm, (size_t)c.hidden * 2, cudaMemcpyDefault, s),
            "set_embeddings final norm");
  e->emb_set = true;
  return bm::ok();
}

bm_status bm_engine_sync(bm_engine* e, void* stream) {
  if (!e) return set_error(BM_ERR_INVALID_ARG, "bm_engine_sync: null engine");
  BM_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream synchronise");
  int flag = 0;
  BM_CUDA(cudaMemcpy(&flag, e->d_err, sizeof(int), cudaMemcpyDeviceToHost), "device check read");
  if (flag) {
    BM_CUDA(cudaMemset(e->d_err, 0, sizeof(int)), "device check reset");
    // a kernel that stopped early may have left its arrival counters short:
    // every counter goes back to zero so the next launches start clean
    const size_t S = e->cfg.max_streams;
    BM_CUDA(cudaMemset(e->route_cnt, 0, (S + 1) * 4), "counter reset");
    BM_CUDA(cudaMemset(e->attn_cnt, 0, attn_counter_count(S, e->cfg.kv_heads) * 4), "counter reset");
    BM_CUDA(cudaMemset(e->lm_counter, 0, 4), "counter reset");
    BM_CUDA(cudaMemset(e->lm_keys, 0, S * 8), "counter reset");
    if (e->tc_counters) BM_CUDA(cudaMemset(e->tc_counters, 0, e->tc_counter_count * 4), "counter reset");
    static const char* what[] = {"", "an out-of-range slot id was skipped", "an out-of-range position was skipped",
                                 "an out-of-range token id was skipped",
                                 "a tensor-core projection's pipeline wait timed out",
                                 "an expert projection's pipeline wait timed out (the CTA stopped consuming)",
                                 "a wait of the persistent decode step timed out (every CTA left the step)"};
    return set_error(BM_ERR_DEVICE_CHECK, std::string("device check code ") + std::to_string(flag) + ": " +
                                              (flag >= 1 && flag <= 6 ? what[flag] : "unknown"));
  }
  return bm::ok();
}

bm_status bm_engine_stats(const bm_engine* e, bm_stats* out) {
  if (!e || !out) return set_error(BM_ERR_INVALID_ARG, "bm_engine_stats: null argument");
  *out = e->st;
  return bm::ok();
}

int bm_engine_kernel_family(const bm_engine* e) { return e ? e->family : -1; }

// ------------------------------------------------------------------ slots

bm_status kv_slot_seed(bm_engine* e, const uint16_t* K, const uint16_t* V, int len, int* slot_out, void* stream) {
  if (!e || !slot_out) return set_error(BM_ERR_INVALID_ARG, "kv_slot_seed: null argument");
  if (len > 0 && (!K || !V)) return set_error(BM_ERR_INVALID_ARG, "kv_slot_seed: null K or V with len > 0");
  std::lock_guard<std::mutex> lk(e->mu);
  std::string err;
  int slot = -1;
  bm_status st = e->slots.acquire(len, &slot, &err);
  if (st != BM_OK) return set_error(st, "kv_slot_seed: " + err);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const AttnArena& ar = e->arena;
  const size_t d = ar.d;
  cudaError_t ce = cudaSuccess;
  for (int l = 0; l < ar.layers && len > 0 && ce == cudaSuccess; ++l) {
    const size_t src_off = (size_t)l * ar.kvh * len * d;
    const size_t dst_off = l * ar.layer_stride() + slot * ar.slot_stride();
    ce = cudaMemcpy2DAsync(ar.K + dst_off, ar.cap * d * 2, K + src_off, len * d * 2, len * d * 2, ar.kvh,
                           cudaMemcpyDefault, s);
    if (ce == cudaSuccess)
      ce = cudaMemcpy2DAsync(ar.V + dst_off, ar.cap * d * 2, V + src_off, len * d * 2, len * d * 2, ar.kvh,
                             cudaMemcpyDefault, s);
  }
  if (ce == cudaSuccess) ce = launch_set_len(ar.len, slot, len, s);
  if (ce != cudaSuccess) {
    e->slots.release(slot, &err);
    return set_error(BM_ERR_CUDA, std::string("kv_slot_seed: ") + cudaGetErrorString(ce));
  }
  *slot_out = slot;
  return bm::ok();
}

bm_status kv_slot_append(bm_engine* e, int layer, const int32_t* slots, const uint16_t* Knew, const uint16_t* Vnew,
                         int B, void* stream) {
  if (!e || !Knew || !Vnew) return set_error(BM_ERR_INVALID_ARG, "kv_slot_append: null argument");
  std::lock_guard<std::mutex> lk(e->mu);
  if (layer < 0 || layer >= e->cfg.layers) return set_error(BM_ERR_INVALID_ARG, "kv_slot_append: layer out of range");
  std::string err;
  bm_status st = e->slots.check_batch(slots, B, &err);
  if (st != BM_OK) return set_error(st, "kv_slot_append: " + err);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = stage_aux_slots(e, slots, B, s)) != BM_OK) return st;
  BM_CUDA(launch_kv_append(e->arena, layer, e->d_slots_aux, reinterpret_cast<const bf16*>(Knew),
                           reinterpret_cast<const bf16*>(Vnew), B, chk_of(e), s),
          "kv_slot_append launch");
  e->st.kernel_launches += 1;
  return bm::ok();
}

bm_status kv_slot_attend(bm_engine* e, int layer, const int32_t* slots, const uint16_t* Q, uint16_t* O, int B,
                         void* stream) {
  if (!e || !Q || !O) return set_error(BM_ERR_INVALID_ARG, "kv_slot_attend: null argument");
  std::lock_guard<std::mutex> lk(e->mu);
  if (layer < 0 || layer >= e->cfg.layers) return set_error(BM_ERR_INVALID_ARG, "kv_slot_attend: layer out of range");
  std::string err;
  bm_status st = e->slots.check_batch(slots, B, &err);
  if (st != BM_OK) return set_error(st, "kv_slot_attend: " + err);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = stage_aux_slots(e, slots, B, s)) != BM_OK) return st;
  int n = 0;
  BM_CUDA(launch_attention(e->arena, layer, e->d_slots_aux, reinterpret_cast<const bf16*>(Q),
                           reinterpret_cast<bf16*>(O), e->cfg.q_heads, B, e->attn_part, chk_of(e), s, &n),
          "kv_slot_attend launch");
  e->st.kernel_launches += n;
  return bm::ok();
}

bm_status kv_slot_advance(bm_engine* e, const int32_t* slots, int B, void* stream) {
  if (!e) return set_error(BM_ERR_INVALID_ARG, "kv_slot_advance: null engine");
  std::lock_guard<std::mutex> lk(e->mu);
  std::string err;
  bm_status st = e->slots.check_batch(slots, B, &err);
  if (st != BM_OK) return set_error(st, "kv_slot_advance: " + err);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = stage_aux_slots(e, slots, B, s)) != BM_OK) return st;
  BM_CUDA(launch_advance(e->arena.len, e->d_slots_aux, B, s), "kv_slot_advance launch");
  e->slots.advance(slots, B);
  e->st.kernel_launches += 1;
  return bm::ok();
}

bm_status kv_slot_release(bm_engine* e, int slot) {
  if (!e) return set_error(BM_ERR_INVALID_ARG, "kv_slot_release: null engine");
  std::lock_guard<std::mutex> lk(e->mu);
  std::string err;
  const bm_status st = e->slots.release(slot, &err);
  return st == BM_OK ? bm::ok() : set_error(st, "kv_slot_release: " + err);
}

bm_status kv_slot_length(const bm_engine* e, int slot, int* len_out) {
  if (!e || !len_out) return set_error(BM_ERR_INVALID_ARG, "kv_slot_length: null argument");
  if (!e->slots.active(slot)) return set_error(BM_ERR_SLOT_FREE, "kv_slot_length: slot is not active");
  *len_out = e->slots.length(slot);
  return bm::ok();
}

bm_status kv_slot_read(bm_engine* e, int layer, int slot, int count, uint16_t* K_out, uint16_t* V_out,
                       void* stream) {
  if (!e || !K_out || !V_out) return set_error(BM_ERR_INVALID_ARG, "kv_slot_read: null argument");
  const AttnArena& ar = e->arena;
  if (layer < 0 || layer >= ar.layers || slot < 0 || slot >= ar.S || count < 0 || count > ar.cap)
    return set_error(BM_ERR_INVALID_ARG, "kv_slot_read: layer, slot or count out of range");
  if (count == 0) return bm::ok();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t d = ar.d, src = layer * ar.layer_stride() + slot * ar.slot_stride();
  BM_CUDA(cudaMemcpy2DAsync(K_out, count * d * 2, ar.K + src, ar.cap * d * 2, count * d * 2, ar.kvh,
                            cudaMemcpyDefault, s),
          "kv_slot_read K");
  BM_CUDA(cudaMemcpy2DAsync(V_out, count * d * 2, ar.V + src, ar.cap * d * 2, count * d * 2, ar.kvh,
                            cudaMemcpyDefault, s),
          "kv_slot_read V");
  return bm::ok();
}

// ------------------------------------------------------------------ step

}  // extern "C"

namespace bm {
namespace {

// Checks shared by decode_step and bm_engine_profile_step, then the upload of
// slot ids and tokens into the step's static device inputs (through the next
// entry of the pinned staging ring).
bm_status stage_inputs(bm_engine* e, int B, const int32_t* slots, const int32_t* tokens, cudaStream_t s);

bm_status prepare_step(bm_engine* e, int B, const int32_t* slots, const int32_t* tokens, int32_t* next_tokens,
                       cudaStream_t s, const char* who) {
  if (!e || !slots || !tokens || !next_tokens) return set_error(BM_ERR_INVALID_ARG, std::string(who) + ": null argument");
  const bm_config& c = e->cfg;
  if (!e->emb_set) return set_error(BM_ERR_NOT_READY, std::string(who) + ": embeddings not set");
  for (int l = 0; l < c.layers; ++l)
    if (!e->L[l].set) return set_error(BM_ERR_NOT_READY, std::string(who) + ": layer " + std::to_string(l) + " not set");
  std::string err;
  const bm_status st = e->slots.check_batch(slots, B, &err);
  if (st != BM_OK) return set_error(st, std::string(who) + ": " + err);
  return stage_inputs(e, B, slots, tokens, s);
}

// Copy B slot ids (host) and B tokens (host or device) to e->d_slots and
// e->d_tokens through the pinned staging ring.
bm_status stage_inputs(bm_engine* e, int B, const int32_t* slots, const int32_t* tokens, cudaStream_t s) {
  const size_t S = e->cfg.max_streams;
  const int slot = e->ring_pos;
  e->ring_pos = (e->ring_pos + 1) % bm_engine::kStageRing;
  int32_t* stage = e->h_stage + 2 * S * slot;
  BM_CUDA(cudaEventSynchronize(e->ev_ring[slot]), "staging event");
  std::memcpy(stage, slots, sizeof(int32_t) * B);
  BM_CUDA(cudaMemcpyAsync(e->d_slots, stage, sizeof(int32_t) * B, cudaMemcpyHostToDevice, s), "slot upload");
  if (is_device_ptr(tokens)) {
    BM_CUDA(cudaMemcpyAsync(e->d_tokens, tokens, sizeof(int32_t) * B, cudaMemcpyDeviceToDevice, s), "token copy");
  } else {
    std::memcpy(stage + S, tokens, sizeof(int32_t) * B);
    BM_CUDA(cudaMemcpyAsync(e->d_tokens, stage + S, sizeof(int32_t) * B, cudaMemcpyHostToDevice, s), "token upload");
  }
  BM_CUDA(cudaEventRecord(e->ev_ring[slot], s), "staging event");
  return BM_OK;
}

// Enqueue one step (or prompt block) of B rows from e->d_slots / e->d_tokens:
// through the cached CUDA graph of (B, prompt) when graphs are on, else
// eagerly.  *n_out = the kernels it launches.
bm_status run_step(bm_engine* e, int B, int prompt, cudaStream_t s, int* n_out, const char* who) {
  int n = 0;
  if (e->cfg.persistent_step && e->players_dirty) {
    BM_CUDA(cudaMemcpyAsync(e->d_players, e->h_players.data(), sizeof(PersistLayer) * e->h_players.size(),
                            cudaMemcpyHostToDevice, s),
            "persistent step layer table");
    BM_CUDA(cudaStreamSynchronize(s), "persistent step layer table");
    e->players_dirty = false;
  }
  if (e->cfg.use_graph) {
    const int key = prompt == kDecode ? B : -(4 * B + prompt);   // prompt graphs under negative keys
    auto it = e->graphs.find(key);
    if (it == e->graphs.end()) {
      cudaGraph_t graph = nullptr;
      BM_CUDA(cudaStreamBeginCapture(e->cap_stream, cudaStreamCaptureModeThreadLocal), "graph capture begin");
      const cudaError_t ce = enqueue_step(e, B, e->cap_stream, &n, Marker(), prompt);
      const cudaError_t ee = cudaStreamEndCapture(e->cap_stream, &graph);
      if (ce != cudaSuccess) {
        if (graph) cudaGraphDestroy(graph);
        return set_error(BM_ERR_CUDA, std::string(who) + " capture: " + cudaGetErrorString(ce));
      }
      BM_CUDA(ee, "graph capture end");
      cudaGraphExec_t exec = nullptr;
      const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
      cudaGraphDestroy(graph);
      BM_CUDA(ie, "graph instantiate");
      it = e->graphs.emplace(key, exec).first;
      e->graph_kernels[key] = n;
      e->st.graph_captures += 1;
    }
    BM_CUDA(cudaGraphLaunch(it->second, s), "graph launch");
    e->st.graph_launches += 1;
    n = e->graph_kernels[key];
  } else {
    const cudaError_t ce = enqueue_step(e, B, s, &n, Marker(), prompt);
    if (ce != cudaSuccess) return set_error(BM_ERR_CUDA, std::string(who) + " launch: " + cudaGetErrorString(ce));
  }
  e->st.kernel_launches += n;
  *n_out = n;
  return BM_OK;
}

struct ProfCtx {
  bm_engine* e;
  cudaStream_t s;
  std::vector<int> tags;
  cudaError_t err = cudaSuccess;
};

void prof_mark(void* ctx, int tag) {
  ProfCtx* p = static_cast<ProfCtx*>(ctx);
  const size_t i = p->tags.size() + 1;
  while (p->e->prof_events.size() <= i) {
    cudaEvent_t ev;
    if (cudaEventCreate(&ev) != cudaSuccess) {
      p->err = cudaErrorMemoryAllocation;
      return;
    }
    p->e->prof_events.push_back(ev);
  }
  if (p->err == cudaSuccess) p->err = cudaEventRecord(p->e->prof_events[i], p->s);
  p->tags.push_back(tag);
}

}  // namespace
}  // namespace bm

extern "C" {

bm_status decode_step(bm_engine* e, int B, const int32_t* slots, const int32_t* tokens, int32_t* next_tokens,
                      float* logits, void* stream) {
  if (!e) return set_error(BM_ERR_INVALID_ARG, "decode_step: null engine");
  std::lock_guard<std::mutex> lk(e->mu);
  const bm_config& c = e->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bm_status st = prepare_step(e, B, slots, tokens, next_tokens, s, "decode_step");
  if (st != BM_OK) return st;
  int n = 0;
  if ((st = run_step(e, B, kDecode, s, &n, "decode_step")) != BM_OK) return st;
  e->st.kernels_per_step = n;
  BM_CUDA(cudaMemcpyAsync(next_tokens, e->d_next, sizeof(int32_t) * B, cudaMemcpyDefault, s), "next token copy");
  if (logits)
    BM_CUDA(cudaMemcpyAsync(logits, e->logits, sizeof(float) * B * (size_t)c.vocab, cudaMemcpyDefault, s),
            "logits copy");
  e->slots.advance(slots, B);
  e->st.steps += 1;
  e->st.tokens += B;
  return bm::ok();
}

bm_status kv_slot_prefill(bm_engine* e, int slot, int n_tokens, const int32_t* tokens, int32_t* next_token,
                          float* logits, void* stream) {
  if (!e || !tokens || !next_token) return set_error(BM_ERR_INVALID_ARG, "kv_slot_prefill: null argument");
  std::lock_guard<std::mutex> lk(e->mu);
  const bm_config& c = e->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (n_tokens < 1) return set_error(BM_ERR_INVALID_ARG, "kv_slot_prefill: n_tokens must be >= 1");
  if (slot < 0 || slot >= c.max_streams) return set_error(BM_ERR_INVALID_ARG, "kv_slot_prefill: slot out of range");
  if (!e->slots.active(slot)) return set_error(BM_ERR_SLOT_FREE, "kv_slot_prefill: slot is not active");
  if (!e->emb_set) return set_error(BM_ERR_NOT_READY, "kv_slot_prefill: embeddings not set");
  for (int l = 0; l < c.layers; ++l)
    if (!e->L[l].set) return set_error(BM_ERR_NOT_READY, "kv_slot_prefill: layer " + std::to_string(l) + " not set");
  if (e->family != BM_POLICY_MMA || !attention_fused_supports(e->arena, c.q_heads))
    return set_error(BM_ERR_UNSUPPORTED, "kv_slot_prefill: needs the warp-MMA kernel family and fused attention");
  if ((long)e->slots.length(slot) + n_tokens > c.ctx_cap)
    return set_error(BM_ERR_CTX_CAP, "kv_slot_prefill: the prompt does not fit the context cap");
  if (c.prefill_tc) {
    const int T = e->pf_rows;
    for (int i = 0; i < n_tokens; i += T) {
      const int b = n_tokens - i < T ? n_tokens - i : T;
      BM_CUDA(cudaMemcpyAsync(e->pf_tokens, tokens + i, sizeof(int32_t) * b, cudaMemcpyDefault, s), "prompt tokens");
      BM_CUDA(launch_fill_i32(e->pf_slots, slot, b, s), "prompt slots");
      int n = 0;
      const cudaError_t ce = enqueue_prefill_tc(e, b, i + b == n_tokens, s, &n);
      if (ce != cudaSuccess) return set_error(BM_ERR_CUDA, std::string("kv_slot_prefill launch: ") + cudaGetErrorString(ce));
      e->st.kernel_launches += n + 1;
    }
    BM_CUDA(cudaMemcpyAsync(next_token, e->d_next, sizeof(int32_t), cudaMemcpyDefault, s), "next token copy");
    if (logits)
      BM_CUDA(cudaMemcpyAsync(logits, e->logits, sizeof(float) * (size_t)c.vocab, cudaMemcpyDefault, s), "logits copy");
    e->slots.advance_by(slot, n_tokens);
    e->st.tokens += n_tokens;
    return bm::ok();
  }
  const int T = c.max_streams;
  std::vector<int32_t> rows(T, slot);
  for (int i = 0; i < n_tokens; i += T) {
    const int b = n_tokens - i < T ? n_tokens - i : T;
    const int32_t* tok = tokens + i;
    bm_status st = stage_inputs(e, b, rows.data(), tok, s);
    if (st != BM_OK) return st;
    int n = 0;
    if ((st = run_step(e, b, i + b == n_tokens ? kPromptLast : kPromptBlock, s, &n, "kv_slot_prefill")) != BM_OK)
      return st;
  }
  BM_CUDA(cudaMemcpyAsync(next_token, e->d_next, sizeof(int32_t), cudaMemcpyDefault, s), "next token copy");
  if (logits)
    BM_CUDA(cudaMemcpyAsync(logits, e->logits, sizeof(float) * (size_t)c.vocab, cudaMemcpyDefault, s), "logits copy");
  e->slots.advance_by(slot, n_tokens);
  e->st.tokens += n_tokens;
  return bm::ok();
}

bm_status bm_engine_profile_step(bm_engine* e, int B, const int32_t* slots, const int32_t* tokens,
                                 int32_t* next_tokens, bm_kernel_profile* out, int max_out, int* n_out,
                                 void* stream) {
  if (!e || !out || !n_out || max_out < 1) return set_error(BM_ERR_INVALID_ARG, "bm_engine_profile_step: null argument");
  std::lock_guard<std::mutex> lk(e->mu);
  const bm_config& c = e->cfg;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bm_status st = prepare_step(e, B, slots, tokens, next_tokens, s, "bm_engine_profile_step");
  if (st != BM_OK) return st;
  double kv_pos = 0;
  for (int i = 0; i < B; ++i) kv_pos += e->slots.length(slots[i]) + 1;
  // prof_events[0] marks the start; kernel i (tags[i]) ends at prof_events[i + 1].
  if (e->prof_events.empty()) {
    cudaEvent_t ev;
    BM_CUDA(cudaEventCreate(&ev), "profile event");
    e->prof_events.push_back(ev);
  }
  ProfCtx ctx{e, s, {}};
  int n = 0;
  Marker mark{prof_mark, &ctx};
  BM_CUDA(cudaEventRecord(e->prof_events[0], s), "profile start event");
  BM_CUDA(enqueue_step(e, B, s, &n, mark), "bm_engine_profile_step launch");
  BM_CUDA(ctx.err, "profile events");
  BM_CUDA(cudaMemcpyAsync(next_tokens, e->d_next, sizeof(int32_t) * B, cudaMemcpyDefault, s), "next token copy");
  BM_CUDA(cudaStreamSynchronize(s), "profile synchronise");
  std::vector<int32_t> ulog(c.layers);
  BM_CUDA(cudaMemcpy(ulog.data(), e->d_u_log, sizeof(int32_t) * c.layers, cudaMemcpyDeviceToHost), "expert count read");
  std::vector<double> ms(KT_COUNT, 0.0), bytes(KT_COUNT, 0.0), flops(KT_COUNT, 0.0);
  std::vector<int> cnt(KT_COUNT, 0);
  int layer = 0;
  for (size_t i = 0; i < ctx.tags.size(); ++i) {
    const int tag = ctx.tags[i];
    float t = 0.f;
    BM_CUDA(cudaEventElapsedTime(&t, e->prof_events[i], e->prof_events[i + 1]), "event time");
    double b = 0, f = 0;
    const double U = ulog[layer < c.layers ? layer : c.layers - 1];
    algo_cost(c, e->qkv_rows, tag, B, U, kv_pos, &b, &f);
    ms[tag] += t;
    bytes[tag] += b;
    flops[tag] += f;
    cnt[tag] += 1;
    if (tag == KT_COMBINE) ++layer;
  }
  int k = 0;
  for (int tag = 0; tag < KT_COUNT && k < max_out; ++tag) {
    if (!cnt[tag]) continue;
    bm_kernel_profile& p = out[k++];
    std::memset(p.name, 0, sizeof(p.name));
    std::strncpy(p.name, kTagNames[tag], sizeof(p.name) - 1);
    p.launches = cnt[tag];
    p.ms = (float)ms[tag];
    p.bytes = bytes[tag];
    p.flops = flops[tag];
  }
  *n_out = k;
  e->slots.advance(slots, B);
  e->st.steps += 1;
  e->st.tokens += B;
  e->st.kernel_launches += n;
  return bm::ok();
}

// ------------------------------------------------------------------ ops

bm_status w4_gemm_batched(const uint8_t* W, const uint16_t* S, const uint16_t* X, uint16_t* Y, const uint16_t* R,
                          int M, int N, int K, int g, void* stream) {
  if (!W || !S || !X || !Y) return set_error(BM_ERR_INVALID_ARG, "w4_gemm_batched: null pointer");
  if (M < 1 || N < 1 || K < 32 || K % 32 || (g != 32 && g != 64 && g != 128) || K % g)
    return set_error(BM_ERR_INVALID_ARG, "w4_gemm_batched: need M, N >= 1, K % 32 == 0, g in {32, 64, 128}, K % g == 0");
  if (!simt_supports_k(K)) return set_error(BM_ERR_UNSUPPORTED, "w4_gemm_batched: no kernel shape for this K");
  bm_status st = ensure_attributes();
  if (st != BM_OK) return st;
  GemvArgs a{W, reinterpret_cast<const __half*>(S), reinterpret_cast<const bf16*>(X), K,
             reinterpret_cast<const bf16*>(R), N, reinterpret_cast<bf16*>(Y), N, M, N, K, g, 0, nullptr, 0.f};
  BM_CUDA(launch_w4_gemv(a, static_cast<cudaStream_t>(stream)), "w4_gemm_batched launch");
  return bm::ok();
}

bm_status bm_w4_repack_tc(const uint8_t* W, const uint16_t* S, int N, int K, int g, uint8_t* Wtc, uint16_t* Stc,
                          void* stream) {
  if (!W || !S || !Wtc || !Stc) return set_error(BM_ERR_INVALID_ARG, "bm_w4_repack_tc: null pointer");
  if (!tc_supports(N, K, g))
    return set_error(BM_ERR_INVALID_ARG, "bm_w4_repack_tc: need N % 128 == 0, K % 64 == 0, K <= 4096, "
                                         "g in {32, 64, 128}, K % g == 0");
  BM_CUDA(launch_repack_tc(W, reinterpret_cast<const __half*>(S), nullptr, nullptr, N, K, g, Wtc,
                           reinterpret_cast<__half*>(Stc), static_cast<cudaStream_t>(stream)),
          "bm_w4_repack_tc launch");
  return bm::ok();
}

bm_status bm_w4_repack_mma(const uint8_t* W, const uint16_t* S, int N, int K, int g, uint8_t* Wm, uint32_t* Sm,
                           void* stream) {
  if (!W || !S || !Wm || !Sm) return set_error(BM_ERR_INVALID_ARG, "bm_w4_repack_mma: null pointer");
  if (!mma_supports(N, K, g))
    return set_error(BM_ERR_INVALID_ARG, "bm_w4_repack_mma: need N % 32 == 0, K % 128 == 0, K <= 4096, "
                                         "g in {32, 64, 128}, K % g == 0");
  BM_CUDA(launch_repack_mma(W, reinterpret_cast<const __half*>(S), nullptr, nullptr, N, K, g, Wm, Sm,
                            static_cast<cudaStream_t>(stream)),
          "bm_w4_repack_mma launch");
  return bm::ok();
}

bm_status w4_gemm_batched_mma(const uint8_t* Wm, const uint32_t* Sm, const uint16_t* X, uint16_t* Y,
                              const uint16_t* R, int M, int N, int K, int g, void* stream) {
  if (!Wm || !Sm || !X || !Y) return set_error(BM_ERR_INVALID_ARG, "w4_gemm_batched_mma: null pointer");
  if (M < 1 || !mma_supports(N, K, g))
    return set_error(BM_ERR_INVALID_ARG, "w4_gemm_batched_mma: need M >= 1, N % 32 == 0, K % 128 == 0, "
                                         "K <= 4096, g in {32, 64, 128}, K % g == 0");
  bm_status st = ensure_attributes();
  if (st != BM_OK) return st;
  MmaArgs a{};
  a.W = Wm; a.S = Sm; a.rows = N; a.K = K; a.g = g;
  a.X = X; a.ldx = K; a.ntok = M; a.x_bf16 = 1;
  a.Res = reinterpret_cast<const bf16*>(R); a.ldr = N; a.Y = reinterpret_cast<bf16*>(Y); a.ldy = N;
  BM_CUDA(launch_w4_mma_dense(a, static_cast<cudaStream_t>(stream)), "w4_gemm_batched_mma launch");
  return bm::ok();
}

bm_status w4_gemm_prompt_tc(const uint8_t* Wm, const uint32_t* Sm, const uint16_t* X16, uint16_t* Y,
                            const uint16_t* R, int M, int N, int K, int g, void* stream) {
  if (!Wm || !Sm || !X16 || !Y) return set_error(BM_ERR_INVALID_ARG, "w4_gemm_prompt_tc: null pointer");
  if (M < 1 || !mma_supports(N, K, g) || !prefill_gemm_supports(N, K, g))
    return set_error(BM_ERR_INVALID_ARG, "w4_gemm_prompt_tc: need M >= 1, N % 128 == 0, K % 256 == 0, K <= 4096, "
                                         "g in {32, 64, 128}, K % g == 0");
  bm_status st = ensure_attributes();
  if (st != BM_OK) return st;
  PrefillGemmArgs a{};
  a.W = Wm; a.S = Sm; a.rows = N; a.K = K; a.g = g;
  a.X = X16; a.ldx = K; a.ntok = M;
  a.Res = reinterpret_cast<const bf16*>(R); a.ldr = N; a.Y = reinterpret_cast<bf16*>(Y); a.ldy = N;
  TmapBytes tm{};
  BM_CUDA(encode_rows_tmap(&tm, X16, M, K, K), "w4_gemm_prompt_tc tensor map");
  BM_CUDA(launch_prefill_dense(a, tm, static_cast<cudaStream_t>(stream)), "w4_gemm_prompt_tc launch");
  return bm::ok();
}

bm_status w4_gemm_batched_tc(const uint8_t* Wtc, const uint16_t* Stc, const uint16_t* X, uint16_t* Y,
                             const uint16_t* R, int M, int N, int K, int g, void* stream) {
  if (!Wtc || !Stc || !X || !Y) return set_error(BM_ERR_INVALID_ARG, "w4_gemm_batched_tc: null pointer");
  if (M < 1 || !tc_supports(N, K, g))
    return set_error(BM_ERR_INVALID_ARG, "w4_gemm_batched_tc: need M >= 1, N % 128 == 0, K % 64 == 0, "
                                         "K <= 4096, g in {32, 64, 128}, K % g == 0");
  bm_status st = ensure_attributes();
  if (st != BM_OK) return st;
  TcArgs a{};
  a.W = Wtc; a.S = reinterpret_cast<const __half*>(Stc); a.rows = N; a.K = K; a.g = g;
  a.X = reinterpret_cast<const bf16*>(X); a.ldx = K; a.ntok = M;
  a.Res = reinterpret_cast<const bf16*>(R); a.ldr = N; a.Y = reinterpret_cast<bf16*>(Y); a.ldy = N;
  a.ksplit = 1;
  BM_CUDA(launch_w4_tc_dense(a, static_cast<cudaStream_t>(stream)), "w4_gemm_batched_tc launch");
  return bm::ok();
}

size_t bm_moe_workspace_bytes(int B, int experts, int top_k, int hidden, int ffn) {
  if (B < 1 || experts < 1 || top_k < 1 || hidden < 1 || ffn < 1) return 0;
  return moe_scratch_bytes(B, experts, top_k, hidden, ffn);
}

bm_status moe_grouped_w4(const bm_moe_weights* w, const uint16_t* X, const uint16_t* Hres, uint16_t* Y,
                         int32_t* topk_ids, float* topk_w, int B, void* ws, size_t ws_bytes, void* stream) {
  if (!w || !X || !Y || !ws || !w->wr || !w->wg || !w->wg_s || !w->wu || !w->wu_s || !w->wd || !w->wd_s)
    return set_error(BM_ERR_INVALID_ARG, "moe_grouped_w4: null pointer");
  if (B < 1 || w->experts < 1 || w->experts > 256 || w->top_k < 1 || w->top_k > 16 || w->top_k > w->experts ||
      B * w->top_k > 1024)
    return set_error(BM_ERR_INVALID_ARG, "moe_grouped_w4: need 1 <= top_k <= min(16, experts), experts <= 256, "
                                         "B * top_k <= 1024");
  if ((w->group != 32 && w->group != 64 && w->group != 128) || w->hidden % w->group || w->ffn % w->group ||
      w->hidden % 32 || w->ffn % 32)
    return set_error(BM_ERR_INVALID_ARG, "moe_grouped_w4: bad group or sizes");
  if (!simt_supports_k(w->hidden) || !simt_supports_k(w->ffn))
    return set_error(BM_ERR_UNSUPPORTED, "moe_grouped_w4: no kernel shape for these sizes");
  const size_t need = moe_scratch_bytes(B, w->experts, w->top_k, w->hidden, w->ffn);
  if (ws_bytes < need)
    return set_error(BM_ERR_INVALID_ARG, "moe_grouped_w4: workspace of " + std::to_string(ws_bytes) +
                                             " bytes, need " + std::to_string(need));
  bm_status st = ensure_attributes();
  if (st != BM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MoeBufs b = moe_carve(ws, B, w->experts, w->top_k, w->hidden, w->ffn);
  MoeArgs a{B, w->experts, w->top_k, w->hidden, w->ffn, w->group, w->renorm_topk,
            w->wr, w->wg, reinterpret_cast<const __half*>(w->wg_s), w->wu,
            reinterpret_cast<const __half*>(w->wu_s), w->wd, reinterpret_cast<const __half*>(w->wd_s),
            reinterpret_cast<const bf16*>(X), 0, nullptr, 0.f, reinterpret_cast<const bf16*>(Hres),
            reinterpret_cast<bf16*>(Y)};
  BM_CUDA(launch_moe(a, b, s, nullptr), "moe_grouped_w4 launch");
  if (topk_ids)
    BM_CUDA(cudaMemcpyAsync(topk_ids, b.topk_ids, sizeof(int32_t) * B * w->top_k, cudaMemcpyDeviceToDevice, s),
            "topk ids copy");
  if (topk_w)
    BM_CUDA(cudaMemcpyAsync(topk_w, b.topk_w, sizeof(float) * B * w->top_k, cudaMemcpyDeviceToDevice, s),
            "topk weights copy");
  return bm::ok();
}

bm_status bm_engine_moe(bm_engine* e, int layer, const uint16_t* h, uint16_t* y, int32_t* topk_ids, float* topk_w,
                        int B, void* stream) {
  if (!e || !h || !y) return set_error(BM_ERR_INVALID_ARG, "bm_engine_moe: null argument");
  std::lock_guard<std::mutex> lk(e->mu);
  const bm_config& c = e->cfg;
  if (layer < 0 || layer >= c.layers) return set_error(BM_ERR_INVALID_ARG, "bm_engine_moe: layer out of range");
  if (B < 1 || B > c.max_streams) return set_error(BM_ERR_INVALID_ARG, "bm_engine_moe: B out of range");
  if (!e->L[layer].set) return set_error(BM_ERR_NOT_READY, "bm_engine_moe: layer weights not set");
  if (e->family != BM_POLICY_MMA)
    return set_error(BM_ERR_UNSUPPORTED, "bm_engine_moe: needs an engine on the warp-MMA kernel family");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const LayerW& w = e->L[layer];
  const int H = c.hidden, F = c.ffn, g = c.group;
  auto u32 = [](const __half* p) { return reinterpret_cast<const uint32_t*>(p); };
  const bf16* hin = reinterpret_cast<const bf16*>(h);
  MoeArgs ma{B, c.experts, c.top_k, H, F, g, c.renorm_topk,
             w.wr, w.wg, w.wg_s, w.wu, w.wu_s, w.wd, w.wd_s,
             hin, 1, w.has_ffn_norm ? w.ffn_norm_buf : nullptr, c.rms_eps, hin, reinterpret_cast<bf16*>(y),
             e->d_u_log + layer, 1};
  const MoeBufs mb = moe_carve(e->moe_ws, B, c.experts, c.top_k, H, F);
  BM_CUDA(launch_moe_route_fused(ma, mb, e->route_cnt, e->route_cnt + c.max_streams, s, Marker(), false),
          "bm_engine_moe routing");
  MmaArgs m3{};
  m3.W = w.wg; m3.S = u32(w.wg_s); m3.rows = 2 * F; m3.K = H; m3.g = g; m3.X = mb.xn; m3.ldx = H;
  m3.pair_token = mb.pair_token; m3.n_jobs = mb.n_jobs; m3.jobs = mb.jobs;
  m3.max_jobs = moe_max_jobs(B, c.experts, c.top_k);
  m3.w_expert_stride = (size_t)2 * F * H / 2; m3.s_expert_stride = (size_t)F * (H / g);
  m3.act16 = reinterpret_cast<__half*>(mb.act); m3.F = F; m3.err = e->d_err;
  m3.drop_item1 = e->test_drop_item + 1;
  BM_CUDA(launch_w4_mma_gateup(m3, s), "bm_engine_moe gate/up");
  MmaArgs m4{};
  m4.W = w.wd; m4.S = u32(w.wd_s); m4.rows = H; m4.K = F; m4.g = g; m4.X = mb.act; m4.ldx = F;
  m4.pair_token = mb.pair_token; m4.n_jobs = mb.n_jobs; m4.jobs = mb.jobs; m4.max_jobs = m3.max_jobs;
  m4.w_expert_stride = (size_t)H * F / 2; m4.s_expert_stride = (size_t)H * (F / g) / 2;
  m4.out = mb.out; m4.H = H; m4.err = e->d_err;
  BM_CUDA(launch_w4_mma_down(m4, s), "bm_engine_moe down");
  BM_CUDA(launch_moe_combine_norm(ma, mb, nullptr, e->xn, 1, s, Marker(), false), "bm_engine_moe combine");
  if (topk_ids)
    BM_CUDA(cudaMemcpyAsync(topk_ids, mb.topk_ids, sizeof(int32_t) * B * c.top_k, cudaMemcpyDefault, s),
            "bm_engine_moe ids copy");
  if (topk_w)
    BM_CUDA(cudaMemcpyAsync(topk_w, mb.topk_w, sizeof(float) * B * c.top_k, cudaMemcpyDefault, s),
            "bm_engine_moe weights copy");
  e->st.kernel_launches += 4;
  return bm::ok();
}

bm_status bm_engine_attention(bm_engine* e, int layer, const int32_t* slots, const uint16_t* qkv, uint16_t* out,
                              int B, void* stream) {
  if (!e || !slots || !qkv || !out) return set_error(BM_ERR_INVALID_ARG, "bm_engine_attention: null argument");
  std::lock_guard<std::mutex> lk(e->mu);
  const bm_config& c = e->cfg;
  if (layer < 0 || layer >= c.layers) return set_error(BM_ERR_INVALID_ARG, "bm_engine_attention: layer out of range");
  if (e->family != BM_POLICY_MMA || !attention_fused_supports(e->arena, c.q_heads))
    return set_error(BM_ERR_UNSUPPORTED, "bm_engine_attention: needs the warp-MMA kernel family and fused attention");
  std::string err;
  bm_status st = e->slots.check_batch(slots, B, &err);
  if (st != BM_OK) return set_error(st, "bm_engine_attention: " + err);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = stage_aux_slots(e, slots, B, s)) != BM_OK) return st;
  AttnFusedArgs fa{e->arena, layer, e->d_slots_aux, reinterpret_cast<const bf16*>(qkv), e->qkv_rows, c.q_heads,
                   e->d_rope, reinterpret_cast<__half*>(out), e->attn_part, (c.ctx_cap + kAttnChunk - 1) / kAttnChunk,
                   e->attn_cnt, B, chk_of(e), 0};
  BM_CUDA(launch_attention_fused(fa, s, false), "bm_engine_attention launch");
  e->st.kernel_launches += 1;
  return bm::ok();
}

bm_status bm_engine_read_hidden(bm_engine* e, int B, uint16_t* out, void* stream) {
  if (!e || !out) return set_error(BM_ERR_INVALID_ARG, "bm_engine_read_hidden: null argument");
  if (B < 1 || B > e->cfg.max_streams) return set_error(BM_ERR_INVALID_ARG, "bm_engine_read_hidden: B out of range");
  BM_CUDA(cudaMemcpyAsync(out, e->x, sizeof(uint16_t) * B * (size_t)e->cfg.hidden, cudaMemcpyDefault,
                          static_cast<cudaStream_t>(stream)),
          "bm_engine_read_hidden copy");
  return bm::ok();
}

bm_status bm_engine_test_drop_expert_item(bm_engine* e, int item) {
  if (!e) return set_error(BM_ERR_INVALID_ARG, "bm_engine_test_drop_expert_item: null engine");
  std::lock_guard<std::mutex> lk(e->mu);
  e->test_drop_item = item < 0 ? -1 : item;
  return bm::ok();
}

bm_status bm_engine_set_persistent_step(bm_engine* e, int enable) {
  if (!e) return set_error(BM_ERR_INVALID_ARG, "bm_engine_set_persistent_step: null engine");
  std::lock_guard<std::mutex> lk(e->mu);
  const bm_config& c = e->cfg;
  if (!c.persistent_step)
    return set_error(BM_ERR_UNSUPPORTED, "bm_engine_set_persistent_step: the engine was created without persistent_step");
  const int rows = enable ? std::min(std::min(c.max_streams, kPMaxRows), 64 / c.top_k) : 0;
  if (rows != e->persist_rows) {
    e->persist_rows = rows;
    for (auto it = e->graphs.begin(); it != e->graphs.end();) {   // decode graphs of the other path
      if (it->first > 0) {
        cudaGraphExecDestroy(it->second);
        e->graph_kernels.erase(it->first);
        it = e->graphs.erase(it);
      } else {
        ++it;
      }
    }
  }
  return bm::ok();
}

bm_status bm_engine_test_drop_persist_unit(bm_engine* e, int unit) {
  if (!e) return set_error(BM_ERR_INVALID_ARG, "bm_engine_test_drop_persist_unit: null engine");
  std::lock_guard<std::mutex> lk(e->mu);
  e->test_drop_unit = unit < 0 ? -1 : unit;
  // the captured decode graphs hold the old setting: capture again
  for (auto it = e->graphs.begin(); it != e->graphs.end();) {
    if (it->first > 0) {
      cudaGraphExecDestroy(it->second);
      e->graph_kernels.erase(it->first);
      it = e->graphs.erase(it);
    } else {
      ++it;
    }
  }
  return bm::ok();
}

bm_status bm_w4_quantize(const float* W, int N, int K, int g, uint8_t* packed, uint16_t* scales, void* stream) {
  if (!W || !packed || !scales) return set_error(BM_ERR_INVALID_ARG, "bm_w4_quantize: null pointer");
  if (N < 1 || K < 2 || (g != 32 && g != 64 && g != 128) || K % g)
    return set_error(BM_ERR_INVALID_ARG, "bm_w4_quantize: need N >= 1, g in {32, 64, 128}, K % g == 0");
  BM_CUDA(launch_quantize(W, N, K, g, packed, reinterpret_cast<__half*>(scales), static_cast<cudaStream_t>(stream)),
          "bm_w4_quantize launch");
  return bm::ok();
}

}  // extern "C"
