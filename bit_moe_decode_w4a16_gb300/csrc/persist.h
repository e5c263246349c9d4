// Host interface of the persistent small-batch decode step (persist.cu).
#pragma once

#include "kernels.cuh"

namespace bm {

constexpr int kPMaxRows = 8;   // rows of a persistent step (and rows x top_k <= 64)

// One layer's weights in the warp-MMA layout (device pointers).
struct PersistLayer {
  const uint8_t* wqkv; const uint32_t* sqkv;
  const uint8_t* wo; const uint32_t* so;
  const float* wr;
  const uint8_t* wg; const uint32_t* sg;   // gate/up bank, rows interleaved by 8
  const uint8_t* wd; const uint32_t* sd;
  const bf16* attn_nw;                     // RMSNorm weights or null (ones)
  const bf16* ffn_nw;
};

// Shared-memory plan of the kernel (bytes) and its grid.
struct PersistGeo {
  uint32_t ring_bytes;  // the weight ring
  uint32_t ring_off, red_off, uni_off, uni_bytes;
  int grid;             // CTAs: one per SM
};

struct PersistArgs {
  const PersistLayer* L;   // [layers], device
  int layers, B;
  int H, qd, qkv_rows, F, E, k;
  float eps;
  const bf16* final_nw;
  bf16* x;                 // residual stream [B][H]: the embedding rows in, each layer's output out
  const __half* xn16;      // RMSNorm of the embedding rows (layer 0 input), fp16 [B][H]
  bf16* xn_out;            // final RMSNorm rows for the output projection, bf16 [B][H]
  bf16* qkv;               // [B][qkv_rows]
  __half* attn;            // [B][qd]
  bf16* h;                 // [B][H]
  MoeArgs moe;             // routing arguments (x = h, the ffn norm fused); wr / norm_w set per layer
  MoeBufs mb;              // routing and expert scratch of B rows
  __half* mb_act16;        // mb.act as fp16
  AttnFusedArgs at;        // attention arguments; layer set per layer
  size_t wg_stride, wd_stride;   // bytes of one expert's matrix
  size_t sg_stride, sd_stride;   // 32-bit scale words of one expert's matrix
  int32_t* u_log;          // [layers] active experts, or null
  unsigned int* bar;       // grid barrier counter, zero at launch
  int* err;                // device error flag (code 6: a bounded wait gave up)
  int drop_unit1;          // failure-detection tests only: 1 + the index of a weight item (tile job) the
                           // producer does not issue (its consumers' bounded wait runs out); 0 = none
  PersistGeo geo;
};

// Shared-memory plan for a model geometry and at most max_rows rows; false
// (with a reason) if the persistent step cannot run it.
bool persist_plan(int H, int qd, int qkv_rows, int F, int E, int k, int g, int d, int cap, int max_rows,
                  PersistGeo* geo, const char** why);
// Kernel attributes and the grid (one CTA per SM, all resident).
cudaError_t persist_init(const PersistGeo& geo, int d, int g, int* grid);
// One cooperative launch.
cudaError_t launch_persist_step(const PersistArgs& a, int d, int g, cudaStream_t st);

}  // namespace bm
