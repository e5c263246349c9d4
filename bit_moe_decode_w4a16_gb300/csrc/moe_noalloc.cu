// The grouped expert op for callers that cannot allocate device memory.
//
// moe_grouped_w4 needs a caller-supplied workspace.  Some callers have no way
// to provide one: a plugin running inside a host engine that owns the whole
// device memory pool and forbids cudaMalloc (an extra allocation would fail or
// break the pool's accounting), or a caller on a latency-critical path where
// cudaMalloc / cudaFree, which can synchronise the device, are not allowed.
// This variant keeps its workspace in a fixed array compiled into the
// library, so it allocates nothing when it runs.
#include <map>
#include <mutex>
#include <string>

#include "errors.h"
#include "kernels.cuh"

namespace bm {

cudaError_t init_moe_attributes();

// The workspace: one array per device that loads this library, reserved for
// the life of the process.  Every call on a device reuses the same bytes.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;   // 4 MiB
static __device__ __align__(256) unsigned char g_moe_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_mu;
std::map<int, void*> g_scratch_addr;   // device -> device address of the array

// Once per device, with that device current: look up the array's device
// address (host code cannot use the symbol itself as a device pointer) and
// set the expert kernels' shared-memory limits.
bm_status scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(BM_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  std::lock_guard<std::mutex> lk(g_mu);
  auto it = g_scratch_addr.find(dev);
  if (it != g_scratch_addr.end()) {
    *out = it->second;
    return BM_OK;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_moe_noalloc_scratch);
  if (e != cudaSuccess || !p)
    return set_error(BM_ERR_CUDA, std::string("cudaGetSymbolAddress of the static workspace: ") +
                                      cudaGetErrorString(e));
  e = init_moe_attributes();
  if (e != cudaSuccess)
    return set_error(BM_ERR_CUDA, std::string("expert kernel attributes: ") + cudaGetErrorString(e));
  g_scratch_addr[dev] = p;
  *out = p;
  return BM_OK;
}

}  // namespace
}  // namespace bm

extern "C" {

size_t bm_moe_noalloc_max_bytes(void) { return bm::kNoAllocScratchBytes; }

bm_status moe_grouped_w4_noalloc(const bm_moe_weights* w, const uint16_t* X, const uint16_t* Hres, uint16_t* Y,
                                 int32_t* topk_ids, float* topk_w, int B, void* stream) {
  using namespace bm;
  if (!w || !X || !Y || !w->wr || !w->wg || !w->wg_s || !w->wu || !w->wu_s || !w->wd || !w->wd_s)
    return set_error(BM_ERR_INVALID_ARG, "moe_grouped_w4_noalloc: null pointer");
  if (B < 1 || w->experts < 1 || w->experts > 256 || w->top_k < 1 || w->top_k > 16 || w->top_k > w->experts ||
      B * w->top_k > 1024)
    return set_error(BM_ERR_INVALID_ARG, "moe_grouped_w4_noalloc: need 1 <= top_k <= min(16, experts), "
                                         "experts <= 256, B * top_k <= 1024");
  if ((w->group != 32 && w->group != 64 && w->group != 128) || w->hidden % w->group || w->ffn % w->group ||
      w->hidden % 32 || w->ffn % 32)
    return set_error(BM_ERR_INVALID_ARG, "moe_grouped_w4_noalloc: bad group or sizes");
  if (!simt_supports_k(w->hidden) || !simt_supports_k(w->ffn))
    return set_error(BM_ERR_UNSUPPORTED, "moe_grouped_w4_noalloc: no kernel shape for these sizes");
  const size_t need = moe_scratch_bytes(B, w->experts, w->top_k, w->hidden, w->ffn);
  if (need > kNoAllocScratchBytes)
    return set_error(BM_ERR_INVALID_ARG, "moe_grouped_w4_noalloc: these sizes need " + std::to_string(need) +
                                             " bytes of workspace, more than the built-in " +
                                             std::to_string(kNoAllocScratchBytes) +
                                             "; use moe_grouped_w4 with a caller-owned workspace");
  void* ws = nullptr;
  bm_status st = scratch_for_current_device(&ws);
  if (st != BM_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Every workspace element the kernels read is first written by the same
  // call, so nothing has to be cleared between calls.
  MoeBufs b = moe_carve(ws, B, w->experts, w->top_k, w->hidden, w->ffn);
  MoeArgs a{B, w->experts, w->top_k, w->hidden, w->ffn, w->group, w->renorm_topk,
            w->wr, w->wg, reinterpret_cast<const __half*>(w->wg_s), w->wu,
            reinterpret_cast<const __half*>(w->wu_s), w->wd, reinterpret_cast<const __half*>(w->wd_s),
            reinterpret_cast<const bf16*>(X), 0, nullptr, 0.f, reinterpret_cast<const bf16*>(Hres),
            reinterpret_cast<bf16*>(Y), nullptr};
  cudaError_t e = launch_moe(a, b, s, nullptr);
  if (e == cudaSuccess && topk_ids)
    e = cudaMemcpyAsync(topk_ids, b.topk_ids, sizeof(int32_t) * B * w->top_k, cudaMemcpyDeviceToDevice, s);
  if (e == cudaSuccess && topk_w)
    e = cudaMemcpyAsync(topk_w, b.topk_w, sizeof(float) * B * w->top_k, cudaMemcpyDeviceToDevice, s);
  if (e != cudaSuccess) return set_error(BM_ERR_CUDA, std::string("moe_grouped_w4_noalloc: ") + cudaGetErrorString(e));
  return ok();
}

}  // extern "C"
