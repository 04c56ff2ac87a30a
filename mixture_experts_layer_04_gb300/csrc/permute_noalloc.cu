// moe_permute_noalloc: the dispatch permutation for callers that cannot allocate
// device memory.
//
// Some callers of this library cannot call cudaMalloc, or hand out any workspace:
// an inference server that carves every device buffer out of pools it sizes once at
// start-up and forbids allocation afterwards, or a plug-in host that passes only its
// input and output tensors to the plug-in.  moe_permute needs a little scratch (the
// per-block expert counts of the counting sort), which it normally takes from the
// caller's workspace.  This variant takes it instead from a fixed array compiled into
// the library (below), so the caller only passes inputs and outputs.
//
// The array lives in device memory of every GPU that loads the library, from load
// time until the process exits.  It is shared by every call on that GPU and keeps what
// the last call left in it; calls that may overlap on the GPU (on different streams,
// or from several host threads) race on it and must be serialised by the caller.  No
// word of it needs to start at zero: the permutation writes every scratch word it
// reads earlier in the same call.
#include <mutex>

#include "../../include/moe.h"
#include "kernels.h"

namespace moe {
namespace {

// The scratch of the counting sort: one int32 count per (block of 256 tokens, expert).
static __device__ __align__(256) int32_t g_permute_scratch[MOE_PERMUTE_NOALLOC_MAX_WORDS];

constexpr int kMaxDevices = 64;

int32_t* g_noalloc_scratch[kMaxDevices];  // device address of g_permute_scratch, per device
std::mutex g_noalloc_mu;

// One-time set-up per device, done by the first call on that device with the device
// current: the symbol above is a host-side stand-in, so its device address has to be
// looked up with cudaGetSymbolAddress before a kernel may be given it.  Which devices are
// supported is decided by the library's common device check.
moe_status_t noalloc_setup(int32_t** scratch) {
  const moe_status_t sd = check_current_device();
  if (sd != MOE_OK) return sd;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_scratch[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || p == nullptr)
      return MOE_ERR_CUDA;
    g_noalloc_scratch[dev] = static_cast<int32_t*>(p);
  }
  *scratch = g_noalloc_scratch[dev];
  return MOE_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_permute_noalloc(const moe_config_t* cfg, const void* x,
                                            const int32_t* topk_ids, int32_t* counts,
                                            int32_t* offsets, int32_t* perm, int32_t* inv,
                                            void* x_perm, moe_stream_t stream) {
  using namespace moe;
  const moe_status_t sf = fault_point("moe_permute_noalloc");
  if (sf != MOE_OK) return sf;
  size_t ignored = 0;
  const moe_status_t st = moe_workspace_size(cfg, &ignored);  // validates cfg on the host
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (x == nullptr || topk_ids == nullptr || counts == nullptr || offsets == nullptr ||
      perm == nullptr || inv == nullptr || x_perm == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(topk_ids) || !aligned16(counts) || !aligned16(offsets) ||
      !aligned16(perm) || !aligned16(inv) || !aligned16(x_perm))
    return MOE_ERR_MISALIGNED;
  if (permute_ws_words(cfg->T, cfg->E) > static_cast<size_t>(MOE_PERMUTE_NOALLOC_MAX_WORDS))
    return MOE_ERR_WORKSPACE;  // more scratch than the fixed array holds
  int32_t* scratch = nullptr;
  const moe_status_t su = noalloc_setup(&scratch);
  if (su != MOE_OK) return su;
  const cudaError_t e =
      launch_permute(cfg->dtype, x, topk_ids, cfg->T, cfg->H, cfg->E, cfg->K, counts, offsets,
                     perm, inv, x_perm, scratch, nullptr, nullptr, 0, nullptr, nullptr,
                     static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
