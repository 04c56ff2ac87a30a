// C ABI of the MoE layer (include/moe.h): argument validation, the workspace plan and
// the order of launches.  Every check happens on the host before the first launch; the
// library never allocates, frees or synchronises on the compute paths.
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

// Device error word (bits MOE_DEVERR_*), one per device that loads the library.
__device__ unsigned g_error_word;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  bool supported = false;
  int num_sms = 0;
  unsigned* err = nullptr;
  // Prefill layers with a shared expert run it on a second stream, concurrently with the
  // dispatch permutation (see side_stream()); created on first use, kept until exit.
  bool side_tried = false;
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  std::mutex side_mu;  // one layer at a time enqueues work on the side stream
};

DeviceInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

// Per-device setup on first use: checks for an sm_103 device and looks up the device
// address of the error word (the host-side symbol is not a device address).
const DeviceInfo* device_info() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return nullptr;
    d.supported = (prop.major == 10 && prop.minor == 3);
    d.num_sms = prop.multiProcessorCount;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    d.err = static_cast<unsigned*>(p);
    d.ready = true;
  }
  return &d;
}

// The device's side stream (lowest priority, not synchronising with the legacy stream)
// and its fork/join events, created by the first call that asks for them, or null if they
// cannot be created.  Not called while `s` is being captured into a graph.
DeviceInfo* side_stream(const DeviceInfo* dc) {
  DeviceInfo* d = const_cast<DeviceInfo*>(dc);
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (!d->side_tried) {
    d->side_tried = true;
    int lo = 0, hi = 0;
    cudaStream_t st = nullptr;
    cudaEvent_t f = nullptr, j = nullptr;
    if (cudaDeviceGetStreamPriorityRange(&lo, &hi) == cudaSuccess &&
        cudaStreamCreateWithPriority(&st, cudaStreamNonBlocking, lo) == cudaSuccess &&
        cudaEventCreateWithFlags(&f, cudaEventDisableTiming) == cudaSuccess &&
        cudaEventCreateWithFlags(&j, cudaEventDisableTiming) == cudaSuccess) {
      d->side = st;
      d->fork = f;
      d->join = j;
    } else {
      cudaGetLastError();  // leave no sticky error behind; the layer then runs in order
    }
  }
  return d->side != nullptr ? d : nullptr;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t check_config(const moe_config_t* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if ((c->flags & ~static_cast<uint32_t>(MOE_FLAG_FUSED_COMBINE | MOE_FLAG_CAPACITY |
                                         MOE_FLAG_FP8)) != 0u)
    return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->H <= 0 || c->E <= 0 || c->K <= 0 || c->I <= 0 || c->I_shared < 0)
    return MOE_ERR_INVALID_ARG;
  if (c->K > c->E || c->K > 16 || c->E > 1024) return MOE_ERR_INVALID_ARG;
  if (c->H % 64 != 0 || c->I % 64 != 0 || c->I_shared % 64 != 0) return MOE_ERR_INVALID_ARG;
  if (c->H > 65536 || c->I > 65536 || c->I_shared > 65536) return MOE_ERR_INVALID_ARG;
  if (!(c->gate_threshold >= 0.0f && c->gate_threshold < 1.0f)) return MOE_ERR_INVALID_ARG;
  if (static_cast<long long>(c->T) * c->K >= (1ll << 31)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

bool use_tc_router(const moe_config_t* c) {
  return c->dtype == MOE_BF16 && c->T >= 256 && c->E >= 32 && c->E % 16 == 0;
}

// Workspace plan: every region 256-byte aligned.
struct Plan {
  size_t logits, partial, ids, w, counts, offsets, perm, inv, perm_ws, table, num_mt, x_perm, h,
      out_perm, row_w, y32, x_codes, x_scales, xs_perm, h_codes, h_scales,
      shared_h, shared_out, tile_counter, total;
};

inline size_t up256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

Plan make_plan(const moe_config_t* c) {
  const size_t T = c->T, H = c->H, E = c->E, K = c->K, I = c->I, Is = c->I_shared;
  const size_t ab = act_bytes(c->dtype);
  const int bm = c->dtype == MOE_BF16 ? kTcBM : kF32TileRows;
  Plan p;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o += up256(bytes);
    return at;
  };
  p.logits = take(T * E * 4);
  // H-slice partial logits of the CUDA-core router (when neither the tensor-core nor the
  // shared-memory router serves this shape)
  const bool part_router = !use_tc_router(c) && !router_uses_wsmem(c->dtype, c->T, c->H, c->E);
  p.partial = take(part_router ? static_cast<size_t>(router_slices(c->T, c->H, c->E, c->dtype)) *
                                     T * E * 4
                               : 0);
  p.ids = take(T * K * 4);
  p.w = take(T * K * 4);
  p.counts = take(E * 4);
  p.offsets = take((E + 1) * 4);
  p.perm = take(T * K * 4);
  p.inv = take(T * K * 4);
  p.perm_ws = take(permute_ws_words(c->T, c->E) * 4);
  p.table = take(static_cast<size_t>(max_mtiles(c->T, c->K, c->E, bm)) * sizeof(int4));
  p.num_mt = take(16);
  p.x_perm = take(T * K * H * ab);
  p.h = take(T * K * I * ab);
  p.out_perm = take(T * K * H * 4);
  p.shared_h = take(T * Is * ab);
  p.shared_out = take(Is > 0 ? T * H * 4 : 0);
  const bool fused = (c->flags & MOE_FLAG_FUSED_COMBINE) != 0u;
  p.row_w = take(fused ? T * K * 4 : 0);
  p.y32 = take(fused ? T * H * 4 : 0);
  // FP8 experts (moe_layer_forward_fp8): x's codes and scales, the scales in row order, and
  // h's codes and scales (the permuted codes reuse x_perm)
  const bool fp8 = (c->flags & MOE_FLAG_FP8) != 0u;
  p.x_codes = take(fp8 ? T * H : 0);
  p.x_scales = take(fp8 ? T * 4 : 0);
  p.xs_perm = take(fp8 ? T * K * 4 : 0);
  p.h_codes = take(fp8 ? T * K * I : 0);
  p.h_scales = take(fp8 ? T * K * 4 : 0);
  p.tile_counter = take(4);
  p.total = o;
  return p;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                      \
  do {                                     \
    moe_status_t st__ = (expr);            \
    if (st__ != MOE_OK) return st__;       \
  } while (0)

#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))

moe_status_t check_device(const DeviceInfo** out) {
  const DeviceInfo* d = device_info();
  if (d == nullptr) return MOE_ERR_CUDA;
  if (!d->supported) return MOE_ERR_UNSUPPORTED;
  *out = d;
  return MOE_OK;
}


// Routing launches (shared by moe_route and moe_layer_forward).
// Routing launches (shared by moe_route and moe_layer_forward).  `partial` is scratch
// for the CUDA-core router's H-slice partial sums (at least slices*T*E floats), or null
// to use one slice written straight into `logits`.  With `defer_topk` (layer forward,
// small T) the router only writes the partials and *deferred_slices tells the caller to
// take the top-k inside the fused small permutation.
moe_status_t run_route(const moe_config_t* c, const DeviceInfo* d, const void* x,
                       const void* w_router, const float* bias, float* logits, int32_t* ids,
                       float* w, float* partial, bool defer_topk, int* deferred_slices,
                       cudaStream_t s) {
  if (deferred_slices != nullptr) *deferred_slices = 0;
  if (c->T == 0) return MOE_OK;
  if (x == nullptr) {
    return cuda_status(launch_topk(logits, 1, nullptr, nullptr, ids, w, c->T, c->E, c->K,
                                   c->gate_threshold, s));
  }
  if (route_cluster_ok(c->dtype, c->T, c->H, c->E, c->K))  // decode-sized: one cluster
    return cuda_status(launch_route_cluster(x, w_router, bias, logits, ids, w, c->gate_threshold,
                                            c->T, c->H, c->E, c->K, nullptr, nullptr, nullptr,
                                            nullptr, nullptr, nullptr, d->err, s));
  if (use_tc_router(c)) {
    GroupedGemm g{};
    g.mode = kPlain;
    g.dtype = kBF16;
    g.A = x;
    g.rows_alloc = c->T;
    g.Kd = c->H;
    g.B = w_router;
    g.G = 1;
    g.Nb = c->E;
    g.N_out = c->E;
    g.C = logits;
    g.col_bias = bias;
    if (c->E <= 256) {
      // one tile spans all experts: the top-k, softmax and gate drop run in its epilogue
      g.mode = kTopK;
      g.topk_k = c->K;
      g.topk_theta = c->gate_threshold;
      g.topk_ids = ids;
      g.topk_w = w;
      return cuda_status(launch_grouped_gemm_tc(g, d->err, d->num_sms, s));
    }
    MOE_CUDA(launch_grouped_gemm_tc(g, d->err, d->num_sms, s));
    return cuda_status(
        launch_topk(logits, 1, nullptr, nullptr, ids, w, c->T, c->E, c->K, c->gate_threshold, s));
  }
  if (router_uses_wsmem(c->dtype, c->T, c->H, c->E))
    return cuda_status(launch_router_wsmem(c->dtype, x, w_router, bias, logits, ids, w, c->T, c->H,
                                           c->E, c->K, c->gate_threshold, d->err, s));
  const int S = partial != nullptr ? router_slices(c->T, c->H, c->E, c->dtype) : 1;
  float* part = partial != nullptr ? partial : logits;
  MOE_CUDA(launch_router_partial(c->dtype, x, w_router, part, S, c->T, c->H, c->E, s));
  if (defer_topk && topk_permute_fusable(c->T, c->E, c->K)) {
    *deferred_slices = S;
    return MOE_OK;
  }
  return cuda_status(launch_topk(part, S, bias, logits, ids, w, c->T, c->E, c->K,
                                 c->gate_threshold, s));
}

// Grouped-GEMM launch descriptions of the two expert GEMMs.  Groups come from `offsets`
// (bf16 engine) or from the m-tile table (float32 engine); with neither, A is one
// dense group of rows_alloc rows (the shared expert).
struct Groups {
  const int32_t* offsets;
  const int4* table;
  const int32_t* num_mt;
  int max_mt;
  int G;
};

// Decode-sized batches: with at most kSwapMaxTokens tokens no group can have more rows
// than that, so the tensor-core GEMMs put the weights on the 128-row side of the MMA.
constexpr int kSwapMaxTokens = 128;
// Batches routed by one cluster launch with at most this many tokens gather token rows in
// the gate/up GEMM instead of copying them.
constexpr int kGatherMaxTokens = 16;
constexpr int kPairMinRowsPerGroup = 768;
// batches from this many tokens run the shared expert on the side stream
constexpr int kSharedSideMinTokens = 1024;
constexpr int kPairMinRowsSwiGLU = 384;
constexpr int kPairWideDim = 4096;

// The routed gate/up GEMM of a prefill-sized bf16 batch runs on CTA pairs in the normal
// operand order, where the pairs draw their tiles from a counter in the workspace (the
// SwiGLU launch measured faster so on GB300: Qwen3-, Mixtral- and DeepSeek-shaped gate/up
// 1-4%, FP8 Mixtral-shaped 22%; the down projections and single-CTA launches were not).
// The layer's permutation kernel zeroes the counter; a standalone call, a memset.
bool dynamic_tiles(const moe_config_t* c) {
  return c->dtype == MOE_BF16 && c->T > kSwapMaxTokens;
}

// The tile counter of a standalone gate/up call (zeroed first), or null.
int* standalone_counter(const moe_config_t* c, void* ws, const Plan& p, cudaStream_t s,
                        cudaError_t* e) {
  *e = cudaSuccess;
  if (!dynamic_tiles(c)) return nullptr;
  int* ctr = at<int>(ws, p.tile_counter);
  *e = cudaMemsetAsync(ctr, 0, sizeof(int), s);
  return ctr;
}

// CTA pairs (256-row tiles, 2/3 of the shared-memory traffic per MMA) pay for the padding
// of each group's last tile when groups are large (>= 768 rows on average), or half that
// size with a long reduction or a wide output to amortise it; otherwise single CTAs with
// 128-row tiles (measured on GB300 with the workloads' groups).  The gate/up GEMM (bf16
// output, a light epilogue) gains from pairs from 384 rows per group; a short-reduction down
// projection with its fp32 output does not (Qwen3-shaped layer on GB300: gate/up on pairs
// 0.650 -> 0.637 ms per layer, down on pairs +70 us).
bool use_pairs(const GroupedGemm& g) {
  const long long rows_per_group = g.rows_alloc / (g.G > 0 ? g.G : 1);
  const bool big = rows_per_group >= kPairMinRowsPerGroup ||
                   (rows_per_group >= kPairMinRowsPerGroup / 3 &&
                    (g.Kd >= kPairWideDim || g.N_out >= kPairWideDim)) ||
                   (g.mode == kSwiGLU && rows_per_group >= kPairMinRowsSwiGLU);
  return g.swap_tokens == 0 && big && g.gather_rows == nullptr;
}

moe_status_t launch_gemm(const moe_config_t* c, const DeviceInfo* d, const GroupedGemm& g0,
                         cudaStream_t s) {
  if (c->dtype == MOE_BF16) {
    GroupedGemm g = g0;
    g.swap_tokens = c->T <= kSwapMaxTokens ? c->T : 0;
    g.pair = use_pairs(g) ? 1 : 0;
    return cuda_status(launch_grouped_gemm_tc(g, d->err, d->num_sms, s));
  }
  return cuda_status(launch_grouped_gemm_tf32(g0, d->err, d->num_sms, s));
}

// h = silu(A W_g^T) * (A W_u^T) per group.  With `gather_rows`, row r of the groups is
// row gather_rows[r] of A (A then has c->T rows).
moe_status_t run_gate_up(const moe_config_t* c, const DeviceInfo* d, const void* A,
                         int rows_alloc, const void* w_gate_up, int I, void* h, const Groups& gr,
                         cudaStream_t s, const int32_t* gather_rows = nullptr,
                         float* clear = nullptr, long long clear_n = 0, int* ctr = nullptr) {
  if (rows_alloc == 0) return MOE_OK;
  GroupedGemm g{};
  g.tile_counter = ctr;
  g.zero_ptr = clear;
  g.zero_n = clear_n;
  g.gather_rows = gather_rows;
  g.src_rows = c->T;
  g.mode = kSwiGLU;
  g.dtype = c->dtype;
  g.A = A;
  g.rows_alloc = rows_alloc;
  g.Kd = c->H;
  g.B = w_gate_up;
  g.G = gr.G;
  g.Nb = 2 * I;
  g.N_out = I;
  g.up_offset = I;
  g.C = h;
  g.offsets = gr.offsets;
  g.mtile_table = gr.table;
  g.num_mtiles = gr.num_mt;
  g.max_mtiles = gr.max_mt;
  return launch_gemm(c, d, g, s);
}

// out = h W_d^T per group.
moe_status_t run_down(const moe_config_t* c, const DeviceInfo* d, const void* h, int rows_alloc,
                      const void* w_down, int I, float* out, const Groups& gr, cudaStream_t s) {
  if (rows_alloc == 0) return MOE_OK;
  GroupedGemm g{};
  g.mode = kPlain;
  g.dtype = c->dtype;
  g.A = h;
  g.rows_alloc = rows_alloc;
  g.Kd = I;
  g.B = w_down;
  g.G = gr.G;
  g.Nb = c->H;
  g.N_out = c->H;
  g.C = out;
  g.offsets = gr.offsets;
  g.mtile_table = gr.table;
  g.num_mtiles = gr.num_mt;
  g.max_mtiles = gr.max_mt;
  return launch_gemm(c, d, g, s);
}

// The fused combine: y32[perm[r]] += row_w[r] * (h[r] W_d^T) for every kept row r, with
// the additions done at L2 (bf16 layers on the tensor cores only).
moe_status_t run_down_scatter(const moe_config_t* c, const DeviceInfo* d, const void* h,
                              int rows_alloc, const void* w_down, int I, float* y32,
                              const Groups& gr, const int32_t* perm, const float* row_w,
                              cudaStream_t s) {
  if (rows_alloc == 0) return MOE_OK;
  GroupedGemm g{};
  g.mode = kScatter;
  g.dtype = c->dtype;
  g.A = h;
  g.rows_alloc = rows_alloc;
  g.Kd = I;
  g.B = w_down;
  g.G = gr.G;
  g.Nb = c->H;
  g.N_out = c->H;
  g.C = y32;
  g.offsets = gr.offsets;
  g.row_token = perm;
  g.row_w = row_w;
  g.c_rows = c->T;
  return launch_gemm(c, d, g, s);
}

// Groups of the routed experts: bf16 reads `offsets` directly; float builds the m-tile
// table into the workspace first (unless `table_ready`).
moe_status_t routed_groups(const moe_config_t* c, const int32_t* offsets, void* ws,
                           const Plan& p, bool table_ready, cudaStream_t s, Groups* out) {
  Groups gr{};
  gr.G = c->E;
  if (c->dtype == MOE_BF16) {
    gr.offsets = offsets;
  } else {
    gr.table = at<int4>(ws, p.table);
    gr.num_mt = at<int32_t>(ws, p.num_mt);
    gr.max_mt = max_mtiles(c->T, c->K, c->E, kF32TileRows);
    if (!table_ready)
      MOE_CUDA(launch_build_mtile_table(offsets, c->E, c->T * c->K, kF32TileRows,
                                        const_cast<int4*>(gr.table),
                                        const_cast<int32_t*>(gr.num_mt), s));
  }
  *out = gr;
  return MOE_OK;
}

moe_status_t check_ws(const moe_config_t* c, void* ws, size_t ws_bytes, Plan* p) {
  *p = make_plan(c);
  if (ws == nullptr || ws_bytes < p->total) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_MISALIGNED;
  return MOE_OK;
}

bool any_misaligned(std::initializer_list<const void*> ps) {
  for (const void* q : ps)
    if (q != nullptr && !aligned16(q)) return true;
  return false;
}

// A wait that is meant to run out: one thread waits on an mbarrier that nothing arrives
// at, with a short limit, through the same bounded wait every kernel of the library uses.
__global__ void wait_timeout_probe_kernel(unsigned* err, unsigned long long limit_ns,
                                          int* done) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  abort_flag = 0;
  const bool ok = mbar_wait(b, 0, &abort_flag, err, limit_ns);
  *done = ok ? 1 : 2;
}

}  // namespace

std::atomic<unsigned long long> g_kernel_launches{0};

unsigned* device_error_word() {
  const DeviceInfo* d = device_info();
  return d != nullptr ? d->err : nullptr;
}

// ------------------------------------------------------------- fault injection ----
// A one-shot host-side fault for testing callers' error handling: once armed (by
// moe_debug_set_fault, or by MOE_FAULT=<point>:<n> in the environment when the library
// loads), the n-th pass through the named point returns MOE_ERR_CUDA there, as a failed
// launch would, and disarms.  Unarmed, a point costs one relaxed atomic load.
namespace {

const char* const kFaultPoints[] = {
    "moe_workspace_size",      "moe_route",                 "moe_permute",
    "moe_permute_noalloc",     "moe_grouped_ffn",           "moe_expert_gate_up",
    "moe_expert_gate_up_gather", "moe_expert_down",         "moe_quantize_fp8",
    "moe_expert_gate_up_fp8",  "moe_expert_down_fp8",       "moe_combine",
    "moe_layer_forward",       "moe_layer_forward_fp8",     "moe_sync_check",
    "moe_layer_forward.route", "moe_layer_forward.permute", "moe_layer_forward.gate_up",
    "moe_layer_forward.shared", "moe_layer_forward.down",   "moe_layer_forward.combine"};

struct Fault {
  std::mutex mu;
  std::atomic<bool> armed{false};
  char point[64] = {0};
  long long n = 0;
  long long seen = 0;
};

Fault& fault() {
  static Fault f;
  return f;
}

bool known_fault_point(const char* name) {
  for (const char* q : kFaultPoints)
    if (std::strcmp(q, name) == 0) return true;
  return false;
}

moe_status_t arm_fault(const char* point, long long n) {
  Fault& f = fault();
  std::lock_guard<std::mutex> lock(f.mu);
  if (point == nullptr || n <= 0) {
    f.armed.store(false);
    f.point[0] = 0;
    f.n = f.seen = 0;
    return MOE_OK;
  }
  if (!known_fault_point(point)) return MOE_ERR_INVALID_ARG;
  std::snprintf(f.point, sizeof(f.point), "%s", point);
  f.n = n;
  f.seen = 0;
  f.armed.store(true);
  return MOE_OK;
}

// MOE_FAULT=<point>:<n> arms the injector when the library is loaded.
struct FaultFromEnvironment {
  FaultFromEnvironment() {
    const char* e = std::getenv("MOE_FAULT");
    if (e == nullptr || *e == 0) return;
    const char* colon = std::strrchr(e, ':');
    char point[64] = {0};
    char* end = nullptr;
    const long long n = colon != nullptr ? std::strtoll(colon + 1, &end, 10) : 0;
    const size_t len = colon != nullptr ? static_cast<size_t>(colon - e) : 0;
    if (colon == nullptr || len == 0 || len >= sizeof(point) || end == colon + 1 || *end != 0 ||
        n <= 0) {
      std::fprintf(stderr, "moe_gb300: MOE_FAULT=%s ignored (expected <point>:<n>, n >= 1)\n", e);
      return;
    }
    std::memcpy(point, e, len);
    if (arm_fault(point, n) != MOE_OK)
      std::fprintf(stderr, "moe_gb300: MOE_FAULT=%s ignored (unknown point)\n", e);
  }
};
FaultFromEnvironment g_fault_from_environment;

}  // namespace

moe_status_t fault_point(const char* name) {
  Fault& f = fault();
  if (!f.armed.load(std::memory_order_relaxed)) return MOE_OK;
  std::lock_guard<std::mutex> lock(f.mu);
  if (!f.armed.load() || std::strcmp(f.point, name) != 0) return MOE_OK;
  if (++f.seen < f.n) return MOE_OK;
  f.armed.store(false);
  return MOE_ERR_CUDA;
}

// NVTX ranges over the stages of the layer, on the host: profilers that record NVTX
// (ncu --nvtx, Nsight Systems) attribute each stage's kernels to its range.  With no tool
// attached a range costs a few branches.  next() closes the open range and opens another.
struct StageRanges {
  bool open = false;
  void next(const char* name) {
    if (open) nvtxRangePop();
    nvtxRangePushA(name);
    open = true;
  }
  ~StageRanges() {
    if (open) nvtxRangePop();
  }
};

moe_status_t check_current_device() {
  const DeviceInfo* d = nullptr;
  return check_device(&d);
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_INTERNAL: return "MOE_ERR_INTERNAL";
    case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
  }
  return "MOE_ERR_UNKNOWN";
}

const char* moe_version(void) { return "moe_gb300 0.1 sm_103a"; }

moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes) {
  MOE_TRY(fault_point("moe_workspace_size"));
  MOE_TRY(check_config(cfg));
  if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
  *bytes = make_plan(cfg).total;
  return MOE_OK;
}

moe_status_t moe_workspace_views(const moe_config_t* cfg, void* ws, float** logits,
                                 int32_t** topk_ids, float** topk_w, int32_t** counts,
                                 int32_t** offsets, int32_t** perm, int32_t** inv, void** x_perm,
                                 float** out_perm, float** shared_out) {
  MOE_TRY(check_config(cfg));
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  const Plan p = make_plan(cfg);
  if (logits) *logits = at<float>(ws, p.logits);
  if (topk_ids) *topk_ids = at<int32_t>(ws, p.ids);
  if (topk_w) *topk_w = at<float>(ws, p.w);
  if (counts) *counts = at<int32_t>(ws, p.counts);
  if (offsets) *offsets = at<int32_t>(ws, p.offsets);
  if (perm) *perm = at<int32_t>(ws, p.perm);
  if (inv) *inv = at<int32_t>(ws, p.inv);
  if (x_perm) *x_perm = at<void>(ws, p.x_perm);
  if (out_perm) *out_perm = at<float>(ws, p.out_perm);
  if (shared_out) *shared_out = cfg->I_shared > 0 ? at<float>(ws, p.shared_out) : nullptr;
  return MOE_OK;
}

moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* w_router,
                       const float* router_bias, float* logits, int32_t* topk_ids, float* topk_w,
                       moe_stream_t stream) {
  MOE_TRY(fault_point("moe_route"));
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (logits == nullptr || topk_ids == nullptr || topk_w == nullptr) return MOE_ERR_INVALID_ARG;
  if (x != nullptr && w_router == nullptr) return MOE_ERR_INVALID_ARG;
  for (const void* q : std::initializer_list<const void*>{x, w_router, static_cast<const void*>(router_bias),
                        static_cast<const void*>(logits), static_cast<const void*>(topk_ids),
                        static_cast<const void*>(topk_w)})
    if (q != nullptr && !aligned16(q)) return MOE_ERR_MISALIGNED;
  if (cfg->T == 0) return MOE_OK;
  const DeviceInfo* d = nullptr;
  MOE_TRY(check_device(&d));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MOE_TRY(run_route(cfg, d, x, w_router, router_bias, logits, topk_ids, topk_w, nullptr, false,
                    nullptr, s));
  if ((cfg->flags & MOE_FLAG_CAPACITY) == 0u) return MOE_OK;
  return cuda_status(launch_capacity_route(logits, topk_ids, topk_w, cfg->T, cfg->E, cfg->K,
                                           cfg->gate_threshold,
                                           capacity_limit(cfg->T, cfg->K, cfg->E), d->err, s));
}

moe_status_t moe_permute(const moe_config_t* cfg, const void* x, const int32_t* topk_ids,
                         int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                         void* x_perm, void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(fault_point("moe_permute"));
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (x == nullptr || topk_ids == nullptr || counts == nullptr || offsets == nullptr ||
      perm == nullptr || inv == nullptr || x_perm == nullptr)
    return MOE_ERR_INVALID_ARG;
  for (const void* q : std::initializer_list<const void*>{x, static_cast<const void*>(topk_ids), static_cast<const void*>(counts),
                        static_cast<const void*>(offsets), static_cast<const void*>(perm),
                        static_cast<const void*>(inv), static_cast<const void*>(x_perm)})
    if (!aligned16(q)) return MOE_ERR_MISALIGNED;
  const Plan p = make_plan(cfg);
  if (ws == nullptr || ws_bytes < p.total) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_MISALIGNED;
  const DeviceInfo* d = nullptr;
  MOE_TRY(check_device(&d));
  return cuda_status(launch_permute(cfg->dtype, x, topk_ids, cfg->T, cfg->H, cfg->E, cfg->K,
                                    counts, offsets, perm, inv, x_perm, at<int32_t>(ws, p.perm_ws),
                                    nullptr, nullptr, 0, nullptr, nullptr,
                                    static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_grouped_ffn(const moe_config_t* cfg, const void* x_perm, const int32_t* offsets,
                             const void* w_gate_up, const void* w_down, float* out_perm, void* ws,
                             size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(fault_point("moe_grouped_ffn"));
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (x_perm == nullptr || offsets == nullptr || w_gate_up == nullptr || w_down == nullptr ||
      out_perm == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (any_misaligned({x_perm, offsets, w_gate_up, w_down, out_perm})) return MOE_ERR_MISALIGNED;
  Plan p;
  MOE_TRY(check_ws(cfg, ws, ws_bytes, &p));
  if (cfg->T == 0) return MOE_OK;
  const DeviceInfo* d = nullptr;
  MOE_TRY(check_device(&d));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Groups gr;
  MOE_TRY(routed_groups(cfg, offsets, ws, p, false, s, &gr));
  void* h = at<void>(ws, p.h);
  const int rows = cfg->T * cfg->K;
  cudaError_t e;
  int* ctr = standalone_counter(cfg, ws, p, s, &e);
  MOE_CUDA(e);
  MOE_TRY(run_gate_up(cfg, d, x_perm, rows, w_gate_up, cfg->I, h, gr, s, nullptr, nullptr, 0, ctr));
  return run_down(cfg, d, h, rows, w_down, cfg->I, out_perm, gr, s);
}

moe_status_t moe_expert_gate_up(const moe_config_t* cfg, const void* x_perm,
                                const int32_t* offsets, const void* w_gate_up, void* h, void* ws,
                                size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(fault_point("moe_expert_gate_up"));
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (x_perm == nullptr || offsets == nullptr || w_gate_up == nullptr || h == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (any_misaligned({x_perm, offsets, w_gate_up, h})) return MOE_ERR_MISALIGNED;
  Plan p;
  MOE_TRY(check_ws(cfg, ws, ws_bytes, &p));
  if (cfg->T == 0) return MOE_OK;
  const DeviceInfo* d = nullptr;
  MOE_TRY(check_device(&d));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Groups gr;
  MOE_TRY(routed_groups(cfg, offsets, ws, p, false, s, &gr));
  cudaError_t e;
  int* ctr = standalone_counter(cfg, ws, p, s, &e);
  MOE_CUDA(e);
  return run_gate_up(cfg, d, x_perm, cfg->T * cfg->K, w_gate_up, cfg->I, h, gr, s, nullptr,
                     nullptr, 0, ctr);
}

moe_status_t moe_quantize_fp8(const void* in, int64_t rows, int32_t cols, uint8_t* codes,
                              float* scales, moe_stream_t stream) {
  MOE_TRY(fault_point("moe_quantize_fp8"));
  if (rows < 0 || cols <= 0 || cols % 8 != 0) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (in == nullptr || codes == nullptr || scales == nullptr) return MOE_ERR_INVALID_ARG;
  if (any_misaligned({in, codes})) return MOE_ERR_MISALIGNED;
  const DeviceInfo* d = nullptr;
  MOE_TRY(check_device(&d));
  return cuda_status(launch_quantize_fp8(in, rows, cols, codes, scales,
                                         static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_expert_gate_up_fp8(const moe_config_t* cfg, const uint8_t* x_codes,
                                    const float* x_scales, const int32_t* offsets,
                                    const uint8_t* w_codes, const float* w_scales, void* h,
                                    void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(fault_point("moe_expert_gate_up_fp8"));
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (cfg->dtype != MOE_BF16 || cfg->H % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (x_codes == nullptr || x_scales == nullptr || offsets == nullptr || w_codes == nullptr ||
      w_scales == nullptr || h == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (any_misaligned({x_codes, offsets, w_codes, h})) return MOE_ERR_MISALIGNED;
  Plan p;
  MOE_TRY(check_ws(cfg, ws, ws_bytes, &p));
  const DeviceInfo* d = nullptr;
  MOE_TRY(check_device(&d));
  GroupedGemm g{};
  g.mode = kSwiGLU;
  g.dtype = cfg->dtype;
  g.A = x_codes;
  g.rows_alloc = cfg->T * cfg->K;
  g.Kd = cfg->H;
  g.B = w_codes;
  g.G = cfg->E;
  g.Nb = 2 * cfg->I;
  g.N_out = cfg->I;
  g.up_offset = cfg->I;
  g.C = h;
  g.offsets = offsets;
  g.swap_tokens = cfg->T <= kSwapMaxTokens ? cfg->T : 0;
  g.pair = use_pairs(g) ? 1 : 0;
  cudaError_t e;
  g.tile_counter = standalone_counter(cfg, ws, p, static_cast<cudaStream_t>(stream), &e);
  MOE_CUDA(e);
  return cuda_status(launch_gate_up_fp8(g, x_scales, w_scales, d->err, d->num_sms,
                                        static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_expert_down_fp8(const moe_config_t* cfg, const uint8_t* h_codes,
                                 const float* h_scales, const int32_t* offsets,
                                 const uint8_t* w_codes, const float* w_scales, float* out_perm,
                                 void* ws, size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(fault_point("moe_expert_down_fp8"));
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (cfg->dtype != MOE_BF16 || cfg->I % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (h_codes == nullptr || h_scales == nullptr || offsets == nullptr || w_codes == nullptr ||
      w_scales == nullptr || out_perm == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (any_misaligned({h_codes, offsets, w_codes, out_perm})) return MOE_ERR_MISALIGNED;
  Plan p;
  MOE_TRY(check_ws(cfg, ws, ws_bytes, &p));
  const DeviceInfo* d = nullptr;
  MOE_TRY(check_device(&d));
  GroupedGemm g{};
  g.mode = kPlain;
  g.dtype = cfg->dtype;
  g.A = h_codes;
  g.rows_alloc = cfg->T * cfg->K;
  g.Kd = cfg->I;
  g.B = w_codes;
  g.G = cfg->E;
  g.Nb = cfg->H;
  g.N_out = cfg->H;
  g.C = out_perm;
  g.offsets = offsets;
  g.swap_tokens = cfg->T <= kSwapMaxTokens ? cfg->T : 0;
  g.pair = use_pairs(g) ? 1 : 0;
  return cuda_status(launch_down_fp8(g, h_scales, w_scales, d->err, d->num_sms,
                                     static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_expert_gate_up_gather(const moe_config_t* cfg, const void* x,
                                       const int32_t* perm, const int32_t* offsets,
                                       const void* w_gate_up, void* h, void* ws, size_t ws_bytes,
                                       moe_stream_t stream) {
  MOE_TRY(fault_point("moe_expert_gate_up_gather"));
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (x == nullptr || perm == nullptr || offsets == nullptr || w_gate_up == nullptr ||
      h == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (cfg->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  if (any_misaligned({x, perm, offsets, w_gate_up, h})) return MOE_ERR_MISALIGNED;
  Plan p;
  MOE_TRY(check_ws(cfg, ws, ws_bytes, &p));
  const DeviceInfo* d = nullptr;
  MOE_TRY(check_device(&d));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Groups gr;
  MOE_TRY(routed_groups(cfg, offsets, ws, p, false, s, &gr));
  return run_gate_up(cfg, d, x, cfg->T * cfg->K, w_gate_up, cfg->I, h, gr, s, perm);
}

moe_status_t moe_expert_down(const moe_config_t* cfg, const void* h, const int32_t* offsets,
                             const void* w_down, float* out_perm, void* ws, size_t ws_bytes,
                             moe_stream_t stream) {
  MOE_TRY(fault_point("moe_expert_down"));
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (h == nullptr || offsets == nullptr || w_down == nullptr || out_perm == nullptr)
    return MOE_ERR_INVALID_ARG;
  if (any_misaligned({h, offsets, w_down, out_perm})) return MOE_ERR_MISALIGNED;
  Plan p;
  MOE_TRY(check_ws(cfg, ws, ws_bytes, &p));
  if (cfg->T == 0) return MOE_OK;
  const DeviceInfo* d = nullptr;
  MOE_TRY(check_device(&d));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  Groups gr;
  MOE_TRY(routed_groups(cfg, offsets, ws, p, false, s, &gr));
  return run_down(cfg, d, h, cfg->T * cfg->K, w_down, cfg->I, out_perm, gr, s);
}

moe_status_t moe_combine(const moe_config_t* cfg, const float* out_perm, const int32_t* inv,
                         const float* topk_w, const float* shared_out, void* y, float* y_f32,
                         moe_stream_t stream) {
  MOE_TRY(fault_point("moe_combine"));
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (out_perm == nullptr || inv == nullptr || topk_w == nullptr || y == nullptr)
    return MOE_ERR_INVALID_ARG;
  for (const void* q : std::initializer_list<const void*>{static_cast<const void*>(out_perm), static_cast<const void*>(inv),
                        static_cast<const void*>(topk_w), static_cast<const void*>(shared_out), y,
                        static_cast<const void*>(y_f32)})
    if (q != nullptr && !aligned16(q)) return MOE_ERR_MISALIGNED;
  if (cfg->T == 0) return MOE_OK;
  const DeviceInfo* d = nullptr;
  MOE_TRY(check_device(&d));
  return cuda_status(launch_combine(cfg->dtype, out_perm, inv, topk_w, shared_out, y, y_f32,
                                    cfg->T, cfg->H, cfg->K, static_cast<cudaStream_t>(stream)));
}

moe_status_t moe_layer_forward_fp8(const moe_config_t* cfg, const void* x, const void* w_router,
                                   const float* router_bias, const uint8_t* w_gate_up_codes,
                                   const float* w_gate_up_scales, const uint8_t* w_down_codes,
                                   const float* w_down_scales, const void* w_shared_gate_up,
                                   const void* w_shared_down, void* y, float* y_f32, void* ws,
                                   size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(fault_point("moe_layer_forward_fp8"));
  MOE_TRY(check_config(cfg));
  if ((cfg->flags & MOE_FLAG_FP8) == 0u) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (cfg->dtype != MOE_BF16 || cfg->H % 128 != 0 || cfg->I % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (x == nullptr || w_router == nullptr || w_gate_up_codes == nullptr ||
      w_gate_up_scales == nullptr || w_down_codes == nullptr || w_down_scales == nullptr ||
      y == nullptr)
    return MOE_ERR_INVALID_ARG;
  const bool shared = cfg->I_shared > 0;
  if (shared != (w_shared_gate_up != nullptr) || shared != (w_shared_down != nullptr))
    return MOE_ERR_INVALID_ARG;
  if (any_misaligned({x, w_router, w_gate_up_codes, w_down_codes, y, w_shared_gate_up,
                      w_shared_down, y_f32}))
    return MOE_ERR_MISALIGNED;
  const Plan p = make_plan(cfg);
  if (ws == nullptr || ws_bytes < p.total) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_MISALIGNED;
  const DeviceInfo* d = nullptr;
  MOE_TRY(check_device(&d));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int T = cfg->T, H = cfg->H, E = cfg->E, K = cfg->K, I = cfg->I;
  float* logits = at<float>(ws, p.logits);
  int32_t* ids = at<int32_t>(ws, p.ids);
  float* w = at<float>(ws, p.w);
  int32_t* counts = at<int32_t>(ws, p.counts);
  int32_t* offsets = at<int32_t>(ws, p.offsets);
  int32_t* perm = at<int32_t>(ws, p.perm);
  int32_t* inv = at<int32_t>(ws, p.inv);
  uint8_t* x_codes = at<uint8_t>(ws, p.x_codes);
  float* x_scales = at<float>(ws, p.x_scales);
  float* xs_perm = at<float>(ws, p.xs_perm);
  uint8_t* xq_perm = at<uint8_t>(ws, p.x_perm);
  void* h = at<void>(ws, p.h);
  uint8_t* h_codes = at<uint8_t>(ws, p.h_codes);
  float* h_scales = at<float>(ws, p.h_scales);
  float* out_perm = at<float>(ws, p.out_perm);
  // 1. routing (capacity-limited with MOE_FLAG_CAPACITY)
  MOE_TRY(run_route(cfg, d, x, w_router, router_bias, logits, ids, w, at<float>(ws, p.partial),
                    false, nullptr, s));
  if ((cfg->flags & MOE_FLAG_CAPACITY) != 0u)
    MOE_CUDA(launch_capacity_route(logits, ids, w, T, E, K, cfg->gate_threshold,
                                   capacity_limit(T, K, E), d->err, s));
  // 2. x's rows to E4M3 codes, then the dispatch moves the one-byte rows (as rows of H/2
  //    bf16 units) and the scales follow the permutation
  MOE_CUDA(launch_quantize_fp8(x, T, H, x_codes, x_scales, s));
  const bool fused = (cfg->flags & MOE_FLAG_FUSED_COMBINE) != 0u;
  float* row_w = fused ? at<float>(ws, p.row_w) : nullptr;
  // the permutation zeroes the routed gate/up GEMM's tile counter
  int* ctr = dynamic_tiles(cfg) ? at<int>(ws, p.tile_counter) : nullptr;
  MOE_CUDA(launch_permute(MOE_BF16, x_codes, ids, T, H / 2, E, K, counts, offsets, perm, inv,
                          xq_perm, at<int32_t>(ws, p.perm_ws), nullptr, nullptr, kF32TileRows, w,
                          row_w, s, ctr));
  MOE_CUDA(launch_gather_scales(x_scales, perm, offsets + E, xs_perm, T * K, s));
  // 3. FP8 gate/up -> bf16 h -> E4M3 h -> FP8 down
  GroupedGemm g{};
  g.mode = kSwiGLU;
  g.dtype = MOE_BF16;
  g.A = xq_perm;
  g.rows_alloc = T * K;
  g.Kd = H;
  g.B = w_gate_up_codes;
  g.G = E;
  g.Nb = 2 * I;
  g.N_out = I;
  g.up_offset = I;
  g.C = h;
  g.offsets = offsets;
  g.swap_tokens = T <= kSwapMaxTokens ? T : 0;
  g.pair = use_pairs(g) ? 1 : 0;
  g.tile_counter = ctr;
  // the fused combine's fp32 sum is initialised by the shared expert or cleared here
  float* y32 = fused ? (y_f32 != nullptr ? y_f32 : at<float>(ws, p.y32)) : nullptr;
  if (fused && !shared) {
    g.zero_ptr = y32;
    g.zero_n = static_cast<long long>(T) * H;
  }
  MOE_CUDA(launch_gate_up_fp8(g, xs_perm, w_gate_up_scales, d->err, d->num_sms, s));
  MOE_CUDA(launch_quantize_fp8(h, static_cast<long long>(T) * K, I, h_codes, h_scales, s));
  GroupedGemm gd{};
  gd.mode = kPlain;
  gd.dtype = MOE_BF16;
  gd.A = h_codes;
  gd.rows_alloc = T * K;
  gd.Kd = I;
  gd.B = w_down_codes;
  gd.G = E;
  gd.Nb = H;
  gd.N_out = H;
  gd.C = out_perm;
  gd.offsets = offsets;
  gd.swap_tokens = g.swap_tokens;
  if (fused) {
    // the combine in the down projection: the shared expert writes the fp32 sum (or the
    // gate/up GEMM cleared it), every routed row adds its gated output into its token's
    // row, then one rounding pass
    if (shared) {
      Groups one{};
      one.G = 1;
      void* hs = at<void>(ws, p.shared_h);
      MOE_TRY(run_gate_up(cfg, d, x, T, w_shared_gate_up, cfg->I_shared, hs, one, s));
      MOE_TRY(run_down(cfg, d, hs, T, w_shared_down, cfg->I_shared, y32, one, s));
    }
    gd.mode = kScatter;
    gd.C = y32;
    gd.row_token = perm;
    gd.row_w = row_w;
    gd.c_rows = T;
    gd.pair = use_pairs(gd) ? 1 : 0;
    MOE_CUDA(launch_down_fp8(gd, h_scales, w_down_scales, d->err, d->num_sms, s));
    return cuda_status(launch_finalize(cfg->dtype, y32, y, static_cast<long long>(T) * H, s));
  }
  gd.pair = use_pairs(gd) ? 1 : 0;
  MOE_CUDA(launch_down_fp8(gd, h_scales, w_down_scales, d->err, d->num_sms, s));
  // 4. shared expert (bf16), 5. combine
  float* shared_out = nullptr;
  if (shared) {
    shared_out = at<float>(ws, p.shared_out);
    Groups one{};
    one.G = 1;
    void* hs = at<void>(ws, p.shared_h);
    MOE_TRY(run_gate_up(cfg, d, x, T, w_shared_gate_up, cfg->I_shared, hs, one, s));
    MOE_TRY(run_down(cfg, d, hs, T, w_shared_down, cfg->I_shared, shared_out, one, s));
  }
  return cuda_status(launch_combine(cfg->dtype, out_perm, inv, w, shared_out, y, y_f32, T, H, K, s));
}

moe_status_t moe_layer_forward(const moe_config_t* cfg, const void* x, const void* w_router,
                               const float* router_bias, const void* w_gate_up,
                               const void* w_down, const void* w_shared_gate_up,
                               const void* w_shared_down, void* y, float* y_f32, void* ws,
                               size_t ws_bytes, moe_stream_t stream) {
  MOE_TRY(fault_point("moe_layer_forward"));
  MOE_TRY(check_config(cfg));
  if ((cfg->flags & MOE_FLAG_FP8) != 0u) return MOE_ERR_INVALID_ARG;  // moe_layer_forward_fp8
  if (cfg->T == 0) return MOE_OK;
  if (x == nullptr || w_router == nullptr || w_gate_up == nullptr || w_down == nullptr ||
      y == nullptr)
    return MOE_ERR_INVALID_ARG;
  const bool shared = cfg->I_shared > 0;
  if (shared != (w_shared_gate_up != nullptr) || shared != (w_shared_down != nullptr))
    return MOE_ERR_INVALID_ARG;
  for (const void* q : std::initializer_list<const void*>{x, w_router, static_cast<const void*>(router_bias), w_gate_up, w_down,
                        w_shared_gate_up, w_shared_down, y, static_cast<const void*>(y_f32)})
    if (q != nullptr && !aligned16(q)) return MOE_ERR_MISALIGNED;
  const Plan p = make_plan(cfg);
  if (ws == nullptr || ws_bytes < p.total) return MOE_ERR_WORKSPACE;
  if (!aligned16(ws)) return MOE_ERR_MISALIGNED;
  if (cfg->T == 0) return MOE_OK;
  const DeviceInfo* d = nullptr;
  MOE_TRY(check_device(&d));
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  float* logits = at<float>(ws, p.logits);
  int32_t* ids = at<int32_t>(ws, p.ids);
  float* w = at<float>(ws, p.w);
  int32_t* counts = at<int32_t>(ws, p.counts);
  int32_t* offsets = at<int32_t>(ws, p.offsets);
  int32_t* perm = at<int32_t>(ws, p.perm);
  int32_t* inv = at<int32_t>(ws, p.inv);
  int4* table = at<int4>(ws, p.table);
  int32_t* num_mt = at<int32_t>(ws, p.num_mt);
  void* x_perm = at<void>(ws, p.x_perm);
  float* out_perm = at<float>(ws, p.out_perm);
  const bool f32 = cfg->dtype == MOE_F32;
  // the fused combine needs the tensor-core engine; float32 layers keep the gather combine
  const bool fused = (cfg->flags & MOE_FLAG_FUSED_COMBINE) != 0u && !f32;
  // Larger batches: the gate/up GEMM reads the permuted copy x_perm.  Its row-gather
  // variant (TMA tile::gather4, four 128-byte rows per request) measured about 3x slower
  // than the copy plus whole-tile TMA loads when every group has hundreds of rows.

  // 1. router scores, top-k, gate drop
  // 2. dispatch: stable permutation, inverse map, row gather (+ the float32 m-tile table);
  //    decode-sized bf16 batches do both in one cluster launch, other small batches run
  //    the top-k inside the permutation's launch
  float* row_w = fused ? at<float>(ws, p.row_w) : nullptr;
  // Decode-sized bf16 batches route and dispatch in one cluster launch, and the gate/up
  // GEMM then gathers each group's token rows from x itself (few rows per group, so the
  // gather is cheap next to the weight stream): no permuted copy of x is made.
  // capacity-limited routing rewrites the router's choices before the dispatch, so the
  // one-launch routing + dispatch of small batches does not apply
  const bool capacity = (cfg->flags & MOE_FLAG_CAPACITY) != 0u;
  const bool cluster =
      !capacity && route_cluster_ok(cfg->dtype, cfg->T, cfg->H, cfg->E, cfg->K);
  const bool gather = cluster && cfg->T <= kGatherMaxTokens;
  // Prefill batches with a shared expert run it on the device's side stream, concurrently
  // with the dispatch permutation and the routed gate/up GEMM: it needs only x, and it is
  // tensor-bound while the permutation is memory-bound.  The routed down projection (or
  // the combine) waits for it.  Not while the caller's stream is being captured.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  const bool conc_wanted = shared && !f32 && cfg->T >= kSharedSideMinTokens &&
                           cudaStreamIsCapturing(s, &cap) == cudaSuccess &&
                           cap == cudaStreamCaptureStatusNone;
  DeviceInfo* side = conc_wanted ? side_stream(d) : nullptr;
  std::unique_lock<std::mutex> side_lock;
  if (side != nullptr) side_lock = std::unique_lock<std::mutex>(side->side_mu);
  // once the shared expert is on the side stream, every return makes `s` wait for it
  struct JoinOnExit {
    DeviceInfo* side = nullptr;
    cudaStream_t s = nullptr;
    bool armed = false;
    ~JoinOnExit() {
      if (armed) cudaStreamWaitEvent(s, side->join, 0);
    }
  } join_guard;
  void* hs = at<void>(ws, p.shared_h);
  float* y32 = fused ? (y_f32 != nullptr ? y_f32 : at<float>(ws, p.y32)) : nullptr;
  float* shared_out = nullptr;
  if (shared && !fused) shared_out = at<float>(ws, p.shared_out);
  auto run_shared = [&](cudaStream_t st) -> moe_status_t {
    Groups one{};
    one.G = 1;
    MOE_TRY(run_gate_up(cfg, d, x, cfg->T, w_shared_gate_up, cfg->I_shared, hs, one, st));
    return run_down(cfg, d, hs, cfg->T, w_shared_down, cfg->I_shared, fused ? y32 : shared_out,
                    one, st);
  };
  int* gu_counter = nullptr;  // set where the permutation zeroes it
  StageRanges nv;
  nv.next("moe_layer_forward.route");
  MOE_TRY(fault_point("moe_layer_forward.route"));
  if (cluster) {
    nv.next("moe_layer_forward.permute");
    MOE_TRY(fault_point("moe_layer_forward.permute"));  // the cluster launch dispatches too
    MOE_CUDA(launch_route_cluster(x, w_router, router_bias, logits, ids, w, cfg->gate_threshold,
                                  cfg->T, cfg->H, cfg->E, cfg->K, counts, offsets, perm, inv,
                                  row_w, gather ? nullptr : x_perm, d->err, s));
  } else {
    int deferred = 0;
    float* partial = at<float>(ws, p.partial);
    MOE_TRY(run_route(cfg, d, x, w_router, router_bias, logits, ids, w, partial, !capacity,
                      &deferred, s));
    if (capacity)
      MOE_CUDA(launch_capacity_route(logits, ids, w, cfg->T, cfg->E, cfg->K, cfg->gate_threshold,
                                     capacity_limit(cfg->T, cfg->K, cfg->E), d->err, s));
    if (side != nullptr) {
      nv.next("moe_layer_forward.shared");
      MOE_TRY(fault_point("moe_layer_forward.shared"));
      MOE_CUDA(cudaEventRecord(side->fork, s));
      MOE_CUDA(cudaStreamWaitEvent(side->side, side->fork, 0));
      const moe_status_t st_shared = run_shared(side->side);
      const cudaError_t e_join = cudaEventRecord(side->join, side->side);
      join_guard.side = side;
      join_guard.s = s;
      join_guard.armed = e_join == cudaSuccess;
      MOE_TRY(st_shared);
      MOE_CUDA(e_join);
    }
    nv.next("moe_layer_forward.permute");
    MOE_TRY(fault_point("moe_layer_forward.permute"));
    // the permutation zeroes the routed gate/up GEMM's tile counter
    gu_counter = dynamic_tiles(cfg) ? at<int>(ws, p.tile_counter) : nullptr;
    if (deferred > 0) {
      MOE_CUDA(launch_topk_permute_small(partial, deferred, router_bias, logits, ids, w,
                                         cfg->gate_threshold, cfg->dtype, x, cfg->T, cfg->H,
                                         cfg->E, cfg->K, counts, offsets, perm, inv, x_perm,
                                         f32 ? table : nullptr, f32 ? num_mt : nullptr, kF32TileRows,
                                         row_w, s, gu_counter));
    } else {
      MOE_CUDA(launch_permute(cfg->dtype, x, ids, cfg->T, cfg->H, cfg->E, cfg->K, counts,
                              offsets, perm, inv, x_perm, at<int32_t>(ws, p.perm_ws),
                              f32 ? table : nullptr, f32 ? num_mt : nullptr, kF32TileRows, w, row_w,
                              s, gu_counter));
    }
  }
  // 3-4. grouped SwiGLU FFN of the routed experts
  Groups gr;
  MOE_TRY(routed_groups(cfg, offsets, ws, p, true, s, &gr));
  void* h = at<void>(ws, p.h);
  const int rows = cfg->T * cfg->K;
  // the fused combine's fp32 sum: the shared expert's down projection initialises it, or
  // else the routed gate/up GEMM clears it (a memset node between the two expert GEMMs
  // would keep the down projection from launching early), except for 17..128 tokens,
  // where a memset measured about 1% faster
  const bool memset_sum = fused && !shared && cfg->T > 16 && cfg->T <= 128;
  float* clear = fused && !shared && !memset_sum ? y32 : nullptr;
  const long long clear_n = static_cast<long long>(cfg->T) * cfg->H;
  nv.next("moe_layer_forward.gate_up");
  MOE_TRY(fault_point("moe_layer_forward.gate_up"));
  if (gather)
    MOE_TRY(run_gate_up(cfg, d, x, rows, w_gate_up, cfg->I, h, gr, s, perm, clear, clear_n));
  else
    MOE_TRY(run_gate_up(cfg, d, x_perm, rows, w_gate_up, cfg->I, h, gr, s, nullptr, clear,
                        clear_n, gu_counter));
  if (fused) {
    // 5'. shared expert written straight into the fp32 sum (cleared above otherwise), then
    //     the down projection adds every routed row, scaled by its gate, into its token's
    //     row, and one pass rounds the sum to the output type
    if (side == nullptr) {
      nv.next("moe_layer_forward.shared");
      MOE_TRY(fault_point("moe_layer_forward.shared"));
    }
    if (shared && side == nullptr) {
      MOE_TRY(run_shared(s));
    } else if (memset_sum) {
      MOE_CUDA(cudaMemsetAsync(y32, 0, static_cast<size_t>(cfg->T) * cfg->H * sizeof(float), s));
    }
    nv.next("moe_layer_forward.down");
    MOE_TRY(fault_point("moe_layer_forward.down"));
    if (side != nullptr) {  // the shared expert has written the fp32 sum
      join_guard.armed = false;
      MOE_CUDA(cudaStreamWaitEvent(s, side->join, 0));
    }
    MOE_TRY(run_down_scatter(cfg, d, h, rows, w_down, cfg->I, y32, gr, perm,
                             at<float>(ws, p.row_w), s));
    nv.next("moe_layer_forward.combine");
    MOE_TRY(fault_point("moe_layer_forward.combine"));
    return cuda_status(
        launch_finalize(cfg->dtype, y32, y, static_cast<long long>(cfg->T) * cfg->H, s));
  }
  nv.next("moe_layer_forward.down");
  MOE_TRY(fault_point("moe_layer_forward.down"));
  MOE_TRY(run_down(cfg, d, h, rows, w_down, cfg->I, out_perm, gr, s));
  // 5. shared expert: the same engine on all T rows of x as one group (already enqueued on
  //    the side stream for prefill batches)
  if (side == nullptr) {
    nv.next("moe_layer_forward.shared");
    MOE_TRY(fault_point("moe_layer_forward.shared"));
    if (shared) MOE_TRY(run_shared(s));
  }
  // 6. un-permute and weighted combine
  nv.next("moe_layer_forward.combine");
  MOE_TRY(fault_point("moe_layer_forward.combine"));
  if (side != nullptr) {  // the shared expert's output is complete
    join_guard.armed = false;
    MOE_CUDA(cudaStreamWaitEvent(s, side->join, 0));
  }
  return cuda_status(launch_combine(cfg->dtype, out_perm, inv, w, shared_out, y, y_f32, cfg->T,
                                    cfg->H, cfg->K, s));
}

moe_status_t moe_debug_wait_timeout(unsigned limit_us, int* done, moe_stream_t stream) {
  if (done == nullptr || limit_us == 0 || limit_us > 1000000u) return MOE_ERR_INVALID_ARG;
  if (!aligned16(done)) return MOE_ERR_MISALIGNED;
  const DeviceInfo* d = nullptr;
  MOE_TRY(check_device(&d));
  wait_timeout_probe_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
      d->err, static_cast<unsigned long long>(limit_us) * 1000ull, done);
  return cuda_status(count_launch(cudaGetLastError()));
}

moe_status_t moe_debug_set_fault(const char* point, int n) {
  return arm_fault(point, static_cast<long long>(n));
}

unsigned long long moe_kernel_launch_count(void) {
  return moe::g_kernel_launches.load(std::memory_order_relaxed);
}

moe_status_t moe_sync_check(moe_stream_t stream) {
  MOE_TRY(fault_point("moe_sync_check"));
  const DeviceInfo* d = device_info();
  if (d == nullptr) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, d->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (word != 0) {
    const unsigned zero = 0;
    if (cudaMemcpy(d->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
      return MOE_ERR_CUDA;
    return (word & MOE_DEVERR_TIMEOUT) ? MOE_ERR_TIMEOUT : MOE_ERR_INTERNAL;
  }
  return MOE_OK;
}

}  // extern "C"
