// Internal launchers of the MoE layer kernels (host side).  The public C ABI in
// include/moe.h validates arguments and then calls these.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

#include <atomic>
#include <cstring>
#include <utility>

namespace moe {

enum DType : int { kF32 = 0, kBF16 = 1 };

inline size_t act_bytes(int dtype) { return dtype == kBF16 ? 2 : 4; }

// Kernels this library has launched in this process (launches the runtime accepted, on
// every device; a launch into a stream being captured counts once, at capture).
extern std::atomic<unsigned long long> g_kernel_launches;

inline cudaError_t count_launch(cudaError_t e) {
  if (e == cudaSuccess) g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  return e;
}

// Launch with programmatic stream serialization: the kernel may be scheduled while the
// previous kernel on the stream is still running; every kernel of this library calls
// griddepcontrol.wait before reading what an earlier kernel wrote.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t lc;
  std::memset(&lc, 0, sizeof(lc));
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return count_launch(cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...));
}

// Rows per m-tile of the bf16 grouped GEMM and of the float32 grouped GEMM (whose groups
// come from an m-tile table of 64-row tiles).
constexpr int kTcBM = 128;
constexpr int kF32TileRows = 64;

// ------------------------------------------------------------------ routing ----
// Router logits on the CUDA cores (see route.cu for when each is used).
// Few experts with W_r in shared memory; top-k fused (one launch).
bool router_uses_wsmem(int dtype, int T, int H, int E);
cudaError_t launch_router_wsmem(int dtype, const void* x, const void* w_router,
                                const float* bias, float* logits, int32_t* ids, float* w, int T,
                                int H, int E, int K, float theta, unsigned* err, cudaStream_t s);
// Number of H slices of the partial-logits router for this shape (deterministic).
int router_slices(int T, int H, int E, int dtype);
// partial[s][t][e] over H slice s (no bias), S = router_slices(...) slices.
cudaError_t launch_router_partial(int dtype, const void* x, const void* w_router, float* partial,
                                  int S, int T, int H, int E, cudaStream_t s);

// Decode-sized bf16 batches (T <= 64, E <= 256, K <= 16): router logits on the tensor
// core, top-k, gate drop and (when `counts` is non-null) the whole dispatch permutation,
// in one launch of one thread-block cluster (route_cluster.cu).  Token rows are copied
// into x_perm unless it is null (the gate/up GEMM then gathers them from x).
bool route_cluster_ok(int dtype, int T, int H, int E, int K);
cudaError_t launch_route_cluster(const void* x, const void* w_router, const float* bias,
                                 float* logits, int32_t* ids, float* w, float theta, int T, int H,
                                 int E, int K, int32_t* counts, int32_t* offsets, int32_t* perm,
                                 int32_t* inv, float* row_w, void* x_perm, unsigned* err,
                                 cudaStream_t s);
// Capacity-limited routing (capacity.cu): ceil(1.2 T K / E) kept assignments per expert, and
// the in-place rewrite of the router's choices ids/w [T,K] (from logits [T,E]) into the
// token-by-token capacity routing.  E <= 1024, K <= 16; one thread-block cluster (16 CTAs
// where the device holds it).
int capacity_limit(int T, int K, int E);
cudaError_t launch_capacity_route(const float* logits, int32_t* ids, float* w, int T, int E, int K,
                                  float theta, int cap, unsigned* err, cudaStream_t s);
// 2D TMA map of a row-major bf16 [rows, cols] matrix, box = 64 columns x box_rows rows,
// 128-byte swizzle (gemm_tc.cu).
bool make_tma_2d_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows);

// Top-k, softmax over the kept logits and gate drop, one warp per token.  The logits are
// the sum of S partial slices [S][T][E] (S = 1: plain logits) plus `bias` (may be null);
// they are written to `logits_out` when non-null (which may alias `partial` if S == 1).
cudaError_t launch_topk(const float* partial, int S, const float* bias, float* logits_out,
                        int32_t* ids, float* w, int T, int E, int K, float theta,
                        cudaStream_t s);

// ---------------------------------------------------------------- dispatch ----
// Workspace (int32 words) the permutation needs for T tokens, E experts.
size_t permute_ws_words(int T, int E);

// Device address of the current device's error word (MOE_DEVERR_* bits, reported by
// moe_sync_check), or null when the device cannot be set up.  Launchers pass it to kernels
// that check indices in the debug build.
unsigned* device_error_word();

// Host-side fault injection (moe_debug_set_fault, MOE_FAULT): MOE_ERR_CUDA when the armed
// fault is due at the named point, else MOE_OK.
moe_status_t fault_point(const char* name);

// MOE_OK when the current device is an sm_103 GPU this library runs on (the same check
// every entry point makes), MOE_ERR_UNSUPPORTED when it is not, MOE_ERR_CUDA when the
// device cannot be queried.
moe_status_t check_current_device();
// Maximum number of m-tiles of `bm` rows over all groups of T*K rows and E experts.
inline int max_mtiles(int T, int K, int E, int bm) {
  return static_cast<int>((static_cast<long long>(T) * K + bm - 1) / bm) + E;
}

// Stable counting-sort permutation: counts, offsets, perm, inv and the row gather
// x_perm[r] = x[perm[r]].  If `mtile_table` is non-null the m-tile table of `bm`
// rows per tile is written as well (entries {expert, row0, row_end, 0}) with its
// length in *num_mtiles.  If `row_w` is non-null, row_w[r] = gate_w of row r's slot.
// If `zero_word` is non-null it is set to 0 (the tile counter of a later grouped GEMM on
// the same stream, so that no memset sits between the launches).
cudaError_t launch_permute(int dtype, const void* x, const int32_t* ids, int T, int H, int E,
                           int K, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                           void* x_perm, int32_t* ws_words, int4* mtile_table,
                           int32_t* num_mtiles, int bm, const float* gate_w, float* row_w,
                           cudaStream_t s, int32_t* zero_word = nullptr);

// Routing and the permutation in one launch for small batches: logits = sum of the
// router's S partial slices + bias (written to `logits`), top-k/softmax/gate drop
// (written to ids/w), then the permutation as launch_permute.
bool topk_permute_fusable(int T, int E, int K);
cudaError_t launch_topk_permute_small(const float* partial, int S, const float* bias,
                                      float* logits, int32_t* ids, float* w, float theta,
                                      int dtype, const void* x, int T, int H, int E, int K,
                                      int32_t* counts, int32_t* offsets, int32_t* perm,
                                      int32_t* inv, void* x_perm, int4* mtile_table,
                                      int32_t* num_mtiles, int bm, float* row_w, cudaStream_t s,
                                      int32_t* zero_word = nullptr);

// The m-tile table of a grouped GEMM from offsets alone.
// `rows`: rows of the grouped matrix (offsets[E] must not exceed it).
cudaError_t launch_build_mtile_table(const int32_t* offsets, int E, int rows, int bm,
                                     int4* table, int32_t* num_mtiles, cudaStream_t s);

// ----------------------------------------------------------------- combine ----
// y = act(y_f32) elementwise (the last step of the fused combine).
cudaError_t launch_finalize(int dtype, const float* y_f32, void* y, long long n, cudaStream_t s);
cudaError_t launch_combine(int dtype, const float* out_perm, const int32_t* inv, const float* w,
                           const float* shared_out, void* y, float* y_f32, int T, int H, int K,
                           cudaStream_t s);

// --------------------------------------------------------- grouped GEMMs ----
// Grouped NT GEMM description shared by the float32 (tf32 split) and the bf16 / FP8
// engines: for every m-tile (group g, rows row0..row_end-1 of A):
//   C[row, n] = sum_k A[row, k] * B[g, n, k]                      (mode kPlain)
//   C[row, n] = silu(sum_k A B[g, n, k]) * (sum_k A B[g, up + n, k])  (mode kSwiGLU)
// A: [rows_alloc, Kd] row-major; B: [G, Nb, Kd] row-major; C: [rows_alloc, N_out].
//   C[row_token[row], n] += row_w[row] * sum_k A[row, k] * B[g, n, k]  (mode kScatter:
//   the combine fused into the down projection; fp32 additions at L2, order not fixed)
// kTopK: kPlain (the router logits, + col_bias) whose epilogue also takes each row's top-k
// over all N_out <= 256 columns (one tile spans them) with the softmax and gate drop.
enum GemmMode : int { kPlain = 0, kSwiGLU = 1, kScatter = 2, kTopK = 3 };

struct GroupedGemm {
  int mode;
  int dtype;                 // act type of A and B; C is act for kSwiGLU, float for kPlain
  const void* A;
  int rows_alloc;            // rows of A/C that exist in memory
  int Kd;                    // reduction length
  const void* B;
  int G;                     // groups in B
  int Nb;                    // rows of one group of B
  int N_out;                 // output columns
  int up_offset;             // kSwiGLU: first row of the up block in a group of B
  void* C;
  const float* col_bias;     // kPlain only: added per output column, or null
  // Groups: device row offsets [G+1] of the groups in A (tensor-core engine), or
  // null for a single group 0 covering rows 0..rows_alloc-1.
  const int32_t* offsets;
  // float32 engine: a device m-tile table {group, row0, row_end, 0} with a device count,
  // or null for a single group.
  const int4* mtile_table;
  const int32_t* num_mtiles;
  int max_mtiles;            // upper bound of the device count (grid sizing)
  // Tensor-core engine only: 0 = token rows on the 128-row MMA side (prefill); > 0 =
  // the largest number of token rows a group can have, with weights on the 128-row side
  // and tokens in tiles of 16/32/64 (decode).
  int swap_tokens;
  const int32_t* row_token;  // kScatter only
  const float* row_w;        // kScatter only
  int c_rows;                // kScatter: rows of C (checked in the debug build; 0 = unknown)
  // Tensor-core engine: a float array that the launch clears (n floats, n % 4 == 0,
  // 16-byte aligned) before the scatter-add of a later launch, or null.  The fused
  // combine's fp32 sum is cleared this way by the gate/up GEMM that precedes its down
  // projection, so no separate memset sits between the two launches.
  float* zero_ptr;
  long long zero_n;
  // Tensor-core engine, normal order: a device int, zero when the launch starts, from
  // which the CTAs draw tile indices in order as they become free; or null for a fixed
  // round-robin assignment of the tiles.
  int* tile_counter;
  // Tensor-core engine, normal order only: run on CTA pairs (cta_group::2, 256-row tiles)
  int pair;
  // Tensor-core engine, single CTAs: row r of the (grouped) A is row gather_rows[r] of the
  // src_rows x Kd matrix at A, fetched by TMA row gathers (no permuted copy of A), or null.
  const int32_t* gather_rows;
  int src_rows;
  // kTopK only: K (<= 16), gate threshold, outputs ids [rows, K] and weights [rows, K]
  int topk_k;
  float topk_theta;
  int32_t* topk_ids;
  float* topk_w;
};


// float32 layers on the tensor cores (gemm_tf32.cu): three kind::tf32 MMAs per k-step on
// operands split into a tf32 part and a remainder; groups from the m-tile table (64 rows).
cudaError_t launch_grouped_gemm_tf32(const GroupedGemm& g, unsigned* err, int num_sms,
                                     cudaStream_t s);
// FP8 (E4M3) per-row quantisation of a bf16 [rows, cols] matrix (quant.cu); cols % 8 == 0.
cudaError_t launch_quantize_fp8(const void* in, long long rows, int cols, uint8_t* codes,
                                float* scales, cudaStream_t s);
// dst[r] = src[perm[r]] for r < offsets_end[0] (device), 0 for r < n beyond it (quant.cu).
cudaError_t launch_gather_scales(const float* src, const int32_t* perm, const int32_t* offsets_end,
                                 float* dst, int n, cudaStream_t s);
// The gate/up GEMM on E4M3 operands (A [rows_alloc, Kd] and B [G, Nb, Kd] codes, Kd % 128
// == 0) with per-row scales a_scale [rows_alloc] and b_scale [G, Nb]; single CTAs (swapped
// for decode-sized batches), bf16 h.
cudaError_t launch_gate_up_fp8(const GroupedGemm& g, const float* a_scale, const float* b_scale,
                               unsigned* err, int num_sms, cudaStream_t s);
// The down projection (kPlain, or kScatter for the fused combine) on E4M3 operands: h codes
// [rows_alloc, Kd] with a_scale per row, W_d codes [G, Nb, Kd] with b_scale per output channel.
cudaError_t launch_down_fp8(const GroupedGemm& g, const float* a_scale, const float* b_scale,
                            unsigned* err, int num_sms, cudaStream_t s);
cudaError_t launch_grouped_gemm_tc(const GroupedGemm& g, unsigned* err, int num_sms,
                                   cudaStream_t s);

}  // namespace moe
