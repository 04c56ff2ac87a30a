/*
 * moe.h -- C ABI of a single-GPU Mixture-of-Experts feed-forward layer (forward pass)
 * for NVIDIA GB300 (sm_103a).
 *
 * The layer follows the pipeline that the page opening
 * "MoE通过稀疏激活降低每个token的计算量但增加了服务系统的复杂度" describes in its section
 * "单机MoE执行流水线": the router scores every expert, top-k keeps the chosen expert ids
 * and weights, a permutation writes the token rows in expert order and records an
 * inverse map, a grouped GEMM runs every expert's ragged row block in one launch, each
 * expert applies its activation and output projection, and an un-permute restores token
 * order, applies the route weights and sums the contributions of each token.  The
 * routing rule (softmax over the top-k logits, then drop gates below a threshold and
 * renormalise) is section 2.2 of the page "MoE大模型的智能调度：从1.8万亿参数到每token仅激活
 * 2%的工程真相".
 *
 * Notation: T tokens, H hidden size, E routed experts, K experts per token, I expert
 * intermediate size, I_shared intermediate size of the always-on shared expert (0 =
 * none), theta the gate-drop threshold (0 = off), M the number of kept assignments
 * (M = T*K when theta = 0).
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - Every tensor pointer is DEVICE memory owned by the caller, row-major and
 *    contiguous, 16-byte aligned.  "act" below means the configured activation/weight
 *    type: bfloat16 when cfg->dtype == MOE_BF16, float when cfg->dtype == MOE_F32.
 *  - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL = legacy default
 *    stream) and the call returns without synchronising.  The library never allocates
 *    or frees device memory on these paths and never synchronises the device.
 *  - Arguments are validated on the host before any launch; on any error nothing is
 *    launched and the outputs are untouched.  No C++ exception crosses this boundary.
 *  - T == 0 is a valid no-op: the call returns MOE_OK after checking `cfg` only (the
 *    pointers of an empty batch may be NULL).
 *  - Supported shapes: 1 <= K <= min(E, 16), E <= 1024, H and I multiples of 64,
 *    0 <= theta < 1, H <= 65536, I <= 65536, T*K < 2^31.
 *  - Asynchronous device errors (a bounded wait that timed out inside a kernel) are
 *    recorded in a device error word and reported by moe_sync_check().
 *  - Calls are deterministic: the same inputs give bitwise-identical outputs.
 *  - Calls with separate workspaces may run concurrently on different streams.
 */
#ifndef MOE_GB300_MOE_H
#define MOE_GB300_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad shape, bad threshold */
  MOE_ERR_UNSUPPORTED = 2,   /* shape/type outside the supported set, or no sm_103a device */
  MOE_ERR_WORKSPACE = 3,     /* workspace missing or smaller than moe_workspace_size() */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed (launch error, ...) */
  MOE_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up (see moe_sync_check) */
  MOE_ERR_INTERNAL = 6,      /* an internal consistency check failed */
  MOE_ERR_MISALIGNED = 7     /* a pointer is not 16-byte aligned */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;

/* moe_config_t.flags */
enum {
  /* moe_layer_forward only, bf16 layers: fuse the combine into the down projection.  Each
   * routed row of the down GEMM is scaled by its gate and added in fp32 straight into its
   * token's row of the fp32 sum (which the shared expert initialises, else it starts at
   * zero); one pass then rounds the sum to bf16.  This removes the [T*K, H] fp32
   * intermediate and the separate combine.  The K additions of a token happen in no fixed
   * order, so y and y_f32 are correct to fp32 rounding but not bitwise reproducible from
   * run to run.  Without this flag (default) the combine gathers in slot order and every
   * output is deterministic.  Float32 layers ignore the flag. */
  MOE_FLAG_FUSED_COMBINE = 1u,
  /* moe_route and moe_layer_forward: capacity-limited routing ("MoE大模型的智能调度…" §3.2,
   * trap 2).  Each expert takes at most cap = ceil(1.2 * T * K / E) kept assignments.
   * Tokens are routed in token order: an expert that earlier tokens have filled is
   * unavailable (its logit counts as -inf), and the token takes its top-k of the available
   * experts, with the softmax over them and the gate drop as usual; dropped assignments do
   * not use capacity.  If fewer than K experts are available the missing slots hold -1 / 0
   * (a suffix, like dropped slots).  E <= 1024.  The result is deterministic and equals
   * the token-by-token rule; it runs as one extra single-CTA launch after the router. */
  MOE_FLAG_CAPACITY = 2u,
  /* moe_workspace_size and moe_layer_forward_fp8: the routed experts run on FP8 (E4M3)
   * codes (see moe_layer_forward_fp8); the workspace then also holds the codes and scales
   * of x and h.  moe_layer_forward rejects this flag. */
  MOE_FLAG_FP8 = 4u
};

typedef struct {
  int32_t T;               /* tokens */
  int32_t H;               /* hidden size */
  int32_t E;               /* routed experts */
  int32_t K;               /* experts per token (top-k) */
  int32_t I;               /* routed expert intermediate size */
  int32_t I_shared;        /* shared expert intermediate size, 0 = no shared expert */
  float gate_threshold;    /* theta: drop kept gates below it (slot 0 never), 0 = off */
  int32_t dtype;           /* moe_dtype_t of activations and weights */
  uint32_t flags;          /* MOE_FLAG_* bits; 0 = defaults */
} moe_config_t;

typedef void* moe_stream_t; /* a cudaStream_t */

/* Bytes of device workspace that moe_layer_forward, moe_permute and moe_grouped_ffn
 * need for `cfg` (the largest of the three).  The workspace is scratch: its contents
 * are undefined between calls, and it must not be shared by calls that may run
 * concurrently.  Among the intermediates, a call with more than 128 tokens keeps in it
 * the counter from which the gate/up GEMM's CTA pairs draw their tiles; the call zeroes
 * it first (in the permutation's launch, or with a memset in the standalone GEMM calls),
 * so no state carries from one call to the next.  Returns MOE_ERR_INVALID_ARG for an
 * unsupported config. */
moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* bytes);

/* Router scores and routing.
 * Defined by: "MoE大模型的智能调度…" §2.2 routing steps 1-3 (logits per expert, softmax
 * over the top-k logits, drop gates below the threshold and renormalise) and the
 * page section "单机MoE执行流水线" (the router scores every candidate expert; top-k keeps
 * the chosen ids and weights).
 *   x           [T,H] act, or NULL: then `logits` is an INPUT [T,E] float that is read
 *               (router_bias is then ignored).
 *   w_router    [E,H] act (ignored when x == NULL).
 *   router_bias [E] float added to every token's logits, or NULL for none.
 *   logits      [T,E] float: written with x*W_r^T + bias (fp32 accumulation) when x != NULL.
 *   topk_ids    [T,K] int32 out: slot 0 = largest logit, descending, ties to the lower
 *               expert id; a dropped slot holds -1 (dropped slots form a suffix).
 *   topk_w      [T,K] float out: softmax over the K kept logits, after the drop the
 *               survivors renormalised to sum 1; dropped slots hold 0.
 * The selection is taken on float32 logits.  With MOE_FLAG_CAPACITY the choices are
 * capacity-limited (see the flag). */
moe_status_t moe_route(const moe_config_t* cfg, const void* x, const void* w_router,
                       const float* router_bias, float* logits, int32_t* topk_ids,
                       float* topk_w, moe_stream_t stream);

/* Dispatch: group the assignments by expert (a stable permutation) and gather rows.
 * Defined by: page section "一个批次如何变成各专家专属的矩阵" (assignments grouped by
 * expert into matrices, the source token id kept beside each row) and section
 * "单机MoE执行流水线" (the permutation writes token rows in expert order and records an
 * inverse map for the combine).
 *   x         [T,H] act in.
 *   topk_ids  [T,K] int32 in (from moe_route; -1 = dropped, not dispatched).
 *   counts    [E] int32 out: rows per expert.
 *   offsets   [E+1] int32 out: exclusive prefix sum of counts; offsets[E] = M.
 *   perm      [T*K] int32 out: perm[r] = source token of row r, rows ordered by
 *             (expert ascending, token ascending); entries r >= M are untouched.
 *   inv       [T*K] int32 out: inv[t*K+k] = row of assignment (t,k), -1 if dropped.
 *   x_perm    [T*K,H] act out: x_perm[r] = x[perm[r]]; rows r >= M untouched.
 *   ws        workspace of at least moe_workspace_size() bytes. */
moe_status_t moe_permute(const moe_config_t* cfg, const void* x, const int32_t* topk_ids,
                         int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                         void* x_perm, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Largest scratch (int32 words) moe_permute_noalloc can use: it needs
 * ceil(T/256) * E words, so E = 128 allows T <= 524288 and E = 1024 allows T <= 65536. */
#define MOE_PERMUTE_NOALLOC_MAX_WORDS 262144

/* moe_permute without a workspace, for callers that cannot allocate device memory (an
 * inference server that sizes all its device pools once at start-up and allows no
 * allocation later, a plug-in host that passes a kernel only its inputs and outputs).
 * No counterpart on the pages: it is a deployment variant of moe_permute.
 * Same arguments, outputs and results as moe_permute, minus ws/ws_bytes.  The scratch of
 * the counting sort comes from a fixed 1 MiB array inside the library
 * (MOE_PERMUTE_NOALLOC_MAX_WORDS int32 words), held on every GPU that loads the library
 * until the process exits.  It allocates and frees nothing.
 *  - A problem that needs more than MOE_PERMUTE_NOALLOC_MAX_WORDS words of scratch is
 *    rejected with MOE_ERR_WORKSPACE before anything is launched.
 *  - The first call on a device looks up the array's device address on that device
 *    (the device must be current); make that first call before any stream capture.
 *  - Every call on a device shares the one array and leaves its contents behind; calls
 *    that can overlap on the GPU (other streams, other host threads) race on it, so the
 *    caller must serialise them.  No part of the array needs to start at zero. */
moe_status_t moe_permute_noalloc(const moe_config_t* cfg, const void* x, const int32_t* topk_ids,
                                 int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                                 void* x_perm, moe_stream_t stream);

/* Grouped expert FFN over ragged row groups (one launch per GEMM for all experts).
 * Defined by: page section "单机MoE执行流水线" (a grouped GEMM runs several experts'
 * matrices of different row counts in one launch, then each expert applies its
 * activation and output projection) and "MoE大模型的智能调度…" §2.2 expert layer (every
 * expert is a two-layer FFN of the same shape with its own weights).  Activation:
 * SwiGLU, out = (silu(x W_g^T) * (x W_u^T)) W_d^T; the intermediate h is rounded to
 * `act` between the two GEMMs; accumulation is fp32.  Float32 layers multiply on the
 * tensor cores with each operand split into a tf32 part and its remainder (three tf32
 * products per step), which keeps the accuracy of a float32 dot product.
 *   x_perm    [T*K,H] act in; rows offsets[e]..offsets[e+1]-1 belong to expert e.
 *   offsets   [E+1] int32 in (device).
 *   w_gate_up [E,2I,H] act: rows 0..I-1 of expert e = W_g, rows I..2I-1 = W_u.
 *   w_down    [E,H,I] act.
 *   out_perm  [T*K,H] float out; rows r >= offsets[E] untouched.
 *   ws        workspace of at least moe_workspace_size() bytes. */
moe_status_t moe_grouped_ffn(const moe_config_t* cfg, const void* x_perm, const int32_t* offsets,
                             const void* w_gate_up, const void* w_down, float* out_perm,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* The first GEMM of the grouped FFN alone: gate/up projection with SwiGLU.
 * Defined by: page section "单机MoE执行流水线" (grouped GEMM over ragged expert row
 * groups; each expert applies its activation).  For every row r of group e:
 *   h[r] = silu(x_perm[r] W_g[e]^T) * (x_perm[r] W_u[e]^T), fp32 accumulation, rounded
 *   once to `act`.
 *   x_perm [T*K,H] act in; offsets [E+1] int32 in; w_gate_up [E,2I,H] act;
 *   h [T*K,I] act out (rows >= offsets[E] untouched); ws as for moe_grouped_ffn. */
moe_status_t moe_expert_gate_up(const moe_config_t* cfg, const void* x_perm,
                                const int32_t* offsets, const void* w_gate_up, void* h, void* ws,
                                size_t ws_bytes, moe_stream_t stream);

/* The same gate/up projection with the dispatch row gather folded into its loads: row r
 * of the groups is token row perm[r] of x, so no permuted copy of x is needed.
 * Defined by: page section "单机MoE执行流水线" (moving token rows to their experts is
 * part of the cost at small batches; a fused kernel need not write intermediates back to
 * device memory).  For every row r of group e:
 *   h[r] = silu(x[perm[r]] W_g[e]^T) * (x[perm[r]] W_u[e]^T), as moe_expert_gate_up.
 *   x [T,H] act in; perm [T*K] int32 in (device; entries below offsets[E] are token ids in
 *   0..T-1, the rest are not read); offsets [E+1] int32 in; w_gate_up [E,2I,H] act;
 *   h [T*K,I] act out (rows >= offsets[E] untouched); ws as for moe_grouped_ffn.
 * bf16 only (MOE_ERR_UNSUPPORTED for float32 layers). */
moe_status_t moe_expert_gate_up_gather(const moe_config_t* cfg, const void* x,
                                       const int32_t* perm, const int32_t* offsets,
                                       const void* w_gate_up, void* h, void* ws,
                                       size_t ws_bytes, moe_stream_t stream);

/* The whole layer with FP8 (E4M3) routed experts, as moe_layer_forward otherwise: routing
 * (capacity-limited with MOE_FLAG_CAPACITY), then x quantised per token row, the dispatch
 * of the one-byte rows, the FP8 gate/up (moe_expert_gate_up_fp8) to bf16 h, h quantised
 * per row, the FP8 down projection (moe_expert_down_fp8), the bf16 shared expert and the
 * gather combine.
 * Defined by: page section "单机MoE执行流水线" (the layer's stages) and
 * "MoE大模型的智能调度…" §4.1 (8-bit expert weights).
 *   w_gate_up_codes [E,2I,H] uint8 and w_gate_up_scales [E,2I] float, w_down_codes [E,H,I]
 *   uint8 and w_down_scales [E,H] float, from moe_quantize_fp8 of the bf16 weights (rows =
 *   output channels); the other arguments as moe_layer_forward.
 * cfg->flags must include MOE_FLAG_FP8 (the workspace size depends on it); with
 * MOE_FLAG_FUSED_COMBINE the combine is done in the FP8 down projection as in
 * moe_layer_forward.  bf16 layers with H % 128 == 0 and I % 128 == 0 (else
 * MOE_ERR_UNSUPPORTED). */
moe_status_t moe_layer_forward_fp8(const moe_config_t* cfg, const void* x, const void* w_router,
                                   const float* router_bias, const uint8_t* w_gate_up_codes,
                                   const float* w_gate_up_scales, const uint8_t* w_down_codes,
                                   const float* w_down_scales, const void* w_shared_gate_up,
                                   const void* w_shared_down, void* y, float* y_f32, void* ws,
                                   size_t ws_bytes, moe_stream_t stream);

/* Per-row FP8 (E4M3) quantisation, for low-precision experts.
 * Defined by: "MoE大模型的智能调度…" §4.1 (the resident experts' weights are quantised to 8
 * bits to save memory).  Reading: E4M3, the 8-bit format the tensor cores run at full rate,
 * one float32 scale per row.  For every row r:
 *   scales[r] = max_c |in[r,c]| / 448 (1 for an all-zero row), float32;
 *   codes[r,c] = E4M3(in[r,c] * (1 / scales[r])) (the reciprocal and the product each
 *   rounded to float32, then round to nearest even, saturating at +-448), one byte each.
 *   in [rows, cols] bf16 (device); codes [rows, cols] uint8 out; scales [rows] float out.
 *   cols % 8 == 0; rows >= 0.  Expert weights quantise as rows = E*2I (gate/up, per output
 *   channel); token rows as rows = T*K (the permuted x). */
moe_status_t moe_quantize_fp8(const void* in, int64_t rows, int32_t cols, uint8_t* codes,
                              float* scales, moe_stream_t stream);

/* The gate/up projection on FP8 operands: moe_expert_gate_up with E4M3 codes and per-row
 * scales (see moe_quantize_fp8) in place of the bf16 activations and weights.
 * Defined by: page section "单机MoE执行流水线" (each expert's gate/up GEMM) and
 * "MoE大模型的智能调度…" §4.1 (8-bit expert weights).  For every row r of group e:
 *   g[r,n] = xs[r] * ws[e,n] * sum_k xq[r,k] wq[e,n,k] (fp32 accumulation of exact
 *   products), u likewise with the up rows I+n, h[r,n] = silu(g) * u rounded once to bf16.
 *   x_codes [T*K,H] uint8, x_scales [T*K] float; offsets [E+1] int32; w_codes [E,2I,H]
 *   uint8, w_scales [E,2I] float; h [T*K,I] bf16 out (rows >= offsets[E] untouched);
 *   ws as for moe_grouped_ffn.  bf16 layers only, H % 128 == 0 (else MOE_ERR_UNSUPPORTED). */
moe_status_t moe_expert_gate_up_fp8(const moe_config_t* cfg, const uint8_t* x_codes,
                                    const float* x_scales, const int32_t* offsets,
                                    const uint8_t* w_codes, const float* w_scales, void* h,
                                    void* ws, size_t ws_bytes, moe_stream_t stream);

/* The output projection on FP8 operands: moe_expert_down with E4M3 codes and per-row
 * scales (see moe_quantize_fp8): h quantised per row (T*K rows of I), W_d per output
 * channel (E*H rows of I).  For every row r of group e:
 *   out_perm[r,n] = hs[r] * ws[e,n] * sum_k hq[r,k] wq[e,n,k] (fp32 accumulation).
 *   h_codes [T*K,I] uint8, h_scales [T*K] float; offsets [E+1] int32; w_codes [E,H,I]
 *   uint8, w_scales [E,H] float; out_perm [T*K,H] float out (rows >= offsets[E]
 *   untouched); ws as for moe_grouped_ffn.  bf16 layers only, I % 128 == 0 (else
 *   MOE_ERR_UNSUPPORTED).
 * Defined by: page section "单机MoE执行流水线" (each expert's output projection) and
 * "MoE大模型的智能调度…" §4.1 (8-bit expert weights). */
moe_status_t moe_expert_down_fp8(const moe_config_t* cfg, const uint8_t* h_codes,
                                 const float* h_scales, const int32_t* offsets,
                                 const uint8_t* w_codes, const float* w_scales, float* out_perm,
                                 void* ws, size_t ws_bytes, moe_stream_t stream);

/* The second GEMM of the grouped FFN alone: the output projection.
 * Defined by: page section "单机MoE执行流水线" (each expert applies its output
 * projection).  For every row r of group e: out_perm[r] = h[r] W_d[e]^T (fp32).
 *   h [T*K,I] act in; offsets [E+1] int32 in; w_down [E,H,I] act;
 *   out_perm [T*K,H] float out (rows >= offsets[E] untouched); ws as above. */
moe_status_t moe_expert_down(const moe_config_t* cfg, const void* h, const int32_t* offsets,
                             const void* w_down, float* out_perm, void* ws, size_t ws_bytes,
                             moe_stream_t stream);

/* Un-permute and gated weighted sum back to token order.
 * Defined by: "MoE大模型的智能调度…" §2.2 fusion layer (output = sum of gate_i *
 * Expert_i(h)) and page sections "MoE层的结构与token路由" (y = sum over the selected
 * experts S(x) of w_e(x) E_e(x)) and "单机MoE执行流水线" (restore token order with the
 * inverse map, apply the route weights, add contributions of the same token id).
 *   y[t] = sum_{k=0..K-1, inv[t,k] >= 0} topk_w[t,k] * out_perm[inv[t,k]]  (+ shared_out[t])
 * summed in fp32 in slot order, then rounded once to `act`.
 *   out_perm   [T*K,H] float in;  inv [T*K] int32 in;  topk_w [T*K] float in.
 *   shared_out [T,H] float in or NULL.
 *   y          [T,H] act out.
 *   y_f32      [T,H] float out (the fp32 sum before rounding) or NULL. */
moe_status_t moe_combine(const moe_config_t* cfg, const float* out_perm, const int32_t* inv,
                         const float* topk_w, const float* shared_out, void* y, float* y_f32,
                         moe_stream_t stream);

/* The whole layer: moe_route -> moe_permute -> moe_grouped_ffn -> (shared expert) ->
 * moe_combine, on one stream, with every intermediate in `ws`.
 * The shared expert (page section "MoE层的结构与token路由": not scored by the router, run
 * for every token) is a SwiGLU FFN of size I_shared added with weight 1.
 *   x [T,H] act; w_router [E,H] act; router_bias [E] float or NULL;
 *   w_gate_up [E,2I,H] act; w_down [E,H,I] act;
 *   w_shared_gate_up [2*I_shared,H] act and w_shared_down [H,I_shared] act, both NULL
 *   when I_shared == 0;
 *   y [T,H] act out; y_f32 [T,H] float out or NULL;
 *   ws workspace of at least moe_workspace_size() bytes.
 * Batches of 1024 tokens or more with a shared expert run it on a stream the library owns
 * (one per device, created by the first such call), concurrently with the dispatch and the
 * routed gate/up GEMM; `stream` waits for it before the routed down projection, so work
 * the caller enqueues on `stream` afterwards sees the whole layer, as with one stream.
 * While `stream` is being captured into a CUDA graph the layer runs in stream order. */
moe_status_t moe_layer_forward(const moe_config_t* cfg, const void* x, const void* w_router,
                               const float* router_bias, const void* w_gate_up,
                               const void* w_down, const void* w_shared_gate_up,
                               const void* w_shared_down, void* y, float* y_f32, void* ws,
                               size_t ws_bytes, moe_stream_t stream);

/* Intermediates of the last moe_layer_forward that used `ws` (views into ws; valid
 * until ws is reused).  Any output pointer may be NULL.  Useful to check every stage.
 * x_perm is not written by decode-sized bf16 layers (T <= 16, E <= 256, K <= 16), whose
 * gate/up GEMM gathers token rows from x through perm instead; out_perm is not written
 * with MOE_FLAG_FUSED_COMBINE. */
moe_status_t moe_workspace_views(const moe_config_t* cfg, void* ws, float** logits,
                                 int32_t** topk_ids, float** topk_w, int32_t** counts,
                                 int32_t** offsets, int32_t** perm, int32_t** inv,
                                 void** x_perm, float** out_perm, float** shared_out);

/* Synchronise `stream` and report (then clear) the device error word of the current
 * device: MOE_ERR_TIMEOUT if a bounded device-side wait gave up since the last check,
 * MOE_ERR_INTERNAL if a kernel of the debug build (compiled with -DMOE_DEBUG) found an
 * index out of range in its inputs (an expert id >= E, group offsets that decrease or
 * exceed the rows, an inverse-map or gather row out of range) and skipped that access,
 * MOE_ERR_CUDA if the stream reports a CUDA error, MOE_OK otherwise. */
moe_status_t moe_sync_check(moe_stream_t stream);

/* Failure-handling self-test (no counterpart on the pages).  Launches one thread that
 * waits, through the library's bounded device-side wait, on an mbarrier that nothing
 * arrives at.  After `limit_us` microseconds (1..1e6) the wait gives up.  The kernel then
 * stores 2 to *done (1 would mean the wait completed) and records MOE_ERR_TIMEOUT in the
 * device error word, which the next moe_sync_check() reports and clears.  The kernel
 * exits normally, so the CUDA context stays usable.  `done` is an int in device memory. */
moe_status_t moe_debug_wait_timeout(unsigned limit_us, int* done, moe_stream_t stream);

/* Host-side fault injection, for testing how a caller handles errors (no counterpart on
 * the pages: section 3.2 of "MoE大模型的智能调度…" recounts production failures of the
 * routing step, one an out-of-memory crash; this lets a caller rehearse its clean-up
 * after a failed call without causing a real failure).
 * Arms one fault: the n-th time (n >= 1, counted from this call) the library passes the
 * named point, the call returns MOE_ERR_CUDA there, as a failed launch would, and the
 * fault disarms itself.  point == NULL or n <= 0 disarms.  Returns MOE_ERR_INVALID_ARG
 * for an unknown point.  The same fault can be armed when the library loads by setting
 * MOE_FAULT=<point>:<n> in the environment.  Points:
 *  - every entry point by its own name ("moe_route", "moe_layer_forward", ...,
 *    "moe_workspace_size", "moe_sync_check"): checked first, before any argument check,
 *    so nothing is launched and no output is written;
 *  - the stages inside moe_layer_forward: "moe_layer_forward.route", ".permute",
 *    ".gate_up", ".shared", ".down", ".combine": checked before that stage's launches, so
 *    the earlier stages have been enqueued on the stream.  y is then untouched; the
 *    workspace (and y_f32 with MOE_FLAG_FUSED_COMBINE) may hold partial results.
 * Thread-safe; the fault is process-wide.  No GPU state is involved. */
moe_status_t moe_debug_set_fault(const char* point, int n);

/* Number of kernels this library has launched in this process, on every device: each
 * launch the CUDA runtime accepted counts once.  A launch issued while a stream is being
 * captured into a CUDA graph counts once, at capture; replays of the graph are not
 * counted.  Memset and copy operations are not kernels of this library and do not count.
 * No counterpart on the pages: a diagnostic for callers that check which work ran. */
unsigned long long moe_kernel_launch_count(void);

/* Static, human-readable name of a status code. */
const char* moe_status_string(moe_status_t status);

/* Library version string ("moe_gb300 <major>.<minor> sm_103a"). */
const char* moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_MOE_H */
