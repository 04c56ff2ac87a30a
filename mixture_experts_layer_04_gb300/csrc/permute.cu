// Dispatch kernels: the stable counting-sort permutation of the assignments and the
// row gather.
//
// Page opening "MoE通过稀疏激活降低每个token的计算量但增加了服务系统的复杂度", section
// "一个批次如何变成各专家专属的矩阵": each (token, expert, weight) assignment is grouped by
// expert into a matrix whose rows keep their source token id; section "单机MoE执行流水线":
// the permutation reads token vectors, writes them in expert order and records an
// inverse map for the combine.  Rows inside a group are in ascending token order, so
// the result does not depend on the order in which threads run.
//
// Three launches:
//   1. rank:    per block of 256 tokens, the rank of every assignment among the
//               block's assignments to the same expert (shared-memory bit masks, one
//               32-bit mask per warp and expert; rank = popcount of lower lanes), and
//               the block's per-expert counts.
//   2. scan:    one block: per-expert totals, the exclusive scan `offsets`, every
//               block's base row per expert, and the m-tile table of the grouped GEMM.
//   3. scatter: one warp per token: row = base + rank, inv/perm, and the 16-byte
//               vectorised copy of the token row to each of its K rows.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kRankTokens = 256;  // tokens per rank block (8 warps x 32 lanes)
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kRankTokens)
    permute_rank_kernel(const int32_t* __restrict__ ids, int T, int E, int K,
                        int32_t* __restrict__ rank_out, int32_t* __restrict__ block_counts,
                        unsigned* __restrict__ err) {
  extern __shared__ uint32_t masks[];  // [8][E]
  grid_dep_wait();
  grid_dep_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 8 * E; i += kRankTokens) masks[i] = 0u;
  __syncthreads();
  const int t = blockIdx.x * kRankTokens + tid;
  if (t < T) {
    for (int k = 0; k < K; ++k) {
      const int e = ids[static_cast<size_t>(t) * K + k];
      if (e >= 0 && dcheck(e < E, err)) atomicOr(&masks[warp * E + e], 1u << lane);
    }
  }
  __syncthreads();
  if (t < T) {
    const uint32_t lower = (1u << lane) - 1u;
    for (int k = 0; k < K; ++k) {
      const int e = ids[static_cast<size_t>(t) * K + k];
      int r = -1;
      if (e >= 0 && dcheck(e < E, nullptr)) {
        r = __popc(masks[warp * E + e] & lower);
        for (int w = 0; w < warp; ++w) r += __popc(masks[w * E + e]);
      }
      rank_out[static_cast<size_t>(t) * K + k] = r;
    }
  }
  for (int e = tid; e < E; e += kRankTokens) {
    int c = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) c += __popc(masks[w * E + e]);
    block_counts[static_cast<size_t>(blockIdx.x) * E + e] = c;
  }
}

// Writes the m-tile entries of expert e (count rows starting at row `base`).
__device__ void write_mtiles(int4* table, int e, int base, int count, int first, int bm) {
  const int nt = (count + bm - 1) / bm;
  for (int j = 0; j < nt; ++j) table[first + j] = make_int4(e, base + j * bm, base + count, 0);
}

__global__ void __launch_bounds__(kScanThreads)
    permute_scan_kernel(int32_t* __restrict__ block_counts, int nblocks, int E,
                        int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                        int4* __restrict__ mtile_table, int32_t* __restrict__ num_mtiles, int bm,
                        int32_t* __restrict__ zero_word) {
  __shared__ int scratch[32];
  grid_dep_wait();
  grid_dep_trigger();
  const int e = threadIdx.x;
  if (zero_word != nullptr && e == 0) *zero_word = 0;
  constexpr int kChunk = 16;  // counts loaded at once (independent loads in flight)
  // pass 1: the expert's total over all rank blocks
  int total = 0;
  if (e < E) {
    for (int b0 = 0; b0 < nblocks; b0 += kChunk) {
      int c[kChunk];
#pragma unroll
      for (int j = 0; j < kChunk; ++j)
        c[j] = b0 + j < nblocks ? block_counts[static_cast<size_t>(b0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < kChunk; ++j) total += c[j];
    }
  }
  int M = 0;
  const int base = block_exclusive_scan(total, scratch, &M);
  // pass 2: each block's count becomes its first row of the expert's group
  if (e < E) {
    counts[e] = total;
    offsets[e] = base;
    int run = base;
    for (int b0 = 0; b0 < nblocks; b0 += kChunk) {
      int c[kChunk];
#pragma unroll
      for (int j = 0; j < kChunk; ++j)
        c[j] = b0 + j < nblocks ? block_counts[static_cast<size_t>(b0 + j) * E + e] : 0;
#pragma unroll
      for (int j = 0; j < kChunk; ++j) {
        if (b0 + j < nblocks) block_counts[static_cast<size_t>(b0 + j) * E + e] = run;
        run += c[j];
      }
    }
  }
  if (e == 0) offsets[E] = M;
  if (mtile_table != nullptr) {
    const int nt = e < E ? (total + bm - 1) / bm : 0;
    int all = 0;
    const int first = block_exclusive_scan(nt, scratch, &all);
    if (e < E) write_mtiles(mtile_table, e, base, total, first, bm);
    if (e == 0) *num_mtiles = all;
  }
}

__global__ void __launch_bounds__(kScanThreads)
    mtile_table_kernel(const int32_t* __restrict__ offsets, int E, int rows,
                       int4* __restrict__ table, int32_t* __restrict__ num_mtiles, int bm,
                       unsigned* __restrict__ err) {
  __shared__ int scratch[32];
  grid_dep_wait();
  grid_dep_trigger();
  const int e = threadIdx.x;
  const int base = e < E ? offsets[e] : 0;
  const int count = e < E ? offsets[e + 1] - base : 0;
#ifdef MOE_DEBUG
  // offsets must be non-decreasing within [0, rows]: otherwise no tile is emitted
  const bool bad = e < E && (base < 0 || count < 0 || base + count > rows);
  if (__syncthreads_or(bad)) {
    if (e == 0) {
      report_error(err, MOE_DEVERR_BOUNDS);
      *num_mtiles = 0;
    }
    return;
  }
#else
  (void)rows;
  (void)err;
#endif
  const int nt = (count + bm - 1) / bm;
  int all = 0;
  const int first = block_exclusive_scan(nt, scratch, &all);
  if (e < E) write_mtiles(table, e, base, count, first, bm);
  if (e == 0) *num_mtiles = all;
}

constexpr int kScatterWarps = 8;

__global__ void __launch_bounds__(kScatterWarps * 32)
    permute_scatter_kernel(const int32_t* __restrict__ ids,
                           const int32_t* __restrict__ block_base, int T, int E, int K,
                           int row_units, int32_t* __restrict__ inv, int32_t* __restrict__ perm,
                           const uint4* __restrict__ x, uint4* __restrict__ x_perm,
                           const float* __restrict__ gate_w, float* __restrict__ row_w) {
  grid_dep_wait();
  grid_dep_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kScatterWarps + warp;
  if (t >= T) return;
  int row = -1;
  if (lane < K) {
    const int e = ids[static_cast<size_t>(t) * K + lane];
    if (e >= 0 && dcheck(e < E, nullptr)) {  // an id out of range was reported by the rank pass
      const int b = t / kRankTokens;
      row = block_base[static_cast<size_t>(b) * E + e] + inv[static_cast<size_t>(t) * K + lane];
      inv[static_cast<size_t>(t) * K + lane] = row;
      perm[row] = t;
      if (row_w != nullptr) row_w[row] = gate_w[static_cast<size_t>(t) * K + lane];
    }
  }
  // The token row is read once (bursts of 8 independent 16-byte loads per lane) and
  // written to each of its K destination rows.
  const uint4* src = x + static_cast<size_t>(t) * row_units;
  constexpr int kBurst = 8;
  for (int i0 = 0; i0 < row_units; i0 += 32 * kBurst) {
    uint4 v[kBurst];
#pragma unroll
    for (int b = 0; b < kBurst; ++b) {
      const int i = i0 + b * 32 + lane;
      if (i < row_units) v[b] = __ldg(src + i);
    }
    for (int k = 0; k < K; ++k) {
      const int r = __shfl_sync(0xffffffffu, row, k);
      if (r < 0) continue;
      uint4* dst = x_perm + static_cast<size_t>(r) * row_units;
#pragma unroll
      for (int b = 0; b < kBurst; ++b) {
        const int i = i0 + b * 32 + lane;
        if (i < row_units) dst[i] = v[b];
      }
    }
  }
}

constexpr int kSmallThreads = 1024;

struct SmallRoute {
  const float* partial;  // [S][T][E] router partial logits
  int S;
  const float* bias;
  float* logits;         // [T][E] out
  int32_t* ids_out;      // [T][K] out
  float* w_out;          // [T][K] out
  float theta;
};
constexpr int kSmallMaxT = 256;                 // token bit masks of 8 words per expert
constexpr int kSmallMaskWords = kSmallMaxT / 32;
constexpr int kSmallFusedMaxT = 64;                // routing fused into the permutation

// The whole permutation in one launch for small batches (T <= 256).  Every block
// recomputes the (cheap) index math of all T*K assignments in shared memory -- counts by
// shared atomics, offsets by a block scan, ranks from per-expert token bit masks -- so no
// block depends on another; block 0 stores counts/offsets/perm/inv (and the m-tile table
// when asked), and every block copies its share of the rows into x_perm, one warp per row.
template <bool kRoute>
__global__ void __launch_bounds__(kSmallThreads)
    permute_small_kernel(const int32_t* __restrict__ ids_in, SmallRoute rt, int T, int E, int K,
                         int row_units, int32_t* __restrict__ counts,
                         int32_t* __restrict__ offsets, int32_t* __restrict__ perm,
                         int32_t* __restrict__ inv, const uint4* __restrict__ x,
                         uint4* __restrict__ x_perm, int4* __restrict__ mtile_table,
                         int32_t* __restrict__ num_mtiles, int bm,
                         const float* __restrict__ gate_w, float* __restrict__ row_w,
                         unsigned* __restrict__ err, int32_t* __restrict__ zero_word) {
  extern __shared__ uint32_t smem_u[];
  uint32_t* masks = smem_u;                                        // [E][8]
  int* cnt = reinterpret_cast<int*>(masks + E * kSmallMaskWords);  // [E]
  int* off = cnt + E;                                              // [E+1]
  int* rows = off + E + 1;                                         // [T*K]
  __shared__ int scratch[32];
  grid_dep_wait();
  grid_dep_trigger();
  const int tid = threadIdx.x;
  if (zero_word != nullptr && blockIdx.x == 0 && tid == 0) *zero_word = 0;
  const int TK = T * K;
  const int32_t* ids = ids_in;
  const float* gates = gate_w;
  if constexpr (kRoute) {
    // routing of all T tokens (every block computes it; block 0 stores it): logits = sum
    // of the router's H-slice partials in slice order + bias, then the warp top-k
    float* Ls = reinterpret_cast<float*>(rows + TK);     // [T][E]
    int32_t* sids = reinterpret_cast<int32_t*>(Ls + T * E);  // [T*K]
    float* sw = reinterpret_cast<float*>(sids + TK);     // [T*K]
    for (int i = tid; i < T * E; i += blockDim.x) {
      float v = 0.f;
      for (int s0 = 0; s0 < rt.S; s0 += 8) {  // 8 slice loads in flight, summed in order
        float q[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          q[j] = s0 + j < rt.S ? rt.partial[static_cast<size_t>(s0 + j) * T * E + i] : 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (s0 + j < rt.S) v += q[j];
      }
      if (rt.bias != nullptr) v += rt.bias[i % E];
      Ls[i] = v;
      if (blockIdx.x == 0) rt.logits[i] = v;
    }
    __syncthreads();
    const int nwarps = blockDim.x >> 5;
    for (int t = tid >> 5; t < T; t += nwarps)
      warp_topk_softmax(Ls + t * E, E, K, rt.theta, sids + t * K, sw + t * K);
    __syncthreads();
    if (blockIdx.x == 0)
      for (int i = tid; i < TK; i += blockDim.x) {
        rt.ids_out[i] = sids[i];
        rt.w_out[i] = sw[i];
      }
    ids = sids;
    gates = sw;
  }
  for (int i = tid; i < E * kSmallMaskWords; i += blockDim.x) masks[i] = 0u;
  __syncthreads();
  for (int a = tid; a < TK; a += blockDim.x) {
    const int e = ids[a];
    if (e >= 0 && dcheck(e < E, blockIdx.x == 0 ? err : nullptr)) {
      const int t = a / K;
      atomicOr(&masks[e * kSmallMaskWords + (t >> 5)], 1u << (t & 31));
    }
  }
  __syncthreads();
  int c = 0;
  if (tid < E) {
#pragma unroll
    for (int w = 0; w < kSmallMaskWords; ++w) c += __popc(masks[tid * kSmallMaskWords + w]);
  }
  int M = 0;
  const int base = block_exclusive_scan(tid < E ? c : 0, scratch, &M);
  if (tid < E) {
    cnt[tid] = c;
    off[tid] = base;
  }
  if (tid == 0) off[E] = M;
  __syncthreads();
  for (int a = tid; a < TK; a += blockDim.x) {
    const int e = ids[a];
    int row = -1;
    if (e >= 0 && dcheck(e < E, nullptr)) {
      const int t = a / K;
      const uint32_t* m = masks + e * kSmallMaskWords;
      int r = __popc(m[t >> 5] & ((1u << (t & 31)) - 1u));
      for (int w = 0; w < (t >> 5); ++w) r += __popc(m[w]);
      row = off[e] + r;
    }
    rows[a] = row;
  }
  __syncthreads();
  if (blockIdx.x == 0) {
    if (tid < E) counts[tid] = cnt[tid];
    for (int i = tid; i <= E; i += blockDim.x) offsets[i] = off[i];
    for (int a = tid; a < TK; a += blockDim.x) {
      inv[a] = rows[a];
      if (rows[a] >= 0) {
        perm[rows[a]] = a / K;
        if (row_w != nullptr) row_w[rows[a]] = gates[a];
      }
    }
    if (mtile_table != nullptr) {
      const int nt = tid < E ? (cnt[tid] + bm - 1) / bm : 0;
      int all = 0;
      const int first = block_exclusive_scan(nt, scratch, &all);
      if (tid < E)
        for (int j = 0; j < nt; ++j)
          mtile_table[first + j] = make_int4(tid, off[tid] + j * bm, off[tid] + cnt[tid], 0);
      if (tid == 0) *num_mtiles = all;
    }
  }
  // row copies: assignment a -> x_perm[rows[a]] = x[a / K], one warp per assignment,
  // each lane with 8 independent 16-byte loads in flight before its stores
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int kBurst = 8;
  for (int a = blockIdx.x * (kSmallThreads / 32) + warp; a < TK;
       a += gridDim.x * (kSmallThreads / 32)) {
    const int r = rows[a];
    if (r < 0) continue;
    const uint4* src = x + static_cast<size_t>(a / K) * row_units;
    uint4* dst = x_perm + static_cast<size_t>(r) * row_units;
    for (int i0 = 0; i0 < row_units; i0 += 32 * kBurst) {
      uint4 v[kBurst];
#pragma unroll
      for (int b = 0; b < kBurst; ++b) {
        const int i = i0 + b * 32 + lane;
        if (i < row_units) v[b] = __ldg(src + i);
      }
#pragma unroll
      for (int b = 0; b < kBurst; ++b) {
        const int i = i0 + b * 32 + lane;
        if (i < row_units) dst[i] = v[b];
      }
    }
  }
}


size_t small_smem_bytes(int T, int E, int K, bool route) {
  size_t b = static_cast<size_t>(E) * kSmallMaskWords * 4 + (2 * E + 1) * 4 +
             static_cast<size_t>(T) * K * 4;
  if (route) b += static_cast<size_t>(T) * E * 4 + static_cast<size_t>(T) * K * 8;
  return b;
}

constexpr size_t kSmallMaxSmem = 200 * 1024;

template <bool kRoute>
cudaError_t launch_small_t(int dtype, const void* x, const int32_t* ids, const SmallRoute* rt,
                           int T, int H, int E, int K, int32_t* counts, int32_t* offsets,
                           int32_t* perm, int32_t* inv, void* x_perm, int4* mtile_table,
                           int32_t* num_mtiles, int bm, const float* gate_w, float* row_w,
                           int32_t* zero_word, cudaStream_t s) {
  static int attr_dev = -1;  // opt in to more than 48 KB of dynamic shared memory once
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(permute_small_kernel<kRoute>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmallMaxSmem));
    if (e != cudaSuccess) return e;
    attr_dev = dev;
  }
  const size_t smem = small_smem_bytes(T, E, K, kRoute);
  if (smem > kSmallMaxSmem) return cudaErrorInvalidValue;
  const int row_units = static_cast<int>(static_cast<size_t>(H) * act_bytes(dtype) / 16);
  int blocks = (T * K + 31) / 32;
  blocks = blocks < 148 ? blocks : 148;
  SmallRoute r{};
  if (rt != nullptr) r = *rt;
  return launch_pdl(permute_small_kernel<kRoute>, dim3(blocks), dim3(kSmallThreads), smem, s, ids,
                    r, T, E, K, row_units, counts, offsets, perm, inv,
                    static_cast<const uint4*>(x), static_cast<uint4*>(x_perm), mtile_table,
                    num_mtiles, bm, gate_w, row_w, device_error_word(), zero_word);
}

cudaError_t launch_small(int dtype, const void* x, const int32_t* ids, const SmallRoute* rt,
                         int T, int H, int E, int K, int32_t* counts, int32_t* offsets,
                         int32_t* perm, int32_t* inv, void* x_perm, int4* mtile_table,
                         int32_t* num_mtiles, int bm, const float* gate_w, float* row_w,
                         int32_t* zero_word, cudaStream_t s) {
  if (rt != nullptr)
    return launch_small_t<true>(dtype, x, ids, rt, T, H, E, K, counts, offsets, perm, inv, x_perm,
                                mtile_table, num_mtiles, bm, gate_w, row_w, zero_word, s);
  return launch_small_t<false>(dtype, x, ids, rt, T, H, E, K, counts, offsets, perm, inv, x_perm,
                               mtile_table, num_mtiles, bm, gate_w, row_w, zero_word, s);
}

}  // namespace

bool topk_permute_fusable(int T, int E, int K) {
  return T > 0 && T <= kSmallFusedMaxT && small_smem_bytes(T, E, K, true) <= kSmallMaxSmem;
}

cudaError_t launch_topk_permute_small(const float* partial, int S, const float* bias,
                                      float* logits, int32_t* ids, float* w, float theta,
                                      int dtype, const void* x, int T, int H, int E, int K,
                                      int32_t* counts, int32_t* offsets, int32_t* perm,
                                      int32_t* inv, void* x_perm, int4* mtile_table,
                                      int32_t* num_mtiles, int bm, float* row_w, cudaStream_t s,
                                      int32_t* zero_word) {
  SmallRoute rt{partial, S, bias, logits, ids, w, theta};
  return launch_small(dtype, x, nullptr, &rt, T, H, E, K, counts, offsets, perm, inv, x_perm,
                      mtile_table, num_mtiles, bm, nullptr, row_w, zero_word, s);
}

size_t permute_ws_words(int T, int E) {
  const size_t nb = (static_cast<size_t>(T) + kRankTokens - 1) / kRankTokens;
  return nb * static_cast<size_t>(E);
}

cudaError_t launch_permute(int dtype, const void* x, const int32_t* ids, int T, int H, int E,
                           int K, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                           void* x_perm, int32_t* ws_words, int4* mtile_table,
                           int32_t* num_mtiles, int bm, const float* gate_w, float* row_w,
                           cudaStream_t s, int32_t* zero_word) {
  if (T > 0 && T <= kSmallMaxT)
    return launch_small(dtype, x, ids, nullptr, T, H, E, K, counts, offsets, perm, inv, x_perm,
                        mtile_table, num_mtiles, bm, gate_w, row_w, zero_word, s);
  const int nb = (T + kRankTokens - 1) / kRankTokens;
  if (nb > 0) {
    cudaError_t err = launch_pdl(permute_rank_kernel, dim3(nb), dim3(kRankTokens),
                                 8 * E * sizeof(uint32_t), s, ids, T, E, K, inv, ws_words,
                                 device_error_word());
    if (err != cudaSuccess) return err;
  }
  cudaError_t err = launch_pdl(permute_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, ws_words,
                               nb, E, counts, offsets, mtile_table, num_mtiles, bm, zero_word);
  if (err != cudaSuccess || T == 0) return err;
  const int row_units = static_cast<int>(static_cast<size_t>(H) * act_bytes(dtype) / 16);
  return launch_pdl(permute_scatter_kernel, dim3((T + kScatterWarps - 1) / kScatterWarps),
                    dim3(kScatterWarps * 32), 0, s, ids, static_cast<const int32_t*>(ws_words), T,
                    E, K, row_units, inv, perm, static_cast<const uint4*>(x),
                    static_cast<uint4*>(x_perm), gate_w, row_w);
}

cudaError_t launch_build_mtile_table(const int32_t* offsets, int E, int rows, int bm,
                                     int4* table, int32_t* num_mtiles, cudaStream_t s) {
  return launch_pdl(mtile_table_kernel, dim3(1), dim3(kScanThreads), 0, s, offsets, E, rows,
                    table, num_mtiles, bm, device_error_word());
}

}  // namespace moe
