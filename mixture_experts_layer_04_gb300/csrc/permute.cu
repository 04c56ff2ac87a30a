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

namespace moe {
namespace {

constexpr int kRankTokens = 256;  // tokens per rank block (8 warps x 32 lanes)
constexpr int kScanThreads = 1024;

__global__ void __launch_bounds__(kRankTokens)
    permute_rank_kernel(const int32_t* __restrict__ ids, int T, int E, int K,
                        int32_t* __restrict__ rank_out, int32_t* __restrict__ block_counts) {
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
      if (e >= 0) atomicOr(&masks[warp * E + e], 1u << lane);
    }
  }
  __syncthreads();
  if (t < T) {
    const uint32_t lower = (1u << lane) - 1u;
    for (int k = 0; k < K; ++k) {
      const int e = ids[static_cast<size_t>(t) * K + k];
      int r = -1;
      if (e >= 0) {
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
                        int4* __restrict__ mtile_table, int32_t* __restrict__ num_mtiles, int bm) {
  __shared__ int scratch[32];
  grid_dep_wait();
  grid_dep_trigger();
  const int e = threadIdx.x;
  int total = 0;
  if (e < E) {
    for (int b = 0; b < nblocks; ++b) {
      const int c = block_counts[static_cast<size_t>(b) * E + e];
      block_counts[static_cast<size_t>(b) * E + e] = total;
      total += c;
    }
  }
  int M = 0;
  const int base = block_exclusive_scan(total, scratch, &M);
  if (e < E) {
    counts[e] = total;
    offsets[e] = base;
    for (int b = 0; b < nblocks; ++b) block_counts[static_cast<size_t>(b) * E + e] += base;
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
    mtile_table_kernel(const int32_t* __restrict__ offsets, int E, int4* __restrict__ table,
                       int32_t* __restrict__ num_mtiles, int bm) {
  __shared__ int scratch[32];
  grid_dep_wait();
  grid_dep_trigger();
  const int e = threadIdx.x;
  const int base = e < E ? offsets[e] : 0;
  const int count = e < E ? offsets[e + 1] - base : 0;
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
                           const uint4* __restrict__ x, uint4* __restrict__ x_perm) {
  grid_dep_wait();
  grid_dep_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kScatterWarps + warp;
  if (t >= T) return;
  int row = -1;
  if (lane < K) {
    const int e = ids[static_cast<size_t>(t) * K + lane];
    if (e >= 0) {
      const int b = t / kRankTokens;
      row = block_base[static_cast<size_t>(b) * E + e] + inv[static_cast<size_t>(t) * K + lane];
      inv[static_cast<size_t>(t) * K + lane] = row;
      perm[row] = t;
    }
  }
  const uint4* src = x + static_cast<size_t>(t) * row_units;
  for (int k = 0; k < K; ++k) {
    const int r = __shfl_sync(0xffffffffu, row, k);
    if (r < 0) continue;
    uint4* dst = x_perm + static_cast<size_t>(r) * row_units;
    for (int i = lane; i < row_units; i += 32) dst[i] = src[i];
  }
}

}  // namespace

size_t permute_ws_words(int T, int E) {
  const size_t nb = (static_cast<size_t>(T) + kRankTokens - 1) / kRankTokens;
  return nb * static_cast<size_t>(E);
}

cudaError_t launch_permute(int dtype, const void* x, const int32_t* ids, int T, int H, int E,
                           int K, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* inv,
                           void* x_perm, int32_t* ws_words, int4* mtile_table,
                           int32_t* num_mtiles, int bm, cudaStream_t s) {
  const int nb = (T + kRankTokens - 1) / kRankTokens;
  if (nb > 0) {
    cudaError_t err = launch_pdl(permute_rank_kernel, dim3(nb), dim3(kRankTokens),
                                 8 * E * sizeof(uint32_t), s, ids, T, E, K, inv, ws_words);
    if (err != cudaSuccess) return err;
  }
  cudaError_t err = launch_pdl(permute_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, ws_words,
                               nb, E, counts, offsets, mtile_table, num_mtiles, bm);
  if (err != cudaSuccess || T == 0) return err;
  const int row_units = static_cast<int>(static_cast<size_t>(H) * act_bytes(dtype) / 16);
  return launch_pdl(permute_scatter_kernel, dim3((T + kScatterWarps - 1) / kScatterWarps),
                    dim3(kScatterWarps * 32), 0, s, ids, static_cast<const int32_t*>(ws_words), T,
                    E, K, row_units, inv, perm, static_cast<const uint4*>(x),
                    static_cast<uint4*>(x_perm));
}

cudaError_t launch_build_mtile_table(const int32_t* offsets, int E, int bm, int4* table,
                                     int32_t* num_mtiles, cudaStream_t s) {
  return launch_pdl(mtile_table_kernel, dim3(1), dim3(kScanThreads), 0, s, offsets, E, table,
                    num_mtiles, bm);
}

}  // namespace moe
