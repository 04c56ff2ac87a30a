// Capacity-limited routing.
//
// "MoE大模型的智能调度：从1.8万亿参数到每token仅激活2%的工程真相" §3.2, trap 2: a capacity
// check goes into routing, capacity = (batch_size * seq_len * k) / num_experts * 1.2, and an
// expert chosen that many times gets logit -inf so that the token chooses again.  Tokens are
// routed in token order: an expert is available to token t while fewer than `cap` kept
// assignments of earlier tokens (after their gate drop) went to it, and t takes its top-k of
// the available experts (softmax over them, then the gate drop; missing slots -1).
//
// The rule is sequential in t, but each token depends on earlier tokens only through, per
// expert, the index of the token that takes its last free place.  One CTA sweeps the batch in
// blocks of 256 tokens with the exact counts of the earlier blocks.  Inside a block it
// iterates to a fixed point: fb[e] = the block token holding e's (cap - count[e])-th kept
// assignment under the current choices, and every token whose availability changed chooses
// again among the experts with count[e] < cap and fb[e] >= its index.  Token 0 of the block is
// final after the first pass and each pass fixes at least the next token, so the fixed point
// (the sequential routing) is reached within 257 passes; in practice in a few.  Tokens that no
// capacity touches keep the router's choice.  No global scratch, no atomics on global memory:
// the result is deterministic.
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kCapThreads = 1024;
constexpr int kCapWarps = kCapThreads / 32;
constexpr int kCapBlock = 256;              // tokens per block of the sweep
constexpr int kCapWords = kCapBlock / 32;   // token bits per expert
constexpr int kNone = kCapBlock;            // fb value: the expert does not fill in the block

// Position of the n-th (0-based) set bit of v (n < popc(v)).
__device__ __forceinline__ int nth_set_bit(uint32_t v, int n) {
  for (int i = 0; i < n; ++i) v &= v - 1u;
  return __ffs(v) - 1;
}

// Inverse of float_key (the key of -0 gives +0, which the softmax cannot tell apart).
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <int NJ>  // candidates per lane: experts lane + 32 j, j < NJ (E <= 32 NJ)
__device__ __forceinline__ void masked_topk_t(const float* __restrict__ L, int E, int K,
                                              float theta, int tl, const int* cnt, const int* fb, int cap,
                                              int32_t* ids, float* w) {
  const int lane = threadIdx.x & 31;
  uint32_t key[NJ];
  uint32_t live = 0u;  // bit j: expert lane + 32 j is available
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    key[j] = 0u;
    if (e < E && cnt[e] < cap && fb[e] >= tl) {
      key[j] = float_key(L[e]);
      live |= 1u << j;
    }
  }
  float my_v = 0.f, v0 = 0.f;
  int my_e = -1, nsel = 0;
  for (int k = 0; k < K; ++k) {
    uint32_t kbest = 0u, ebest = 0xffffffffu;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (((live >> j) & 1u) && (key[j] > kbest || ebest == 0xffffffffu)) {
        kbest = key[j];
        ebest = static_cast<uint32_t>(lane + 32 * j);
      }
    }
    const bool has = ebest != 0xffffffffu;
    if (!__any_sync(0xffffffffu, has)) break;
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, has ? kbest : 0u);
    const int e_win = static_cast<int>(
        __reduce_min_sync(0xffffffffu, (has && kbest == kmax) ? ebest : 0xffffffffu));
    if ((e_win & 31) == lane) live &= ~(1u << (e_win >> 5));
    const float v_win = key_float(kmax);
    if (k == 0) v0 = v_win;
    if (lane == k) {
      my_v = v_win;
      my_e = e_win;
    }
    ++nsel;
  }
  float z = (lane < nsel) ? expf(my_v - v0) : 0.f;
  float g = nsel > 0 ? z / warp_sum(z) : 0.f;
  if (theta > 0.f && nsel > 0) {
    if (lane >= 1 && lane < nsel && g < theta) {
      g = 0.f;
      my_e = -1;
    }
    g = g / warp_sum(g);
  }
  if (lane < K) {
    ids[lane] = lane < nsel ? my_e : -1;
    w[lane] = lane < nsel ? g : 0.f;
  }
}

// One warp: token `tl` of the block (logits row L) takes its top-k among the available experts
// (count < cap and fb >= tl), with the softmax and gate drop of the warp top-k (same sums in
// the same order), and writes its K slots to ids/w (dropped or missing slots -1 / 0).  The
// candidates' keys are loaded once and kept in registers.
__device__ __forceinline__ void masked_topk(const float* __restrict__ L, int E, int K, float theta,
                                            int tl, const int* cnt, const int* fb, int cap,
                                            int32_t* ids, float* w) {
  if (E <= 128)
    masked_topk_t<4>(L, E, K, theta, tl, cnt, fb, cap, ids, w);
  else if (E <= 256)
    masked_topk_t<8>(L, E, K, theta, tl, cnt, fb, cap, ids, w);
  else
    masked_topk_t<32>(L, E, K, theta, tl, cnt, fb, cap, ids, w);
}

__global__ void __launch_bounds__(kCapThreads, 1)
    capacity_route_kernel(const float* __restrict__ logits, int32_t* __restrict__ ids,
                          float* __restrict__ w, int T, int E, int K, float theta, int cap,
                          unsigned* err) {
  extern __shared__ int smem_i[];
  int* cnt = smem_i;                                        // [E] kept before the block
  int* fb = cnt + E;                                        // [E]
  uint32_t* mask = reinterpret_cast<uint32_t*>(fb + E);     // [E][kCapWords]
  int32_t* bid = reinterpret_cast<int32_t*>(mask + E * kCapWords);  // [kCapBlock * K]
  float* bw = reinterpret_cast<float*>(bid + kCapBlock * K);        // [kCapBlock * K]
  int* chg = reinterpret_cast<int*>(bw + kCapBlock * K);           // [3 * E]: e, old, new fb
  __shared__ int s_nchg;
  __shared__ int s_dirty[kCapBlock];

  grid_dep_wait();  // the router's logits and choices
  grid_dep_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < E; e += kCapThreads) cnt[e] = 0;
  for (int t0 = 0; t0 < T; t0 += kCapBlock) {
    const int nb = min(kCapBlock, T - t0);
    for (int i = tid; i < nb * K; i += kCapThreads) {
      bid[i] = ids[static_cast<size_t>(t0) * K + i];
      bw[i] = w[static_cast<size_t>(t0) * K + i];
    }
    for (int e = tid; e < E; e += kCapThreads) fb[e] = kNone;
    __syncthreads();
    for (int pass = 0;; ++pass) {
      // 1. tokens whose available set may have changed choose again.  First pass: with a
      //    gate drop the router's dropped slots hide part of its choice, so every token
      //    chooses again; without one, only tokens that chose an expert already full.
      for (int tl = warp; tl < nb; tl += kCapWarps) {
        bool dirty;
        if (pass == 0) {
          const int e = lane < K ? bid[tl * K + lane] : -1;
          dirty = theta > 0.f || __any_sync(0xffffffffu, e >= 0 && cnt[e] >= cap);
        } else {
          dirty = s_dirty[tl] != 0;
        }
        if (dirty)
          masked_topk(logits + static_cast<size_t>(t0 + tl) * E, E, K, theta, tl, cnt, fb, cap,
                      bid + tl * K, bw + tl * K);
      }
      __syncthreads();  // every warp has read the dirty flags and written its tokens' choices
      for (int i = tid; i < E * kCapWords; i += kCapThreads) mask[i] = 0u;
      if (tid == 0) s_nchg = 0;
      __syncthreads();
      // 2. which block tokens hold each expert
      for (int i = tid; i < nb * K; i += kCapThreads) {
        const int e = bid[i];
        const int tl = i / K;
        if (e >= 0) atomicOr(&mask[e * kCapWords + (tl >> 5)], 1u << (tl & 31));
      }
      __syncthreads();
      // 3. fb[e]: the block token that takes e's last free place, if any
      for (int e = tid; e < E; e += kCapThreads) {
        const int need = cap - cnt[e];
        int f = kNone;
        if (need > 0) {
          int run = 0;
          for (int wd = 0; wd < kCapWords; ++wd) {
            const uint32_t m = mask[e * kCapWords + wd];
            const int c = __popc(m);
            if (run + c >= need) {
              f = wd * 32 + nth_set_bit(m, need - run - 1);
              break;
            }
            run += c;
          }
        }
        if (f != fb[e]) {
          const int j = atomicAdd(&s_nchg, 1);
          chg[3 * j] = e;
          chg[3 * j + 1] = fb[e];
          chg[3 * j + 2] = f;
          fb[e] = f;
        }
      }
      __syncthreads();
      const int nchg = s_nchg;
      if (nchg == 0) break;
      // 4. which tokens must choose again: e's last free place moved from a to b.  Earlier
      //    (b < a): tokens in (b, a] lose e, which matters to those holding it.  Later
      //    (b > a): tokens in (a, b] gain e, which matters if its logit ties or beats the
      //    token's weakest choice or the token has an empty slot (a dropped slot hides a
      //    choice, so it counts as empty).
      for (int tl = tid; tl < nb; tl += kCapThreads) {
        const float* Lt = logits + static_cast<size_t>(t0 + tl) * E;
        float weakest = 0.f;
        bool has_empty = false;
        for (int k = 0; k < K; ++k) {
          const int e = bid[tl * K + k];
          if (e < 0) {
            has_empty = true;
          } else {
            const float v = Lt[e];
            weakest = k == 0 ? v : fminf(weakest, v);
          }
        }
        int d = 0;
        for (int j = 0; j < nchg && !d; ++j) {
          const int e = chg[3 * j], a = chg[3 * j + 1], b = chg[3 * j + 2];
          if (b < a) {
            if (tl > b && tl <= a) {
              for (int k = 0; k < K; ++k) d |= bid[tl * K + k] == e;
            }
          } else if (tl > a && tl <= b) {
            d = has_empty || Lt[e] >= weakest;
          }
        }
        s_dirty[tl] = d;
      }
      __syncthreads();
      if (pass > nb + 1) {  // cannot happen: each pass fixes at least one more token
        if (tid == 0) report_error(err, MOE_DEVERR_BOUNDS);
        break;
      }
    }
    // 4. commit the block: its kept assignments count against the capacity
    for (int e = tid; e < E; e += kCapThreads) {
      int c = 0;
      for (int wd = 0; wd < kCapWords; ++wd) c += __popc(mask[e * kCapWords + wd]);
      cnt[e] += c;
    }
    for (int i = tid; i < nb * K; i += kCapThreads) {
      ids[static_cast<size_t>(t0) * K + i] = bid[i];
      w[static_cast<size_t>(t0) * K + i] = bw[i];
    }
    __syncthreads();
  }
}

}  // namespace

int capacity_limit(int T, int K, int E) {
  const long long c = (12LL * T * K + 10LL * E - 1) / (10LL * E);
  return static_cast<int>(c);
}

cudaError_t launch_capacity_route(const float* logits, int32_t* ids, float* w, int T, int E, int K,
                                  float theta, int cap, unsigned* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (E < 1 || E > 1024 || K < 1 || K > 16) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(E) * (2 * 4 + kCapWords * 4 + 3 * 4) +
                      static_cast<size_t>(kCapBlock) * K * 8;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static int attr_dev = -1;
  if (attr_dev != dev) {
    e = cudaFuncSetAttribute(capacity_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kCapBlock * 16 * 8 + 1024 * (8 + kCapWords * 4 + 12)));
    if (e != cudaSuccess) return e;
    attr_dev = dev;
  }
  return launch_pdl(capacity_route_kernel, dim3(1), dim3(kCapThreads), smem, s, logits, ids, w, T,
                    E, K, theta, cap, err);
}

}  // namespace moe
