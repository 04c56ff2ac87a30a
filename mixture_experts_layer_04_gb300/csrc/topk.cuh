// Warp-level top-k with softmax and gate drop, shared by the routing kernels.
//
// Routing rule ("MoE大模型的智能调度：从1.8万亿参数到每token仅激活2%的工程真相", §2.2,
// routing steps 2-3): the K largest logits are kept and normalised with a softmax; a kept
// gate below the threshold is set to zero and the survivors are renormalised.  Selection
// is on float32 logits, descending, ties to the lower expert id; slot 0 is never dropped.
#pragma once

#include "common.cuh"

namespace moe {

// Order-preserving map of a float to uint32 (larger float -> larger key); -0 is
// folded into +0 so that the two compare equal, as floats do.
__device__ __forceinline__ uint32_t float_key(float v) {
  if (v == 0.0f) v = 0.0f;
  uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp: top-K of the E logits in shared memory `L`, softmax over the kept
// logits, gate drop, and the stores of ids[K] / w[K] for this token.
__device__ __forceinline__ void warp_topk_softmax(const float* L, int E, int K, float theta, int32_t* ids_out,
                                  float* w_out) {
  const int lane = threadIdx.x & 31;
  uint32_t taken = 0;  // bit j: expert lane + 32 j already selected
  float my_v = 0.f;
  int my_e = -1;
  float v0 = 0.f;
  if (E <= 256) {
    // up to 8 candidates per lane, keys kept in registers for all K rounds
    uint32_t key[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) key[j] = lane + 32 * j < E ? float_key(L[lane + 32 * j]) : 0u;
    for (int k = 0; k < K; ++k) {
      // this lane's best untaken candidate (the first of equal keys is the lower id), then
      // the warp's largest key and, among the lanes holding it, the lowest expert id
      uint32_t kbest = 0u, ebest = 0xffffffffu;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const bool live = lane + 32 * j < E && !(taken & (1u << j));
        if (live && (key[j] > kbest || ebest == 0xffffffffu)) {
          kbest = key[j];
          ebest = static_cast<uint32_t>(lane + 32 * j);
        }
      }
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, ebest != 0xffffffffu ? kbest : 0u);
      const int e_win = static_cast<int>(__reduce_min_sync(
          0xffffffffu, (ebest != 0xffffffffu && kbest == kmax) ? ebest : 0xffffffffu));
      if ((e_win & 31) == lane) taken |= 1u << (e_win >> 5);
      const float v_win = L[e_win];
      if (k == 0) v0 = v_win;
      if (lane == k) {
        my_v = v_win;
        my_e = e_win;
      }
    }
  } else {
    for (int k = 0; k < K; ++k) {
      uint32_t kbest = 0u, ebest = 0xffffffffu;
      for (int j = 0, e = lane; e < E; ++j, e += 32) {
        if (taken & (1u << j)) continue;
        const uint32_t kk = float_key(L[e]);
        if (kk > kbest || ebest == 0xffffffffu) {
          kbest = kk;
          ebest = static_cast<uint32_t>(e);
        }
      }
      const uint32_t kmax = __reduce_max_sync(0xffffffffu, ebest != 0xffffffffu ? kbest : 0u);
      const int e_win = static_cast<int>(__reduce_min_sync(
          0xffffffffu, (ebest != 0xffffffffu && kbest == kmax) ? ebest : 0xffffffffu));
      if ((e_win & 31) == lane) taken |= 1u << (e_win >> 5);
      const float v_win = L[e_win];
      if (k == 0) v0 = v_win;
      if (lane == k) {
        my_v = v_win;
        my_e = e_win;
      }
    }
  }
  float z = (lane < K) ? expf(my_v - v0) : 0.f;
  float w = z / warp_sum(z);
  if (theta > 0.f) {
    if (lane >= 1 && lane < K && w < theta) {
      w = 0.f;
      my_e = -1;
    }
    w = w / warp_sum(w);
  }
  if (lane < K) {
    ids_out[lane] = my_e;
    w_out[lane] = w;
  }
}

}  // namespace moe
