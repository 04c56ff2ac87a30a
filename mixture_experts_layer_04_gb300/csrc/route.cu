// Routing kernels: router logits and the warp-per-token top-k.
//
// Routing rule ("MoE大模型的智能调度：从1.8万亿参数到每token仅激活2%的工程真相", §2.2,
// routing steps 1-3): the router gives one logit per expert; the K largest are kept and
// normalised with a softmax; a kept gate below the threshold is set to zero and the
// survivors are renormalised.  Selection is on float32 logits, descending, ties to the
// lower expert id; slot 0 is never dropped.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

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
__device__ void warp_topk_softmax(const float* L, int E, int K, float theta, int32_t* ids_out,
                                  float* w_out) {
  const int lane = threadIdx.x & 31;
  uint32_t taken = 0;  // bit j: expert lane + 32 j already selected
  float my_v = 0.f;
  int my_e = -1;
  float v0 = 0.f;
  for (int k = 0; k < K; ++k) {
    unsigned long long best = 0ull;
    for (int j = 0, e = lane; e < E; ++j, e += 32) {
      if (taken & (1u << j)) continue;
      unsigned long long key = (static_cast<unsigned long long>(float_key(L[e])) << 32) |
                               static_cast<uint32_t>(~static_cast<uint32_t>(e));
      best = key > best ? key : best;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      unsigned long long other = __shfl_xor_sync(0xffffffffu, best, o);
      best = other > best ? other : best;
    }
    const int e_win = static_cast<int>(~static_cast<uint32_t>(best & 0xffffffffull));
    if ((e_win & 31) == lane) taken |= 1u << (e_win >> 5);
    const float v_win = L[e_win];
    if (k == 0) v0 = v_win;
    if (lane == k) {
      my_v = v_win;
      my_e = e_win;
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

// Widens the 16-byte chunk i of a row of TIn into floats (8 bf16 or 4 float).
template <typename TIn> struct Vec;
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, int i, float (&f)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p) + i);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 v = __bfloat1622float2(h[j]);
      f[2 * j] = v.x;
      f[2 * j + 1] = v.y;
    }
  }
};
template <> struct Vec<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void load(const float* p, int i, float (&f)[8]) {
    const float4 u = __ldg(reinterpret_cast<const float4*>(p) + i);
    f[0] = u.x;
    f[1] = u.y;
    f[2] = u.z;
    f[3] = u.w;
  }
};

constexpr int kRouterExperts = 8;  // warps per block, one expert each
constexpr int kRouterTokens = 8;   // tokens per block

// logits[t, e] = x[t] . W_r[e] + bias[e] for 8 experts x 8 tokens per block.  Each warp
// keeps its expert's weights streaming through registers once and reuses them for the
// block's 8 tokens (whose rows the 8 warps share through L1).  With E <= 8 one block
// holds every logit of its tokens, and warp t then takes token t's top-k (fuse_topk).
template <typename TIn>
__global__ void __launch_bounds__(kRouterExperts * 32)
    router_logits_kernel(const TIn* __restrict__ x, const TIn* __restrict__ w_router,
                         const float* __restrict__ bias, float* __restrict__ logits,
                         int32_t* __restrict__ ids, float* __restrict__ w, int T, int H, int E,
                         int K, float theta, int fuse_topk) {
  __shared__ float Ls[kRouterTokens][kRouterExperts];
  grid_dep_wait();
  grid_dep_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * kRouterExperts + warp;
  constexpr int V = Vec<TIn>::N;
  for (int t0 = blockIdx.y * kRouterTokens; t0 < T; t0 += gridDim.y * kRouterTokens) {
  const int nt = min(kRouterTokens, T - t0);
  if (e < E) {
    float acc[kRouterTokens];
#pragma unroll
    for (int tt = 0; tt < kRouterTokens; ++tt) acc[tt] = 0.f;
    const TIn* wr = w_router + static_cast<size_t>(e) * H;
    const int chunks = H / V;
#pragma unroll 2
    for (int i = lane; i < chunks; i += 32) {
      float wv[8];
      Vec<TIn>::load(wr, i, wv);
#pragma unroll
      for (int tt = 0; tt < kRouterTokens; ++tt) {
        if (tt < nt) {
          float xv[8];
          Vec<TIn>::load(x + static_cast<size_t>(t0 + tt) * H, i, xv);
#pragma unroll
          for (int j = 0; j < V; ++j) acc[tt] = fmaf(xv[j], wv[j], acc[tt]);
        }
      }
    }
    const float b = bias != nullptr ? bias[e] : 0.f;
#pragma unroll
    for (int tt = 0; tt < kRouterTokens; ++tt) {
      const float v = warp_sum(acc[tt]) + b;
      if (tt < nt && lane == 0) {
        logits[static_cast<size_t>(t0 + tt) * E + e] = v;
        Ls[tt][warp] = v;
      }
    }
  }
  if (fuse_topk) {
    __syncthreads();
    if (warp < nt)
      warp_topk_softmax(Ls[warp], E, K, theta, ids + static_cast<size_t>(t0 + warp) * K,
                        w + static_cast<size_t>(t0 + warp) * K);
    __syncthreads();
  }
  }
}

constexpr int kTopkWarps = 4;

// One warp per token, logits from memory (optionally biased and written back).
__global__ void __launch_bounds__(kTopkWarps * 32)
    topk_kernel(const float* __restrict__ logits_in, const float* __restrict__ bias,
                float* __restrict__ logits_out, int32_t* __restrict__ ids, float* __restrict__ w,
                int T, int E, int K, float theta) {
  extern __shared__ float Ls_all[];
  grid_dep_wait();
  grid_dep_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t >= T) return;
  float* Ls = Ls_all + warp * E;
  const float* src = logits_in + static_cast<size_t>(t) * E;
  for (int e = lane; e < E; e += 32) {
    float v = src[e];
    if (bias != nullptr) {
      v += bias[e];
      logits_out[static_cast<size_t>(t) * E + e] = v;
    }
    Ls[e] = v;
  }
  __syncwarp();
  warp_topk_softmax(Ls, E, K, theta, ids + static_cast<size_t>(t) * K,
                    w + static_cast<size_t>(t) * K);
}

}  // namespace

cudaError_t launch_router_simt(int dtype, const void* x, const void* w_router,
                               const float* bias, float* logits, int32_t* ids, float* w,
                               int T, int H, int E, int K, float theta, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int fuse = E <= kRouterExperts ? 1 : 0;
  const int tblocks = (T + kRouterTokens - 1) / kRouterTokens;
  const dim3 grid((E + kRouterExperts - 1) / kRouterExperts, tblocks < 65535 ? tblocks : 65535);
  cudaError_t err;
  if (dtype == kBF16)
    err = launch_pdl(router_logits_kernel<__nv_bfloat16>, grid, dim3(kRouterExperts * 32), 0, s,
                     static_cast<const __nv_bfloat16*>(x),
                     static_cast<const __nv_bfloat16*>(w_router), bias, logits, ids, w, T, H, E,
                     K, theta, fuse);
  else
    err = launch_pdl(router_logits_kernel<float>, grid, dim3(kRouterExperts * 32), 0, s,
                     static_cast<const float*>(x), static_cast<const float*>(w_router), bias,
                     logits, ids, w, T, H, E, K, theta, fuse);
  if (err != cudaSuccess || fuse) return err;
  return launch_topk(logits, nullptr, nullptr, ids, w, T, E, K, theta, s);
}

cudaError_t launch_topk(const float* logits_in, const float* bias, float* logits_out,
                        int32_t* ids, float* w, int T, int E, int K, float theta,
                        cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kTopkWarps - 1) / kTopkWarps;
  const size_t smem = static_cast<size_t>(kTopkWarps) * E * sizeof(float);
  return launch_pdl(topk_kernel, dim3(blocks), dim3(kTopkWarps * 32), smem, s, logits_in, bias,
                    logits_out, ids, w, T, E, K, theta);
}

}  // namespace moe
