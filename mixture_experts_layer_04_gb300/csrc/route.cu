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

template <typename TIn>
__device__ __forceinline__ float dot_row(const TIn* a, const TIn* b, int H, int lane);

template <>
__device__ __forceinline__ float dot_row<float>(const float* a, const float* b, int H, int lane) {
  float acc = 0.f;
  const float4* a4 = reinterpret_cast<const float4*>(a);
  const float4* b4 = reinterpret_cast<const float4*>(b);
  for (int i = lane; i < H / 4; i += 32) {
    float4 p = a4[i], q = __ldg(b4 + i);
    acc = fmaf(p.x, q.x, acc);
    acc = fmaf(p.y, q.y, acc);
    acc = fmaf(p.z, q.z, acc);
    acc = fmaf(p.w, q.w, acc);
  }
  return warp_sum(acc);
}

template <>
__device__ __forceinline__ float dot_row<__nv_bfloat16>(const __nv_bfloat16* a,
                                                        const __nv_bfloat16* b, int H, int lane) {
  float acc = 0.f;
  const uint4* a4 = reinterpret_cast<const uint4*>(a);
  const uint4* b4 = reinterpret_cast<const uint4*>(b);
  for (int i = lane; i < H / 8; i += 32) {
    uint4 p = a4[i], q = __ldg(b4 + i);
    const __nv_bfloat162* pp = reinterpret_cast<const __nv_bfloat162*>(&p);
    const __nv_bfloat162* qq = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float2 fp = __bfloat1622float2(pp[j]);
      float2 fq = __bfloat1622float2(qq[j]);
      acc = fmaf(fp.x, fq.x, acc);
      acc = fmaf(fp.y, fq.y, acc);
    }
  }
  return warp_sum(acc);
}

constexpr int kRouterWarps = 8;

// One block per token: warp w computes the logits of experts w, w+8, ...; then warp 0
// takes the top-k.  Used when the router GEMM is too small for the tensor cores
// (few tokens or few experts) and for float32 layers.
template <typename TIn>
__global__ void __launch_bounds__(kRouterWarps * 32)
    router_simt_topk_kernel(const TIn* __restrict__ x, const TIn* __restrict__ w_router,
                            const float* __restrict__ bias, float* __restrict__ logits,
                            int32_t* __restrict__ ids, float* __restrict__ w, int H, int E, int K,
                            float theta) {
  extern __shared__ float Ls[];
  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const TIn* xr = x + static_cast<size_t>(t) * H;
  for (int e = warp; e < E; e += kRouterWarps) {
    float d = dot_row<TIn>(xr, w_router + static_cast<size_t>(e) * H, H, lane);
    if (lane == 0) Ls[e] = bias != nullptr ? d + bias[e] : d;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) logits[static_cast<size_t>(t) * E + e] = Ls[e];
  if (warp == 0)
    warp_topk_softmax(Ls, E, K, theta, ids + static_cast<size_t>(t) * K,
                      w + static_cast<size_t>(t) * K);
}

constexpr int kTopkWarps = 4;

// One warp per token, logits from memory (optionally biased and written back).
__global__ void __launch_bounds__(kTopkWarps * 32)
    topk_kernel(const float* __restrict__ logits_in, const float* __restrict__ bias,
                float* __restrict__ logits_out, int32_t* __restrict__ ids, float* __restrict__ w,
                int T, int E, int K, float theta) {
  extern __shared__ float Ls_all[];
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

cudaError_t launch_router_simt_topk(int dtype, const void* x, const void* w_router,
                                    const float* bias, float* logits, int32_t* ids, float* w,
                                    int T, int H, int E, int K, float theta, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const size_t smem = static_cast<size_t>(E) * sizeof(float);
  if (dtype == kBF16) {
    router_simt_topk_kernel<__nv_bfloat16><<<T, kRouterWarps * 32, smem, s>>>(
        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(w_router), bias,
        logits, ids, w, H, E, K, theta);
  } else {
    router_simt_topk_kernel<float><<<T, kRouterWarps * 32, smem, s>>>(
        static_cast<const float*>(x), static_cast<const float*>(w_router), bias, logits, ids, w,
        H, E, K, theta);
  }
  return cudaGetLastError();
}

cudaError_t launch_topk(const float* logits_in, const float* bias, float* logits_out,
                        int32_t* ids, float* w, int T, int E, int K, float theta,
                        cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kTopkWarps - 1) / kTopkWarps;
  const size_t smem = static_cast<size_t>(kTopkWarps) * E * sizeof(float);
  topk_kernel<<<blocks, kTopkWarps * 32, smem, s>>>(logits_in, bias, logits_out, ids, w, T, E, K,
                                                     theta);
  return cudaGetLastError();
}

}  // namespace moe
