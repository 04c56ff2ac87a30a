// Combine kernel: un-permute and gated weighted sum back to token order.
//
// "MoE大模型的智能调度：从1.8万亿参数到每token仅激活2%的工程真相" §2.2, fusion layer: the
// output is the gate-weighted sum of the selected experts' outputs.  Page opening
// "MoE通过稀疏激活降低每个token的计算量…", section "单机MoE执行流水线": the inverse map
// restores token order, the route weights are applied and contributions with the same
// token id are added.  Each token gathers its K rows (no atomics), sums in fp32 in slot
// order, adds the shared expert, and rounds once to the output type.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kCombineThreads = 128;
constexpr int kMaxK = 16;

__device__ __forceinline__ void store4(float* y, size_t i, float4 v) {
  reinterpret_cast<float4*>(y)[i] = v;
}
__device__ __forceinline__ void store4(__nv_bfloat16* y, size_t i, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  reinterpret_cast<uint2*>(y)[i] = u;
}

// Many tokens: one block per token walks its row, four columns per thread per step.
template <typename TOut>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float* __restrict__ out_perm, const int32_t* __restrict__ inv,
                   const float* __restrict__ w, const float* __restrict__ shared_out,
                   TOut* __restrict__ y, float* __restrict__ y_f32, int H, int K,
                   unsigned* __restrict__ err) {
  __shared__ int rows[kMaxK];
  __shared__ float gates[kMaxK];
  grid_dep_wait();
  grid_dep_trigger();
  const int t = blockIdx.x;
  if (threadIdx.x < K) {
    // the grid has one x-block per token, so the rows of out_perm number gridDim.x * K
    const int r = inv[static_cast<size_t>(t) * K + threadIdx.x];
    rows[threadIdx.x] = dcheck(r < static_cast<int>(gridDim.x) * K, err) ? r : -1;
    gates[threadIdx.x] = w[static_cast<size_t>(t) * K + threadIdx.x];
  }
  __syncthreads();
  const int H4 = H / 4;
  const float4* o4 = reinterpret_cast<const float4*>(out_perm);
  for (int c = threadIdx.x; c < H4; c += kCombineThreads) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < K; ++k) {
      const int r = rows[k];
      if (r < 0) continue;
      const float g = gates[k];
      const float4 v = o4[static_cast<size_t>(r) * H4 + c];
      acc.x = fmaf(g, v.x, acc.x);
      acc.y = fmaf(g, v.y, acc.y);
      acc.z = fmaf(g, v.z, acc.z);
      acc.w = fmaf(g, v.w, acc.w);
    }
    if (shared_out != nullptr) {
      const float4 sv = reinterpret_cast<const float4*>(shared_out)[static_cast<size_t>(t) * H4 + c];
      acc.x += sv.x;
      acc.y += sv.y;
      acc.z += sv.z;
      acc.w += sv.w;
    }
    const size_t i = static_cast<size_t>(t) * H4 + c;
    store4(y, i, acc);
    if (y_f32 != nullptr) reinterpret_cast<float4*>(y_f32)[i] = acc;
  }
}

// Few tokens: block (t, by) handles token t's columns [512 by, 512 by + 512), one float4
// per thread with its K row loads issued together, so a small batch still spreads over
// many blocks.  Same arithmetic (fp32, slot order) as combine_kernel.
template <typename TOut>
__global__ void __launch_bounds__(kCombineThreads)
    combine_split_kernel(const float* __restrict__ out_perm, const int32_t* __restrict__ inv,
                         const float* __restrict__ w, const float* __restrict__ shared_out,
                         TOut* __restrict__ y, float* __restrict__ y_f32, int H, int K,
                         unsigned* __restrict__ err) {
  __shared__ int rows[kMaxK];
  __shared__ float gates[kMaxK];
  grid_dep_wait();
  grid_dep_trigger();
  const int t = blockIdx.x;
  if (threadIdx.x < K) {
    // the grid has one x-block per token, so the rows of out_perm number gridDim.x * K
    const int r = inv[static_cast<size_t>(t) * K + threadIdx.x];
    rows[threadIdx.x] = dcheck(r < static_cast<int>(gridDim.x) * K, err) ? r : -1;
    gates[threadIdx.x] = w[static_cast<size_t>(t) * K + threadIdx.x];
  }
  __syncthreads();
  const int H4 = H / 4;
  const int c = blockIdx.y * kCombineThreads + threadIdx.x;
  if (c >= H4) return;
  const float4* o4 = reinterpret_cast<const float4*>(out_perm);
  float4 v[kMaxK];
#pragma unroll
  for (int k = 0; k < kMaxK; ++k)
    if (k < K && rows[k] >= 0) v[k] = o4[static_cast<size_t>(rows[k]) * H4 + c];
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kMaxK; ++k) {
    if (k < K && rows[k] >= 0) {
      const float g = gates[k];
      acc.x = fmaf(g, v[k].x, acc.x);
      acc.y = fmaf(g, v[k].y, acc.y);
      acc.z = fmaf(g, v[k].z, acc.z);
      acc.w = fmaf(g, v[k].w, acc.w);
    }
  }
  if (shared_out != nullptr) {
    const float4 sv = reinterpret_cast<const float4*>(shared_out)[static_cast<size_t>(t) * H4 + c];
    acc.x += sv.x;
    acc.y += sv.y;
    acc.z += sv.z;
    acc.w += sv.w;
  }
  const size_t i = static_cast<size_t>(t) * H4 + c;
  store4(y, i, acc);
  if (y_f32 != nullptr) reinterpret_cast<float4*>(y_f32)[i] = acc;
}

// y[i] = act(y_f32[i]), four elements per thread.
template <typename TOut>
__global__ void __launch_bounds__(256)
    finalize_kernel(const float* __restrict__ y_f32, TOut* __restrict__ y, long long n4) {
  grid_dep_wait();
  grid_dep_trigger();
  for (long long i = blockIdx.x * 256ll + threadIdx.x; i < n4; i += static_cast<long long>(gridDim.x) * 256)
    store4(y, static_cast<size_t>(i), reinterpret_cast<const float4*>(y_f32)[i]);
}

}  // namespace

cudaError_t launch_finalize(int dtype, const float* y_f32, void* y, long long n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const long long n4 = n / 4;
  const long long want = (n4 + 255) / 256;
  const unsigned blocks = static_cast<unsigned>(want < 4096 ? want : 4096);
  if (dtype == kBF16)
    return launch_pdl(finalize_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), 0, s, y_f32,
                      static_cast<__nv_bfloat16*>(y), n4);
  return launch_pdl(finalize_kernel<float>, dim3(blocks), dim3(256), 0, s, y_f32,
                    static_cast<float*>(y), n4);
}

cudaError_t launch_combine(int dtype, const float* out_perm, const int32_t* inv, const float* w,
                           const float* shared_out, void* y, float* y_f32, int T, int H, int K,
                           cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (T < 1024) {  // few tokens: spread each token's columns over several blocks
    const dim3 grid(T, (H / 4 + kCombineThreads - 1) / kCombineThreads);
    if (dtype == kBF16)
      return launch_pdl(combine_split_kernel<__nv_bfloat16>, grid, dim3(kCombineThreads), 0, s,
                        out_perm, inv, w, shared_out, static_cast<__nv_bfloat16*>(y), y_f32, H, K,
                      device_error_word());
    return launch_pdl(combine_split_kernel<float>, grid, dim3(kCombineThreads), 0, s, out_perm,
                      inv, w, shared_out, static_cast<float*>(y), y_f32, H, K,
                      device_error_word());
  }
  if (dtype == kBF16)
    return launch_pdl(combine_kernel<__nv_bfloat16>, dim3(T), dim3(kCombineThreads), 0, s,
                      out_perm, inv, w, shared_out, static_cast<__nv_bfloat16*>(y), y_f32, H, K,
                      device_error_word());
  return launch_pdl(combine_kernel<float>, dim3(T), dim3(kCombineThreads), 0, s, out_perm, inv, w,
                    shared_out, static_cast<float*>(y), y_f32, H, K,
                      device_error_word());
}

}  // namespace moe
