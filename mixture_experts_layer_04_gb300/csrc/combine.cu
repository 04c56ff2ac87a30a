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

template <typename TOut>
__global__ void __launch_bounds__(kCombineThreads)
    combine_kernel(const float* __restrict__ out_perm, const int32_t* __restrict__ inv,
                   const float* __restrict__ w, const float* __restrict__ shared_out,
                   TOut* __restrict__ y, float* __restrict__ y_f32, int H, int K) {
  __shared__ int rows[kMaxK];
  __shared__ float gates[kMaxK];
  grid_dep_wait();
  grid_dep_trigger();
  const int t = blockIdx.x;
  if (threadIdx.x < K) {
    rows[threadIdx.x] = inv[static_cast<size_t>(t) * K + threadIdx.x];
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
      const float4 s = reinterpret_cast<const float4*>(shared_out)[static_cast<size_t>(t) * H4 + c];
      acc.x += s.x;
      acc.y += s.y;
      acc.z += s.z;
      acc.w += s.w;
    }
    const size_t i = static_cast<size_t>(t) * H4 + c;
    store4(y, i, acc);
    if (y_f32 != nullptr) reinterpret_cast<float4*>(y_f32)[i] = acc;
  }
}

}  // namespace

cudaError_t launch_combine(int dtype, const float* out_perm, const int32_t* inv, const float* w,
                           const float* shared_out, void* y, float* y_f32, int T, int H, int K,
                           cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (dtype == kBF16)
    return launch_pdl(combine_kernel<__nv_bfloat16>, dim3(T), dim3(kCombineThreads), 0, s,
                      out_perm, inv, w, shared_out, static_cast<__nv_bfloat16*>(y), y_f32, H, K);
  return launch_pdl(combine_kernel<float>, dim3(T), dim3(kCombineThreads), 0, s, out_perm, inv, w,
                    shared_out, static_cast<float*>(y), y_f32, H, K);
}

}  // namespace moe
