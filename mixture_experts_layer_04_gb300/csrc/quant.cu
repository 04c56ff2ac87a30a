// Per-row FP8 (E4M3) quantisation for the low-precision experts.
//
// "MoE大模型的智能调度：从1.8万亿参数到每token仅激活2%的工程真相" §4.1 quantises the resident
// experts' weights to 8 bits to save memory.  Here the 8-bit format is E4M3, the one the tensor
// cores run at full rate, with one float32 scale per row: scale = amax(|row|) / 448 (1 for an
// all-zero row) and code = E4M3(value * (1 / scale)), the reciprocal (once per row) and the
// product each rounded to float32, then rounded to nearest even, saturating at 448.  (A float32
// division per value instead took most of the kernel's time.)  Used for the expert weights
// (rows = output channels) and for the token rows fed to the FP8 gate/up GEMM.
#include <cuda_fp8.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kQThreads = 256;

// One warp per row; each lane handles 8 consecutive values at a time (16-byte loads).
__global__ void __launch_bounds__(kQThreads)
    quantize_rows_fp8_kernel(const __nv_bfloat16* __restrict__ in, long long rows, int cols,
                             uint8_t* __restrict__ codes, float* __restrict__ scales) {
  grid_dep_wait();
  grid_dep_trigger();
  const int lane = threadIdx.x & 31;
  const long long warps = static_cast<long long>(gridDim.x) * (kQThreads / 32);
  for (long long r = blockIdx.x * (kQThreads / 32) + (threadIdx.x >> 5); r < rows; r += warps) {
    const uint4* src = reinterpret_cast<const uint4*>(in + r * cols);
    const int units = cols / 8;
    float amax = 0.f;
    for (int u = lane; u < units; u += 32) {
      const uint4 v = __ldg(src + u);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.f ? amax / 448.f : 1.f;
    const float inv = 1.f / scale;  // correctly rounded: an IEEE division, once per row
    if (lane == 0) scales[r] = scale;
    uint2* dst = reinterpret_cast<uint2*>(codes + r * cols);
    for (int u = lane; u < units; u += 32) {
      const uint4 v = __ldg(src + u);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
      uint32_t packed[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const float2 a = __bfloat1622float2(h[2 * i]);
        const float2 b = __bfloat1622float2(h[2 * i + 1]);
        const uint32_t lo = __nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(a.x, inv), __fmul_rn(a.y, inv)), __NV_SATFINITE, __NV_E4M3);
        const uint32_t hi = __nv_cvt_float2_to_fp8x2(
            make_float2(__fmul_rn(b.x, inv), __fmul_rn(b.y, inv)), __NV_SATFINITE, __NV_E4M3);
        packed[i] = lo | (hi << 16);
      }
      dst[u] = make_uint2(packed[0], packed[1]);
    }
  }
}

// The same for rows of up to 32 * 8 * U values, read once: each lane keeps its U 16-byte
// units of the row in registers (all loads issued before the first use) for the amax and
// the conversion, instead of reading the row a second time.
template <int U>
__global__ void __launch_bounds__(kQThreads)
    quantize_rows_fp8_reg_kernel(const __nv_bfloat16* __restrict__ in, long long rows, int cols,
                                 uint8_t* __restrict__ codes, float* __restrict__ scales) {
  grid_dep_wait();
  grid_dep_trigger();
  const int lane = threadIdx.x & 31;
  const int units = cols / 8;
  const long long warps = static_cast<long long>(gridDim.x) * (kQThreads / 32);
  for (long long r = blockIdx.x * (kQThreads / 32) + (threadIdx.x >> 5); r < rows; r += warps) {
    const uint4* src = reinterpret_cast<const uint4*>(in + r * cols);
    uint4 v[U];
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int u = lane + 32 * i;
      v[i] = u < units ? __ldg(src + u) : make_uint4(0u, 0u, 0u, 0u);
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(h[q]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = amax > 0.f ? amax / 448.f : 1.f;
    const float inv = 1.f / scale;  // correctly rounded: an IEEE division, once per row
    if (lane == 0) scales[r] = scale;
    uint2* dst = reinterpret_cast<uint2*>(codes + r * cols);
#pragma unroll
    for (int i = 0; i < U; ++i) {
      const int u = lane + 32 * i;
      if (u < units) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
        auto four = [&](int k) {  // values 4k .. 4k+3 of the unit as four codes
          const float2 a = __bfloat1622float2(h[2 * k]);
          const float2 b = __bfloat1622float2(h[2 * k + 1]);
          const uint32_t lo = __nv_cvt_float2_to_fp8x2(
              make_float2(__fmul_rn(a.x, inv), __fmul_rn(a.y, inv)), __NV_SATFINITE, __NV_E4M3);
          const uint32_t hi = __nv_cvt_float2_to_fp8x2(
              make_float2(__fmul_rn(b.x, inv), __fmul_rn(b.y, inv)), __NV_SATFINITE, __NV_E4M3);
          return lo | (hi << 16);
        };
        dst[u] = make_uint2(four(0), four(1));
      }
    }
  }
}

// dst[r] = src[perm[r]] for the dispatched rows r < offsets_end[0], 0 for the rest: the
// token-row scales in the permuted row order.
__global__ void __launch_bounds__(kQThreads)
    gather_scales_kernel(const float* __restrict__ src, const int32_t* __restrict__ perm,
                         const int32_t* __restrict__ offsets_end, float* __restrict__ dst,
                         int n) {
  grid_dep_wait();
  grid_dep_trigger();
  const int m = *offsets_end;
  for (int r = blockIdx.x * kQThreads + threadIdx.x; r < n; r += gridDim.x * kQThreads)
    dst[r] = r < m ? __ldg(src + __ldg(perm + r)) : 0.f;
}

}  // namespace

cudaError_t launch_gather_scales(const float* src, const int32_t* perm, const int32_t* offsets_end,
                                 float* dst, int n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const int want = (n + kQThreads - 1) / kQThreads;
  return launch_pdl(gather_scales_kernel, dim3(want < 1024 ? want : 1024), dim3(kQThreads), 0, s,
                    src, perm, offsets_end, dst, n);
}

cudaError_t launch_quantize_fp8(const void* in, long long rows, int cols, uint8_t* codes,
                                float* scales, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  if (cols % 8 != 0) return cudaErrorInvalidValue;
  const long long want = (rows + kQThreads / 32 - 1) / (kQThreads / 32);
  const unsigned blocks = static_cast<unsigned>(want < 8192 ? want : 8192);
  const auto* src = static_cast<const __nv_bfloat16*>(in);
  const int per_lane = (cols / 8 + 31) / 32;  // 16-byte units per lane
  if (per_lane <= 4)
    return launch_pdl(quantize_rows_fp8_reg_kernel<4>, dim3(blocks), dim3(kQThreads), 0, s, src,
                      rows, cols, codes, scales);
  if (per_lane <= 8)
    return launch_pdl(quantize_rows_fp8_reg_kernel<8>, dim3(blocks), dim3(kQThreads), 0, s, src,
                      rows, cols, codes, scales);
  // (9-16 units per lane, e.g. H = 4096, measured about 8% slower read once than twice)
  if (per_lane > 16 && per_lane <= 28)  // H = 7168: 896 units, 2.82 GB in 541 us against 640
    return launch_pdl(quantize_rows_fp8_reg_kernel<28>, dim3(blocks), dim3(kQThreads), 0, s, src,
                      rows, cols, codes, scales);
  return launch_pdl(quantize_rows_fp8_kernel, dim3(blocks), dim3(kQThreads), 0, s, src, rows,
                    cols, codes, scales);
}

}  // namespace moe
