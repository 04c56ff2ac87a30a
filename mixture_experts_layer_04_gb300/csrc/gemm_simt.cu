// Grouped GEMM on the CUDA cores for float32 layers.
//
// The float32 layer keeps every operand in float32 (the tensor cores would round the
// inputs to tf32), so its expert FFN runs as a classic shared-memory tiled SIMT GEMM:
// 64x64 output tiles, k-steps of 16, 4x4 outputs per thread.  It walks the same ragged
// m-tile table as the tensor-core engine (one tile never mixes two experts' rows) and
// supports the same two epilogues: plain fp32 store (+ optional column bias) and the
// SwiGLU pair silu(gate) * up, whose gate and up columns come from the two halves of
// the expert's stacked [W_g; W_u] weight.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kBM = kSimtBM;  // 64
constexpr int kBN = 64;
constexpr int kBK = 16;
constexpr int kThreads = 256;

template <bool kSwi>
__global__ void __launch_bounds__(kThreads)
    grouped_gemm_simt_kernel(const float* __restrict__ A, const float* __restrict__ B,
                             float* __restrict__ C, const float* __restrict__ col_bias,
                             const int4* __restrict__ table, const int32_t* __restrict__ num_mt,
                             int rows_alloc, int Kd, int Nb, int N_out, int up_offset) {
  __shared__ float As[kBK][kBM + 4];
  __shared__ float Bg[kBK][kBN + 4];
  __shared__ float Bu[kSwi ? kBK : 1][kSwi ? kBN + 4 : 1];

  grid_dep_wait();
  grid_dep_trigger();
  const int mt = blockIdx.y;
  int g, row0, row_end;
  if (table != nullptr) {
    if (mt >= *num_mt) return;
    const int4 ent = table[mt];
    g = ent.x;
    row0 = ent.y;
    row_end = ent.z;
  } else {
    g = 0;
    row0 = mt * kBM;
    row_end = rows_alloc;
    if (row0 >= row_end) return;
  }
  const int n0 = blockIdx.x * kBN;
  const int tid = threadIdx.x;
  const int ty = tid / 16, tx = tid % 16;
  const float* Bgrp = B + static_cast<size_t>(g) * Nb * Kd;

  float accg[4][4] = {};
  float accu[4][4] = {};

  const int lr = tid / 4;        // 0..63: row of the tile this thread loads
  const int lk = (tid % 4) * 4;  // 0,4,8,12: k offset inside the 16-wide step
  for (int k0 = 0; k0 < Kd; k0 += kBK) {
    {
      const int r = row0 + lr;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r < row_end) v = *reinterpret_cast<const float4*>(A + static_cast<size_t>(r) * Kd + k0 + lk);
      As[lk + 0][lr] = v.x;
      As[lk + 1][lr] = v.y;
      As[lk + 2][lr] = v.z;
      As[lk + 3][lr] = v.w;
    }
    {
      const int n = n0 + lr;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (n < N_out) v = *reinterpret_cast<const float4*>(Bgrp + static_cast<size_t>(n) * Kd + k0 + lk);
      Bg[lk + 0][lr] = v.x;
      Bg[lk + 1][lr] = v.y;
      Bg[lk + 2][lr] = v.z;
      Bg[lk + 3][lr] = v.w;
      if constexpr (kSwi) {
        float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
        if (n < N_out)
          u = *reinterpret_cast<const float4*>(Bgrp + static_cast<size_t>(up_offset + n) * Kd + k0 + lk);
        Bu[lk + 0][lr] = u.x;
        Bu[lk + 1][lr] = u.y;
        Bu[lk + 2][lr] = u.z;
        Bu[lk + 3][lr] = u.w;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      float a[4], bg[4], bu[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bg[j] = Bg[kk][tx * 4 + j];
        if constexpr (kSwi) bu[j] = Bu[kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          accg[i][j] = fmaf(a[i], bg[j], accg[i][j]);
          if constexpr (kSwi) accu[i][j] = fmaf(a[i], bu[j], accu[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = row0 + ty * 4 + i;
    if (r >= row_end) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N_out) continue;
      float v;
      if constexpr (kSwi)
        v = silu_f(accg[i][j]) * accu[i][j];
      else
        v = accg[i][j] + (col_bias != nullptr ? col_bias[n] : 0.f);
      C[static_cast<size_t>(r) * N_out + n] = v;
    }
  }
}

}  // namespace

cudaError_t launch_grouped_gemm_simt(const GroupedGemm& p, cudaStream_t s) {
  if (p.dtype != kF32) return cudaErrorInvalidValue;
  const int mt = p.mtile_table != nullptr ? p.max_mtiles : (p.rows_alloc + kBM - 1) / kBM;
  if (mt == 0) return cudaSuccess;
  dim3 grid((p.N_out + kBN - 1) / kBN, mt);
  auto kernel = p.mode == kSwiGLU ? grouped_gemm_simt_kernel<true> : grouped_gemm_simt_kernel<false>;
  return launch_pdl(kernel, grid, dim3(kThreads), 0, s, static_cast<const float*>(p.A),
                    static_cast<const float*>(p.B), static_cast<float*>(p.C),
                    p.mode == kSwiGLU ? nullptr : p.col_bias, p.mtile_table, p.num_mtiles,
                    p.rows_alloc, p.Kd, p.Nb, p.N_out, p.up_offset);
}

}  // namespace moe
