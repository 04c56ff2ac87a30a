// Grouped GEMM on the CUDA cores for float32 layers.
//
// The float32 layer keeps every operand in float32 (the tensor cores would round the
// inputs to tf32), so its expert FFN runs as a classic shared-memory tiled SIMT GEMM:
// 64x64 output tiles, k-steps of 16 double-buffered in shared memory, 4x4 outputs per
// thread.  It walks the same ragged m-tile table as the tensor-core engine (one tile
// never mixes two experts' rows) and supports the same two epilogues: plain fp32 store (+ optional column bias) and the
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
  // two shared-memory buffers: the global loads of k-step s+1 are in flight (in
  // registers) while k-step s is computed from the other buffer
  __shared__ float As[2][kBK][kBM + 4];
  __shared__ float Bg[2][kBK][kBN + 4];
  __shared__ float Bu[2][kSwi ? kBK : 1][kSwi ? kBN + 4 : 1];

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
  const bool a_ok = row0 + lr < row_end, b_ok = n0 + lr < N_out;
  const float* a_src = A + static_cast<size_t>(a_ok ? row0 + lr : 0) * Kd + lk;
  const float* g_src = Bgrp + static_cast<size_t>(b_ok ? n0 + lr : 0) * Kd + lk;
  const float* u_src = Bgrp + static_cast<size_t>(b_ok ? up_offset + n0 + lr : 0) * Kd + lk;
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 va, vg, vu = zero;
  auto load = [&](int k0) {
    va = a_ok ? *reinterpret_cast<const float4*>(a_src + k0) : zero;
    vg = b_ok ? *reinterpret_cast<const float4*>(g_src + k0) : zero;
    if constexpr (kSwi) vu = b_ok ? *reinterpret_cast<const float4*>(u_src + k0) : zero;
  };
  auto stash = [&](int buf) {
    As[buf][lk + 0][lr] = va.x;
    As[buf][lk + 1][lr] = va.y;
    As[buf][lk + 2][lr] = va.z;
    As[buf][lk + 3][lr] = va.w;
    Bg[buf][lk + 0][lr] = vg.x;
    Bg[buf][lk + 1][lr] = vg.y;
    Bg[buf][lk + 2][lr] = vg.z;
    Bg[buf][lk + 3][lr] = vg.w;
    if constexpr (kSwi) {
      Bu[buf][lk + 0][lr] = vu.x;
      Bu[buf][lk + 1][lr] = vu.y;
      Bu[buf][lk + 2][lr] = vu.z;
      Bu[buf][lk + 3][lr] = vu.w;
    }
  };
  load(0);
  stash(0);
  __syncthreads();
  int buf = 0;
  for (int k0 = 0; k0 < Kd; k0 += kBK) {
    const bool more = k0 + kBK < Kd;
    if (more) load(k0 + kBK);
#pragma unroll
    for (int kk = 0; kk < kBK; ++kk) {
      float a[4], bg[4], bu[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[buf][kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bg[j] = Bg[buf][kk][tx * 4 + j];
        if constexpr (kSwi) bu[j] = Bu[buf][kk][tx * 4 + j];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          accg[i][j] = fmaf(a[i], bg[j], accg[i][j]);
          if constexpr (kSwi) accu[i][j] = fmaf(a[i], bu[j], accu[i][j]);
        }
    }
    // the other buffer was last read before the previous barrier, so it can be refilled
    if (more) stash(buf ^ 1);
    __syncthreads();
    buf ^= 1;
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
