// Routing kernels: router logits on the CUDA cores and the warp-per-token top-k.
//
// Routing rule ("MoE大模型的智能调度：从1.8万亿参数到每token仅激活2%的工程真相", §2.2,
// routing steps 1-3): the router gives one logit per expert; the K largest are kept and
// normalised with a softmax; a kept gate below the threshold is set to zero and the
// survivors are renormalised.  Selection is on float32 logits, descending, ties to the
// lower expert id; slot 0 is never dropped.
//
// Router logits x.W_r^T + b (fp32 accumulation) take one of three routes:
//   * few experts whose weights fit in shared memory (E <= 16): router_wsmem_kernel
//     stages W_r per block and streams each token's x row once, top-k fused;
//   * otherwise on the CUDA cores (decode-sized batches): router_partial_kernel splits
//     the work over (8 experts) x (8 tokens) x (a slice of H) per block so that every SM
//     gets blocks and each block needs one round of loads; the slices' partial sums are
//     added in a fixed order by the top-k kernel (deterministic);
//   * large bf16 batches with E % 16 == 0 use the tensor-core GEMM (gemm_tc.cu).
#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {
namespace {

// Widens the 16-byte chunk u of a row of TIn into floats (8 bf16 or 4 float).
template <typename TIn> struct Vec;
template <> struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void widen(const uint4& u, float (&f)[8]) {
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
  static __device__ __forceinline__ void widen(const uint4& u, float (&f)[8]) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
};

// ------------------------------------------------------------ few experts ----
constexpr int kWsMaxE = 16;
constexpr size_t kWsMaxWeightBytes = 96 * 1024;  // W_r staged in shared memory up to this
constexpr int kWsMaxBlocks = 456;                // 3 blocks per SM on 152 SMs
constexpr int kWsBurst = 8;                      // 16-byte x loads in flight per lane

// Every block stages W_r once; each warp then takes one token at a time, loads its whole
// x row in bursts of kWsBurst independent 16-byte loads per lane (so the row read is not
// a chain of dependent round trips), dots it with all E weight rows from shared memory,
// and takes the top-k.  Persistent over tokens.
template <typename TIn>
__global__ void __launch_bounds__(256, 3)
    router_wsmem_kernel(const TIn* __restrict__ x, const TIn* __restrict__ w_router,
                        const float* __restrict__ bias, float* __restrict__ logits,
                        int32_t* __restrict__ ids, float* __restrict__ w, int T, int H, int E,
                        int K, float theta, unsigned* err) {
  extern __shared__ uint4 wsm[];  // [E][H] TIn, then 8 warps x kWsMaxE floats
  __shared__ uint64_t wbar;
  __shared__ int wfail;
  grid_dep_wait();
  grid_dep_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int V = Vec<TIn>::N;
  const int row_units = H / V;    // 16-byte units per row
  const int units = E * row_units;
  // W_r -> shared memory with one bulk copy (no chain of per-thread round trips)
  const uint32_t bar = smem_u32(&wbar);
  if (threadIdx.x == 0) {
    wfail = 0;
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(units) * 16u);
    bulk_copy_g2s(smem_u32(wsm), w_router, static_cast<uint32_t>(units) * 16u, bar);
  }
  __syncthreads();
  if (!mbar_wait(bar, 0, &wfail, nullptr)) wfail = 1;
  __syncthreads();
  if (wfail) {
    if (threadIdx.x == 0) report_error(err, MOE_DEVERR_TIMEOUT);
    return;
  }
  float* Ls = reinterpret_cast<float*>(wsm + units) + warp * kWsMaxE;
  for (int t = blockIdx.x * 8 + warp; t < T; t += gridDim.x * 8) {
    float acc[kWsMaxE];
#pragma unroll
    for (int e = 0; e < kWsMaxE; ++e) acc[e] = 0.f;
    const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
    for (int i0 = 0; i0 < row_units; i0 += 32 * kWsBurst) {
      uint4 xb[kWsBurst];
#pragma unroll
      for (int b = 0; b < kWsBurst; ++b) {
        const int i = i0 + b * 32 + lane;
        xb[b] = i < row_units ? __ldg(xr + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int b = 0; b < kWsBurst; ++b) {
        const int i = i0 + b * 32 + lane;
        if (i < row_units) {
          float xv[8];
          Vec<TIn>::widen(xb[b], xv);
#pragma unroll
          for (int e = 0; e < kWsMaxE; ++e) {
            if (e < E) {
              float wv[8];
              Vec<TIn>::widen(wsm[e * row_units + i], wv);
#pragma unroll
              for (int j = 0; j < V; ++j) acc[e] = fmaf(xv[j], wv[j], acc[e]);
            }
          }
        }
      }
    }
    float mine = 0.f;
#pragma unroll
    for (int e = 0; e < kWsMaxE; ++e) {
      if (e < E) {
        const float v = warp_sum(acc[e]);
        if (lane == e) mine = v + (bias != nullptr ? bias[e] : 0.f);
      }
    }
    if (lane < E) {
      Ls[lane] = mine;
      logits[static_cast<size_t>(t) * E + lane] = mine;
    }
    __syncwarp();
    warp_topk_softmax(Ls, E, K, theta, ids + static_cast<size_t>(t) * K,
                      w + static_cast<size_t>(t) * K);
    __syncwarp();
  }
}

// ---------------------------------------------------------- partial logits ----
constexpr int kPartExperts = 8;   // warps per block, one expert each
constexpr int kPartTokens = 8;    // tokens per block
constexpr int kPartMaxUnits = 8;  // 16-byte weight units per lane in one slice (burst)
constexpr int kRouterTargetBlocks = 608;  // about 4 blocks per SM

// partial[s][t][e] = sum over slice s of H of x[t, h] * W_r[e, h]  (no bias).
// Block (bx, by, s): experts 8bx..8bx+7, tokens 8by..8by+7, the s-th slice of H.  The slice
// is walked in bursts of 256 16-byte units: the block stages the 8 tokens' burst in shared
// memory (all loads issued at once) while each warp loads its expert's burst (8 units per
// lane, all in flight), then dots it with the 8 staged rows.  Slices are chosen so that a
// layer normally needs a single burst per block.
template <typename TIn>
__global__ void __launch_bounds__(kPartExperts * 32)
    router_partial_kernel(const TIn* __restrict__ x, const TIn* __restrict__ w_router,
                          float* __restrict__ partial, int T, int H, int E, int slice_units) {
  __shared__ uint4 xs[kPartTokens * 32 * kPartMaxUnits];  // [8 tokens][256 units]: 32 KB
  grid_dep_wait();
  grid_dep_trigger();
  constexpr int kBurst = 32 * kPartMaxUnits;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int V = Vec<TIn>::N;
  const int t0 = blockIdx.y * kPartTokens;
  const int nt = min(kPartTokens, T - t0);
  const int s = blockIdx.z;
  const int e = blockIdx.x * kPartExperts + warp;
  const uint4* wr = reinterpret_cast<const uint4*>(w_router + static_cast<size_t>(min(e, E - 1)) * H);
  float acc[kPartTokens];
#pragma unroll
  for (int tt = 0; tt < kPartTokens; ++tt) acc[tt] = 0.f;
  for (int b0 = 0; b0 < slice_units; b0 += kBurst) {
    const int u0 = s * slice_units + b0;
    const int nb = min(kBurst, slice_units - b0);
    for (int i = threadIdx.x; i < kPartTokens * nb; i += blockDim.x) {
      const int tt = i / nb, u = i - tt * nb;
      xs[tt * kBurst + u] =
          tt < nt ? __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0 + tt) * H) + u0 + u)
                  : make_uint4(0, 0, 0, 0);
    }
    uint4 wb[kPartMaxUnits];
#pragma unroll
    for (int b = 0; b < kPartMaxUnits; ++b) {
      const int u = b * 32 + lane;
      wb[b] = (e < E && u < nb) ? __ldg(wr + u0 + u) : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();
#pragma unroll
    for (int b = 0; b < kPartMaxUnits; ++b) {
      const int u = b * 32 + lane;
      if (u < nb) {
        float wv[8];
        Vec<TIn>::widen(wb[b], wv);
#pragma unroll
        for (int tt = 0; tt < kPartTokens; ++tt) {
          float xv[8];
          Vec<TIn>::widen(xs[tt * kBurst + u], xv);
#pragma unroll
          for (int j = 0; j < V; ++j) acc[tt] = fmaf(xv[j], wv[j], acc[tt]);
        }
      }
    }
    __syncthreads();
  }
  if (e >= E) return;
#pragma unroll
  for (int tt = 0; tt < kPartTokens; ++tt) {
    const float v = warp_sum(acc[tt]);
    if (lane == 0 && tt < nt) partial[(static_cast<size_t>(s) * T + t0 + tt) * E + e] = v;
  }
}

constexpr int kTopkWarps = 4;

// One warp per token: logits = sum of `S` partial slices (in slice order) + bias, written
// to logits_out when given; then the warp top-k.
__global__ void __launch_bounds__(kTopkWarps * 32)
    topk_kernel(const float* __restrict__ partial, int S, const float* __restrict__ bias,
                float* __restrict__ logits_out, int32_t* __restrict__ ids, float* __restrict__ w,
                int T, int E, int K, float theta) {
  extern __shared__ float Ls_all[];
  grid_dep_wait();
  grid_dep_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTopkWarps + warp;
  if (t >= T) return;
  float* Ls = Ls_all + warp * E;
  for (int e = lane; e < E; e += 32) {
    float v = 0.f;
    for (int s0 = 0; s0 < S; s0 += 8) {  // 8 slice loads in flight, summed in order
      float q[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        q[j] = s0 + j < S ? partial[(static_cast<size_t>(s0 + j) * T + t) * E + e] : 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (s0 + j < S) v += q[j];
    }
    if (bias != nullptr) v += bias[e];
    if (logits_out != nullptr) logits_out[static_cast<size_t>(t) * E + e] = v;
    Ls[e] = v;
  }
  __syncwarp();
  warp_topk_softmax(Ls, E, K, theta, ids + static_cast<size_t>(t) * K,
                    w + static_cast<size_t>(t) * K);
}

}  // namespace

int router_slices(int T, int H, int E, int dtype) {
  const int row_units = static_cast<int>(static_cast<size_t>(H) * act_bytes(dtype) / 16);
  const int eb = (E + kPartExperts - 1) / kPartExperts;
  const int tb = (T + kPartTokens - 1) / kPartTokens;
  const int min_su = row_units < 32 ? row_units : 32;  // at least one unit per lane
  int best = row_units;                                // one unit per slice always divides
  // the fewest slices (each a divisor of the row, 32..256 units) that give enough blocks
  for (int s = 1; s <= row_units; ++s) {
    if (row_units % s != 0) continue;
    const int su = row_units / s;
    if (su > 32 * kPartMaxUnits) continue;
    if (su < min_su) break;
    best = s;
    if (static_cast<long long>(eb) * tb * s >= kRouterTargetBlocks) break;
  }
  return best;
}

bool router_uses_wsmem(int dtype, int T, int H, int E) {
  return E <= kWsMaxE && static_cast<size_t>(E) * H * act_bytes(dtype) <= kWsMaxWeightBytes &&
         T >= 64;
}

cudaError_t launch_router_wsmem(int dtype, const void* x, const void* w_router,
                                const float* bias, float* logits, int32_t* ids, float* w, int T,
                                int H, int E, int K, float theta, unsigned* err, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(E) * H * act_bytes(dtype) + 8 * kWsMaxE * sizeof(float);
  static int attr_dev = -1;  // opt in to more than 48 KB of dynamic shared memory once
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_dev != dev) {
    cudaError_t e1 = cudaFuncSetAttribute(router_wsmem_kernel<__nv_bfloat16>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(kWsMaxWeightBytes + 1024));
    cudaError_t e2 = cudaFuncSetAttribute(router_wsmem_kernel<float>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(kWsMaxWeightBytes + 1024));
    if (e1 != cudaSuccess) return e1;
    if (e2 != cudaSuccess) return e2;
    attr_dev = dev;
  }
  const int blocks = (T + 7) / 8 < kWsMaxBlocks ? (T + 7) / 8 : kWsMaxBlocks;
  if (dtype == kBF16)
    return launch_pdl(router_wsmem_kernel<__nv_bfloat16>, dim3(blocks), dim3(256), smem, s,
                      static_cast<const __nv_bfloat16*>(x),
                      static_cast<const __nv_bfloat16*>(w_router), bias, logits, ids, w, T, H, E,
                      K, theta, err);
  return launch_pdl(router_wsmem_kernel<float>, dim3(blocks), dim3(256), smem, s,
                    static_cast<const float*>(x), static_cast<const float*>(w_router), bias,
                    logits, ids, w, T, H, E, K, theta, err);
}

cudaError_t launch_router_partial(int dtype, const void* x, const void* w_router, float* partial,
                                  int S, int T, int H, int E, cudaStream_t s) {
  const int row_units = static_cast<int>(static_cast<size_t>(H) * act_bytes(dtype) / 16);
  const int su = row_units / S;
  const size_t smem = 0;
  const int tb = (T + kPartTokens - 1) / kPartTokens;
  if (tb > 65535 || S > 65535) return cudaErrorInvalidValue;
  const dim3 grid((E + kPartExperts - 1) / kPartExperts, tb, S);
  if (dtype == kBF16)
    return launch_pdl(router_partial_kernel<__nv_bfloat16>, grid, dim3(kPartExperts * 32), smem, s,
                      static_cast<const __nv_bfloat16*>(x),
                      static_cast<const __nv_bfloat16*>(w_router), partial, T, H, E, su);
  return launch_pdl(router_partial_kernel<float>, grid, dim3(kPartExperts * 32), smem, s,
                    static_cast<const float*>(x), static_cast<const float*>(w_router), partial, T,
                    H, E, su);
}

cudaError_t launch_topk(const float* partial, int S, const float* bias, float* logits_out,
                        int32_t* ids, float* w, int T, int E, int K, float theta,
                        cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kTopkWarps - 1) / kTopkWarps;
  const size_t smem = static_cast<size_t>(kTopkWarps) * E * sizeof(float);
  return launch_pdl(topk_kernel, dim3(blocks), dim3(kTopkWarps * 32), smem, s, partial, S, bias,
                    logits_out, ids, w, T, E, K, theta);
}

}  // namespace moe
