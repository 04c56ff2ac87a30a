// Grouped GEMM on the tensor cores for float32 layers, at float32 accuracy.
//
// Page opening "MoE通过稀疏激活降低每个token的计算量…", section "单机MoE执行流水线": each
// expert's rows form one matrix and the experts run as one grouped GEMM.  The float32
// layer keeps its operands in float32.  The tensor cores take them as tf32 (10 mantissa
// bits), so every operand v is split into a tf32 part and a remainder,
//     hi = v with its low 13 mantissa bits cleared,   lo = v - hi   (exact in float32),
// and each k-step issues three kind::tf32 MMAs: hi*hi + hi*lo + lo*hi.  The dropped lo*lo
// term and the tf32 reading of lo each contribute about 2^-20 of |a*b|, so the sums keep
// the accuracy of a float32 dot product.
//
// Tiles: the weights on the MMA's 128-row side (128 weight rows; for SwiGLU 64 gate rows
// and the 64 matching up rows), 64 token rows of one group (an entry of the m-tile table)
// as N.  TMEM lane = weight row (output feature), column = token row.  Per CTA one tile:
//   warp 0    TMA producer: weights [G, Nb, Kd] and token rows [rows, Kd] in 128-byte
//             k-steps (32 floats) with the 128-byte swizzle, 4 stages ahead (2, with two
//             CTAs per SM, when the grid has more tiles than the GPU has SMs);
//   warps 2-5 split every landed stage into hi (in place) and lo (a second buffer), then
//             run the epilogue;
//   warp 1    allocates TMEM and issues the MMAs; tcgen05.commit frees each stage.
// Epilogue: plain (fp32 store, optional column bias) or SwiGLU (the up half reaches the
// gate half's warps through shared memory; h = silu(g) * u in float32).
// Every wait is bounded and reports through the device error word.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kTfThreads = 192;
constexpr int kTfRowsW = 128;   // weight rows per tile (MMA M)
constexpr int kTfRowsT = kF32TileRows;  // token rows per tile (MMA N), one m-tile table entry
constexpr int kTfKStep = 32;    // floats per 128-byte k-step
constexpr int kWBytes = kTfRowsW * 128;  // 16 KB
constexpr int kTBytes = kTfRowsT * 128;  // 8 KB
constexpr int kHiBytes = kWBytes + kTBytes;
constexpr int kStageBytes = 2 * kHiBytes;  // hi (weights, tokens) then lo (same layout)
constexpr int kXchgStride = kTfRowsT + 1;  // floats per exchange row (bank spread)
constexpr int kXchgBytes = 64 * kXchgStride * 4;  // reuses stage 0 once the MMAs are done
// Stages: 4 with one CTA per SM, or 2 with two CTAs per SM when the grid has more tiles
// than the GPU has SMs (the same bytes in flight per SM, and one wave instead of two).
template <int S>
constexpr int tf_smem() {
  return 1024 + S * kStageBytes + 256;
}
static_assert(kXchgBytes <= kStageBytes, "exchange buffer inside stage 0");
static_assert(kTfRowsT == 64, "MMA N = 64 token rows");
static_assert(tf_smem<4>() <= 232448, "shared memory per CTA");
static_assert(2 * (tf_smem<2>() + 1024) <= 233472, "two CTAs per SM");

struct TfParams {
  CUtensorMap tmW;  // [G, Nb, Kd] fp32, box 32 x (64 or 128) x 1
  CUtensorMap tmA;  // [rows_alloc, Kd] fp32, box 32 x 64
  float* C;
  const float* col_bias;
  const int4* table;  // {group, row0, group end, 0} per m-tile, or null (one group)
  const int32_t* num_mt;
  unsigned* err;
  int rows_alloc, num_kb, N_out, up_offset;
};

// tcgen05 instruction descriptor, kind::tf32: D f32 (bits 4-5 = 1), A and B tf32 (bits
// 7-9 and 10-12 = 2), both K-major, N >> 3 at bit 17, M >> 4 at bit 24.
constexpr uint32_t idesc_tf32_f32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Generic-proxy writes to shared memory become visible to the tensor core (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier of the four split/epilogue warps.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// The same barrier, returning to every one of the four warps whether any thread passed
// `pred` true, so that they leave a loop together or not at all.
__device__ __forceinline__ bool epi_bar_any_tf(bool pred) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, 128, q;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(out)
      : "r"(pred ? 1u : 0u)
      : "memory");
  return out != 0u;
}

__device__ __forceinline__ float4 split_hi(float4& v) {
  float4 hi;
  hi.x = __uint_as_float(__float_as_uint(v.x) & 0xFFFFE000u);
  hi.y = __uint_as_float(__float_as_uint(v.y) & 0xFFFFE000u);
  hi.z = __uint_as_float(__float_as_uint(v.z) & 0xFFFFE000u);
  hi.w = __uint_as_float(__float_as_uint(v.w) & 0xFFFFE000u);
  v.x -= hi.x;
  v.y -= hi.y;
  v.z -= hi.z;
  v.w -= hi.w;
  return hi;
}

template <int MODE, int kTfStages>
__global__ void __launch_bounds__(kTfThreads, kTfStages == 2 ? 2 : 1)
    tf32x3_gemm_kernel(const __grid_constant__ TfParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // SwiGLU epilogue exchange: stage 0's buffer, free once the last MMA has completed
  float* xchg = reinterpret_cast<float*>(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kTfStages * kStageBytes);
  // bars: full[S], split[S], empty[S], tfull, mma_done; then the TMEM slot and abort flag
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * kTfStages + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  static_assert(8 * (3 * kTfStages + 2) + 8 <= 256, "barrier region");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto split_bar = [&](int s) { return bar0 + 8u * (kTfStages + s); };
  auto empty_bar = [&](int s) { return bar0 + 8u * (2 * kTfStages + s); };
  const uint32_t tfull_bar = bar0 + 8u * (3 * kTfStages);
  const uint32_t mma_done_bar = bar0 + 8u * (3 * kTfStages + 1);

  grid_dep_wait();
  grid_dep_trigger();
  // the tile: m-tile table entry blockIdx.y, weight tile blockIdx.x
  const int mt = blockIdx.y;
  int g, row0, row_end;
  if (p.table != nullptr) {
    if (mt >= *p.num_mt) return;
    const int4 ent = p.table[mt];
    g = ent.x;
    row0 = ent.y;
    row_end = min(ent.z, ent.y + kTfRowsT);
  } else {
    g = 0;
    row0 = mt * kTfRowsT;
    row_end = min(p.rows_alloc, row0 + kTfRowsT);
    if (row0 >= p.rows_alloc) return;
  }
  constexpr int kColsOut = MODE == kSwiGLU ? kTfRowsW / 2 : kTfRowsW;
  const int n0 = blockIdx.x * kColsOut;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kTfStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(split_bar(s), 4);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(tfull_bar, 1);
    mbar_init(mma_done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmW);
    tma_prefetch_desc(&p.tmA);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int nk = p.num_kb;

  if (warp == 0) {
    // ------------------------------------------------------------ producer ----
    if (elect_one_sync()) {
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) break;
        const uint32_t base = smem_u32(smem + stage * kStageBytes);
        const uint32_t fb = full_bar(stage);
        mbar_arrive_expect_tx(fb, kHiBytes);
        if constexpr (MODE == kSwiGLU) {
          tma_load_3d(base, &p.tmW, fb, kb * kTfKStep, n0, g);
          tma_load_3d(base + kWBytes / 2, &p.tmW, fb, kb * kTfKStep, p.up_offset + n0, g);
        } else {
          tma_load_3d(base, &p.tmW, fb, kb * kTfKStep, n0, g);
        }
        tma_load_2d(base + kWBytes, &p.tmA, fb, kb * kTfKStep, row0);
        ++issued;
        if (++stage == kTfStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // every load issued must land before the CTA may exit
      const int n = issued < kTfStages ? issued : kTfStages;
      int s = stage;
      uint32_t ph = phase;
      volatile int no_abort = 0;
      for (int j = 0; j < n; ++j) {
        if (--s < 0) {
          s = kTfStages - 1;
          ph ^= 1u;
        }
        mbar_wait(full_bar(s), ph, &no_abort, p.err);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA ----
    if (elect_one_sync()) {
      constexpr uint32_t idesc = idesc_tf32_f32(kTfRowsW, kTfRowsT);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {
        if (!mbar_wait(split_bar(stage), phase, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t w_hi = smem_u32(smem + stage * kStageBytes);
        const uint32_t t_hi = w_hi + kWBytes;
        const uint32_t w_lo = w_hi + kHiBytes;
        const uint32_t t_lo = t_hi + kHiBytes;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {  // 8 floats (32 bytes) per MMA
          const uint32_t o = kk * 32;
          tc_mma_tf32(tmem_base, smem_desc_sw128(w_hi + o), smem_desc_sw128(t_hi + o), idesc,
                      (kb | kk) != 0 ? 1u : 0u);
          tc_mma_tf32(tmem_base, smem_desc_sw128(w_hi + o), smem_desc_sw128(t_lo + o), idesc, 1u);
          tc_mma_tf32(tmem_base, smem_desc_sw128(w_lo + o), smem_desc_sw128(t_hi + o), idesc, 1u);
        }
        tc_commit(empty_bar(stage));
        if (++stage == kTfStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) {
        tc_commit(tfull_bar);
      } else {
        // no MMA may still read shared memory or write TMEM when the CTA exits
        tc_commit(mma_done_bar);
        volatile int no_abort = 0;
        mbar_wait(mma_done_bar, 0, &no_abort, p.err);
      }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------- split, epilogue ----
    const int et = threadIdx.x - 64;  // 0..127
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int kb = 0; kb < nk; ++kb) {
      const bool landed = mbar_wait(full_bar(stage), phase, abort_flag, p.err);
      if (epi_bar_any_tf(!landed || *abort_flag != 0)) {
        ok = false;
        break;
      }
      float4* hi = reinterpret_cast<float4*>(smem + stage * kStageBytes);
      float4* lo = reinterpret_cast<float4*>(smem + stage * kStageBytes + kHiBytes);
#pragma unroll
      for (int i = 0; i < kHiBytes / 16 / 128; ++i) {
        const int idx = et + 128 * i;
        float4 v = hi[idx];
        const float4 h = split_hi(v);
        hi[idx] = h;
        lo[idx] = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(split_bar(stage));
      if (++stage == kTfStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (ok) ok = mbar_wait(tfull_bar, 0, abort_flag, p.err);
    ok = !epi_bar_any_tf(!ok);
    if (ok) {
      tc_fence_after();
      const int quad = warp & 3;          // TMEM lanes 32*quad .. 32*quad+31
      const int L = quad * 32 + lane;     // weight row of the tile
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
      if constexpr (MODE == kSwiGLU) {
        // lanes 64-127: up rows, handed to the gate lanes through shared memory
        if (quad >= 2) {
          const int r = L - 64;
#pragma unroll 1
          for (int c = 0; c < kTfRowsT; c += 32) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_row + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) xchg[r * kXchgStride + c + j] = __uint_as_float(v[j]);
          }
        }
        epi_sync();
        if (quad < 2) {
          const int col = n0 + L;
#pragma unroll 1
          for (int c = 0; c < kTfRowsT; c += 32) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(t_row + c, v);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int row = row0 + c + j;
              if (row < row_end && col < p.N_out) {
                const float u = xchg[L * kXchgStride + c + j];
                p.C[static_cast<size_t>(row) * p.N_out + col] = silu_f(__uint_as_float(v[j])) * u;
              }
            }
          }
        }
      } else {
        const int col = n0 + L;
        const float b = (p.col_bias != nullptr && col < p.N_out) ? __ldg(p.col_bias + col) : 0.f;
#pragma unroll 1
        for (int c = 0; c < kTfRowsT; c += 32) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(t_row + c, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int row = row0 + c + j;
            if (row < row_end && col < p.N_out)
              p.C[static_cast<size_t>(row) * p.N_out + col] = __uint_as_float(v[j]) + b;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, 64);
}

// ------------------------------------------------------------------ host ----
PFN_cuTensorMapEncodeTiled_v12000 tf_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// fp32 maps, 128-byte swizzle, box = 32 floats (one 128-byte row) x box_rows
bool make_map_f32(CUtensorMap* m, const void* base, int rank, const uint64_t* dims_rows_first,
                  uint32_t box_rows) {
  auto fn = tf_encode_fn();
  if (fn == nullptr) return false;
  // dims_rows_first: {cols, rows} or {cols, rows, G}
  cuuint64_t dims[3] = {dims_rows_first[0], dims_rows_first[1], rank == 3 ? dims_rows_first[2] : 1};
  cuuint64_t strides[2] = {dims[0] * 4, dims[0] * dims[1] * 4};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kTfKStep), box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int S>
cudaError_t launch_tf32(const GroupedGemm& g, unsigned* err, dim3 grid, cudaStream_t s) {
  static int attr_set_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  auto kernel = tf32x3_gemm_kernel<MODE, S>;
  if (attr_set_dev != dev) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tf_smem<S>());
    if (e != cudaSuccess) return e;
    attr_set_dev = dev;
  }
  TfParams p;
  std::memset(&p, 0, sizeof(p));
  const uint64_t wdims[3] = {static_cast<uint64_t>(g.Kd), static_cast<uint64_t>(g.Nb),
                             static_cast<uint64_t>(g.G)};
  const uint64_t adims[2] = {static_cast<uint64_t>(g.Kd), static_cast<uint64_t>(g.rows_alloc)};
  if (!make_map_f32(&p.tmW, g.B, 3, wdims, MODE == kSwiGLU ? kTfRowsW / 2 : kTfRowsW) ||
      !make_map_f32(&p.tmA, g.A, 2, adims, kTfRowsT))
    return cudaErrorInvalidValue;
  p.C = static_cast<float*>(g.C);
  p.col_bias = MODE == kSwiGLU ? nullptr : g.col_bias;
  p.table = g.mtile_table;
  p.num_mt = g.num_mtiles;
  p.err = err;
  p.rows_alloc = g.rows_alloc;
  p.num_kb = g.Kd / kTfKStep;
  p.N_out = g.N_out;
  p.up_offset = g.up_offset;
  return launch_pdl(kernel, grid, dim3(kTfThreads), tf_smem<S>(), s, p);
}

template <int MODE>
cudaError_t launch_tf32_mode(const GroupedGemm& g, unsigned* err, int num_sms, cudaStream_t s) {
  constexpr int kColsOut = MODE == kSwiGLU ? kTfRowsW / 2 : kTfRowsW;
  const int mt = g.mtile_table != nullptr ? g.max_mtiles : (g.rows_alloc + kTfRowsT - 1) / kTfRowsT;
  if (mt == 0) return cudaSuccess;
  const dim3 grid((g.N_out + kColsOut - 1) / kColsOut, mt);
  if (static_cast<long long>(grid.x) * grid.y > num_sms)
    return launch_tf32<MODE, 2>(g, err, grid, s);
  return launch_tf32<MODE, 4>(g, err, grid, s);
}

}  // namespace

cudaError_t launch_grouped_gemm_tf32(const GroupedGemm& g, unsigned* err, int num_sms,
                                     cudaStream_t s) {
  if (g.dtype != kF32 || g.Kd % kTfKStep != 0 || g.rows_alloc == 0) return cudaErrorInvalidValue;
  if (g.mode == kSwiGLU) return launch_tf32_mode<kSwiGLU>(g, err, num_sms, s);
  if (g.mode == kPlain) return launch_tf32_mode<kPlain>(g, err, num_sms, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
