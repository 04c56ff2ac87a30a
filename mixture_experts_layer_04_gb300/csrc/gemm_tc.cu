// Grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
// Page opening "MoE通过稀疏激活降低每个token的计算量…", section "单机MoE执行流水线": a
// grouped GEMM runs several experts' matrices, whose row counts differ, in one kernel
// launch; grouping changes the number of launches, not the matrices.  Section
// "一个批次如何变成各专家专属的矩阵": prefill gives experts many rows (matrix efficiency
// matters), decode gives them few (weight reads dominate).
//
// Design (one persistent CTA per SM, 192 threads):
//   warp 0     TMA producer: for every tile and k-block, loads a 128x64 bf16 tile of A
//              (token rows) and a BNx64 bf16 tile of B (expert weight rows) into a
//              STAGES-deep shared-memory ring (128-byte swizzle), signalling an mbarrier.
//   warp 1     MMA issuer: one elected thread issues tcgen05.mma (M=128, N=BN, K=16,
//              bf16 x bf16 -> fp32) into one of two TMEM accumulators, frees each smem
//              stage with tcgen05.commit, and signals the epilogue per finished tile.
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (each warp owns 32 TMEM lanes =
//              32 rows), SwiGLU or plain fp32 (+ column bias), staging through a swizzled
//              per-warp shared buffer, then coalesced row-masked global stores.
// The two accumulators let the epilogue of tile i overlap the main loop of tile i+1.
//
// Ragged groups: the m-tile table lists, per 128-row tile, its expert and the row range
// it owns.  A tile's TMA load may read rows of the next expert (or zero-filled rows past
// the end of A); those rows are computed but never stored.  Tiles are rasterised in
// groups of `swz` m-tiles so that the CTAs resident at one time share weight tiles in L2.
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int BM = kTcBM;  // 128
constexpr int BK = 64;     // bf16 elements = 128 bytes = one swizzle row
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kSwz = 8;

struct __align__(64) TcParams {
  CUtensorMap tmA;
  CUtensorMap tmB;
  void* C;
  const float* col_bias;
  const int32_t* offsets;  // [num_groups+1] row offsets of the groups in A, or null
  unsigned* err;
  int num_groups;
  int rows_alloc;
  int num_kb;
  int N_out;
  int n_tiles;
  int up_offset;
  int swz;
};

template <int BN, int MODE>
struct TcCfg {
  static constexpr int kABytes = BM * BK * 2;
  static constexpr int kBBytes = BN * BK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStagesRaw = (200 * 1024) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
  static constexpr int kBnOut = MODE == kSwiGLU ? BN / 2 : BN;
  static constexpr int kTmemCols = 2 * BN;
  static constexpr int kRowBytes = MODE == kSwiGLU ? 64 : 128;  // staged bytes per row per chunk
  static constexpr int kStgBytes = kEpiWarps * 32 * kRowBytes;
  static constexpr int kBarBytes = 256;
  static constexpr int kSchedBytes = 2 * 1028 * 4 + 32 * 4;  // offsets, m-tile prefix, scratch
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kStgBytes + kBarBytes + kSchedBytes;
  static_assert(kTmemCols >= 32 && kTmemCols <= 512 && (kTmemCols & (kTmemCols - 1)) == 0,
                "TMEM columns must be a power of two in [32, 512]");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M=128");
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

// Tile idx -> (group g, rows row0..row_end-1 of A, n_tile).  s_off holds the group row
// offsets and s_mt the exclusive prefix of m-tiles per group (both in shared memory).
__device__ __forceinline__ void decode_tile(const TcParams& p, const int* s_off, const int* s_mt,
                                            int num_mt, int idx, int& g, int& row0,
                                            int& row_end, int& n_tile) {
  const int gsz = p.swz * p.n_tiles;
  const int grp = idx / gsz;
  const int rem = idx - grp * gsz;
  const int m_first = grp * p.swz;
  const int m_cnt = min(p.swz, num_mt - m_first);
  n_tile = rem / m_cnt;
  const int mt = m_first + (rem - n_tile * m_cnt);
  if (p.offsets != nullptr) {
    int lo = 0, hi = p.num_groups - 1;  // last group with s_mt[g] <= mt
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_mt[mid] <= mt) lo = mid; else hi = mid - 1;
    }
    g = lo;
    row0 = s_off[g] + (mt - s_mt[g]) * BM;
    row_end = s_off[g + 1];
  } else {
    g = 0;
    row0 = mt * BM;
    row_end = p.rows_alloc;
  }
}

// Swizzled offset of 16-byte unit u of row r in a per-warp staging buffer.
template <int RB>
__device__ __forceinline__ uint32_t stg_off(int r, int u) {
  if constexpr (RB == 128)
    return static_cast<uint32_t>(r * 128 + ((u ^ (r & 7)) << 4));
  else
    return static_cast<uint32_t>(r * 64 + ((u ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

template <int BN, int MODE>
__global__ void __launch_bounds__(kThreads, 1) tc_grouped_gemm_kernel(const __grid_constant__ TcParams p) {
  using Cfg = TcCfg<BN, MODE>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * Cfg::kABytes;
  uint8_t* sStg = sB + S * Cfg::kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + Cfg::kStgBytes);
  // bars: full[S], empty[S], tfull[2], tempty[2], mma_done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_off = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + Cfg::kBarBytes);
  int* s_mt = s_off + 1028;
  int* s_scan = s_mt + 1028;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t mma_done_bar = bar0 + 8u * (2 * S + 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kEpiWarps);
    }
    mbar_init(mma_done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmA);
    tma_prefetch_desc(&p.tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Ragged schedule: every CTA derives the m-tiles of every group from the offsets.
  int num_mt;
  if (p.offsets != nullptr) {
    const int G = p.num_groups;
    for (int i = threadIdx.x; i <= G; i += blockDim.x) s_off[i] = p.offsets[i];
    __syncthreads();
    const int per = (G + blockDim.x - 1) / blockDim.x;
    const int beg = min(G, static_cast<int>(threadIdx.x) * per), end = min(G, beg + per);
    int mine = 0;
    for (int q = beg; q < end; ++q) mine += (s_off[q + 1] - s_off[q] + BM - 1) / BM;
    int all = 0;
    int run = block_exclusive_scan(mine, s_scan, &all);
    for (int q = beg; q < end; ++q) {
      s_mt[q] = run;
      run += (s_off[q + 1] - s_off[q] + BM - 1) / BM;
    }
    if (threadIdx.x == 0) s_mt[G] = all;
    __syncthreads();
    num_mt = all;
  } else {
    num_mt = (p.rows_alloc + BM - 1) / BM;
  }
  const int total = num_mt * p.n_tiles;

  if (warp == 0) {
    // ------------------------------------------------------------ producer ----
    if (elect_one_sync()) {
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int idx = blockIdx.x; idx < total && ok; idx += gridDim.x) {
        int g, row0, row_end, n_tile;
        decode_tile(p, s_off, s_mt, num_mt, idx, g, row0, row_end, n_tile);
        const int n0 = n_tile * Cfg::kBnOut;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
          const uint32_t a_dst = smem_u32(sA + stage * Cfg::kABytes);
          const uint32_t b_dst = smem_u32(sB + stage * Cfg::kBBytes);
          tma_load_2d(a_dst, &p.tmA, fb, kb * BK, row0);
          if constexpr (MODE == kSwiGLU) {
            tma_load_3d(b_dst, &p.tmB, fb, kb * BK, n0, g);
            tma_load_3d(b_dst + (BN / 2) * 128, &p.tmB, fb, kb * BK, p.up_offset + n0, g);
          } else {
            tma_load_3d(b_dst, &p.tmB, fb, kb * BK, n0, g);
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: the most recent load of every stage must have landed before the CTA
      // may exit (they all have in a normal run; this matters only after an abort).
      const int n = issued < S ? static_cast<int>(issued) : S;
      int s = stage;
      uint32_t ph = phase;
      volatile int no_abort = 0;
      for (int j = 0; j < n; ++j) {
        if (--s < 0) {
          s = S - 1;
          ph ^= 1u;
        }
        mbar_wait(full_bar(s), ph, &no_abort, p.err);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA ----
    if (elect_one_sync()) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int idx = blockIdx.x; idx < total && ok; idx += gridDim.x, ++local) {
        const int acc = local & 1;
        const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
        if (!mbar_wait(tempty_bar(acc), acc_phase ^ 1u, abort_flag, p.err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(full_bar(stage), phase, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(sA + stage * Cfg::kABytes);
          const uint32_t b_base = smem_u32(sB + stage * Cfg::kBBytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(a_base + kk * 32);
            const uint64_t bd = smem_desc_sw128(b_base + kk * 32);
            tc_mma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          tc_commit(empty_bar(stage));
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc_commit(tfull_bar(acc));
      }
      if (!ok || *abort_flag) {
        // make sure no MMA is still reading shared memory or writing TMEM
        tc_commit(mma_done_bar);
        volatile int no_abort = 0;
        mbar_wait(mma_done_bar, 0, &no_abort, p.err);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue ----
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    const uint32_t stg = smem_u32(sStg) + static_cast<uint32_t>((warp - 2) * 32 * Cfg::kRowBytes);
    int local = 0;
    for (int idx = blockIdx.x; idx < total; idx += gridDim.x, ++local) {
      int g, row0, row_end, n_tile;
      decode_tile(p, s_off, s_mt, num_mt, idx, g, row0, row_end, n_tile);
      const int acc = local & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
      if (!mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.err)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
      const int tile_row0 = row0 + quad * 32;  // first global row of this warp's 32 rows
      const int col0 = n_tile * Cfg::kBnOut;
      if constexpr (MODE == kSwiGLU) {
        __nv_bfloat16* C = static_cast<__nv_bfloat16*>(p.C);
#pragma unroll 1
        for (int c = 0; c < BN / 2; c += 32) {
          uint32_t gr[32], ur[32];
          tmem_ld_32x32b_x32(t_row + c, gr);
          tmem_ld_32x32b_x32(t_row + BN / 2 + c, ur);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float h0 = silu_f(__uint_as_float(gr[2 * j])) * __uint_as_float(ur[2 * j]);
            const float h1 =
                silu_f(__uint_as_float(gr[2 * j + 1])) * __uint_as_float(ur[2 * j + 1]);
            pk[j] = pack_bf16x2(h0, h1);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u)
            st_shared_v4(stg + stg_off<64>(lane, u), pk[4 * u], pk[4 * u + 1], pk[4 * u + 2],
                         pk[4 * u + 3]);
          __syncwarp();
#pragma unroll
          for (int pass = 0; pass < 4; ++pass) {
            const int rr = pass * 8 + (lane >> 2), u = lane & 3;
            const uint4 v = ld_shared_v4(stg + stg_off<64>(rr, u));
            const int grow = tile_row0 + rr;
            const int col = col0 + c + u * 8;
            if (grow < row_end && col < p.N_out)
              *reinterpret_cast<uint4*>(C + static_cast<size_t>(grow) * p.N_out + col) = v;
          }
          __syncwarp();
        }
      } else {
        float* C = static_cast<float*>(p.C);
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_row + c, r);
          tmem_ld_wait();
          if (p.col_bias != nullptr) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int col = col0 + c + j;
              const float b = col < p.N_out ? __ldg(p.col_bias + col) : 0.f;
              r[j] = __float_as_uint(__uint_as_float(r[j]) + b);
            }
          }
#pragma unroll
          for (int u = 0; u < 8; ++u)
            st_shared_v4(stg + stg_off<128>(lane, u), r[4 * u], r[4 * u + 1], r[4 * u + 2],
                         r[4 * u + 3]);
          __syncwarp();
#pragma unroll
          for (int pass = 0; pass < 8; ++pass) {
            const int rr = pass * 4 + (lane >> 3), u = lane & 7;
            const uint4 v = ld_shared_v4(stg + stg_off<128>(rr, u));
            const int grow = tile_row0 + rr;
            const int col = col0 + c + u * 4;
            if (grow < row_end && col < p.N_out)
              *reinterpret_cast<uint4*>(C + static_cast<size_t>(grow) * p.N_out + col) = v;
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty_bar(acc));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, Cfg::kTmemCols);
}

// ------------------------------------------------------------------ host ----
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 2D bf16 map of a row-major [rows, cols] matrix, box = box_rows x 64 columns.
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3D bf16 map of [G, rows, cols], box = 1 x box_rows x 64 columns.
bool make_map_3d(CUtensorMap* m, const void* base, uint64_t G, uint64_t rows, uint64_t cols,
                 uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {cols, rows, G};
  cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int MODE>
cudaError_t launch_one(const GroupedGemm& g, unsigned* err, int num_sms, cudaStream_t s) {
  using Cfg = TcCfg<BN, MODE>;
  static int attr_set_dev = -1;  // per-process: the attribute is per function and device
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_set_dev != dev) {
    cudaError_t e = cudaFuncSetAttribute(tc_grouped_gemm_kernel<BN, MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    attr_set_dev = dev;
  }
  TcParams p;
  memset(&p, 0, sizeof(p));
  const uint32_t b_box = MODE == kSwiGLU ? BN / 2 : BN;
  if (!make_map_2d(&p.tmA, g.A, static_cast<uint64_t>(g.rows_alloc), static_cast<uint64_t>(g.Kd), BM))
    return cudaErrorInvalidValue;
  if (!make_map_3d(&p.tmB, g.B, static_cast<uint64_t>(g.G), static_cast<uint64_t>(g.Nb),
                   static_cast<uint64_t>(g.Kd), b_box))
    return cudaErrorInvalidValue;
  p.C = g.C;
  p.col_bias = g.col_bias;
  p.offsets = g.offsets;
  p.num_groups = g.G;
  p.err = err;
  p.rows_alloc = g.rows_alloc;
  p.num_kb = g.Kd / BK;
  p.N_out = g.N_out;
  p.n_tiles = (g.N_out + Cfg::kBnOut - 1) / Cfg::kBnOut;
  p.up_offset = g.up_offset;
  p.swz = kSwz;
  const long long max_mt =
      g.offsets != nullptr ? (g.rows_alloc + BM - 1) / BM + g.G : (g.rows_alloc + BM - 1) / BM;
  const long long max_tiles = max_mt * p.n_tiles;
  if (max_tiles == 0) return cudaSuccess;
  const int grid = static_cast<int>(max_tiles < num_sms ? max_tiles : num_sms);
  tc_grouped_gemm_kernel<BN, MODE><<<grid, kThreads, Cfg::kSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm_tc(const GroupedGemm& g, unsigned* err, int num_sms,
                                   cudaStream_t s) {
  if (g.dtype != kBF16) return cudaErrorInvalidValue;
  if (g.mode == kSwiGLU) return launch_one<256, kSwiGLU>(g, err, num_sms, s);
  if (g.N_out > 128) return launch_one<256, kPlain>(g, err, num_sms, s);
  if (g.N_out > 64) return launch_one<128, kPlain>(g, err, num_sms, s);
  return launch_one<64, kPlain>(g, err, num_sms, s);
}

}  // namespace moe
