// Routing and dispatch of a decode-sized batch in one launch: one thread-block cluster.
//
// Page opening "MoE通过稀疏激活降低每个token的计算量但增加了服务系统的复杂度", section
// "单机MoE执行流水线": the router scores every expert, top-k keeps the chosen ids and
// weights, and the permutation writes token rows in expert order with an inverse map.
// Routing rule: "MoE大模型的智能调度：从1.8万亿参数到每token仅激活2%的工程真相" §2.2 steps 1-3.
//
// With a handful of tokens every step is latency-bound, and separate launches (router,
// top-k, counting sort, row copy) cost more than their work.  Here a cluster of nc CTAs
// (16 when the device allows it, else 8) does all of it, synchronised by cluster
// barriers and distributed shared memory instead of global counters.
//
// Up to kRdMaxT tokens (route_dispatch_dot_kernel), the logits are split by expert:
//   1. CTA c takes experts [c*E/nc, (c+1)*E/nc); warp w of it computes an expert's full-H
//      dot products with every token on the CUDA cores (the tokens staged in shared
//      memory, the router row read straight into registers), adds the bias and stores the
//      logit into every CTA's logit table through distributed shared memory.
//   2. One cluster barrier: every CTA now holds all T x E logits, takes every token's
//      top-k itself and runs step 3 below with no further exchange.
//   At one token this saves two of the three cluster barriers and the 16-way partial
//   sums (the routing of the Qwen3-shaped decode layer 12.5 -> 9.1 us); from 8 tokens on,
//   the dot products on the CUDA cores cost more than that.
// With more tokens (route_dispatch_cluster_kernel), the H dimension is split instead:
//   1. CTA c computes the partial logits of its share of the H dimension on the tensor
//      core: D[e][t] = sum over its k-blocks of W_r[e, k] x[t, k] (tcgen05.mma, experts
//      on the 128-row side, tokens zero-padded to npad columns), TMA-fed, and parks
//      them in shared memory as part[t][e] (fp32).
//   2. Cluster barrier.  Warp j of CTA c takes token t = c + nc*j: its logits are the
//      nc partials read through distributed shared memory and added in rank order (so
//      the result is the same on every run), plus the bias; then the warp top-k with
//      softmax and gate drop.
//   3. Cluster barrier.  Every CTA gathers all T*K expert ids and recomputes the stable
//      counting sort (per-expert token bit masks, a block scan for the offsets, ranks by
//      popcount), identically; CTA 0 stores counts, offsets, perm and inv; and, unless the
//      caller gathers rows itself, every CTA copies some token rows into x_perm.
// (Pushing the partials and the ids into the owners' shared memory with remote stores
// instead, one barrier fewer, measured slower: 4-byte remote stores from the TMEM
// read-out cost more than the loads they replace, 5 us more per layer at 64 tokens.)
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kRcThreads = 256;
constexpr int kRcWarps = kRcThreads / 32;
constexpr int kRcMaxT = 64;
constexpr int kRcMaxE = 256;
constexpr int kRcMaxK = 16;
constexpr int kRcMaxStages = 4;
constexpr int kRcSmemBudget = 200 * 1024;
constexpr int kRdMaxT = 4;    // tokens up to which the logits are CUDA-core dot products
constexpr int kRdChunk = 8;   // 16-byte units of a router row each lane holds at a time

struct RcParams {
  CUtensorMap tmX;  // x [T, H] bf16, box 64 columns x npad rows (rows >= T read as zero)
  CUtensorMap tmW;  // W_r [E, H] bf16, box 64 columns x 128 rows (rows >= E read as zero)
  const float* bias;
  float* logits;    // [T, E]
  int32_t* ids;     // [T, K]
  float* w;         // [T, K]
  int32_t* counts;  // [E] (null: routing only, no permutation)
  int32_t* offsets; // [E + 1]
  int32_t* perm;    // [T*K]
  int32_t* inv;     // [T*K]
  float* row_w;     // [T*K] gate of every row, or null
  const uint4* x;   // token rows (H*2/16 units each)
  const uint4* wr;  // router rows (H*2/16 units each)
  uint4* x_perm;    // x_perm[r] = x[perm[r]], or null: rows not copied
  unsigned* err;
  int T, H, E, K;
  int npad;       // tokens padded to a multiple of 16 (MMA N)
  int nmt;        // 128-row expert tiles (MMA M)
  int kb_total;   // k-blocks of 64 columns in H
  int stages;
  int tmem_cols;
  float theta;
};

struct RcLayout {
  int stage_bytes, stages_off, part_off, ls_off, bias_off, sid_off, sw_off, aid_off, agate_off,
      rows_off, masks_off, cnt_off, off_off, bar_off, total;
};

__host__ __device__ inline int rc_align(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline RcLayout rc_layout(int npad, int nmt, int E, int K, int T, int stages) {
  RcLayout L;
  L.stage_bytes = nmt * 128 * 128 + npad * 128;
  int o = 0;
  L.stages_off = o;
  o += stages * L.stage_bytes;
  L.part_off = o;
  o = rc_align(o + npad * E * 4, 16);
  L.ls_off = o;
  o = rc_align(o + kRcWarps * E * 4, 16);
  L.bias_off = o;
  o = rc_align(o + E * 4, 16);
  L.sid_off = o;
  o = rc_align(o + kRcWarps * K * 4, 16);
  L.sw_off = o;
  o = rc_align(o + kRcWarps * K * 4, 16);
  L.aid_off = o;
  o = rc_align(o + T * K * 4, 16);
  L.agate_off = o;
  o = rc_align(o + T * K * 4, 16);
  L.rows_off = o;
  o = rc_align(o + T * K * 4, 16);
  L.masks_off = o;
  o = rc_align(o + E * 2 * 4, 16);
  L.cnt_off = o;
  o = rc_align(o + E * 4, 16);
  L.off_off = o;
  o = rc_align(o + (E + 1) * 4, 16);
  L.bar_off = o;
  o += 8 * (2 * kRcMaxStages + 1) + 16 + 32 * 4;  // barriers, tmem slot, abort, scan scratch
  L.total = o + 1024;                            // slack for the 1024-byte alignment
  return L;
}

// Shared memory of the expert-split kernel: the tokens, the logit table, the top-k of every
// token and the counting-sort scratch.
struct RdLayout {
  int x_off, ls_off, sid_off, sw_off, rows_off, masks_off, cnt_off, off_off, scratch_off, total;
};

__host__ __device__ inline RdLayout rd_layout(int T, int H, int E, int K) {
  RdLayout L;
  int o = 0;
  L.x_off = o;
  o = rc_align(o + T * H * 2, 16);
  L.ls_off = o;
  o = rc_align(o + T * E * 4, 16);
  L.sid_off = o;
  o = rc_align(o + T * K * 4, 16);
  L.sw_off = o;
  o = rc_align(o + T * K * 4, 16);
  L.rows_off = o;
  o = rc_align(o + T * K * 4, 16);
  L.masks_off = o;
  o = rc_align(o + E * 2 * 4, 16);
  L.cnt_off = o;
  o = rc_align(o + E * 4, 16);
  L.off_off = o;
  o = rc_align(o + (E + 1) * 4, 16);
  L.scratch_off = o;
  L.total = o + 32 * 4;
  return L;
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t cluster_addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(cluster_addr) : "memory");
  return v;
}
__device__ __forceinline__ int ld_dsmem_s32(uint32_t cluster_addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(cluster_addr) : "memory");
  return v;
}
// Split cluster barrier: arrive now, wait later (no memory ordering: it only tells a CTA
// that every CTA of the cluster is running, before the first write into their shared memory).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// bf16 pair -> two floats (exact)
__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// Step 3 of both kernels, once every CTA holds all T*K expert ids `aid` (-1: dropped)
// and gates `agate` and has zeroed `masks`: the stable counting sort (redundantly in every
// CTA), CTA 0's stores of counts, offsets, perm, inv and row_w, and the row copies, dealt
// over the warps of the whole cluster.  No remote shared memory access.
__device__ __forceinline__ void rc_sort_and_dispatch(const RcParams& p, int c, int nc,
                                                     const int32_t* aid, const float* agate,
                                                     uint32_t* masks, int* cnt, int* off,
                                                     int32_t* rows, int* scratch) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int TK = p.T * p.K;
  for (int a = tid; a < TK; a += kRcThreads) {
    const int e = aid[a];
    if (e >= 0) {
      const int t = a / p.K;
      atomicOr(&masks[2 * e + (t >> 5)], 1u << (t & 31));
    }
  }
  __syncthreads();
  int cnt_e = 0;
  if (tid < p.E) cnt_e = __popc(masks[2 * tid]) + __popc(masks[2 * tid + 1]);
  int M = 0;
  const int base = block_exclusive_scan(cnt_e, scratch, &M);
  if (tid < p.E) {
    cnt[tid] = cnt_e;
    off[tid] = base;
  }
  if (tid == 0) off[p.E] = M;
  __syncthreads();
  for (int a = tid; a < TK; a += kRcThreads) {
    const int e = aid[a];
    int row = -1;
    if (e >= 0) {
      const int t = a / p.K;
      const uint32_t* m = masks + 2 * e;
      int r = __popc(m[t >> 5] & ((1u << (t & 31)) - 1u));
      if (t >= 32) r += __popc(m[0]);
      row = off[e] + r;
    }
    rows[a] = row;
  }
  __syncthreads();
  if (c == 0) {
    for (int e = tid; e < p.E; e += kRcThreads) p.counts[e] = cnt[e];
    for (int e = tid; e <= p.E; e += kRcThreads) p.offsets[e] = off[e];
    for (int a = tid; a < TK; a += kRcThreads) {
      const int r = rows[a];
      p.inv[a] = r;
      if (r >= 0) {
        p.perm[r] = a / p.K;
        if (p.row_w != nullptr) p.row_w[r] = agate[a];
      }
    }
  }
  // row copies: the T*K kept assignments are dealt to all warps of the cluster, two at a
  // time per warp (both rows' loads in flight, then both rows' stores), so every SM of the
  // cluster shares the stores; each lane moves 16-byte units in bursts of 4 per row
  if (p.x_perm != nullptr) {
    const int row_units = p.H / 8;
    constexpr int kBurst = 4;
    const int nw = nc * kRcWarps;
    for (int a0 = c * kRcWarps + warp; a0 < TK; a0 += 2 * nw) {
      const int a1 = a0 + nw;
      const int r0 = rows[a0], r1 = a1 < TK ? rows[a1] : -1;
      const uint4* s0 = p.x + static_cast<size_t>(a0 / p.K) * row_units;
      const uint4* s1 = p.x + static_cast<size_t>((a1 < TK ? a1 : a0) / p.K) * row_units;
      for (int i0 = 0; i0 < row_units; i0 += 32 * kBurst) {
        uint4 v0[kBurst], v1[kBurst];
#pragma unroll
        for (int b = 0; b < kBurst; ++b) {
          const int i = i0 + b * 32 + lane;
          if (i < row_units) {
            if (r0 >= 0) v0[b] = __ldg(s0 + i);
            if (r1 >= 0) v1[b] = __ldg(s1 + i);
          }
        }
#pragma unroll
        for (int b = 0; b < kBurst; ++b) {
          const int i = i0 + b * 32 + lane;
          if (i < row_units) {
            if (r0 >= 0) p.x_perm[static_cast<size_t>(r0) * row_units + i] = v0[b];
            if (r1 >= 0) p.x_perm[static_cast<size_t>(r1) * row_units + i] = v1[b];
          }
        }
      }
    }
  }
}

__global__ void __launch_bounds__(kRcThreads, 1)
    route_dispatch_cluster_kernel(const __grid_constant__ RcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const RcLayout L = rc_layout(p.npad, p.nmt, p.E, p.K, p.T, p.stages);
  float* part = reinterpret_cast<float*>(smem + L.part_off);
  float* Ls = reinterpret_cast<float*>(smem + L.ls_off);
  float* bias_s = reinterpret_cast<float*>(smem + L.bias_off);
  int32_t* sid = reinterpret_cast<int32_t*>(smem + L.sid_off);
  float* sw = reinterpret_cast<float*>(smem + L.sw_off);
  int32_t* aid = reinterpret_cast<int32_t*>(smem + L.aid_off);
  float* agate = reinterpret_cast<float*>(smem + L.agate_off);
  int32_t* rows = reinterpret_cast<int32_t*>(smem + L.rows_off);
  uint32_t* masks = reinterpret_cast<uint32_t*>(smem + L.masks_off);
  int* cnt = reinterpret_cast<int*>(smem + L.cnt_off);
  int* off = reinterpret_cast<int*>(smem + L.off_off);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L.bar_off);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kRcMaxStages + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* scratch = reinterpret_cast<int*>(tmem_slot + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = static_cast<int>(cluster_ctarank());
  const int nc = static_cast<int>(cluster_nctarank());
  const int S = p.stages;
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kRcMaxStages + s); };
  const uint32_t done_bar = bar0 + 8u * (2 * kRcMaxStages);
  // this CTA's tokens are t = c + nc*j, j < ntok
  const int ntok = c < p.T ? (p.T - 1 - c) / nc + 1 : 0;
  const bool dispatch = p.counts != nullptr;

  // this CTA's k-blocks of H
  const int kb0 = c * p.kb_total / nc, kb1 = (c + 1) * p.kb_total / nc;
  const int n = kb1 - kb0;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmX);
    tma_prefetch_desc(&p.tmW);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), static_cast<uint32_t>(p.tmem_cols));
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  grid_dep_wait();  // x may come from the previous kernel on the stream
  grid_dep_trigger();

  // the bias is read once per CTA, by the warps that have nothing to do in step 1
  if (warp >= 4)
    for (int e = tid - 128; e < p.E; e += kRcThreads - 128)
      bias_s[e] = p.bias != nullptr ? p.bias[e] : 0.f;

  // ---- 1. partial logits of this CTA's k-blocks on the tensor core --------------------
  const int w_bytes = p.nmt * 128 * 128;
  if (tid == 0 && n > 0) {
    const uint32_t idesc = idesc_bf16_f32(128, p.npad);
    auto issue = [&](int i, int s) {
      const uint32_t dst = smem_u32(smem + L.stages_off + s * L.stage_bytes);
      mbar_arrive_expect_tx(full_bar(s), static_cast<uint32_t>(L.stage_bytes));
      const int kc = (kb0 + i) * 64;
      for (int m = 0; m < p.nmt; ++m) tma_load_2d(dst + m * 16384, &p.tmW, full_bar(s), kc, m * 128);
      tma_load_2d(dst + w_bytes, &p.tmX, full_bar(s), kc, 0);
    };
    const int pre = n < S ? n : S;
    for (int i = 0; i < pre; ++i) issue(i, i);
    bool ok = true;
    int issued_to = pre;
    for (int i = 0; i < n && ok; ++i) {
      const int s = i % S;
      const uint32_t ph = static_cast<uint32_t>(i / S) & 1u;
      if (!mbar_wait(full_bar(s), ph, abort_flag, p.err)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t base = smem_u32(smem + L.stages_off + s * L.stage_bytes);
      for (int m = 0; m < p.nmt; ++m) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc_mma_bf16(tmem_base + static_cast<uint32_t>(m * p.npad),
                      smem_desc_sw128(base + m * 16384 + kk * 32),
                      smem_desc_sw128(base + w_bytes + kk * 32), idesc, (i | kk) != 0 ? 1u : 0u);
      }
      tc_commit(empty_bar(s));
      if (i + S < n) {
        if (!mbar_wait(empty_bar(s), ph, abort_flag, p.err)) {
          ok = false;
          break;
        }
        issue(i + S, s);
        issued_to = i + S + 1;
      }
    }
    tc_commit(done_bar);  // arrives when every MMA issued above is complete
    if (!ok) {
      // the loads issued into each stage must land before the CTA may exit
      volatile int no_abort = 0;
      for (int i = (issued_to > S ? issued_to - S : 0); i < issued_to; ++i)
        mbar_wait(full_bar(i % S), static_cast<uint32_t>(i / S) & 1u, &no_abort, p.err);
    }
  }
  __syncthreads();
  bool have = n > 0;
  if (have) {
    volatile int no_abort = 0;
    have = mbar_wait(done_bar, 0, &no_abort, p.err);
  }
  tc_fence_after();
  if (warp < 4) {
    // TMEM lane = expert (warp w owns lanes 32w..32w+31 of every 128-row tile), column = token
    for (int m = 0; m < p.nmt; ++m) {
      const int e = m * 128 + warp * 32 + lane;
      for (int t0 = 0; t0 < p.npad; t0 += 16) {
        uint32_t r[16];
        if (have) {
          tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(warp * 32) << 16) +
                                 static_cast<uint32_t>(m * p.npad + t0),
                             r);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 16; ++j) r[j] = 0u;
        }
        if (e < p.E) {
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (t0 + j < p.T) part[(t0 + j) * p.E + e] = __uint_as_float(r[j]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem_base, static_cast<uint32_t>(p.tmem_cols));

  // ---- 2. logits = partials of all CTAs in rank order + bias; warp top-k -------------
  // This CTA's tokens are t = c + nc*j, j < ntok.  Every thread adds up some of their
  // (token, expert) logits from the nc partials; then warp j takes token j's top-k.
  // Global stores wait until after the last cluster barrier (a release there would
  // otherwise wait for them to drain).
  cluster_sync_all();
  const uint32_t part_addr = smem_u32(part);
  for (int i = tid; i < ntok * p.E; i += kRcThreads) {
    const int j = i / p.E, e = i - j * p.E;
    const uint32_t a = part_addr + static_cast<uint32_t>(((c + nc * j) * p.E + e) * 4);
    float q[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) q[r] = r < nc ? ld_dsmem_f32(mapa_shared(a, r)) : 0.f;
    float v = 0.f;
#pragma unroll
    for (int r = 0; r < 16; ++r)
      if (r < nc) v += q[r];
    Ls[j * p.E + e] = v + bias_s[e];
  }
  __syncthreads();
  if (warp < ntok) {
    warp_topk_softmax(Ls + warp * p.E, p.E, p.K, p.theta, sid + warp * p.K, sw + warp * p.K);
    __syncwarp();
  }
  cluster_sync_all();  // every CTA's ids are in place (and no one reads `part` any more)

  // ---- 3. stable counting sort of the T*K assignments, redundantly in every CTA ------
  const int TK = p.T * p.K;
  if (dispatch) {
    const uint32_t sid_addr = smem_u32(sid), sw_addr = smem_u32(sw);
    for (int a = tid; a < TK; a += kRcThreads) {
      const int t = a / p.K, k = a - t * p.K;
      const uint32_t o = static_cast<uint32_t>(((t / nc) * p.K + k) * 4);
      aid[a] = ld_dsmem_s32(mapa_shared(sid_addr + o, static_cast<uint32_t>(t % nc)));
      if (p.row_w != nullptr)
        agate[a] = ld_dsmem_f32(mapa_shared(sw_addr + o, static_cast<uint32_t>(t % nc)));
    }
    for (int i = tid; i < 2 * p.E; i += kRcThreads) masks[i] = 0u;
  }
  cluster_sync_all();  // last remote access: after this a CTA may exit on its own

  // this CTA's routing results
  for (int i = tid; i < ntok * p.E; i += kRcThreads) {
    const int j = i / p.E, e = i - j * p.E;
    p.logits[static_cast<size_t>(c + nc * j) * p.E + e] = Ls[i];
  }
  for (int i = tid; i < ntok * p.K; i += kRcThreads) {
    const int j = i / p.K, k = i - j * p.K;
    p.ids[static_cast<size_t>(c + nc * j) * p.K + k] = sid[i];
    p.w[static_cast<size_t>(c + nc * j) * p.K + k] = sw[i];
  }
  if (!dispatch) return;

  rc_sort_and_dispatch(p, c, nc, aid, agate, masks, cnt, off, rows, scratch);
}

// Sums a[t] over the warp for NT (a power of two up to 32) values at once: at each of the
// first log2(NT) butterfly steps a lane keeps half of its values and adds its partner's
// copy of them, so the shuffles halve with the values (NT - 1 + 5 - log2(NT) in all).
// Returns the full sum of value t_out, which the lane's bits 4, 3, ... select; the 32 / NT
// lanes of a block of consecutive lanes share t_out and the same sum.
template <int NT>
__device__ __forceinline__ float warp_sum_scatter(float (&a)[NT], int lane, int& t_out) {
  int t = 0;
#pragma unroll
  for (int n = NT, o = 16; n > 1; n >>= 1, o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float keep = upper ? a[i + n / 2] : a[i];
      const float send = upper ? a[i] : a[i + n / 2];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
    if (upper) t += n / 2;
  }
  float v = a[0];
#pragma unroll
  for (int o = 16 / NT; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  t_out = t;
  return v;
}

// NT: the token count rounded up to a power of two (the tokens from T on are zero rows).
template <int NT>
__global__ void __launch_bounds__(kRcThreads, 1)
    route_dispatch_dot_kernel(const __grid_constant__ RcParams p) {
  extern __shared__ __align__(16) uint8_t smem_rd[];
  const RdLayout L = rd_layout(NT, p.H, p.E, p.K);
  uint4* xs = reinterpret_cast<uint4*>(smem_rd + L.x_off);
  float* Ls = reinterpret_cast<float*>(smem_rd + L.ls_off);
  int32_t* sid = reinterpret_cast<int32_t*>(smem_rd + L.sid_off);
  float* sw = reinterpret_cast<float*>(smem_rd + L.sw_off);
  int32_t* rows = reinterpret_cast<int32_t*>(smem_rd + L.rows_off);
  uint32_t* masks = reinterpret_cast<uint32_t*>(smem_rd + L.masks_off);
  int* cnt = reinterpret_cast<int*>(smem_rd + L.cnt_off);
  int* off = reinterpret_cast<int*>(smem_rd + L.off_off);
  int* scratch = reinterpret_cast<int*>(smem_rd + L.scratch_off);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = static_cast<int>(cluster_ctarank());
  const int nc = static_cast<int>(cluster_nctarank());
  const int e0 = c * p.E / nc, e1 = (c + 1) * p.E / nc;
  const int units = p.H / 8;  // 16-byte units per row
  for (int i = tid; i < 2 * p.E; i += kRcThreads) masks[i] = 0u;
  cluster_arrive_relaxed();  // waited on after the tokens are staged

  grid_dep_wait();  // x may come from the previous kernel on the stream
  grid_dep_trigger();

  // Warp w takes experts e0 + w, e0 + w + 8, ...: the first chunk of its first router row
  // is in flight while the tokens are staged.  (An L2 bulk prefetch of the rows before
  // griddepcontrol.wait measured no faster.)
  uint4 wv[kRdChunk];
  auto load_chunk = [&](int e, int u0) {
    const uint4* row = p.wr + static_cast<size_t>(e) * units;
#pragma unroll
    for (int j = 0; j < kRdChunk; ++j) {
      const int u = u0 + 32 * j + lane;
      wv[j] = u < units ? __ldg(row + u) : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  if (e0 + warp < e1) load_chunk(e0 + warp, 0);

  // ---- 1. the tokens into shared memory (all of a thread's loads in flight at once) ----
  {
    const int n = p.T * units;
#pragma unroll 8
    for (int i = tid; i < n; i += kRcThreads) xs[i] = __ldg(p.x + i);
    for (int i = n + tid; i < NT * units; i += kRcThreads) xs[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();
  cluster_wait();  // every CTA of the cluster is running: its shared memory may be written

  // ---- 2. logits of this CTA's experts: warp per expert, lanes over H ------------------
  // Each lane adds its units in order and the warp sums the lanes by a fixed butterfly, so
  // a logit is the same on every run; the lanes holding it store it into every CTA's table.
  const uint32_t ls_addr = smem_u32(Ls);
  for (int e = e0 + warp; e < e1; e += kRcWarps) {
    const float be = p.bias != nullptr ? __ldg(p.bias + e) : 0.f;
    float acc[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) acc[t] = 0.f;
    for (int u0 = 0; u0 < units; u0 += 32 * kRdChunk) {
      if (u0 != 0 || e != e0 + warp) load_chunk(e, u0);
#pragma unroll
      for (int j = 0; j < kRdChunk; ++j) {
        const int u = u0 + 32 * j + lane;
        if (u < units) {
          const float2 w0 = bf2_to_f2(wv[j].x), w1 = bf2_to_f2(wv[j].y);
          const float2 w2 = bf2_to_f2(wv[j].z), w3 = bf2_to_f2(wv[j].w);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const uint4 xv = xs[t * units + u];
            const float2 x0 = bf2_to_f2(xv.x), x1 = bf2_to_f2(xv.y);
            const float2 x2 = bf2_to_f2(xv.z), x3 = bf2_to_f2(xv.w);
            float a = acc[t];
            a = fmaf(w0.x, x0.x, a);
            a = fmaf(w0.y, x0.y, a);
            a = fmaf(w1.x, x1.x, a);
            a = fmaf(w1.y, x1.y, a);
            a = fmaf(w2.x, x2.x, a);
            a = fmaf(w2.y, x2.y, a);
            a = fmaf(w3.x, x3.x, a);
            a = fmaf(w3.y, x3.y, a);
            acc[t] = a;
          }
        }
      }
    }
    int t = 0;
    const float v = warp_sum_scatter<NT>(acc, lane, t) + be;
    if (t < p.T) {
      constexpr int kGroup = 32 / NT;  // lanes holding token t
      const uint32_t a = ls_addr + static_cast<uint32_t>((t * p.E + e) * 4);
      for (int r = lane & (kGroup - 1); r < nc; r += kGroup)
        st_shared_cluster(mapa_shared(a, static_cast<uint32_t>(r)), __float_as_int(v));
    }
  }
  cluster_sync_all();  // every CTA holds all logits; the last remote access

  // ---- 3. top-k of every token, in every CTA ---------------------------------------------
  if (warp < p.T) {
    warp_topk_softmax(Ls + warp * p.E, p.E, p.K, p.theta, sid + warp * p.K, sw + warp * p.K);
    __syncwarp();
  }
  __syncthreads();
  // CTA c stores the routing results of tokens c, c + nc, ...
  for (int t = c; t < p.T; t += nc) {
    for (int e = tid; e < p.E; e += kRcThreads)
      p.logits[static_cast<size_t>(t) * p.E + e] = Ls[t * p.E + e];
    if (tid < p.K) {
      p.ids[static_cast<size_t>(t) * p.K + tid] = sid[t * p.K + tid];
      p.w[static_cast<size_t>(t) * p.K + tid] = sw[t * p.K + tid];
    }
  }
  if (p.counts == nullptr) return;
  rc_sort_and_dispatch(p, c, nc, sid, sw, masks, cnt, off, rows, scratch);
}

struct RcDevice {
  bool ready = false;
  bool dot_ready = false;
  int nc = 0;  // cluster size that fits (16 or 8), 0 if none
};

RcDevice g_rc[64];

int rc_stages(int npad, int nmt, int E, int K, int T, int kb_total, int nc) {
  const int per_cta = (kb_total + nc - 1) / nc;
  int s = per_cta < kRcMaxStages ? per_cta : kRcMaxStages;
  if (s < 1) s = 1;
  while (s > 1 && rc_layout(npad, nmt, E, K, T, s).total > kRcSmemBudget) --s;
  return s;
}

}  // namespace

bool route_cluster_ok(int dtype, int T, int H, int E, int K) {
  if (dtype != kBF16 || T < 1 || T > kRcMaxT || E < 1 || E > kRcMaxE || K > kRcMaxK) return false;
  const int npad = (T + 15) / 16 * 16, nmt = (E + 127) / 128;
  return rc_layout(npad, nmt, E, K, T, 1).total <= kRcSmemBudget && H % 64 == 0;
}

cudaError_t launch_route_cluster(const void* x, const void* w_router, const float* bias,
                                 float* logits, int32_t* ids, float* w, float theta, int T, int H,
                                 int E, int K, int32_t* counts, int32_t* offsets, int32_t* perm,
                                 int32_t* inv, float* row_w, void* x_perm, unsigned* err,
                                 cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  RcDevice& d = g_rc[dev];
  const int npad = (T + 15) / 16 * 16, nmt = (E + 127) / 128;
  const int kb_total = H / 64;
  if (!d.ready) {
    e = cudaFuncSetAttribute(route_dispatch_cluster_kernel,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kRcSmemBudget);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(route_dispatch_cluster_kernel,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    d.nc = 0;
    for (int nc : {16, 8}) {
      cudaLaunchConfig_t lc;
      std::memset(&lc, 0, sizeof(lc));
      lc.gridDim = dim3(nc);
      lc.blockDim = dim3(kRcThreads);
      lc.dynamicSmemBytes = kRcSmemBudget;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = nc;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      lc.attrs = at;
      lc.numAttrs = 1;
      int nclusters = 0;
      if (cudaOccupancyMaxActiveClusters(&nclusters, route_dispatch_cluster_kernel, &lc) ==
              cudaSuccess &&
          nclusters >= 1) {
        d.nc = nc;
        break;
      }
      cudaGetLastError();  // clear a refused query before trying the smaller cluster
    }
    d.ready = true;
  }
  if (d.nc == 0) return cudaErrorNotSupported;
  // up to kRdMaxT tokens, when the tokens fit in shared memory: the expert-split kernel
  int nt = 1;
  while (nt < T) nt <<= 1;
  const bool dot = T <= kRdMaxT && rd_layout(nt, H, E, K).total <= kRcSmemBudget;
  if (dot && !d.dot_ready) {
    for (const void* f : {reinterpret_cast<const void*>(route_dispatch_dot_kernel<1>),
                          reinterpret_cast<const void*>(route_dispatch_dot_kernel<2>),
                          reinterpret_cast<const void*>(route_dispatch_dot_kernel<4>)}) {
      e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, kRcSmemBudget);
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    d.dot_ready = true;
  }
  RcParams p;
  std::memset(&p, 0, sizeof(p));
  if (dot) {
    // the rows are read in 16-byte units
    if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w_router)) & 15u) != 0u)
      return cudaErrorInvalidValue;
  } else if (!make_tma_2d_bf16(&p.tmX, x, static_cast<uint64_t>(T), static_cast<uint64_t>(H),
                               static_cast<uint32_t>(npad)) ||
             !make_tma_2d_bf16(&p.tmW, w_router, static_cast<uint64_t>(E),
                               static_cast<uint64_t>(H), 128)) {
    return cudaErrorInvalidValue;
  }
  p.bias = bias;
  p.logits = logits;
  p.ids = ids;
  p.w = w;
  p.counts = counts;
  p.offsets = offsets;
  p.perm = perm;
  p.inv = inv;
  p.row_w = row_w;
  p.x = static_cast<const uint4*>(x);
  p.wr = static_cast<const uint4*>(w_router);
  p.x_perm = static_cast<uint4*>(x_perm);
  p.err = err;
  p.T = T;
  p.H = H;
  p.E = E;
  p.K = K;
  p.npad = npad;
  p.nmt = nmt;
  p.kb_total = kb_total;
  p.stages = rc_stages(npad, nmt, E, K, T, kb_total, d.nc);
  int cols = 32;
  while (cols < nmt * npad) cols <<= 1;
  p.tmem_cols = cols;
  p.theta = theta;
  const int smem = dot ? rd_layout(nt, H, E, K).total : rc_layout(npad, nmt, E, K, T, p.stages).total;

  cudaLaunchConfig_t lc;
  std::memset(&lc, 0, sizeof(lc));
  lc.gridDim = dim3(d.nc);
  lc.blockDim = dim3(kRcThreads);
  lc.dynamicSmemBytes = static_cast<size_t>(smem);
  lc.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = d.nc;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 2;
  if (!dot) return count_launch(cudaLaunchKernelEx(&lc, route_dispatch_cluster_kernel, p));
  switch (nt) {
    case 1: return count_launch(cudaLaunchKernelEx(&lc, route_dispatch_dot_kernel<1>, p));
    case 2: return count_launch(cudaLaunchKernelEx(&lc, route_dispatch_dot_kernel<2>, p));
    default: return count_launch(cudaLaunchKernelEx(&lc, route_dispatch_dot_kernel<4>, p));
  }
}

}  // namespace moe
