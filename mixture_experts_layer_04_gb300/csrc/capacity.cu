// Capacity-limited routing.
//
// "MoE大模型的智能调度：从1.8万亿参数到每token仅激活2%的工程真相" §3.2, trap 2: a capacity
// check goes into routing, capacity = (batch_size * seq_len * k) / num_experts * 1.2, and an
// expert chosen that many times gets logit -inf so that the token chooses again.  Tokens are
// routed in token order: an expert is available to token t while fewer than `cap` kept
// assignments of earlier tokens (after their gate drop) went to it, and t takes its top-k of
// the available experts (softmax over them, then the gate drop; missing slots -1).
//
// The rule is sequential in t, but each token depends on earlier tokens only through, per
// expert, the index of the token that takes its last free place.  The batch is swept in blocks
// of 256 tokens with the exact counts of the earlier blocks.  Inside a block the routing
// iterates to a fixed point: fb[e] = the block token holding e's (cap - count[e])-th kept
// assignment under the current choices, and every token whose availability changed chooses
// again among the experts with count[e] < cap and fb[e] >= its index.  Token 0 of the block is
// final after the first pass and each pass fixes at least the next token, so the fixed point
// (the sequential routing) is reached within 257 passes; in practice in a few.  Tokens that no
// capacity touches keep the router's choice.
//
// One thread-block cluster runs the sweep (16 CTAs where the device allows it, else fewer).
// CTA c owns block tokens [c * 256 / nc, (c + 1) * 256 / nc), one token per warp at nc = 16,
// with their logit rows staged in shared memory.  Each pass, every CTA re-chooses its dirty
// tokens and sets the bits of its tokens in its slice of the per-expert block masks (16 bits
// per expert at nc = 16, u16 [E] contiguous), then stores the slice, in 16-byte stores, into
// every CTA of the cluster; one cluster barrier later every CTA holds the whole block's masks
// and derives the same fb[], the same change list and the same decision to stop.  The block
// masks are double-buffered by pass parity, so one cluster barrier per pass suffices: a CTA
// can only overwrite a buffer after every CTA has passed the next barrier, i.e. has finished
// reading it.  No global scratch, no atomics on global memory: the result is deterministic.
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int kCapThreads = 512;
constexpr int kCapWarps = kCapThreads / 32;
constexpr int kCapBlock = 256;              // tokens per block of the sweep
constexpr int kCapWords = kCapBlock / 32;   // token bits per expert
constexpr int kNone = kCapBlock;            // fb value: the expert does not fill in the block
constexpr int kCapMaxE = 1024;
constexpr int kCapMaxK = 16;
constexpr int kCapStageMax = 96 * 1024;     // largest logit stage kept in shared memory

// Shared-memory layout of one CTA (byte offsets, 16-byte aligned); tpc = tokens per CTA.
struct CapLayout {
  int lg, cnt, fb, mask, own, chg, bid, bw, dirty, total;
  int src_bytes;  // one CTA's slice of every expert's block mask: u16 [E][tpc / 16], padded
};

__host__ __device__ inline int cap_align16(int b) { return (b + 15) / 16 * 16; }

__host__ __device__ inline bool cap_stages_logits(int E, int tpc) {
  return tpc * E * 4 <= kCapStageMax;
}

__host__ __device__ inline CapLayout cap_layout(int E, int K, int tpc) {
  CapLayout L;
  L.src_bytes = cap_align16(E * (tpc / 16) * 2);
  int o = 0;
  L.lg = o;
  o += cap_stages_logits(E, tpc) ? cap_align16(tpc * E * 4) : 0;  // float [tpc][E]
  L.cnt = o;
  o += cap_align16(E * 4);                                         // int [E]
  L.fb = o;
  o += cap_align16(E * 4);                                         // int [E]
  L.mask = o;
  o += 2 * (kCapBlock / tpc) * L.src_bytes;                        // [2][nc] slices
  L.own = o;
  o += L.src_bytes;                                                // this CTA's slice
  L.chg = o;
  o += cap_align16(3 * E * 4);                                     // int [E][3]
  L.bid = o;
  o += cap_align16(tpc * K * 4);                                   // int [tpc][K]
  L.bw = o;
  o += cap_align16(tpc * K * 4);                                   // float [tpc][K]
  L.dirty = o;
  o += cap_align16(tpc * 4);                                       // int [tpc]
  L.total = o;
  return L;
}

__device__ __forceinline__ uint32_t cap_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// 16-byte store into the shared memory of a CTA of the cluster (a shared::cluster address).
__device__ __forceinline__ void st_dsmem_v4(uint32_t cluster_addr, uint4 v) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(cluster_addr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Position of the n-th (0-based) set bit of v (n < popc(v)).
__device__ __forceinline__ int nth_set_bit(uint32_t v, int n) {
  for (int i = 0; i < n; ++i) v &= v - 1u;
  return __ffs(v) - 1;
}

// Inverse of float_key (the key of -0 gives +0, which the softmax cannot tell apart).
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Word wd (block tokens [32 wd, 32 wd + 32)) of expert e's block mask, from the slices of one
// pass: slice r holds u16 [E][upc], unit j of expert e covering block tokens
// [16 (r upc + j), +16); upc = 1 << ulog.
__device__ __forceinline__ uint32_t block_word(const unsigned char* mk, int src_bytes, int ulog,
                                               int e, int wd) {
  const int u0 = 2 * wd, u1 = u0 + 1, um = (1 << ulog) - 1;
  const uint16_t* s0 = reinterpret_cast<const uint16_t*>(mk + (u0 >> ulog) * src_bytes);
  const uint16_t* s1 = reinterpret_cast<const uint16_t*>(mk + (u1 >> ulog) * src_bytes);
  return static_cast<uint32_t>(s0[(e << ulog) + (u0 & um)]) |
         (static_cast<uint32_t>(s1[(e << ulog) + (u1 & um)]) << 16);
}

template <int NJ>  // candidates per lane: experts lane + 32 j, j < NJ (E <= 32 NJ)
__device__ __forceinline__ void masked_topk_t(const float* __restrict__ L, int E, int K,
                                              float theta, int tl, const int* cnt, const int* fb, int cap,
                                              int32_t* ids, float* w) {
  const int lane = threadIdx.x & 31;
  uint32_t key[NJ];
  uint32_t live = 0u;  // bit j: expert lane + 32 j is available
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const int e = lane + 32 * j;
    key[j] = 0u;
    if (e < E && cnt[e] < cap && fb[e] >= tl) {
      key[j] = float_key(L[e]);
      live |= 1u << j;
    }
  }
  float my_v = 0.f, v0 = 0.f;
  int my_e = -1, nsel = 0;
  for (int k = 0; k < K; ++k) {
    uint32_t kbest = 0u, ebest = 0xffffffffu;
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      if (((live >> j) & 1u) && (key[j] > kbest || ebest == 0xffffffffu)) {
        kbest = key[j];
        ebest = static_cast<uint32_t>(lane + 32 * j);
      }
    }
    const bool has = ebest != 0xffffffffu;
    if (!__any_sync(0xffffffffu, has)) break;
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, has ? kbest : 0u);
    const int e_win = static_cast<int>(
        __reduce_min_sync(0xffffffffu, (has && kbest == kmax) ? ebest : 0xffffffffu));
    if ((e_win & 31) == lane) live &= ~(1u << (e_win >> 5));
    const float v_win = key_float(kmax);
    if (k == 0) v0 = v_win;
    if (lane == k) {
      my_v = v_win;
      my_e = e_win;
    }
    ++nsel;
  }
  float z = (lane < nsel) ? expf(my_v - v0) : 0.f;
  float g = nsel > 0 ? z / warp_sum(z) : 0.f;
  if (theta > 0.f && nsel > 0) {
    if (lane >= 1 && lane < nsel && g < theta) {
      g = 0.f;
      my_e = -1;
    }
    g = g / warp_sum(g);
  }
  if (lane < K) {
    ids[lane] = lane < nsel ? my_e : -1;
    w[lane] = lane < nsel ? g : 0.f;
  }
}

// One warp: token `tl` of the block (logits row L) takes its top-k among the available experts
// (count < cap and fb >= tl), with the softmax and gate drop of the warp top-k (same sums in
// the same order), and writes its K slots to ids/w (dropped or missing slots -1 / 0).  The
// candidates' keys are loaded once and kept in registers.
__device__ __forceinline__ void masked_topk(const float* __restrict__ L, int E, int K, float theta,
                                            int tl, const int* cnt, const int* fb, int cap,
                                            int32_t* ids, float* w) {
  if (E <= 128)
    masked_topk_t<4>(L, E, K, theta, tl, cnt, fb, cap, ids, w);
  else if (E <= 256)
    masked_topk_t<8>(L, E, K, theta, tl, cnt, fb, cap, ids, w);
  else
    masked_topk_t<32>(L, E, K, theta, tl, cnt, fb, cap, ids, w);
}

__global__ void __launch_bounds__(kCapThreads, 1)
    capacity_route_kernel(const float* __restrict__ logits, int32_t* __restrict__ ids,
                          float* __restrict__ w, int T, int E, int K, float theta, int cap,
                          unsigned* err) {
  extern __shared__ __align__(16) unsigned char smem_c[];
  __shared__ int s_nchg;
  const int c = static_cast<int>(cluster_ctarank());
  const int nc = static_cast<int>(cap_nctarank());
  const int tpc = kCapBlock / nc;  // block tokens owned by this CTA (a multiple of 16)
  const int upc = tpc / 16;        // 16-token units of this CTA per expert
  const int ulog = 31 - __clz(upc);
  const bool stage = cap_stages_logits(E, tpc);
  const CapLayout lay = cap_layout(E, K, tpc);
  float* lg = reinterpret_cast<float*>(smem_c + lay.lg);
  int* cnt = reinterpret_cast<int*>(smem_c + lay.cnt);          // kept before the block
  int* fb = reinterpret_cast<int*>(smem_c + lay.fb);
  unsigned char* mask = smem_c + lay.mask;  // [2][nc] slices, written by every CTA
  uint32_t* own = reinterpret_cast<uint32_t*>(smem_c + lay.own);  // this CTA's slice
  const int sb = lay.src_bytes;
  int* chg = reinterpret_cast<int*>(smem_c + lay.chg);          // e, old fb, new fb
  int32_t* bid = reinterpret_cast<int32_t*>(smem_c + lay.bid);
  float* bw = reinterpret_cast<float*>(smem_c + lay.bw);
  int* s_dirty = reinterpret_cast<int*>(smem_c + lay.dirty);
  const uint32_t mask_sa = smem_u32(mask);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < E; e += kCapThreads) cnt[e] = 0;
  for (int i = tid; i < sb / 4; i += kCapThreads) own[i] = 0u;
  grid_dep_wait();  // the router's logits and choices
  grid_dep_trigger();
  cluster_sync_all();  // every CTA of the cluster is running before the first remote store
  int parity = 0;
  for (int t0 = 0; t0 < T; t0 += kCapBlock) {
    const int nb = min(kCapBlock, T - t0);
    const int b0 = c * tpc;                    // this CTA's first token in the block
    const int nt = max(0, min(tpc, nb - b0));  // this CTA's tokens in the block
    const size_t g0 = static_cast<size_t>(t0) + b0;
    for (int i = tid; i < nt * K; i += kCapThreads) {
      bid[i] = ids[g0 * K + i];
      bw[i] = w[g0 * K + i];
    }
    if (stage)
      for (int i = tid; i < nt * E; i += kCapThreads) lg[i] = logits[g0 * E + i];
    for (int e = tid; e < E; e += kCapThreads) fb[e] = kNone;
    __syncthreads();
    for (int pass = 0;; ++pass) {
      parity ^= 1;
      const unsigned char* mk = mask + parity * nc * sb;
      // 1. tokens whose available set may have changed choose again.  First pass: with a
      //    gate drop the router's dropped slots hide part of its choice, so every token
      //    chooses again; without one, only tokens that chose an expert already full.
      //    Then every token sets its bit in the masks of the experts it holds.
      for (int tl = warp; tl < nt; tl += kCapWarps) {
        bool dirty;
        if (pass == 0) {
          const int e = lane < K ? bid[tl * K + lane] : -1;
          dirty = theta > 0.f || __any_sync(0xffffffffu, e >= 0 && cnt[e] >= cap);
        } else {
          dirty = s_dirty[tl] != 0;
        }
        const float* Lt = stage ? lg + static_cast<size_t>(tl) * E : logits + (g0 + tl) * E;
        if (dirty) masked_topk(Lt, E, K, theta, b0 + tl, cnt, fb, cap, bid + tl * K, bw + tl * K);
        __syncwarp();
        const int e = lane < K ? bid[tl * K + lane] : -1;
        if (e >= 0) {
          const int u = e * upc + (tl >> 4);  // 16-bit unit of the slice
          atomicOr(&own[u >> 1], 1u << (16 * (u & 1) + (tl & 15)));
        }
      }
      if (tid == 0) s_nchg = 0;
      __syncthreads();
      // 2. this CTA's slice of every expert's block mask goes to every CTA of the cluster, in
      //    16-byte stores
      {
        const int chunks = sb / 16;
        const uint32_t dst = mask_sa + static_cast<uint32_t>((parity * nc + c) * sb);
        for (int i = tid; i < nc * chunks; i += kCapThreads) {
          const int r = i / chunks, ch = i - r * chunks;
          const uint4 v = reinterpret_cast<const uint4*>(own)[ch];
          st_dsmem_v4(mapa_shared(dst + 16u * ch, static_cast<uint32_t>(r)), v);
        }
      }
      cluster_sync_all();  // every CTA's slices are in place (and all reads of `own` done)
      for (int i = tid; i < sb / 4; i += kCapThreads) own[i] = 0u;
      // 3. fb[e]: the block token that takes e's last free place, if any (the same in every CTA)
      for (int e = tid; e < E; e += kCapThreads) {
        const int need = cap - cnt[e];
        int f = kNone;
        if (need > 0) {
          int run = 0;
          for (int wd = 0; wd < kCapWords; ++wd) {
            const uint32_t m = block_word(mk, sb, ulog, e, wd);
            const int pc = __popc(m);
            if (run + pc >= need) {
              f = wd * 32 + nth_set_bit(m, need - run - 1);
              break;
            }
            run += pc;
          }
        }
        if (f != fb[e]) {
          const int j = atomicAdd(&s_nchg, 1);
          chg[3 * j] = e;
          chg[3 * j + 1] = fb[e];
          chg[3 * j + 2] = f;
          fb[e] = f;
        }
      }
      __syncthreads();
      const int nchg = s_nchg;
      if (nchg == 0) break;
      // 4. which of this CTA's tokens must choose again: e's last free place moved from a to
      //    b.  Earlier (b < a): tokens in (b, a] lose e, which matters to those holding it.
      //    Later (b > a): tokens in (a, b] gain e, which matters if its logit ties or beats
      //    the token's weakest choice or the token has an empty slot (a dropped slot hides a
      //    choice, so it counts as empty).
      for (int tl = tid; tl < nt; tl += kCapThreads) {
        const float* Lt = stage ? lg + static_cast<size_t>(tl) * E : logits + (g0 + tl) * E;
        const int tb = b0 + tl;
        float weakest = 0.f;
        bool has_empty = false;
        for (int k = 0; k < K; ++k) {
          const int e = bid[tl * K + k];
          if (e < 0) {
            has_empty = true;
          } else {
            const float v = Lt[e];
            weakest = k == 0 ? v : fminf(weakest, v);
          }
        }
        int d = 0;
        for (int j = 0; j < nchg && !d; ++j) {
          const int e = chg[3 * j], a = chg[3 * j + 1], b = chg[3 * j + 2];
          if (b < a) {
            if (tb > b && tb <= a) {
              for (int k = 0; k < K; ++k) d |= bid[tl * K + k] == e;
            }
          } else if (tb > a && tb <= b) {
            d = has_empty || Lt[e] >= weakest;
          }
        }
        s_dirty[tl] = d;
      }
      __syncthreads();
      if (pass > nb + 1) {  // cannot happen: each pass fixes at least one more token
        if (tid == 0 && c == 0) report_error(err, MOE_DEVERR_BOUNDS);
        break;
      }
    }
    // 5. commit the block: its kept assignments count against the capacity
    const unsigned char* mk = mask + parity * nc * sb;
    for (int e = tid; e < E; e += kCapThreads) {
      int n = 0;
      for (int wd = 0; wd < kCapWords; ++wd) n += __popc(block_word(mk, sb, ulog, e, wd));
      cnt[e] += n;
    }
    for (int i = tid; i < nt * K; i += kCapThreads) {
      ids[g0 * K + i] = bid[i];
      w[g0 * K + i] = bw[i];
    }
    __syncthreads();
  }
}

}  // namespace

int capacity_limit(int T, int K, int E) {
  const long long c = (12LL * T * K + 10LL * E - 1) / (10LL * E);
  return static_cast<int>(c);
}

cudaError_t launch_capacity_route(const float* logits, int32_t* ids, float* w, int T, int E, int K,
                                  float theta, int cap, unsigned* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (E < 1 || E > kCapMaxE || K < 1 || K > kCapMaxK) return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  // the largest cluster (16, 8, 4, 2 or 1 CTAs) that the device can hold at the largest
  // layout (E = 1024, K = 16), found once per device
  static int cap_nc[64] = {0};
  if (cap_nc[dev] == 0) {
    int smem_max = 0;
    for (int nc = 1; nc <= 16; nc *= 2) {
      const int b = cap_layout(kCapMaxE, kCapMaxK, kCapBlock / nc).total;
      smem_max = b > smem_max ? b : smem_max;
    }
    e = cudaFuncSetAttribute(capacity_route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem_max);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(capacity_route_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed,
                             1);
    if (e != cudaSuccess) return e;
    int found = 1;
    for (int nc : {16, 8, 4, 2}) {
      cudaLaunchConfig_t lc;
      std::memset(&lc, 0, sizeof(lc));
      lc.gridDim = dim3(nc);
      lc.blockDim = dim3(kCapThreads);
      lc.dynamicSmemBytes = static_cast<size_t>(cap_layout(kCapMaxE, kCapMaxK, kCapBlock / nc).total);
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = nc;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      lc.attrs = at;
      lc.numAttrs = 1;
      int nclusters = 0;
      if (cudaOccupancyMaxActiveClusters(&nclusters, capacity_route_kernel, &lc) == cudaSuccess &&
          nclusters >= 1) {
        found = nc;
        break;
      }
      cudaGetLastError();  // clear a refused query before trying the smaller cluster
    }
    cap_nc[dev] = found;
  }
  const int nc = cap_nc[dev];
  cudaLaunchConfig_t lc;
  std::memset(&lc, 0, sizeof(lc));
  lc.gridDim = dim3(nc);
  lc.blockDim = dim3(kCapThreads);
  lc.dynamicSmemBytes = static_cast<size_t>(cap_layout(E, K, kCapBlock / nc).total);
  lc.stream = s;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = nc;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = at;
  lc.numAttrs = 2;
  return count_launch(cudaLaunchKernelEx(&lc, capacity_route_kernel, logits, ids, w, T, E, K, theta, cap, err));
}

}  // namespace moe
