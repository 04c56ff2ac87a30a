// Grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
// Page opening "MoE通过稀疏激活降低每个token的计算量…", section "单机MoE执行流水线": a
// grouped GEMM runs several experts' matrices, whose row counts differ, in one kernel
// launch; grouping changes the number of launches, not the matrices.  Section
// "一个批次如何变成各专家专属的矩阵": prefill gives experts many rows (matrix efficiency
// matters), decode gives them few (weight reads dominate).
//
// One persistent CTA per SM, 192 threads:
//   warp 0     TMA producer: for every tile and k-block (64 bf16 = one 128-byte swizzle
//              row), loads an activation tile (token rows) and a weight tile (expert
//              weight rows) into a STAGES-deep shared-memory ring, signalling an mbarrier.
//   warp 1     MMA issuer: one elected thread issues tcgen05.mma (M=128, K=16, bf16 x bf16
//              -> fp32) into one of two TMEM accumulators, frees each smem stage with
//              tcgen05.commit, and signals the epilogue when a tile is complete.
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (each warp owns 32 TMEM lanes),
//              SwiGLU or plain fp32 (+ column bias), row/column-masked global stores.
// The two accumulators let the epilogue of tile i overlap the main loop of tile i+1.
//
// Two operand orders:
//   normal  (prefill): A = 128 token rows, B = BN weight rows.  TMEM lane = token row,
//           column = output feature.  SwiGLU: the weight tile is BN/2 gate rows followed
//           by the BN/2 matching up rows, so a thread holds both halves of its outputs.
//   swapped (decode, few rows per expert): A = 128 weight rows, B = BN token rows (BN =
//           16..64), so the tensor core does no work on empty token rows and every CTA
//           streams distinct weight bytes.  TMEM lane = output feature, column = token.
//           SwiGLU: lanes 0-63 hold gate rows, 64-127 the matching up rows; the up half
//           goes through shared memory to the warps that own the gate half.
//
// Ragged groups: each CTA derives, from the group row offsets, how many token tiles
// every group has (a block-wide scan in shared memory) and maps a tile index to (group,
// first row, end row, weight tile) by binary search.  A tile's TMA load may read rows of
// the next group (or zero-filled rows past the end of A); those rows are computed but
// never stored.  Tiles are rasterised in groups of `swz` token tiles so that the CTAs
// resident at one time share weight tiles in L2.
//
// Launches use programmatic dependent launch: the prologue (barrier init, TMEM
// allocation, descriptor prefetch) overlaps the previous kernel, and griddepcontrol.wait
// precedes the first read of anything an earlier kernel wrote.
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {
namespace {

constexpr int BK = 64;  // bf16 elements = 128 bytes = one swizzle row
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kSwz = 8;  // token tiles per raster chunk
constexpr int kMaxGroups = 1024;

struct TcParams {
  CUtensorMap tmAct;  // [rows_alloc, Kd] activations (token rows)
  // CTA pairs only, for tail tiles in swapped order: the activations in boxes of 16, 32
  // and 64 rows, and (SwiGLU) the weights as [G][2][I][Kd] in boxes of 64 gate rows plus
  // the 64 matching up rows
  CUtensorMap tmActS16;
  CUtensorMap tmActS32;
  CUtensorMap tmActS64;
  CUtensorMap tmWgtS;
  CUtensorMap tmWgt;  // [G, Nb, Kd] weights
  void* C;
  const float* col_bias;
  const int32_t* offsets;  // [num_groups+1] row offsets of the groups, or null
  const int32_t* row_token;  // kScatter: destination row (token) of every A row
  const float* row_w;        // kScatter: scale of every A row (its route weight)
  unsigned* err;
  int num_groups;
  int rows_alloc;
  int num_kb;
  int N_out;
  int n_tiles;
  int up_offset;
  int swz;
  const int32_t* gather_rows;  // A row r is row gather_rows[r] of the mapped tensor, or null
  int topk_k;                  // kTopK: experts kept per row, gate threshold, outputs
  float topk_theta;
  int32_t* topk_ids;
  float* topk_w;
  // FP8 gate/up (E4M3 operands): per A row and per B row ([G][b_rows]) scales, applied to
  // the accumulators before the SwiGLU; null for bf16
  const float* a_scale;
  const float* b_scale;
  int b_rows;
  // grouped launches in the normal operand order: interleave the tiles of groups that
  // have a single token tile with the tiles of the larger groups (see build_schedule)
  int interleave;
  float* zero_ptr;  // cleared by the epilogue warps before the first tile (n floats), or null
  long long zero_n;
  int a_rows;  // rows of the tensor behind tmAct (the gather's source rows with a row gather)
  // CTA pairs: tiles are taken in index order from this counter (zero at launch) as pairs
  // become free (see ring_publish), or null for every npairs-th tile per pair
  int* tile_counter;
  int c_rows;  // kScatter: rows of C, 0 = unknown (both checked in the debug build only)
};

// Epilogue warps of a single-CTA launch: FP8 plain / scatter tiles in the normal order
// take eight (two per TMEM lane quarter, each draining every other 32-column chunk): their
// MMAs take half the time of bf16 ones, and with four warps the fp32 epilogue set the pace
// (a per-tile timeline at the Qwen3 shape: MMA 1.9 us, epilogue 3.8-4.9 us per tile; the
// FP8 layer went from 530 to 508 us with eight).
__host__ __device__ constexpr int tc_epi_warps(int MODE, bool SWAP, bool F8) {
  return (F8 && !SWAP && (MODE == kPlain || MODE == kScatter)) ? 8 : kEpiWarps;
}
__host__ __device__ constexpr int tc_threads(int MODE, bool SWAP, bool GATHER, bool F8) {
  return 64 + 32 * tc_epi_warps(MODE, SWAP, F8) + (GATHER ? 32 : 0);
}

template <int BN, int MODE, bool SWAP, int EPI = kEpiWarps>
struct TcCfg {
  static constexpr int kActRows = SWAP ? BN : 128;   // token rows per tile
  static constexpr int kWgtRows = SWAP ? 128 : BN;   // weight rows per tile
  static constexpr int kActBytes = kActRows * BK * 2;
  static constexpr int kWgtBytes = kWgtRows * BK * 2;
  static constexpr int kStageBytes = kActBytes + kWgtBytes;
  static constexpr int kWgtBox = MODE == kSwiGLU ? kWgtRows / 2 : kWgtRows;  // rows per TMA box
  static constexpr int kColsOut = MODE == kSwiGLU ? kWgtRows / 2 : kWgtRows; // outputs per tile
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
  static constexpr int kStgBytes =
      SWAP ? (MODE == kSwiGLU ? 64 * BN * 4 : 0) : EPI * 32 * (MODE == kSwiGLU ? 64 : 128);
  static constexpr int kBarBytes = 256;
  static constexpr int kSchedBytes = 3 * (kMaxGroups + 4) * 4 + 32 * 4;
  // as many stages as shared memory holds (up to 12): the bytes a CTA keeps in flight set
  // its load rate, which is what bounds the small-tile decode kernels
  static constexpr int kStagesRaw =
      (232448 - 1024 - kStgBytes - kBarBytes - kSchedBytes) / kStageBytes;
  static constexpr int kStages = kStagesRaw > 12 ? 12 : kStagesRaw;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kStgBytes + kBarBytes + kSchedBytes;
  static_assert((kTmemCols & (kTmemCols - 1)) == 0 && kTmemCols <= 512, "TMEM columns");
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M=128");
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

// The tile schedule of one launch, which every CTA derives from the group row offsets.
//   s_off[0..G]   the group row offsets;
//   s_mt[0..G]    exclusive prefix of the token tiles of the groups in the "heavy" order;
//   s_light[j]    with interleaving, the j-th group that has exactly one token tile.
// Groups with a single token tile (up to `tile_rows` rows) stream a whole expert's weights
// for a few rows of MMA work: their tiles are bound by DRAM, while the tiles of large
// groups reuse each weight tile from L2 across many token tiles and are bound by the
// tensor cores.  In group order the two kinds come in long runs of one kind (a run of
// small experts leaves the tensor cores idle while DRAM saturates, a large expert leaves
// DRAM idle), so with `p.interleave` the single-tile groups are taken out of the heavy
// order and their tiles are spread evenly through it: out of every N tiles of the launch,
// N_light/N are single-tile-group tiles.  CTAs that run at the same time then mix both
// kinds, and the weight streaming of the small experts overlaps the MMAs of the large.
struct Sched {
  int num_mt;     // token tiles in the heavy order
  int num_light;  // groups taken out of the heavy order (interleaved)
  int total;      // tiles of the launch: (num_mt + num_light) * n_tiles
};

__device__ __forceinline__ Sched build_schedule(const TcParams& p, int* s_off, int* s_mt,
                                                int* s_light, int* s_scan, int tile_rows) {
  Sched sc;
  sc.num_light = 0;
  if (p.offsets == nullptr) {
    sc.num_mt = (p.rows_alloc + tile_rows - 1) / tile_rows;
    sc.total = sc.num_mt * p.n_tiles;
    return sc;
  }
  const int G = p.num_groups;
  for (int i = threadIdx.x; i <= G; i += blockDim.x) s_off[i] = p.offsets[i];
  __syncthreads();
#ifdef MOE_DEBUG
  // the offsets must be non-decreasing within [0, rows_alloc]: otherwise the launch does
  // nothing (every CTA sees the same offsets and takes the same decision)
  bool bad = threadIdx.x == 0 && (s_off[0] < 0 || s_off[G] > p.rows_alloc);
  for (int q = threadIdx.x; q < G; q += blockDim.x) bad = bad || s_off[q] > s_off[q + 1];
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report_error(p.err, MOE_DEVERR_BOUNDS);
    sc.num_mt = 0;
    sc.total = 0;
    return sc;
  }
#endif
  const int per = (G + blockDim.x - 1) / blockDim.x;
  const int beg = min(G, static_cast<int>(threadIdx.x) * per), end = min(G, beg + per);
  auto tiles_of = [&](int q) { return (s_off[q + 1] - s_off[q] + tile_rows - 1) / tile_rows; };
  auto light = [&](int q) { return p.interleave != 0 && tiles_of(q) == 1; };
  int mine = 0, mine_light = 0;
  for (int q = beg; q < end; ++q) {
    if (light(q)) ++mine_light;
    else mine += tiles_of(q);
  }
  int all = 0, all_light = 0;
  int run = block_exclusive_scan(mine, s_scan, &all);
  int run_light = block_exclusive_scan(mine_light, s_scan, &all_light);
  for (int q = beg; q < end; ++q) {
    s_mt[q] = run;
    if (light(q)) s_light[run_light++] = q;
    else run += tiles_of(q);
  }
  if (threadIdx.x == 0) s_mt[G] = all;
  __syncthreads();
  sc.num_mt = all;
  sc.num_light = all_light;
  sc.total = (all + all_light) * p.n_tiles;
  return sc;
}

// Tile idx -> (group g, token rows row0..row_end-1, weight tile n_tile).
// Heavy order: groups one after another; inside a group, chunks of up to `swz` token tiles,
// and inside a chunk the weight tiles outer, token tiles inner.  CTAs running at the same
// time thus share a weight tile (read once from HBM) and keep a chunk's token rows in L2
// while they sweep the weight tiles, and no chunk mixes two groups' weights.  With
// interleaved single-tile groups, tile idx is one of theirs when floor(idx * NL / N) steps
// up at idx (NL of the N tiles are theirs, taken group by group, weight tiles inner);
// otherwise it is heavy tile idx - floor(idx * NL / N).
__device__ __forceinline__ void decode_tile(const TcParams& p, const int* s_off, const int* s_mt,
                                            const int* s_light, const Sched& sc, int tile_rows,
                                            int idx, int& g, int& row0, int& row_end,
                                            int& n_tile) {
  const int nt = p.n_tiles;
  int mt;  // token tile index inside its group
  if (p.offsets != nullptr) {
    if (sc.num_light > 0) {
      const long long NL = static_cast<long long>(sc.num_light) * nt;
      const long long N = sc.total;
      const long long cl = static_cast<long long>(idx) * NL / N;
      const long long cl1 = (static_cast<long long>(idx) + 1) * NL / N;
      if (cl1 > cl) {
        const int j = static_cast<int>(cl / nt);
        n_tile = static_cast<int>(cl - static_cast<long long>(j) * nt);
        g = s_light[j];
        row0 = s_off[g];
        row_end = s_off[g + 1];
        return;
      }
      idx -= static_cast<int>(cl);
    }
    const int mi = idx / nt;  // the group holding tile idx: s_mt[g] * nt <= idx
    int lo = 0, hi = p.num_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_mt[mid] <= mi) lo = mid; else hi = mid - 1;
    }
    g = lo;
    const int m_g = s_mt[g + 1] - s_mt[g];
    const int local = idx - s_mt[g] * nt;
    const int chunk = local / (p.swz * nt);
    const int rem = local - chunk * p.swz * nt;
    const int cm = min(p.swz, m_g - chunk * p.swz);
    n_tile = rem / cm;
    mt = chunk * p.swz + (rem - n_tile * cm);
    row0 = s_off[g] + mt * tile_rows;
    row_end = s_off[g + 1];
  } else {
    g = 0;
    const int chunk = idx / (p.swz * nt);
    const int rem = idx - chunk * p.swz * nt;
    const int cm = min(p.swz, sc.num_mt - chunk * p.swz);
    n_tile = rem / cm;
    mt = chunk * p.swz + (rem - n_tile * cm);
    row0 = mt * tile_rows;
    row_end = p.rows_alloc;
  }
}

// True when tile (g, row0..row_end) is its group's only token tile: each of the group's
// weight tiles is then read by this one tile and never again in the launch.
__device__ __forceinline__ bool read_once(const TcParams& p, const int* s_off, int g, int row0,
                                          int row_end, int tile_rows) {
  const int first = p.offsets != nullptr ? s_off[g] : 0;
  return row0 == first && row_end - row0 <= tile_rows;
}

// ------------------------------------------------------- dynamic tile order ----
// With p.tile_counter, CTA pairs take tiles in index order as they become free instead of
// every npairs-th tile each: the even CTA's producer thread draws tile indices from the
// counter and hands them to the pair's other roles (its own MMA thread and epilogue warps,
// the odd CTA's producer and epilogue warps) through a ring of kTileRing slots in shared
// memory.  Tiles that share a weight tile then start close together in time whichever
// pairs run them, and no pair is left running a whole tile after the others have finished.
// The drawing thread keeps two tiles ahead: it draws the index of tile j + 2 when it starts
// loading tile j and publishes it once tile j's loads are issued, so the atomic's latency
// and the odd CTA's wait are off the load path.  Every pair's last two draws are past the
// end, so the counter ends at total + 2 x pairs.
constexpr int kTileRing = 6;

struct TileRing {
  uint32_t full0;   // kTileRing barriers (count 1): the slot holds the next index
  uint32_t empty0;  // kTileRing barriers of the even CTA: every consumer has read the slot
  uint32_t slot0;   // kTileRing ints
};

// Publishes tile index v (-1: stop) as tile number j of this pair, in both CTAs.  The slot
// is written even when the wait for it fails, so that the consumers stop; returns false then.
__device__ __forceinline__ bool ring_publish(const TileRing& r, int j, int v,
                                             volatile int* abort, unsigned* err) {
  const int s = j % kTileRing;
  const uint32_t ph = static_cast<uint32_t>(j / kTileRing) & 1u;
  const bool ok = mbar_wait<true>(r.empty0 + 8u * s, ph ^ 1u, abort, err);
  if (!ok) v = -1;
  const uint32_t slot = r.slot0 + 4u * s;
  asm volatile("st.shared.u32 [%0], %1;" ::"r"(slot), "r"(v) : "memory");
  mbar_arrive(r.full0 + 8u * s);
  st_shared_cluster(mapa_shared(slot, 1), v);
  mbar_arrive_cluster(mapa_shared(r.full0 + 8u * s, 1));
  return ok;
}
__device__ __forceinline__ int ring_index(int ticket, int total) {
  return ticket < total ? ticket : -1;
}

// A consumer thread: tile number j (-1: stop), after which it releases the slot.  kRemote:
// the thread is in the odd CTA, whose slot the even CTA wrote.
template <bool kRemote>
__device__ __forceinline__ int ring_take(const TileRing& r, int j, volatile int* abort,
                                         unsigned* err) {
  const int s = j % kTileRing;
  const uint32_t ph = static_cast<uint32_t>(j / kTileRing) & 1u;
  int v = -1;
  if (mbar_wait<kRemote>(r.full0 + 8u * s, ph, abort, err))
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(r.slot0 + 4u * s) : "memory");
  if constexpr (kRemote)
    mbar_arrive_cluster(mapa_shared(r.empty0 + 8u * s, 0));
  else
    mbar_arrive(r.empty0 + 8u * s);
  return v;
}

// This CTA's share of the array to clear (see TcParams::zero_ptr), by the `nthreads`
// epilogue threads before they wait for the first accumulator; the writes need no ordering
// with the rest of this launch, only with later launches.
__device__ __forceinline__ void clear_share(const TcParams& p, int part, int parts, int t,
                                            int nthreads) {
  if (p.zero_ptr == nullptr) return;
  const long long n4 = p.zero_n / 4;
  const long long per = (n4 + parts - 1) / parts;
  const long long beg = per * part;
  const long long end = beg + per < n4 ? beg + per : n4;
  float4* q = reinterpret_cast<float4*>(p.zero_ptr);
  for (long long i = beg + t; i < end; i += nthreads) q[i] = make_float4(0.f, 0.f, 0.f, 0.f);
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

// Fire-and-forget fp32 additions into global memory (performed at L2).
__device__ __forceinline__ void red_add_v4(float* p, const uint4& v) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(__uint_as_float(v.x)),
               "f"(__uint_as_float(v.y)), "f"(__uint_as_float(v.z)), "f"(__uint_as_float(v.w))
               : "memory");
}
__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}

// Barrier among the four epilogue warps only (named barrier 1, 128 threads).
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// Barrier of the four epilogue warps that also returns, to every one of them, whether
// any thread passed `pred` true: a decision to leave the tile loop taken by all or none
// (a plain barrier followed by separate reads of the abort flag could split the warps
// if the flag is set in between, and the next barrier would then never fill).
__device__ __forceinline__ bool epi_bar_any(bool pred) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, 128, q;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(out)
      : "r"(pred ? 1u : 0u)
      : "memory");
  return out != 0u;
}

// Reads NC (16 or 32) consecutive columns of this warp's 32 TMEM lanes into v[0..NC).
template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&v)[32]) {
  if constexpr (NC == 16) {
    uint32_t r[16];
    tmem_ld_32x32b_x16(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
  } else {
    uint32_t r[32];
    tmem_ld_32x32b_x32(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
  }
}

// Epilogue of one accumulator tile in the normal operand order.  This warp owns the 32
// TMEM lanes at t_row (token rows tile_row0 .. tile_row0+31 of A, stored when < row_end);
// accumulator column j is output feature col0 + j (SwiGLU: columns BN/2 + j hold the up
// half).  `stg` is this warp's staging buffer in shared memory.
template <int BN, int MODE>
__device__ __forceinline__ void epilogue_rows(const TcParams& p, uint32_t t_row, uint32_t stg,
                                              int lane, int tile_row0, int row_end, int col0,
                                              int group = 0, int c_first = 0, int c_step = 32) {
  if constexpr (MODE == kSwiGLU) {
    __nv_bfloat16* C = static_cast<__nv_bfloat16*>(p.C);
    // FP8 operands: this thread's token-row scale, and the group's weight-row scales
    float sa = 1.f;
    const float* sb = nullptr;
    // the weight-row scales of every chunk, loaded at once (one coalesced load per chunk,
    // broadcast by shuffles below) so their latency is paid once, not once per chunk
    constexpr int kChunks = BN / 64;
    float sgv[kChunks], suv[kChunks];
    if (p.a_scale != nullptr) {
      sa = tile_row0 + lane < row_end ? __ldg(p.a_scale + tile_row0 + lane) : 0.f;
      sb = p.b_scale + static_cast<size_t>(group) * p.b_rows;
#pragma unroll
      for (int k = 0; k < kChunks; ++k) {
        const int cl = col0 + 32 * k + lane;
        sgv[k] = cl < p.N_out ? __ldg(sb + cl) : 0.f;
        suv[k] = cl < p.N_out ? __ldg(sb + p.up_offset + cl) : 0.f;
      }
    }
#pragma unroll 1
    for (int c = 0; c < BN / 2; c += 32) {
      uint32_t gr[32], ur[32];
      tmem_ld_32x32b_x32(t_row + c, gr);
      tmem_ld_32x32b_x32(t_row + BN / 2 + c, ur);
      tmem_ld_wait();
      if (sb != nullptr) {
        float sg = 0.f, su = 0.f;
#pragma unroll
        for (int k = 0; k < kChunks; ++k)
          if (32 * k == c) {
            sg = sgv[k];
            su = suv[k];
          }
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          gr[j] = __float_as_uint(__uint_as_float(gr[j]) * (sa * __shfl_sync(0xffffffffu, sg, j)));
          ur[j] = __float_as_uint(__uint_as_float(ur[j]) * (sa * __shfl_sync(0xffffffffu, su, j)));
        }
      }
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float h0 = silu_bf16out(__uint_as_float(gr[2 * j])) * __uint_as_float(ur[2 * j]);
        const float h1 =
            silu_bf16out(__uint_as_float(gr[2 * j + 1])) * __uint_as_float(ur[2 * j + 1]);
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
    // The scaling is applied after the transpose through shared memory, where each lane
    // holds 4 consecutive columns of one row per pass: row r = 4 pass + lane / 8 of the
    // warp's 32, columns 4 (lane % 8) .. + 3 of the chunk.  A lane then needs one factor per
    // pass (loaded once per tile) and four column factors per chunk, and no shuffles.
    //   kScatter: the row is scaled by its route weight and added into the output row of
    //             its token (the fused combine);
    //   FP8:      the row's token-row scale and the columns' weight-row scales;
    //   bias:     added per column after the scaling.
    const bool f8 = p.a_scale != nullptr;
    const bool row_scaled = MODE == kScatter || f8;
    const float* sb = f8 ? p.b_scale + static_cast<size_t>(group) * p.b_rows : nullptr;
    float rsc[8];
    int tok[8];
#pragma unroll
    for (int pass = 0; pass < 8; ++pass) {
      const int gr = tile_row0 + pass * 4 + (lane >> 3);
      const bool live = gr < row_end;
      float f = 1.f;
      tok[pass] = 0;
      if constexpr (MODE == kScatter) {
        f = live ? __ldg(p.row_w + gr) : 0.f;
        tok[pass] = live ? __ldg(p.row_token + gr) : 0;
      }
      if (f8) f *= live ? __ldg(p.a_scale + gr) : 0.f;
      rsc[pass] = f;
    }
    const int u = lane & 7;
    // FP8: this lane's four columns' weight-row scales for every chunk, loaded once per
    // tile (their latency is then paid once, not once per chunk)
    constexpr int kChunks = BN / 32;
    float csv[kChunks][4];
    if (f8) {
#pragma unroll
      for (int k = 0; k < kChunks; ++k)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int cl = col0 + 32 * k + u * 4 + q;
          csv[k][q] = cl < p.N_out ? __ldg(sb + cl) : 0.f;
        }
    }
#pragma unroll 1
    for (int c = c_first; c < BN; c += c_step) {
      uint32_t r[32];
      tmem_ld_32x32b_x32(t_row + c, r);
      // this lane's four columns' weight-row scales and biases for the chunk
      const int col = col0 + c + u * 4;
      float cs[4] = {1.f, 1.f, 1.f, 1.f}, bs[4] = {0.f, 0.f, 0.f, 0.f};
      if (f8) {
#pragma unroll
        for (int k = 0; k < kChunks; ++k)
          if (32 * k == c) {
#pragma unroll
            for (int q = 0; q < 4; ++q) cs[q] = csv[k][q];
          }
      }
      if (p.col_bias != nullptr) {
#pragma unroll
        for (int q = 0; q < 4; ++q) bs[q] = col + q < p.N_out ? __ldg(p.col_bias + col + q) : 0.f;
      }
      tmem_ld_wait();
#pragma unroll
      for (int w = 0; w < 8; ++w)
        st_shared_v4(stg + stg_off<128>(lane, w), r[4 * w], r[4 * w + 1], r[4 * w + 2],
                     r[4 * w + 3]);
      __syncwarp();
#pragma unroll
      for (int pass = 0; pass < 8; ++pass) {
        const int rr = pass * 4 + (lane >> 3);
        uint4 v = ld_shared_v4(stg + stg_off<128>(rr, u));
        if (row_scaled) {
          const float f = rsc[pass];
          v.x = __float_as_uint(__uint_as_float(v.x) * (f * cs[0]));
          v.y = __float_as_uint(__uint_as_float(v.y) * (f * cs[1]));
          v.z = __float_as_uint(__uint_as_float(v.z) * (f * cs[2]));
          v.w = __float_as_uint(__uint_as_float(v.w) * (f * cs[3]));
        }
        if (p.col_bias != nullptr) {
          v.x = __float_as_uint(__uint_as_float(v.x) + bs[0]);
          v.y = __float_as_uint(__uint_as_float(v.y) + bs[1]);
          v.z = __float_as_uint(__uint_as_float(v.z) + bs[2]);
          v.w = __float_as_uint(__uint_as_float(v.w) + bs[3]);
        }
        const int grow = tile_row0 + rr;
        if (grow < row_end && col < p.N_out) {
          if constexpr (MODE == kScatter) {
            const int t = tok[pass];
            if (dcheck(t >= 0 && (p.c_rows == 0 || t < p.c_rows), p.err))
              red_add_v4(C + static_cast<size_t>(t) * p.N_out + col, v);
          } else {
            *reinterpret_cast<uint4*>(C + static_cast<size_t>(grow) * p.N_out + col) = v;
          }
        }
      }
      __syncwarp();
    }
  }
}

// Sum of 16 values in the order of a 32-lane xor-butterfly whose lanes 16-31 hold zero
// (warp_sum), so that the gates below equal the warp top-k's bit for bit.
__device__ __forceinline__ float butterfly_sum16(const float (&z)[16]) {
  const float a0 = (z[0] + z[8]) + (z[4] + z[12]), a2 = (z[2] + z[10]) + (z[6] + z[14]);
  const float a1 = (z[1] + z[9]) + (z[5] + z[13]), a3 = (z[3] + z[11]) + (z[7] + z[15]);
  return (a0 + a2) + (a1 + a3);
}

// kTopK epilogue (router logits): each thread owns one token row of the tile, which spans
// all N_out experts.  The logits (+ bias) are stored as in kPlain, and on the way the
// thread keeps the KS >= K best (logit, expert) pairs in registers, sorted by logit
// descending and expert ascending on ties (the warp top-k's order); KS is the smallest of
// 2, 4, 8, 16 that holds K, so the insertion costs no more slots than needed.  Then the
// softmax over the K kept logits, the gate drop and the renormalisation, as the warp
// top-k computes them (the same sums in the same order).
template <int BN, int KS>
__device__ __forceinline__ void epilogue_topk(const TcParams& p, uint32_t t_row, uint32_t stg,
                                              int lane, int tile_row0, int row_end) {
  float* C = static_cast<float*>(p.C);
  const int K = p.topk_k;
  uint32_t kk[KS];
  int ki[KS];
#pragma unroll
  for (int j = 0; j < KS; ++j) {
    kk[j] = 0u;  // below the key of every non-NaN float
    ki[j] = -1;
  }
  uint32_t thr = 0u;  // key of the K-th best so far
  const uint32_t kmask = 1u << (K - 1);
#pragma unroll 1
  for (int c = 0; c < BN; c += 32) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_row + c, r);
    tmem_ld_wait();
    if (p.col_bias != nullptr) {
      // one coalesced load of the chunk's 32 biases, then broadcast by shuffles
      const float bl = c + lane < p.N_out ? __ldg(p.col_bias + c + lane) : 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        r[j] = __float_as_uint(__uint_as_float(r[j]) + __shfl_sync(0xffffffffu, bl, j));
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
      const int col = c + u * 4;
      if (grow < row_end && col < p.N_out)
        *reinterpret_cast<uint4*>(C + static_cast<size_t>(grow) * p.N_out + col) = v;
    }
    __syncwarp();
    // this thread's 32 logits, read back from its own staging row
#pragma unroll 1
    for (int u = 0; u < 8; ++u) {
      const uint4 v4 = ld_shared_v4(stg + stg_off<128>(lane, u));
      const uint32_t vv[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int col = c + 4 * u + t;
        const uint32_t key = float_key(__uint_as_float(vv[t]));
        if (col < p.N_out && key > thr) {  // enters the top K: insertion into the sorted KS
#pragma unroll
          for (int q = KS - 1; q >= 1; --q) {  // selects only: every slot stays in a register
            const bool shift = key > kk[q - 1];
            const bool here = key > kk[q];
            kk[q] = shift ? kk[q - 1] : (here ? key : kk[q]);
            ki[q] = shift ? ki[q - 1] : (here ? col : ki[q]);
          }
          const bool first = key > kk[0];
          kk[0] = first ? key : kk[0];
          ki[0] = first ? col : ki[0];
          if (K == KS) {
            thr = kk[KS - 1];
          } else {  // the K-th key, picked with a one-hot mask (no indexed access)
            uint32_t t_new = 0u;
#pragma unroll
            for (int q = 0; q < KS; ++q) t_new |= kk[q] & ((kmask >> q) & 1u ? 0xffffffffu : 0u);
            thr = t_new;
          }
        }
      }
    }
  }
  const int grow = tile_row0 + lane;
  if (grow >= row_end) return;
  // keys back to logits (float_key is monotone; -0 came in as +0); the sums below run
  // over 16 terms (zeros past K) in the warp top-k's butterfly order
  float z[16], lv[KS];
#pragma unroll
  for (int q = 0; q < KS; ++q)
    lv[q] = __uint_as_float((kk[q] & 0x80000000u) ? (kk[q] & 0x7fffffffu) : ~kk[q]);
#pragma unroll
  for (int q = 0; q < 16; ++q) z[q] = (q < KS && q < K) ? expf(lv[q < KS ? q : 0] - lv[0]) : 0.f;
  const float s = butterfly_sum16(z);
  float w[16];
#pragma unroll
  for (int q = 0; q < 16; ++q) w[q] = z[q] / s;
  if (p.topk_theta > 0.f) {
#pragma unroll
    for (int q = 1; q < KS; ++q)
      if (q < K && w[q] < p.topk_theta) {
        w[q] = 0.f;
        ki[q] = -1;
      }
    const float s2 = butterfly_sum16(w);
#pragma unroll
    for (int q = 0; q < 16; ++q) w[q] = w[q] / s2;
  }
  int32_t* ids = p.topk_ids + static_cast<size_t>(grow) * K;
  float* wo = p.topk_w + static_cast<size_t>(grow) * K;
#pragma unroll
  for (int q = 0; q < KS; ++q)
    if (q < K) {
      ids[q] = ki[q];
      wo[q] = w[q];
    }
}

template <int BN, int MODE, bool SWAP, bool GATHER, bool F8 = false>
__global__ void __launch_bounds__(tc_threads(MODE, SWAP, GATHER, F8), 1)
    tc_grouped_gemm_kernel(const __grid_constant__ TcParams p) {
  constexpr int kEpi = tc_epi_warps(MODE, SWAP, F8);
  // With a row gather two producer warps (0 and 2 + kEpiWarps) take alternate k-steps: the
  // gather's many small requests then come from two warps (decode at one token: layer
  // 41.5 -> 39.6 us on GB300; without a gather a second producer measured no faster).
  constexpr int kProducers = GATHER ? 2 : 1;
  using Cfg = TcCfg<BN, MODE, SWAP, kEpi>;
  constexpr int S = Cfg::kStages;
  constexpr int kKStep = F8 ? 128 : BK;  // elements per 128-byte k-step
  constexpr int kTileRows = Cfg::kActRows;
  constexpr int kNC = BN < 32 ? BN : 32;  // TMEM columns per load in the swapped epilogue
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sAct = smem;
  uint8_t* sWgt = sAct + S * Cfg::kActBytes;
  uint8_t* sStg = sWgt + S * Cfg::kWgtBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + Cfg::kStgBytes);
  // bars: full[S], empty[S], tfull[2], tempty[2], mma_done
  static_assert(8 * (2 * S + 5) + 8 <= Cfg::kBarBytes, "barrier region");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_off = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + Cfg::kBarBytes);
  int* s_mt = s_off + kMaxGroups + 4;
  int* s_scan = s_mt + kMaxGroups + 4;
  int* s_light = s_scan + 32;

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
      mbar_init(tempty_bar(a), kEpi);
    }
    mbar_init(mma_done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmAct);
    tma_prefetch_desc(&p.tmWgt);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Everything below may read what earlier kernels on the stream wrote.
  grid_dep_wait();
  grid_dep_trigger();

  // Ragged schedule: every CTA derives the token tiles of every group from the offsets.
  const Sched sc = build_schedule(p, s_off, s_mt, s_light, s_scan, kTileRows);
  const int total = sc.total;

  if (warp == 0 || (kProducers == 2 && warp == 2 + kEpi)) {
    const int pid = warp == 0 ? 0 : 1;
    // ------------------------------------------------------------ producer ----
    // One elected lane waits for a free stage, arms its barrier and loads the weight and
    // activation tiles.  With a row gather, the whole warp runs the loop: lane 0 as
    // above for the weights, and lane l < rows/4 loads activation rows 4l..4l+3 of the
    // tile, each from its own source row (tile::gather4).
    constexpr bool gather = GATHER;
    constexpr int kGatherLanes = kTileRows / 4;
    static_assert(kGatherLanes <= 32, "one gather4 per lane");
    if (gather || elect_one_sync()) {
      const bool leader = !gather || lane == 0;
      const uint64_t pol_once = l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int idx = blockIdx.x; idx < total && ok; idx += gridDim.x) {
        int g, row0, row_end, n_tile;
        decode_tile(p, s_off, s_mt, s_light, sc, kTileRows, idx, g, row0, row_end, n_tile);
        const int n0 = n_tile * Cfg::kColsOut;  // first weight row of the tile
        const bool once = read_once(p, s_off, g, row0, row_end, kTileRows);
        // With a row gather only the lanes whose four rows start inside the group load
        // anything: the rest of the tile's rows are never stored, so whatever an earlier
        // stage left in that part of the buffer is harmless.  Within a lane, rows past
        // the group's end repeat a row of the tile.
        const int live_rows = min(row_end - row0, kTileRows);
        const int gather_lanes = GATHER ? (live_rows + 3) / 4 : 0;
        const uint32_t stage_tx =
            GATHER ? static_cast<uint32_t>(Cfg::kWgtBytes + gather_lanes * 512) : Cfg::kStageBytes;
        int src[4] = {0, 0, 0, 0};
        if (GATHER && lane < gather_lanes) {
          const int pad = p.gather_rows[row0];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = row0 + 4 * lane + i;
            src[i] = r < row_end ? p.gather_rows[r] : pad;
            if (!dcheck(src[i] >= 0 && src[i] < p.a_rows, p.err)) src[i] = 0;
          }
        }
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (kProducers > 1 && (issued % kProducers) != pid) {  // the other producer's step
            ++issued;
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          bool good = true;
          if (leader) good = mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err);
          if constexpr (GATHER) good = __shfl_sync(0xffffffffu, good ? 1 : 0, 0) != 0;
          if (!good) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(stage);
          const uint32_t a_dst = smem_u32(sAct + stage * Cfg::kActBytes);
          const uint32_t w_dst = smem_u32(sWgt + stage * Cfg::kWgtBytes);
          if (leader) {
            mbar_arrive_expect_tx(fb, stage_tx);
            if constexpr (!GATHER) tma_load_2d(a_dst, &p.tmAct, fb, kb * kKStep, row0);
            if (once) {
              tma_load_3d_hint(w_dst, &p.tmWgt, fb, kb * kKStep, n0, g, pol_once);
              if constexpr (MODE == kSwiGLU)
                tma_load_3d_hint(w_dst + Cfg::kWgtBox * 128, &p.tmWgt, fb, kb * kKStep,
                                 p.up_offset + n0, g, pol_once);
            } else {
              tma_load_3d(w_dst, &p.tmWgt, fb, kb * kKStep, n0, g);
              if constexpr (MODE == kSwiGLU)
                tma_load_3d(w_dst + Cfg::kWgtBox * 128, &p.tmWgt, fb, kb * kKStep,
                            p.up_offset + n0, g);
            }
          }
          if constexpr (GATHER) {
            __syncwarp();
            if (lane < gather_lanes)
              tma_gather4(a_dst + 512u * lane, &p.tmAct, fb, kb * kKStep, src[0], src[1], src[2],
                          src[3]);
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Drain: the most recent load of every stage must have landed before the CTA may
      // exit (they all have in a normal run; this matters only after an abort).  Both
      // producers of a gather wait for the same last S k-steps, whoever issued them.
      if (leader) {
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
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA ----
    if (elect_one_sync()) {
      constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(128, BN) : idesc_bf16_f32(128, BN);
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
          const uint32_t act = smem_u32(sAct + stage * Cfg::kActBytes);
          const uint32_t wgt = smem_u32(sWgt + stage * Cfg::kWgtBytes);
          const uint32_t a_base = SWAP ? wgt : act;
          const uint32_t b_base = SWAP ? act : wgt;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(a_base + kk * 32);
            const uint64_t bd = smem_desc_sw128(b_base + kk * 32);
            if constexpr (F8)
              tc_mma_e4m3(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            else
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
    clear_share(p, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x),
                static_cast<int>(threadIdx.x) - 64, 32 * kEpi);
    int local = 0;
    for (int idx = blockIdx.x; idx < total; idx += gridDim.x, ++local) {
      int g, row0, row_end, n_tile;
      decode_tile(p, s_off, s_mt, s_light, sc, kTileRows, idx, g, row0, row_end, n_tile);
      const int acc = local & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
      const bool ready = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.err);
      if constexpr (SWAP && MODE == kSwiGLU) {
        // the four epilogue warps meet at named barriers below: leave together or not at all
        if (epi_bar_any(!ready || *abort_flag != 0)) break;
      } else if (!ready) {
        break;
      }
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
      const int col0 = n_tile * Cfg::kColsOut;
      if constexpr (!SWAP) {
        const uint32_t stg =
            smem_u32(sStg) + static_cast<uint32_t>((warp - 2) * 32 * (MODE == kSwiGLU ? 64 : 128));
        const int tile_row0 = row0 + quad * 32;  // first global row of this warp's 32 rows
        if constexpr (MODE == kTopK) {
          if (p.topk_k <= 2)
            epilogue_topk<BN, 2>(p, t_row, stg, lane, tile_row0, row_end);
          else if (p.topk_k <= 4)
            epilogue_topk<BN, 4>(p, t_row, stg, lane, tile_row0, row_end);
          else if (p.topk_k <= 8)
            epilogue_topk<BN, 8>(p, t_row, stg, lane, tile_row0, row_end);
          else
            epilogue_topk<BN, 16>(p, t_row, stg, lane, tile_row0, row_end);
        } else
          epilogue_rows<BN, MODE>(p, t_row, stg, lane, tile_row0, row_end, col0, g,
                                  32 * ((warp - 2) / 4), 32 * (kEpi / 4));
      } else {
        // swapped: lane = weight row of the tile, column j = token row0 + j
        // FP8 operands: the token-row scales of every chunk, loaded before the chunk loops
        // (lane l of chunk k holds token row0 + k kNC + l's scale)
        constexpr int kSwChunks = BN / kNC;
        float sxv[kSwChunks];
        if (p.a_scale != nullptr) {
#pragma unroll
          for (int k = 0; k < kSwChunks; ++k) {
            const int r = row0 + k * kNC + lane;
            sxv[k] = r < row_end ? __ldg(p.a_scale + r) : 0.f;
          }
        }
        auto chunk_sx = [&](int c) {
          float sx = 0.f;
#pragma unroll
          for (int k = 0; k < kSwChunks; ++k)
            if (k * kNC == c) sx = sxv[k];
          return sx;
        };
        if constexpr (MODE == kSwiGLU) {
          // lanes 0-63: gate rows (quads 0, 1); lanes 64-127: up rows (quads 2, 3).
          // xchg[r][j] holds up row r for token j, rotated by r to spread the banks.
          float* xchg = reinterpret_cast<float*>(sStg);
          // FP8 operands: this lane's weight-row scale; token-row scales per column below
          float sw = 1.f;
          if (p.a_scale != nullptr) {
            const int wr = quad < 2 ? col0 + quad * 32 + lane
                                    : p.up_offset + col0 + (quad - 2) * 32 + lane;
            sw = col0 + (quad & 1) * 32 + lane < p.N_out
                     ? __ldg(p.b_scale + static_cast<size_t>(g) * p.b_rows + wr)
                     : 0.f;
          }
          if (quad >= 2) {
            const int r = (quad - 2) * 32 + lane;
#pragma unroll 1
            for (int c = 0; c < BN; c += kNC) {
              float v[32];
              tmem_ld_cols<kNC>(t_row + c, v);
              if (p.a_scale != nullptr) {
                const float sx = chunk_sx(c);
#pragma unroll
                for (int j = 0; j < kNC; ++j) v[j] *= sw * __shfl_sync(0xffffffffu, sx, j);
              }
#pragma unroll
              for (int j = 0; j < kNC; ++j) xchg[r * BN + ((c + j + r) % BN)] = v[j];
            }
          }
          epi_bar();
          if (quad < 2) {
            __nv_bfloat16* C = static_cast<__nv_bfloat16*>(p.C);
            const int r = quad * 32 + lane;
            const int col = col0 + r;
#pragma unroll 1
            for (int c = 0; c < BN; c += kNC) {
              float v[32];
              tmem_ld_cols<kNC>(t_row + c, v);
              if (p.a_scale != nullptr) {
                const float sx = chunk_sx(c);
#pragma unroll
                for (int j = 0; j < kNC; ++j) v[j] *= sw * __shfl_sync(0xffffffffu, sx, j);
              }
#pragma unroll
              for (int j = 0; j < kNC; ++j) {
                const int tok = row0 + c + j;
                if (tok < row_end && col < p.N_out) {
                  const float u = xchg[r * BN + ((c + j + r) % BN)];
                  C[static_cast<size_t>(tok) * p.N_out + col] =
                      __float2bfloat16_rn(silu_bf16out(v[j]) * u);
                }
              }
            }
          }
          epi_bar();
        } else {
          float* C = static_cast<float*>(p.C);
          const int col = col0 + quad * 32 + lane;
          const float b = (p.col_bias != nullptr && col < p.N_out) ? __ldg(p.col_bias + col) : 0.f;
          // FP8 operands: this lane's output-channel scale; token-row scales per column
          const float sw = (p.a_scale != nullptr && col < p.N_out)
                               ? __ldg(p.b_scale + static_cast<size_t>(g) * p.b_rows + col)
                               : 1.f;
#pragma unroll 1
          for (int c = 0; c < BN; c += kNC) {
            float v[32];
            tmem_ld_cols<kNC>(t_row + c, v);
            // kScatter: lane j loads row c + j's token and route weight; shuffles hand
            // them out
            int tok_l = 0;
            float w_l = 0.f;
            if constexpr (MODE == kScatter) {
              const int rl = row0 + c + lane;
              if (lane < kNC && rl < row_end) {
                tok_l = __ldg(p.row_token + rl);
                w_l = __ldg(p.row_w + rl);
              }
            }
            if (p.a_scale != nullptr) {
              const float sx = chunk_sx(c);
#pragma unroll
              for (int j = 0; j < kNC; ++j) v[j] *= sw * __shfl_sync(0xffffffffu, sx, j);
            }
#pragma unroll
            for (int j = 0; j < kNC; ++j) {
              const int row = row0 + c + j;
              int tok = 0;
              float wj = 0.f;
              if constexpr (MODE == kScatter) {
                tok = __shfl_sync(0xffffffffu, tok_l, j);
                wj = __shfl_sync(0xffffffffu, w_l, j);
              }
              if (row < row_end && col < p.N_out) {
                if constexpr (MODE == kScatter) {
                  if (dcheck(tok >= 0 && (p.c_rows == 0 || tok < p.c_rows), p.err))
                    red_add_f32(C + static_cast<size_t>(tok) * p.N_out + col, wj * v[j]);
                } else {
                  C[static_cast<size_t>(row) * p.N_out + col] = v[j] + b;
                }
              }
            }
          }
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


// ------------------------------------------------------ CTA pairs (2 SMs) ----
// The same grouped GEMM on pairs of CTAs (a cluster of 2) with tcgen05.mma.cta_group::2:
// one 256 x 256 accumulator tile per pair, rows 0-127 in the even CTA's TMEM and 128-255
// in the odd CTA's.  Each CTA loads its own 128 rows of A and one half of the 256 B rows
// (SwiGLU: the even CTA the 128 gate rows, the odd CTA the matching 128 up rows), so a
// stage is 32 KB per CTA and 6 stages fit; per SM the L2->shared traffic per MMA FLOP is
// two thirds of the single-CTA kernel's.
//   * both CTAs' TMA loads complete on the even CTA's full barrier (cta_group::2 loads);
//   * the even CTA's single MMA thread issues the pair MMAs and commits with a multicast
//     arrive on both CTAs' empty (per stage) and tmem-full (per accumulator) barriers;
//   * both CTAs' epilogue warps arrive on the even CTA's tmem-empty barrier (count 8);
//   * a cluster barrier after initialisation and before TMEM release keeps every
//     remote arrive and shared-memory read inside the peer's lifetime.
// A group's last tile holds r < 256 rows.  Padded to 256 token rows it costs a full pair
// step (512 MMA rows x 256 columns per k-block); in swapped order (the tile's 256 weight
// rows on the MMA's M side, 128 per CTA, and its r token rows, rounded up to N, a multiple
// of 32, as the MMA's N split 2 x N/2 between the CTAs) a k-block moves 16 KB + 64 N bytes
// per CTA instead of 32 KB.  Tails up to kPairTailMaxN rows are run that way.
constexpr int kPairTailMaxN = 192;

__device__ __forceinline__ int pair_tail_n(int row0, int row_end) {
  const int r = row_end - row0;
  if (r >= 256) return 0;
  const int n = (r + 31) / 32 * 32;
  return n <= kPairTailMaxN ? n : 0;
}

// Epilogue of a swapped pair tail (see pair_tail_n) in one CTA of the pair: TMEM lane L
// (quad * 32 + lane) is weight row L of this CTA's 128, accumulator column j is token row
// row0 + j (j < tn).  SwiGLU: lanes 0-63 hold gate rows n0 + 64 rank + L, lanes 64-127 the
// matching up rows, whose values reach the gate lanes through `stg` (64 x 32 floats per
// round).  Plain / scatter: lane L is output column n0 + 128 rank + L.
template <int MODE>
__device__ __forceinline__ void epilogue_pair_tail(const TcParams& p, uint32_t t_row, uint8_t* stg,
                                                   int quad, int lane, int rank, int tn, int row0,
                                                   int row_end, int n0, int group) {
  const int L = quad * 32 + lane;
  // FP8 operands: v[j] (token row0 + c + j) is scaled by this lane's weight-row scale and
  // that token row's scale.  The token-row scales of every chunk and the lane's weight-row
  // scale are loaded once, before the chunk loop (one dependent load, not one per chunk).
  constexpr int kMaxChunks = kPairTailMaxN / 32;
  float sxv[kMaxChunks];
  if (p.a_scale != nullptr) {
#pragma unroll
    for (int k = 0; k < kMaxChunks; ++k) {
      const int r = row0 + 32 * k + lane;
      sxv[k] = 32 * k < tn && r < row_end ? __ldg(p.a_scale + r) : 0.f;
    }
  }
  auto weight_scale = [&](int wrow, bool live) {
    return p.a_scale != nullptr && live
               ? __ldg(p.b_scale + static_cast<size_t>(group) * p.b_rows + wrow)
               : 0.f;
  };
  auto scale = [&](float (&v)[32], int c, float sw) {
    if (p.a_scale == nullptr) return;
    float sx = 0.f;
#pragma unroll
    for (int k = 0; k < kMaxChunks; ++k)
      if (32 * k == c) sx = sxv[k];
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] *= sw * __shfl_sync(0xffffffffu, sx, j);
  };
  if constexpr (MODE == kSwiGLU) {
    float* xchg = reinterpret_cast<float*>(stg);  // [64][32], rotated by row
    __nv_bfloat16* C = static_cast<__nv_bfloat16*>(p.C);
    const int col = n0 + 64 * rank + (L & 63);
    const float sw = weight_scale(quad >= 2 ? p.up_offset + col : col, col < p.N_out);
#pragma unroll 1
    for (int c = 0; c < tn; c += 32) {
      float v[32];
      if (quad >= 2) {
        const int r = L - 64;
        tmem_ld_cols<32>(t_row + c, v);
        scale(v, c, sw);
#pragma unroll
        for (int j = 0; j < 32; ++j) xchg[r * 32 + ((j + r) & 31)] = v[j];
      }
      epi_bar();
      if (quad < 2) {
        tmem_ld_cols<32>(t_row + c, v);
        scale(v, c, sw);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int tok = row0 + c + j;
          if (tok < row_end && col < p.N_out) {
            const float u = xchg[L * 32 + ((j + L) & 31)];
            C[static_cast<size_t>(tok) * p.N_out + col] = __float2bfloat16_rn(silu_bf16out(v[j]) * u);
          }
        }
      }
      epi_bar();
    }
  } else {
    float* C = static_cast<float*>(p.C);
    const int col = n0 + 128 * rank + L;
    const float b = (p.col_bias != nullptr && col < p.N_out) ? __ldg(p.col_bias + col) : 0.f;
    const float sw = weight_scale(col, col < p.N_out);
#pragma unroll 1
    for (int c = 0; c < tn; c += 32) {
      float v[32];
      tmem_ld_cols<32>(t_row + c, v);
      // kScatter: lane j loads row c + j's token and route weight; shuffles hand them out
      int dst_l = 0;
      float w_l = 0.f;
      if constexpr (MODE == kScatter) {
        const int tk = row0 + c + lane;
        if (tk < row_end) {
          dst_l = __ldg(p.row_token + tk);
          w_l = __ldg(p.row_w + tk);
        }
      }
      scale(v, c, sw);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int tok = row0 + c + j;
        int dst = 0;
        float wj = 0.f;
        if constexpr (MODE == kScatter) {
          dst = __shfl_sync(0xffffffffu, dst_l, j);
          wj = __shfl_sync(0xffffffffu, w_l, j);
        }
        if (tok < row_end && col < p.N_out) {
          if constexpr (MODE == kScatter) {
            if (dcheck(dst >= 0 && (p.c_rows == 0 || dst < p.c_rows), p.err))
              red_add_f32(C + static_cast<size_t>(dst) * p.N_out + col, wj * v[j]);
          } else {
            C[static_cast<size_t>(tok) * p.N_out + col] = v[j] + b;
          }
        }
      }
    }
  }
}

template <int MODE>
struct TcPairCfg {
  static constexpr int kABytes = 128 * BK * 2;  // this CTA's 128 rows of A
  static constexpr int kBBytes = 128 * BK * 2;  // this CTA's half of the 256 B rows
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = 6;
  static constexpr int kBN = 256;  // MMA N over the pair
  static constexpr int kColsOut = MODE == kSwiGLU ? 128 : 256;
  static constexpr int kTmemCols = 512;
  static constexpr int kStgBytes = kEpiWarps * 32 * (MODE == kSwiGLU ? 64 : 128);
  static constexpr int kBarBytes = 384;
  static constexpr int kSchedBytes = 3 * (kMaxGroups + 4) * 4 + 32 * 4;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kStgBytes + kBarBytes + kSchedBytes;
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

template <int MODE, bool F8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    tc_pair_gemm_kernel(const __grid_constant__ TcParams p) {
  using Cfg = TcPairCfg<MODE>;
  constexpr int S = Cfg::kStages;
  constexpr int kKStep = F8 ? 128 : BK;  // elements per 128-byte k-step
  constexpr int BN = Cfg::kBN;
  constexpr int kTileRows = 256;  // token rows per pair tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + S * Cfg::kABytes;
  uint8_t* sStg = sB + S * Cfg::kBBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + Cfg::kStgBytes);
  // bars: full[S], empty[S], tfull[2], tempty[2], mma_done, {tmem slot, abort flag},
  // tile ring full[kTileRing], empty[kTileRing], slots
  static_assert(8 * (2 * S + 6 + 2 * kTileRing) + 4 * kTileRing <= Cfg::kBarBytes,
                "barrier region");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_off = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(bars) + Cfg::kBarBytes);
  int* s_mt = s_off + kMaxGroups + 4;
  int* s_scan = s_mt + kMaxGroups + 4;
  int* s_light = s_scan + 32;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t mma_done_bar = bar0 + 8u * (2 * S + 4);
  // dynamic tile order: the even CTA's producer draws; consumers are the even CTA's MMA
  // thread and epilogue warps and the odd CTA's producer and epilogue warps
  const bool dyn = p.tile_counter != nullptr;
  const TileRing ring{bar0 + 8u * (2 * S + 6), bar0 + 8u * (2 * S + 6 + kTileRing),
                      bar0 + 8u * (2 * S + 6 + 2 * kTileRing)};

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), 2 * kEpiWarps);
    }
    mbar_init(mma_done_bar, 1);
    for (int r = 0; r < kTileRing; ++r) {
      mbar_init(ring.full0 + 8u * r, 1);
      mbar_init(ring.empty0 + 8u * r, 2 + 2 * kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&p.tmAct);
    tma_prefetch_desc(&p.tmWgt);
    tma_prefetch_desc(&p.tmActS16);
    tma_prefetch_desc(&p.tmActS32);
    tma_prefetch_desc(&p.tmActS64);
    if constexpr (MODE == kSwiGLU) tma_prefetch_desc(&p.tmWgtS);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // the peer's barriers exist before anything arrives on them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  grid_dep_wait();
  grid_dep_trigger();

  const Sched sc = build_schedule(p, s_off, s_mt, s_light, s_scan, kTileRows);
  const int total = sc.total;
  const int pair = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);

  if (warp == 0) {
    // ------------------------------------------------------------ producer ----
    if (elect_one_sync()) {
      const uint64_t pol_once = l2_policy_evict_first();
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      const bool draws = dyn && rank == 0;  // the even CTA draws, the odd one takes
      int cur = -1, nxt = -1;                // (drawing) tiles j and j + 1, already published
      if (draws) {
        const int t0 = atomicAdd(p.tile_counter, 1), t1 = atomicAdd(p.tile_counter, 1);
        cur = ring_index(t0, total);
        nxt = ring_index(t1, total);
        ok = ring_publish(ring, 0, cur, abort_flag, p.err) &&
             ring_publish(ring, 1, nxt, abort_flag, p.err);
      }
      for (int j = 0; ok; ++j) {
        int idx = pair + j * npairs;
        if (draws) idx = cur;
        else if (dyn) idx = ring_take<true>(ring, j, abort_flag, p.err);
        if (idx < 0 || idx >= total) break;
        const int ticket = draws ? atomicAdd(p.tile_counter, 1) : 0;  // tile j + 2
        int g, row0, row_end, n_tile;
        decode_tile(p, s_off, s_mt, s_light, sc, kTileRows, idx, g, row0, row_end, n_tile);
        const int n0 = n_tile * Cfg::kColsOut;
        const int a_row = row0 + static_cast<int>(rank) * 128;
        const int b_row = MODE == kSwiGLU ? (rank == 0 ? n0 : p.up_offset + n0)
                                          : n0 + static_cast<int>(rank) * 128;
        // swapped tail: sA takes this CTA's 128 weight rows, sB its N/2 token rows
        const int tn = pair_tail_n(row0, row_end);
        const int t_row = row0 + static_cast<int>(rank) * (tn / 2);
        const bool once = read_once(p, s_off, g, row0, row_end, kTileRows);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(empty_bar(stage), phase ^ 1u, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const uint32_t fb_leader = mapa_shared(full_bar(stage), 0);
          const uint32_t a_dst = smem_u32(sA + stage * Cfg::kABytes);
          const uint32_t b_dst = smem_u32(sB + stage * Cfg::kBBytes);
          if (tn > 0) {
            if (rank == 0)
              mbar_arrive_expect_tx(full_bar(stage), 2u * (Cfg::kABytes + tn * 64));
            if constexpr (MODE == kSwiGLU) {  // gate rows w0.. then the matching up rows
              if (once)
                tma_load_4d_pair_hint(a_dst, &p.tmWgtS, fb_leader, kb * kKStep,
                                      n0 + static_cast<int>(rank) * 64, 0, g, pol_once);
              else
                tma_load_4d_pair(a_dst, &p.tmWgtS, fb_leader, kb * kKStep,
                                 n0 + static_cast<int>(rank) * 64, 0, g);
            } else if (once) {
              tma_load_3d_pair_hint(a_dst, &p.tmWgt, fb_leader, kb * kKStep, b_row, g, pol_once);
            } else {
              tma_load_3d_pair(a_dst, &p.tmWgt, fb_leader, kb * kKStep, b_row, g);
            }
            // this CTA's tn/2 token rows in boxes of 64, 32 and 16 rows
            int rr = 0;
            for (; rr + 64 <= tn / 2; rr += 64)
              tma_load_2d_pair(b_dst + 128u * rr, &p.tmActS64, fb_leader, kb * kKStep, t_row + rr);
            if (rr + 32 <= tn / 2) {
              tma_load_2d_pair(b_dst + 128u * rr, &p.tmActS32, fb_leader, kb * kKStep, t_row + rr);
              rr += 32;
            }
            if (rr < tn / 2)
              tma_load_2d_pair(b_dst + 128u * rr, &p.tmActS16, fb_leader, kb * kKStep, t_row + rr);
            ++issued;
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (rank == 0) mbar_arrive_expect_tx(full_bar(stage), 2 * Cfg::kStageBytes);
          tma_load_2d_pair(a_dst, &p.tmAct, fb_leader, kb * kKStep, a_row);
          if (once)
            tma_load_3d_pair_hint(b_dst, &p.tmWgt, fb_leader, kb * kKStep, b_row, g, pol_once);
          else
            tma_load_3d_pair(b_dst, &p.tmWgt, fb_leader, kb * kKStep, b_row, g);
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (draws && ok) {
          ok = ring_publish(ring, j + 2, ring_index(ticket, total), abort_flag, p.err);
          cur = nxt;
          nxt = ring_index(ticket, total);
        }
      }
      if (rank == 0) {
        // Drain: both CTAs' loads complete on the even CTA's full barriers.
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
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA ----
    if (rank == 0 && elect_one_sync()) {
      constexpr uint32_t idesc = F8 ? idesc_e4m3_f32(256, BN) : idesc_bf16_f32(256, BN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int j = 0; ok; ++j, ++local) {
        int idx = pair + j * npairs;
        if (dyn) idx = ring_take<false>(ring, j, abort_flag, p.err);
        if (idx < 0 || idx >= total) break;
        const int acc = local & 1;
        const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
        int g, row0, row_end, n_tile;
        decode_tile(p, s_off, s_mt, s_light, sc, kTileRows, idx, g, row0, row_end, n_tile);
        const int tn = pair_tail_n(row0, row_end);
        const uint32_t idesc_t =
            tn > 0 ? (F8 ? idesc_e4m3_f32(256, tn) : idesc_bf16_f32(256, tn)) : idesc;
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
          for (int kk = 0; kk < BK / 16; ++kk)
            if constexpr (F8)
              tc_mma_e4m3_pair(d_tmem, smem_desc_sw128(a_base + kk * 32),
                               smem_desc_sw128(b_base + kk * 32), idesc_t, (kb | kk) != 0 ? 1u : 0u);
            else
              tc_mma_bf16_pair(d_tmem, smem_desc_sw128(a_base + kk * 32),
                               smem_desc_sw128(b_base + kk * 32), idesc_t, (kb | kk) != 0 ? 1u : 0u);
          tc_commit_pair(empty_bar(stage), 0x3);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc_commit_pair(tfull_bar(acc), 0x3);
      }
      if (!ok || *abort_flag) {
        tc_commit_pair(mma_done_bar, 0x1);
        volatile int no_abort = 0;
        mbar_wait(mma_done_bar, 0, &no_abort, p.err);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue ----
    const int quad = warp & 3;
    clear_share(p, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x),
                static_cast<int>(threadIdx.x) - 64, 32 * kEpiWarps);
    const uint32_t stg =
        smem_u32(sStg) + static_cast<uint32_t>((warp - 2) * 32 * (MODE == kSwiGLU ? 64 : 128));
    int local = 0;
    for (int j = 0;; ++j, ++local) {
      int idx = pair + j * npairs;
      if (dyn) {
        if (lane == 0)
          idx = rank == 0 ? ring_take<false>(ring, j, abort_flag, p.err)
                          : ring_take<true>(ring, j, abort_flag, p.err);
        idx = __shfl_sync(0xffffffffu, idx, 0);
        if (epi_bar_any(idx < 0)) break;  // the four warps stop together
      }
      if (idx >= total) break;
      int g, row0, row_end, n_tile;
      decode_tile(p, s_off, s_mt, s_light, sc, kTileRows, idx, g, row0, row_end, n_tile);
      const int acc = local & 1;
      const uint32_t acc_phase = static_cast<uint32_t>(local >> 1) & 1u;
      const bool ready = mbar_wait(tfull_bar(acc), acc_phase, abort_flag, p.err);
      // swapped tails meet at named barriers: the four epilogue warps leave together
      if (epi_bar_any(!ready || *abort_flag != 0)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
      const int tn = pair_tail_n(row0, row_end);
      if (tn > 0) {
        epilogue_pair_tail<MODE>(p, t_row, sStg, quad, lane, static_cast<int>(rank), tn, row0,
                                 row_end, n_tile * Cfg::kColsOut, g);
      } else {
        const int tile_row0 = row0 + static_cast<int>(rank) * 128 + quad * 32;
        epilogue_rows<BN, MODE>(p, t_row, stg, lane, tile_row0, row_end, n_tile * Cfg::kColsOut,
                                g);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // no peer still reads this CTA's shared memory or arrives on it
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
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

// 2D / 3D maps of FP8 (one byte per element) matrices: box = 128 columns (128 bytes, one
// swizzle row, the same smem layout as 64 bf16 columns) x box_rows rows.
bool make_map_2d_u8(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                    uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool make_map_3d_u8(CUtensorMap* m, const void* base, uint64_t G, uint64_t rows, uint64_t cols,
                    uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {cols, rows, G};
  cuuint64_t strides[2] = {cols, rows * cols};
  cuuint32_t box[3] = {128, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4D bf16 map of [G][2][half][cols] (two stacked blocks of `half` rows per group), box =
// 1 x 2 x 64 rows x 64 columns: rows r..r+63 of both blocks in one load.
bool make_map_4d_halves(CUtensorMap* m, const void* base, uint64_t G, uint64_t half,
                        uint64_t cols, bool u8 = false) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  const uint64_t eb = u8 ? 1 : 2;  // bytes per element; the box is 128 bytes wide either way
  cuuint64_t dims[4] = {cols, half, 2, G};
  cuuint64_t strides[3] = {cols * eb, half * cols * eb, 2 * half * cols * eb};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / eb), 64, 2, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN, int MODE, bool SWAP, bool GATHER = false, bool F8 = false>
cudaError_t launch_one(const GroupedGemm& g, unsigned* err, int num_sms, cudaStream_t s,
                       const float* a_scale = nullptr, const float* b_scale = nullptr) {
  using Cfg = TcCfg<BN, MODE, SWAP, tc_epi_warps(MODE, SWAP, F8)>;  // the kernel's own layout
  auto kernel = tc_grouped_gemm_kernel<BN, MODE, SWAP, GATHER, F8>;
  if (GATHER != (g.gather_rows != nullptr)) return cudaErrorInvalidValue;
  static int attr_set_dev = -1;  // the attribute is per function and device
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_set_dev != dev) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    attr_set_dev = dev;
  }
  TcParams p;
  memset(&p, 0, sizeof(p));
  // with a row gather the map covers the source rows, one row per box
  const bool ok_map =
      F8 ? make_map_2d_u8(&p.tmAct, g.A, static_cast<uint64_t>(g.rows_alloc),
                          static_cast<uint64_t>(g.Kd), Cfg::kActRows)
      : g.gather_rows != nullptr
          ? make_map_2d(&p.tmAct, g.A, static_cast<uint64_t>(g.src_rows),
                        static_cast<uint64_t>(g.Kd), 1)
          : make_map_2d(&p.tmAct, g.A, static_cast<uint64_t>(g.rows_alloc),
                        static_cast<uint64_t>(g.Kd), Cfg::kActRows);
  if (!ok_map) return cudaErrorInvalidValue;
  p.gather_rows = g.gather_rows;
  p.topk_k = g.topk_k;
  p.topk_theta = g.topk_theta;
  p.topk_ids = g.topk_ids;
  p.topk_w = g.topk_w;
  if (F8 ? !make_map_3d_u8(&p.tmWgt, g.B, static_cast<uint64_t>(g.G), static_cast<uint64_t>(g.Nb),
                           static_cast<uint64_t>(g.Kd), Cfg::kWgtBox)
         : !make_map_3d(&p.tmWgt, g.B, static_cast<uint64_t>(g.G), static_cast<uint64_t>(g.Nb),
                        static_cast<uint64_t>(g.Kd), Cfg::kWgtBox))
    return cudaErrorInvalidValue;
  p.a_scale = a_scale;
  p.b_scale = b_scale;
  p.b_rows = g.Nb;
  p.C = g.C;
  p.col_bias = g.col_bias;
  p.offsets = g.offsets;
  p.row_token = g.row_token;
  p.row_w = g.row_w;
  p.num_groups = g.G;
  p.err = err;
  p.rows_alloc = g.rows_alloc;
  p.num_kb = F8 ? g.Kd / 128 : g.Kd / BK;  // 128-byte k-steps either way
  p.N_out = g.N_out;
  p.n_tiles = (g.N_out + Cfg::kColsOut - 1) / Cfg::kColsOut;
  p.up_offset = g.up_offset;
  p.swz = kSwz;
  p.interleave = (!SWAP && g.offsets != nullptr) ? 1 : 0;
  p.a_rows = GATHER ? g.src_rows : g.rows_alloc;
  p.c_rows = g.c_rows;
  p.zero_ptr = g.zero_ptr;
  p.zero_n = g.zero_n;
  const long long rows_tiles = (g.rows_alloc + Cfg::kActRows - 1) / Cfg::kActRows;
  const long long max_mt = g.offsets != nullptr ? rows_tiles + g.G : rows_tiles;
  const long long max_tiles = max_mt * p.n_tiles;
  if (max_tiles == 0) return cudaSuccess;
  return launch_pdl(kernel, dim3(static_cast<unsigned>(max_tiles < num_sms ? max_tiles : num_sms)),
                    dim3(tc_threads(MODE, SWAP, GATHER, F8)), Cfg::kSmem, s, p);
}


template <int MODE, bool F8 = false>
cudaError_t launch_pair(const GroupedGemm& g, unsigned* err, int num_sms, cudaStream_t s,
                        const float* a_scale = nullptr, const float* b_scale = nullptr) {
  using Cfg = TcPairCfg<MODE>;
  auto kernel = tc_pair_gemm_kernel<MODE, F8>;
  static int attr_set_dev = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (attr_set_dev != dev) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (e != cudaSuccess) return e;
    attr_set_dev = dev;
  }
  TcParams p;
  memset(&p, 0, sizeof(p));
  const uint64_t rows = static_cast<uint64_t>(g.rows_alloc), kd = static_cast<uint64_t>(g.Kd);
  auto act = [&](CUtensorMap* m, uint32_t box) {
    return F8 ? make_map_2d_u8(m, g.A, rows, kd, box) : make_map_2d(m, g.A, rows, kd, box);
  };
  if (!act(&p.tmAct, 128) ||
      !(F8 ? make_map_3d_u8(&p.tmWgt, g.B, static_cast<uint64_t>(g.G),
                            static_cast<uint64_t>(g.Nb), kd, 128)
           : make_map_3d(&p.tmWgt, g.B, static_cast<uint64_t>(g.G), static_cast<uint64_t>(g.Nb),
                         kd, 128)))
    return cudaErrorInvalidValue;
  if (!act(&p.tmActS16, 16) || !act(&p.tmActS32, 32) || !act(&p.tmActS64, 64))
    return cudaErrorInvalidValue;
  if (MODE == kSwiGLU) {
    // [G][2][I][Kd]: the gate block then the up block of each expert
    if (g.up_offset * 2 != g.Nb || g.up_offset % 64 != 0 ||
        !make_map_4d_halves(&p.tmWgtS, g.B, static_cast<uint64_t>(g.G),
                            static_cast<uint64_t>(g.up_offset), kd, F8))
      return cudaErrorInvalidValue;
  }
  p.a_scale = a_scale;
  p.b_scale = b_scale;
  p.b_rows = g.Nb;
  p.C = g.C;
  p.col_bias = g.col_bias;
  p.offsets = g.offsets;
  p.row_token = g.row_token;
  p.row_w = g.row_w;
  p.num_groups = g.G;
  p.err = err;
  p.rows_alloc = g.rows_alloc;
  p.num_kb = F8 ? g.Kd / 128 : g.Kd / BK;  // 128-byte k-steps either way
  p.N_out = g.N_out;
  p.n_tiles = (g.N_out + Cfg::kColsOut - 1) / Cfg::kColsOut;
  p.up_offset = g.up_offset;
  p.swz = kSwz;
  p.interleave = g.offsets != nullptr ? 1 : 0;
  p.tile_counter = g.tile_counter;
  p.a_rows = g.rows_alloc;
  p.c_rows = g.c_rows;
  p.zero_ptr = g.zero_ptr;
  p.zero_n = g.zero_n;
  const long long rows_tiles = (g.rows_alloc + 255) / 256;
  const long long max_mt = g.offsets != nullptr ? rows_tiles + g.G : rows_tiles;
  const long long max_tiles = max_mt * p.n_tiles;
  if (max_tiles == 0) return cudaSuccess;
  const long long pairs = max_tiles < num_sms / 2 ? max_tiles : num_sms / 2;
  return launch_pdl(kernel, dim3(static_cast<unsigned>(2 * pairs)), dim3(kThreads), Cfg::kSmem, s,
                    p);
}
}  // namespace

bool make_tma_2d_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols,
                      uint32_t box_rows) {
  return make_map_2d(m, base, rows, cols, box_rows);
}

int tc_swap_tokens(int max_rows_per_group) {
  if (max_rows_per_group <= 16) return 16;
  if (max_rows_per_group <= 32) return 32;
  return 64;
}

cudaError_t launch_gate_up_fp8(const GroupedGemm& g, const float* a_scale, const float* b_scale,
                               unsigned* err, int num_sms, cudaStream_t s) {
  if (g.mode != kSwiGLU || g.G > kMaxGroups || g.Kd % 128 != 0 || a_scale == nullptr ||
      b_scale == nullptr || g.gather_rows != nullptr)
    return cudaErrorInvalidValue;
  if (g.pair && g.swap_tokens == 0)
    return launch_pair<kSwiGLU, true>(g, err, num_sms, s, a_scale, b_scale);
  if (g.swap_tokens > 0) {
    const int bt = tc_swap_tokens(g.swap_tokens);
    if (bt == 16) return launch_one<16, kSwiGLU, true, false, true>(g, err, num_sms, s, a_scale, b_scale);
    if (bt == 32) return launch_one<32, kSwiGLU, true, false, true>(g, err, num_sms, s, a_scale, b_scale);
    return launch_one<64, kSwiGLU, true, false, true>(g, err, num_sms, s, a_scale, b_scale);
  }
  return launch_one<256, kSwiGLU, false, false, true>(g, err, num_sms, s, a_scale, b_scale);
}

cudaError_t launch_down_fp8(const GroupedGemm& g, const float* a_scale, const float* b_scale,
                            unsigned* err, int num_sms, cudaStream_t s) {
  if ((g.mode != kPlain && g.mode != kScatter) || g.G > kMaxGroups || g.Kd % 128 != 0 ||
      a_scale == nullptr || b_scale == nullptr || g.gather_rows != nullptr)
    return cudaErrorInvalidValue;
  if (g.pair && g.swap_tokens == 0) {
    if (g.mode == kScatter) return launch_pair<kScatter, true>(g, err, num_sms, s, a_scale, b_scale);
    if (g.N_out > 128) return launch_pair<kPlain, true>(g, err, num_sms, s, a_scale, b_scale);
  }
  if (g.swap_tokens > 0) {
    const int bt = tc_swap_tokens(g.swap_tokens);
    if (g.mode == kScatter) {
      if (bt == 16) return launch_one<16, kScatter, true, false, true>(g, err, num_sms, s, a_scale, b_scale);
      if (bt == 32) return launch_one<32, kScatter, true, false, true>(g, err, num_sms, s, a_scale, b_scale);
      return launch_one<64, kScatter, true, false, true>(g, err, num_sms, s, a_scale, b_scale);
    }
    if (bt == 16) return launch_one<16, kPlain, true, false, true>(g, err, num_sms, s, a_scale, b_scale);
    if (bt == 32) return launch_one<32, kPlain, true, false, true>(g, err, num_sms, s, a_scale, b_scale);
    return launch_one<64, kPlain, true, false, true>(g, err, num_sms, s, a_scale, b_scale);
  }
  if (g.mode == kScatter)
    return launch_one<256, kScatter, false, false, true>(g, err, num_sms, s, a_scale, b_scale);
  return launch_one<256, kPlain, false, false, true>(g, err, num_sms, s, a_scale, b_scale);
}

cudaError_t launch_grouped_gemm_tc(const GroupedGemm& g, unsigned* err, int num_sms,
                                   cudaStream_t s) {
  if (g.dtype != kBF16) return cudaErrorInvalidValue;
  if (g.G > kMaxGroups) return cudaErrorInvalidValue;
  if (g.gather_rows != nullptr && g.src_rows <= 0) return cudaErrorInvalidValue;
  if (g.mode == kTopK) {  // router logits with the top-k in the epilogue: one tile spans E
    if (g.swap_tokens > 0 || g.pair || g.gather_rows != nullptr || g.offsets != nullptr ||
        g.N_out > 256 || g.topk_k < 1 || g.topk_k > 16 || g.topk_ids == nullptr ||
        g.topk_w == nullptr)
      return cudaErrorInvalidValue;
    if (g.N_out <= 64) return launch_one<64, kTopK, false>(g, err, num_sms, s);
    if (g.N_out <= 128) return launch_one<128, kTopK, false>(g, err, num_sms, s);
    return launch_one<256, kTopK, false>(g, err, num_sms, s);
  }
  if (g.gather_rows != nullptr) {  // the row-gather gate/up variant
    if (g.mode != kSwiGLU) return cudaErrorInvalidValue;
    if (g.swap_tokens > 0) {
      const int bt = tc_swap_tokens(g.swap_tokens);
      if (bt == 16) return launch_one<16, kSwiGLU, true, true>(g, err, num_sms, s);
      if (bt == 32) return launch_one<32, kSwiGLU, true, true>(g, err, num_sms, s);
      return launch_one<64, kSwiGLU, true, true>(g, err, num_sms, s);
    }
    return launch_one<256, kSwiGLU, false, true>(g, err, num_sms, s);
  }
  if (g.swap_tokens > 0) {
    const int bt = tc_swap_tokens(g.swap_tokens);
    if (g.mode == kSwiGLU) {
      if (bt == 16) return launch_one<16, kSwiGLU, true>(g, err, num_sms, s);
      if (bt == 32) return launch_one<32, kSwiGLU, true>(g, err, num_sms, s);
      return launch_one<64, kSwiGLU, true>(g, err, num_sms, s);
    }
    if (g.mode == kScatter) {
      if (bt == 16) return launch_one<16, kScatter, true>(g, err, num_sms, s);
      if (bt == 32) return launch_one<32, kScatter, true>(g, err, num_sms, s);
      return launch_one<64, kScatter, true>(g, err, num_sms, s);
    }
    if (bt == 16) return launch_one<16, kPlain, true>(g, err, num_sms, s);
    if (bt == 32) return launch_one<32, kPlain, true>(g, err, num_sms, s);
    return launch_one<64, kPlain, true>(g, err, num_sms, s);
  }
  if (g.pair) {
    if (g.mode == kSwiGLU) return launch_pair<kSwiGLU>(g, err, num_sms, s);
    if (g.mode == kScatter) return launch_pair<kScatter>(g, err, num_sms, s);
    if (g.N_out > 128) return launch_pair<kPlain>(g, err, num_sms, s);
  }
  if (g.mode == kScatter) return launch_one<256, kScatter, false>(g, err, num_sms, s);
  if (g.mode == kSwiGLU) return launch_one<256, kSwiGLU, false>(g, err, num_sms, s);
  if (g.N_out > 128) return launch_one<256, kPlain, false>(g, err, num_sms, s);
  if (g.N_out > 64) return launch_one<128, kPlain, false>(g, err, num_sms, s);
  return launch_one<64, kPlain, false>(g, err, num_sms, s);
}

}  // namespace moe
