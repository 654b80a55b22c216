// A1 + A2: DSA indexer scores and Top-K selection.
//
// [P3] "From 1M total to 15+ x 1M: GLM-5.3 KV-cache offload", section
// "起点" (starting point): the DSA indexer selects the Top-2048 history
// positions; section "第一次决策" (first decision): the selection is the exact
// GPU path with a BF16 query.
// [W7] "How a dual 8-card AMD W7900D machine runs GLM5.3", section
// "Kernel 快了，整条链却可能更慢" (a faster kernel can still slow the chain):
// the radix select's serial tail and its extra launches cost more than the
// kernel time they saved, so here the whole select is one clustered launch.
//
// Design (GB300):
//  * k_dsa_score: a persistent grid, as many CTAs per SM as shared and tensor
//    memory allow (4 on the whole device, 5 on an SM partition of fewer SMs,
//    for one query row), walks the flattened (unit, tile) space, whole CTAs
//    per unit where the grid holds one per unit. Three roles per CTA meet
//    only at mbarriers: a producer warp copies each 128-position tile of bf16
//    keys (16 KB) by tiled TMA through a per-unit tensor map made on the
//    device, landing 128-byte swizzled as MMA operand A; an MMA warp issues
//    four tcgen05.mma kind::f16 (bf16 x bf16 -> fp32, M = 128 positions,
//    N = 8 heads per query row padded to 16, K = 64) against the unit's query
//    rows held as operand B, into one of two TMEM accumulators; four epilogue
//    warps read the accumulator (one position per thread), apply ReLU and the
//    head weights, and turn each score into an order-preserving uint32 key
//    (written coalesced) counted in a shared histogram of its top 12 bits
//    (two 16-bit bins per word, one shared atomic per distinct bin per warp),
//    merged into the call's per-(unit, row) histogram when the CTA leaves a
//    unit; each warp also writes the largest key of its 32 positions.
//  * k_topk_select: one 8-CTA thread-block cluster per (unit, row). The
//    histogram gives the bin b1 of the K-th largest key. Each warp of a CTA
//    owns a run of 32-key groups and reads only the groups whose largest key
//    reaches b1; it counts the keys above b1, pushes the candidates inside b1
//    to every CTA of the cluster through distributed shared memory, and keeps
//    every key of bin >= b1 with its position in an ordered per-warp list.
//    Every CTA finds the exact threshold key T (and how many keys equal to T
//    are taken) by a local radix select over the candidates; if they do not
//    fit, refinement passes with cluster-summed histograms find T instead.
//    Each warp compacts its own list at the offset the counts before it give
//    (or, if a list overflowed, the CTA compacts from its whole range): keys
//    above T, and keys equal to T lowest position first.
#include <algorithm>
#include <cooperative_groups.h>
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int HIST1_BINS = 4096;         // top 12 bits of the ordered key
constexpr int SEL_CLUSTER = 8;
constexpr int SEL_THREADS = 512;
constexpr int SEL_WARPS = 16;           // SEL_THREADS / 32
constexpr int SEL_LIST_CAP = 2048;       // keys of bin >= b1 kept per CTA, in order
constexpr int SEL_WLIST = SEL_LIST_CAP / SEL_WARPS;   // per warp
constexpr int SEL_ROUND = 256;           // groups of 32 keys a warp screens per round (8 per lane)
constexpr int SEL_NLD = 4;               // 16-byte loads in flight per lane: 16 groups per warp
constexpr int SEL_ALL_CAP = 8192;        // candidates per cluster (fast path)
constexpr int SEL_PER_SRC = SEL_ALL_CAP / SEL_CLUSTER;   // candidates each CTA may push

constexpr int SEL_GROUP = 32;            // keys per group (one warp of the score epilogue)

struct TopkWs {
  uint32_t* hist;   // [U*R][4096]
  uint32_t* keys;   // [U*R][stride]
  uint32_t* gmax;   // [U*R][stride / 32]: largest key of each group of 32 positions
  uint8_t* tmaps;   // tensor-map slots of the score kernel's CTAs
  int64_t stride;
};

// Keys per (unit, row): whole groups, so that every group is one 128-byte line.
inline int64_t key_stride(int64_t max_len) { return (max_len + SEL_GROUP - 1) / SEL_GROUP * SEL_GROUP; }

inline size_t topk_hist_bytes(int32_t U, int32_t R) { return dsa_align((size_t)U * R * HIST1_BINS * 4, 256); }
inline size_t topk_keys_bytes(int32_t U, int32_t R, int64_t max_len) {
  return dsa_align((size_t)U * R * key_stride(max_len) * 4, 256);
}
inline size_t topk_gmax_bytes(int32_t U, int32_t R, int64_t max_len) {
  return dsa_align((size_t)U * R * (key_stride(max_len) / SEL_GROUP) * 4, 256);
}

inline TopkWs topk_ws(void* ws, int32_t U, int32_t R, int64_t max_len) {
  TopkWs w;
  char* b = static_cast<char*>(ws);
  w.hist = reinterpret_cast<uint32_t*>(b);
  w.keys = reinterpret_cast<uint32_t*>(b + topk_hist_bytes(U, R));
  w.gmax = reinterpret_cast<uint32_t*>(b + topk_hist_bytes(U, R) + topk_keys_bytes(U, R, max_len));
  w.stride = key_stride(max_len);
  w.tmaps = reinterpret_cast<uint8_t*>(w.gmax) + topk_gmax_bytes(U, R, max_len);
  return w;
}

// Order-preserving map float -> uint32 (larger float, larger key); -0 == +0.
__device__ __forceinline__ uint32_t ordered_key(float s) {
  uint32_t b = __float_as_uint(s == 0.0f ? 0.0f : s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ---------------------------------------------------------------------------
// Scores on the tensor cores. For a tile of 128 positions the 8 indexer heads
// of every query row are one small contraction:
//     D[p][8r + h] = sum_d keys[p][d] * q[r][h][d]       (M = 128, N = 8R, K = 64)
// issued as tcgen05.mma kind::f16 with bf16 operands and an fp32 accumulator
// in tensor memory. With the workloads' integer-grid values every product and
// partial sum is exactly representable in fp32, so the result equals the
// CUDA-core fp32 (and the fp64) dot products bit for bit. ReLU, head weights
// and the sum over heads follow on the CUDA cores, one thread per position.

constexpr int SCORE_EPI_THREADS = 128;   // epilogue warps 0-3: one position (TMEM lane) per thread
constexpr int SCORE_PRODUCER_WARP = 4;   // issues the key copies
constexpr int SCORE_MMA_WARP = 5;        // issues the MMAs, owns the tensor memory
constexpr int SCORE_THREADS = 192;
constexpr int SCORE_TILE = 128;          // positions per tile = MMA M
constexpr int SCORE_STAGE = SCORE_TILE * 128;   // 16 KB of bf16 keys
constexpr int SCORE_MAX_STAGES = 6;
// CTAs per SM: on an SM partition (fewer SMs than the device's) the stream
// of keys per SM is what bounds the kernel, and every CTA's stages add to
// the bytes in flight (5 CTAs: 375 vs 392 us for 2.15 GB on 104 SMs). On the
// whole device HBM bounds it at 4 already (333 us either way), and a fifth
// CTA only crowds out the gather copy that shares its SMs (0.90 vs 0.83 ms
// per step for the capacity batch in two session groups).
constexpr int SCORE_MAX_CTAS_PER_SM = 6;
constexpr int SCORE_FULL_DEVICE_CTAS_PER_SM = 4;
constexpr int SCORE_TMEM_PER_SM = 512;   // tensor-memory columns of an SM
// The shared histogram holds two 16-bit bin counts per 32-bit word. A CTA
// flushes it to the call's histogram at least every SCORE_FLUSH_TILES tiles
// of a unit (511 x 128 = 65,408 positions), so no count passes 65,535.
constexpr int SCORE_HIST_WORDS = HIST1_BINS / 2;
constexpr int SCORE_FLUSH_TILES = 511;

// N of the MMA: 8 heads per query row, padded to a multiple of 16.
__host__ __device__ inline int score_npad(int R) { return (8 * R + 15) / 16 * 16; }
// Tensor-memory columns of one accumulator (two per CTA).
__host__ __device__ inline int score_acc_cols(int R) { return score_npad(R) <= 32 ? 32 : 64; }

struct ScoreLayout {
  int nst;            // key stages (operand A of one tile each)
  size_t b_off;       // query operand B: nb buffers of npad rows x 128 B (one
                      // when every CTA stays within one unit, else two)
  size_t b_bytes;
  size_t hist_off;    // R x 2048 words (4096 16-bit bins)
  size_t bar_off;     // barriers (full and empty per stage, full and empty per
                      // accumulator), TMEM address, failure flag
  size_t bytes;
};

__host__ __device__ inline ScoreLayout score_layout(int R, int nst, int nb) {
  ScoreLayout l;
  l.nst = nst;
  l.b_off = (size_t)nst * SCORE_STAGE;
  l.b_bytes = dsa_align((size_t)score_npad(R) * 128, 1024);
  l.hist_off = l.b_off + (size_t)nb * l.b_bytes;
  l.bar_off = dsa_align(l.hist_off + (size_t)R * SCORE_HIST_WORDS * 4, 16);
  l.bytes = l.bar_off + (2 * SCORE_MAX_STAGES + 4) * 8 + 16;
  return l;
}

// The stage count and CTAs per SM for R query rows and nb operand-B
// buffers: as many CTAs per SM as shared and tensor memory allow, up to
// max_ctas (the bytes in flight per SM are the stages of all its CTAs, and a
// CTA's roles overlap only within one tile's chain), then as many stages as
// still fit.
inline void score_config(int R, int nb, int max_ctas, int* nst, int* per_sm) {
  constexpr size_t SM_BYTES = 228 * 1024;
  // dynamic bytes + alignment slack, static shared memory, the per-CTA reserve
  auto cta_bytes = [R, nb](int s) { return score_layout(R, s, nb).bytes + 1024 + 1024 + 1024; };
  const int tmem_cap = SCORE_TMEM_PER_SM / (2 * score_acc_cols(R));
  int c = (int)std::max<size_t>(1, std::min<size_t>(std::min(max_ctas, tmem_cap), SM_BYTES / cta_bytes(2)));
  int s = 2;
  while (s < SCORE_MAX_STAGES && (size_t)c * cta_bytes(s + 1) <= SM_BYTES) ++s;
  *nst = s;
  *per_sm = c;
}

// Per-unit tensor maps. The keys of a unit are a bf16 [L][64] tensor whose
// 128-position boxes a tiled TMA copy lands in shared memory already in the
// 128-byte-swizzled K-major layout of the MMA's operand A. The units' key
// pointers live in device memory, so the maps are made on the device: a
// template encoded on the host (128 B, passed as a kernel parameter) is
// copied into a CTA-private slot in the workspace, and tensormap.replace
// sets the unit's address and row count.
constexpr int SCORE_TMAP_SLOTS = 8;              // per CTA, reused cyclically by unit
static_assert(SCORE_TMAP_SLOTS > SCORE_MAX_STAGES, "a map slot outlives the copies in flight");
constexpr int SCORE_MAX_GRID = 1024;
constexpr size_t SCORE_TMAP_BYTES = (size_t)SCORE_MAX_GRID * SCORE_TMAP_SLOTS * 128;

__device__ __forceinline__ void tmap_set_unit(uint8_t* slot, const void* keys, int rows) {
  asm volatile("tensormap.replace.tile.global_address.global.b1024.b64 [%0], %1;" ::"l"(slot), "l"(keys) : "memory");
  asm volatile("tensormap.replace.tile.global_dim.global.b1024.b32 [%0], 1, %1;" ::"l"(slot), "r"(rows) : "memory");
  asm volatile("fence.proxy.tensormap::generic.release.gpu;" ::: "memory");
  asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(slot) : "memory");
}

// One 128 x 64 bf16 box (rows y .. y + 127; rows past the map's row count
// read as zeros) into shared memory, completion counted on `bar` (16 KB).
__device__ __forceinline__ void tma_tile(void* dst, const uint8_t* tmap, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(tc::smem_u32(dst)), "l"(tmap), "r"(0), "r"(y), "r"(tc::smem_u32(bar))
      : "memory");
}

// 8 consecutive fp32 TMEM columns of this thread's lane (no wait).
__device__ __forceinline__ void tmem_ld8_nowait(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

struct ScoreArgs {
  const dsa_unit* units;
  const uint16_t* q;
  const float* w;
  uint32_t* hist;
  uint32_t* okeys;
  uint32_t* gmax;
  int64_t stride;
  int64_t max_len;
  int tpu;              // tiles per unit
  int cpu;              // CTAs per unit (each CTA within one unit), or 0: flattened ranges
  int U;
  int R, K;
  int nst;
  uint32_t idesc;
  uint8_t* tmaps;       // [grid][SCORE_TMAP_SLOTS][128 B]
  int32_t* dev_err;
};

// Per CTA: a contiguous range of the flattened (unit, tile) space. Its valid
// tiles j = 0, 1, ... pass through three roles that meet only at mbarriers:
//   producer (warp 4)   one tiled TMA copy per tile into stage j % NST (the
//                       keys land swizzled, ready for the MMA), once the MMAs
//                       that read the stage's previous tile are done;
//   MMA (warp 5)        once tile j's keys have landed and accumulator j & 1
//                       is free, four tcgen05.mma into it; their completion
//                       frees the key stage and hands the accumulator on;
//   epilogue (warps 0-3, one position per thread) reads the accumulator,
//                       frees it, then ReLU, head weights, order-preserving
//                       key, warp-aggregated shared histogram and the largest
//                       key of each warp's 32 positions (for the select).
// No role waits for another except at these barriers, so the stream of a CTA
// is bounded by its copies in flight and the slowest role, not by the sum of
// a tile's steps. The query rows of the tile's unit sit in operand-B buffer
// (unit change count & 1); the MMA warp writes a new unit's rows once every
// MMA it issued before is done.
__global__ void __launch_bounds__(SCORE_THREADS) k_dsa_score(const __grid_constant__ CUtensorMap tmpl, ScoreArgs a) {
  extern __shared__ __align__(1024) uint8_t sm_raw[];
  // the swizzled operand layouts need a 1024-byte aligned base
  uint8_t* sm = sm_raw + ((1024u - (tc::smem_u32(sm_raw) & 1023u)) & 1023u);
  const int R = a.R, NST = a.nst;
  if (NST < 2 || NST > SCORE_MAX_STAGES) return;   // the launch never passes these (barrier slots)
  const ScoreLayout lay = score_layout(R, NST, a.cpu > 0 ? 1 : 2);
  const int npad = score_npad(R);
  const uint32_t acols = (uint32_t)score_acc_cols(R);
  uint32_t* hs = reinterpret_cast<uint32_t*>(sm + lay.hist_off);
  uint64_t* full = reinterpret_cast<uint64_t*>(sm + lay.bar_off);   // [NST] keys landed
  uint64_t* empty = full + SCORE_MAX_STAGES;                        // [NST] stage read by its MMAs
  uint64_t* acc_full = empty + SCORE_MAX_STAGES;                    // [2] accumulator written
  uint64_t* acc_empty = acc_full + 2;                               // [2] accumulator read
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* s_fail = reinterpret_cast<int*>(s_tmem + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // this CTA's tiles: [f0, f1) of the flattened (unit, tile) space. With
  // a.cpu CTAs per unit every range lies inside one unit (one query operand,
  // one histogram flush); otherwise the flattened space is cut evenly.
  const long long total = (long long)a.U * a.tpu;
  long long f0, f1;
  if (a.cpu > 0) {
    const int uu = blockIdx.x / a.cpu, sub = blockIdx.x % a.cpu;
    const int per = (a.tpu + a.cpu - 1) / a.cpu;
    f0 = (long long)uu * a.tpu + min(sub * per, a.tpu);
    f1 = (long long)uu * a.tpu + min(sub * per + per, a.tpu);
  } else {
    const long long per = (total + gridDim.x - 1) / gridDim.x;
    f0 = (long long)blockIdx.x * per;
    f1 = min(f0 + per, total);
  }
  if (f0 >= f1) return;
  const int u0 = (int)(f0 / a.tpu);
  const int t0 = (int)(f0 - (long long)u0 * a.tpu);
  const int ntiles = (int)(f1 - f0);

  constexpr int UCACHE = 8;
  __shared__ int s_ntv[UCACHE];               // valid tiles of the unit (0 if L <= K)
  __shared__ int s_len[UCACHE];
  __shared__ const uint16_t* s_keys[UCACHE];
  for (int i = tid; i < R * SCORE_HIST_WORDS; i += SCORE_THREADS) hs[i] = 0;
  uint8_t* my_tmaps = a.tmaps + (size_t)blockIdx.x * SCORE_TMAP_SLOTS * 128;
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int c = 0; c < 2; ++c) {
      tc::mbar_init(&acc_full[c], 1);
      tc::mbar_init(&acc_empty[c], SCORE_EPI_THREADS / 32);   // one arrival per epilogue warp
    }
    *s_fail = 0;
    tc::fence_mbar_init();
  }
  if (warp == SCORE_MMA_WARP) tc::tmem_alloc(s_tmem, 2 * acols);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;
  pdl_wait();
  // every slot starts as a copy of the template (8 x 16 B each)
  for (int i = tid; i < SCORE_TMAP_SLOTS * 8; i += SCORE_THREADS)
    reinterpret_cast<uint4*>(my_tmaps)[i] = reinterpret_cast<const uint4*>(&tmpl)[i & 7];
  if (tid < UCACHE) {
    const int u = u0 + tid;
    s_ntv[tid] = 0;
    if (u < a.U && (long long)(u - u0) * a.tpu <= (long long)t0 + ntiles) {
      const int64_t L = min(a.units[u].state[DSA_ST_LEN], a.max_len);
      const bool ok = unit_aligned(a.units[u]);
      s_len[tid] = (int)L;
      s_keys[tid] = a.units[u].keys;
      s_ntv[tid] = (L > a.K && ok) ? (int)((L + SCORE_TILE - 1) / SCORE_TILE) : 0;
      if (!ok) dsa_flag(a.dev_err, DSA_DEVERR_BOUNDS);
    }
  }
  __syncthreads();     // the map slots hold the template; the unit cache is filled

  auto tile_of = [&](int k, int& u, int& t) {
    int tt = t0 + k;
    u = u0;
    while (tt >= a.tpu) {
      tt -= a.tpu;
      ++u;
    }
    t = tt;
  };
  auto unit_len = [&](int u) -> int {
    return u - u0 < UCACHE ? s_len[u - u0] : (int)min(a.units[u].state[DSA_ST_LEN], a.max_len);
  };
  auto unit_keys = [&](int u) -> const uint16_t* {
    return u - u0 < UCACHE ? s_keys[u - u0] : a.units[u].keys;
  };
  auto valid = [&](int u, int t) -> bool {
    const int i = u - u0;
    int ntv;
    if (i < UCACHE) {
      ntv = s_ntv[i];
    } else {
      const int L = unit_len(u);
      ntv = (L > a.K && unit_aligned(a.units[u])) ? (L + SCORE_TILE - 1) / SCORE_TILE : 0;
    }
    return t < ntv;
  };
  auto next_valid = [&](int k) -> int {
    for (; k < ntiles; ++k) {
      int u, t;
      tile_of(k, u, t);
      if (valid(u, t)) return k;
    }
    return ntiles;
  };
  // Bounded wait of one lane. A lane whose wait runs out flags the call and
  // the CTA; every other wait then gives up too, so all roles leave their
  // loops (this does not happen in normal runs).
  volatile int* vfail = s_fail;
  auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    const long long c0 = clock64();
    while (!tc::mbar_try_wait(bar, parity)) {
      if (*vfail) return false;
      if (clock64() - c0 > (1LL << 32)) {
        atomicOr(s_fail, 1);
        dsa_flag(a.dev_err, DSA_DEVERR_TIMEOUT);
        return false;
      }
    }
    return true;
  };
  // lane 0 waits, the warp follows its verdict
  auto warp_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
    bool ok = true;
    if (lane == 0) ok = wait(bar, parity);
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  };

  long long issued = 0;     // producer: copies issued
  long long last_mma = -1;  // MMA warp: the last tile whose MMAs were issued
  int hist_u = -1;          // epilogue: unit whose counts the shared histogram holds
  auto flush_hist = [&](int u) {
    uint32_t* gh = a.hist + (size_t)u * R * HIST1_BINS;
    for (int i = tid; i < R * SCORE_HIST_WORDS; i += SCORE_EPI_THREADS) {
      const uint32_t c = hs[i];
      if (c) {
        const int r = i / SCORE_HIST_WORDS;
        uint32_t* g = gh + (size_t)r * HIST1_BINS + 2 * (i - r * SCORE_HIST_WORDS);
        if (c & 0xFFFFu) atomicAdd(g, c & 0xFFFFu);
        if (c >> 16) atomicAdd(g + 1, c >> 16);
        hs[i] = 0;
      }
    }
  };

  if (warp == SCORE_PRODUCER_WARP) {
    // ---- producer. A unit's tensor map is made when its first tile is
    // issued, in the next slot in turn: every unit issued has at least one
    // tile, so a slot is rewritten only SCORE_TMAP_SLOTS units (and as many
    // tiles, more than the NST copies in flight) after its last use.
    // Stage s = j % NST and the parity of its use j / NST advance with j
    // (no integer division in the loop).
    int tmap_u = -1, tmap_n = -1;
    int s = 0;
    uint32_t use_par = 0;
    long long j = 0;
    for (int k = next_valid(0); k < ntiles; k = next_valid(k + 1), ++j) {
      if (j >= NST && !warp_wait(&empty[s], use_par ^ 1u)) break;   // the stage's previous use is read
      if (lane == 0) {
        int u, t;
        tile_of(k, u, t);
        if (u != tmap_u) {
          tmap_u = u;
          ++tmap_n;
          tmap_set_unit(my_tmaps + (size_t)(tmap_n & (SCORE_TMAP_SLOTS - 1)) * 128, unit_keys(u), unit_len(u));
        }
        tc::mbar_arrive_expect_tx(&full[s], (uint32_t)SCORE_STAGE);
        tma_tile(sm + s * SCORE_STAGE, my_tmaps + (size_t)(tmap_n & (SCORE_TMAP_SLOTS - 1)) * 128,
                 t * SCORE_TILE, &full[s]);
      }
      __syncwarp();
      issued = j + 1;
      if (++s == NST) {
        s = 0;
        use_par ^= 1u;
      }
    }
  } else if (warp == SCORE_MMA_WARP) {
    // ---- MMA issue
    int mma_u = -1, bsel = 1;
    int s = 0;
    uint32_t use_par = 0;     // parity of stage s's use j / NST
    long long j = 0;
    for (int k = next_valid(0); k < ntiles; k = next_valid(k + 1), ++j) {
      int u, t;
      tile_of(k, u, t);
      if (u != mma_u) {
        // new unit: its query rows into the other B buffer, once every MMA
        // issued so far (the last reader of that buffer among them) is done
        if (j > 0 && !warp_wait(&acc_full[(j - 1) & 1], (uint32_t)(((j - 1) >> 1) & 1))) break;
        mma_u = u;
        bsel ^= 1;
        uint8_t* sB = sm + lay.b_off + bsel * lay.b_bytes;
        const uint16_t* qu = a.q + (size_t)u * R * 512;
        for (int i = lane; i < npad * 8; i += 32) {
          const int row = i >> 3, c = i & 7;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (row < 8 * R) v = *reinterpret_cast<const uint4*>(qu + (size_t)row * 64 + 8 * c);
          *reinterpret_cast<uint4*>(sB + (row >> 3) * 1024 + (row & 7) * 128 + ((c ^ (row & 7)) << 4)) = v;
        }
        tc::fence_async_shared();
        __syncwarp();
      }
      const int acc = (int)(j & 1);
      bool ok = true;
      if (lane == 0) {
        ok = wait(&full[s], use_par);
        if (ok && j >= 2) ok = wait(&acc_empty[acc], (uint32_t)(((j >> 1) - 1) & 1));
        if (ok) {
          tc::fence_after_sync();
          const uint32_t aa = tc::smem_u32(sm + s * SCORE_STAGE);
          const uint32_t bb = tc::smem_u32(sm + lay.b_off + bsel * lay.b_bytes);
          const uint32_t d = tmem + (uint32_t)acc * acols;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            tc::mma_f16(d, tc::sdesc_sw128(aa + kk * 32, 16, 1024), tc::sdesc_sw128(bb + kk * 32, 16, 1024),
                        a.idesc, kk > 0);
          tc::mma_commit(&empty[s]);
          tc::mma_commit(&acc_full[acc]);
          last_mma = j;
        }
      }
      if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      if (++s == NST) {
        s = 0;
        use_par ^= 1u;
      }
    }
  } else {
    // ---- epilogue. A warp whose wait gave up keeps walking the tiles
    // without touching them, so that every epilogue thread meets the same
    // histogram barriers.
    bool dead = false;
    int since = 0;            // tiles counted into the shared histogram since its last flush
    long long j = 0;
    for (int k = next_valid(0); k < ntiles; k = next_valid(k + 1), ++j) {
      int u, t;
      tile_of(k, u, t);
      if (u != hist_u || since == SCORE_FLUSH_TILES) {
        // the histogram moves to a new unit, or its 16-bit counts could
        // overflow with one more tile: all counts so far are in (barrier),
        // each thread flushes and clears its own words, and the second
        // barrier keeps new counts out until then
        if (hist_u >= 0) {
          asm volatile("bar.sync 1, %0;" ::"r"(SCORE_EPI_THREADS) : "memory");
          flush_hist(hist_u);
          asm volatile("bar.sync 1, %0;" ::"r"(SCORE_EPI_THREADS) : "memory");
        }
        hist_u = u;
        since = 0;
      }
      ++since;
      const int acc = (int)(j & 1);
      if (!dead) dead = !warp_wait(&acc_full[acc], (uint32_t)((j >> 1) & 1));
      if (dead) continue;
      tc::fence_after_sync();
      const int n = min(SCORE_TILE, unit_len(u) - t * SCORE_TILE);
      const float* wu = a.w + (size_t)u * R * 8;
      const int p = tid;
      for (int r = 0; r < R; ++r) {
        uint32_t d[8];
        tmem_ld8_nowait(tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)acc * acols + 8 * r, d);
        tmem_ld_wait();
        if (r == R - 1) {
          // the accumulator is read: the MMA two tiles on may overwrite it
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(&acc_empty[acc]);
        }
        uint32_t key = 0u;   // positions past the history count as the smallest key
        if (p < n) {
          float sc = 0.f;
#pragma unroll
          for (int h = 0; h < 8; ++h) sc = fmaf(__ldg(wu + r * 8 + h), fmaxf(__uint_as_float(d[h]), 0.f), sc);
          key = ordered_key(sc);
          a.okeys[((size_t)u * R + r) * a.stride + (size_t)t * SCORE_TILE + p] = key;
          const uint32_t bin = key >> 20;
          const unsigned amask = __activemask();
          const unsigned peers = __match_any_sync(amask, bin);
          if (lane == __ffs(peers) - 1)
            atomicAdd(&hs[r * SCORE_HIST_WORDS + (bin >> 1)], (uint32_t)__popc(peers) << (16 * (bin & 1)));
        }
        // the warp's 32 positions form one group: its largest key lets the
        // selection skip groups that hold no key of the threshold bin. A
        // row holds stride / 32 groups; the last tile's groups past it
        // (positions >= max_len only) have no slot and are not written.
        const uint32_t gk = __reduce_max_sync(0xffffffffu, key);
        const int64_t gi = (int64_t)t * (SCORE_TILE / SEL_GROUP) + warp;
        if (lane == 0 && gi < a.stride / SEL_GROUP) a.gmax[((size_t)u * R + r) * (a.stride / SEL_GROUP) + gi] = gk;
      }
    }
    if (hist_u >= 0) {
      asm volatile("bar.sync 1, %0;" ::"r"(SCORE_EPI_THREADS) : "memory");
      flush_hist(hist_u);
    }
  }

  tc::fence_before_sync();
  __syncthreads();     // every role has left its loop
  tc::fence_after_sync();
  if (*vfail) {
    // A wait gave up: the call's selection is void. Nothing may land after
    // the CTA is gone: the MMAs and copies still in flight get one more
    // bounded wait each.
    if (warp == SCORE_MMA_WARP && lane == 0 && last_mma >= 0)
      tc::mbar_wait(&acc_full[last_mma & 1], (uint32_t)((last_mma >> 1) & 1));
    if (warp == SCORE_PRODUCER_WARP && lane == 0) {
      for (int s = 0; s < NST && s < issued; ++s) {
        const long long last = s + (issued - 1 - s) / NST * NST;   // the stage's last copy
        tc::mbar_wait(&full[s], (uint32_t)((last / NST) & 1));
      }
    }
  }
  if (warp == SCORE_MMA_WARP) {
    __syncwarp();
    tc::tmem_dealloc(tmem, 2 * acols);
  }
}

// Among `nb` histogram bins (held by threads 0..nb-1, thread t <-> bin
// nb-1-t, i.e. highest bin first), find the bin where the count of keys
// from the top reaches `need`. Returns the bin and the count strictly above it.
template <int NT>
__device__ __forceinline__ void find_digit(const uint32_t* h, int nb, int need, int* tmp,
                                           int* s_bin, int* s_above) {
  const int t = threadIdx.x;
  const int c = t < nb ? (int)h[nb - 1 - t] : 0;
  const int inc = block_inclusive_scan<NT>(c, tmp);
  const int exc = inc - c;
  if (t < nb && exc < need && need <= inc) {
    *s_bin = nb - 1 - t;
    *s_above = exc;
  }
  __syncthreads();
}

// Like find_digit, for up to 8 * NT bins: thread t sums the bins
// [nb - per*(t+1), nb - per*t) and scans them highest first.
template <int NT>
__device__ __forceinline__ void find_digit_wide(const uint32_t* h, int nb, int need, int* tmp,
                                                int* s_bin, int* s_above) {
  const int per = (nb + NT - 1) / NT;
  const int t = threadIdx.x;
  const int hi = nb - 1 - per * t;
  int c = 0;
  for (int i = 0; i < per; ++i)
    if (hi - i >= 0) c += (int)h[hi - i];
  const int inc = block_inclusive_scan<NT>(c, tmp);
  int exc = inc - c;
  if (c > 0 && exc < need && need <= inc) {
    for (int i = 0; i < per; ++i) {
      const int cb = hi - i >= 0 ? (int)h[hi - i] : 0;
      if (exc + cb >= need) {
        *s_bin = hi - i;
        *s_above = exc;
        break;
      }
      exc += cb;
    }
  }
  __syncthreads();
}

struct SelShared {
  uint32_t hl[2][256];
  uint32_t hg[256];
  int tmp[32];
  int bin, above;
  int ncand;
  int wcnt[SEL_WARPS];        // entries of each warp's list (above SEL_WLIST: it overflowed)
  int wgt[SEL_WARPS];         // keys of each warp's range above bin b1
  int wg[SEL_WARPS], we[SEL_WARPS];   // entries of each warp's list above / at the threshold key
  int csum[2];                // this CTA's candidates above / at the threshold key
  int srcn[SEL_CLUSTER];      // candidates pushed here by each CTA (-1: it overflowed)
  long long rcnt[SEL_CLUSTER][2];   // (gt, eq) of each CTA, read once for the prefix
  long long cnt[2];           // this CTA's (gt, eq) counts
};
// Shared memory after SelShared (each part 128-byte aligned): the 4096-bin
// radix histogram, the per-warp ordered lists (positions, keys), the
// candidates of the whole cluster.
constexpr size_t SEL_H_OFF = (sizeof(SelShared) + 127) / 128 * 128;
constexpr size_t SEL_LIST_OFF = SEL_H_OFF + (size_t)HIST1_BINS * 4;
constexpr size_t SEL_ALLC_OFF = SEL_LIST_OFF + (size_t)SEL_LIST_CAP * 8;
constexpr size_t SEL_GL_OFF = SEL_ALLC_OFF + (size_t)SEL_ALL_CAP * 4;
constexpr size_t SEL_SMEM = SEL_GL_OFF + (size_t)SEL_WARPS * SEL_ROUND * 4;
static_assert(SEL_WARPS * 32 == SEL_THREADS, "one list per warp");

__global__ void __cluster_dims__(SEL_CLUSTER, 1, 1) __launch_bounds__(SEL_THREADS, 2)
k_topk_select(const dsa_unit* __restrict__ units, int R, int K, uint32_t* __restrict__ hist,
              const uint32_t* __restrict__ okeys, const uint32_t* __restrict__ gmax, int64_t stride, int32_t* __restrict__ topk_idx,
              int64_t max_len, int32_t* dev_err) {
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int ur = blockIdx.y;
  const int u = ur / R;
  pdl_wait();
  tc::fence_async_global();   // score keys are read by bulk copies below
  const int64_t Lu = units[u].state[DSA_ST_LEN];
  const int64_t L = min(Lu, max_len);
  if (Lu > max_len && crank == 0 && threadIdx.x == 0) dsa_flag(dev_err, DSA_DEVERR_BOUNDS);
  int32_t* out = topk_idx + (size_t)ur * K;

  if (L <= K) {  // every position is selected; no cluster communication
    for (int j = crank * SEL_THREADS + threadIdx.x; j < K; j += SEL_CLUSTER * SEL_THREADS)
      out[j] = j < L ? j : -1;
    return;
  }

  // every CTA of the cluster must be running before any remote shared store:
  // arrive now, wait just before the first one
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  extern __shared__ __align__(128) uint8_t smem_sel[];
  SelShared* S = reinterpret_cast<SelShared*>(smem_sel);
  uint32_t* h1 = reinterpret_cast<uint32_t*>(smem_sel + SEL_H_OFF);           // [4096]
  int32_t* lpos = reinterpret_cast<int32_t*>(smem_sel + SEL_LIST_OFF);        // [SEL_LIST_CAP]
  uint32_t* lkey = reinterpret_cast<uint32_t*>(lpos + SEL_LIST_CAP);          // [SEL_LIST_CAP]
  uint32_t* allc = reinterpret_cast<uint32_t*>(smem_sel + SEL_ALLC_OFF);      // [SEL_ALL_CAP]
  const int tid = threadIdx.x;
  // this CTA's key range: whole groups of 32 keys (a trailing range may be empty)
  const int64_t chunk = ((L + SEL_CLUSTER - 1) / SEL_CLUSTER + SEL_GROUP - 1) / SEL_GROUP * SEL_GROUP;
  const int64_t beg = min((int64_t)crank * chunk, L);
  const int64_t end = min(beg + chunk, L);
  const uint32_t* kk = okeys + (size_t)ur * stride;
  if (tid == 0) {
    S->bin = 0;
    S->above = 0;
    S->ncand = 0;
  }

  // Warp w owns a contiguous run of groups of 32 positions; the largest
  // key of each group of its first round is loaded now (8 per lane, all in
  // flight) and lands while the histogram is scanned.
  const int warp = tid >> 5, lane = tid & 31;
  // (positions and group indices of one unit fit in 32 bits: L < 2^31)
  const int begi = (int)beg, endi = (int)end;
  const int gr0 = begi / SEL_GROUP, gr1 = (endi + SEL_GROUP - 1) / SEL_GROUP;   // beg: whole groups
  const int gpw = (gr1 - gr0 + SEL_WARPS - 1) / SEL_WARPS;
  const int wg0 = min(gr0 + warp * gpw, gr1), wg1 = min(wg0 + gpw, gr1);
  const uint32_t* gm = gmax + (size_t)ur * (stride / SEL_GROUP);
  uint32_t gmr[SEL_ROUND / 32];
  auto load_round = [&](int rb) {
#pragma unroll
    for (int j = 0; j < SEL_ROUND / 32; ++j) {
      const int gi = rb + 32 * j + lane;
      gmr[j] = gi < wg1 ? __ldcg(gm + gi) : 0u;
    }
  };
  load_round(wg0);

  // ---- level 1: top 12 bits from the global histogram (read in place)
  uint32_t* gh = hist + (size_t)ur * HIST1_BINS;
  find_digit_wide<SEL_THREADS>(gh, HIST1_BINS, K, S->tmp, &S->bin, &S->above);
  const uint32_t b1 = (uint32_t)S->bin;
  int need = K - S->above;

  // four keys [4q, 4q + 4) of the range from global memory (the fallbacks)
  auto key4 = [&](int64_t q) -> uint4 { return __ldcg(reinterpret_cast<const uint4*>(kk + 4 * q)); };
  // quads covering [beg, end); beg is a multiple of 4 whenever the range is
  // not empty (a trailing CTA whose range is empty gets no quads)
  const int64_t q0 = beg / 4, q1 = end > beg ? (end + 3) / 4 : q0;
  // visit every key of the range with coalesced 16-byte loads, UNR quads in
  // flight per thread
  auto for_keys = [&](auto&& f) {
    constexpr int UNR = 4;
    for (int64_t qb = q0 + tid; qb < q1; qb += (int64_t)UNR * SEL_THREADS) {
      uint4 v[UNR];
#pragma unroll
      for (int k = 0; k < UNR; ++k) {
        const int64_t q = qb + (int64_t)k * SEL_THREADS;
        v[k] = q < q1 ? key4(q) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < UNR; ++k) {
        const int64_t q = qb + (int64_t)k * SEL_THREADS;
        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (q < q1 && 4 * q + e < end) f(4 * q + e, w[e]);
      }
    }
  };

  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  // candidates go to region [crank] of every CTA's candidate buffer (the
  // remote addresses are formed where a candidate is pushed: it is rare, and
  // the pass keeps its registers for loads in flight)
  uint32_t* const own_region = allc + crank * SEL_PER_SRC;

  // ---- one pass over the range: count the keys above bin b1, push the
  //      candidates inside b1 to the cluster, and keep every key of bin >= b1
  //      with its position in an ordered list. Per round of 256 groups a
  //      warp lists, in order, the groups whose largest key reaches bin b1
  //      (the score kernel wrote these maxima; the other groups hold nothing
  //      of interest and are not read), then reads the listed groups 16 at
  //      a time, 8 lanes x 16 bytes per group. The warp's own list of keys
  //      is filled in position order, so the warps' lists concatenated in
  //      warp order are ordered; no block barrier is needed.
  const uint32_t kb1 = b1 << 20;     // smallest key of bin b1
  int32_t* wpos = lpos + warp * SEL_WLIST;
  uint32_t* wkey = lkey + warp * SEL_WLIST;
  int32_t* wgl = reinterpret_cast<int32_t*>(smem_sel + SEL_GL_OFF) + warp * SEL_ROUND;
  long long gt1 = 0;
  int wn = 0;          // entries of this warp's list so far (may pass SEL_WLIST)
  const unsigned lt_mask = (1u << lane) - 1u;
  const int seg = lane >> 3, sl = lane & 7;   // group slot of a load, 16-byte piece of the group
  for (int rb = wg0; rb < wg1; rb += SEL_ROUND) {
    if (rb != wg0) load_round(rb);
    int ng = 0;
#pragma unroll
    for (int j = 0; j < SEL_ROUND / 32; ++j) {
      const int gi = rb + 32 * j + lane;
      const bool hit = gi < wg1 && gmr[j] >= kb1;
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (hit) wgl[ng + __popc(m & lt_mask)] = gi - rb;
      ng += __popc(m);
    }
    __syncwarp();
    for (int e0 = 0; e0 < ng; e0 += 4 * SEL_NLD) {
      uint4 v[SEL_NLD];
#pragma unroll
      for (int k = 0; k < SEL_NLD; ++k) {
        const int e = e0 + 4 * k + seg;
        v[k] = e < ng ? __ldcg(reinterpret_cast<const uint4*>(kk + (size_t)(rb + wgl[e]) * SEL_GROUP) + sl)
                      : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int k = 0; k < SEL_NLD; ++k) {
        if (e0 + 4 * k >= ng) break;   // warp-uniform
        const int e = e0 + 4 * k + seg;
        const int p0 = e < ng ? (rb + wgl[e]) * SEL_GROUP + 4 * sl : -1;
        const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
        int c = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int pos = p0 + q;
          const bool in = p0 >= 0 && pos >= begi && pos < endi;
          gt1 += in && (w[q] >> 20) > b1;
          c += in && w[q] >= kb1;
          if (in && (w[q] >> 20) == b1) {
            const int kc = atomicAdd(&S->ncand, 1);
            if (kc < SEL_PER_SRC) {
#pragma unroll
              for (int cc = 0; cc < SEL_CLUSTER; ++cc) cluster.map_shared_rank(own_region, cc)[kc] = w[q];
            }
          }
        }
        // lanes hold consecutive pieces of consecutive listed groups, so an
        // exclusive prefix over the lanes gives each taken key its place
        int inc = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        int o = wn + inc - c;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int pos = p0 + q;
          if (p0 >= 0 && pos >= begi && pos < endi && w[q] >= kb1) {
            if (o < SEL_WLIST) {
              wpos[o] = pos;
              wkey[o] = w[q];
            }
            ++o;
          }
        }
        wn += __shfl_sync(0xffffffffu, inc, 31);
      }
    }
    __syncwarp();   // the group list is rewritten by the next round
  }
  {
    const int gw = __reduce_add_sync(0xffffffffu, (int)gt1);
    if (lane == 0) {
      S->wcnt[warp] = wn;
      S->wgt[warp] = gw;
    }
    if (tid < 2) S->csum[tid] = 0;
  }
  __syncthreads();
  bool list_ok = true;
  int gt1_cta = 0;
  for (int i = 0; i < SEL_WARPS; ++i) {
    list_ok &= S->wcnt[i] <= SEL_WLIST;
    gt1_cta += S->wgt[i];
  }
  if (tid < SEL_CLUSTER)
    cluster.map_shared_rank(S, tid)->srcn[crank] = S->ncand > SEL_PER_SRC ? -1 : S->ncand;
  cluster.sync();
  if (crank == 0) {
    // every CTA read the global histogram before the barrier: clear it for the next call
    for (int i = tid; i < HIST1_BINS; i += SEL_THREADS) gh[i] = 0;
  }
  int total = 0, any_over = 0;
  for (int c = 0; c < SEL_CLUSTER; ++c) {
    const int nc = S->srcn[c];
    any_over |= nc < 0;
    total += max(nc, 0);
  }
  const bool fast = !any_over && total <= SEL_ALL_CAP;

  uint32_t T;
  int ties;
  long long gt_cta, eq_cta;
  if (fast) {
    // ---- every CTA holds all candidates (pushed into per-source regions):
    //      exact local radix select on bits 19..8 and 7..0
    for (int i = tid; i < HIST1_BINS; i += SEL_THREADS) h1[i] = 0;
    // the valid candidates, flattened: source c's are entries [off[c], off[c + 1])
    int off[SEL_CLUSTER + 1];
    off[0] = 0;
#pragma unroll
    for (int c = 0; c < SEL_CLUSTER; ++c) off[c + 1] = off[c] + S->srcn[c];
    auto cand = [&](int i) -> uint32_t {
      int c = 0;
#pragma unroll
      for (int cc = 1; cc < SEL_CLUSTER; ++cc) c += i >= off[cc];
      return allc[c * SEL_PER_SRC + (i - off[c])];
    };
    __syncthreads();
    const uint32_t p1 = b1 << 20;
    for (int i = tid; i < total; i += SEL_THREADS) {
      const uint32_t key = cand(i);
      if ((key & 0xFFF00000u) == p1) atomicAdd(&h1[(key >> 8) & 0xFFF], 1u);
    }
    __syncthreads();
    find_digit_wide<SEL_THREADS>(h1, HIST1_BINS, need, S->tmp, &S->bin, &S->above);
    need -= S->above;
    const uint32_t p2 = p1 | ((uint32_t)S->bin << 8);
    for (int i = tid; i < 256; i += SEL_THREADS) S->hg[i] = 0;
    __syncthreads();
    for (int i = tid; i < total; i += SEL_THREADS) {
      const uint32_t key = cand(i);
      if ((key & 0xFFFFFF00u) == p2) atomicAdd(&S->hg[key & 0xFF], 1u);
    }
    __syncthreads();
    find_digit<SEL_THREADS>(S->hg, 256, need, S->tmp, &S->bin, &S->above);
    need -= S->above;
    T = p2 | (uint32_t)S->bin;
    ties = need;
    // this CTA's counts from its own candidates
    const int nc = S->srcn[crank];
    const uint32_t* own = allc + crank * SEL_PER_SRC;
    int g = 0, e = 0;
    for (int i = tid; i < nc; i += SEL_THREADS) {
      g += own[i] > T;
      e += own[i] == T;
    }
    g = __reduce_add_sync(0xffffffffu, g);
    e = __reduce_add_sync(0xffffffffu, e);
    if (lane == 0 && (g | e)) {
      atomicAdd(&S->csum[0], g);
      atomicAdd(&S->csum[1], e);
    }
    __syncthreads();
    gt_cta = (long long)gt1_cta + S->csum[0];
    eq_cta = S->csum[1];
  } else {
    // ---- refinement passes with cluster-summed histograms (8, 8, 4 bits)
    long long local_gt = gt1_cta;
    long long local_eq = 0;
    uint32_t prefix = b1 << 20, mask = 0xFFF00000u;
    const int shifts[3] = {12, 4, 0};
    const int nbins[3] = {256, 256, 16};
    for (int lvl = 0; lvl < 3; ++lvl) {
      uint32_t* hl = S->hl[lvl & 1];
      for (int i = tid; i < 256; i += SEL_THREADS) hl[i] = 0;
      __syncthreads();
      const int sh = shifts[lvl];
      const uint32_t dm = (uint32_t)nbins[lvl] - 1;
      for_keys([&](int64_t, uint32_t key) {
        if ((key & mask) == prefix) atomicAdd(&hl[(key >> sh) & dm], 1u);
      });
      __syncthreads();
      cluster.sync();
      for (int i = tid; i < nbins[lvl]; i += SEL_THREADS) {
        uint32_t s = 0;
        for (int c = 0; c < SEL_CLUSTER; ++c) s += cluster.map_shared_rank(hl, c)[i];
        S->hg[i] = s;
      }
      __syncthreads();
      find_digit<SEL_THREADS>(S->hg, nbins[lvl], need, S->tmp, &S->bin, &S->above);
      const uint32_t b = (uint32_t)S->bin;
      need -= S->above;
      {
        const int c = (tid < nbins[lvl] && (uint32_t)tid > b) ? (int)hl[tid] : 0;
        int tot;
        block_inclusive_scan<SEL_THREADS>(c, S->tmp, &tot);
        local_gt += tot;
        if (lvl == 2) local_eq = hl[b];
      }
      prefix |= b << sh;
      mask |= dm << sh;
    }
    T = prefix;
    ties = need;
    gt_cta = local_gt;
    eq_cta = local_eq;
  }
  if (tid == 0) {
    S->cnt[0] = gt_cta;
    S->cnt[1] = eq_cta;
  }
  __syncthreads();
  cluster.sync();
  if (tid < SEL_CLUSTER) {   // one round of remote loads
    const SelShared* rs = cluster.map_shared_rank(S, tid);
    S->rcnt[tid][0] = rs->cnt[0];
    S->rcnt[tid][1] = rs->cnt[1];
  }
  __syncthreads();
  long long eq_before = 0, sel_before = 0;
  for (int c = 0; c < crank; ++c) {
    const long long g = S->rcnt[c][0], e = S->rcnt[c][1];
    long long take = (long long)ties - eq_before;
    take = take < 0 ? 0 : (take > e ? e : take);
    sel_before += g + take;
    eq_before += e;
  }
  // ---- ordered compaction: keys above T, and keys equal to T lowest position
  //      first, written at the CTA's offset. From the ordered list when it
  //      held every key of bin >= b1 (all selected keys are among them), else
  //      from the whole range. Per group of entries: thread t owns NPT
  //      consecutive entries; two block scans give its tie rank and offset.
  auto compact = [&](int64_t nent, auto&& entry) {
    constexpr int NPT = 8;
    long long run_eq = eq_before, run_sel = sel_before;
    for (int64_t gb = 0; gb < nent; gb += (int64_t)NPT * SEL_THREADS) {
      const int64_t e0 = gb + (int64_t)NPT * tid;
      int32_t pos[NPT];
      uint32_t key[NPT];
      int g = 0, e = 0;
#pragma unroll
      for (int k = 0; k < NPT; ++k) {
        entry(e0 + k, pos[k], key[k]);           // pos < 0: no entry
        g += pos[k] >= 0 && key[k] > T;
        e += pos[k] >= 0 && key[k] == T;
      }
      int etot, stot;
      const int einc = block_inclusive_scan<SEL_THREADS>(e, S->tmp, &etot);
      const long long estart = run_eq + einc - e;
      long long take = (long long)ties - estart;
      take = take < 0 ? 0 : (take > e ? e : take);
      const int sel = g + (int)take;
      const int sinc = block_inclusive_scan<SEL_THREADS>(sel, S->tmp, &stot);
      long long o = run_sel + sinc - sel;
      long long er = estart;
#pragma unroll
      for (int k = 0; k < NPT; ++k) {
        bool pick = pos[k] >= 0 && key[k] > T;
        if (pos[k] >= 0 && key[k] == T) {
          pick = er < ties;
          ++er;
        }
        if (pick) {
          if (o < K) out[o] = pos[k];
          ++o;
        }
      }
      run_eq += etot;
      run_sel += stot;
    }
  };
  if (list_ok) {
    // Every warp walks its own list (in position order; the warps' lists
    // follow each other in position order). Its place in the CTA's output
    // and its first tie rank come from the counts of the warps before it.
    const int nw = S->wcnt[warp];
    int g = 0, e = 0;
    for (int j = lane; j < nw; j += 32) {
      const uint32_t k = wkey[j];
      g += k > T;
      e += k == T;
    }
    g = __reduce_add_sync(0xffffffffu, g);
    e = __reduce_add_sync(0xffffffffu, e);
    if (lane == 0) {
      S->wg[warp] = g;
      S->we[warp] = e;
    }
    __syncthreads();
    long long eqb = eq_before, selb = sel_before;
    for (int i = 0; i < warp; ++i) {
      const long long ei = S->we[i];
      long long take = (long long)ties - eqb;
      take = take < 0 ? 0 : (take > ei ? ei : take);
      selb += S->wg[i] + take;
      eqb += ei;
    }
    for (int j0 = 0; j0 < nw; j0 += 32) {
      const int j = j0 + lane;
      const bool v = j < nw;
      const uint32_t k = v ? wkey[j] : 0u;
      const bool eq = v && k == T;
      const unsigned em = __ballot_sync(0xffffffffu, eq);
      const bool pick = (v && k > T) || (eq && eqb + __popc(em & lt_mask) < ties);
      const unsigned pm = __ballot_sync(0xffffffffu, pick);
      const long long o = selb + __popc(pm & lt_mask);
      if (pick && o < K) out[o] = wpos[j];
      selb += __popc(pm);
      eqb += __popc(em);
    }
  } else {
    const int64_t nq = q1 - q0;   // the whole range, 4 keys per quad from global memory
    compact(4 * nq, [&](int64_t i, int32_t& p, uint32_t& k) {
      const int64_t pp = 4 * q0 + i;
      const bool in = pp >= beg && pp < end;
      p = in ? (int32_t)pp : -1;
      k = in ? __ldcg(kk + pp) : 0u;
    });
  }
  cluster.sync();   // keep this CTA's shared memory alive for its peers
}

inline size_t select_smem() { return SEL_SMEM; }

DsaPerDevice g_setup;   // kernel attributes and SM count, per device

// The tensor-map template of the score kernel, per device: bf16 [rows][64],
// 128-byte rows, 64 x 128 boxes, 128-byte swizzle. It is encoded over a
// small array of this library (the kernels always replace the address and
// the row count before a copy).
static __device__ __align__(256) uint8_t g_tmap_dummy[SCORE_STAGE];
CUtensorMap g_tmpl[DSA_MAX_DEVICES];

int encode_template(int dev) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return DSA_ERR_CUDA;
  void* base = nullptr;
  if (cudaGetSymbolAddress(&base, g_tmap_dummy) != cudaSuccess) return DSA_ERR_CUDA;
  const cuuint64_t dims[2] = {64, SCORE_TILE};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {64, SCORE_TILE};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn)(
      &g_tmpl[dev], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr,
      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace

extern "C" size_t dsa_score_topk_workspace(int32_t U, int32_t R, int64_t max_len) {
  if (U < 1 || R < 1 || max_len < 0) return 0;
  return topk_hist_bytes(U, R) + topk_keys_bytes(U, R, max_len) + topk_gmax_bytes(U, R, max_len) +
         SCORE_TMAP_BYTES;
}

namespace {

// Argument checks shared by the scoring and selection entry points.
int check_score_args(const dsa_unit* units, int32_t U, int32_t R, int32_t K, int64_t max_len, const void* ws,
                     size_t ws_bytes) {
  if (!units) return DSA_ERR_ARG;
  if (U < 1 || U > 65535 || R < 1 || R > DSA_MAX_ROWS || max_len < 0) return DSA_ERR_ARG;
  if ((int64_t)U * R > 65535) return DSA_ERR_ARG;
  if (K < 1 || K > DSA_MAX_K) return DSA_ERR_SHAPE;
  if (!ws || ws_bytes < dsa_score_topk_workspace(U, R, max_len)) return DSA_ERR_WS;
  if (reinterpret_cast<uintptr_t>(ws) & 15u) return DSA_ERR_ARG;   // its keys are read by bulk copies
  return DSA_OK;
}

int score_setup(int* dev) {
  return dsa_device_setup(g_setup, dev, [](int d) {
    if (encode_template(d) != DSA_OK) return DSA_ERR_CUDA;
    size_t mx = 0;
    for (int r = 1; r <= DSA_MAX_ROWS; ++r) {
      for (int nb = 1; nb <= 2; ++nb) {
        for (int cap : {SCORE_FULL_DEVICE_CTAS_PER_SM, SCORE_MAX_CTAS_PER_SM}) {
          int nst = 2, per_sm = 1;
          score_config(r, nb, cap, &nst, &per_sm);
          mx = std::max(mx, score_layout(r, nst, nb).bytes + 1024);
        }
      }
    }
    DSA_CUDA_TRY(dsa_prefer_shared(k_dsa_score));
    DSA_CUDA_TRY(dsa_prefer_shared(k_topk_select));
    DSA_CUDA_TRY(cudaFuncSetAttribute(k_dsa_score, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mx));
    DSA_CUDA_TRY(cudaFuncSetAttribute(k_topk_select, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)select_smem()));
    return DSA_OK;
  });
}

}  // namespace

extern "C" int dsa_score(const dsa_unit* units, int32_t U, int32_t R, int32_t K, const uint16_t* q,
                         const float* w, int64_t max_len, void* ws, size_t ws_bytes, int32_t* dev_err,
                         void* stream) {
  if (!q || !w) return DSA_ERR_ARG;
  const int chk = check_score_args(units, U, R, K, max_len, ws, ws_bytes);
  if (chk != DSA_OK) return chk;
  if (reinterpret_cast<uintptr_t>(q) & 15u) return DSA_ERR_ARG;   // query rows are read as 16-byte vectors
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TopkWs tw = topk_ws(ws, U, R, max_len);
  int dev = 0;
  const int ok = score_setup(&dev);
  if (ok != DSA_OK) return ok;
  const int64_t tpu = (max_len + SCORE_TILE - 1) / SCORE_TILE;
  if (tpu == 0) return DSA_OK;
  if (tpu * U > 0x7fffffffLL) return DSA_ERR_ARG;
  // The persistent grid fills the SMs the stream may use: all of the
  // device's, or those of the SM partition the stream belongs to.
  const int num_sms = dsa_stream_sms(st, g_setup.num_sms[dev]);
  // one operand-B buffer when every CTA stays within one unit (the grid
  // holds at least one CTA per unit), else two
  const int cap = num_sms < g_setup.num_sms[dev] ? SCORE_MAX_CTAS_PER_SM : SCORE_FULL_DEVICE_CTAS_PER_SM;
  int nst = 2, per_sm = 1;
  score_config(R, 1, cap, &nst, &per_sm);
  int nb = 1;
  if (U > std::min<int64_t>((int64_t)per_sm * num_sms, SCORE_MAX_GRID)) {
    nb = 2;
    score_config(R, nb, cap, &nst, &per_sm);
  }
  ScoreArgs a;
  a.units = units;
  a.q = q;
  a.w = w;
  a.hist = tw.hist;
  a.okeys = tw.keys;
  a.gmax = tw.gmax;
  a.stride = tw.stride;
  a.max_len = max_len;
  a.tpu = (int)tpu;
  a.U = U;
  a.R = R;
  a.K = K;
  a.nst = nst;
  a.idesc = tc::idesc_bf16_f32(SCORE_TILE, score_npad(R));
  a.tmaps = tw.tmaps;
  a.dev_err = dev_err;
  const int64_t slots = std::min<int64_t>((int64_t)per_sm * num_sms, SCORE_MAX_GRID);
  int64_t grid;
  if (nb == 1) {
    // whole CTAs per unit
    a.cpu = (int)std::min<int64_t>(slots / U, tpu);
    grid = (int64_t)a.cpu * U;
  } else {
    a.cpu = 0;
    grid = std::min<int64_t>(tpu * U, slots);
  }
  return launch_pdl(k_dsa_score, dim3((unsigned)grid), dim3(SCORE_THREADS), score_layout(R, nst, nb).bytes + 1024,
                    st, g_tmpl[dev], a);
}

extern "C" int dsa_topk_select(const dsa_unit* units, int32_t U, int32_t R, int32_t K, int32_t* topk_idx,
                               int64_t max_len, void* ws, size_t ws_bytes, int32_t* dev_err, void* stream) {
  if (!topk_idx) return DSA_ERR_ARG;
  const int chk = check_score_args(units, U, R, K, max_len, ws, ws_bytes);
  if (chk != DSA_OK) return chk;
  TopkWs tw = topk_ws(ws, U, R, max_len);
  int dev = 0;
  const int ok = score_setup(&dev);
  if (ok != DSA_OK) return ok;
  return launch_pdl(k_topk_select, dim3(SEL_CLUSTER, U * R), dim3(SEL_THREADS), select_smem(),
                    static_cast<cudaStream_t>(stream), units, R, K, tw.hist, tw.keys, tw.gmax, tw.stride, topk_idx,
                    max_len, dev_err);
}

extern "C" int dsa_score_topk(const dsa_unit* units, int32_t U, int32_t R, int32_t K,
                              const uint16_t* q, const float* w, int32_t* topk_idx,
                              int64_t max_len, void* ws, size_t ws_bytes, int32_t* dev_err,
                              void* stream) {
  if (!topk_idx) return DSA_ERR_ARG;
  const int st = dsa_score(units, U, R, K, q, w, max_len, ws, ws_bytes, dev_err, stream);
  if (st != DSA_OK) return st;
  return dsa_topk_select(units, U, R, K, topk_idx, max_len, ws, ws_bytes, dev_err, stream);
}

// ---------------------------------------------------------------------------
// Selection reuse across layers: unit u takes the selection held in row
// src_of[u] of a compact buffer of the scored (source) units.

namespace {

__global__ void __launch_bounds__(256)
k_reuse_selection(int32_t* __restrict__ topk, const int32_t* __restrict__ src_topk, int Us, int R, int K,
                  const int32_t* __restrict__ src_of, int32_t* dev_err) {
  const int u = blockIdx.y;
  pdl_wait();
  const int s = src_of[u];
  if (s < 0 || s >= Us) {
    if (blockIdx.x == 0 && threadIdx.x == 0) dsa_flag(dev_err, DSA_DEVERR_BOUNDS);
    return;
  }
  const size_t n = (size_t)R * K;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    topk[(size_t)u * n + i] = src_topk[(size_t)s * n + i];
}

}  // namespace

extern "C" int dsa_reuse_selection(int32_t* topk_idx, const int32_t* src_topk, int32_t U, int32_t Us, int32_t R,
                                   int32_t K, const int32_t* src_of, int32_t* dev_err, void* stream) {
  if (!topk_idx || !src_topk || !src_of || U < 1 || U > 65535 || Us < 1 || R < 1 || R > DSA_MAX_ROWS)
    return DSA_ERR_ARG;
  if (K < 1 || K > DSA_MAX_K) return DSA_ERR_SHAPE;
  static DsaPerDevice pd;
  int dev = 0;
  const int ok = dsa_device_setup(pd, &dev, [](int) {
    DSA_CUDA_TRY(dsa_prefer_shared(k_reuse_selection));
    return DSA_OK;
  });
  if (ok != DSA_OK) return ok;
  const int bx = (int)std::min<int64_t>(((int64_t)R * K + 255) / 256, 64);
  return launch_pdl(k_reuse_selection, dim3(bx, U), dim3(256), 0, static_cast<cudaStream_t>(stream), topk_idx,
                    src_topk, Us, R, K, src_of, dev_err);
}

// ---------------------------------------------------------------------------
// dsa_score_topk_noalloc: the same scoring and selection for callers that may
// not allocate device memory. Its scratch (selection histograms and ordered
// score keys) lives in one fixed array compiled into this library.

namespace {

constexpr int64_t NOALLOC_MAX_UR = 16;          // units x query rows per call
constexpr int64_t NOALLOC_MAX_LEN = 65536;      // history positions per unit
constexpr size_t NOALLOC_HIST_BYTES = (size_t)NOALLOC_MAX_UR * HIST1_BINS * 4;   // 256 KiB
// histograms, ordered keys (4 MiB), group maxima (128 KiB), tensor-map slots
// (1 MiB); each part a multiple of 256 bytes at these limits
constexpr size_t NOALLOC_BYTES = NOALLOC_HIST_BYTES + (size_t)NOALLOC_MAX_UR * NOALLOC_MAX_LEN * 4 +
                                 (size_t)NOALLOC_MAX_UR * (NOALLOC_MAX_LEN / SEL_GROUP) * 4 + SCORE_TMAP_BYTES;
static __device__ __align__(256) uint8_t g_topk_scratch[NOALLOC_BYTES];

// Device address of g_topk_scratch, per device ordinal (looked up once, under
// a lock so that host threads making first calls at the same time agree).
std::atomic<void*> g_topk_scratch_addr[DSA_MAX_DEVICES];
std::mutex g_topk_scratch_mu;

}  // namespace

extern "C" int dsa_score_topk_noalloc(const dsa_unit* units, int32_t U, int32_t R, int32_t K,
                                      const uint16_t* q, const float* w, int32_t* topk_idx,
                                      int64_t max_len, int32_t* dev_err, void* stream) {
  if (!units || !q || !w || !topk_idx) return DSA_ERR_ARG;
  if (U < 1 || R < 1 || R > DSA_MAX_ROWS || max_len < 0) return DSA_ERR_ARG;
  if (K < 1 || K > DSA_MAX_K) return DSA_ERR_SHAPE;
  if ((int64_t)U * R > NOALLOC_MAX_UR || max_len > NOALLOC_MAX_LEN) return DSA_ERR_SCRATCH_LIMIT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= DSA_MAX_DEVICES) return DSA_ERR_CUDA;
  void* scratch = g_topk_scratch_addr[dev].load(std::memory_order_acquire);
  if (!scratch) {
    // First call on this device: host code cannot use the array's name as a
    // device address, so ask the runtime for it (the device must be current).
    std::lock_guard<std::mutex> lock(g_topk_scratch_mu);
    scratch = g_topk_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!scratch) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || !p) return DSA_ERR_CUDA;
      g_topk_scratch_addr[dev].store(p, std::memory_order_release);
      scratch = p;
    }
  }
  const size_t need = dsa_score_topk_workspace(U, R, max_len);
  if (need > NOALLOC_BYTES) return DSA_ERR_SCRATCH_LIMIT;
  // The array keeps whatever the previous call left; the histograms must
  // start at zero, so clear them (an interrupted earlier call may have left
  // counts behind).
  if (cudaMemsetAsync(scratch, 0, (size_t)U * R * HIST1_BINS * 4, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return DSA_ERR_CUDA;
  return dsa_score_topk(units, U, R, K, q, w, topk_idx, max_len, scratch, NOALLOC_BYTES, dev_err, stream);
}
