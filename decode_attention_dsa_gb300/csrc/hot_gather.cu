// A3: GPU-managed hot-cache gather.
//
// [P3] "From 1M total to 15+ x 1M: GLM-5.3 KV-cache offload", section
// "第三次决策：让 GPU 直接管理热缓存" (third decision: the GPU manages the hot
// cache): the selection stays on the GPU, the GPU looks up the hot slots, hits
// read VRAM and misses read the registered RAM mirror, forming the compact set
// attention uses. Section "GPU 管缓存也会犯错：跨 block 可见性与置换长扫描"
// (cross-block visibility and long replacement sweeps): slots filled in a
// round are hit sources only from the next round and duplicate misses read
// RAM (an early version let one block read a slot another block was still
// filling); slots in use are pinned; rows not yet written back are served by
// the recent ring; replacement is a ring that skips pinned slots (the
// reference-bit clock's long sweeps cost ~1 ms per gather).
//
// Two launches per call, each over all units:
//  1. k_assign    one 1024-thread CTA per unit: classification of every
//                 selected entry with the state as it is at call start and
//                 pins of the HOT slots (pin_epoch = call id) -- nothing is
//                 filled before a block barrier, so no entry can see a slot
//                 filled in this call and the visibility rule holds by
//                 construction -- then counts, the ascending list of
//                 distinct unmapped misses (first occurrence across rows found
//                 by binary search in the lower rows, rank by per-row prefix
//                 counts), the eligible slots in cyclic order from the hand
//                 (block scans over 1024-slot windows), and the map update.
//                 The parallel assignment reproduces the sequential rule
//                 "i-th miss takes the i-th eligible slot" exactly.
//  2. k_copy      one warp per 656-byte row: a fill reads the mirror row once
//                 (zero-copy over the host link) and writes the victim slot,
//                 the compact row of the position's first occurrence and the
//                 compact rows of its later occurrences in the other query
//                 rows (all RAM-class: they get the RAM bytes, never the slot
//                 being filled); every other entry copies from its source
//                 (slot / ring / mirror).
#include <algorithm>

#include "common.cuh"
#include "gather_internal.cuh"

namespace {

constexpr int ASSIGN_THREADS = 1024;
constexpr int COPY_THREADS = 256;
constexpr int COPY_WARPS = COPY_THREADS / 32;
// Blocks per SM of the row copies (grid-stride beyond). A small call is bound
// by the latency of its dependent loads and spreads over COPY_BLOCKS_PER_SM
// blocks per SM. From COPY_BW_ENTRIES selected entries per call on, the copies
// are bound by the host link, which one block per SM already keeps busy
// (the same copy time as four); the extra reads in flight would only queue at
// the link, and that queueing slows the HBM reads of a kernel running beside
// the copy (the next step's scoring, when steps are pipelined), measured
// 0.90 vs 1.02 ms per step on 32 units x Top-2048 with 1 vs 4 blocks per SM.
constexpr int COPY_BLOCKS_PER_SM = 4;
constexpr int64_t COPY_BW_ENTRIES = 65536;
// On an SM partition of its own (no kernel beside it to slow), the copy keeps
// as many reads in flight as its blocks allow: 8 blocks of 256 threads per SM.
constexpr int COPY_MAX_BLOCKS_PER_SM = 8;
// Between COPY_MID_ENTRIES and COPY_BW_ENTRIES the kernel decides itself: if
// the call's fills (rows read over the host link) reach COPY_BW_FILLS, only
// one block per SM copies (the rest leave at once); a call with that many
// selected entries but few misses stays latency-bound and keeps them all.
constexpr int64_t COPY_MID_ENTRIES = 16384;
constexpr int COPY_BW_FILLS = 16384;

// lower_bound of p in an ascending row whose tail is -1 padding (-1 = +inf).
__device__ __forceinline__ int row_lower_bound(const int32_t* row, int K, int32_t p) {
  int lo = 0, hi = K;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    const int32_t v = row[mid];
    if (v >= 0 && v < p) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Shared working set of k_assign for R*K entries: the selected rows (when
// they fit), classes, owner flags and per-row owner prefix counts.
constexpr int ASSIGN_TK_SMEM_MAX = 16384;   // entries whose rows are kept in shared memory

inline size_t assign_smem(int RK) {
  return (size_t)RK * (1 + 1 + 2) + (RK <= ASSIGN_TK_SMEM_MAX ? (size_t)RK * 4 : 0) + 64;
}

__global__ void __launch_bounds__(ASSIGN_THREADS)
k_assign(const dsa_unit* __restrict__ units, int R, int K, int round,
         const int32_t* __restrict__ topk_all, uint8_t* cls_all,
         int32_t* __restrict__ counters, GatherWs g, int32_t* dev_err) {
  __shared__ int s_tmp[32];
  __shared__ int s_cnt[4];
  extern __shared__ __align__(16) uint8_t asm_[];
  const int u = blockIdx.x;
  const int RK = R * K;
  const bool tk_in_smem = RK <= ASSIGN_TK_SMEM_MAX;
  int32_t* s_tk = reinterpret_cast<int32_t*>(asm_);                          // [RK] if it fits
  uint16_t* s_opc = reinterpret_cast<uint16_t*>(asm_ + (tk_in_smem ? (size_t)RK * 4 : 0));   // [RK]
  uint8_t* s_cl = reinterpret_cast<uint8_t*>(s_opc + RK);                      // [RK]
  uint8_t* s_fl = s_cl + RK;                                                   // [RK] owner flags
  if (threadIdx.x < 4) s_cnt[threadIdx.x] = 0;   // totals: HOT, RING, RAM, owners
  __syncthreads();
  pdl_wait();
  const dsa_unit& un = units[u];
  const int32_t epoch = (int32_t)(un.state[DSA_ST_EPOCH] + 1);
  if (round < 0) round = epoch - 1;
  // a unit whose arrays are misaligned, or a round below the unit's previous
  // one (it would break the visibility rule), is skipped: every entry PAD
  // (k_copy zeroes its compact row), no fill, state untouched
  const bool clock = un.policy == DSA_POLICY_CLOCK;
  const bool misaligned = !unit_aligned(un) || (clock && !un.ref) ||
                          (un.policy != DSA_POLICY_RING && !clock);   // (or an unknown policy)
  if (misaligned || (int64_t)round + 1 < un.state[DSA_ST_ROUND]) {
    if (threadIdx.x == 0) {
      dsa_flag(dev_err, misaligned ? DSA_DEVERR_BOUNDS : DSA_DEVERR_ROUND);
      g.nfill[u] = 0;
      for (int i = 0; i < 4; ++i) counters[(size_t)u * 4 + i] = 0;
    }
    for (int e = threadIdx.x; e < RK; e += ASSIGN_THREADS) {
      cls_all[(size_t)u * RK + e] = DSA_CLS_PAD;
      g.served[(size_t)u * RK + e] = 0;
      g.fill_of[(size_t)u * RK + e] = -1;
    }
    return;
  }
  const int32_t* gtopk = topk_all + (size_t)u * RK;
  const int32_t* tk = tk_in_smem ? s_tk : gtopk;
  uint8_t* cls = cls_all + (size_t)u * RK;
  int32_t* fill_pos = g.fill_pos + (size_t)u * RK;
  int32_t* fill_slot = g.fill_slot + (size_t)u * RK;
  int32_t* fill_entry = g.fill_entry + (size_t)u * RK;
  uint8_t* served = g.served + (size_t)u * RK;
  const int S = un.slots_n;
  const int64_t len = un.state[DSA_ST_LEN];
  const int64_t ram = un.state[DSA_ST_RAM];

  // 0. classify every entry with the state as it is now, pinning HOT slots
  //    (nothing is filled before the block barriers below, so no entry can see
  //    a slot filled in this call); flag RAM positions that hold no slot
  // batches of CB entries per thread: the three dependent lookups of an
  // entry (position -> slot -> fill round) are issued for the whole batch at
  // once, so a thread waits three memory latencies per batch, not per entry
  int hot = 0, ring = 0, rm = 0;
  constexpr int CB = 8;
  for (int e0 = threadIdx.x; e0 < RK; e0 += CB * ASSIGN_THREADS) {
    int32_t pv[CB], sv[CB], fv[CB];
#pragma unroll
    for (int b = 0; b < CB; ++b) {
      const int e = e0 + b * ASSIGN_THREADS;
      pv[b] = e < RK ? gtopk[e] : -1;
    }
#pragma unroll
    for (int b = 0; b < CB; ++b) {
      const int32_t p = pv[b];
      sv[b] = (p >= 0 && p < ram) ? un.pos_slot[p] : -1;
    }
#pragma unroll
    for (int b = 0; b < CB; ++b) fv[b] = (sv[b] >= 0 && sv[b] < S) ? un.fill_round[sv[b]] : 0;
#pragma unroll
    for (int b = 0; b < CB; ++b) {
      const int e = e0 + b * ASSIGN_THREADS;
      if (e >= RK) break;
      const int32_t p = pv[b];
      if (tk_in_smem) s_tk[e] = p;
      uint8_t c = DSA_CLS_PAD, unmapped = 0;
      if (p >= 0) {
        if (p >= len) {
          dsa_flag(dev_err, DSA_DEVERR_BOUNDS);
        } else if (p >= ram) {
          c = DSA_CLS_RING;
        } else {
          const int32_t sl = sv[b];
          if (sl >= 0 && sl < S && fv[b] < round) {
            c = DSA_CLS_HOT;
            un.pin_epoch[sl] = epoch;
            if (clock) un.ref[sl] = 1;        // a hit sets the reference bit
          } else {
            c = DSA_CLS_RAM;
            unmapped = sl < 0;
          }
        }
      }
      cls[e] = c;
      s_cl[e] = c;
      s_fl[e] = unmapped;
      hot += c == DSA_CLS_HOT;
      ring += c == DSA_CLS_RING;
      rm += c == DSA_CLS_RAM;
    }
  }
  {
    // per-warp totals, one shared atomic each
    hot = __reduce_add_sync(0xffffffffu, hot);
    ring = __reduce_add_sync(0xffffffffu, ring);
    rm = __reduce_add_sync(0xffffffffu, rm);
    if ((threadIdx.x & 31) == 0) {
      if (hot) atomicAdd(&s_cnt[0], hot);
      if (ring) atomicAdd(&s_cnt[1], ring);
      if (rm) atomicAdd(&s_cnt[2], rm);
    }
  }
  __syncthreads();   // s_tk, s_cl, s_fl and the totals are complete

  // 1. owners: the first occurrence (lowest query row) of an unmapped RAM
  //    position; per-row exclusive prefix counts of owners
  if (R > 1) {
    for (int e = threadIdx.x; e < RK; e += ASSIGN_THREADS) {
      if (!s_fl[e]) continue;
      const int r = e / K;
      const int32_t p = tk[e];
      for (int r2 = 0; r2 < r; ++r2) {
        const int32_t* o = tk + (size_t)r2 * K;
        const int lb = row_lower_bound(o, K, p);
        if (lb < K && o[lb] == p) {
          s_fl[e] = 0;
          break;
        }
      }
    }
    __syncthreads();
  }
  const int per = (K + ASSIGN_THREADS - 1) / ASSIGN_THREADS;   // contiguous run per thread
  for (int r = 0; r < R; ++r) {
    const int j0 = min(threadIdx.x * per, K), j1 = min(j0 + per, K);
    int own = 0;
    for (int j = j0; j < j1; ++j) own += s_fl[r * K + j];
    const int inc = block_inclusive_scan<ASSIGN_THREADS>(own, s_tmp);
    int run = inc - own;
    for (int j = j0; j < j1; ++j) {
      s_opc[r * K + j] = (uint16_t)run;
      run += s_fl[r * K + j];
    }
  }
  __syncthreads();

  // 2. rank of each owner among all owners (ascending position)
  int nM_local = 0;
  for (int e = threadIdx.x; e < RK; e += ASSIGN_THREADS) {
    if (!s_fl[e]) continue;
    const int r = e / K;
    const int32_t p = tk[e];
    int rank = s_opc[e];
    for (int r2 = 0; r2 < R; ++r2) {
      if (r2 == r) continue;
      const int32_t* o = tk + (size_t)r2 * K;
      const int lb = row_lower_bound(o, K, p);
      rank += lb < K ? s_opc[r2 * K + lb] : (s_opc[r2 * K + K - 1] + s_fl[r2 * K + K - 1]);
    }
    if (rank < RK) {
      fill_pos[rank] = p;
      fill_entry[rank] = e;
      int32_t* dp = g.dup + ((size_t)u * RK + rank) * (DSA_MAX_ROWS - 1);
      for (int k = 0; k < R - 1; ++k) dp[k] = -1;     // only the first R - 1 are ever read
      int nd = 0;
      for (int r2 = r + 1; r2 < R; ++r2) {
        const int32_t* o = tk + (size_t)r2 * K;
        const int lb = row_lower_bound(o, K, p);
        if (lb < K && o[lb] == p) dp[nd++] = r2 * K + lb;
      }
    } else {
      dsa_flag(dev_err, DSA_DEVERR_BOUNDS);
    }
    ++nM_local;
  }
  nM_local = __reduce_add_sync(0xffffffffu, nM_local);
  if ((threadIdx.x & 31) == 0 && nM_local) atomicAdd(&s_cnt[3], nM_local);
  __syncthreads();
  const int nM = s_cnt[3];

  // 3. victims in cyclic order from the hand. Ring: the eligible slots (not
  //    pinned in this call, not filled in this round). Clock: the eligible
  //    slots whose reference bit is clear (the hand's first turn), then those
  //    whose bit is set (its second turn, after the first cleared them).
  const int hand0 = (int)un.state[DSA_ST_HAND];
  int found = 0, found_first = 0;
  for (int pass = 0; pass < (clock ? 2 : 1) && found < nM; ++pass) {
    for (int base = 0; base < S && found < nM; base += ASSIGN_THREADS) {
      const int t = base + threadIdx.x;
      int sidx = -1;
      int elig = 0;
      if (t < S) {
        sidx = hand0 + t;
        if (sidx >= S) sidx -= S;
        elig = (un.pin_epoch[sidx] != epoch) && (un.fill_round[sidx] < round);
        if (clock && elig) elig = (un.ref[sidx] != 0) == (pass == 1);
      }
      int tot;
      const int inc = block_inclusive_scan<ASSIGN_THREADS>(elig, s_tmp, &tot);
      const int rank = found + inc - elig;
      if (elig && rank < nM) fill_slot[rank] = sidx;
      found += tot;
    }
    if (pass == 0) found_first = found;
  }
  const int n = min(found, nM);
  __syncthreads();
  if (clock && n > 0) {
    // the bits the first turn passed are cleared: up to the last victim if
    // the first turn found them all, else every eligible slot's
    int limit = S;
    if (n <= found_first) {
      const int last = fill_slot[n - 1];
      limit = last >= hand0 ? last - hand0 : last + S - hand0;
    }
    for (int t = threadIdx.x; t < limit; t += ASSIGN_THREADS) {
      int sidx = hand0 + t;
      if (sidx >= S) sidx -= S;
      if (un.pin_epoch[sidx] != epoch && un.fill_round[sidx] < round && un.ref[sidx]) un.ref[sidx] = 0;
    }
    __syncthreads();
  }

  // 4. map update (distinct slots, distinct new positions, and old positions
  //    that are neither new positions nor pinned: safe in parallel)
  for (int i = threadIdx.x; i < n; i += ASSIGN_THREADS) {
    const int sl = fill_slot[i];
    const int32_t p = fill_pos[i];
    const int32_t old = un.slot_pos[sl];
    if (old >= 0 && old < un.lmax) un.pos_slot[old] = -1;
    un.slot_pos[sl] = p;
    un.pos_slot[p] = sl;
    un.fill_round[sl] = round;
    if (clock) un.ref[sl] = 1;                // a fill sets the reference bit
  }
  // served[e] = 1 for owners that received a slot and for the later
  // occurrences of their position: the fill reads the mirror row once and
  // hands the same RAM bytes to every occurrence
  int32_t* fill_of = g.fill_of + (size_t)u * RK;
  for (int e = threadIdx.x; e < RK; e += ASSIGN_THREADS) {
    served[e] = 0;
    fill_of[e] = -1;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < n; i += ASSIGN_THREADS) {
    served[fill_entry[i]] = 1;
    fill_of[fill_entry[i]] = i;
    const int32_t* dp = g.dup + ((size_t)u * RK + i) * (DSA_MAX_ROWS - 1);
    for (int k = 0; k < R - 1 && dp[k] >= 0; ++k) served[dp[k]] = 1;
  }
  if (threadIdx.x == 0) {
    if (n > 0) {
      int h = fill_slot[n - 1] + 1;
      un.state[DSA_ST_HAND] = h >= S ? 0 : h;
    }
    un.state[DSA_ST_EPOCH] = epoch;
    un.state[DSA_ST_ROUND] = (int64_t)round + 1;
    g.nfill[u] = n;
    int32_t* cu = counters + (size_t)u * 4;
    cu[0] = s_cnt[0];
    cu[1] = s_cnt[1];
    cu[2] = s_cnt[2];
    cu[3] = n;
  }
}

__global__ void __launch_bounds__(COPY_THREADS)
k_copy(const dsa_unit* __restrict__ units, int U, int R, int K, const int32_t* __restrict__ topk_all,
       const uint8_t* __restrict__ cls_all, uint8_t* __restrict__ rows_all, GatherWs g, int32_t* dev_err,
       int bw_blocks) {
  const int lane = threadIdx.x & 31;
  pdl_wait();
  const int RK = R * K;
  int nblocks = gridDim.x;
  if (bw_blocks > 0) {
    __shared__ int s_fills;
    if (threadIdx.x == 0) s_fills = 0;
    __syncthreads();
    int f = 0;
    for (int u = threadIdx.x; u < U; u += COPY_THREADS) f += g.nfill[u];
    f = __reduce_add_sync(0xffffffffu, f);
    if ((threadIdx.x & 31) == 0 && f) atomicAdd(&s_fills, f);
    __syncthreads();
    if (s_fills >= COPY_BW_FILLS) {
      if ((int)blockIdx.x >= bw_blocks) return;   // (the whole block)
      nblocks = bw_blocks;
    }
  }
  // warps walk the flattened (unit, item) space in order: per unit its RK
  // entries, then its fills in ascending position order (mirror rows are
  // read in position order, unit by unit, which suits the host's page
  // translations)
  const int64_t nitems = (int64_t)U * 2 * RK;
  for (int64_t idx = (int64_t)blockIdx.x * COPY_WARPS + (threadIdx.x >> 5); idx < nitems;
       idx += (int64_t)nblocks * COPY_WARPS) {
    const int u = (int)(idx / (2 * RK));
    const int item = (int)(idx - (int64_t)u * 2 * RK);
    const dsa_unit& un = units[u];
    uint8_t* rows = rows_all + (size_t)u * RK * DSA_ROW_BYTES;
    if (item < RK) {
      const int e = item;
      if (g.served[(size_t)u * RK + e]) continue;   // written by its fill
      const uint8_t c = cls_all[(size_t)u * RK + e];
      const int32_t p = topk_all[(size_t)u * RK + e];
      uint8_t* dst = rows + (size_t)e * DSA_ROW_BYTES;
      if (c == DSA_CLS_HOT) {
        const int32_t sl = un.pos_slot[p];
        if (sl >= 0 && sl < un.slots_n) {
          warp_copy_row(dst, un.slots + (size_t)sl * DSA_ROW_BYTES, lane);
        } else {   // the map changed under this copy (a later assign ran first)
          warp_zero_row(dst, lane);
          if (lane == 0) dsa_flag(dev_err, DSA_DEVERR_BOUNDS);
        }
      } else if (c == DSA_CLS_RING) {
        warp_copy_row(dst, un.ring + (size_t)(p & (DSA_RING_ROWS - 1)) * DSA_ROW_BYTES, lane);
      } else if (c == DSA_CLS_RAM) {
        warp_copy_row(dst, un.mirror + (size_t)p * DSA_ROW_BYTES, lane);
      } else {
        warp_zero_row(dst, lane);
      }
    } else {
      const int f = item - RK;
      if (f >= g.nfill[u]) continue;
      const size_t o = (size_t)u * RK + f;
      const int32_t p = g.fill_pos[o];
      const int32_t s = g.fill_slot[o];
      const int32_t e = g.fill_entry[o];
      const uint4* src = reinterpret_cast<const uint4*>(un.mirror + (size_t)p * DSA_ROW_BYTES);
      uint4* d1 = reinterpret_cast<uint4*>(un.slots + (size_t)s * DSA_ROW_BYTES);
      uint4* d2 = reinterpret_cast<uint4*>(rows + (size_t)e * DSA_ROW_BYTES);
      const uint4 a = ldg_nc_v4(src + lane);
      uint4 b;
      if (lane < 9) b = ldg_nc_v4(src + 32 + lane);
      d1[lane] = a;
      d2[lane] = a;
      if (lane < 9) {
        d1[32 + lane] = b;
        d2[32 + lane] = b;
      }
      const int32_t* dp = g.dup + o * (DSA_MAX_ROWS - 1);
      for (int k = 0; k < R - 1; ++k) {
        const int32_t ed = dp[k];
        if (ed < 0) break;
        uint4* d3 = reinterpret_cast<uint4*>(rows + (size_t)ed * DSA_ROW_BYTES);
        d3[lane] = a;
        if (lane < 9) d3[32 + lane] = b;
      }
    }
  }
}

}  // namespace

extern "C" size_t hot_gather_workspace(int32_t U, int32_t R, int32_t K) {
  if (U < 1 || R < 1 || K < 1) return 0;
  const size_t rk = (size_t)R * K;
  return 4 * dsa_align((size_t)U * rk * 4, 256) + dsa_align((size_t)U * 4, 256) +
         dsa_align((size_t)U * rk, 256) + dsa_align((size_t)U * rk * (DSA_MAX_ROWS - 1) * 4, 256);
}

int dsa_launch_assign(const dsa_unit* units, int32_t U, int32_t R, int32_t K, int32_t round,
                      const int32_t* topk_idx, uint8_t* cls, int32_t* counters, void* ws, int32_t* dev_err,
                      cudaStream_t st) {
  GatherWs g = gather_ws(ws, U, R, K);
  const int RK = R * K;
  static DsaPerDevice pd;
  int dev = 0;
  const int ok = dsa_device_setup(pd, &dev, [](int) {
    DSA_CUDA_TRY(dsa_prefer_shared(k_assign));
    DSA_CUDA_TRY(cudaFuncSetAttribute(k_assign, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)assign_smem(DSA_MAX_ROWS * DSA_MAX_K)));
    return DSA_OK;
  });
  if (ok != DSA_OK) return ok;
  return launch_pdl(k_assign, dim3(U), dim3(ASSIGN_THREADS), assign_smem(RK), st, units, R, K, round, topk_idx,
                    cls, counters, g, dev_err);
}

static int gather_args_ok(const dsa_unit* units, int32_t U, int32_t R, int32_t K, const int32_t* topk_idx,
                          const void* cls, void* ws, size_t ws_bytes) {
  if (!units || !topk_idx || !cls) return DSA_ERR_ARG;
  if (U < 1 || U > 65535 || R < 1 || R > DSA_MAX_ROWS) return DSA_ERR_ARG;
  if (K < 1 || K > DSA_MAX_K) return DSA_ERR_SHAPE;
  if (!ws || ws_bytes < hot_gather_workspace(U, R, K)) return DSA_ERR_WS;
  return DSA_OK;
}

extern "C" int hot_gather_assign(const dsa_unit* units, int32_t U, int32_t R, int32_t K, int32_t round,
                                 const int32_t* topk_idx, uint8_t* cls, int32_t* counters, void* ws,
                                 size_t ws_bytes, int32_t* dev_err, void* stream) {
  const int st = gather_args_ok(units, U, R, K, topk_idx, cls, ws, ws_bytes);
  if (st != DSA_OK) return st;
  if (!counters) return DSA_ERR_ARG;
  return dsa_launch_assign(units, U, R, K, round, topk_idx, cls, counters, ws, dev_err,
                           static_cast<cudaStream_t>(stream));
}

extern "C" int hot_gather_copy(const dsa_unit* units, int32_t U, int32_t R, int32_t K, const int32_t* topk_idx,
                               const uint8_t* cls, uint8_t* rows, void* ws, size_t ws_bytes, int32_t* dev_err,
                               void* stream) {
  const int st = gather_args_ok(units, U, R, K, topk_idx, cls, ws, ws_bytes);
  if (st != DSA_OK) return st;
  if (!rows || (reinterpret_cast<uintptr_t>(rows) & 15u)) return DSA_ERR_ARG;
  static DsaPerDevice pd;
  int dev = 0;
  const int ok = dsa_device_setup(pd, &dev, [](int) {
    DSA_CUDA_TRY(dsa_prefer_shared(k_copy));
    return DSA_OK;
  });
  if (ok != DSA_OK) return ok;
  const int64_t entries = (int64_t)U * R * K;
  const int sms = dsa_stream_sms(static_cast<cudaStream_t>(stream), pd.num_sms[dev]);
  const bool own_sms = sms < pd.num_sms[dev];   // the stream has an SM partition of its own
  // Beside other kernels (a scoring that holds the SMs) host-link reads in
  // flight beyond what the link serves only slow those kernels: the copy
  // takes one block per SM from COPY_BW_ENTRIES selected entries on, and
  // mid-size calls do so once their fills turn out to bind on the host link.
  // On an SM partition of its own, it fills the partition instead.
  const int64_t per_sm = own_sms ? COPY_MAX_BLOCKS_PER_SM : entries >= COPY_BW_ENTRIES ? 1 : COPY_BLOCKS_PER_SM;
  const int64_t blocks =
      std::max<int64_t>(1, std::min<int64_t>((2 * entries + COPY_WARPS - 1) / COPY_WARPS, per_sm * sms));
  const int bw_blocks = (!own_sms && entries >= COPY_MID_ENTRIES && entries < COPY_BW_ENTRIES) ? sms : 0;
  return launch_pdl(k_copy, dim3((unsigned)blocks), dim3(COPY_THREADS), 0, static_cast<cudaStream_t>(stream),
                    units, (int)U, (int)R, (int)K, topk_idx, cls, rows, gather_ws(ws, U, R, K), dev_err,
                    bw_blocks);
}

extern "C" int hot_gather(const dsa_unit* units, int32_t U, int32_t R, int32_t K, int32_t round,
                          const int32_t* topk_idx, uint8_t* cls, uint8_t* rows, int32_t* counters,
                          void* ws, size_t ws_bytes, int32_t* dev_err, void* stream) {
  if (!rows || !counters) return DSA_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(rows) & 15u) return DSA_ERR_ARG;
  const int st = hot_gather_assign(units, U, R, K, round, topk_idx, cls, counters, ws, ws_bytes, dev_err, stream);
  if (st != DSA_OK) return st;
  return hot_gather_copy(units, U, R, K, topk_idx, cls, rows, ws, ws_bytes, dev_err, stream);
}
