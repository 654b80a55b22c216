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
//  * k_dsa_score: one CTA per (tile of positions, unit). Keys stream from HBM
//    with 16-byte read-only loads; the R query rows and head weights sit
//    in shared memory as fp32; scores accumulate in fp32 FMA (exact for
//    integer-grid data). Each score becomes an order-preserving uint32 key,
//    written to the workspace, and a 4096-bin histogram of its top 12 bits is
//    built in shared memory and merged into a global per-(unit,row) histogram.
//  * k_topk_select: one 8-CTA thread-block cluster per (unit, row). The global
//    histogram gives the top digit of the K-th largest key; three refinement
//    passes (8, 8 and 4 bits) over the cluster's key ranges, with histograms
//    summed through distributed shared memory, give the exact threshold key T
//    and how many keys equal to T are taken. A last pass writes the selected
//    positions in ascending order (ballot-based ordered compaction); keys equal
//    to T are taken lowest position first.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int SCORE_THREADS = 256;
constexpr int SCORE_TILE = 512;          // positions per CTA
constexpr int HIST1_BINS = 4096;         // top 12 bits of the ordered key
constexpr int SEL_CLUSTER = 8;
constexpr int SEL_THREADS = 512;

struct TopkWs {
  uint32_t* hist;   // [U*R][4096]
  uint32_t* keys;   // [U*R][stride]
  int64_t stride;
};

inline int64_t key_stride(int64_t max_len) { return (max_len + 3) / 4 * 4; }

inline TopkWs topk_ws(void* ws, int32_t U, int32_t R, int64_t max_len) {
  TopkWs w;
  w.hist = static_cast<uint32_t*>(ws);
  size_t hb = dsa_align((size_t)U * R * HIST1_BINS * 4, 256);
  w.keys = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + hb);
  w.stride = key_stride(max_len);
  return w;
}

// Order-preserving map float -> uint32 (larger float, larger key); -0 == +0.
__device__ __forceinline__ uint32_t ordered_key(float s) {
  uint32_t b = __float_as_uint(s == 0.0f ? 0.0f : s);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__global__ void __launch_bounds__(SCORE_THREADS)
k_dsa_score(const dsa_unit* __restrict__ units, int R, int K,
            const uint16_t* __restrict__ q, const float* __restrict__ w,
            uint32_t* __restrict__ hist, uint32_t* __restrict__ okeys, int64_t stride,
            int64_t max_len) {
  const int u = blockIdx.y;
  const int64_t L = min(units[u].state[DSA_ST_LEN], max_len);
  const int64_t p0 = (int64_t)blockIdx.x * SCORE_TILE;
  if (p0 >= L || L <= K) return;   // L <= K: the select emits 0..L-1 directly

  extern __shared__ float sm[];
  float* sq = sm;                                  // [R][8][64]
  float* sw = sq + R * 512;                        // [R][8]
  uint32_t* sh = reinterpret_cast<uint32_t*>(sw + R * 8);  // [R][4096]

  const uint16_t* qu = q + (size_t)u * R * 512;
  for (int i = threadIdx.x; i < R * 512; i += SCORE_THREADS) sq[i] = bf16f(qu[i]);
  for (int i = threadIdx.x; i < R * 8; i += SCORE_THREADS) sw[i] = w[(size_t)u * R * 8 + i];
  for (int i = threadIdx.x; i < R * HIST1_BINS; i += SCORE_THREADS) sh[i] = 0;
  __syncthreads();

  const uint4* kp = reinterpret_cast<const uint4*>(units[u].keys);
  const int64_t pend = min(p0 + (int64_t)SCORE_TILE, L);
  uint32_t* ok = okeys + (size_t)u * R * stride;
  for (int64_t p = p0 + threadIdx.x; p < pend; p += SCORE_THREADS) {
    uint4 v[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) v[c] = ldg_v4(kp + p * 8 + c);
    float k[64];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint32_t ww[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        k[c * 8 + 2 * e] = bf16_lo(ww[e]);
        k[c * 8 + 2 * e + 1] = bf16_hi(ww[e]);
      }
    }
    for (int r = 0; r < R; ++r) {
      float acc = 0.0f;
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float4* qh = reinterpret_cast<const float4*>(sq + (r * 8 + h) * 64);
        float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float4 qq = qh[i];
          d0 = fmaf(qq.x, k[4 * i + 0], d0);
          d1 = fmaf(qq.y, k[4 * i + 1], d1);
          d2 = fmaf(qq.z, k[4 * i + 2], d2);
          d3 = fmaf(qq.w, k[4 * i + 3], d3);
        }
        const float dot = (d0 + d1) + (d2 + d3);
        acc = fmaf(sw[r * 8 + h], fmaxf(dot, 0.0f), acc);
      }
      const uint32_t key = ordered_key(acc);
      ok[(size_t)r * stride + p] = key;
      atomicAdd(&sh[r * HIST1_BINS + (key >> 20)], 1u);
    }
  }
  __syncthreads();
  uint32_t* gh = hist + (size_t)u * R * HIST1_BINS;
  for (int i = threadIdx.x; i < R * HIST1_BINS; i += SCORE_THREADS) {
    const uint32_t c = sh[i];
    if (c) atomicAdd(&gh[i], c);
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

__global__ void __cluster_dims__(SEL_CLUSTER, 1, 1) __launch_bounds__(SEL_THREADS)
k_topk_select(const dsa_unit* __restrict__ units, int R, int K, uint32_t* __restrict__ hist,
              const uint32_t* __restrict__ okeys, int64_t stride, int32_t* __restrict__ topk_idx,
              int64_t max_len, int32_t* dev_err) {
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int ur = blockIdx.y;
  const int u = ur / R;
  const int64_t Lu = units[u].state[DSA_ST_LEN];
  const int64_t L = min(Lu, max_len);
  if (Lu > max_len && crank == 0 && threadIdx.x == 0) dsa_flag(dev_err, DSA_DEVERR_BOUNDS);
  int32_t* out = topk_idx + (size_t)ur * K;

  if (L <= K) {  // every position is selected; no cluster communication
    for (int j = crank * SEL_THREADS + threadIdx.x; j < K; j += SEL_CLUSTER * SEL_THREADS)
      out[j] = j < L ? j : -1;
    return;
  }

  __shared__ uint32_t s_h1[HIST1_BINS];
  __shared__ uint32_t s_hl[2][256];   // local refinement histograms (double buffer)
  __shared__ uint32_t s_hg[256];      // cluster-summed refinement histogram
  __shared__ int s_tmp[32];
  __shared__ int s_bin, s_above;
  __shared__ long long s_cnt[2];      // this CTA's (gt, eq) counts
  __shared__ int s_wsum[SEL_THREADS / 32];
  if (threadIdx.x == 0) {
    s_bin = 0;
    s_above = 0;
  }

  // ---- level 1: top 12 bits from the global histogram
  uint32_t* gh = hist + (size_t)ur * HIST1_BINS;
  for (int i = threadIdx.x; i < HIST1_BINS; i += SEL_THREADS) s_h1[i] = gh[i];
  __syncthreads();
  // 4096 bins over 512 threads: each thread sums 8 bins, highest first.
  {
    const int t = threadIdx.x;
    int c = 0;
    const int hi = HIST1_BINS - 1 - 8 * t;
#pragma unroll
    for (int i = 0; i < 8; ++i) c += (int)s_h1[hi - i];
    const int inc = block_inclusive_scan<SEL_THREADS>(c, s_tmp);
    int exc = inc - c;
    if (exc < K && K <= inc) {
      for (int i = 0; i < 8; ++i) {
        const int cb = (int)s_h1[hi - i];
        if (exc + cb >= K) {
          s_bin = hi - i;
          s_above = exc;
          break;
        }
        exc += cb;
      }
    }
    __syncthreads();
  }
  const uint32_t b1 = (uint32_t)s_bin;
  int need = K - s_above;

  const int64_t chunk = (L + SEL_CLUSTER - 1) / SEL_CLUSTER;
  const int64_t beg = min((int64_t)crank * chunk, L);
  const int64_t end = min(beg + chunk, L);
  const uint32_t* kk = okeys + (size_t)ur * stride;

  long long local_gt = 0;
  uint32_t prefix = b1 << 20, mask = 0xFFF00000u;
  const int shifts[3] = {12, 4, 0};
  const int nbins[3] = {256, 256, 16};
  for (int lvl = 0; lvl < 3; ++lvl) {
    uint32_t* hl = s_hl[lvl & 1];
    for (int i = threadIdx.x; i < 256; i += SEL_THREADS) hl[i] = 0;
    __syncthreads();
    const int sh = shifts[lvl];
    const uint32_t dm = (uint32_t)nbins[lvl] - 1;
    long long gt_top = 0;   // level 1 only: keys whose top digit is above b1
    for (int64_t p = beg + threadIdx.x; p < end; p += SEL_THREADS) {
      const uint32_t key = kk[p];
      if ((key & mask) == prefix) atomicAdd(&hl[(key >> sh) & dm], 1u);
      else if (lvl == 0 && (key >> 20) > b1) ++gt_top;
    }
    if (lvl == 0) {
      int tot;
      block_inclusive_scan<SEL_THREADS>((int)gt_top, s_tmp, &tot);
      local_gt += tot;
    }
    __syncthreads();
    cluster.sync();
    // sum the cluster's histograms of this level
    for (int i = threadIdx.x; i < nbins[lvl]; i += SEL_THREADS) {
      uint32_t s = 0;
      for (int c = 0; c < SEL_CLUSTER; ++c) s += cluster.map_shared_rank(hl, c)[i];
      s_hg[i] = s;
    }
    if (lvl == 0 && crank == 0) {
      // every CTA of the cluster read the global histogram before the
      // cluster barrier above: clear it for the next call
      for (int i = threadIdx.x; i < HIST1_BINS; i += SEL_THREADS) gh[i] = 0;
    }
    __syncthreads();
    find_digit<SEL_THREADS>(s_hg, nbins[lvl], need, s_tmp, &s_bin, &s_above);
    const uint32_t b = (uint32_t)s_bin;
    need -= s_above;
    // this CTA's keys above the digit at this level
    {
      const int t = threadIdx.x;
      int c = (t < nbins[lvl] && (uint32_t)t > b) ? (int)hl[t] : 0;
      int tot;
      block_inclusive_scan<SEL_THREADS>(c, s_tmp, &tot);
      local_gt += tot;
      if (lvl == 2 && t == 0) s_cnt[1] = hl[b];
    }
    prefix |= b << sh;
    mask |= dm << sh;
  }
  const uint32_t T = prefix;
  const int ties = need;            // keys equal to T that are taken
  if (threadIdx.x == 0) s_cnt[0] = local_gt;
  __syncthreads();
  cluster.sync();
  long long eq_before = 0, sel_before = 0;
  {
    for (int c = 0; c < crank; ++c) {
      const long long* rc = cluster.map_shared_rank(s_cnt, c);
      const long long g = rc[0], e = rc[1];
      long long take = (long long)ties - eq_before;
      take = take < 0 ? 0 : (take > e ? e : take);
      sel_before += g + take;
      eq_before += e;
    }
  }
  // ordered compaction of this CTA's range
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long run_eq = eq_before, run_sel = sel_before;
  for (int64_t base = beg; base < end; base += SEL_THREADS) {
    const int64_t p = base + threadIdx.x;
    const uint32_t key = p < end ? kk[p] : 0u;
    const bool gt = p < end && key > T;
    const bool eq = p < end && key == T;
    const unsigned beq = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) s_wsum[warp] = __popc(beq);
    __syncthreads();
    int weq = 0, teq = 0;
    for (int i = 0; i < SEL_THREADS / 32; ++i) {
      const int v = s_wsum[i];
      if (i < warp) weq += v;
      teq += v;
    }
    const long long eq_rank = run_eq + weq + __popc(beq & ((1u << lane) - 1u));
    const bool sel = gt || (eq && eq_rank < ties);
    __syncthreads();
    const unsigned bs = __ballot_sync(0xffffffffu, sel);
    if (lane == 0) s_wsum[warp] = __popc(bs);
    __syncthreads();
    int wsel = 0, tsel = 0;
    for (int i = 0; i < SEL_THREADS / 32; ++i) {
      const int v = s_wsum[i];
      if (i < warp) wsel += v;
      tsel += v;
    }
    if (sel) {
      const long long o = run_sel + wsel + __popc(bs & ((1u << lane) - 1u));
      if (o < K) out[o] = (int32_t)p;
    }
    run_eq += teq;
    run_sel += tsel;
    __syncthreads();
  }
  cluster.sync();   // keep this CTA's shared memory alive for its peers
}

}  // namespace

extern "C" size_t dsa_score_topk_workspace(int32_t U, int32_t R, int64_t max_len) {
  if (U < 1 || R < 1 || max_len < 0) return 0;
  return dsa_align((size_t)U * R * HIST1_BINS * 4, 256) +
         dsa_align((size_t)U * R * key_stride(max_len) * 4, 256);
}

extern "C" int dsa_score_topk(const dsa_unit* units, int32_t U, int32_t R, int32_t K,
                              const uint16_t* q, const float* w, int32_t* topk_idx,
                              int64_t max_len, void* ws, size_t ws_bytes, int32_t* dev_err,
                              void* stream) {
  if (!units || !q || !w || !topk_idx) return DSA_ERR_ARG;
  if (U < 1 || U > 65535 || R < 1 || R > DSA_MAX_ROWS || max_len < 0) return DSA_ERR_ARG;
  if (K < 1 || K > DSA_MAX_K) return DSA_ERR_SHAPE;
  if (!ws || ws_bytes < dsa_score_topk_workspace(U, R, max_len)) return DSA_ERR_WS;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  TopkWs tw = topk_ws(ws, U, R, max_len);
  const int64_t tiles = (max_len + SCORE_TILE - 1) / SCORE_TILE;
  if (tiles > 0) {
    const size_t smem = (size_t)R * (512 + 8) * 4 + (size_t)R * HIST1_BINS * 4;
    static bool attr_done = false;
    if (!attr_done) {
      DSA_CUDA_TRY(cudaFuncSetAttribute(k_dsa_score, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)((size_t)DSA_MAX_ROWS * (520 + HIST1_BINS) * 4)));
      attr_done = true;
    }
    if (tiles > 0x7fffffff) return DSA_ERR_ARG;
    k_dsa_score<<<dim3((unsigned)tiles, U), SCORE_THREADS, smem, st>>>(units, R, K, q, w, tw.hist,
                                                                     tw.keys, tw.stride, max_len);
    if (dsa_launch_status() != DSA_OK) return DSA_ERR_CUDA;
  }
  k_topk_select<<<dim3(SEL_CLUSTER, U * R), SEL_THREADS, 0, st>>>(units, R, K, tw.hist, tw.keys,
                                                                  tw.stride, topk_idx, max_len,
                                                                  dev_err);
  return dsa_launch_status();
}

// ---------------------------------------------------------------------------
// dsa_score_topk_noalloc: the same scoring and selection for callers that may
// not allocate device memory. Its scratch (selection histograms and ordered
// score keys) lives in one fixed array compiled into this library.

namespace {

constexpr int64_t NOALLOC_MAX_UR = 16;          // units x query rows per call
constexpr int64_t NOALLOC_MAX_LEN = 65536;      // history positions per unit
constexpr size_t NOALLOC_HIST_BYTES = (size_t)NOALLOC_MAX_UR * HIST1_BINS * 4;   // 256 KiB
constexpr size_t NOALLOC_BYTES =
    NOALLOC_HIST_BYTES + (size_t)NOALLOC_MAX_UR * NOALLOC_MAX_LEN * 4;           // 4.25 MiB
constexpr int NOALLOC_MAX_DEVICES = 64;

static __device__ __align__(256) uint8_t g_topk_scratch[NOALLOC_BYTES];

// Device address of g_topk_scratch, per device ordinal (looked up once).
void* g_topk_scratch_addr[NOALLOC_MAX_DEVICES];

}  // namespace

extern "C" int dsa_score_topk_noalloc(const dsa_unit* units, int32_t U, int32_t R, int32_t K,
                                      const uint16_t* q, const float* w, int32_t* topk_idx,
                                      int64_t max_len, int32_t* dev_err, void* stream) {
  if (!units || !q || !w || !topk_idx) return DSA_ERR_ARG;
  if (U < 1 || R < 1 || R > DSA_MAX_ROWS || max_len < 0) return DSA_ERR_ARG;
  if (K < 1 || K > DSA_MAX_K) return DSA_ERR_SHAPE;
  if ((int64_t)U * R > NOALLOC_MAX_UR || max_len > NOALLOC_MAX_LEN) return DSA_ERR_SCRATCH_LIMIT;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NOALLOC_MAX_DEVICES) return DSA_ERR_CUDA;
  if (!g_topk_scratch_addr[dev]) {
    // First call on this device: host code cannot use the array's name as a
    // device address, so ask the runtime for it (the device must be current).
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_topk_scratch) != cudaSuccess || !p) return DSA_ERR_CUDA;
    g_topk_scratch_addr[dev] = p;
  }
  void* scratch = g_topk_scratch_addr[dev];
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
