// A4 + A5: Q8G64 dequantisation and absorbed-MLA decode attention.
//
// [ALG] "Algorithm layer: from attention and KV cache to FFN and MoE",
// section "2. Attention": softmax(Q K^T / sqrt(d_k)) V; section "3. KV Cache":
// MLA keeps the normalised latent and the RoPE part, the latent as INT8 per
// group. [QNT] "Quantization is not a zip file", section "三、基本思路":
// w_hat = scale * q, one scale per group of 64 (G64). [P3] "From 1M total to
// 15+ x 1M", section "起点": a row is 512 B latent + 16 B scales + 128 B RoPE.
//
// One thread-block cluster per (unit, query row), of ceil(K / 128) CTAs
// rounded up to a power of two; CTA c of the cluster owns selected rows
// [128c, 128c + 128) (none for the padding CTAs):
//  1. one 1-D bulk TMA copy brings the CTA's rows (up to 128 x 656 B) into
//     shared memory region X;
//  2. dequantisation writes an fp16 tile [128 rows][576] (latent int8 * fp16
//     scale rounded once to fp16; RoPE bf16 -> fp16) in the K-major
//     128-byte-swizzled layout into region Y. The same bytes serve as the
//     K-major B operand of S = Q K^T and, read as an MN-major operand, as the
//     B operand of O = P V;
//  3. the query block (64 heads x 576, bf16 -> fp16) goes into X;
//  4. tcgen05.mma kind::f16, M = 128 (heads, 64 real), N = 128 for S and
//     2 x 256 for O, fp32 accumulators in tensor memory, one issuing thread,
//     completion through tcgen05.commit on an mbarrier;
//  5. softmax of the CTA's 128 columns per head in registers; P (fp16) goes to
//     X as the A operand of PV;
//  6. each CTA stores its O (64 x 512 fp32) to its workspace slot (it stays in
//     L2) and its max/sum to shared memory; after a cluster barrier CTA c
//     merges columns [c*W, c*W + W) of every CTA's O with the max/sum
//     rescaling of split softmax (maxima and sums read through distributed
//     shared memory) and writes the final out (and lse) directly.
// fp16 operands keep 11 significant bits: each operand's rounding is <= 2^-11
// relative, far inside the 1e-3 * max|out| budget. Waits are bounded; on a
// timeout the kernel sets DSA_DEVERR_TIMEOUT, frees its tensor memory and
// still takes part in every cluster barrier so no peer is left waiting.
#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "gather_internal.cuh"
#include "tc.cuh"

namespace cg = cooperative_groups;

namespace {

constexpr int NC = 128;                         // selected rows per CTA
constexpr int MAX_CLUSTER = 16;                 // -> K <= 2048
constexpr int THREADS = 256;
constexpr int QATOM = 8192;                     // 64 rows x 128 B (query and P atoms)
constexpr int BATOM = NC * 128;                 // 128 rows x 128 B (row-tile atoms)
constexpr int X_OFF = 0;
constexpr int X_BYTES = NC * DSA_ROW_BYTES;     // 83,968 = 82 KB
constexpr int Y_OFF = X_BYTES;
constexpr int Y_BYTES = 9 * BATOM;              // 147,456
constexpr int MISC_OFF = Y_OFF + Y_BYTES;
constexpr int SMEM_BYTES = MISC_OFF + 1024;     // 232,448: the whole opt-in budget
constexpr int OSTR = 516;                       // fp32 row stride of the staged O
constexpr int TMEM_COLS = 512;
constexpr uint32_t IDESC_QK = tc::idesc_f16_f32(128, NC, 0, 0);
constexpr uint32_t IDESC_PV = tc::idesc_f16_f32(128, 256, 0, 1);

static_assert(X_BYTES % 1024 == 0, "region X must keep Y 1024-aligned");
static_assert(64 * OSTR * 4 <= Y_BYTES, "staged O must fit in Y");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

struct Misc {
  uint64_t bar[2];        // [0] TMA, [1] MMA
  uint32_t tmem;
  int fail;
  float m[64];
  float l[64];
  uint32_t vmask[NC / 32];    // validity of this CTA's rows
};

// Softmax partials, in region X beyond the P atoms (the query block is dead
// once S is computed).
struct SoftmaxScratch {
  float pm[2][64];            // partial max per column half
  float pl[2][64];            // partial sum per column half
};
constexpr int SMX_OFF = 4 * QATOM;
static_assert(sizeof(Misc) <= 1024, "misc block");

// Merge-phase scratch, placed in region X once P is no longer needed.
struct MergeScratch {
  float rm[MAX_CLUSTER][64];  // every source CTA's max per head
  float rl[MAX_CLUSTER][64];  // every source CTA's sum per head
  float f[MAX_CLUSTER][64];   // exp(m_c - M) per source CTA and head
  float inv[64];              // 1 / L per head
};
static_assert(sizeof(MergeScratch) <= X_BYTES, "merge scratch");

// CTAs per cluster for K selected rows: ceil(K / 128) rounded up to a power
// of two (at most 16 for K <= 2048). The merge splits the 512 output columns
// evenly over the cluster, so the count must divide 512; the CTAs past the
// last row hold no rows and add an empty softmax part (max -inf, sum 0).
inline int cluster_ctas(int K) {
  const int need = (K + NC - 1) / NC;
  int C = 1;
  while (C < need) C *= 2;
  return C;
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst_smem)), "l"(src) : "memory");
}

// GATHER = false: the rows come compact from hot_gather (one bulk copy).
// GATHER = true: the rows are read from their sources (HOT slot, ring, RAM
// mirror) as classified by the gather's assign kernel, and each inserted
// miss's row is also written to its victim slot.
template <bool GATHER>
__global__ void __launch_bounds__(THREADS, 1)
k_mla_attn(int R, int H, int K, const uint16_t* __restrict__ q_lat, const uint16_t* __restrict__ q_rope,
           const uint8_t* __restrict__ rows, const int32_t* __restrict__ topk, float scale,
           float* __restrict__ out, float* __restrict__ lse, float* __restrict__ ws_o, int32_t* dev_err,
           const dsa_unit* __restrict__ units, const uint8_t* __restrict__ cls, GatherWs g) {
  extern __shared__ __align__(1024) uint8_t sm[];
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int crank = (int)cluster.block_rank();
  uint8_t* sX = sm + X_OFF;
  uint8_t* sY = sm + Y_OFF;
  Misc* ms = reinterpret_cast<Misc*>(sm + MISC_OFF);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ur = blockIdx.y;
  const int j0 = crank * NC;
  const int nrows = max(0, min(NC, K - j0));

  if (tid == 0) {
    tc::mbar_init(&ms->bar[0], 1);
    tc::mbar_init(&ms->bar[1], 1);
    tc::fence_mbar_init();
    ms->fail = (tc::smem_u32(sm) & 1023u) != 0;   // the tile layouts need 1024-byte alignment
  }
  if (warp == 0) tc::tmem_alloc(&ms->tmem, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ms->tmem;
  bool failed = ms->fail != 0;
  pdl_wait();   // everything above touched only this CTA's shared and tensor memory

  // The rows of a CTA arrive by one bulk copy on phase 0 of bar[0]; a CTA
  // without rows (the cluster is padded to a power of two) issues none, so
  // the merge's copies below complete phase 0 there and phase 1 elsewhere.
  const bool rows_copy = !GATHER && !failed && nrows > 0;
  if (rows_copy && tid == 0) {
    const uint32_t bytes = (uint32_t)nrows * DSA_ROW_BYTES;
    tc::mbar_arrive_expect_tx(&ms->bar[0], bytes);
    tc::bulk_g2s(sX, rows + ((size_t)ur * K + j0) * DSA_ROW_BYTES, bytes, &ms->bar[0]);
  }
  if (GATHER && !failed) {
    // source and fill destination of each of this CTA's rows (kept in Y, which
    // is free until the dequantised tile is written)
    const uint8_t** s_src = reinterpret_cast<const uint8_t**>(sY);
    uint8_t** s_dst = reinterpret_cast<uint8_t**>(sY + NC * sizeof(void*));
    if (tid < NC) {
      const uint8_t* src = nullptr;
      uint8_t* dst = nullptr;
      if (tid < nrows) {
        const size_t e = (size_t)ur * K + j0 + tid;    // = u * R * K + entry
        const int u = ur / R;
        const dsa_unit& un = units[u];
        const int32_t p = topk[e];
        const uint8_t c = cls[e];
        if (c == DSA_CLS_HOT) {
          const int32_t sl = un.pos_slot[p];
          if (sl >= 0 && sl < un.slots_n) src = un.slots + (size_t)sl * DSA_ROW_BYTES;
        } else if (c == DSA_CLS_RING) {
          src = un.ring + (size_t)(p & (DSA_RING_ROWS - 1)) * DSA_ROW_BYTES;
        } else if (c == DSA_CLS_RAM) {
          src = un.mirror + (size_t)p * DSA_ROW_BYTES;
          const int32_t f = g.fill_of[e];
          if (f >= 0) {
            const int32_t sl = g.fill_slot[(size_t)u * R * K + f];
            if (sl >= 0 && sl < un.slots_n) dst = un.slots + (size_t)sl * DSA_ROW_BYTES;
          }
        }
      }
      s_src[tid] = src;
      s_dst[tid] = dst;
    }
    __syncthreads();
    // every 16-byte piece of every row in flight at once (no registers held)
    for (int t = tid; t < nrows * 41; t += THREADS) {
      const int jj = t / 41, c = t % 41;
      const uint8_t* src = s_src[jj];
      uint8_t* d = sX + jj * DSA_ROW_BYTES + 16 * c;
      if (src) cp_async16(d, src + 16 * c);
      else *reinterpret_cast<uint4*>(d) = make_uint4(0, 0, 0, 0);
    }
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    // inserted misses: their RAM bytes also go to the victim slot
    for (int t = tid; t < nrows * 41; t += THREADS) {
      const int jj = t / 41, c = t % 41;
      uint8_t* dst = s_dst[jj];
      if (dst) *reinterpret_cast<uint4*>(dst + 16 * c) = *reinterpret_cast<const uint4*>(sX + jj * DSA_ROW_BYTES + 16 * c);
    }
  }
  if (tid < NC) {
    const bool v = (tid < nrows) && topk[(size_t)ur * K + j0 + tid] >= 0;
    const unsigned b = __ballot_sync(0xffffffffu, v);
    if (lane == 0) ms->vmask[warp] = b;
  }

  // query block loads, in flight while the rows arrive: 64 heads x 72 chunks of 8 dims
  constexpr int QCH = 64 * 72 / THREADS;        // 18 chunks per thread
  uint4 qv[QCH];
#pragma unroll
  for (int i = 0; i < QCH; ++i) {
    const int t = tid + i * THREADS;
    const int h = t / 72, c = t % 72;
    qv[i] = make_uint4(0, 0, 0, 0);
    if (h < H) {
      const size_t qo = (size_t)ur * H + h;
      qv[i] = c < 64 ? *reinterpret_cast<const uint4*>(q_lat + qo * 512 + 8 * c)
                     : *reinterpret_cast<const uint4*>(q_rope + qo * 64 + 8 * (c - 64));
    }
  }
  if (rows_copy && !tc::mbar_wait(&ms->bar[0], 0)) atomicOr(&ms->fail, 1);
  __syncthreads();
  failed = ms->fail != 0;

  // ---- dequantise the rows: region X (raw) -> region Y (fp16 tile)
  if (!failed) {
    bool bad = false;
    for (int t = tid; t < NC * 36; t += THREADS) {
      const int j = t % NC, c = t / NC;     // consecutive threads: consecutive rows
      uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
      if (j < nrows) {
        const uint8_t* row = sX + j * DSA_ROW_BYTES;
        uint32_t o[8];
        if (c < 32) {
          const float s = __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(row + 512)[c >> 2]));
          const uint4 raw = *reinterpret_cast<const uint4*>(row + 16 * c);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a0 = (float)(int8_t)(w[e] & 0xFF) * s;
            const float a1 = (float)(int8_t)((w[e] >> 8) & 0xFF) * s;
            const float a2 = (float)(int8_t)((w[e] >> 16) & 0xFF) * s;
            const float a3 = (float)(int8_t)(w[e] >> 24) * s;
            bad |= fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(a2), fabsf(a3))) >= 65504.f;
            o[2 * e] = pack_h2(a0, a1);
            o[2 * e + 1] = pack_h2(a2, a3);
          }
        } else {
          const uint4 r0 = *reinterpret_cast<const uint4*>(row + 528 + 32 * (c - 32));
          const uint4 r1 = *reinterpret_cast<const uint4*>(row + 528 + 32 * (c - 32) + 16);
          const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = pack_h2(bf16_lo(w[e]), bf16_hi(w[e]));
        }
        lo = make_uint4(o[0], o[1], o[2], o[3]);
        hi = make_uint4(o[4], o[5], o[6], o[7]);
      }
      const int d0 = 16 * c;
      uint8_t* atom = sY + (d0 >> 6) * BATOM;
      *reinterpret_cast<uint4*>(atom + tc::sw128_off(j, d0 & 63)) = lo;
      *reinterpret_cast<uint4*>(atom + tc::sw128_off(j, (d0 & 63) + 8)) = hi;
    }
    if (bad) dsa_flag(dev_err, DSA_DEVERR_QRANGE);
  }
  __syncthreads();   // raw rows are dead: X takes the query block
  if (!failed) {
    bool bad = false;
#pragma unroll
    for (int i = 0; i < QCH; ++i) {
      const int t = tid + i * THREADS;
      const int h = t / 72, c = t % 72;
      const uint32_t w[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
      uint32_t o[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
        bad |= fmaxf(fabsf(a), fabsf(b)) >= 65504.f;
        o[e] = pack_h2(a, b);
      }
      const int d0 = 8 * c;
      *reinterpret_cast<uint4*>(sX + (d0 >> 6) * QATOM + tc::sw128_off(h, d0 & 63)) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (bad) dsa_flag(dev_err, DSA_DEVERR_QRANGE);
  }
  tc::fence_async_shared();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();

  // ---- S = Q K^T: TMEM columns [0, 128)
  if (tid == 0 && !failed) {
    const uint32_t qa = tc::smem_u32(sX), ba = tc::smem_u32(sY);
    for (int kb = 0; kb < 9; ++kb) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t ad = tc::sdesc_sw128(qa + kb * QATOM + kk * 32, 16, 1024);
        const uint64_t bd = tc::sdesc_sw128(ba + kb * BATOM + kk * 32, 16, 1024);
        tc::mma_f16(tmem, ad, bd, IDESC_QK, (kb | kk) != 0);
      }
    }
    tc::mma_commit(&ms->bar[1]);
  }
  if (!failed && !tc::mbar_wait(&ms->bar[1], 0)) atomicOr(&ms->fail, 1);
  tc::fence_after_sync();
  __syncthreads();
  failed = ms->fail != 0;

  // ---- softmax over this CTA's columns. Warps 0,1,4,5 can read TMEM lanes
  // 0..63 (head rows); warp w takes lane quarter w & 3 and column half w >> 2.
  const bool sm_warp = (warp & 3) < 2;
  const int hr = 32 * (warp & 3) + lane;      // head row of this thread (sm_warp only)
  const int half = warp >> 2;
  SoftmaxScratch* sx = reinterpret_cast<SoftmaxScratch*>(sX + SMX_OFF);
  float s[64];
  if (sm_warp && !failed) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v[32];
      tc::tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 64 * half + 32 * c, v);
      const uint32_t vm = ms->vmask[2 * half + c];
#pragma unroll
      for (int i = 0; i < 32; ++i) s[32 * c + i] = ((vm >> i) & 1u) ? v[i] * scale : -INFINITY;
    }
    float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
#pragma unroll
    for (int j = 0; j < 64; j += 4) {
      m0 = fmaxf(m0, s[j]);
      m1 = fmaxf(m1, s[j + 1]);
      m2 = fmaxf(m2, s[j + 2]);
      m3 = fmaxf(m3, s[j + 3]);
    }
    sx->pm[half][hr] = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
  }
  __syncthreads();
  if (sm_warp && !failed) {
    const float m = fmaxf(sx->pm[0][hr], sx->pm[1][hr]);
    float l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int j = 0; j < 64; j += 2) {
      s[j] = (m == -INFINITY) ? 0.f : __expf(s[j] - m);
      s[j + 1] = (m == -INFINITY) ? 0.f : __expf(s[j + 1] - m);
      l0 += s[j];
      l1 += s[j + 1];
    }
    sx->pl[half][hr] = l0 + l1;
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      const uint4 v = make_uint4(pack_h2(s[8 * c8], s[8 * c8 + 1]), pack_h2(s[8 * c8 + 2], s[8 * c8 + 3]),
                                 pack_h2(s[8 * c8 + 4], s[8 * c8 + 5]), pack_h2(s[8 * c8 + 6], s[8 * c8 + 7]));
      *reinterpret_cast<uint4*>(sX + half * QATOM + tc::sw128_off(hr, 8 * c8)) = v;
    }
    if (half == 0) ms->m[hr] = m;
  }
  tc::fence_async_shared();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid < 64) ms->l[tid] = sx->pl[0][tid] + sx->pl[1][tid];

  // ---- O = P V: TMEM columns [0, 512)
  if (tid == 0 && !failed) {
    const uint32_t pa = tc::smem_u32(sX), ba = tc::smem_u32(sY);
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int kk = 0; kk < NC / 16; ++kk) {
        const uint64_t ad = tc::sdesc_sw128(pa + (kk >> 2) * QATOM + (kk & 3) * 32, 16, 1024);
        const uint64_t bd = tc::sdesc_sw128(ba + half * 4 * BATOM + kk * 2048, BATOM, 1024);
        tc::mma_f16(tmem + half * 256, ad, bd, IDESC_PV, kk > 0);
      }
    }
    tc::mma_commit(&ms->bar[1]);
  }
  if (!failed && !tc::mbar_wait(&ms->bar[1], 1)) atomicOr(&ms->fail, 1);
  tc::fence_after_sync();
  __syncthreads();
  failed = ms->fail != 0;

  // ---- this CTA's O (64 x 512 fp32) to its slot of the workspace (L2):
  //      warps 0,1,4,5 (lane quarters 0 and 1), 128 contiguous bytes per store run
  //      The slot is slice-major: the W = 512 / C columns that CTA c merges
  //      form one contiguous [64][W] block, so the merge fetches each source's
  //      block with one bulk copy. Each 32 x 32 block goes through a padded
  //      shared-memory transpose so every store writes whole 128-byte rows.
  const int W = 512 / C;                                 // C in {1, 2, 4, 8, 16}
  float* gO = ws_o + ((size_t)ur * MAX_CLUSTER + crank) * 64 * 512;
  if ((warp & 3) < 2 && !failed) {
    const int q = warp & 3;                              // lane quarter: head rows 32q..32q+31
    const int c0 = 256 * (warp >> 2);
    float* tb = reinterpret_cast<float*>(sY) + (2 * (warp >> 2) + q) * 32 * 36;   // [32][36]
    for (int c = 0; c < 8; ++c) {
      float v[32];
      tc::tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + c0 + 32 * c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        reinterpret_cast<float4*>(tb + lane * 36)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      __syncwarp();
      const int col = c0 + 32 * c;                       // first column of the block
      float* blk = gO + (size_t)(col / W) * 64 * W + (col % W);
#pragma unroll
      for (int r4 = 0; r4 < 8; ++r4) {
        const int r = 4 * r4 + (lane >> 3);              // row within the block
        const float4 x = reinterpret_cast<const float4*>(tb + r * 36)[lane & 7];
        reinterpret_cast<float4*>(blk + (size_t)(32 * q + r) * W)[lane & 7] = x;
      }
      __syncwarp();
    }
  }
  if (failed && tid < 64) {   // an empty contribution keeps the peers' merge well defined
    ms->m[tid] = -INFINITY;
    ms->l[tid] = 0.f;
  }
  tc::fence_async_global();   // the partial stores are read by bulk copies
  tc::fence_before_sync();
  __syncthreads();
  cluster.sync();
  tc::fence_async_global();

  // ---- merge columns [crank*W, crank*W + W) of all C CTAs' outputs: one
  //      bulk copy per source brings its contiguous [64][W] block into Y
  {
    MergeScratch* mg = reinterpret_cast<MergeScratch*>(sX);
    float* buf = reinterpret_cast<float*>(sY);           // [C][64][W] = 128 KB
    const uint32_t blk_bytes = 64u * (uint32_t)W * 4u;
    // (a CTA that already failed issues no copy: nothing of it stays in flight)
    if (tid == 0 && !failed) {
      tc::mbar_arrive_expect_tx(&ms->bar[0], blk_bytes * (uint32_t)C);
      for (int c = 0; c < C; ++c)
        tc::bulk_g2s(buf + (size_t)c * 64 * W,
                     ws_o + (((size_t)ur * MAX_CLUSTER + c) * 64 * 512 + (size_t)crank * 64 * W), blk_bytes,
                     &ms->bar[0]);
    }
    // one round of remote loads: every source CTA's (m, l) for every head
    for (int t = tid; t < C * 64; t += THREADS) {
      const Misc* rm = cluster.map_shared_rank(ms, t >> 6);
      mg->rm[t >> 6][t & 63] = rm->m[t & 63];
      mg->rl[t >> 6][t & 63] = rm->l[t & 63];
    }
    __syncthreads();
    if (tid < 64) {
      const int h = tid;
      float M = -INFINITY;
      for (int c = 0; c < C; ++c) M = fmaxf(M, mg->rm[c][h]);
      float L = 0.f;
      for (int c = 0; c < C; ++c) {
        const float f = mg->rm[c][h] == -INFINITY ? 0.f : __expf(mg->rm[c][h] - M);
        mg->f[c][h] = f;
        L += f * mg->rl[c][h];
      }
      mg->inv[h] = L > 0.f ? 1.f / L : 0.f;
      if (crank == 0 && lse && h < H) lse[(size_t)ur * H + h] = L > 0.f ? M + logf(L) : -INFINITY;
    }
    const bool got = !failed && tc::mbar_wait(&ms->bar[0], rows_copy ? 1u : 0u);   // the merge copies' phase
    if (!got) atomicOr(&ms->fail, 1);
    __syncthreads();
    const int nq = W / 4;
    for (int t = tid; t < 64 * nq && got; t += THREADS) {
      const int h = t / nq, q4 = t % nq;
      if (h >= H) continue;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int c = 0; c < C; ++c) {
        const float f = mg->f[c][h];
        if (f == 0.f) continue;   // skip empty sources (their blocks may be undefined)
        const float4 v = reinterpret_cast<const float4*>(buf + ((size_t)c * 64 + h) * W)[q4];
        acc.x = fmaf(f, v.x, acc.x);
        acc.y = fmaf(f, v.y, acc.y);
        acc.z = fmaf(f, v.z, acc.z);
        acc.w = fmaf(f, v.w, acc.w);
      }
      const float inv = mg->inv[h];
      *reinterpret_cast<float4*>(out + ((size_t)ur * H + h) * 512 + crank * W + 4 * q4) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    failed = ms->fail != 0;
  }
  if (failed && tid == 0) dsa_flag(dev_err, DSA_DEVERR_TIMEOUT);
  tc::fence_before_sync();
  cluster.sync();   // peers may still read this CTA's shared memory until here
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace

extern "C" size_t mla_decode_attn_workspace(int32_t U, int32_t R, int32_t H, int32_t K) {
  (void)H; (void)K;
  if (U < 1 || R < 1) return 0;
  return (size_t)U * R * MAX_CLUSTER * 64 * 512 * 4;   // one 64 x 512 fp32 partial per CTA
}

namespace {

template <bool GATHER>
int launch_attn(int32_t U, int32_t R, int32_t H, int32_t K, const uint16_t* q_lat, const uint16_t* q_rope,
                const uint8_t* rows, const int32_t* topk_idx, float scale, float* out, float* lse, float* ws_o,
                int32_t* dev_err, const dsa_unit* units, const uint8_t* cls, GatherWs g, cudaStream_t st) {
  static DsaPerDevice pd;
  int dev = 0;
  const int ok = dsa_device_setup(pd, &dev, [](int) {
    DSA_CUDA_TRY(cudaFuncSetAttribute(k_mla_attn<GATHER>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
    DSA_CUDA_TRY(cudaFuncSetAttribute(k_mla_attn<GATHER>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1));
    DSA_CUDA_TRY(dsa_prefer_shared(k_mla_attn<GATHER>));
    return DSA_OK;
  });
  if (ok != DSA_OK) return ok;
  const int C = cluster_ctas(K);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, U * R, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (cudaLaunchKernelEx(&cfg, k_mla_attn<GATHER>, (int)R, (int)H, (int)K, q_lat, q_rope, rows, topk_idx, scale,
                         out, lse, ws_o, dev_err, units, cls, g) != cudaSuccess)
    return DSA_ERR_CUDA;
  return dsa_launch_status();
}

}  // namespace

extern "C" int mla_decode_attn(int32_t U, int32_t R, int32_t H, int32_t K, const uint16_t* q_lat,
                               const uint16_t* q_rope, const uint8_t* rows,
                               const int32_t* topk_idx, float scale, float* out, float* lse,
                               void* ws, size_t ws_bytes, int32_t* dev_err, void* stream) {
  if (!q_lat || !q_rope || !rows || !topk_idx || !out) return DSA_ERR_ARG;
  if (U < 1 || U > 65535 || R < 1 || R > DSA_MAX_ROWS || !(scale > 0.0f)) return DSA_ERR_ARG;
  if (K < 1 || K > NC * MAX_CLUSTER || H < 16 || H > 64 || (H % 16) != 0) return DSA_ERR_SHAPE;
  if ((size_t)U * R > 65535) return DSA_ERR_ARG;
  if (!ws || ws_bytes < mla_decode_attn_workspace(U, R, H, K)) return DSA_ERR_WS;
  // rows and the workspace are read by bulk copies: 16-byte alignment
  if ((reinterpret_cast<uintptr_t>(rows) | reinterpret_cast<uintptr_t>(ws)) & 15u) return DSA_ERR_ARG;
  GatherWs none = {};
  return launch_attn<false>(U, R, H, K, q_lat, q_rope, rows, topk_idx, scale, out, lse, static_cast<float*>(ws),
                            dev_err, nullptr, nullptr, none, static_cast<cudaStream_t>(stream));
}

extern "C" size_t hot_gather_attn_workspace(int32_t U, int32_t R, int32_t H, int32_t K) {
  if (U < 1 || R < 1 || H < 1 || K < 1) return 0;
  return dsa_align(hot_gather_workspace(U, R, K), 256) + mla_decode_attn_workspace(U, R, H, K);
}

extern "C" int hot_gather_attn(const dsa_unit* units, int32_t U, int32_t R, int32_t K, int32_t H, int32_t round,
                               const int32_t* topk_idx, const uint16_t* q_lat, const uint16_t* q_rope,
                               float scale, uint8_t* cls, int32_t* counters, float* out, float* lse, void* ws,
                               size_t ws_bytes, int32_t* dev_err, void* stream) {
  if (!units || !topk_idx || !q_lat || !q_rope || !cls || !counters || !out) return DSA_ERR_ARG;
  if (U < 1 || U > 65535 || R < 1 || R > DSA_MAX_ROWS || !(scale > 0.0f)) return DSA_ERR_ARG;
  if (K < 1 || K > NC * MAX_CLUSTER || H < 16 || H > 64 || (H % 16) != 0) return DSA_ERR_SHAPE;
  if ((size_t)U * R > 65535) return DSA_ERR_ARG;
  if (!ws || ws_bytes < hot_gather_attn_workspace(U, R, H, K)) return DSA_ERR_WS;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return DSA_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* gws = ws;
  float* aws = reinterpret_cast<float*>(static_cast<char*>(ws) + dsa_align(hot_gather_workspace(U, R, K), 256));
  if (dsa_launch_assign(units, U, R, K, round, topk_idx, cls, counters, gws, dev_err, st) != DSA_OK)
    return DSA_ERR_CUDA;
  return launch_attn<true>(U, R, H, K, q_lat, q_rope, nullptr, topk_idx, scale, out, lse, aws, dev_err, units,
                           cls, gather_ws(gws, U, R, K), st);
}
