// A4 + A5: Q8G64 dequantisation and absorbed-MLA decode attention.
//
// [ALG] "Algorithm layer: from attention and KV cache to FFN and MoE",
// section "2. Attention": softmax(Q K^T / sqrt(d_k)) V; section "3. KV Cache":
// MLA keeps the normalised latent and the RoPE part, the latent as INT8 per
// group. [QNT] "Quantization is not a zip file", section "三、基本思路":
// w_hat = scale * q, one scale per group of 64 (G64). [P3] "From 1M total to
// 15+ x 1M", section "起点": a row is 512 B latent + 16 B scales + 128 B RoPE.
//
// Two launches per call:
//  A. k_attn_parts: the K selected rows of a (unit, query row) are cut into
//     chunks of 64 and the chunks into `parts` contiguous runs, one CTA per
//     run (runs sized so that all CTAs fill the stream's SMs once). A CTA
//     keeps the query block (64 heads x 576, fp16) in shared memory and, per
//     chunk:
//  1. bulk TMA copies bring the chunk's rows (up to 64 x 656 B) into a
//     staging buffer: one copy of the compact rows (mla_decode_attn), or with
//     the gather fused in (hot_gather_attn) one copy per row from its source
//     (HBM slot, ring or host mirror), the fills then written to their slots
//     from shared memory; the copies of the next chunk are issued as soon as
//     this chunk is dequantised, so they land while this chunk's products run;
//  2. dequantisation writes an fp16 tile [64 rows][576] (latent int8 * fp16
//     scale rounded once to fp16; RoPE bf16 -> fp16), 128-byte swizzled;
//  3. S = Q K^T on the tensor cores (tcgen05.mma kind::f16, M = 128: the 64
//     heads, the other 64 lanes unused; N = 64 rows, K = 576; fp32 in tensor
//     memory);
//  4. an online softmax per head (a thread holds one head and 32 rows). The
//     running maximum of a head moves only when a chunk exceeds it by more
//     than TAU, so P = exp(x - m) stays below e^TAU in fp16 and the
//     accumulated output is rescaled only then;
//  5. P (fp16, [64 heads][64 rows]) goes over the tile's RoPE part, which S
//     no longer needs, and O^T += V^T P^T accumulates in tensor memory
//     (M = 128 latent dims per block, 4 blocks, N = 64 heads, K = 64 rows):
//     the tile is the K-major B operand of the first product and the
//     MN-major A operand of the second.
//     The run's O (64 x 512 fp32, unnormalised), running maxima and sums go to
//     the run's slot of the workspace (they stay in L2).
//  B. k_attn_merge: one block per (unit, query row) and 32-column slice
//     rescales the runs' outputs by exp(m_c - M) (split softmax), sums them,
//     divides by the total L and writes out (and lse).
// fp16 operands keep 11 significant bits: each operand's rounding is <= 2^-11
// relative, far inside the 1e-3 * max|out| budget. The latent is dequantised
// in fp16 arithmetic: the byte b + 128 placed under the exponent of 1024 is
// the fp16 number 1024 + (b + 128), exactly; subtracting 1152 gives b exactly
// and one fp16 multiply by the scale rounds once, the same value as the fp32
// product rounded to fp16. Waits are bounded; on a timeout the kernel sets
// DSA_DEVERR_TIMEOUT, frees its tensor memory and leaves an empty part (max
// -inf, sum 0) for the merge.
#include <algorithm>
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "gather_internal.cuh"
#include "tc.cuh"

namespace {

constexpr int NC = 64;                          // selected rows per chunk
constexpr int MAX_CTAS = 16;                    // runs per (unit, query row)
constexpr int THREADS = 256;
constexpr int QATOM = 64 * 128;                 // 64 rows x 128 B: query and tile atoms
constexpr int Q_OFF = 0;                        // query block: 9 atoms of 64 dims
constexpr int T_OFF = 9 * QATOM;                // row tile: 9 atoms of 64 dims (atom 8: RoPE, then P)
constexpr int P_OFF = T_OFF + 8 * QATOM;
constexpr int R_OFF = T_OFF + 9 * QATOM;        // staging of the raw rows (64 x 656 B)
constexpr int MISC_OFF = R_OFF + NC * DSA_ROW_BYTES;
constexpr float TAU = 8.f;                      // allowed growth of a chunk maximum before a rescale
// Tensor memory: O^T block b (latent dims 128b..128b+127 in lanes, heads in
// columns) at columns [64b, 64b + 64); S (heads in lanes 0..63, rows in
// columns) at columns [256, 320).
constexpr int TMEM_COLS = 512;
constexpr uint32_t S_COL = 256;
constexpr uint32_t IDESC_QK = tc::idesc_f16_f32(128, NC, 0, 0);
constexpr uint32_t IDESC_PV = tc::idesc_f16_f32(128, 64, 1, 0);
// Partial outputs in the workspace, per (unit, query row) and run: O as 16
// slices of 32 columns, each a contiguous [64 heads][32] block (the merge
// block of a slice reads one block per run), then the 64 row maxima and the
// 64 row sums.
constexpr int SLICE = 32;
constexpr int NSLICE = 512 / SLICE;
constexpr size_t PART_O = (size_t)64 * 512;     // floats per run
constexpr size_t PART_ML = 128;                 // floats per run

struct Misc {
  uint64_t bar_t;             // rows staged (one phase per chunk, compact rows)
  uint64_t bar_s;             // S product done (one phase per chunk)
  uint64_t bar_o;             // O^T product done (one phase per chunk)
  uint32_t tmem;
  int fail;
  int rescale;                // this chunk moved a running maximum: rescale O^T
  uint32_t vmask[NC / 32];    // validity of the chunk's rows
  float m_run[64];            // running maximum per head (logit units)
  float alpha[64];            // this chunk's rescale factor per head
  float red[2][64];           // per half of the rows: maximum, then sum, per head
  const uint8_t* src[NC];     // (gathered rows) source of each row
  uint8_t* dst[NC];           // (gathered rows) hot slot an inserted miss also goes to
};
constexpr int SMEM_BYTES = MISC_OFF + (int)((sizeof(Misc) + 127) / 128 * 128);
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(T_OFF % 1024 == 0 && P_OFF % 1024 == 0 && R_OFF % 16 == 0, "operand alignment");
// the M = 128 query operand reads 64 rows past each atom: the last atom's
// extra rows fall inside the tile
static_assert(T_OFF + QATOM <= MISC_OFF, "padded query rows stay inside shared memory");

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}

// Four int8 (one 32-bit word, lowest byte first) times the fp16 scale s2, as
// two fp16 pairs (bytes 0,1 and 2,3).
__device__ __forceinline__ void dequant4(uint32_t w, __half2 s2, __half2& lo, __half2& hi) {
  const uint32_t x = w ^ 0x80808080u;                  // b + 128 per byte
  const uint32_t a = prmt(x, 0x64646464u, 0x4140u);   // {0x64, b0 + 128}, {0x64, b1 + 128}
  const uint32_t b = prmt(x, 0x64646464u, 0x4342u);
  const __half2 off = __half2half2(__ushort_as_half((unsigned short)0x6480u));   // 1152
  lo = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&a), off), s2);
  hi = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&b), off), s2);
}

__device__ __forceinline__ uint32_t h2_bits(__half2 v) { return *reinterpret_cast<const uint32_t*>(&v); }

// 32 lanes x 32 bits, 32 consecutive columns, from registers (then waits).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Dequantise the staged raw rows [0, nrows) into the fp16 tile (rows past
// nrows: zeros). Work item (row j, piece c): c < 32 is 16 latent bytes (one
// fp16 scale), c >= 32 is 16 RoPE values; consecutive threads take
// consecutive rows. Returns the largest |value| written.
__device__ __forceinline__ float dequant_tile(const uint8_t* raw, uint8_t* tile, int nrows, int tid) {
  __half2 vmax = __float2half2_rn(0.f);
  for (int t = tid; t < NC * 36; t += THREADS) {
    const int j = t % NC, c = t / NC;
    uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = make_uint4(0u, 0u, 0u, 0u);
    if (j < nrows) {
      const uint8_t* row = raw + j * DSA_ROW_BYTES;
      uint32_t o[8];
      if (c < 32) {
        const __half2 s2 = __half2half2(reinterpret_cast<const __half*>(row + 512)[c >> 2]);
        const uint4 w4 = *reinterpret_cast<const uint4*>(row + 16 * c);
        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          __half2 a, b;
          dequant4(w[e], s2, a, b);
          vmax = __hmax2(vmax, __hmax2(__habs2(a), __habs2(b)));
          o[2 * e] = h2_bits(a);
          o[2 * e + 1] = h2_bits(b);
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
    const int d0 = 16 * c;   // first of the item's 16 dims
    uint8_t* atom = tile + (d0 >> 6) * QATOM;
    *reinterpret_cast<uint4*>(atom + tc::sw128_off(j, d0 & 63)) = lo;
    *reinterpret_cast<uint4*>(atom + tc::sw128_off(j, (d0 & 63) + 8)) = hi;
  }
  return fmaxf(__low2float(vmax), __high2float(vmax));
}

// A: one run of chunks [cpp * part, cpp * part + cpp) of (unit, query row)
// ur = blockIdx.y, part = blockIdx.x.
template <bool GATHER>
__global__ void __launch_bounds__(THREADS, 1)
k_attn_parts(int R, int H, int K, int cpp, const uint16_t* __restrict__ q_lat, const uint16_t* __restrict__ q_rope,
             const uint8_t* __restrict__ rows, const int32_t* __restrict__ topk, float scale,
             float* __restrict__ ws_o, float* __restrict__ ws_ml, int32_t* dev_err,
             const dsa_unit* __restrict__ units, const uint8_t* __restrict__ cls, GatherWs g) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint8_t* sQ = sm + Q_OFF;
  uint8_t* sT = sm + T_OFF;
  uint8_t* sP = sm + P_OFF;
  uint8_t* sR = sm + R_OFF;
  Misc* ms = reinterpret_cast<Misc*>(sm + MISC_OFF);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int part = blockIdx.x, ur = blockIdx.y;
  const int nchunks = (K + NC - 1) / NC;
  const int c0 = part * cpp, c1 = min(c0 + cpp, nchunks);
  // softmax threads: warps 0, 1, 4, 5 read S lanes 0..63 (the heads); head
  // 32 * (warp & 1) + lane, rows 32 * (warp >> 2) .. + 31 of the chunk
  const bool sm_warp = (warp & 3) < 2;
  const int hd = 32 * (warp & 1) + lane, rh = warp >> 2;

  if (tid == 0) {
    tc::mbar_init(&ms->bar_t, 1);
    tc::mbar_init(&ms->bar_s, 1);
    tc::mbar_init(&ms->bar_o, 1);
    tc::fence_mbar_init();
    ms->fail = (tc::smem_u32(sm) & 1023u) != 0;   // the tile layouts need 1024-byte alignment
    ms->rescale = 0;
  }
  if (tid < 64) ms->m_run[tid] = -INFINITY;
  if (warp == 0) tc::tmem_alloc(&ms->tmem, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = ms->tmem;
  bool failed = ms->fail != 0;
  pdl_wait();   // everything above touched only this CTA's shared and tensor memory

  // Stage chunk c's rows, completion counted on bar_t (one phase per chunk).
  // Compact rows: one bulk copy (thread 0). Gathered rows: one bulk copy per
  // row from its source (an HBM slot, the ring or the host mirror; 656 bytes,
  // 16-byte aligned), so a host row crosses the link as whole sectors; rows
  // without a source are zero-filled by their thread (the caller's barrier
  // after the wait publishes them).
  auto stage = [&](int c) {
    const int j0 = c * NC, n = min(NC, K - j0);
    if (!GATHER) {
      if (tid == 0) {
        const uint32_t bytes = (uint32_t)n * DSA_ROW_BYTES;
        tc::mbar_arrive_expect_tx(&ms->bar_t, bytes);
        tc::bulk_g2s(sR, rows + ((size_t)ur * K + j0) * DSA_ROW_BYTES, bytes, &ms->bar_t);
      }
    } else {
      if (tid < NC) {
        uint8_t* dst = nullptr;
        const uint8_t* src = nullptr;
        if (tid < n) {
          const size_t ei = (size_t)ur * K + j0 + tid;   // = u * R * K + entry
          const int u = ur / R;
          const dsa_unit& un = units[u];
          const int32_t p = topk[ei];
          const uint8_t cl = cls[ei];
          if (cl == DSA_CLS_HOT) {
            const int32_t sl = un.pos_slot[p];
            if (sl >= 0 && sl < un.slots_n) src = un.slots + (size_t)sl * DSA_ROW_BYTES;
          } else if (cl == DSA_CLS_RING) {
            src = un.ring + (size_t)(p & (DSA_RING_ROWS - 1)) * DSA_ROW_BYTES;
          } else if (cl == DSA_CLS_RAM) {
            src = un.mirror + (size_t)p * DSA_ROW_BYTES;
            const int32_t f = g.fill_of[ei];
            if (f >= 0) {
              const int32_t sl = g.fill_slot[(size_t)u * R * K + f];
              if (sl >= 0 && sl < un.slots_n) dst = un.slots + (size_t)sl * DSA_ROW_BYTES;
            }
          }
        }
        ms->src[tid] = src;
        ms->dst[tid] = dst;
      }
      __syncthreads();
      if (tid == 0) {
        uint32_t bytes = 0;
        for (int jj = 0; jj < n; ++jj) bytes += ms->src[jj] ? (uint32_t)DSA_ROW_BYTES : 0u;
        tc::mbar_arrive_expect_tx(&ms->bar_t, bytes);
      }
      if (tid < n) {
        const uint8_t* src = ms->src[tid];
        uint8_t* d = sR + tid * DSA_ROW_BYTES;
        if (src) {
          tc::bulk_g2s(d, src, DSA_ROW_BYTES, &ms->bar_t);
        } else {
          for (int q = 0; q < DSA_ROW_BYTES / 16; ++q)
            reinterpret_cast<uint4*>(d)[q] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
  };
  if (!failed && c0 < c1) stage(c0);

  // query block: 64 heads x 72 pieces of 8 dims, bf16 -> fp16, K-major swizzled
  constexpr int QCH = 64 * 72 / THREADS;        // 18 pieces per thread
  if (!failed) {
    uint4 qv[QCH];
#pragma unroll
    for (int i = 0; i < QCH; ++i) {
      const int t = tid + i * THREADS;
      const int h = t / 72, c = t % 72;
      qv[i] = make_uint4(0u, 0u, 0u, 0u);
      if (h < H) {
        const size_t qo = (size_t)ur * H + h;
        qv[i] = c < 64 ? *reinterpret_cast<const uint4*>(q_lat + qo * 512 + 8 * c)
                       : *reinterpret_cast<const uint4*>(q_rope + qo * 64 + 8 * (c - 64));
      }
    }
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
      *reinterpret_cast<uint4*>(sQ + (c >> 3) * QATOM + tc::sw128_off(h, 8 * (c & 7))) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (bad) dsa_flag(dev_err, DSA_DEVERR_QRANGE);
  }

  float lsum = 0.f;    // (softmax threads) this thread's share of its head's row sum
  float vmax = 0.f;
  int ns = 0, no = 0;  // (thread 0) product groups committed on bar_s / bar_o
  int nt = (!failed && c0 < c1) ? 1 : 0;   // (thread 0) row copies issued on bar_t
  for (int c = c0; c < c1; ++c) {
    const int i = c - c0;
    const int j0 = c * NC;
    const int nrows = min(NC, K - j0);
    // ---- rows staged; the tile and P are free once the previous chunk's
    //      O^T product is done
    if (!failed) {
      if (!tc::mbar_wait(&ms->bar_t, (uint32_t)(i & 1))) atomicOr(&ms->fail, 1);
      if (i > 0 && !tc::mbar_wait(&ms->bar_o, (uint32_t)((i - 1) & 1))) atomicOr(&ms->fail, 1);
    }
    if (tid < NC) {
      const bool v = tid < nrows && topk[(size_t)ur * K + j0 + tid] >= 0;
      const unsigned b = __ballot_sync(0xffffffffu, v);
      if (lane == 0) ms->vmask[warp] = b;
    }
    tc::fence_after_sync();
    __syncthreads();
    failed = ms->fail != 0;
    // ---- dequantise (an inserted miss's bytes also go to its hot slot)
    if (!failed) {
      if (GATHER) {
        for (int t = tid; t < nrows * 41; t += THREADS) {
          const int jj = t / 41, q = t % 41;
          uint8_t* dst = ms->dst[jj];
          if (dst) *reinterpret_cast<uint4*>(dst + 16 * q) = *reinterpret_cast<const uint4*>(sR + jj * DSA_ROW_BYTES + 16 * q);
        }
      }
      vmax = fmaxf(vmax, dequant_tile(sR, sT, nrows, tid));
    }
    tc::fence_async_shared();
    tc::fence_before_sync();
    __syncthreads();   // staging consumed, tile written
    tc::fence_after_sync();
    failed = ms->fail != 0;
    // ---- the next chunk's rows land while this chunk's products run
    if (!failed && c + 1 < c1) {
      stage(c + 1);
      ++nt;
    }

    // ---- S = Q K^T: heads in lanes 0..63, rows in columns [S_COL, S_COL + 64)
    if (tid == 0 && !failed) {
      const uint32_t ta = tc::smem_u32(sT), qa = tc::smem_u32(sQ);
      for (int kb = 0; kb < 9; ++kb) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          tc::mma_f16(tmem + S_COL, tc::sdesc_sw128(qa + kb * QATOM + kk * 32, 16, 1024),
                      tc::sdesc_sw128(ta + kb * QATOM + kk * 32, 16, 1024), IDESC_QK, (kb | kk) != 0);
      }
      tc::mma_commit(&ms->bar_s);
      ++ns;
    }
    if (!failed && !tc::mbar_wait(&ms->bar_s, (uint32_t)(i & 1))) atomicOr(&ms->fail, 1);
    tc::fence_after_sync();
    __syncthreads();
    failed = ms->fail != 0;

    // ---- online softmax: head hd, rows 32 rh .. 32 rh + 31 of the chunk
    float x[32];
    if (sm_warp && !failed) {
      float v[32];
      tc::tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + S_COL + 32 * rh, v);
      const uint32_t vm = ms->vmask[rh];
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        x[k] = ((vm >> k) & 1u) ? v[k] * scale : -INFINITY;
        mx = fmaxf(mx, x[k]);
      }
      ms->red[rh][hd] = mx;
    }
    __syncthreads();
    if (tid < 64 && !failed) {
      const int h = tid;
      const float cm = fmaxf(ms->red[0][h], ms->red[1][h]);
      const float mo = ms->m_run[h];
      float a = 1.f;
      if (cm > -INFINITY && (mo == -INFINITY || cm > mo + TAU)) {
        a = mo == -INFINITY ? 0.f : __expf(mo - cm);
        ms->m_run[h] = cm;
        if (i > 0) ms->rescale = 1;
      }
      ms->alpha[h] = a;
    }
    __syncthreads();
    if (!failed) {
      if (ms->rescale) {
        // (rare) a running maximum moved: O^T *= alpha per head column. This
        // thread owns latent dim 32 * (warp & 3) + lane of blocks
        // 2 * (warp >> 2) and 2 * (warp >> 2) + 1.
#pragma unroll 1
        for (int b = 0; b < 2; ++b) {
#pragma unroll 1
          for (int x2 = 0; x2 < 2; ++x2) {
            const uint32_t ta =
                tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 64 * (2 * (warp >> 2) + b) + 32 * x2;
            float o[32];
            tc::tmem_ld32(ta, o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] *= ms->alpha[32 * x2 + k];
            tmem_st32(ta, o);
          }
        }
      }
      if (sm_warp) {
        // P = exp(x - m) (0 for masked rows) -> row hd of P, columns 32 rh ..
        const float m = ms->m_run[hd];
        uint32_t pw[16];
        float sum = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float p0 = (x[2 * k] == -INFINITY || m == -INFINITY) ? 0.f : __expf(x[2 * k] - m);
          const float p1 = (x[2 * k + 1] == -INFINITY || m == -INFINITY) ? 0.f : __expf(x[2 * k + 1] - m);
          sum += p0 + p1;
          pw[k] = pack_h2(p0, p1);
        }
        lsum = fmaf(lsum, ms->alpha[hd], sum);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4)
          *reinterpret_cast<uint4*>(sP + tc::sw128_off(hd, 32 * rh + 8 * q4)) =
              make_uint4(pw[4 * q4], pw[4 * q4 + 1], pw[4 * q4 + 2], pw[4 * q4 + 3]);
      }
    }
    tc::fence_async_shared();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0) ms->rescale = 0;
    failed = ms->fail != 0;

    // ---- O^T += V^T P^T: latent dims 128 mb .. + 127 in lanes, heads in columns
    if (tid == 0 && !failed) {
      const uint32_t ta = tc::smem_u32(sT), pa = tc::smem_u32(sP);
      for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
        for (int kk = 0; kk < NC / 16; ++kk)
          tc::mma_f16(tmem + 64 * mb, tc::sdesc_sw128(ta + 2 * mb * QATOM + kk * 2048, QATOM, 1024),
                      tc::sdesc_sw128(pa + kk * 32, 16, 1024), IDESC_PV, (i > 0 || kk > 0));
      }
      tc::mma_commit(&ms->bar_o);
      ++no;
    }
  }

  // ---- the run's O^T, maxima and sums -> its workspace slot
  const int nch = c1 - c0;
  if (nch > 0 && !failed && !tc::mbar_wait(&ms->bar_o, (uint32_t)((nch - 1) & 1))) atomicOr(&ms->fail, 1);
  tc::fence_after_sync();
  __syncthreads();
  failed = ms->fail != 0;
  if (sm_warp) ms->red[rh][hd] = lsum;
  float* gO = ws_o + ((size_t)ur * MAX_CTAS + part) * PART_O;
  if (!failed && nch > 0) {
    // this thread: latent dim d = 128 mb + 32 (warp & 3) + lane of blocks
    // mb = 2 (warp >> 2) + b; for each head the warp stores 32 consecutive
    // floats of slice d / 32
#pragma unroll 1
    for (int b = 0; b < 2; ++b) {
      const int mb = 2 * (warp >> 2) + b;
      float* blk = gO + (size_t)(4 * mb + (warp & 3)) * 64 * SLICE;
#pragma unroll 1
      for (int x2 = 0; x2 < 2; ++x2) {
        float o[32];
        tc::tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 64 * mb + 32 * x2, o);
#pragma unroll
        for (int k = 0; k < 32; ++k) blk[(32 * x2 + k) * SLICE + lane] = o[k];
      }
    }
  }
  __syncthreads();
  if (tid < 64) {   // a failed or empty run leaves an empty part (its O is never read)
    const bool empty = failed || nch <= 0;
    float* ml = ws_ml + ((size_t)ur * MAX_CTAS + part) * PART_ML;
    ml[tid] = empty ? -INFINITY : ms->m_run[tid];
    ml[64 + tid] = empty ? 0.f : ms->red[0][tid] + ms->red[1][tid];
  }
  // (a value whose fp16 rounding reaches 65504, including an overflow)
  if (vmax >= 65504.f) dsa_flag(dev_err, DSA_DEVERR_QRANGE);
  if (failed && tid == 0) {
    dsa_flag(dev_err, DSA_DEVERR_TIMEOUT);
    // nothing may still land in shared memory or run on tensor memory once
    // the CTA is gone
    if (nt > 0) tc::mbar_wait(&ms->bar_t, (uint32_t)((nt - 1) & 1));
    if (ns > 0) tc::mbar_wait(&ms->bar_s, (uint32_t)((ns - 1) & 1));
    if (no > 0) tc::mbar_wait(&ms->bar_o, (uint32_t)((no - 1) & 1));
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// B: merge of the C runs of one (unit, query row), output columns
// [32 s, 32 s + 32) with s = blockIdx.x. The loops over the runs are unrolled
// to MAX_CTAS with predicated loads, so every run's value is in flight at
// once (a run-time bound would chain one L2 round trip per run).
__global__ void __launch_bounds__(256) k_attn_merge(int H, int C, const float* __restrict__ ws_o,
                                                     const float* __restrict__ ws_ml, float* __restrict__ out,
                                                     float* __restrict__ lse) {
  __shared__ float f[MAX_CTAS][64];   // exp(m_c - M) per run and head
  __shared__ float inv[64];           // 1 / L per head
  const int s = blockIdx.x, ur = blockIdx.y, tid = threadIdx.x;
  pdl_wait();
  const float* ml = ws_ml + (size_t)ur * MAX_CTAS * PART_ML;
  if (tid < 64) {
    const int h = tid;
    float mc[MAX_CTAS], lc[MAX_CTAS];
#pragma unroll
    for (int c = 0; c < MAX_CTAS; ++c) {
      mc[c] = c < C ? ml[c * PART_ML + h] : -INFINITY;
      lc[c] = c < C ? ml[c * PART_ML + 64 + h] : 0.f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < MAX_CTAS; ++c) M = fmaxf(M, mc[c]);
    float L = 0.f;
#pragma unroll
    for (int c = 0; c < MAX_CTAS; ++c) {
      const float fc = mc[c] == -INFINITY ? 0.f : __expf(mc[c] - M);
      f[c][h] = fc;
      L += fc * lc[c];
    }
    inv[h] = L > 0.f ? 1.f / L : 0.f;
    if (s == 0 && lse && h < H) lse[(size_t)ur * H + h] = L > 0.f ? M + logf(L) : -INFINITY;
  }
  __syncthreads();
  // 64 heads x 8 float4 columns: two items per thread
  const float* po = ws_o + (size_t)ur * MAX_CTAS * PART_O + (size_t)s * 64 * SLICE;
#pragma unroll 1
  for (int t = tid; t < 64 * (SLICE / 4); t += 256) {
    const int h = t / (SLICE / 4), q4 = t % (SLICE / 4);
    if (h >= H) continue;
    float4 v[MAX_CTAS];
#pragma unroll
    for (int c = 0; c < MAX_CTAS; ++c)
      v[c] = (c < C && f[c][h] != 0.f)   // an empty run's block may be undefined
                 ? reinterpret_cast<const float4*>(po + (size_t)c * PART_O + h * SLICE)[q4]
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int c = 0; c < MAX_CTAS; ++c) {
      const float fc = c < C ? f[c][h] : 0.f;
      acc.x = fmaf(fc, v[c].x, acc.x);
      acc.y = fmaf(fc, v[c].y, acc.y);
      acc.z = fmaf(fc, v[c].z, acc.z);
      acc.w = fmaf(fc, v[c].w, acc.w);
    }
    const float iv = inv[h];
    *reinterpret_cast<float4*>(out + ((size_t)ur * H + h) * 512 + s * SLICE + 4 * q4) =
        make_float4(acc.x * iv, acc.y * iv, acc.z * iv, acc.w * iv);
  }
}

}  // namespace

extern "C" size_t mla_decode_attn_workspace(int32_t U, int32_t R, int32_t H, int32_t K) {
  (void)H; (void)K;
  if (U < 1 || R < 1) return 0;
  // per (unit, query row): MAX_CTAS partial outputs, then their maxima and sums
  return (size_t)U * R * MAX_CTAS * (PART_O + PART_ML) * sizeof(float);
}

namespace {

template <bool GATHER>
int launch_attn(int32_t U, int32_t R, int32_t H, int32_t K, const uint16_t* q_lat, const uint16_t* q_rope,
                const uint8_t* rows, const int32_t* topk_idx, float scale, float* out, float* lse, float* ws,
                int32_t* dev_err, const dsa_unit* units, const uint8_t* cls, GatherWs g, cudaStream_t st) {
  static DsaPerDevice pd;
  int dev = 0;
  const int ok = dsa_device_setup(pd, &dev, [](int) {
    DSA_CUDA_TRY(cudaFuncSetAttribute(k_attn_parts<GATHER>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
    DSA_CUDA_TRY(dsa_prefer_shared(k_attn_parts<GATHER>));
    DSA_CUDA_TRY(dsa_prefer_shared(k_attn_merge));
    return DSA_OK;
  });
  if (ok != DSA_OK) return ok;
  // runs of chunks: as many runs per (unit, query row) as one CTA per SM
  // allows for all of them, at most MAX_CTAS, at least one chunk per run
  const int nchunks = (K + NC - 1) / NC;
  const int64_t UR = (int64_t)U * R;
  const int sms = dsa_stream_sms(st, pd.num_sms[dev]);   // the stream's SM partition, if any
  const int64_t want = std::min<int64_t>(std::min<int64_t>(std::max<int64_t>(1, sms / UR), nchunks), MAX_CTAS);
  const int cpp = (int)((nchunks + want - 1) / want);
  const int parts = (nchunks + cpp - 1) / cpp;
  float* ws_o = ws;
  float* ws_ml = ws + (size_t)UR * MAX_CTAS * PART_O;
  if (launch_pdl(k_attn_parts<GATHER>, dim3(parts, (unsigned)UR), dim3(THREADS), SMEM_BYTES, st, (int)R, (int)H,
                 (int)K, cpp, q_lat, q_rope, rows, topk_idx, scale, ws_o, ws_ml, dev_err, units, cls, g) != DSA_OK)
    return DSA_ERR_CUDA;
  return launch_pdl(k_attn_merge, dim3(NSLICE, (unsigned)UR), dim3(256), 0, st, (int)H, parts,
                    static_cast<const float*>(ws_o), static_cast<const float*>(ws_ml), out, lse);
}

}  // namespace

extern "C" int mla_decode_attn(int32_t U, int32_t R, int32_t H, int32_t K, const uint16_t* q_lat,
                               const uint16_t* q_rope, const uint8_t* rows,
                               const int32_t* topk_idx, float scale, float* out, float* lse,
                               void* ws, size_t ws_bytes, int32_t* dev_err, void* stream) {
  if (!q_lat || !q_rope || !rows || !topk_idx || !out) return DSA_ERR_ARG;
  if (U < 1 || U > 65535 || R < 1 || R > DSA_MAX_ROWS || !(scale > 0.0f)) return DSA_ERR_ARG;
  if (K < 1 || K > DSA_MAX_ATTN_K || H < 16 || H > 64 || (H % 16) != 0) return DSA_ERR_SHAPE;
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
  if (K < 1 || K > DSA_MAX_ATTN_K || H < 16 || H > 64 || (H % 16) != 0) return DSA_ERR_SHAPE;
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
