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
//  A. k_mla_attn: ceil(K / 128) CTAs per (unit, query row); CTA c owns the
//     selected rows [128c, 128c + 128):
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
//     X as the A operand of PV, its 64 head rows written twice (rows 64..127
//     repeat them) so that tensor-memory lanes 64..127 of O repeat lanes
//     0..63 and all eight warps can read O out;
//  6. the CTA's O (64 x 512 fp32), row max and row sum go to its slot of the
//     workspace (they stay in L2).
//  B. k_attn_merge: one block per (unit, query row) and 32-column slice
//     rescales the CTAs' partial outputs by exp(m_c - M) (split softmax),
//     sums them, divides by the total L and writes out (and lse).
// fp16 operands keep 11 significant bits: each operand's rounding is <= 2^-11
// relative, far inside the 1e-3 * max|out| budget. The latent is
// dequantised in fp16 arithmetic: the byte b + 128 placed under the exponent
// of 1024 is the fp16 number 1024 + (b + 128), exactly; subtracting 1152 gives
// b exactly and one fp16 multiply by the scale rounds once, the same value as
// the fp32 product rounded to fp16. Waits are bounded; on a timeout the kernel
// sets DSA_DEVERR_TIMEOUT, frees its tensor memory and leaves an empty part
// (max -inf, sum 0) for the merge.
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "gather_internal.cuh"
#include "tc.cuh"

namespace {

constexpr int NC = 128;                         // selected rows per CTA
constexpr int MAX_CTAS = 16;                    // per (unit, query row) -> K <= 2048
constexpr int THREADS = 256;
constexpr int QATOM = 8192;                     // 64 rows x 128 B (query atoms)
constexpr int PATOM = 16384;                    // 128 rows x 128 B (P atoms: the 64 rows twice)
constexpr int BATOM = NC * 128;                 // 128 rows x 128 B (row-tile atoms)
constexpr int X_OFF = 0;
constexpr int X_BYTES = NC * DSA_ROW_BYTES;     // 83,968 = 82 KB
constexpr int Y_OFF = X_BYTES;
constexpr int Y_BYTES = 9 * BATOM;              // 147,456
constexpr int MISC_OFF = Y_OFF + Y_BYTES;
constexpr int SMEM_BYTES = MISC_OFF + 1024;     // 232,448: the whole opt-in budget
constexpr int TMEM_COLS = 512;
constexpr uint32_t IDESC_QK = tc::idesc_f16_f32(128, NC, 0, 0);
constexpr uint32_t IDESC_PV = tc::idesc_f16_f32(128, 256, 0, 1);
// Partial outputs in the workspace, per (unit, query row) and CTA: O as 16
// slices of 32 columns, each a contiguous [64 heads][32] block (the merge
// block of a slice reads one block per CTA), then the 64 row maxima and the
// 64 row sums.
constexpr int SLICE = 32;
constexpr int NSLICE = 512 / SLICE;
constexpr size_t PART_O = (size_t)64 * 512;     // floats per CTA
constexpr size_t PART_ML = 128;                 // floats per CTA

static_assert(X_BYTES % 1024 == 0, "region X must keep Y 1024-aligned");
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
constexpr int SMX_OFF = 2 * PATOM;
static_assert(SMX_OFF + (int)sizeof(SoftmaxScratch) <= X_BYTES, "softmax scratch");
static_assert(sizeof(Misc) <= 1024, "misc block");
static_assert(8 * 32 * 36 * 4 <= Y_BYTES, "O transpose buffers");

// CTAs per (unit, query row) for K selected rows.
inline int attn_ctas(int K) { return (K + NC - 1) / NC; }

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
           float* __restrict__ ws_o, float* __restrict__ ws_ml, int32_t* dev_err,
           const dsa_unit* __restrict__ units, const uint8_t* __restrict__ cls, GatherWs g) {
  extern __shared__ __align__(1024) uint8_t sm[];
  const int crank = blockIdx.x;
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

  // The rows of a CTA arrive by one bulk copy on phase 0 of bar[0].
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
    __half2 vmax = __float2half2_rn(0.f);   // largest |dequantised value| of this thread
    for (int t = tid; t < NC * 36; t += THREADS) {
      const int j = t % NC, c = t / NC;     // consecutive threads: consecutive rows
      uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
      if (j < nrows) {
        const uint8_t* row = sX + j * DSA_ROW_BYTES;
        uint32_t o[8];
        if (c < 32) {
          const __half2 s2 = __half2half2(reinterpret_cast<const __half*>(row + 512)[c >> 2]);
          const uint4 raw = *reinterpret_cast<const uint4*>(row + 16 * c);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
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
      const int d0 = 16 * c;
      uint8_t* atom = sY + (d0 >> 6) * BATOM;
      *reinterpret_cast<uint4*>(atom + tc::sw128_off(j, d0 & 63)) = lo;
      *reinterpret_cast<uint4*>(atom + tc::sw128_off(j, (d0 & 63) + 8)) = hi;
    }
    // (a value whose fp16 rounding reaches 65504, including an overflow)
    if (fmaxf(__low2float(vmax), __high2float(vmax)) >= 65504.f) dsa_flag(dev_err, DSA_DEVERR_QRANGE);
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
      *reinterpret_cast<uint4*>(sX + half * PATOM + tc::sw128_off(hr, 8 * c8)) = v;
      *reinterpret_cast<uint4*>(sX + half * PATOM + tc::sw128_off(hr + 64, 8 * c8)) = v;
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
        const uint64_t ad = tc::sdesc_sw128(pa + (kk >> 2) * PATOM + (kk & 3) * 32, 16, 1024);
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

  // ---- this CTA's O (64 x 512 fp32) to its slot of the workspace (L2). Warp
  //      w reads tensor-memory lane quarter w & 3 (heads 32 * (w & 1) + lane:
  //      lanes 64..127 repeat 0..63) and 128-column range 2 * (w >> 2) +
  //      ((w & 3) >> 1). Each 32 x 32 block goes through a padded shared-memory
  //      transpose so every store writes whole 128-byte rows of a slice.
  float* gO = ws_o + ((size_t)ur * MAX_CTAS + crank) * PART_O;
  if (!failed) {
    const int q = warp & 3;
    const int hb = 32 * (q & 1);
    const int c0 = 128 * (2 * (warp >> 2) + (q >> 1));
    float* tb = reinterpret_cast<float*>(sY) + warp * 32 * 36;   // [32][36]
    for (int c = 0; c < 4; ++c) {
      float v[32];
      const int col = c0 + 32 * c;                       // first column of the block = slice start
      tc::tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + col, v);
#pragma unroll
      for (int i = 0; i < 8; ++i)
        reinterpret_cast<float4*>(tb + lane * 36)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      __syncwarp();
      float* blk = gO + (size_t)(col / SLICE) * 64 * SLICE;
#pragma unroll
      for (int r4 = 0; r4 < 8; ++r4) {
        const int r = 4 * r4 + (lane >> 3);              // row within the block
        const float4 x = reinterpret_cast<const float4*>(tb + r * 36)[lane & 7];
        reinterpret_cast<float4*>(blk + (size_t)(hb + r) * SLICE)[lane & 7] = x;
      }
      __syncwarp();
    }
  }
  failed = failed || ms->fail != 0;
  if (tid < 64) {   // a failed CTA leaves an empty part (its O is never read)
    float* ml = ws_ml + ((size_t)ur * MAX_CTAS + crank) * PART_ML;
    ml[tid] = failed ? -INFINITY : ms->m[tid];
    ml[64 + tid] = failed ? 0.f : ms->l[tid];
  }
  if (failed && tid == 0) dsa_flag(dev_err, DSA_DEVERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// B: merge of the C parts of one (unit, query row), output columns
// [32 s, 32 s + 32) with s = blockIdx.x.
__global__ void __launch_bounds__(256) k_attn_merge(int H, int C, const float* __restrict__ ws_o,
                                                     const float* __restrict__ ws_ml, float* __restrict__ out,
                                                     float* __restrict__ lse) {
  __shared__ float f[MAX_CTAS][64];   // exp(m_c - M) per part and head
  __shared__ float inv[64];           // 1 / L per head
  const int s = blockIdx.x, ur = blockIdx.y, tid = threadIdx.x;
  pdl_wait();
  const float* ml = ws_ml + (size_t)ur * MAX_CTAS * PART_ML;
  if (tid < 64) {
    const int h = tid;
    float M = -INFINITY;
    for (int c = 0; c < C; ++c) M = fmaxf(M, ml[c * PART_ML + h]);
    float L = 0.f;
    for (int c = 0; c < C; ++c) {
      const float mc = ml[c * PART_ML + h];
      const float fc = mc == -INFINITY ? 0.f : __expf(mc - M);
      f[c][h] = fc;
      L += fc * ml[c * PART_ML + 64 + h];
    }
    inv[h] = L > 0.f ? 1.f / L : 0.f;
    if (s == 0 && lse && h < H) lse[(size_t)ur * H + h] = L > 0.f ? M + logf(L) : -INFINITY;
  }
  __syncthreads();
  // 64 heads x 8 float4 columns
  const float* po = ws_o + (size_t)ur * MAX_CTAS * PART_O + (size_t)s * 64 * SLICE;
  for (int t = tid; t < 64 * (SLICE / 4); t += 256) {
    const int h = t / (SLICE / 4), q4 = t % (SLICE / 4);
    if (h >= H) continue;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < C; ++c) {
      const float fc = f[c][h];
      if (fc == 0.f) continue;   // an empty part (its block may be undefined)
      const float4 v = reinterpret_cast<const float4*>(po + (size_t)c * PART_O + h * SLICE)[q4];
      acc.x = fmaf(fc, v.x, acc.x);
      acc.y = fmaf(fc, v.y, acc.y);
      acc.z = fmaf(fc, v.z, acc.z);
      acc.w = fmaf(fc, v.w, acc.w);
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
    DSA_CUDA_TRY(cudaFuncSetAttribute(k_mla_attn<GATHER>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
    DSA_CUDA_TRY(dsa_prefer_shared(k_mla_attn<GATHER>));
    DSA_CUDA_TRY(dsa_prefer_shared(k_attn_merge));
    return DSA_OK;
  });
  if (ok != DSA_OK) return ok;
  const int C = attn_ctas(K);
  const size_t UR = (size_t)U * R;
  float* ws_o = ws;
  float* ws_ml = ws + UR * MAX_CTAS * PART_O;
  if (launch_pdl(k_mla_attn<GATHER>, dim3(C, (unsigned)UR), dim3(THREADS), SMEM_BYTES, st, (int)R, (int)H, (int)K,
                 q_lat, q_rope, rows, topk_idx, scale, ws_o, ws_ml, dev_err, units, cls, g) != DSA_OK)
    return DSA_ERR_CUDA;
  return launch_pdl(k_attn_merge, dim3(NSLICE, (unsigned)UR), dim3(256), 0, st, (int)H, C,
                    static_cast<const float*>(ws_o), static_cast<const float*>(ws_ml), out, lse);
}

}  // namespace

extern "C" int mla_decode_attn(int32_t U, int32_t R, int32_t H, int32_t K, const uint16_t* q_lat,
                               const uint16_t* q_rope, const uint8_t* rows,
                               const int32_t* topk_idx, float scale, float* out, float* lse,
                               void* ws, size_t ws_bytes, int32_t* dev_err, void* stream) {
  if (!q_lat || !q_rope || !rows || !topk_idx || !out) return DSA_ERR_ARG;
  if (U < 1 || U > 65535 || R < 1 || R > DSA_MAX_ROWS || !(scale > 0.0f)) return DSA_ERR_ARG;
  if (K < 1 || K > NC * MAX_CTAS || H < 16 || H > 64 || (H % 16) != 0) return DSA_ERR_SHAPE;
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
  if (K < 1 || K > NC * MAX_CTAS || H < 16 || H > 64 || (H % 16) != 0) return DSA_ERR_SHAPE;
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
