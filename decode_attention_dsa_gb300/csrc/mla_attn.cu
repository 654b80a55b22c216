// A4 + A5: Q8G64 dequantisation and absorbed-MLA decode attention.
//
// [ALG] "Algorithm layer: from attention and KV cache to FFN and MoE",
// section "2. Attention": softmax(Q K^T / sqrt(d_k)) V; section "3. KV Cache":
// MLA keeps the normalised latent and the RoPE part, the latent as INT8 per
// group. [QNT] "Quantization is not a zip file", section "三、基本思路":
// w_hat = scale * q, one scale per group of 64 (G64). [P3] "From 1M total to
// 15+ x 1M", section "起点": a row is 512 B latent + 16 B scales + 128 B RoPE.
//
// Split-K decode attention on the 5th-generation tensor cores:
//  * one CTA (128 threads) per chunk of NC = 64 selected rows of one
//    (unit, query row); the chunk's 64 x 656 B of rows arrive with one 1-D
//    bulk TMA copy into shared memory;
//  * dequantisation writes one fp16 tile [64 rows][576] (latent
//    int8 * fp16 scale, rounded once to fp16; RoPE bf16 -> fp16) in the
//    K-major 128-byte-swizzled layout. The same bytes are the K-major B operand
//    of S = Q K^T and, read as an MN-major operand, the B operand of O = P V;
//  * tcgen05.mma kind::f16 (M = 128 rows of query heads, 64 real, N = 64 for
//    S and 2 x 256 for O, fp32 accumulators in tensor memory), issued by one
//    thread and tracked with tcgen05.commit on an mbarrier;
//  * softmax of the chunk in registers (one thread per head row read from
//    TMEM), P written back to shared memory in fp16 as the A operand of PV;
//  * the unnormalised chunk output with its max and sum goes to the
//    workspace; k_attn_combine merges the chunks.
// fp16 operands keep 11 significant bits (bf16 would keep 8): the relative
// rounding of each operand is <= 2^-12, far inside the 1e-3 * max|out| budget.
// Every wait is bounded; on a timeout the kernel sets DSA_DEVERR_TIMEOUT,
// frees its tensor memory and returns.
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"
#include "tc.cuh"

namespace {

constexpr int NC = 64;                       // selected rows per CTA
constexpr int THREADS = 128;
constexpr int KD = 576;                      // key width
constexpr int ATOM = 8192;                   // one 64-wide K atom of 64 rows (bytes)
constexpr int Q_OFF = 0;                     // Q tile: 9 atoms of 64 head rows
constexpr int B_OFF = 9 * ATOM;              // row tile: 9 atoms of 64 key rows
constexpr int RAW_OFF = 18 * ATOM;           // raw rows (TMA destination); P tile aliases it
constexpr int RAW_BYTES = NC * DSA_ROW_BYTES;
constexpr int MISC_OFF = RAW_OFF + ((RAW_BYTES + 1023) / 1024) * 1024;
constexpr int SMEM_BYTES = MISC_OFF + 1024 + 1024;   // + misc + alignment slack
constexpr int TMEM_COLS = 512;
constexpr int COMB_THREADS = 128;
constexpr uint32_t IDESC_QK = tc::idesc_f16_f32(128, NC, 0, 0);
constexpr uint32_t IDESC_PV = tc::idesc_f16_f32(128, 256, 0, 1);

struct AttnWs {
  float* o;   // [UR][nsplit][H][512] unnormalised chunk outputs
  float* m;   // [UR][nsplit][H] chunk max logit
  float* l;   // [UR][nsplit][H] chunk sum of exp(logit - m)
};

inline int n_split(int K) { return (K + NC - 1) / NC; }

inline AttnWs attn_ws(void* ws, int U, int R, int H, int K) {
  const size_t ns = (size_t)n_split(K);
  const size_t a = dsa_align((size_t)U * R * ns * H * 512 * 4, 256);
  const size_t b = dsa_align((size_t)U * R * ns * H * 4, 256);
  char* c = static_cast<char*>(ws);
  return AttnWs{reinterpret_cast<float*>(c), reinterpret_cast<float*>(c + a),
                reinterpret_cast<float*>(c + a + b)};
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  const __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(THREADS, 1)
k_attn_tc(int R, int H, int K, const uint16_t* __restrict__ q_lat, const uint16_t* __restrict__ q_rope,
          const uint8_t* __restrict__ rows, const int32_t* __restrict__ topk, float scale,
          AttnWs ws, int32_t* dev_err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + Q_OFF;
  uint8_t* sB = sm + B_OFF;
  uint8_t* sRaw = sm + RAW_OFF;
  uint8_t* sP = sRaw;                                   // aliases the raw rows after dequant
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + MISC_OFF);        // [0] TMA, [1] MMA
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + MISC_OFF + 16);
  int* s_valid = reinterpret_cast<int*>(sm + MISC_OFF + 32);         // [NC]
  int* s_fail = reinterpret_cast<int*>(sm + MISC_OFF + 32 + 4 * NC);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x, ur = blockIdx.y, nsplit = gridDim.x;
  const int j0 = split * NC;
  const int nrows = min(NC, K - j0);

  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::fence_mbar_init();
    *s_fail = 0;
  }
  if (warp == 0) tc::tmem_alloc(s_tmem, TMEM_COLS);
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *s_tmem;

  if (tid == 0) {
    const uint32_t bytes = (uint32_t)nrows * DSA_ROW_BYTES;
    tc::mbar_arrive_expect_tx(&bar[0], bytes);
    tc::bulk_g2s(sRaw, rows + ((size_t)ur * K + j0) * DSA_ROW_BYTES, bytes, &bar[0]);
  }
  if (tid < NC) s_valid[tid] = (tid < nrows) && topk[(size_t)ur * K + j0 + tid] >= 0;
  if (!tc::mbar_wait(&bar[0], 0)) atomicOr(s_fail, 1);
  __syncthreads();
  bool failed = *s_fail != 0;

  // ---- dequantise: 16-byte latent chunks (16 int8 -> 16 fp16) and RoPE chunks
  if (!failed) {
    bool bad = false;
    for (int t = tid; t < NC * 36; t += THREADS) {
      const int j = t / 36, c = t % 36;
      uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
      if (j < nrows) {
        const uint8_t* row = sRaw + j * DSA_ROW_BYTES;
        if (c < 32) {
          const int g = c >> 2;
          const float s = __half2float(__ushort_as_half(reinterpret_cast<const uint16_t*>(row + 512)[g]));
          const uint4 raw = *reinterpret_cast<const uint4*>(row + 16 * c);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t o[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a0 = (float)(int8_t)(w[e] & 0xFF) * s;
            const float a1 = (float)(int8_t)((w[e] >> 8) & 0xFF) * s;
            const float a2 = (float)(int8_t)((w[e] >> 16) & 0xFF) * s;
            const float a3 = (float)(int8_t)(w[e] >> 24) * s;
            bad |= fabsf(a0) >= 65504.f || fabsf(a1) >= 65504.f || fabsf(a2) >= 65504.f || fabsf(a3) >= 65504.f;
            o[2 * e] = pack_h2(a0, a1);
            o[2 * e + 1] = pack_h2(a2, a3);
          }
          lo = make_uint4(o[0], o[1], o[2], o[3]);
          hi = make_uint4(o[4], o[5], o[6], o[7]);
        } else {
          const uint4 raw = *reinterpret_cast<const uint4*>(row + 528 + 32 * (c - 32));
          const uint4 raw2 = *reinterpret_cast<const uint4*>(row + 528 + 32 * (c - 32) + 16);
          const uint32_t w[8] = {raw.x, raw.y, raw.z, raw.w, raw2.x, raw2.y, raw2.z, raw2.w};
          uint32_t o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = pack_h2(bf16_lo(w[e]), bf16_hi(w[e]));
          lo = make_uint4(o[0], o[1], o[2], o[3]);
          hi = make_uint4(o[4], o[5], o[6], o[7]);
        }
      }
      // 16 consecutive key dims d0 = 16 * c: atom d0 / 64, in-atom k = d0 % 64
      const int d0 = 16 * c;
      uint8_t* atom = sB + (d0 >> 6) * ATOM;
      *reinterpret_cast<uint4*>(atom + tc::sw128_off(j, d0 & 63)) = lo;
      *reinterpret_cast<uint4*>(atom + tc::sw128_off(j, (d0 & 63) + 8)) = hi;
    }
    if (bad) dsa_flag(dev_err, DSA_DEVERR_QRANGE);
  }
  __syncthreads();   // raw rows are dead from here on (P reuses them)

  uint32_t mma_phase = 0;
  for (int hg = 0; hg < H && !failed; hg += 64) {
    // ---- query block: heads hg .. hg + 63 (rows past H are zero)
    {
      bool bad = false;
      for (int t = tid; t < 64 * 72; t += THREADS) {
        const int hr = t / 72, c = t % 72;     // 72 chunks of 8 dims per head
        const int h = hg + hr;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (h < H) {
          const size_t qo = (size_t)ur * H + h;
          const uint4 raw = c < 64 ? *reinterpret_cast<const uint4*>(q_lat + qo * 512 + 8 * c)
                                   : *reinterpret_cast<const uint4*>(q_rope + qo * 64 + 8 * (c - 64));
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t o[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a = bf16_lo(w[e]), b = bf16_hi(w[e]);
            bad |= fabsf(a) >= 65504.f || fabsf(b) >= 65504.f;
            o[e] = pack_h2(a, b);
          }
          v = make_uint4(o[0], o[1], o[2], o[3]);
        }
        const int d0 = 8 * c;
        *reinterpret_cast<uint4*>(sQ + (d0 >> 6) * ATOM + tc::sw128_off(hr, d0 & 63)) = v;
      }
      if (bad) dsa_flag(dev_err, DSA_DEVERR_QRANGE);
    }
    tc::fence_async_shared();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // ---- S = Q K^T into TMEM columns [0, 64)
    if (tid == 0) {
      const uint32_t qa = tc::smem_u32(sQ), ba = tc::smem_u32(sB);
      uint32_t acc = 0;
      for (int kb = 0; kb < 9; ++kb) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = tc::sdesc_sw128(qa + kb * ATOM + kk * 32, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(ba + kb * ATOM + kk * 32, 16, 1024);
          tc::mma_f16(tmem, ad, bd, IDESC_QK, acc);
          acc = 1;
        }
      }
      tc::mma_commit(&bar[1]);
    }
    if (!tc::mbar_wait(&bar[1], mma_phase & 1)) atomicOr(s_fail, 1);
    ++mma_phase;
    tc::fence_after_sync();
    // ---- softmax of the chunk: warps 0 and 1 hold head rows 0..63
    if (warp < 2) {
      float s[64];
      float tmp[32];
      tc::tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16), tmp);
#pragma unroll
      for (int i = 0; i < 32; ++i) s[i] = tmp[i];
      tc::tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32, tmp);
#pragma unroll
      for (int i = 0; i < 32; ++i) s[32 + i] = tmp[i];
      const int hr = 32 * warp + lane;
      float m = -INFINITY;
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        s[j] = s_valid[j] ? s[j] * scale : -INFINITY;
        m = fmaxf(m, s[j]);
      }
      float l = 0.f;
#pragma unroll
      for (int j = 0; j < NC; ++j) {
        s[j] = (m == -INFINITY) ? 0.f : __expf(s[j] - m);
        l += s[j];
      }
#pragma unroll
      for (int c8 = 0; c8 < NC / 8; ++c8) {
        const uint4 v = make_uint4(pack_h2(s[8 * c8], s[8 * c8 + 1]), pack_h2(s[8 * c8 + 2], s[8 * c8 + 3]),
                                   pack_h2(s[8 * c8 + 4], s[8 * c8 + 5]), pack_h2(s[8 * c8 + 6], s[8 * c8 + 7]));
        *reinterpret_cast<uint4*>(sP + tc::sw128_off(hr, 8 * c8)) = v;
      }
      const int h = hg + hr;
      if (h < H) {
        const size_t mo = ((size_t)ur * nsplit + split) * H + h;
        ws.m[mo] = m;
        ws.l[mo] = l;
      }
    }
    tc::fence_async_shared();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    failed = *s_fail != 0;
    if (failed) break;
    // ---- O = P V into TMEM columns [0, 512)
    if (tid == 0) {
      const uint32_t pa = tc::smem_u32(sP), ba = tc::smem_u32(sB);
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int kk = 0; kk < NC / 16; ++kk) {
          const uint64_t ad = tc::sdesc_sw128(pa + kk * 32, 16, 1024);
          const uint64_t bd = tc::sdesc_sw128(ba + half * 4 * ATOM + kk * 2048, ATOM, 1024);
          tc::mma_f16(tmem + half * 256, ad, bd, IDESC_PV, kk > 0);
        }
      }
      tc::mma_commit(&bar[1]);
    }
    if (!tc::mbar_wait(&bar[1], mma_phase & 1)) atomicOr(s_fail, 1);
    ++mma_phase;
    tc::fence_after_sync();
    if (warp < 2) {
      const int h = hg + 32 * warp + lane;
      float* o = ws.o + (((size_t)ur * nsplit + split) * H + (h < H ? h : 0)) * 512;
      for (int c = 0; c < 16; ++c) {
        float v[32];
        tc::tmem_ld32(tmem + ((uint32_t)(32 * warp) << 16) + 32 * c, v);
        if (h < H) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            reinterpret_cast<float4*>(o + 32 * c)[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    failed = *s_fail != 0;
  }
  if (failed && tid == 0) dsa_flag(dev_err, DSA_DEVERR_TIMEOUT);
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// Merge the chunk outputs of one (unit, query row, head): thread -> 4 dims.
__global__ void __launch_bounds__(COMB_THREADS)
k_attn_combine(int H, int nsplit, AttnWs ws, float* __restrict__ out, float* __restrict__ lse) {
  const int ur = blockIdx.y, h = blockIdx.x, t = threadIdx.x;
  __shared__ float s_f[256];
  __shared__ float s_L;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ws.m[((size_t)ur * nsplit + s) * H + h]);
  for (int s = t; s < nsplit; s += COMB_THREADS) {
    const float m = ws.m[((size_t)ur * nsplit + s) * H + h];
    s_f[s] = (m == -INFINITY) ? 0.f : __expf(m - M);
  }
  __syncthreads();
  if (t == 0) {
    float L = 0.f;
    for (int s = 0; s < nsplit; ++s) L += ws.l[((size_t)ur * nsplit + s) * H + h] * s_f[s];
    s_L = L;
  }
  __syncthreads();
  const float L = s_L;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s = 0; s < nsplit; ++s) {
    const float f = s_f[s];
    if (f == 0.f) continue;
    const float4 v = reinterpret_cast<const float4*>(ws.o + (((size_t)ur * nsplit + s) * H + h) * 512)[t];
    acc.x = fmaf(f, v.x, acc.x);
    acc.y = fmaf(f, v.y, acc.y);
    acc.z = fmaf(f, v.z, acc.z);
    acc.w = fmaf(f, v.w, acc.w);
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  reinterpret_cast<float4*>(out + ((size_t)ur * H + h) * 512)[t] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  if (lse && t == 0) lse[(size_t)ur * H + h] = L > 0.f ? M + logf(L) : -INFINITY;
}

}  // namespace

extern "C" size_t mla_decode_attn_workspace(int32_t U, int32_t R, int32_t H, int32_t K) {
  if (U < 1 || R < 1 || H < 1 || K < 1) return 0;
  const size_t ns = (size_t)n_split(K);
  return dsa_align((size_t)U * R * ns * H * 512 * 4, 256) +
         2 * dsa_align((size_t)U * R * ns * H * 4, 256);
}

extern "C" int mla_decode_attn(int32_t U, int32_t R, int32_t H, int32_t K, const uint16_t* q_lat,
                               const uint16_t* q_rope, const uint8_t* rows,
                               const int32_t* topk_idx, float scale, float* out, float* lse,
                               void* ws, size_t ws_bytes, int32_t* dev_err, void* stream) {
  if (!q_lat || !q_rope || !rows || !topk_idx || !out) return DSA_ERR_ARG;
  if (U < 1 || U > 65535 || R < 1 || R > DSA_MAX_ROWS || !(scale > 0.0f)) return DSA_ERR_ARG;
  if (K < 1 || K > DSA_MAX_K || H < 16 || H > 128 || (H % 16) != 0) return DSA_ERR_SHAPE;
  if (!ws || ws_bytes < mla_decode_attn_workspace(U, R, H, K)) return DSA_ERR_WS;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  AttnWs a = attn_ws(ws, U, R, H, K);
  static bool attr_done = false;
  if (!attr_done) {
    DSA_CUDA_TRY(cudaFuncSetAttribute(k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      SMEM_BYTES));
    attr_done = true;
  }
  const int ns = n_split(K);
  if (ns > 256) return DSA_ERR_SHAPE;
  k_attn_tc<<<dim3(ns, U * R), THREADS, SMEM_BYTES, st>>>(R, H, K, q_lat, q_rope, rows, topk_idx,
                                                          scale, a, dev_err);
  if (dsa_launch_status() != DSA_OK) return DSA_ERR_CUDA;
  k_attn_combine<<<dim3(H, U * R), COMB_THREADS, 0, st>>>(H, ns, a, out, lse);
  return dsa_launch_status();
}
