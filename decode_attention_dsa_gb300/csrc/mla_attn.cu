// A4 + A5: Q8G64 dequantisation and absorbed-MLA decode attention.
//
// [ALG] "Algorithm layer: from attention and KV cache to FFN and MoE",
// section "2. Attention": softmax(Q K^T / sqrt(d_k)) V; section "3. KV Cache":
// MLA keeps the normalised latent and the RoPE part, the latent as INT8 per
// group. [QNT] "Quantization is not a zip file", section "三、基本思路":
// w_hat = scale * q, one scale per group of 64 (G64). [P3] "From 1M total to
// 15+ x 1M", section "起点": a row is 512 B latent + 16 B scales + 128 B RoPE.
//
// Split-K decode attention: each CTA takes a chunk of ATT_KC selected rows of
// one (unit, query row), dequantises them exactly into fp32 in shared memory
// (int8 x fp16 is exact in fp32), computes the logits of every head over the
// 576-wide key, a chunk-local softmax (max m, sum l) and the unnormalised
// P V partial. A second launch merges the chunks with the usual max/sum
// rescaling and writes out and lse.
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"

namespace {

constexpr int ATT_THREADS = 256;
constexpr int ATT_KC = 32;          // selected rows per CTA
constexpr int ATT_HG = 64;          // heads per pass
constexpr int KD = 576;             // key width: 512 latent + 64 RoPE
constexpr int KSTR = 577;           // fp32 row stride of the dequantised chunk (odd: no bank conflicts)
constexpr int QSTR = 578;           // bf16 row stride of the query block
constexpr int COMB_THREADS = 512;

struct AttnWs {
  float* o;   // [UR][nsplit][H][512]
  float* m;   // [UR][nsplit][H]
  float* l;   // [UR][nsplit][H]
};

inline int n_split(int K) { return (K + ATT_KC - 1) / ATT_KC; }

inline AttnWs attn_ws(void* ws, int U, int R, int H, int K) {
  const size_t ns = (size_t)n_split(K);
  const size_t a = dsa_align((size_t)U * R * ns * H * 512 * 4, 256);
  const size_t b = dsa_align((size_t)U * R * ns * H * 4, 256);
  char* c = static_cast<char*>(ws);
  return AttnWs{reinterpret_cast<float*>(c), reinterpret_cast<float*>(c + a),
                reinterpret_cast<float*>(c + a + b)};
}

inline size_t attn_smem() {
  return (size_t)ATT_KC * KSTR * 4 + (size_t)ATT_HG * QSTR * 2 + (size_t)ATT_HG * ATT_KC * 4 +
         ATT_KC * 4;
}

__global__ void __launch_bounds__(ATT_THREADS)
k_attn_partial(int R, int H, int K, const uint16_t* __restrict__ q_lat,
               const uint16_t* __restrict__ q_rope, const uint8_t* __restrict__ rows,
               const int32_t* __restrict__ topk, float scale, AttnWs ws, int32_t* dev_err) {
  extern __shared__ float sm[];
  float* kc = sm;                                              // [KC][KSTR]
  uint16_t* sq = reinterpret_cast<uint16_t*>(kc + ATT_KC * KSTR);  // [HG][QSTR]
  float* sp = reinterpret_cast<float*>(sq + ATT_HG * QSTR);    // [HG][KC]
  int* svalid = reinterpret_cast<int*>(sp + ATT_HG * ATT_KC);  // [KC]

  const int split = blockIdx.x;
  const int ur = blockIdx.y;
  const int nsplit = gridDim.x;
  const int j0 = split * ATT_KC;
  const int t = threadIdx.x;

  // dequantise the chunk: c[d] = int8[d] * scale[d / 64]; RoPE passes through
  for (int jj = 0; jj < ATT_KC; ++jj) {
    const int j = j0 + jj;
    const bool valid = j < K && topk[(size_t)ur * K + j] >= 0;
    if (t == 0) svalid[jj] = valid;
    const uint8_t* row = rows + ((size_t)ur * K + (valid ? j : 0)) * DSA_ROW_BYTES;
    for (int d = t; d < KD; d += ATT_THREADS) {
      float v = 0.0f;
      if (valid) {
        if (d < DSA_LAT_DIM) {
          const float s = __half2float(__ushort_as_half(
              reinterpret_cast<const uint16_t*>(row + DSA_LAT_DIM)[d >> 6]));
          v = (float)reinterpret_cast<const int8_t*>(row)[d] * s;
        } else {
          v = bf16f(reinterpret_cast<const uint16_t*>(row + DSA_LAT_DIM + 16)[d - DSA_LAT_DIM]);
        }
      }
      kc[jj * KSTR + d] = v;
    }
  }

  for (int hg = 0; hg < H; hg += ATT_HG) {
    const int nh = min(ATT_HG, H - hg);
    __syncthreads();
    for (int i = t; i < nh * KD; i += ATT_THREADS) {
      const int h = i / KD, d = i % KD;
      const size_t qo = ((size_t)ur * H + hg + h);
      const uint16_t b = d < DSA_LAT_DIM ? q_lat[qo * DSA_LAT_DIM + d]
                                         : q_rope[qo * DSA_ROPE_DIM + d - DSA_LAT_DIM];
      if (fabsf(bf16f(b)) >= 65504.0f) dsa_flag(dev_err, DSA_DEVERR_QRANGE);
      sq[h * QSTR + d] = b;
    }
    __syncthreads();
    // logits: thread -> head t/4, rows (t%4)*8 .. +8
    {
      const int h = t >> 2, jb = (t & 3) * 8;
      float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (h < nh) {
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(sq + h * QSTR);
        for (int d2 = 0; d2 < KD / 2; ++d2) {
          const uint32_t qq = qrow[d2];
          const float q0 = bf16_lo(qq), q1 = bf16_hi(qq);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float* kr = kc + (jb + i) * KSTR + 2 * d2;
            acc[i] = fmaf(q0, kr[0], acc[i]);
            acc[i] = fmaf(q1, kr[1], acc[i]);
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i)
          sp[h * ATT_KC + jb + i] = svalid[jb + i] ? acc[i] * scale : -INFINITY;
      }
    }
    __syncthreads();
    // chunk softmax per head
    if (t < nh) {
      float m = -INFINITY;
      for (int jj = 0; jj < ATT_KC; ++jj) m = fmaxf(m, sp[t * ATT_KC + jj]);
      float l = 0.0f;
      for (int jj = 0; jj < ATT_KC; ++jj) {
        const float x = sp[t * ATT_KC + jj];
        const float p = (m == -INFINITY) ? 0.0f : expf(x - m);
        sp[t * ATT_KC + jj] = p;
        l += p;
      }
      const size_t mo = ((size_t)ur * nsplit + split) * H + hg + t;
      ws.m[mo] = m;
      ws.l[mo] = l;
    }
    __syncthreads();
    // unnormalised P V: thread -> latent columns t and t + 256
    for (int h0 = 0; h0 < nh; h0 += 16) {
      float a0[16], a1[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) a0[i] = a1[i] = 0.0f;
      for (int jj = 0; jj < ATT_KC; ++jj) {
        const float c0 = kc[jj * KSTR + t];
        const float c1 = kc[jj * KSTR + t + 256];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p = (h0 + i < nh) ? sp[(h0 + i) * ATT_KC + jj] : 0.0f;
          a0[i] = fmaf(p, c0, a0[i]);
          a1[i] = fmaf(p, c1, a1[i]);
        }
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        if (h0 + i < nh) {
          float* o = ws.o + (((size_t)ur * nsplit + split) * H + hg + h0 + i) * DSA_LAT_DIM;
          o[t] = a0[i];
          o[t + 256] = a1[i];
        }
      }
    }
  }
}

__global__ void __launch_bounds__(COMB_THREADS)
k_attn_combine(int H, int nsplit, AttnWs ws, float* __restrict__ out, float* __restrict__ lse) {
  const int ur = blockIdx.x;
  const int t = threadIdx.x;
  for (int h = blockIdx.y; h < H; h += gridDim.y) {
    float M = -INFINITY;
    for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ws.m[((size_t)ur * nsplit + s) * H + h]);
    float Ls = 0.0f, acc = 0.0f;
    for (int s = 0; s < nsplit; ++s) {
      const size_t mo = ((size_t)ur * nsplit + s) * H + h;
      const float m = ws.m[mo];
      if (m == -INFINITY) continue;
      const float f = expf(m - M);
      Ls += ws.l[mo] * f;
      acc += ws.o[mo * DSA_LAT_DIM + t] * f;
    }
    out[((size_t)ur * H + h) * DSA_LAT_DIM + t] = Ls > 0.0f ? acc / Ls : 0.0f;
    if (lse && t == 0) lse[(size_t)ur * H + h] = Ls > 0.0f ? M + logf(Ls) : -INFINITY;
  }
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
    DSA_CUDA_TRY(cudaFuncSetAttribute(k_attn_partial, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)attn_smem()));
    attr_done = true;
  }
  const int ns = n_split(K);
  k_attn_partial<<<dim3(ns, U * R), ATT_THREADS, attn_smem(), st>>>(R, H, K, q_lat, q_rope, rows,
                                                                  topk_idx, scale, a, dev_err);
  if (dsa_launch_status() != DSA_OK) return DSA_ERR_CUDA;
  k_attn_combine<<<dim3(U * R, min(H, 8)), COMB_THREADS, 0, st>>>(H, ns, a, out, lse);
  return dsa_launch_status();
}
