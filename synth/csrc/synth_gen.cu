// GPU implementation of the synth input generator (see synth/rng.py for the
// definition). Counter-based SplitMix64: draw i of stream k is
// mix64(k + (i + 1) * 0x9E3779B97F4A7C15); each draw gives four 16-bit fields,
// least significant first. Every value mapping is integer-exact, so these
// kernels write byte-for-byte what the numpy generator writes. This library
// draws inputs only; it holds none of the decode path's arithmetic.
#include <cstdint>
#include <cuda_runtime.h>

namespace {

constexpr uint64_t GAMMA = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ uint32_t field(uint64_t key, uint64_t f) {
  const uint64_t d = mix64(key + ((f >> 2) + 1) * GAMMA);
  return (uint32_t)((d >> (16 * (f & 3))) & 0xFFFFu);
}

__device__ __forceinline__ int uni(uint32_t f, int lo, int hi) {
  return lo + (int)(((int64_t)f * (hi - lo + 1)) >> 16);
}

// float32 -> bf16 bits, round to nearest even (same bit trick as the host side)
__device__ __forceinline__ uint16_t bf16_rne(float x) {
  const uint32_t u = __float_as_uint(x);
  return (uint16_t)((u + (((u >> 16) & 1u) + 0x7FFFu)) >> 16);
}

// Irwin-Hall numerator: sum of 12 fields + 6 - 6 * 65536
__device__ __forceinline__ int64_t ih_num(uint64_t key, uint64_t f0) {
  int64_t s = 0;
#pragma unroll
  for (int i = 0; i < 12; ++i) s += field(key, f0 + i);
  return s + 6 - 6 * 65536;
}

__global__ void gen_keys(uint64_t key, uint16_t* out, int64_t pos0, int64_t n, int tagged,
                       int64_t hot_lo, int64_t hot_hi) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n * 64) return;
  const int64_t p = pos0 + i / 64;
  const int d = (int)(i % 64);
  int v = uni(field(key, (uint64_t)p * 64 + d), -4, 4);
  if (tagged && d == 63) v = (p >= hot_lo && p < hot_hi) ? 4 : -4;
  out[i] = bf16_rne((float)v);
}

__global__ void gen_rows(uint64_t k_lat, uint64_t k_sc, uint64_t k_rope, uint8_t* out, int64_t pos0,
                       int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  // 512 latent bytes + 8 scales + 64 rope values = 584 items per row
  if (i >= n * 584) return;
  const int64_t r = i / 584;
  const int c = (int)(i % 584);
  const uint64_t p = (uint64_t)(pos0 + r);
  uint8_t* row = out + r * 656;
  if (c < 512) {
    row[c] = (uint8_t)(int8_t)uni(field(k_lat, p * 512 + c), -127, 127);
  } else if (c < 520) {
    const int g = c - 512;
    const int k = uni(field(k_sc, p * 8 + g), 328, 1311);
    // k * 2^-16 is exact in fp16: with 2^e <= k < 2^(e+1) (e in 8..10) the
    // biased exponent is e - 16 + 15 and the 10-bit fraction (k - 2^e) << (10 - e)
    const int e = 31 - __clz(k);
    const uint16_t h = (uint16_t)(((e - 1) << 10) | ((k << (10 - e)) & 0x3FF));
    row[512 + 2 * g] = (uint8_t)(h & 0xFF);
    row[512 + 2 * g + 1] = (uint8_t)(h >> 8);
  } else {
    const int e = c - 520;
    const float z = (float)ih_num(k_rope, (p * 64 + e) * 12) * (1.0f / 65536.0f);
    const uint16_t b = bf16_rne(z);
    row[528 + 2 * e] = (uint8_t)(b & 0xFF);
    row[528 + 2 * e + 1] = (uint8_t)(b >> 8);
  }
}

__global__ void gen_normal(uint64_t key, uint16_t* out, int64_t item0, int64_t n_items, int per) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_items * per) return;
  const uint64_t f0 = ((uint64_t)(item0 + i / per) * per + (uint64_t)(i % per)) * 12;
  out[i] = bf16_rne((float)ih_num(key, f0) * (1.0f / 65536.0f));
}

// Uniform integers in [lo, hi] as bf16; with tag_every > 0 the last value of
// every group of tag_every is replaced by tag16 / 16.
__global__ void gen_uniform_bf16(uint64_t key, uint16_t* out, int64_t item0, int64_t n_items, int per,
                               int lo, int hi, int tag_every, int tag16) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_items * per) return;
  const int v = (int)(i % per);
  float x = (float)uni(field(key, (uint64_t)(item0 + i / per) * per + v), lo, hi);
  if (tag_every > 0 && (v % tag_every) == tag_every - 1) x = (float)tag16 * (1.0f / 16.0f);
  out[i] = bf16_rne(x);
}

// Uniform integers as float32; output item i uses generator item (item0 + i) / rep.
__global__ void gen_uniform_f32(uint64_t key, float* out, int64_t item0, int64_t n_items, int per,
                              int lo, int hi, int rep) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_items * per) return;
  const int64_t it = (item0 + i / per) / rep;
  out[i] = (float)uni(field(key, (uint64_t)it * per + (uint64_t)(i % per)), lo, hi);
}

// MTP verify rows of one step: q16 = clip(16 * base + floor((num * sd16 + 32768) / 65536), -128, 128).
__global__ void gen_mtp(uint64_t k_base, uint64_t k_pert, uint16_t* out, int64_t step, int R, int sd16) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= R * 512) return;
  const int r = i / 512, v = i % 512;
  const int base = uni(field(k_base, (uint64_t)step * 512 + v), -4, 4);
  const int64_t num = ih_num(k_pert, (((uint64_t)step * R + r) * 512 + v) * 12);
  const int64_t m = (num * sd16 + 32768) >> 16;     // arithmetic shift = floor division
  int64_t q16 = (int64_t)base * 16 + m;
  q16 = q16 < -128 ? -128 : (q16 > 128 ? 128 : q16);
  out[i] = bf16_rne((float)q16 * (1.0f / 16.0f));
}

inline unsigned blocks(int64_t n, int t) { return (unsigned)((n + t - 1) / t); }
inline int st(cudaStream_t s) { return cudaGetLastError() == cudaSuccess ? 0 : -4; }

}  // namespace

extern "C" {

int synth_keys(uint64_t key, uint16_t* out, int64_t pos0, int64_t n, int tagged, int64_t hot_lo,
               int64_t hot_hi, void* stream) {
  if (n <= 0) return 0;
  cudaStream_t s = (cudaStream_t)stream;
  gen_keys<<<blocks(n * 64, 256), 256, 0, s>>>(key, out, pos0, n, tagged, hot_lo, hot_hi);
  return st(s);
}

int synth_rows(uint64_t k_lat, uint64_t k_sc, uint64_t k_rope, uint8_t* out, int64_t pos0, int64_t n,
               void* stream) {
  if (n <= 0) return 0;
  cudaStream_t s = (cudaStream_t)stream;
  gen_rows<<<blocks(n * 584, 256), 256, 0, s>>>(k_lat, k_sc, k_rope, out, pos0, n);
  return st(s);
}

int synth_normal_bf16(uint64_t key, uint16_t* out, int64_t item0, int64_t n_items, int per,
                      void* stream) {
  if (n_items <= 0) return 0;
  cudaStream_t s = (cudaStream_t)stream;
  gen_normal<<<blocks(n_items * per, 256), 256, 0, s>>>(key, out, item0, n_items, per);
  return st(s);
}

int synth_uniform_bf16(uint64_t key, uint16_t* out, int64_t item0, int64_t n_items, int per, int lo,
                       int hi, int tag_every, int tag16, void* stream) {
  if (n_items <= 0) return 0;
  cudaStream_t s = (cudaStream_t)stream;
  gen_uniform_bf16<<<blocks(n_items * per, 256), 256, 0, s>>>(key, out, item0, n_items, per, lo, hi,
                                                            tag_every, tag16);
  return st(s);
}

int synth_uniform_f32(uint64_t key, float* out, int64_t item0, int64_t n_items, int per, int lo,
                      int hi, int rep, void* stream) {
  if (n_items <= 0 || rep < 1) return 0;
  cudaStream_t s = (cudaStream_t)stream;
  gen_uniform_f32<<<blocks(n_items * per, 256), 256, 0, s>>>(key, out, item0, n_items, per, lo, hi, rep);
  return st(s);
}

int synth_mtp_qidx(uint64_t k_base, uint64_t k_pert, uint16_t* out, int64_t step, int R, int sd16,
                   void* stream) {
  cudaStream_t s = (cudaStream_t)stream;
  gen_mtp<<<blocks((int64_t)R * 512, 256), 256, 0, s>>>(k_base, k_pert, out, step, R, sd16);
  return st(s);
}

}  // extern "C"
