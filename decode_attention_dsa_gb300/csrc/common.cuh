// Shared helpers of the decode-path kernels (device code for sm_103a).
#pragma once

#include <atomic>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "dsa_decode.h"

#define DSA_CUDA_TRY(expr)                                   \
  do {                                                       \
    cudaError_t e__ = (expr);                                \
    if (e__ != cudaSuccess) return DSA_ERR_CUDA;             \
  } while (0)

// A launch error is reported by cudaGetLastError right after the launch.
static inline int dsa_launch_status() {
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

__host__ __device__ static inline size_t dsa_align(size_t x, size_t a) { return (x + a - 1) / a * a; }

// One-time set-up per device (kernel attributes, SM count), keyed by the
// current device ordinal: a process that uses several GPUs sets every one up,
// and host threads that make their first calls at the same time are
// serialised. `init(dev)` returns a DSA_ status; a failed set-up is retried
// on the next call.
constexpr int DSA_MAX_DEVICES = 64;
struct DsaPerDevice {
  std::mutex mu;
  std::atomic<bool> ready[DSA_MAX_DEVICES] = {};
  int num_sms[DSA_MAX_DEVICES] = {};
};

// SMs that kernels launched on `st` may use: those of the SM partition
// (green context) the stream belongs to, else `device_sms` (partition.cu).
int dsa_stream_sms(cudaStream_t st, int device_sms);

// Every kernel of the library prefers the largest shared-memory carveout. An
// SM whose L1/shared split was set for a kernel with little shared memory
// takes a CTA that needs more only after it has drained, so a small kernel of
// one step (row copies, append) would hold the next step's persistent score
// CTAs off its SMs instead of running beside them.
template <typename T>
static inline cudaError_t dsa_prefer_shared(T* kernel) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

template <typename F>
static inline int dsa_device_setup(DsaPerDevice& pd, int* dev_out, F&& init) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= DSA_MAX_DEVICES) return DSA_ERR_CUDA;
  *dev_out = dev;
  if (pd.ready[dev].load(std::memory_order_acquire)) return DSA_OK;
  std::lock_guard<std::mutex> lock(pd.mu);
  if (pd.ready[dev].load(std::memory_order_relaxed)) return DSA_OK;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return DSA_ERR_CUDA;
  const int st = init(dev);
  if (st != DSA_OK) return st;
  pd.num_sms[dev] = sms;
  pd.ready[dev].store(true, std::memory_order_release);
  return DSA_OK;
}

__device__ __forceinline__ void dsa_flag(int32_t* dev_err, int32_t bit) {
  if (dev_err) atomicOr(dev_err, bit);
}

// bf16 bits -> float (exact).
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// Read-only 16-byte load that bypasses L1 allocation (streamed data, or
// host memory reached through the mapped alias).
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Read-only 16-byte load through L1 (neighbouring lanes reuse the sector).
__device__ __forceinline__ uint4 ldg_v4(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// Copy one 656-byte row (41 x 16 B) with the 32 lanes of a warp. Both
// addresses must be 16-byte aligned.
__device__ __forceinline__ void warp_copy_row(uint8_t* dst, const uint8_t* src, int lane) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  uint4 a = ldg_nc_v4(s + lane);
  uint4 b;
  if (lane < 9) b = ldg_nc_v4(s + 32 + lane);
  d[lane] = a;
  if (lane < 9) d[32 + lane] = b;
}

__device__ __forceinline__ void warp_zero_row(uint8_t* dst, int lane) {
  uint4* d = reinterpret_cast<uint4*>(dst);
  const uint4 z = make_uint4(0, 0, 0, 0);
  d[lane] = z;
  if (lane < 9) d[32 + lane] = z;
}

// Inclusive scan of one int per thread over a block of NT threads.
// `tmp` must hold NT/32 ints in shared memory. Ends with a barrier so that
// `tmp` can be reused right away.
template <int NT>
__device__ __forceinline__ int block_inclusive_scan(int v, int* tmp, int* total = nullptr) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += y;
  }
  if (lane == 31) tmp[warp] = v;
  __syncthreads();
  if (warp == 0) {
    int s = lane < NW ? tmp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < NW) tmp[lane] = s;
  }
  __syncthreads();
  if (warp > 0) v += tmp[warp - 1];
  if (total) *total = tmp[NW - 1];
  __syncthreads();
  return v;
}

// Programmatic dependent launch. Every hot-path kernel is launched with
// programmatic stream serialization, so it may start while the previous
// kernel in the stream is still finishing; it must call pdl_wait() before it
// reads or writes any global memory (inputs may come from that kernel).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
static inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

// The row and key arrays of a unit are moved with 16-byte vector loads and
// bulk copies; a unit whose arrays are not 16-byte aligned is skipped.
__device__ __forceinline__ bool unit_aligned(const dsa_unit& un) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(un.keys) | reinterpret_cast<uintptr_t>(un.slots) |
                      reinterpret_cast<uintptr_t>(un.ring) | reinterpret_cast<uintptr_t>(un.mirror);
  return (a & 15u) == 0;
}
