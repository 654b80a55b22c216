// Housekeeping entry points, cache initialisation (hc_init) and A6: append
// with batched write-back (kv_append_writeback, kv_flush).
//
// [P3] "From 1M total to 15+ x 1M: GLM-5.3 KV-cache offload":
//  * section "第二次决策" (second decision): per-row, per-layer host-mirror
//    updates meant 156 stream operations per token (468 when split further);
//    batching write-back per 64 rows cut the operation count.
//  * section "第三次决策" (third decision) diagram: new KV -> GPU recent ring ->
//    batched write-back -> RAM history.
//  * section "第四次决策" (fourth decision): small logs are copied and packed
//    by compute kernels to cut DMA queue operations.
//  * section "容量优化必须通过会话生命周期" (session lifecycle): before export
//    or restore, flush the log and check RAM rows == logical rows.
// Here the write-back is a plain kernel store of 64 ring rows (41,984 B) into
// the mapped mirror: no DMA operation, no host involvement.
#include <algorithm>
#include <cstring>

#include <unistd.h>

#include <cuda_fp16.h>

#include "common.cuh"
#include "tc.cuh"

namespace {

constexpr int APP_THREADS = 256;
constexpr int INIT_THREADS = 256;

// Store ring rows of positions [from, to) to the mirror (block-wide).
__device__ void write_back(const dsa_unit& un, int64_t from, int64_t to) {
  const int64_t n16 = (to - from) * (DSA_ROW_BYTES / 16);
  for (int64_t i = threadIdx.x; i < n16; i += blockDim.x) {
    const int64_t r = i / (DSA_ROW_BYTES / 16);
    const int c = (int)(i % (DSA_ROW_BYTES / 16));
    const int64_t p = from + r;
    const uint4* src = reinterpret_cast<const uint4*>(un.ring + (p & (DSA_RING_ROWS - 1)) * DSA_ROW_BYTES);
    uint4* dst = reinterpret_cast<uint4*>(un.mirror + p * DSA_ROW_BYTES);
    dst[c] = src[c];
  }
}

// Q8G64-quantise one bf16 row into `dst` (656 bytes): warp g handles latent
// group g (threads 32g..32g+31, two values each). Symmetric group scale
// fp16_rn(amax / 127) and codes clamp(rint(w / scale), -127, 127), IEEE fp32
// division; a zero (or unrepresentable) scale gives all-zero codes.
__device__ void quantize_row_q8g64(uint8_t* dst, const uint16_t* lat, const uint16_t* rope) {
  const int t = threadIdx.x, lane = t & 31, g = t >> 5;
  if (t < 256) {
    const float x0 = bf16f(lat[2 * t]), x1 = bf16f(lat[2 * t + 1]);
    float m = fmaxf(fabsf(x0), fabsf(x1));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const __half h = __float2half_rn(m / 127.0f);
    float sc = __half2float(h);
    const bool zero = !(sc > 0.0f) || isinf(sc);
    int8_t q0 = 0, q1 = 0;
    if (!zero) {
      q0 = (int8_t)fminf(fmaxf(rintf(x0 / sc), -127.0f), 127.0f);
      q1 = (int8_t)fminf(fmaxf(rintf(x1 / sc), -127.0f), 127.0f);
    }
    dst[2 * t] = (uint8_t)q0;
    dst[2 * t + 1] = (uint8_t)q1;
    if (lane == 0) {
      const uint16_t hb = zero ? (uint16_t)0 : __half_as_ushort(h);
      dst[DSA_LAT_DIM + 2 * g] = (uint8_t)(hb & 0xFF);
      dst[DSA_LAT_DIM + 2 * g + 1] = (uint8_t)(hb >> 8);
    }
  }
  if (t < DSA_ROPE_DIM) reinterpret_cast<uint16_t*>(dst + DSA_LAT_DIM + 16)[t] = rope[t];
}

// QUANT = false: new_rows holds ready 656-byte rows. QUANT = true: new_rows
// holds bf16 latents [A][512] and new_rope bf16 RoPE parts [A][64].
template <bool QUANT>
__global__ void __launch_bounds__(APP_THREADS)
k_append(const dsa_unit* __restrict__ units, int A, const uint8_t* __restrict__ new_rows,
         const uint16_t* __restrict__ new_keys, int32_t* dev_err, const uint16_t* __restrict__ new_rope) {
  const int u = blockIdx.x;
  pdl_wait();
  const dsa_unit& un = units[u];
  if (!unit_aligned(un)) {
    if (threadIdx.x == 0) dsa_flag(dev_err, DSA_DEVERR_BOUNDS);
    return;
  }
  __shared__ int64_t s_len, s_ram;
  if (threadIdx.x == 0) {
    s_len = un.state[DSA_ST_LEN];
    s_ram = un.state[DSA_ST_RAM];
  }
  __syncthreads();
  int64_t len = s_len, ram = s_ram;
  int64_t wb = 0;
  for (int a = 0; a < A; ++a) {
    const int64_t p = len;
    if (p >= un.lmax || p - ram >= DSA_RING_ROWS) {
      if (threadIdx.x == 0) dsa_flag(dev_err, DSA_DEVERR_CAPACITY);
      break;
    }
    uint8_t* ring_row = un.ring + (p & (DSA_RING_ROWS - 1)) * DSA_ROW_BYTES;
    if (QUANT) {
      const uint16_t* lat = reinterpret_cast<const uint16_t*>(new_rows) + ((size_t)u * A + a) * DSA_LAT_DIM;
      quantize_row_q8g64(ring_row, lat, new_rope + ((size_t)u * A + a) * DSA_ROPE_DIM);
    } else {
      const uint4* src = reinterpret_cast<const uint4*>(new_rows + ((size_t)u * A + a) * DSA_ROW_BYTES);
      uint4* dst = reinterpret_cast<uint4*>(ring_row);
      for (int c = threadIdx.x; c < DSA_ROW_BYTES / 16; c += APP_THREADS) dst[c] = src[c];
    }
    const uint4* ks = reinterpret_cast<const uint4*>(new_keys + ((size_t)u * A + a) * DSA_IDX_DIM);
    uint4* kd = reinterpret_cast<uint4*>(un.keys + p * DSA_IDX_DIM);
    if (threadIdx.x < 8) kd[threadIdx.x] = ks[threadIdx.x];
    len = p + 1;
    if (len - ram == DSA_RING_ROWS) {
      __syncthreads();              // the ring row just written is part of the batch
      write_back(un, ram, len);
      __syncthreads();              // the batch is read before its ring rows are reused
      ram = len;
      ++wb;
    }
  }
  if (threadIdx.x == 0) {
    un.state[DSA_ST_LEN] = len;
    un.state[DSA_ST_RAM] = ram;
    un.state[DSA_ST_WRITEBACKS] += wb;
  }
}

__global__ void __launch_bounds__(APP_THREADS) k_flush(const dsa_unit* __restrict__ units) {
  const int u = blockIdx.x;
  const dsa_unit& un = units[u];
  if (!unit_aligned(un)) return;
  const int64_t len = un.state[DSA_ST_LEN];
  const int64_t ram = un.state[DSA_ST_RAM];
  if (len <= ram) return;
  write_back(un, ram, len);
  __syncthreads();
  if (threadIdx.x == 0) {
    un.state[DSA_ST_RAM] = len;
    un.state[DSA_ST_WRITEBACKS] += 1;
  }
}

// pos_slot for every position, and the slot arrays, in one pass over
// max(lmax, S) indices per unit.
__global__ void __launch_bounds__(INIT_THREADS)
k_init_map(const dsa_unit* __restrict__ units, int warm, const int64_t* __restrict__ l0v,
           int32_t* dev_err) {
  const int u = blockIdx.y;
  const dsa_unit& un = units[u];
  const int64_t i = (int64_t)blockIdx.x * INIT_THREADS + threadIdx.x;
  const int64_t l0 = l0v[u];
  const int S = un.slots_n;
  if (l0 < 0 || l0 > un.lmax || S < 1) {
    if (i == 0) dsa_flag(dev_err, DSA_DEVERR_BOUNDS);
    return;
  }
  const int64_t n = warm == DSA_WARM_LAST_S ? min((int64_t)S, l0) : 0;
  const int64_t first = l0 - n;
  if (i < un.lmax) un.pos_slot[i] = (i >= first && i < l0) ? (int32_t)(i - first) : -1;
  if (i < S) {
    un.slot_pos[i] = i < n ? (int32_t)(first + i) : -1;
    un.fill_round[i] = -1;
    un.pin_epoch[i] = -1;
    if (un.ref) un.ref[i] = i < n ? 1 : 0;
  }
  if (i < DSA_ST_WORDS) {
    int64_t v = 0;
    if (i == DSA_ST_LEN || i == DSA_ST_RAM) v = l0;
    un.state[i] = v;
  }
}

// Warm slot bytes: slot i <- mirror[l0 - n + i] (one warp per row).
__global__ void __launch_bounds__(INIT_THREADS)
k_init_slots(const dsa_unit* __restrict__ units, int warm, const int64_t* __restrict__ l0v) {
  const int u = blockIdx.y;
  const dsa_unit& un = units[u];
  const int64_t i = (int64_t)blockIdx.x * (INIT_THREADS / 32) + (threadIdx.x >> 5);
  const int64_t l0 = l0v[u];
  const int S = un.slots_n;
  if (warm != DSA_WARM_LAST_S || l0 < 0 || l0 > un.lmax || S < 1 || !unit_aligned(un)) return;
  const int64_t n = min((int64_t)S, l0);
  if (i >= n) return;
  warp_copy_row(un.slots + i * DSA_ROW_BYTES, un.mirror + (l0 - n + i) * DSA_ROW_BYTES,
                threadIdx.x & 31);
}

// One 16-byte read per `stride` bytes of each unit's mirror: the GPU's
// address translations for the whole mirror are set up here, at set-up time,
// instead of by the first decode steps' misses (random rows spread over
// gigabytes of host memory paid several milliseconds per step for them).
__global__ void __launch_bounds__(INIT_THREADS)
k_touch_mirror(const dsa_unit* __restrict__ units, int64_t stride) {
  const dsa_unit& un = units[blockIdx.y];
  if (!unit_aligned(un) || un.lmax <= 0) return;
  const int64_t bytes = un.lmax * DSA_ROW_BYTES;
  for (int64_t i = (int64_t)blockIdx.x * INIT_THREADS + threadIdx.x; i * stride < bytes;
       i += (int64_t)gridDim.x * INIT_THREADS) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(un.mirror + i * stride));
  }
}

// The bounded wait every kernel uses, alone: one CTA waits on a barrier
// phase that completes only if `complete` is set, for at most `limit` cycles.
__global__ void k_wait_selftest(long long limit, int complete, int32_t* dev_err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
  }
  __syncthreads();
  if (complete && threadIdx.x == 0) tc::mbar_arrive(&bar);
  const bool ok = tc::mbar_wait(&bar, 0, limit);
  if (__syncthreads_or(!ok) && threadIdx.x == 0) dsa_flag(dev_err, DSA_DEVERR_TIMEOUT);
}

// ---- session snapshot (export / restore) and the full-history restore

// Byte layout of one unit's snapshot (every part 16-byte aligned).
struct SnapLayout {
  size_t slot_pos, fill_round, ref, ring, keys, bytes;
};
__host__ __device__ inline SnapLayout snap_layout(int32_t S, int64_t lmax) {
  SnapLayout l;
  l.slot_pos = 128;                                   // [0, 64) state words, [64, 80) S, policy, lmax
  l.fill_round = l.slot_pos + dsa_align((size_t)S * 4, 16);
  l.ref = l.fill_round + dsa_align((size_t)S * 4, 16);
  l.ring = l.ref + dsa_align((size_t)S, 16);
  l.keys = l.ring + (size_t)DSA_RING_ROWS * DSA_ROW_BYTES;
  l.bytes = l.keys + (size_t)lmax * DSA_IDX_DIM * 2;
  return l;
}

// 16-byte copy loop over a block's part of [0, n16) chunks (grid x stride).
__device__ __forceinline__ void copy16(void* dst, const void* src, int64_t n16) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (int64_t)gridDim.x * blockDim.x)
    d[i] = s[i];
}

// Export: unit u's state into snap + u * stride. Needs RAM == LEN (flushed).
__global__ void __launch_bounds__(INIT_THREADS)
k_export(const dsa_unit* __restrict__ units, uint8_t* __restrict__ snap, size_t stride, int32_t* dev_err) {
  const dsa_unit& un = units[blockIdx.y];
  const int64_t len = un.state[DSA_ST_LEN];
  if (!unit_aligned(un) || un.state[DSA_ST_RAM] != len) {
    if (blockIdx.x == 0 && threadIdx.x == 0) dsa_flag(dev_err, DSA_DEVERR_STATE);
    return;
  }
  const int S = un.slots_n;
  const SnapLayout l = snap_layout(S, un.lmax);
  if (l.bytes > stride) {   // this unit is larger than the host bounds said
    if (blockIdx.x == 0 && threadIdx.x == 0) dsa_flag(dev_err, DSA_DEVERR_STATE);
    return;
  }
  uint8_t* o = snap + (size_t)blockIdx.y * stride;
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, gs = (int64_t)gridDim.x * blockDim.x;
  if (gt < DSA_ST_WORDS) reinterpret_cast<int64_t*>(o)[gt] = un.state[gt];
  if (gt == 0) {
    reinterpret_cast<int32_t*>(o + 64)[0] = S;
    reinterpret_cast<int32_t*>(o + 64)[1] = un.policy;
    reinterpret_cast<int64_t*>(o + 72)[0] = un.lmax;
  }
  for (int64_t i = gt; i < S; i += gs) {
    reinterpret_cast<int32_t*>(o + l.slot_pos)[i] = un.slot_pos[i];
    reinterpret_cast<int32_t*>(o + l.fill_round)[i] = un.fill_round[i];
    o[l.ref + i] = un.ref ? un.ref[i] : 0;
  }
  copy16(o + l.ring, un.ring, (int64_t)DSA_RING_ROWS * DSA_ROW_BYTES / 16);
  copy16(o + l.keys, un.keys, len * DSA_IDX_DIM * 2 / 16);
}

// Restore, part 1: state words, slot arrays, ring, keys; pos_slot cleared.
__global__ void __launch_bounds__(INIT_THREADS)
k_restore_a(const dsa_unit* __restrict__ units, const uint8_t* __restrict__ snap, size_t stride, int32_t* dev_err) {
  const dsa_unit& un = units[blockIdx.y];
  const uint8_t* o = snap + (size_t)blockIdx.y * stride;
  const int64_t* st = reinterpret_cast<const int64_t*>(o);
  const int S = reinterpret_cast<const int32_t*>(o + 64)[0];
  const int64_t slmax = reinterpret_cast<const int64_t*>(o + 72)[0];
  const int64_t len = st[DSA_ST_LEN];
  if (!unit_aligned(un) || S != un.slots_n || len < 0 || len > un.lmax || len > slmax || st[DSA_ST_RAM] != len ||
      snap_layout(S, slmax).bytes > stride) {
    if (blockIdx.x == 0 && threadIdx.x == 0) dsa_flag(dev_err, DSA_DEVERR_STATE);
    return;
  }
  const SnapLayout l = snap_layout(S, slmax);
  const int64_t gt = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, gs = (int64_t)gridDim.x * blockDim.x;
  if (gt < DSA_ST_WORDS) un.state[gt] = st[gt];
  for (int64_t i = gt; i < S; i += gs) {
    un.slot_pos[i] = reinterpret_cast<const int32_t*>(o + l.slot_pos)[i];
    un.fill_round[i] = reinterpret_cast<const int32_t*>(o + l.fill_round)[i];
    un.pin_epoch[i] = -1;
    if (un.ref) un.ref[i] = o[l.ref + i];
  }
  for (int64_t i = gt; i < un.lmax; i += gs) un.pos_slot[i] = -1;
  copy16(un.ring, o + l.ring, (int64_t)DSA_RING_ROWS * DSA_ROW_BYTES / 16);
  copy16(un.keys, o + l.keys, len * DSA_IDX_DIM * 2 / 16);
}

// Restore, part 2: the position -> slot index and the slot bytes (one warp
// per slot, from the mirror, which holds every row of the flushed history).
__global__ void __launch_bounds__(INIT_THREADS)
k_restore_b(const dsa_unit* __restrict__ units, const uint8_t* __restrict__ snap, size_t stride) {
  const dsa_unit& un = units[blockIdx.y];
  const uint8_t* o = snap + (size_t)blockIdx.y * stride;
  const int64_t len = reinterpret_cast<const int64_t*>(o)[DSA_ST_LEN];
  const int S = reinterpret_cast<const int32_t*>(o + 64)[0];
  const int64_t slmax = reinterpret_cast<const int64_t*>(o + 72)[0];
  if (!unit_aligned(un) || S != un.slots_n || len < 0 || len > un.lmax || len > slmax ||
      reinterpret_cast<const int64_t*>(o)[DSA_ST_RAM] != len || snap_layout(S, slmax).bytes > stride)
    return;
  const int lane = threadIdx.x & 31;
  for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < S;
       i += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int32_t p = un.slot_pos[i];
    if (p < 0 || p >= len) continue;
    if (lane == 0) un.pos_slot[p] = (int32_t)i;
    warp_copy_row(un.slots + i * DSA_ROW_BYTES, un.mirror + (int64_t)p * DSA_ROW_BYTES, lane);
  }
}

// The full history of each unit as dense rows: [0, RAM) from the mirror,
// [RAM, LEN) from the ring. Each warp copies whole rows.
__global__ void __launch_bounds__(INIT_THREADS)
k_restore_full(const dsa_unit* __restrict__ units, uint8_t* __restrict__ dst, int64_t dst_rows) {
  const dsa_unit& un = units[blockIdx.y];
  if (!unit_aligned(un)) return;
  const int64_t len = min(un.state[DSA_ST_LEN], dst_rows);
  const int64_t ram = un.state[DSA_ST_RAM];
  uint8_t* d = dst + (size_t)blockIdx.y * dst_rows * DSA_ROW_BYTES;
  const int lane = threadIdx.x & 31;
  for (int64_t p = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < len;
       p += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const uint8_t* src = p < ram ? un.mirror + p * DSA_ROW_BYTES : un.ring + (p & (DSA_RING_ROWS - 1)) * DSA_ROW_BYTES;
    warp_copy_row(d + p * DSA_ROW_BYTES, src, lane);
  }
}

}  // namespace

extern "C" size_t dsa_snapshot_bytes(int32_t S, int64_t lmax) {
  if (S < 1 || lmax < 0) return 0;
  return snap_layout(S, lmax).bytes;
}

static int grid_for(int64_t items, int per_block) {
  const int64_t b = (items + per_block - 1) / per_block;
  return (int)std::min<int64_t>(std::max<int64_t>(b, 1), 4096);
}

extern "C" int dsa_export(const dsa_unit* units, int32_t U, uint8_t* snap, size_t snap_stride, int32_t max_slots,
                          int64_t max_lmax, int32_t* dev_err, void* stream) {
  if (!units || !snap || U < 1 || U > 65535 || max_slots < 1 || max_lmax < 0) return DSA_ERR_ARG;
  if (snap_stride < dsa_snapshot_bytes(max_slots, max_lmax) || (snap_stride & 15u) ||
      (reinterpret_cast<uintptr_t>(snap) & 15u))
    return DSA_ERR_ARG;
  const int64_t n16 = std::max<int64_t>(max_lmax * DSA_IDX_DIM * 2 / 16, max_slots);
  k_export<<<dim3(grid_for(n16, INIT_THREADS), U), INIT_THREADS, 0, static_cast<cudaStream_t>(stream)>>>(
      units, snap, snap_stride, dev_err);
  return dsa_launch_status();
}

extern "C" int dsa_restore(const dsa_unit* units, int32_t U, const uint8_t* snap, size_t snap_stride,
                           int32_t max_slots, int64_t max_lmax, int32_t* dev_err, void* stream) {
  if (!units || !snap || U < 1 || U > 65535 || max_slots < 1 || max_lmax < 0) return DSA_ERR_ARG;
  if (snap_stride < dsa_snapshot_bytes(max_slots, max_lmax) || (snap_stride & 15u) ||
      (reinterpret_cast<uintptr_t>(snap) & 15u))
    return DSA_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t n = std::max<int64_t>(max_lmax * DSA_IDX_DIM * 2 / 16, std::max<int64_t>(max_lmax, max_slots));
  k_restore_a<<<dim3(grid_for(n, INIT_THREADS), U), INIT_THREADS, 0, st>>>(units, snap, snap_stride, dev_err);
  if (dsa_launch_status() != DSA_OK) return DSA_ERR_CUDA;
  k_restore_b<<<dim3(grid_for(max_slots, INIT_THREADS / 32), U), INIT_THREADS, 0, st>>>(units, snap, snap_stride);
  return dsa_launch_status();
}

extern "C" int kv_restore_full(const dsa_unit* units, int32_t U, uint8_t* dst, int64_t dst_rows,
                               int32_t* dev_err, void* stream) {
  (void)dev_err;
  if (!units || !dst || U < 1 || U > 65535 || dst_rows < 1) return DSA_ERR_ARG;
  if (reinterpret_cast<uintptr_t>(dst) & 15u) return DSA_ERR_ARG;
  k_restore_full<<<dim3(grid_for(dst_rows, INIT_THREADS / 32), U), INIT_THREADS, 0,
                   static_cast<cudaStream_t>(stream)>>>(units, dst, dst_rows);
  return dsa_launch_status();
}

extern "C" int dsa_wait_selftest(int64_t limit_cycles, int32_t complete, int32_t* dev_err, void* stream) {
  if (!dev_err || limit_cycles < 0) return DSA_ERR_ARG;
  k_wait_selftest<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>((long long)limit_cycles, complete ? 1 : 0,
                                                                   dev_err);
  return dsa_launch_status();
}

extern "C" int dsa_abi_version(void) { return 2; }

extern "C" const char* dsa_status_string(int status) {
  switch (status) {
    case DSA_OK: return "ok";
    case DSA_ERR_ARG: return "invalid argument";
    case DSA_ERR_SHAPE: return "unsupported shape";
    case DSA_ERR_WS: return "workspace missing or too small";
    case DSA_ERR_CUDA: return "CUDA runtime or launch error";
    case DSA_ERR_DEVICE_CHECK: return "device-side check failed (see the dev_err bits)";
    case DSA_ERR_SCRATCH_LIMIT: return "problem exceeds the fixed built-in scratch of this entry point";
    default: return "unknown status";
  }
}

extern "C" int dsa_check(int32_t dev_err_value) {
  return dev_err_value == 0 ? DSA_OK : DSA_ERR_DEVICE_CHECK;
}

extern "C" int dsa_host_alloc(void** host_ptr, void** dev_ptr, size_t bytes) {
  if (!host_ptr || !dev_ptr || bytes == 0) return DSA_ERR_ARG;
  *host_ptr = nullptr;
  *dev_ptr = nullptr;
  void* h = nullptr;
  if (cudaHostAlloc(&h, bytes, cudaHostAllocMapped | cudaHostAllocPortable) != cudaSuccess)
    return DSA_ERR_CUDA;
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, h, 0) != cudaSuccess) {
    cudaFreeHost(h);
    return DSA_ERR_CUDA;
  }
  *host_ptr = h;
  *dev_ptr = d;
  return DSA_OK;
}

extern "C" int dsa_host_free(void* host_ptr) {
  if (!host_ptr) return DSA_ERR_ARG;
  return cudaFreeHost(host_ptr) == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

extern "C" int hc_init(const dsa_unit* units, int32_t U, int32_t warm, const int64_t* l0,
                       int32_t max_slots, int64_t max_lmax, int32_t* dev_err, void* stream) {
  if (!units || !l0 || U < 1 || U > 65535 || max_slots < 1 || max_lmax < 0) return DSA_ERR_ARG;
  if (warm != DSA_WARM_EMPTY && warm != DSA_WARM_LAST_S) return DSA_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t n = std::max<int64_t>(std::max<int64_t>(max_lmax, max_slots), DSA_ST_WORDS);
  const int64_t gx = (n + INIT_THREADS - 1) / INIT_THREADS;
  if (gx > 0x7fffffff) return DSA_ERR_ARG;
  k_init_map<<<dim3((unsigned)gx, U), INIT_THREADS, 0, st>>>(units, warm, l0, dev_err);
  if (dsa_launch_status() != DSA_OK) return DSA_ERR_CUDA;
  if (warm == DSA_WARM_LAST_S) {
    const int64_t gs = ((int64_t)max_slots + INIT_THREADS / 32 - 1) / (INIT_THREADS / 32);
    k_init_slots<<<dim3((unsigned)gs, U), INIT_THREADS, 0, st>>>(units, warm, l0);
    if (dsa_launch_status() != DSA_OK) return DSA_ERR_CUDA;
  }
  return dsa_touch_mirror(units, U, max_lmax, stream);
}

extern "C" int dsa_touch_mirror(const dsa_unit* units, int32_t U, int64_t max_lmax, void* stream) {
  if (!units || U < 1 || U > 65535 || max_lmax < 0) return DSA_ERR_ARG;
  // one read per host page of the mirrors (page size of this host)
  const long pg = sysconf(_SC_PAGESIZE);
  const int64_t stride = pg >= 16 ? (int64_t)pg / 16 * 16 : 4096;
  const int64_t pages = (max_lmax * DSA_ROW_BYTES + stride - 1) / stride;
  const int64_t gt = std::min<int64_t>(std::max<int64_t>((pages + INIT_THREADS - 1) / INIT_THREADS, 1), 1024);
  k_touch_mirror<<<dim3((unsigned)gt, U), INIT_THREADS, 0, static_cast<cudaStream_t>(stream)>>>(units, stride);
  return dsa_launch_status();
}

namespace {
DsaPerDevice g_append_setup;
int append_setup() {
  int dev = 0;
  return dsa_device_setup(g_append_setup, &dev, [](int) {
    DSA_CUDA_TRY(dsa_prefer_shared(k_append<false>));
    DSA_CUDA_TRY(dsa_prefer_shared(k_append<true>));
    return DSA_OK;
  });
}
}  // namespace

extern "C" int kv_append_writeback(const dsa_unit* units, int32_t U, int32_t A,
                                   const uint8_t* new_rows, const uint16_t* new_keys,
                                   int32_t* dev_err, void* stream) {
  if (!units || !new_rows || !new_keys || U < 1 || U > 65535 || A < 1 || A > DSA_RING_ROWS)
    return DSA_ERR_ARG;
  if (const int ok = append_setup(); ok != DSA_OK) return ok;
  return launch_pdl(k_append<false>, dim3(U), dim3(APP_THREADS), 0, static_cast<cudaStream_t>(stream), units, A,
                    new_rows, new_keys, dev_err, (const uint16_t*)nullptr);
}

extern "C" int kv_append_quantize(const dsa_unit* units, int32_t U, int32_t A, const uint16_t* new_latent,
                                  const uint16_t* new_rope, const uint16_t* new_keys, int32_t* dev_err,
                                  void* stream) {
  if (!units || !new_latent || !new_rope || !new_keys || U < 1 || U > 65535 || A < 1 || A > DSA_RING_ROWS)
    return DSA_ERR_ARG;
  if (const int ok = append_setup(); ok != DSA_OK) return ok;
  return launch_pdl(k_append<true>, dim3(U), dim3(APP_THREADS), 0, static_cast<cudaStream_t>(stream), units, A,
                    reinterpret_cast<const uint8_t*>(new_latent), new_keys, dev_err, new_rope);
}

extern "C" int kv_flush(const dsa_unit* units, int32_t U, int32_t* dev_err, void* stream) {
  (void)dev_err;
  if (!units || U < 1 || U > 65535) return DSA_ERR_ARG;
  k_flush<<<U, APP_THREADS, 0, static_cast<cudaStream_t>(stream)>>>(units);
  return dsa_launch_status();
}
