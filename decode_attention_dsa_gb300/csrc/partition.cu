// SM partitions of one GPU for the decode step's schedule.
//
// The indexer's score kernel is a persistent grid that holds every SM it may
// use for the whole of its HBM stream, so the rest of a step (selection, slot
// assignment, gather, attention) can run beside it only on SMs it was never
// given. A partition is a green context: a disjoint set of the device's SMs
// whose streams run kernels only there. The device is split in two: the
// scorings run on one partition, the rest of the steps on the other, and
// kernels size their grids to the partition of the stream they are launched
// on (dsa_stream_sms).
//
// Green contexts are driver objects; the calls are reached through the
// runtime's driver entry points, so the library links only the runtime.

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"

struct dsa_partition {
  CUgreenCtx gctx = nullptr;
  std::vector<CUstream> streams;   // owned, destroyed with the partition
  int sms = 0;
};

namespace {

struct DriverFns {
  PFN_cuDeviceGet_v2000 device_get = nullptr;
  PFN_cuDeviceGetDevResource_v12040 get_resource = nullptr;
  PFN_cuDevSmResourceSplitByCount_v12040 split = nullptr;
  PFN_cuDevResourceGenerateDesc_v12040 gen_desc = nullptr;
  PFN_cuGreenCtxCreate_v12040 gctx_create = nullptr;
  PFN_cuGreenCtxDestroy_v12040 gctx_destroy = nullptr;
  PFN_cuGreenCtxStreamCreate_v12050 stream_create = nullptr;
  PFN_cuStreamDestroy_v4000 stream_destroy = nullptr;
  PFN_cuStreamSynchronize_v2000 stream_sync = nullptr;
  PFN_cuStreamGetGreenCtx_v12040 stream_gctx = nullptr;
  PFN_cuStreamGetCtx_v12050 stream_ctx = nullptr;
  PFN_cuGreenCtxGetDevResource_v12040 gctx_resource = nullptr;
  PFN_cuCtxPushCurrent_v4000 ctx_push = nullptr;
  PFN_cuCtxPopCurrent_v4000 ctx_pop = nullptr;
  PFN_cuEventCreate_v2000 event_create = nullptr;
  PFN_cuEventRecord_v2000 event_record = nullptr;
  PFN_cuEventDestroy_v4000 event_destroy = nullptr;
  PFN_cuStreamWaitEvent_v3020 stream_wait = nullptr;
  bool ok = false;
};

template <typename T>
bool entry(const char* name, int version, T* fn) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !p)
    return false;
  *fn = reinterpret_cast<T>(p);
  return true;
}

const DriverFns& driver() {
  static DriverFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    f.ok = entry("cuDeviceGet", 2000, &f.device_get) &&
           entry("cuDeviceGetDevResource", 12040, &f.get_resource) &&
           entry("cuDevSmResourceSplitByCount", 12040, &f.split) &&
           entry("cuDevResourceGenerateDesc", 12040, &f.gen_desc) &&
           entry("cuGreenCtxCreate", 12040, &f.gctx_create) &&
           entry("cuGreenCtxDestroy", 12040, &f.gctx_destroy) &&
           entry("cuGreenCtxStreamCreate", 12050, &f.stream_create) &&
           entry("cuStreamDestroy", 4000, &f.stream_destroy) &&
           entry("cuStreamSynchronize", 2000, &f.stream_sync) &&
           entry("cuStreamGetGreenCtx", 12040, &f.stream_gctx) &&
           entry("cuStreamGetCtx", 12050, &f.stream_ctx) &&
           entry("cuGreenCtxGetDevResource", 12040, &f.gctx_resource) &&
           entry("cuCtxPushCurrent", 4000, &f.ctx_push) && entry("cuCtxPopCurrent", 4000, &f.ctx_pop) &&
           entry("cuEventCreate", 2000, &f.event_create) && entry("cuEventRecord", 2000, &f.event_record) &&
           entry("cuEventDestroy", 4000, &f.event_destroy) &&
           entry("cuStreamWaitEvent", 3020, &f.stream_wait);
  });
  return f;
}

int release(const DriverFns& f, dsa_partition* p) {
  bool ok = true;
  for (CUstream s : p->streams) {
    ok = f.stream_sync(s) == CUDA_SUCCESS && ok;   // its queued work first
    ok = f.stream_destroy(s) == CUDA_SUCCESS && ok;
  }
  if (p->gctx) ok = f.gctx_destroy(p->gctx) == CUDA_SUCCESS && ok;
  delete p;
  return ok ? DSA_OK : DSA_ERR_CUDA;
}

int make_partition(const DriverFns& f, CUdevice dev, CUdevResource* res, unsigned n, unsigned sms,
                   dsa_partition** out) {
  CUdevResourceDesc desc;
  if (f.gen_desc(&desc, res, n) != CUDA_SUCCESS) return DSA_ERR_CUDA;
  dsa_partition* p = new dsa_partition();
  p->sms = (int)sms;
  if (f.gctx_create(&p->gctx, desc, dev, CU_GREEN_CTX_DEFAULT_STREAM) != CUDA_SUCCESS) {
    p->gctx = nullptr;
    release(f, p);
    return DSA_ERR_CUDA;
  }
  *out = p;
  return DSA_OK;
}

}  // namespace

// SMs that kernels launched on `st` may use: the partition's count for a
// stream of a green context, else `device_sms`.
int dsa_stream_sms(cudaStream_t st, int device_sms) {
  if (!st) return device_sms;
  // a stream being captured into a graph is an ordinary stream here (a
  // partition's streams are not captured); no driver query during capture
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess) {
    cudaGetLastError();   // the query's own error
    return device_sms;
  }
  if (cap != cudaStreamCaptureStatusNone) return device_sms;
  const DriverFns& f = driver();
  if (!f.ok) return device_sms;
  CUgreenCtx g = nullptr;
  if (f.stream_gctx(reinterpret_cast<CUstream>(st), &g) != CUDA_SUCCESS || !g) return device_sms;
  CUdevResource r = {};
  if (f.gctx_resource(g, &r, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS || r.sm.smCount < 1) return device_sms;
  return (int)std::min<unsigned>(r.sm.smCount, (unsigned)device_sms);
}

extern "C" int dsa_partition_split(int32_t min_sms, dsa_partition** first, dsa_partition** second) {
  if ((!first && !second) || min_sms < 1) return DSA_ERR_ARG;
  if (first) *first = nullptr;
  if (second) *second = nullptr;
  const DriverFns& f = driver();
  if (!f.ok) return DSA_ERR_CUDA;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  cudaFree(nullptr);   // the primary context exists before a green context retains it
  CUdevice cdev;
  if (f.device_get(&cdev, dev) != CUDA_SUCCESS) return DSA_ERR_CUDA;
  CUdevResource all = {};
  if (f.get_resource(cdev, &all, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS) return DSA_ERR_CUDA;
  if ((unsigned)min_sms >= all.sm.smCount) return DSA_ERR_ARG;
  // The device's SMs as groups that are guaranteed to sit in one GPU
  // processing cluster (the co-scheduling unit), plus the SMs left over. The
  // first partition takes the leftovers (the score kernel launches no thread
  // block clusters), then whole groups until it holds min_sms; the second
  // takes the remaining groups whole, so the clustered kernels of the rest
  // of a step (8-CTA clusters in the Top-K select) find room there.
  const unsigned al = std::max(1u, all.sm.smCoscheduledAlignment);
  unsigned ng = 0;
  if (f.split(nullptr, &ng, &all, nullptr, 0, al) != CUDA_SUCCESS || ng == 0) return DSA_ERR_CUDA;
  std::vector<CUdevResource> res(ng + 1);
  CUdevResource rest = {};
  if (f.split(res.data() + 1, &ng, &all, &rest, 0, al) != CUDA_SUCCESS) return DSA_ERR_CUDA;
  unsigned lo = 1, got = 0;
  if (rest.type == CU_DEV_RESOURCE_TYPE_SM && rest.sm.smCount > 0) {
    res[0] = rest;
    lo = 0;
    got = rest.sm.smCount;
  }
  unsigned end = 1;
  while (end <= ng && got < (unsigned)min_sms) got += res[end++].sm.smCount;
  if (got < (unsigned)min_sms || (second && end > ng)) return DSA_ERR_ARG;   // nothing left for the second
  unsigned got2 = 0;
  for (unsigned i = end; i <= ng; ++i) got2 += res[i].sm.smCount;
  dsa_partition* p1 = nullptr;
  dsa_partition* p2 = nullptr;
  if (first) {
    const int st = make_partition(f, cdev, res.data() + lo, end - lo, got, &p1);
    if (st != DSA_OK) return st;
  }
  if (second) {
    const int st = make_partition(f, cdev, res.data() + end, ng + 1 - end, got2, &p2);
    if (st != DSA_OK) {
      if (p1) release(f, p1);
      return st;
    }
  }
  if (first) *first = p1;
  if (second) *second = p2;
  return DSA_OK;
}

extern "C" int dsa_partition_sms(const dsa_partition* part) { return part ? part->sms : 0; }

extern "C" int dsa_partition_stream(dsa_partition* part, void** stream) {
  if (!part || !stream) return DSA_ERR_ARG;
  *stream = nullptr;
  const DriverFns& f = driver();
  CUstream s = nullptr;
  if (f.stream_create(&s, part->gctx, CU_STREAM_NON_BLOCKING, 0) != CUDA_SUCCESS) return DSA_ERR_CUDA;
  part->streams.push_back(s);
  *stream = s;
  return DSA_OK;
}

extern "C" int dsa_stream_wait_stream(void* waiter, void* signaller) {
  const DriverFns& f = driver();
  if (!f.ok) return DSA_ERR_CUDA;
  // An event must belong to the context of the stream it is recorded on (a
  // partition's stream belongs to its green context); the wait may cross
  // contexts. So the event is made in the signaller's context, used once and
  // released (its resources go once the wait is satisfied).
  CUcontext ctx = nullptr;
  CUgreenCtx g = nullptr;
  CUstream sig = reinterpret_cast<CUstream>(signaller);
  if (f.stream_ctx(sig, &ctx, &g) != CUDA_SUCCESS || !ctx) return DSA_ERR_CUDA;
  if (f.ctx_push(ctx) != CUDA_SUCCESS) return DSA_ERR_CUDA;
  CUevent ev = nullptr;
  const CUresult rc = f.event_create(&ev, CU_EVENT_DISABLE_TIMING);
  CUcontext popped;
  const CUresult rp = f.ctx_pop(&popped);
  if (rc != CUDA_SUCCESS) return DSA_ERR_CUDA;
  CUresult r = rp;
  if (r == CUDA_SUCCESS) r = f.event_record(ev, sig);
  if (r == CUDA_SUCCESS) r = f.stream_wait(reinterpret_cast<CUstream>(waiter), ev, 0);
  f.event_destroy(ev);
  return r == CUDA_SUCCESS ? DSA_OK : DSA_ERR_CUDA;
}

extern "C" int dsa_partition_destroy(dsa_partition* part) {
  if (!part) return DSA_ERR_ARG;
  return release(driver(), part);
}
