// plan_static.cu -- mep_plan_static_scratch: mep_plan for callers that cannot
// allocate device memory.
//
// Some callers have no way to allocate: a host program that reaches the GPU
// only through this C ABI and links no allocator of its own, or a runtime
// whose device memory is owned by one pool allocator and that must not
// create allocations behind that pool's back (a stray cudaMalloc escapes its
// accounting and can fail or fragment memory once the pool has claimed the
// device). For them this entry point takes the planner's scratch from a
// fixed array compiled into the library instead of a caller buffer.
//
// The array below is a file-scope __device__ object: every GPU on which the
// library is loaded holds MEP_PLAN_STATIC_SCRATCH_BYTES of it until the
// process exits. In host code its name is only a host-side stand-in for the
// symbol, never a device address: the device address is looked up with
// cudaGetSymbolAddress on the first call made while a device is current, and
// cached per device together with the unique id of the CUDA context it was
// looked up in. A later call in another context (after cudaDeviceReset, or
// once the primary context has been destroyed and created again, which
// reloads the module) looks the address up again instead of using a stale one.

#include <cuda.h>

#include <mutex>

#include "mep_common.cuh"

namespace {

__device__ __align__(256) unsigned char g_plan_scratch[MEP_PLAN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

// Unique id of the current CUDA context (0 when no context is current yet,
// or on error).
unsigned long long current_context_id() {
  static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
      ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of g_plan_scratch on the current device (nullptr on error).
void* plan_scratch_on_current_device() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  static unsigned long long ctx_of[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (ctx == 0 || addr[dev] == nullptr || ctx_of[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess) return nullptr;
    // the lookup makes the device's primary context current if none was
    if (ctx == 0) ctx = current_context_id();
    if (ctx == 0) return nullptr;
    addr[dev] = p;
    ctx_of[dev] = ctx;
  }
  return addr[dev];
}

}  // namespace

extern "C" int mep_plan_static_scratch(const int32_t* topk_idx, int R, int S, int K, int E,
                                       int B, int32_t* expert_counts, int32_t* cu_seqlens,
                                       int32_t* slot_expert, int32_t* dst_pos, int32_t* status,
                                       void* stream) {
  size_t need = 0;
  const int rc = mep_plan_workspace_bytes(R, S, K, E, B, &need);
  if (rc != MEP_OK) return rc;
  if (need > size_t(MEP_PLAN_STATIC_SCRATCH_BYTES)) return MEP_ERR_INVALID_ARG;
  void* scratch = plan_scratch_on_current_device();
  if (scratch == nullptr) return MEP_ERR_CUDA;
  // Every byte of the scratch that the plan kernels read is written earlier
  // in the same call, so nothing needs clearing between calls.
  return mep_plan(topk_idx, R, S, K, E, B, scratch, size_t(MEP_PLAN_STATIC_SCRATCH_BYTES),
                  expert_counts, cu_seqlens, slot_expert, dst_pos, status, stream);
}
