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
// cudaGetSymbolAddress, once per device, on the first call made while that
// device is current, and cached.

#include <mutex>

#include "mep_common.cuh"

namespace {

__device__ __align__(256) unsigned char g_plan_scratch[MEP_PLAN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of g_plan_scratch on the current device (nullptr on error).
void* plan_scratch_on_current_device() {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess) return nullptr;
    addr[dev] = p;
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
