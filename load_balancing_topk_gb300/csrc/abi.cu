// abi.cu -- library-wide entry points and host helpers of the C ABI (mep.h).

#include <mutex>
#include <unordered_map>

#include "mep_common.cuh"

namespace mep {

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
  return n > 0 ? n : 1;
}

// Raise a kernel's dynamic shared-memory limit once per (kernel, device);
// returns nonzero on failure.
int set_max_dynamic_smem(const void* func, int bytes) {
  static std::mutex mu;
  static std::unordered_map<const void*, int> done[64];
  if (bytes <= 48 * 1024) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  std::lock_guard<std::mutex> lock(mu);
  auto it = done[dev].find(func);
  if (it != done[dev].end() && it->second >= bytes) return 0;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return 1;
  done[dev][func] = bytes;
  return 0;
}

}  // namespace mep

extern "C" int mep_version(void) { return (0 << 16) | 1; }

extern "C" const char* mep_status_string(int code) {
  switch (code) {
    case MEP_OK: return "ok";
    case MEP_ERR_INVALID_ARG: return "invalid argument";
    case MEP_ERR_CUDA: return "CUDA launch failure";
    case MEP_ERR_BAD_ROUTING: return "bad routing: expert index out of range or repeated in a row";
    case MEP_ERR_CAPACITY: return "capacity: a rank needs more than B redundant slots";
    case MEP_ERR_BAD_POSITION: return "bad position: dst_pos entry out of range";
    case MEP_ERR_BAD_SLOT_MAP: return "bad slot map: slot_expert entry out of range";
    case MEP_ERR_TIMEOUT: return "timeout: a bounded wait inside a kernel gave up";
    case MEP_ERR_BAD_SEQLENS: return "bad cu_seqlens: a row decreases, is negative or does not end at S*K";
    default: return "unknown status";
  }
}
