// prefetch.cu -- replica weight prefetch into the redundant slots (mep_prefetch).
//
// Source: "月之暗面开源MoonEP：面向MoE训练的专家并行通信库", section 核心技术
// (the weights of the redundant experts planned from the current routing are
// prefetched before expert compute) and section 内存契约与权重布局 (each
// projection's weight tensor has E home rows, E/R per rank, and B local
// prefetch slot rows [E, E+B)). "Moonshot AI Open-Sources MoonEP for Expert
// Parallelism", paragraph 3: duplicated experts are prefetched before expert
// computation.
//
// slot_w[r][b] = home_w[slot_expert[r][b]] for every used slot: the forward
// twin of reduce_grad. One persistent launch; every CTA lists the used slots
// in ascending (r, b) order (warp ballots), then walks (used slot, 16 KB
// chunk) items grid-stride, each thread moving 4 x 16-byte vectors (all
// loads in flight before the stores).

#include "mep_common.cuh"

namespace mep {
namespace {

constexpr int kThreads = 256;
constexpr int kVec = 4;  // 16-byte vectors per thread per item
#ifndef MEP_PREFETCH_CTAS_PER_SM
#define MEP_PREFETCH_CTAS_PER_SM 16
#endif

__global__ void __launch_bounds__(kThreads)
    k_prefetch(const int32_t* __restrict__ slot_expert, int E, int RB, long long nvec,
               const uint4* __restrict__ home, uint4* __restrict__ slot, int32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  if (read_status(status) != 0) return;
  extern __shared__ int s_used[];  // [RB] used slot ids, ascending
  __shared__ int s_n, s_bad;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int n = 0;
    bool bad = false;
    for (int s0 = 0; s0 < RB; s0 += 32) {
      const int s = s0 + lane;
      const int e = s < RB ? __ldg(slot_expert + s) : -1;
      bad = bad || e < -1 || e >= E;
      const unsigned m = __ballot_sync(MEP_FULL_MASK, e >= 0 && e < E);
      if (e >= 0 && e < E) s_used[n + __popc(m & lanemask_lt())] = s;
      n += __popc(m);
    }
    const bool any_bad = __any_sync(MEP_FULL_MASK, bad);
    if (lane == 0) {
      s_n = n;
      s_bad = any_bad ? 1 : 0;
    }
  }
  __syncthreads();
  if (s_bad) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, MEP_ERR_BAD_SLOT_MAP);
    return;
  }
  const long long per_item = (long long)kThreads * kVec;
  const long long nchunk = (nvec + per_item - 1) / per_item;
  const long long items = (long long)s_n * nchunk;
  for (long long it = blockIdx.x; it < items; it += gridDim.x) {
    const int u = int(it / nchunk);
    const long long c = it - (long long)u * nchunk;
    const int s = s_used[u];
    const int e = __ldg(slot_expert + s);
    const uint4* src = home + (long long)e * nvec;
    uint4* dst = slot + (long long)s * nvec;
    uint4 q[kVec];
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      const long long i = c * per_item + (long long)v * kThreads + threadIdx.x;
      if (i < nvec) q[v] = __ldg(src + i);
    }
#pragma unroll
    for (int v = 0; v < kVec; ++v) {
      const long long i = c * per_item + (long long)v * kThreads + threadIdx.x;
      if (i < nvec) dst[i] = q[v];
    }
  }
}

}  // namespace
}  // namespace mep

using namespace mep;

extern "C" int mep_prefetch(const int32_t* slot_expert, int E, int R, int B, int64_t expert_bytes,
                            const void* home_w, void* slot_w, int32_t* status, void* stream) {
  if (E < 1 || E > MEP_MAX_E || R < 1 || B < 0 || expert_bytes < 0 || expert_bytes % 16 != 0)
    return MEP_ERR_INVALID_ARG;
  if ((long long)R * B > MEP_MAX_SLOTS) return MEP_ERR_INVALID_ARG;
  const int RB = R * B;
  if (RB == 0 || expert_bytes == 0) return MEP_OK;
  if (slot_expert == nullptr || home_w == nullptr || slot_w == nullptr) return MEP_ERR_INVALID_ARG;
  if (!aligned16(home_w) || !aligned16(slot_w)) return MEP_ERR_INVALID_ARG;
  const int smem = int(sizeof(int)) * RB;
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(k_prefetch), smem)) return MEP_ERR_CUDA;
  const int grid = sm_count() * MEP_PREFETCH_CTAS_PER_SM;
  const cudaError_t err =
      launch_pdl(k_prefetch, dim3(grid), dim3(kThreads), smem, static_cast<cudaStream_t>(stream),
                 slot_expert, E, RB, (long long)(expert_bytes / 16),
                 static_cast<const uint4*>(home_w), static_cast<uint4*>(slot_w), status);
  return err == cudaSuccess ? MEP_OK : MEP_ERR_CUDA;
}
