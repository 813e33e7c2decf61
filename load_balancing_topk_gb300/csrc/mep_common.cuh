// mep_common.cuh -- device helpers shared by the sm_103a kernels of the
// dynamic-redundant-expert hot path (warp scans, status word, dependent launch).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "mep.h"

#define MEP_FULL_MASK 0xffffffffu

namespace mep {

// ---------------------------------------------------------------------------
// device status word: the first nonzero code wins, later ones are dropped.
__device__ __forceinline__ void set_status(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

__device__ __forceinline__ int read_status(const int32_t* status) {
  if (status == nullptr) return 0;
  return *reinterpret_cast<const volatile int32_t*>(status);
}

// ---------------------------------------------------------------------------
// warp / block scans (32-wide warps)
__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    int n = __shfl_up_sync(MEP_FULL_MASK, v, d);
    if (lane >= d) v += n;
  }
  return v;
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Exclusive scan of in[0..n) into out[0..n) (may alias), out[n] = total when
// write_total. All threads of the block must call it; s_warp holds >= 33 ints.
// Ends with __syncthreads().
__device__ __forceinline__ void block_excl_scan(const int* in, int* out, int n, int* s_warp,
                                                bool write_total) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = (nthr + 31) >> 5;
  const int per = (n + nthr - 1) / nthr;
  const int beg = min(n, tid * per), end = min(n, beg + per);
  int local = 0;
  for (int i = beg; i < end; ++i) local += in[i];
  int incl = warp_incl_scan(local);
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = (lane < nwarps) ? s_warp[lane] : 0;
    int vi = warp_incl_scan(v);
    s_warp[lane] = vi - v;
    if (lane == 31) s_warp[32] = vi;
  }
  __syncthreads();
  int run = s_warp[warp] + incl - local;
  for (int i = beg; i < end; ++i) {
    int v = in[i];
    out[i] = run;
    run += v;
  }
  if (write_total && tid == 0) out[n] = s_warp[32];
  __syncthreads();
}

// ---------------------------------------------------------------------------
// programmatic dependent launch: a kernel launched with
// launch_pdl() may start while its predecessor in the stream is finishing;
// it must call pdl_wait() before touching anything the predecessor writes.
// pdl_launch_dependents() lets the next kernel in the stream start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Ask L2 for the line that holds p (a valid global address); no value is
// returned, so it may precede pdl_wait() even where p is written upstream.
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(__cvta_generic_to_global(p)));
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------------------
// host helpers (defined in abi.cu)
int sm_count();                                     // SMs of the current device
int set_max_dynamic_smem(const void* func, int bytes);  // cudaFuncSetAttribute, cached

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace mep
