// reduce_grad.cu -- redundant-slot gradients folded into home-expert gradients.
//
// Source: "月之暗面开源MoonEP：面向MoE训练的专家并行通信库", section
// 内存契约与权重布局, gradient paragraph: training keeps fp32 [E+B, H, H']
// gradients whose slot rows [E, E+B) live in a separate reduce buffer; the R
// reduce buffers are seen as one [R, B, H, H'] view; reduce_grad reads the
// matching slots from all ranks, accumulates them into the local parameter
// gradient and zeroes the consumed slots. "Moonshot AI Open-Sources MoonEP for
// Expert Parallelism", paragraph 3: redundant-expert gradients are reduced
// back to their home ranks.
//
// One persistent launch. Every CTA first turns slot_expert [R, B] into, per
// expert, the list of its slots in (r, b) order (warp-aggregated stable
// counting in shared memory), and the list of experts that have slots. The
// work is then (used expert, element chunk) items, walked grid-stride: each
// thread loads the home vector and all of the expert's slot vectors (16-byte
// float4, all in flight together), adds them in (r, b) order in fp32, writes
// the home vector and writes zeros over the consumed slot vectors.

#include "mep_common.cuh"

namespace mep {
namespace {

constexpr int kThreads = 256;
#ifndef MEP_REDUCE_VEC
#define MEP_REDUCE_VEC 4
#endif
#ifndef MEP_REDUCE_CTAS_PER_SM
#define MEP_REDUCE_CTAS_PER_SM 2
#endif
constexpr int kVecPerThread = MEP_REDUCE_VEC;  // float4 vectors per thread per item
#ifndef MEP_REDUCE_SLOT_BATCH
#define MEP_REDUCE_SLOT_BATCH 4
#endif
constexpr int kSlotBatch = MEP_REDUCE_SLOT_BATCH;  // slot vectors loaded together

__device__ __forceinline__ void add4(float4& a, const float4& b) {
  a.x = __fadd_rn(a.x, b.x);
  a.y = __fadd_rn(a.y, b.y);
  a.z = __fadd_rn(a.z, b.z);
  a.w = __fadd_rn(a.w, b.w);
}

template <bool VEC>
__global__ void __launch_bounds__(kThreads)
    k_reduce_grad(const int32_t* __restrict__ slot_expert, int E, int RB, long long HHp,
                  float* __restrict__ home, float* __restrict__ slot, int32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  if (read_status(status) != 0) return;
  extern __shared__ int smem[];
  int* s_cnt = smem;            // [E]   slots per expert
  int* s_beg = s_cnt + E;       // [E+1] exclusive prefix
  int* s_fill = s_beg + E + 1;  // [E+1] running fill, then used-expert numbering
  int* s_list = s_fill + E + 1; // [RB]  flat slot ids grouped by expert, (r,b) order
  int* s_used = s_list + RB;    // [E]   experts with >= 1 slot, ascending
  __shared__ int s_warp[33];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) s_bad = 0;
  for (int e = tid; e < E; e += blockDim.x) {
    s_cnt[e] = 0;
    s_fill[e] = 0;
  }
  __syncthreads();
  for (int s = tid; s < RB; s += blockDim.x) {
    const int e = __ldg(slot_expert + s);
    if (e < -1 || e >= E) s_bad = 1;
    else if (e >= 0) atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  if (s_bad) {
    if (blockIdx.x == 0 && tid == 0) set_status(status, MEP_ERR_BAD_SLOT_MAP);
    return;
  }
  block_excl_scan(s_cnt, s_beg, E, s_warp, true);
  // stable placement by one warp: slots in ascending flat (r, b) order
  if (warp == 0) {
    for (int s0 = 0; s0 < RB; s0 += 32) {
      const int s = s0 + lane;
      const int e = s < RB ? __ldg(slot_expert + s) : -1;
      const unsigned m = __ballot_sync(MEP_FULL_MASK, e >= 0);
      if (e >= 0) {
        const unsigned peers = __match_any_sync(m, e);
        const int cur = s_fill[e];
        s_list[s_beg[e] + cur + __popc(peers & lanemask_lt())] = s;
        __syncwarp(m);
        if (lane == __ffs(peers) - 1) s_fill[e] = cur + __popc(peers);
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // used experts, ascending
  for (int e = tid; e < E; e += blockDim.x) s_fill[e] = s_cnt[e] > 0 ? 1 : 0;
  __syncthreads();
  block_excl_scan(s_fill, s_fill, E, s_warp, true);
  for (int e = tid; e < E; e += blockDim.x)
    if (s_cnt[e] > 0) s_used[s_fill[e]] = e;
  __syncthreads();
  const int nused = s_fill[E];

  const long long nvec = VEC ? HHp / 4 : HHp;  // vectors (or scalars) per matrix
  const long long per_item = (long long)kThreads * kVecPerThread;
  const long long nchunk = (nvec + per_item - 1) / per_item;
  const long long items = (long long)nused * nchunk;
  for (long long it = blockIdx.x; it < items; it += gridDim.x) {
    const int ue = int(it / nchunk);
    const long long c = it - (long long)ue * nchunk;
    const int e = s_used[ue];
    const int nb = s_cnt[e];
    const int* lst = s_list + s_beg[e];
    if constexpr (VEC) {
      float4* h4 = reinterpret_cast<float4*>(home) + (long long)e * nvec;
      float4* sl4 = reinterpret_cast<float4*>(slot);
      float4 acc[kVecPerThread];
      long long idx[kVecPerThread];
#pragma unroll
      for (int v = 0; v < kVecPerThread; ++v) {
        idx[v] = c * per_item + (long long)v * kThreads + tid;
        acc[v] = idx[v] < nvec ? h4[idx[v]] : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int b0 = 0; b0 < nb; b0 += kSlotBatch) {
        float4 q[kSlotBatch][kVecPerThread];
#pragma unroll
        for (int j = 0; j < kSlotBatch; ++j) {
          if (b0 + j < nb) {
            const float4* src = sl4 + (long long)lst[b0 + j] * nvec;
#pragma unroll
            for (int v = 0; v < kVecPerThread; ++v)
              if (idx[v] < nvec) q[j][v] = __ldcs(src + idx[v]);
          }
        }
#pragma unroll
        for (int j = 0; j < kSlotBatch; ++j) {
          if (b0 + j < nb) {
            float4* dst = sl4 + (long long)lst[b0 + j] * nvec;
#pragma unroll
            for (int v = 0; v < kVecPerThread; ++v)
              if (idx[v] < nvec) {
                add4(acc[v], q[j][v]);
                __stcs(dst + idx[v], make_float4(0.f, 0.f, 0.f, 0.f));
              }
          }
        }
      }
#pragma unroll
      for (int v = 0; v < kVecPerThread; ++v)
        if (idx[v] < nvec) h4[idx[v]] = acc[v];
    } else {
      float* h = home + (long long)e * nvec;
#pragma unroll
      for (int v = 0; v < kVecPerThread; ++v) {
        const long long i = c * per_item + (long long)v * kThreads + tid;
        if (i >= nvec) continue;
        float acc = h[i];
        for (int b = 0; b < nb; ++b) {
          float* src = slot + (long long)lst[b] * nvec + i;
          acc = __fadd_rn(acc, *src);
          *src = 0.f;
        }
        h[i] = acc;
      }
    }
  }
}

}  // namespace
}  // namespace mep

using namespace mep;

extern "C" int mep_reduce_grad(const int32_t* slot_expert, int E, int R, int B, int64_t HHp,
                               float* home_grad, float* slot_grad, int32_t* status,
                               void* stream) {
  if (E < 1 || E > MEP_MAX_E || R < 1 || B < 0 || HHp < 0) return MEP_ERR_INVALID_ARG;
  if ((long long)R * B > MEP_MAX_SLOTS) return MEP_ERR_INVALID_ARG;
  const int RB = R * B;
  if (RB == 0 || HHp == 0) return MEP_OK;
  if (slot_expert == nullptr || home_grad == nullptr || slot_grad == nullptr)
    return MEP_ERR_INVALID_ARG;
  if (!aligned16(home_grad) || !aligned16(slot_grad)) return MEP_ERR_INVALID_ARG;
  const bool vec = (HHp % 4) == 0;
  const int smem = int(sizeof(int)) * (4 * E + 2 + RB);
  const void* fn = vec ? reinterpret_cast<const void*>(k_reduce_grad<true>)
                       : reinterpret_cast<const void*>(k_reduce_grad<false>);
  if (set_max_dynamic_smem(fn, smem)) return MEP_ERR_CUDA;
  const int grid = sm_count() * MEP_REDUCE_CTAS_PER_SM;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t err =
      vec ? launch_pdl(k_reduce_grad<true>, dim3(grid), dim3(kThreads), smem, st, slot_expert, E,
                       RB, (long long)HHp, home_grad, slot_grad, status)
          : launch_pdl(k_reduce_grad<false>, dim3(grid), dim3(kThreads), smem, st, slot_expert,
                       E, RB, (long long)HHp, home_grad, slot_grad, status);
  return err == cudaSuccess ? MEP_OK : MEP_ERR_CUDA;
}
