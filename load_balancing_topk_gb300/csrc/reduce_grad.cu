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
// thread loads the home vector and all of the expert's slot vectors (all in
// flight together), adds them in (r, b) order in fp32, writes the home
// vector and writes zeros over the consumed slot vectors. Vectors are
// 32 bytes (8 floats, ld/st .v8) when H*H' % 8 == 0 and both buffers are
// 32-byte aligned, else 16 bytes, else single floats.

#include "mep_common.cuh"

namespace mep {
namespace {

constexpr int kThreads = 256;
#ifndef MEP_REDUCE_CTAS_PER_SM
#define MEP_REDUCE_CTAS_PER_SM 2
#endif
#ifndef MEP_REDUCE_V32
#define MEP_REDUCE_V32 1  // 32-byte accesses when the sizes and addresses allow
#endif
#ifndef MEP_REDUCE_THREAD_BYTES
#define MEP_REDUCE_THREAD_BYTES 64  // bytes of each matrix a thread moves per item
#endif
#ifndef MEP_REDUCE_SLOT_BATCH
#define MEP_REDUCE_SLOT_BATCH 4
#endif
constexpr int kSlotBatch = MEP_REDUCE_SLOT_BATCH;  // slot vectors loaded together
// vectors of W floats per thread per item
template <int W> __host__ __device__ constexpr int vec_per_thread() {
  return MEP_REDUCE_THREAD_BYTES / (4 * W) > 0 ? MEP_REDUCE_THREAD_BYTES / (4 * W) : 1;
}

// W consecutive fp32 values moved as one access: 1 (scalar), 4 (16 bytes) or
// 8 (32 bytes, ld/st .v8, sm_100 and later). Every access is volatile asm or
// volatile-equivalent so that a slot load is never moved past the store of
// zeros to the same address. Home loads and stores use the default caching;
// slot loads and the zero stores stream (.cs): nothing reads them again.
template <int W> struct Vec;
template <> struct Vec<1> {
  float v[1];
  static __device__ __forceinline__ Vec ld(const float* p) { return Vec{{*p}}; }
  static __device__ __forceinline__ Vec ld_cs(const float* p) { return Vec{{__ldcs(p)}}; }
  __device__ __forceinline__ void st(float* p) const { *p = v[0]; }
  static __device__ __forceinline__ void st_zero_cs(float* p) { __stcs(p, 0.f); }
};
template <> struct Vec<4> {
  float v[4];
  static __device__ __forceinline__ Vec from(const float4& q) { return Vec{{q.x, q.y, q.z, q.w}}; }
  static __device__ __forceinline__ Vec ld(const float* p) {
    return from(*reinterpret_cast<const float4*>(p));
  }
  static __device__ __forceinline__ Vec ld_cs(const float* p) {
    return from(__ldcs(reinterpret_cast<const float4*>(p)));
  }
  __device__ __forceinline__ void st(float* p) const {
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  }
  static __device__ __forceinline__ void st_zero_cs(float* p) {
    __stcs(reinterpret_cast<float4*>(p), make_float4(0.f, 0.f, 0.f, 0.f));
  }
};
template <> struct Vec<8> {
  float v[8];
  static __device__ __forceinline__ Vec ld(const float* p) {
    Vec r;
    asm volatile("ld.global.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3]), "=f"(r.v[4]),
                   "=f"(r.v[5]), "=f"(r.v[6]), "=f"(r.v[7])
                 : "l"(p)
                 : "memory");
    return r;
  }
  static __device__ __forceinline__ Vec ld_cs(const float* p) {
    Vec r;
    asm volatile("ld.global.cs.v8.f32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3]), "=f"(r.v[4]),
                   "=f"(r.v[5]), "=f"(r.v[6]), "=f"(r.v[7])
                 : "l"(p)
                 : "memory");
    return r;
  }
  __device__ __forceinline__ void st(float* p) const {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "f"(v[0]),
                 "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
  }
  static __device__ __forceinline__ void st_zero_cs(float* p) {
    asm volatile("st.global.cs.v8.f32 [%0], {%1, %1, %1, %1, %1, %1, %1, %1};" ::"l"(p), "f"(0.f)
                 : "memory");
  }
};

template <int W>
__device__ __forceinline__ void add_rn(Vec<W>& a, const Vec<W>& b) {
#pragma unroll
  for (int j = 0; j < W; ++j) a.v[j] = __fadd_rn(a.v[j], b.v[j]);
}

template <int W>
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

  constexpr int kVecPerThread = vec_per_thread<W>();
  const long long nvec = HHp / W;  // vectors per matrix (the host checks HHp % W == 0)
  const long long per_item = (long long)kThreads * kVecPerThread;
  const long long nchunk = (nvec + per_item - 1) / per_item;
  const long long items = (long long)nused * nchunk;
  for (long long it = blockIdx.x; it < items; it += gridDim.x) {
    const int ue = int(it / nchunk);
    const long long c = it - (long long)ue * nchunk;
    const int e = s_used[ue];
    const int nb = s_cnt[e];
    const int* lst = s_list + s_beg[e];
    float* h = home + (long long)e * HHp;
    Vec<W> acc[kVecPerThread];
    long long off[kVecPerThread];  // float offset of this thread's vector v in a matrix
    bool in[kVecPerThread];
#pragma unroll
    for (int v = 0; v < kVecPerThread; ++v) {
      const long long i = c * per_item + (long long)v * kThreads + tid;
      in[v] = i < nvec;
      off[v] = i * W;
      if (in[v]) acc[v] = Vec<W>::ld(h + off[v]);
    }
    for (int b0 = 0; b0 < nb; b0 += kSlotBatch) {
      Vec<W> q[kSlotBatch][kVecPerThread];
#pragma unroll
      for (int j = 0; j < kSlotBatch; ++j) {
        if (b0 + j < nb) {
          const float* src = slot + (long long)lst[b0 + j] * HHp;
#pragma unroll
          for (int v = 0; v < kVecPerThread; ++v)
            if (in[v]) q[j][v] = Vec<W>::ld_cs(src + off[v]);
        }
      }
#pragma unroll
      for (int j = 0; j < kSlotBatch; ++j) {
        if (b0 + j < nb) {
          float* dst = slot + (long long)lst[b0 + j] * HHp;
#pragma unroll
          for (int v = 0; v < kVecPerThread; ++v)
            if (in[v]) {
              add_rn(acc[v], q[j][v]);
              Vec<W>::st_zero_cs(dst + off[v]);
            }
        }
      }
    }
#pragma unroll
    for (int v = 0; v < kVecPerThread; ++v)
      if (in[v]) acc[v].st(h + off[v]);
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
  // widest access the sizes and addresses allow
  const bool v8 = MEP_REDUCE_V32 && HHp % 8 == 0 && (reinterpret_cast<uintptr_t>(home_grad) & 31u) == 0 &&
                  (reinterpret_cast<uintptr_t>(slot_grad) & 31u) == 0;
  const int W = v8 ? 8 : HHp % 4 == 0 ? 4 : 1;
  const int smem = int(sizeof(int)) * (4 * E + 2 + RB);
  const void* fn = W == 8   ? reinterpret_cast<const void*>(k_reduce_grad<8>)
                   : W == 4 ? reinterpret_cast<const void*>(k_reduce_grad<4>)
                            : reinterpret_cast<const void*>(k_reduce_grad<1>);
  if (set_max_dynamic_smem(fn, smem)) return MEP_ERR_CUDA;
  const int grid = sm_count() * MEP_REDUCE_CTAS_PER_SM;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t err =
      W == 8   ? launch_pdl(k_reduce_grad<8>, dim3(grid), dim3(kThreads), smem, st, slot_expert, E,
                            RB, (long long)HHp, home_grad, slot_grad, status)
      : W == 4 ? launch_pdl(k_reduce_grad<4>, dim3(grid), dim3(kThreads), smem, st, slot_expert, E,
                            RB, (long long)HHp, home_grad, slot_grad, status)
               : launch_pdl(k_reduce_grad<1>, dim3(grid), dim3(kThreads), smem, st, slot_expert, E,
                            RB, (long long)HHp, home_grad, slot_grad, status);
  return err == cudaSuccess ? MEP_OK : MEP_ERR_CUDA;
}
