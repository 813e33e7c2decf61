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
// twin of reduce_grad. One launch of 16 CTAs of 128 threads per SM. Every CTA lists
// the used slots (warp ballots over the slot map, one part of the map per
// warp), so that all CTAs agree on one ascending list without talking to
// each other. The used slots' vectors, concatenated in that order, are cut
// into items of equal length (at most kUnroll 16-byte vectors per thread),
// as many as a whole number of rounds of the grid needs, and the CTAs take
// them grid-stride: at any moment the grid copies one contiguous stretch of
// memory, and every CTA does the same number of rounds. An item may cross
// from one slot into the next; all loads of an item are in flight before its
// stores.

#include "mep_common.cuh"

namespace mep {
namespace {

#ifndef MEP_PREFETCH_THREADS
#define MEP_PREFETCH_THREADS 128
#endif
constexpr int kThreads = MEP_PREFETCH_THREADS;
constexpr int kWarps = kThreads / 32;
#ifndef MEP_PREFETCH_UNROLL
#define MEP_PREFETCH_UNROLL 8
#endif
constexpr int kUnroll = MEP_PREFETCH_UNROLL;  // 16-byte vectors per thread in flight
constexpr int kExpertBits = 12;  // E <= MEP_MAX_E = 4096 fits 12 bits of a list entry
static_assert(MEP_MAX_E <= (1 << kExpertBits), "expert ids must fit a list entry");
static_assert(MEP_MAX_SLOTS <= (1 << (31 - kExpertBits)), "slot ids must fit a list entry");
#ifndef MEP_PREFETCH_CTAS_PER_SM
#define MEP_PREFETCH_CTAS_PER_SM 16
#endif

constexpr int kExpertMask = (1 << kExpertBits) - 1;

// One item of the copy: `len` list vectors from list slot u, offset off
// (this thread's first vector; later ones follow kThreads apart).
struct Item {
  int u, off, len;
};

// Issue the loads of this CTA's item of round r into q; false when the CTA
// has no item in that round.
__device__ __forceinline__ bool load_item(long long r, long long rounds, int ipv, long long V,
                                          int nv, const int* s_list,
                                          const uint4* __restrict__ home, Item& it,
                                          uint4 (&q)[kUnroll]) {
  if (r >= rounds) return false;
  const long long beg = (r * gridDim.x + blockIdx.x) * ipv;
  if (beg >= V) return false;
  it.len = int(min(V - beg, (long long)ipv));
  it.u = int(beg / nv);
  it.off = int(beg - (long long)it.u * nv) + threadIdx.x;
  while (it.off >= nv) {
    it.off -= nv;
    ++it.u;
  }
  int u = it.u, off = it.off;
#pragma unroll
  for (int k = 0; k < kUnroll; ++k) {
    if (k * kThreads + int(threadIdx.x) < it.len) {
      q[k] = __ldg(home + (long long)(s_list[u] & kExpertMask) * nv + off);
      off += kThreads;
      while (off >= nv) {
        off -= nv;
        ++u;
      }
    }
  }
  return true;
}

__device__ __forceinline__ void store_item(const Item& it, int nv, const int* s_list,
                                           uint4* __restrict__ slot, const uint4 (&q)[kUnroll]) {
  int u = it.u, off = it.off;
#pragma unroll
  for (int k = 0; k < kUnroll; ++k) {
    if (k * kThreads + int(threadIdx.x) < it.len) {
      slot[(long long)(s_list[u] >> kExpertBits) * nv + off] = q[k];
      off += kThreads;
      while (off >= nv) {
        off -= nv;
        ++u;
      }
    }
  }
}

#ifndef MEP_PREFETCH_MIN_BLOCKS
#define MEP_PREFETCH_MIN_BLOCKS 8
#endif

__global__ void __launch_bounds__(kThreads, MEP_PREFETCH_MIN_BLOCKS)
    k_prefetch(const int32_t* __restrict__ slot_expert, int E, int RB, long long nvec,
               const uint4* __restrict__ home, uint4* __restrict__ slot, int32_t* status) {
  pdl_wait();
  pdl_launch_dependents();
  extern __shared__ int s_list[];  // [RB] used slots, ascending: (slot << kExpertBits) | expert
  __shared__ int s_cnt[kWarps], s_bad[kWarps], s_stat;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int st = threadIdx.x == 0 ? read_status(status) : 0;  // in flight with the map loads
  // warp w owns the 32-slot steps [j0, j1) of the map
  const int nsteps = (RB + 31) >> 5;
  const int spw = (nsteps + kWarps - 1) / kWarps;
  const int j0 = min(nsteps, warp * spw), j1 = min(nsteps, j0 + spw);
  int n = 0;
  bool bad = false;
  for (int j = j0; j < j1; ++j) {
    const int sl = (j << 5) + lane;
    const int e = sl < RB ? __ldg(slot_expert + sl) : -1;
    bad = bad || e < -1 || e >= E;
    n += __popc(__ballot_sync(MEP_FULL_MASK, e >= 0 && e < E));
  }
  bad = __any_sync(MEP_FULL_MASK, bad);
  if (lane == 0) {
    s_cnt[warp] = n;
    s_bad[warp] = bad ? 1 : 0;
  }
  if (threadIdx.x == 0) s_stat = st;
  __syncthreads();
  int off = 0, used = 0, any_bad = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    off += w < warp ? s_cnt[w] : 0;
    used += s_cnt[w];
    any_bad |= s_bad[w];
  }
  if (s_stat != 0) return;  // uniform: one status word
  if (any_bad) {
    if (blockIdx.x == 0 && threadIdx.x == 0) set_status(status, MEP_ERR_BAD_SLOT_MAP);
    return;
  }
  for (int j = j0; j < j1; ++j) {  // the same loads again (L1), now placed in the list
    const int sl = (j << 5) + lane;
    const int e = sl < RB ? __ldg(slot_expert + sl) : -1;
    const unsigned m = __ballot_sync(MEP_FULL_MASK, e >= 0);
    if (e >= 0) s_list[off + __popc(m & lanemask_lt())] = (sl << kExpertBits) | e;
    off += __popc(m);
  }
  __syncthreads();

  const long long V = (long long)used * nvec;
  if (V == 0) return;
  const long long cap = (long long)gridDim.x * kThreads * kUnroll;  // vectors per round
  const long long rounds = (V + cap - 1) / cap;
  const int ipv = int((V + rounds * gridDim.x - 1) / (rounds * gridDim.x));  // <= kThreads * kUnroll
  const int nv = int(nvec);  // < 2^31 (checked on the host)

  uint4 q[kUnroll];
  Item it;
  for (long long r = 0; load_item(r, rounds, ipv, V, nv, s_list, home, it, q); ++r)
    store_item(it, nv, s_list, slot, q);
}

}  // namespace
}  // namespace mep

using namespace mep;

extern "C" int mep_prefetch(const int32_t* slot_expert, int E, int R, int B, int64_t expert_bytes,
                            const void* home_w, void* slot_w, int32_t* status, void* stream) {
  // in-slot vector offsets are 32-bit and reach nvec + 2 * kThreads before
  // they wrap into the next slot: keep that below 2^31
  if (E < 1 || E > MEP_MAX_E || R < 1 || B < 0 || expert_bytes < 0 || expert_bytes % 16 != 0 ||
      expert_bytes / 16 > 0x7fffffffLL - 2 * kThreads)
    return MEP_ERR_INVALID_ARG;
  if ((long long)R * B > MEP_MAX_SLOTS) return MEP_ERR_INVALID_ARG;
  const int RB = R * B;
  if (RB == 0 || expert_bytes == 0) return MEP_OK;
  if (slot_expert == nullptr || home_w == nullptr || slot_w == nullptr) return MEP_ERR_INVALID_ARG;
  if (!aligned16(home_w) || !aligned16(slot_w)) return MEP_ERR_INVALID_ARG;
  const int smem = int(sizeof(int)) * RB;
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(k_prefetch), smem)) return MEP_ERR_CUDA;
  // 16 CTAs per SM (about 1.6 waves at 47 registers: measured faster than one
  // wave on both a sparse and a full slot map); fewer when even a full slot
  // map holds less work
  const long long nvec = expert_bytes / 16;
  const long long max_rounds = ((long long)RB * nvec + kThreads * kUnroll - 1) / (kThreads * kUnroll);
  const int grid = int(max_rounds < (long long)sm_count() * MEP_PREFETCH_CTAS_PER_SM
                           ? max_rounds
                           : (long long)sm_count() * MEP_PREFETCH_CTAS_PER_SM);
  const cudaError_t err =
      launch_pdl(k_prefetch, dim3(grid), dim3(kThreads), smem, static_cast<cudaStream_t>(stream),
                 slot_expert, E, RB, nvec,
                 static_cast<const uint4*>(home_w), static_cast<uint4*>(slot_w), status);
  return err == cudaSuccess ? MEP_OK : MEP_ERR_CUDA;
}
