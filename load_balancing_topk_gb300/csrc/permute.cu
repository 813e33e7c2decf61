// permute.cu -- fused permute (mep_dispatch) and weighted unpermute (mep_combine).
//
// Source: "月之暗面开源MoonEP：面向MoE训练的专家并行通信库", section 核心技术
// (零拷贝与静态形状: tokens are written straight into preset, expert-grouped
// positions of one fixed S*K buffer per rank, and the unpermute reads them
// back; the shapes are static so no host sync is needed).
//
// dispatch: each token row is read from HBM once and written K times.
//   Rows move as whole units through shared memory with the bulk-copy
//   engine: one global->shared cp.async.bulk per row chunk (completion on an
//   mbarrier), then K shared->global cp.async.bulk stores, one per lane, so
//   a warp keeps several row loads and K times as many row stores in flight
//   without holding the data in registers. A persistent grid walks the
//   (token, chunk) units; a ring of NS stages lets loads run P units ahead.
// combine: one warp per token; each lane owns 16-byte column vectors and
//   issues the K gathers of a vector before its fp32 fused multiply-add
//   chain (k in order), then writes the bf16 result (nearest-even).

#include <cuda_bf16.h>

#include "mep_common.cuh"

#ifndef MEP_DISPATCH_STAGES
#define MEP_DISPATCH_STAGES 8
#endif
#ifndef MEP_DISPATCH_AHEAD
#define MEP_DISPATCH_AHEAD 4
#endif
#ifndef MEP_DISPATCH_CHUNK
#define MEP_DISPATCH_CHUNK 16384
#endif
#ifndef MEP_DISPATCH_MAX_CTAS_PER_SM
#define MEP_DISPATCH_MAX_CTAS_PER_SM 2
#endif
#ifndef MEP_COMBINE_WARPS
#define MEP_COMBINE_WARPS 4
#endif

namespace mep {
namespace {

constexpr int kStages = MEP_DISPATCH_STAGES;
constexpr int kAhead = MEP_DISPATCH_AHEAD;
static_assert(kAhead >= 1 && kAhead < kStages, "loads run ahead of the ring, not around it");
constexpr uint32_t kMaxPolls = 1u << 24;  // bounded mbarrier wait (about a second)

__global__ void __launch_bounds__(32)
    k_dispatch(const uint8_t* __restrict__ hidden, const int32_t* __restrict__ dst_pos,
               int32_t* status, long long N, int K, long long row_bytes, int chunk_bytes,
               int nchunk, long long nrows, uint8_t* __restrict__ buf) {
  pdl_wait();
  pdl_launch_dependents();
  if (read_status(status) != 0) return;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + size_t(kStages) * chunk_bytes);
  const int lane = threadIdx.x;
  const long long units = N * nchunk;
  const long long first = blockIdx.x, stride = gridDim.x;
  if (first >= units) return;
  const long long n = (units - first + stride - 1) / stride;

  if (lane == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();

  auto unit_of = [&](long long i, long long& t, long long& off, uint32_t& bytes) {
    const long long u = first + i * stride;
    t = u / nchunk;
    const int c = int(u - t * nchunk);
    off = (long long)c * chunk_bytes;
    const long long rem = row_bytes - off;
    bytes = uint32_t(rem < chunk_bytes ? rem : chunk_bytes);
  };
  auto issue_load = [&](long long i) {
    long long t, off;
    uint32_t bytes;
    unit_of(i, t, off, bytes);
    const int s = int(i % kStages);
    mbar_arrive_expect_tx(&bars[s], bytes);
    bulk_g2s(smem + size_t(s) * chunk_bytes, hidden + t * row_bytes + off, bytes, &bars[s]);
  };

  if (lane == 0)
    for (long long i = 0; i < n && i < kAhead; ++i) issue_load(i);

  // destination rows of the current unit, lanes k, k+32, ... (K <= 64)
  auto rows_of = [&](long long i, int& r0, int& r1) {
    long long t, off;
    uint32_t bytes;
    unit_of(i, t, off, bytes);
    r0 = lane < K ? __ldg(dst_pos + t * K + lane) : -1;
    r1 = lane + 32 < K ? __ldg(dst_pos + t * K + lane + 32) : -1;
  };
  int cur0, cur1;
  rows_of(0, cur0, cur1);
  long long i = 0;
  bool timed_out = false;
  for (; i < n; ++i) {
    int nxt0 = -1, nxt1 = -1;
    if (i + 1 < n) rows_of(i + 1, nxt0, nxt1);
    const int s = int(i % kStages);
    const uint32_t parity = uint32_t((i / kStages) & 1);
    // every lane polls; the warp leaves together (bounded)
    for (uint32_t tries = 0;; ++tries) {
      const bool ok = mbar_try_wait(&bars[s], parity);
      if (__all_sync(MEP_FULL_MASK, ok)) break;
      if (tries >= kMaxPolls) {
        timed_out = true;
        break;
      }
    }
    if (timed_out) break;
    long long t, off;
    uint32_t bytes;
    unit_of(i, t, off, bytes);
    const uint8_t* src = smem + size_t(s) * chunk_bytes;
    bool bad = false;
    if (lane < K) {
      if (cur0 >= 0 && cur0 < nrows) bulk_s2g(buf + cur0 * row_bytes + off, src, bytes);
      else bad = true;
    }
    if (lane + 32 < K) {
      if (cur1 >= 0 && cur1 < nrows) bulk_s2g(buf + cur1 * row_bytes + off, src, bytes);
      else bad = true;
    }
    if (bad) set_status(status, MEP_ERR_BAD_POSITION);
    bulk_commit();
    if (i + kAhead < n) {
      // the stage that unit i+kAhead reuses was last read by unit
      // i+kAhead-kStages: at most kStages-kAhead newer groups may be pending
      bulk_wait_read<kStages - kAhead>();
      __syncwarp();
      if (lane == 0) issue_load(i + kAhead);
    }
    cur0 = nxt0;
    cur1 = nxt1;
  }
  if (timed_out) {
    set_status(status, MEP_ERR_TIMEOUT);
    // loads of units [i, min(n, i + kAhead)) were issued and not consumed:
    // give each a bounded chance to land before shared memory is released
    if (lane == 0)
      for (long long u = i; u < n && u < i + kAhead; ++u)
        mbar_wait_bounded(&bars[u % kStages], uint32_t((u / kStages) & 1), kMaxPolls);
  }
  bulk_wait_all();
  __syncwarp();
}

// ---------------------------------------------------------------------------
__device__ __forceinline__ void fma8(float (&acc)[8], float w, uint4 q) {
  const uint32_t v[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float lo = __uint_as_float(v[j] << 16);
    const float hi = __uint_as_float(v[j] & 0xffff0000u);
    acc[2 * j] = __fmaf_rn(w, lo, acc[2 * j]);
    acc[2 * j + 1] = __fmaf_rn(w, hi, acc[2 * j + 1]);
  }
}

__device__ __forceinline__ uint4 pack8(const float (&acc)[8]) {
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
    o[j] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// KT > 0: K known at compile time (all K gathers of a vector in flight at
// once). KT == 0: any K, gathered in batches of 8.
template <int KT>
__global__ void __launch_bounds__(32 * MEP_COMBINE_WARPS)
    k_combine(const uint4* __restrict__ y, const float* __restrict__ topk_w,
              const int32_t* __restrict__ dst_pos, int32_t* status, long long N, int Kr,
              long long vpr, long long nrows, uint4* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  if (read_status(status) != 0) return;
  const int K = KT > 0 ? KT : Kr;
  const int lane = threadIdx.x & 31;
  const long long warp0 = (long long)blockIdx.x * MEP_COMBINE_WARPS + (threadIdx.x >> 5);
  const long long nwarp = (long long)gridDim.x * MEP_COMBINE_WARPS;
  for (long long t = warp0; t < N; t += nwarp) {
    const int r0 = lane < K ? __ldg(dst_pos + t * K + lane) : 0;
    const int r1 = lane + 32 < K ? __ldg(dst_pos + t * K + lane + 32) : 0;
    const float w0 = lane < K ? __ldg(topk_w + t * K + lane) : 0.f;
    const bool bad = (lane < K && (r0 < 0 || r0 >= nrows)) ||
                     (lane + 32 < K && (r1 < 0 || r1 >= nrows));
    if (__any_sync(MEP_FULL_MASK, bad)) {
      if (lane == 0) set_status(status, MEP_ERR_BAD_POSITION);
      continue;
    }
    uint4* o = out + t * vpr;
    if constexpr (KT > 0) {
      long long rows[KT];
      float ws[KT];
#pragma unroll
      for (int k = 0; k < KT; ++k) {
        rows[k] = (long long)__shfl_sync(MEP_FULL_MASK, r0, k) * vpr;
        ws[k] = __shfl_sync(MEP_FULL_MASK, w0, k);
      }
      for (long long v = lane; v < vpr; v += 32) {
        uint4 q[KT];
#pragma unroll
        for (int k = 0; k < KT; ++k) q[k] = __ldg(y + rows[k] + v);
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < KT; ++k) fma8(acc, ws[k], q[k]);
        o[v] = pack8(acc);
      }
    } else {
      for (long long v = lane; v < vpr; v += 32) {
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int k0 = 0; k0 < K; k0 += 8) {
          uint4 q[8];
          float ws[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int k = k0 + j;
            if (k < K) {
              const long long row = __ldg(dst_pos + t * K + k);
              ws[j] = __ldg(topk_w + t * K + k);
              q[j] = __ldg(y + row * vpr + v);
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (k0 + j < K) fma8(acc, ws[j], q[j]);
        }
        o[v] = pack8(acc);
      }
    }
  }
}

template <int KT>
cudaError_t launch_combine(const uint4* y, const float* w, const int32_t* dst, int32_t* status,
                           long long N, int K, long long vpr, long long nrows, uint4* out,
                           cudaStream_t st) {
  const long long want = (N + MEP_COMBINE_WARPS - 1) / MEP_COMBINE_WARPS;
  const long long cap = (long long)sm_count() * 64;
  const int grid = int(want < cap ? want : cap);
  return launch_pdl(k_combine<KT>, dim3(grid), dim3(32 * MEP_COMBINE_WARPS), 0, st, y, w, dst,
                    status, N, K, vpr, nrows, out);
}

}  // namespace
}  // namespace mep

using namespace mep;

static int permute_check(const void* a, const void* b, const void* dst, int R, int S, int K,
                         int H) {
  if (R < 1 || S < 0 || K < 1 || K > MEP_MAX_K || H < 8 || H % 8 != 0) return MEP_ERR_INVALID_ARG;
  if ((long long)R * S * K > 0x7fffffffLL) return MEP_ERR_INVALID_ARG;
  if ((long long)R * S == 0) return MEP_OK;
  if (a == nullptr || b == nullptr || dst == nullptr) return MEP_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b)) return MEP_ERR_INVALID_ARG;
  return MEP_OK;
}

extern "C" int mep_dispatch(const mep_bf16* hidden, const int32_t* dst_pos, int32_t* status,
                            int R, int S, int K, int H, mep_bf16* buf, void* stream) {
  int rc = permute_check(hidden, buf, dst_pos, R, S, K, H);
  if (rc != MEP_OK) return rc;
  const long long N = (long long)R * S;
  if (N == 0) return MEP_OK;
  const long long row_bytes = (long long)H * 2;
  const int chunk = int(row_bytes < MEP_DISPATCH_CHUNK ? row_bytes : MEP_DISPATCH_CHUNK);
  const int nchunk = int((row_bytes + chunk - 1) / chunk);
  const int smem = kStages * chunk + kStages * 8;
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(k_dispatch), smem)) return MEP_ERR_CUDA;
  const long long units = N * nchunk;
  // as many rings per SM as fit its shared memory, up to the cap
  int per_sm = (220 * 1024) / smem;
  per_sm = per_sm < 1 ? 1 : (per_sm > MEP_DISPATCH_MAX_CTAS_PER_SM ? MEP_DISPATCH_MAX_CTAS_PER_SM : per_sm);
  const long long cap = (long long)sm_count() * per_sm;
  const int grid = int(units < cap ? units : cap);
  const cudaError_t err =
      launch_pdl(k_dispatch, dim3(grid), dim3(32), smem, static_cast<cudaStream_t>(stream),
                 reinterpret_cast<const uint8_t*>(hidden), dst_pos, status, N, K, row_bytes,
                 chunk, nchunk, N * K, reinterpret_cast<uint8_t*>(buf));
  return err == cudaSuccess ? MEP_OK : MEP_ERR_CUDA;
}

extern "C" int mep_combine(const mep_bf16* y, const float* topk_w, const int32_t* dst_pos,
                           int32_t* status, int R, int S, int K, int H, mep_bf16* out,
                           void* stream) {
  int rc = permute_check(y, out, dst_pos, R, S, K, H);
  if (rc != MEP_OK) return rc;
  const long long N = (long long)R * S;
  if (N == 0) return MEP_OK;
  if (topk_w == nullptr) return MEP_ERR_INVALID_ARG;
  const long long vpr = H / 8;
  const uint4* y4 = reinterpret_cast<const uint4*>(y);
  uint4* o4 = reinterpret_cast<uint4*>(out);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long nrows = N * K;
  cudaError_t err;
  switch (K) {
    case 1: err = launch_combine<1>(y4, topk_w, dst_pos, status, N, K, vpr, nrows, o4, st); break;
    case 2: err = launch_combine<2>(y4, topk_w, dst_pos, status, N, K, vpr, nrows, o4, st); break;
    case 4: err = launch_combine<4>(y4, topk_w, dst_pos, status, N, K, vpr, nrows, o4, st); break;
    case 6: err = launch_combine<6>(y4, topk_w, dst_pos, status, N, K, vpr, nrows, o4, st); break;
    case 8: err = launch_combine<8>(y4, topk_w, dst_pos, status, N, K, vpr, nrows, o4, st); break;
    default: err = launch_combine<0>(y4, topk_w, dst_pos, status, N, K, vpr, nrows, o4, st); break;
  }
  return err == cudaSuccess ? MEP_OK : MEP_ERR_CUDA;
}
