// permute.cu -- fused permute (mep_dispatch), weighted unpermute (mep_combine)
// and the permute's backward pass (mep_dispatch_backward: combine with unit
// weights).
//
// Source: "月之暗面开源MoonEP：面向MoE训练的专家并行通信库", section 核心技术
// (零拷贝与静态形状: tokens are written straight into preset, expert-grouped
// positions of one fixed S*K buffer per rank, and the unpermute reads them
// back; the shapes are static so no host sync is needed).
//
// (mep_combine_backward lives in permute_backward.cu.)
//
// dispatch: each token row is read from HBM once and written K times. One
//   warp per token: every lane loads 8 coalesced 32-byte vectors of the row
//   (16-byte ones when H % 16 != 0 or a pointer is not 32-byte aligned) and
//   stores each to the K destination rows with streaming stores. CTAs of 8
//   warps, up to 64 per SM before the warps loop (one token per warp up to
//   9728 CTAs on 152 SMs): a wave of fresh CTAs keeps enough stores in
//   flight to run at the HBM write rate. (A design that staged rows in shared memory with
//   cp.async.bulk and wrote them back with K bulk stores per row measured
//   4-8% slower on GB300, at 4 KB and at 14 KB rows.)
// combine: one warp per token; each lane owns 16-byte column vectors and
//   issues the K gathers of two vectors before their fp32 fused
//   multiply-add chains (k in order), then writes the bf16 results
//   (nearest-even).

#include <cuda_bf16.h>

#include "mep_common.cuh"
#include "vec.cuh"

#ifndef MEP_DISPATCH_WARPS
#define MEP_DISPATCH_WARPS 8
#endif
#ifndef MEP_DISPATCH_UNROLL
#define MEP_DISPATCH_UNROLL 8
#endif
#ifndef MEP_DISPATCH_V32
#define MEP_DISPATCH_V32 1
#endif
#ifndef MEP_DISPATCH_CTAS_PER_SM
#define MEP_DISPATCH_CTAS_PER_SM 64
#endif
#ifndef MEP_COMBINE_WARPS
#define MEP_COMBINE_WARPS 4
#endif
#ifndef MEP_COMBINE_CTAS_PER_SM
#define MEP_COMBINE_CTAS_PER_SM 64
#endif

namespace mep {
namespace {

constexpr int kUnroll = MEP_DISPATCH_UNROLL;
#ifndef MEP_COMBINE_UNROLL
#define MEP_COMBINE_UNROLL 2
#endif
#ifndef MEP_COMBINE_UNROLL32
#define MEP_COMBINE_UNROLL32 2
#endif
#ifndef MEP_COMBINE_V32
#define MEP_COMBINE_V32 1
#endif
constexpr int kCombineUnroll = MEP_COMBINE_UNROLL;      // 16-byte column vectors per lane in flight
constexpr int kCombineUnroll32 = MEP_COMBINE_UNROLL32;  // 32-byte column vectors per lane in flight


// One warp per token (grid-stride past the grid cap). Each lane holds U
// vectors of the row (U = 16 for rows longer than 8 vectors per lane, so that
// a 7168-wide row moves in one round) and writes each to the K destination
// rows with streaming (evict-first) stores: the buffer is written once here
// and read back by the expert computation, not by this kernel. KT > 0: K
// fixed at compile time, destination offsets held in registers; KT == 0: any
// K, offsets re-read per vector (L1 hits).
template <int KT, typename V, int U>
__global__ void __launch_bounds__(32 * MEP_DISPATCH_WARPS)
    k_dispatch(const V* __restrict__ hidden, const int32_t* __restrict__ dst_pos,
               int32_t* status, long long N, int Kr, long long vpr, long long nrows,
               V* __restrict__ buf) {
  pdl_wait();
  pdl_launch_dependents();
  if (read_status(status) != 0) return;
  const int K = KT > 0 ? KT : Kr;
  const int lane = threadIdx.x & 31;
  const long long warp0 = (long long)blockIdx.x * MEP_DISPATCH_WARPS + (threadIdx.x >> 5);
  const long long nwarp = (long long)gridDim.x * MEP_DISPATCH_WARPS;
  for (long long t = warp0; t < N; t += nwarp) {
    const int r0 = lane < K ? __ldg(dst_pos + t * K + lane) : 0;
    const int r1 = lane + 32 < K ? __ldg(dst_pos + t * K + lane + 32) : 0;
    const bool bad = (lane < K && (r0 < 0 || r0 >= nrows)) ||
                     (lane + 32 < K && (r1 < 0 || r1 >= nrows));
    if (__any_sync(MEP_FULL_MASK, bad) && lane == 0) set_status(status, MEP_ERR_BAD_POSITION);
    const V* src = hidden + t * vpr;
    if constexpr (KT > 0) {
      long long off[KT];
#pragma unroll
      for (int k = 0; k < KT; ++k) {
        const int r = __shfl_sync(MEP_FULL_MASK, r0, k);
        off[k] = (r >= 0 && r < nrows) ? (long long)r * vpr : -1;
      }
      for (long long v0 = lane; v0 < vpr; v0 += 32 * U) {
        V q[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (v0 + 32 * u < vpr) q[u] = ld_nc(src + v0 + 32 * u);
#pragma unroll
        for (int k = 0; k < KT; ++k) {
          if (off[k] < 0) continue;
          V* o = buf + off[k] + v0;
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (v0 + 32 * u < vpr) st_cs(o + 32 * u, q[u]);
        }
      }
    } else {
      for (long long v0 = lane; v0 < vpr; v0 += 32 * U) {
        V q[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (v0 + 32 * u < vpr) q[u] = ld_nc(src + v0 + 32 * u);
        for (int k = 0; k < K; ++k) {
          const int r = __ldg(dst_pos + t * K + k);
          if (r < 0 || r >= nrows) continue;
          V* o = buf + (long long)r * vpr + v0;
#pragma unroll
          for (int u = 0; u < U; ++u)
            if (v0 + 32 * u < vpr) st_cs(o + 32 * u, q[u]);
        }
      }
    }
  }
}

template <int KT>
cudaError_t launch_dispatch(const void* x, const int32_t* dst, int32_t* status, long long N,
                            int K, int H, long long nrows, void* buf, cudaStream_t st) {
  const long long want = (N + MEP_DISPATCH_WARPS - 1) / MEP_DISPATCH_WARPS;
  const long long cap = (long long)sm_count() * MEP_DISPATCH_CTAS_PER_SM;
  const int grid = int(want < cap ? want : cap);
  if (MEP_DISPATCH_V32 && H % 16 == 0 && aligned32(x) && aligned32(buf)) {
    const long long vpr = H / 16;
    if (vpr > 32 * kUnroll)
      return launch_pdl(k_dispatch<KT, Vec32, 2 * kUnroll>, dim3(grid), dim3(32 * MEP_DISPATCH_WARPS),
                        0, st, static_cast<const Vec32*>(x), dst, status, N, K, vpr, nrows,
                        static_cast<Vec32*>(buf));
    return launch_pdl(k_dispatch<KT, Vec32, kUnroll>, dim3(grid), dim3(32 * MEP_DISPATCH_WARPS), 0,
                      st, static_cast<const Vec32*>(x), dst, status, N, K, vpr, nrows,
                      static_cast<Vec32*>(buf));
  }
  return launch_pdl(k_dispatch<KT, uint4, kUnroll>, dim3(grid), dim3(32 * MEP_DISPATCH_WARPS), 0, st,
                    static_cast<const uint4*>(x), dst, status, N, K, (long long)(H / 8), nrows,
                    static_cast<uint4*>(buf));
}

// ---------------------------------------------------------------------------
// acc[i] = fma(w, bf16 element i of q, acc[i]) for the 2n elements of q
template <typename V>
__device__ __forceinline__ void fmaV(float (&acc)[2 * Words<V>::n], float w, const V& q) {
#pragma unroll
  for (int j = 0; j < Words<V>::n; ++j) {
    const uint32_t v = Words<V>::get(q, j);
    acc[2 * j] = __fmaf_rn(w, __uint_as_float(v << 16), acc[2 * j]);
    acc[2 * j + 1] = __fmaf_rn(w, __uint_as_float(v & 0xffff0000u), acc[2 * j + 1]);
  }
}

template <typename V>
__device__ __forceinline__ V packV(const float (&acc)[2 * Words<V>::n]) {
  uint32_t o[Words<V>::n];
#pragma unroll
  for (int j = 0; j < Words<V>::n; ++j) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
    o[j] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return Words<V>::make(o);
}

// KT > 0: K known at compile time (all K gathers of a vector in flight at
// once). KT == 0: any K, gathered in batches of 8. UNIT: every weight is 1
// and topk_w is not read (the backward of dispatch: sum of the K rows; an fma
// with 1 rounds exactly like an add).
template <int KT, bool UNIT, typename V>
__global__ void __launch_bounds__(32 * MEP_COMBINE_WARPS)
    k_combine(const V* __restrict__ y, const float* __restrict__ topk_w,
              const int32_t* __restrict__ dst_pos, int32_t* status, long long N, int Kr,
              long long vpr, long long nrows, V* __restrict__ out) {
  constexpr int U = sizeof(V) == 32 ? kCombineUnroll32 : kCombineUnroll;
  constexpr int NE = 2 * Words<V>::n;  // bf16 elements per vector
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
    const float w0 = UNIT ? 1.f : (lane < K ? __ldg(topk_w + t * K + lane) : 0.f);
    const bool bad = (lane < K && (r0 < 0 || r0 >= nrows)) ||
                     (lane + 32 < K && (r1 < 0 || r1 >= nrows));
    if (__any_sync(MEP_FULL_MASK, bad)) {
      if (lane == 0) set_status(status, MEP_ERR_BAD_POSITION);
      continue;
    }
    V* o = out + t * vpr;
    if constexpr (KT > 0) {
      long long rows[KT];
      float ws[KT];
#pragma unroll
      for (int k = 0; k < KT; ++k) {
        rows[k] = (long long)__shfl_sync(MEP_FULL_MASK, r0, k) * vpr;
        ws[k] = __shfl_sync(MEP_FULL_MASK, w0, k);
      }
      for (long long v0 = lane; v0 < vpr; v0 += 32 * U) {
        V q[U][KT];
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (v0 + 32 * u < vpr) {
#pragma unroll
            for (int k = 0; k < KT; ++k) q[u][k] = ld_nc(y + rows[k] + v0 + 32 * u);
          }
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (v0 + 32 * u < vpr) {
            float acc[NE];
#pragma unroll
            for (int i = 0; i < NE; ++i) acc[i] = 0.f;
#pragma unroll
            for (int k = 0; k < KT; ++k) fmaV<V>(acc, ws[k], q[u][k]);
            st_plain(o + v0 + 32 * u, packV<V>(acc));
          }
      }
    } else {
      for (long long v = lane; v < vpr; v += 32) {
        float acc[NE];
#pragma unroll
        for (int i = 0; i < NE; ++i) acc[i] = 0.f;
        for (int k0 = 0; k0 < K; k0 += 8) {
          V q[8];
          float ws[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int k = k0 + j;
            if (k < K) {
              const long long row = __ldg(dst_pos + t * K + k);
              ws[j] = UNIT ? 1.f : __ldg(topk_w + t * K + k);
              q[j] = ld_nc(y + row * vpr + v);
            }
          }
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (k0 + j < K) fmaV<V>(acc, ws[j], q[j]);
        }
        st_plain(o + v, packV<V>(acc));
      }
    }
  }
}

template <int KT, bool UNIT = false>
cudaError_t launch_combine(const void* y, const float* w, const int32_t* dst, int32_t* status,
                           long long N, int K, int H, long long nrows, void* out,
                           cudaStream_t st) {
  const long long want = (N + MEP_COMBINE_WARPS - 1) / MEP_COMBINE_WARPS;
  const long long cap = (long long)sm_count() * MEP_COMBINE_CTAS_PER_SM;
  const int grid = int(want < cap ? want : cap);
  if (MEP_COMBINE_V32 && H % 16 == 0 && aligned32(y) && aligned32(out))
    return launch_pdl(k_combine<KT, UNIT, Vec32>, dim3(grid), dim3(32 * MEP_COMBINE_WARPS), 0,
                      st, static_cast<const Vec32*>(y), w, dst, status, N, K, (long long)(H / 16),
                      nrows, static_cast<Vec32*>(out));
  return launch_pdl(k_combine<KT, UNIT, uint4>, dim3(grid), dim3(32 * MEP_COMBINE_WARPS), 0, st,
                    static_cast<const uint4*>(y), w, dst, status, N, K, (long long)(H / 8), nrows,
                    static_cast<uint4*>(out));
}

}  // namespace
}  // namespace mep

using namespace mep;


extern "C" int mep_dispatch(const mep_bf16* hidden, const int32_t* dst_pos, int32_t* status,
                            int R, int S, int K, int H, mep_bf16* buf, void* stream) {
  int rc = permute_check(hidden, buf, dst_pos, R, S, K, H);
  if (rc != MEP_OK) return rc;
  const long long N = (long long)R * S;
  if (N == 0) return MEP_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long nrows = N * K;
  cudaError_t err;
  switch (K) {
    case 1: err = launch_dispatch<1>(hidden, dst_pos, status, N, K, H, nrows, buf, st); break;
    case 2: err = launch_dispatch<2>(hidden, dst_pos, status, N, K, H, nrows, buf, st); break;
    case 4: err = launch_dispatch<4>(hidden, dst_pos, status, N, K, H, nrows, buf, st); break;
    case 6: err = launch_dispatch<6>(hidden, dst_pos, status, N, K, H, nrows, buf, st); break;
    case 8: err = launch_dispatch<8>(hidden, dst_pos, status, N, K, H, nrows, buf, st); break;
    default: err = launch_dispatch<0>(hidden, dst_pos, status, N, K, H, nrows, buf, st); break;
  }
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
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long nrows = N * K;
  cudaError_t err;
  switch (K) {
    case 1: err = launch_combine<1>(y, topk_w, dst_pos, status, N, K, H, nrows, out, st); break;
    case 2: err = launch_combine<2>(y, topk_w, dst_pos, status, N, K, H, nrows, out, st); break;
    case 4: err = launch_combine<4>(y, topk_w, dst_pos, status, N, K, H, nrows, out, st); break;
    case 6: err = launch_combine<6>(y, topk_w, dst_pos, status, N, K, H, nrows, out, st); break;
    case 8: err = launch_combine<8>(y, topk_w, dst_pos, status, N, K, H, nrows, out, st); break;
    default: err = launch_combine<0>(y, topk_w, dst_pos, status, N, K, H, nrows, out, st); break;
  }
  return err == cudaSuccess ? MEP_OK : MEP_ERR_CUDA;
}

extern "C" int mep_dispatch_backward(const mep_bf16* dbuf, const int32_t* dst_pos,
                                     int32_t* status, int R, int S, int K, int H,
                                     mep_bf16* dhidden, void* stream) {
  int rc = permute_check(dbuf, dhidden, dst_pos, R, S, K, H);
  if (rc != MEP_OK) return rc;
  const long long N = (long long)R * S;
  if (N == 0) return MEP_OK;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long nrows = N * K;
  cudaError_t err;
  switch (K) {
    case 1: err = launch_combine<1, true>(dbuf, nullptr, dst_pos, status, N, K, H, nrows, dhidden, st); break;
    case 2: err = launch_combine<2, true>(dbuf, nullptr, dst_pos, status, N, K, H, nrows, dhidden, st); break;
    case 4: err = launch_combine<4, true>(dbuf, nullptr, dst_pos, status, N, K, H, nrows, dhidden, st); break;
    case 6: err = launch_combine<6, true>(dbuf, nullptr, dst_pos, status, N, K, H, nrows, dhidden, st); break;
    case 8: err = launch_combine<8, true>(dbuf, nullptr, dst_pos, status, N, K, H, nrows, dhidden, st); break;
    default: err = launch_combine<0, true>(dbuf, nullptr, dst_pos, status, N, K, H, nrows, dhidden, st); break;
  }
  return err == cudaSuccess ? MEP_OK : MEP_ERR_CUDA;
}
