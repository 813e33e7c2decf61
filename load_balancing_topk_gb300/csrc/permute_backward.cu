// permute_backward.cu -- gradient of the weighted unpermute (mep_combine_backward).
//
// Source: "月之暗面开源MoonEP：面向MoE训练的专家并行通信库", section 核心技术 (the
// fused permute/unpermute; a backward pass exists). The arithmetic is this
// library's reading: dy = bf16(fp32(w * dout)), dw = the dot product in fp32.
//
// One warp per token; each lane keeps MEP_CBWD_UNROLL column vectors in
// flight, each with the K rows of y it meets, before the streaming dy
// stores and the per-lane fp32 dot products; a warp butterfly gives dw.

#include <cuda_bf16.h>

#include "mep_common.cuh"
#include "vec.cuh"

#ifndef MEP_COMBINE_WARPS
#define MEP_COMBINE_WARPS 4
#endif
#ifndef MEP_CBWD_V32
#define MEP_CBWD_V32 1
#endif
#ifndef MEP_CBWD_UNROLL
#define MEP_CBWD_UNROLL 2
#endif
#ifndef MEP_CBWD_V32_MIN_H
#define MEP_CBWD_V32_MIN_H 4096
#endif

namespace mep {
namespace {

// ---------------------------------------------------------------------------
// Backward of combine, one warp per token. Per column vector v: load
// dout[t, v] and the K rows y[dst_pos[t,k], v]; write
//   dy[dst_pos[t,k], v] = bf16_rn(fp32(w[t,k] * dout[t, v]))   (streaming)
// and accumulate the K dot products <dout[t], y[dst_pos[t,k]]> per lane with
// fp32 fma (every bf16 x bf16 product is exact in fp32), then reduce them
// across the warp (butterfly) and write dw[t, k] from lane 0.
template <typename V>
__device__ __forceinline__ V scaleV(float w, const V& q) {
  uint32_t o[Words<V>::n];
#pragma unroll
  for (int j = 0; j < Words<V>::n; ++j) {
    const uint32_t v = Words<V>::get(q, j);
    const float lo = __fmul_rn(w, __uint_as_float(v << 16));
    const float hi = __fmul_rn(w, __uint_as_float(v & 0xffff0000u));
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    o[j] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return Words<V>::make(o);
}

template <typename V>
__device__ __forceinline__ float dotV(float acc, const V& a, const V& b) {
#pragma unroll
  for (int j = 0; j < Words<V>::n; ++j) {
    const uint32_t va = Words<V>::get(a, j), vb = Words<V>::get(b, j);
    acc = __fmaf_rn(__uint_as_float(va << 16), __uint_as_float(vb << 16), acc);
    acc = __fmaf_rn(__uint_as_float(va & 0xffff0000u), __uint_as_float(vb & 0xffff0000u), acc);
  }
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) v += __shfl_xor_sync(MEP_FULL_MASK, v, d);
  return v;
}

template <int KT, typename V>
__global__ void __launch_bounds__(32 * MEP_COMBINE_WARPS)
    k_combine_backward(const V* __restrict__ dout, const V* __restrict__ y,
                       const float* __restrict__ topk_w, const int32_t* __restrict__ dst_pos,
                       int32_t* status, long long N, int Kr, long long vpr, long long nrows,
                       V* __restrict__ dy, float* __restrict__ dw) {
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
    const V* d = dout + t * vpr;
    if constexpr (KT > 0) {
      long long rows[KT];
      float ws[KT], acc[KT];
#pragma unroll
      for (int k = 0; k < KT; ++k) {
        rows[k] = (long long)__shfl_sync(MEP_FULL_MASK, r0, k) * vpr;
        ws[k] = __shfl_sync(MEP_FULL_MASK, w0, k);
        acc[k] = 0.f;
      }
      constexpr int U = MEP_CBWD_UNROLL;  // column vectors per lane in flight
      for (long long v0 = lane; v0 < vpr; v0 += 32 * U) {
        V g[U], q[U][KT];
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (v0 + 32 * u < vpr) {
            g[u] = ld_nc(d + v0 + 32 * u);
#pragma unroll
            for (int k = 0; k < KT; ++k) q[u][k] = ld_nc(y + rows[k] + v0 + 32 * u);
          }
#pragma unroll
        for (int u = 0; u < U; ++u)
          if (v0 + 32 * u < vpr) {
#pragma unroll
            for (int k = 0; k < KT; ++k) {
              st_cs(dy + rows[k] + v0 + 32 * u, scaleV<V>(ws[k], g[u]));
              acc[k] = dotV<V>(acc[k], g[u], q[u][k]);
            }
          }
      }
#pragma unroll
      for (int k = 0; k < KT; ++k) {
        const float s = warp_sum(acc[k]);
        if (lane == 0) dw[t * K + k] = s;
      }
    } else {
      for (int k = 0; k < K; ++k) {
        const long long row = (long long)__ldg(dst_pos + t * K + k) * vpr;
        const float wk = __ldg(topk_w + t * K + k);
        float acc = 0.f;
        for (long long v = lane; v < vpr; v += 32) {
          const V g = ld_nc(d + v);
          st_cs(dy + row + v, scaleV<V>(wk, g));
          acc = dotV<V>(acc, g, ld_nc(y + row + v));
        }
        const float s = warp_sum(acc);
        if (lane == 0) dw[t * K + k] = s;
      }
    }
  }
}

template <int KT>
cudaError_t launch_combine_backward(const void* dout, const void* y, const float* w,
                                    const int32_t* dst, int32_t* status, long long N, int K,
                                    int H, long long nrows, void* dy, float* dw,
                                    cudaStream_t st) {
  const long long want = (N + MEP_COMBINE_WARPS - 1) / MEP_COMBINE_WARPS;
  const long long cap = (long long)sm_count() * 64;
  const int grid = int(want < cap ? want : cap);
  // 32-byte vectors pay off once a lane walks 8 or more of them per row;
  // below that the 16-byte form keeps more rows in flight (measured: 3% faster
  // at H = 2048, 4% slower at H = 7168).
  if (MEP_CBWD_V32 && H % 16 == 0 && H >= MEP_CBWD_V32_MIN_H && aligned32(dout) && aligned32(y) &&
      aligned32(dy))
    return launch_pdl(k_combine_backward<KT, Vec32>, dim3(grid), dim3(32 * MEP_COMBINE_WARPS), 0,
                      st, static_cast<const Vec32*>(dout), static_cast<const Vec32*>(y), w, dst,
                      status, N, K, (long long)(H / 16), nrows, static_cast<Vec32*>(dy), dw);
  return launch_pdl(k_combine_backward<KT, uint4>, dim3(grid), dim3(32 * MEP_COMBINE_WARPS), 0,
                    st, static_cast<const uint4*>(dout), static_cast<const uint4*>(y), w, dst,
                    status, N, K, (long long)(H / 8), nrows, static_cast<uint4*>(dy), dw);
}

}  // namespace
}  // namespace mep

using namespace mep;

extern "C" int mep_combine_backward(const mep_bf16* dout, const mep_bf16* y, const float* topk_w,
                                    const int32_t* dst_pos, int32_t* status, int R, int S, int K,
                                    int H, mep_bf16* dy, float* dw, void* stream) {
  int rc = permute_check(dout, y, dst_pos, R, S, K, H);
  if (rc != MEP_OK) return rc;
  const long long N = (long long)R * S;
  if (N == 0) return MEP_OK;
  if (topk_w == nullptr || dy == nullptr || dw == nullptr || !aligned16(dy))
    return MEP_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long nrows = N * K;
  cudaError_t err;
  switch (K) {
    case 1: err = launch_combine_backward<1>(dout, y, topk_w, dst_pos, status, N, K, H, nrows, dy, dw, st); break;
    case 2: err = launch_combine_backward<2>(dout, y, topk_w, dst_pos, status, N, K, H, nrows, dy, dw, st); break;
    case 4: err = launch_combine_backward<4>(dout, y, topk_w, dst_pos, status, N, K, H, nrows, dy, dw, st); break;
    case 6: err = launch_combine_backward<6>(dout, y, topk_w, dst_pos, status, N, K, H, nrows, dy, dw, st); break;
    case 8: err = launch_combine_backward<8>(dout, y, topk_w, dst_pos, status, N, K, H, nrows, dy, dw, st); break;
    default: err = launch_combine_backward<0>(dout, y, topk_w, dst_pos, status, N, K, H, nrows, dy, dw, st); break;
  }
  return err == cudaSuccess ? MEP_OK : MEP_ERR_CUDA;
}
