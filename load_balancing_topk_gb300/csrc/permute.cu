// permute.cu -- fused permute (mep_dispatch), weighted unpermute (mep_combine)
// and their backward passes (mep_dispatch_backward, mep_combine_backward).
//
// Source: "月之暗面开源MoonEP：面向MoE训练的专家并行通信库", section 核心技术
// (零拷贝与静态形状: tokens are written straight into preset, expert-grouped
// positions of one fixed S*K buffer per rank, and the unpermute reads them
// back; the shapes are static so no host sync is needed).
//
// dispatch: each token row is read from HBM once and written K times. One
//   warp per token: every lane loads 8 coalesced 32-byte vectors of the row
//   (16-byte ones when H % 16 != 0 or a pointer is not 32-byte aligned) and
//   stores each to the K destination rows with streaming stores; 16 CTAs
//   of 8 warps per SM keep enough stores in flight to run at the HBM write
//   rate. (A design that staged rows in shared memory with
//   cp.async.bulk and wrote them back with K bulk stores per row measured
//   4-8% slower on GB300, at 4 KB and at 14 KB rows.)
// combine: one warp per token; each lane owns 16-byte column vectors and
//   issues the K gathers of two vectors before their fp32 fused
//   multiply-add chains (k in order), then writes the bf16 results
//   (nearest-even).

#include <cuda_bf16.h>

#include "mep_common.cuh"

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
#define MEP_DISPATCH_CTAS_PER_SM 16
#endif
#ifndef MEP_COMBINE_WARPS
#define MEP_COMBINE_WARPS 4
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
#ifndef MEP_CBWD_V32
#define MEP_CBWD_V32 1
#endif
#ifndef MEP_CBWD_V32_MIN_H
#define MEP_CBWD_V32_MIN_H 4096
#endif
constexpr int kCombineUnroll = MEP_COMBINE_UNROLL;      // 16-byte column vectors per lane in flight
constexpr int kCombineUnroll32 = MEP_COMBINE_UNROLL32;  // 32-byte column vectors per lane in flight

// 16- and 32-byte vectors. The 32-byte forms (ld/st .v8.b32, sm_100 and
// later) halve the memory instructions per byte; they need 32-byte aligned
// addresses, which the host guarantees before choosing them.
struct alignas(32) Vec32 {
  uint32_t w[8];
};

__device__ __forceinline__ uint4 ld_nc(const uint4* p) { return __ldg(p); }
__device__ __forceinline__ void st_cs(uint4* p, const uint4& v) { __stcs(p, v); }

__device__ __forceinline__ Vec32 ld_nc(const Vec32* p) {
  Vec32 v;
  asm("ld.global.nc.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
      : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
        "=r"(v.w[6]), "=r"(v.w[7])
      : "l"(p));
  return v;
}

__device__ __forceinline__ void st_cs(Vec32* p, const Vec32& v) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),
               "r"(v.w[0]), "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]),
               "r"(v.w[6]), "r"(v.w[7])
               : "memory");
}

__device__ __forceinline__ void st_plain(uint4* p, const uint4& v) { *p = v; }
__device__ __forceinline__ void st_plain(Vec32* p, const Vec32& v) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v.w[0]),
               "r"(v.w[1]), "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]),
               "r"(v.w[7])
               : "memory");
}

// 32-bit words of a vector (2 bf16 each): 4 for uint4, 8 for Vec32.
template <typename V> struct Words;
template <> struct Words<uint4> {
  static constexpr int n = 4;
  static __device__ __forceinline__ uint32_t get(const uint4& q, int j) {
    return j == 0 ? q.x : j == 1 ? q.y : j == 2 ? q.z : q.w;
  }
  static __device__ __forceinline__ uint4 make(const uint32_t (&o)[4]) {
    return make_uint4(o[0], o[1], o[2], o[3]);
  }
};
template <> struct Words<Vec32> {
  static constexpr int n = 8;
  static __device__ __forceinline__ uint32_t get(const Vec32& q, int j) { return q.w[j]; }
  static __device__ __forceinline__ Vec32 make(const uint32_t (&o)[8]) {
    Vec32 v;
#pragma unroll
    for (int j = 0; j < 8; ++j) v.w[j] = o[j];
    return v;
  }
};

inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

// One warp per token (grid-stride). Each lane holds kUnroll vectors
// of the row and writes each to the K destination rows with streaming
// (evict-first) stores: the buffer is written once here and read back by the
// expert computation, not by this kernel. KT > 0: K fixed at compile time,
// destination offsets held in registers; KT == 0: any K, offsets re-read
// per vector (L1 hits).
template <int KT, typename V>
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
      for (long long v0 = lane; v0 < vpr; v0 += 32 * kUnroll) {
        V q[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (v0 + 32 * u < vpr) q[u] = ld_nc(src + v0 + 32 * u);
#pragma unroll
        for (int k = 0; k < KT; ++k) {
          if (off[k] < 0) continue;
          V* o = buf + off[k] + v0;
#pragma unroll
          for (int u = 0; u < kUnroll; ++u)
            if (v0 + 32 * u < vpr) st_cs(o + 32 * u, q[u]);
        }
      }
    } else {
      for (long long v0 = lane; v0 < vpr; v0 += 32 * kUnroll) {
        V q[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
          if (v0 + 32 * u < vpr) q[u] = ld_nc(src + v0 + 32 * u);
        for (int k = 0; k < K; ++k) {
          const int r = __ldg(dst_pos + t * K + k);
          if (r < 0 || r >= nrows) continue;
          V* o = buf + (long long)r * vpr + v0;
#pragma unroll
          for (int u = 0; u < kUnroll; ++u)
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
  if (MEP_DISPATCH_V32 && H % 16 == 0 && aligned32(x) && aligned32(buf))
    return launch_pdl(k_dispatch<KT, Vec32>, dim3(grid), dim3(32 * MEP_DISPATCH_WARPS), 0, st,
                      static_cast<const Vec32*>(x), dst, status, N, K, (long long)(H / 16), nrows,
                      static_cast<Vec32*>(buf));
  return launch_pdl(k_dispatch<KT, uint4>, dim3(grid), dim3(32 * MEP_DISPATCH_WARPS), 0, st,
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
  const long long cap = (long long)sm_count() * 64;
  const int grid = int(want < cap ? want : cap);
  if (MEP_COMBINE_V32 && H % 16 == 0 && aligned32(y) && aligned32(out))
    return launch_pdl(k_combine<KT, UNIT, Vec32>, dim3(grid), dim3(32 * MEP_COMBINE_WARPS), 0,
                      st, static_cast<const Vec32*>(y), w, dst, status, N, K, (long long)(H / 16),
                      nrows, static_cast<Vec32*>(out));
  return launch_pdl(k_combine<KT, UNIT, uint4>, dim3(grid), dim3(32 * MEP_COMBINE_WARPS), 0, st,
                    static_cast<const uint4*>(y), w, dst, status, N, K, (long long)(H / 8), nrows,
                    static_cast<uint4*>(out));
}

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
      for (long long v = lane; v < vpr; v += 32) {
        const V g = ld_nc(d + v);
        V q[KT];
#pragma unroll
        for (int k = 0; k < KT; ++k) q[k] = ld_nc(y + rows[k] + v);
#pragma unroll
        for (int k = 0; k < KT; ++k) {
          st_cs(dy + rows[k] + v, scaleV<V>(ws[k], g));
          acc[k] = dotV<V>(acc[k], g, q[k]);
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
