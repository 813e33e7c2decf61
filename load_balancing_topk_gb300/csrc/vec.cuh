// vec.cuh -- 16- and 32-byte vector loads and stores shared by the permute
// kernels (permute.cu, permute_backward.cu), and their common argument check.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "mep_common.cuh"

namespace mep {
namespace {

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

}  // namespace

// Host checks shared by dispatch, combine and their backward passes.
inline int permute_check(const void* a, const void* b, const void* dst, int R, int S, int K,
                         int H) {
  if (R < 1 || S < 0 || K < 1 || K > MEP_MAX_K || H < 8 || H % 8 != 0) return MEP_ERR_INVALID_ARG;
  if ((long long)R * S * K > 0x7fffffffLL) return MEP_ERR_INVALID_ARG;
  if ((long long)R * S == 0) return MEP_OK;
  if (a == nullptr || b == nullptr || dst == nullptr) return MEP_ERR_INVALID_ARG;
  if (!aligned16(a) || !aligned16(b)) return MEP_ERR_INVALID_ARG;
  return MEP_OK;
}

}  // namespace mep
