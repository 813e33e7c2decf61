// grouped_gemm.cu -- the grouped expert product over the static buffer
// (mep_grouped_gemm), on the sm_100-family tensor cores (tcgen05 + TMA).
//
// Source: "月之暗面开源MoonEP：面向MoE训练的专家并行通信库", section
// 内存契约与权重布局: one grouped GEMM per expert projection consumes a single
// [E+B, H, H'] weight tensor (rows [0, E) the experts' own weights, rows
// [E, E+B) the rank's prefetch slots) and cu_seqlens[E+B] says which rows of
// the static S*K buffer each weight row serves.
//
// Two launches on the caller's stream:
//   k_gemm_tiles  (1 CTA) checks every cu_seqlens row and cuts every group
//                 into 128-row tiles {first buffer row, rows, weight row},
//                 padded with empty tiles to a whole number of pairs,
//                 written to the workspace with their count;
//   k_gemm_pair   (default) persistent clusters of two CTAs, one per SM, 192
//                 threads each, over the work units (pair of adjacent tiles
//                 of one group, 256-column block of H'), grid-stride:
//     warp 0      TMA producer of each CTA: per 64-wide K step, its own
//                 128x64 tile of x (K-major, 128-byte swizzle) and its half
//                 (two 64x64 boxes) of the weight row's 256 columns (H'
//                 contiguous: MN-major, 128-byte swizzle) into a ring of
//                 MEP_GEMM_PAIR_STAGES 32 KB stages; both CTAs' copies count
//                 on CTA 0's stage barrier;
//     warp 1      allocates the pair's TMEM (2 x 256 fp32 columns in each
//                 CTA, cta_group::2) and, in CTA 0, issues from one lane the
//                 pair MMAs (tcgen05.mma.cta_group::2: M = 256 over the two
//                 CTAs, N = 256 -- 128 for a last column block of at most
//                 128 columns --, K = 16, bf16 in, fp32 accumulate); every
//                 commit is multicast to both CTAs (stage free, accumulator
//                 ready);
//     warps 2..5  epilogue of each CTA: tcgen05.ld of its 128 TMEM lanes
//                 (= its tile's rows), bf16 (nearest-even); a warp whose 32
//                 rows are all valid writes them through shared memory (two
//                 4 KB boxes in the y map's swizzled layout, alternating) with
//                 bulk tensor stores, a warp with padding rows stores its
//                 valid rows lane by lane (whole sectors); then a release on
//                 CTA 0's accumulator barrier. The accumulator is
//                 double-buffered, so the next unit's MMAs overlap this store.
// Every wait is bounded (MEP_GEMM_TIMEOUT_NS on %globaltimer): a wait that
// gives up raises a CTA-wide abort flag and MEP_ERR_TIMEOUT; every role then
// leaves its loop, the producer waits for its own copies in flight, the MMA
// lane for its own MMAs, and the TMEM is freed before the CTA exits.

#include <cuda.h>
#include <cuda_bf16.h>

#include <mutex>

#include "mep_common.cuh"

#ifndef MEP_GEMM_B_LBO
#define MEP_GEMM_B_LBO 8192  // byte stride between 64-wide H' blocks of a weight stage
#endif
#ifndef MEP_GEMM_B_SBO
#define MEP_GEMM_B_SBO 1024  // byte stride between 8-row K groups of a weight stage
#endif
#ifndef MEP_GEMM_NARROW_N
#define MEP_GEMM_NARROW_N 1  // a last column block of <= 128 columns runs N = 128 pair MMAs
#endif
#ifndef MEP_GEMM_ST32
#define MEP_GEMM_ST32 1  // epilogue stores whole 32-byte sectors when H' % 16 == 0
#endif
#ifndef MEP_GEMM_TIMEOUT_NS
#define MEP_GEMM_TIMEOUT_NS 4000000000ull
#endif

namespace mep {
namespace {

constexpr int kBM = 128;                   // tile rows (TMEM lanes)
constexpr int kBN = 256;                   // tile columns of H' (TMEM columns per accumulator)
constexpr int kBK = 64;                    // K step: one 128-byte swizzle row of bf16
constexpr int kABytes = kBM * kBK * 2;     // 16 KB
constexpr int kBBox = kBK * 64 * 2;        // one 64x64 weight box, 8 KB
constexpr int kThreads = 192;
constexpr int kTmemCols = 2 * kBN;         // double-buffered accumulator
constexpr int kTileThreads = 1024;
constexpr int kPair = 2;                   // CTAs per cluster (one CTA pair)

// ---------------------------------------------------------------------------
// PTX wrappers (mbarrier, TMA, tcgen05)
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for the phase of `bar` with the given parity to complete.
// Returns false on timeout (raising the abort flag and MEP_ERR_TIMEOUT) and,
// when honor_abort, as soon as another role has raised the flag. The drains
// at the end of the kernel pass honor_abort = false: they must see their own
// copies and MMAs land before the CTA frees its TMEM and exits.
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, volatile int* abort,
                                             int32_t* status, bool honor_abort,
                                             uint64_t limit_ns = MEP_GEMM_TIMEOUT_NS) {
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u) {
      if (honor_abort && *abort) return false;
      const uint64_t now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit_ns) {
        *abort = 1;
        set_status(status, MEP_ERR_TIMEOUT);
        return false;
      }
    }
  }
}
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* abort,
                                           int32_t* status, bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_phase_slow(bar, parity, abort, status, honor_abort);
}

// cta_group::2 form: the data lands in this CTA's shared memory, the bytes
// are counted on an mbarrier that may sit in the peer CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar_cluster) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
      : "memory");
}
// Bulk tensor store of one 64-column x 32-row box of y from shared memory
// (128-byte swizzle, the layout of the tensor map); columns at or beyond the
// map's width are not written. Each store is its own bulk group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];\n\t"
      "cp.async.bulk.commit_group;" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(src)
      : "memory");
}
// Wait until at most one of this thread's bulk stores still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Wait until all of this thread's bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Address of the same shared variable in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster)
               : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (all >> 4), descriptor version 1 (bits 46-47) and the
// 128-byte swizzle layout (value 2 in bits 61-63). Stage buffers are
// 1024-byte aligned, so the base-offset field stays 0.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(sbo >> 4) << 32) | (1ull << 46) | (2ull << 61);
}

// The pair form: M = 256 rows over the two CTAs of a pair (each CTA's 128
// rows of A and 128 of the 256 columns of B in its own shared memory, each
// CTA's 128 rows of D in its own TMEM), issued by one thread of CTA 0.
// kIdesc2n: the same with N = 128, for a last column block of at most 128
// columns (each CTA then holds 64 of them).
constexpr uint32_t kIdesc2 = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                             ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
constexpr uint32_t kIdesc2n = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) |
                              ((uint32_t)(128 >> 3) << 17) | ((uint32_t)(256 >> 4) << 24);
__device__ __forceinline__ void tc_mma2(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                        uint32_t accumulate, uint32_t idesc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit2_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}
__device__ __forceinline__ void tc_commit2(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes, one lane (row)
// per thread: tc_ld32_issue starts the load; tc_ld_wait waits for all of
// this thread's loads so far and then ties v to that wait (an empty asm
// that "rewrites" v), so that no use of v can be scheduled above it.
// (Keeping the next chunk's load in flight while one is stored measured the
// same: the epilogue's time goes to its stores, and it overlaps the next
// unit's MMAs through the second accumulator.)
__device__ __forceinline__ void tc_ld32_issue(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tc_ld_wait(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
  asm volatile("" : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31]));
}

__device__ __forceinline__ uint32_t pack_bf16(uint32_t lo, uint32_t hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo), __uint_as_float(hi));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// 32 fp32 accumulator columns of one row -> bf16 (nearest-even) at out[0..32),
// columns at or beyond `left` skipped. st32: whole 32-byte sectors per store
// (needs H' % 16 == 0 and a 32-byte aligned y, checked on the host), else
// 16-byte stores (H' % 8 == 0).
__device__ __forceinline__ void store_chunk(__nv_bfloat16* out, const uint32_t (&v)[32], int left,
                                            bool st32) {
  uint32_t o[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) o[j] = pack_bf16(v[2 * j], v[2 * j + 1]);
  if (st32) {
#pragma unroll
    for (int g = 0; g < 2; ++g)
      if (16 * g < left)
        asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(out + 16 * g),
                     "r"(o[8 * g + 0]), "r"(o[8 * g + 1]), "r"(o[8 * g + 2]), "r"(o[8 * g + 3]),
                     "r"(o[8 * g + 4]), "r"(o[8 * g + 5]), "r"(o[8 * g + 6]), "r"(o[8 * g + 7])
                     : "memory");
  } else {
#pragma unroll
    for (int g = 0; g < 4; ++g)
      if (8 * g < left)
        *reinterpret_cast<uint4*>(out + 8 * g) =
            make_uint4(o[4 * g + 0], o[4 * g + 1], o[4 * g + 2], o[4 * g + 3]);
  }
}

// ---------------------------------------------------------------------------
// Tile table. tiles[i] = {first buffer row, rows (1..128), weight row, 0}
// where weight row < E is a home expert and E + r*B + b is slot b of rank r.
__global__ void __launch_bounds__(kTileThreads)
    k_gemm_tiles(const int32_t* __restrict__ cu, int R, int E, int B, int SK, int pair,
                 int32_t* status, int4* __restrict__ tiles, int* __restrict__ count) {
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int s_warp[33];
  __shared__ int s_bad, s_carry, s_stat;
  const int G = E + B;
  const long long RG = (long long)R * G;
  if (threadIdx.x == 0) {
    s_bad = 0;
    s_carry = 0;
    s_stat = read_status(status);
  }
  __syncthreads();
  if (s_stat != 0) {
    if (threadIdx.x == 0) *count = 0;
    return;
  }
  // every row nondecreasing from >= 0 and ending at S*K
  for (long long p = threadIdx.x; p < RG; p += blockDim.x) {
    const int j = int(p % G);
    const int v = cu[p];
    const int prev = j == 0 ? 0 : cu[p - 1];
    if (v < prev || (j == G - 1 && v != SK)) s_bad = 1;
  }
  __syncthreads();
  if (s_bad) {
    if (threadIdx.x == 0) {
      *count = 0;
      set_status(status, MEP_ERR_BAD_SEQLENS);
    }
    return;
  }
  __shared__ int s_nt[kTileThreads + 1];
  for (long long base = 0; base < RG; base += blockDim.x) {
    const long long p = base + threadIdx.x;
    int lo = 0, len = 0;
    if (p < RG) {
      const int j = int(p % G);
      lo = j == 0 ? 0 : cu[p - 1];
      len = cu[p] - lo;
    }
    const int nt = (len + kBM - 1) / kBM;
    s_nt[threadIdx.x] = (nt + pair - 1) / pair * pair;  // empty tiles complete the last pair
    __syncthreads();
    block_excl_scan(s_nt, s_nt, blockDim.x, s_warp, true);
    if (p < RG && len > 0) {
      const int r = int(p / G), j = int(p % G);
      const int widx = j < E ? j : E + r * B + (j - E);
      const long long row0 = (long long)r * SK + lo;
      const int off = s_carry + s_nt[threadIdx.x];
      const int nt = (len + kBM - 1) / kBM;
      const int padded = (nt + pair - 1) / pair * pair;
      for (int m = 0; m < padded; ++m)
        tiles[off + m] = make_int4(int(row0 + (long long)m * kBM), max(0, min(kBM, len - m * kBM)),
                                   widx, 0);
    }
    __syncthreads();
    if (threadIdx.x == 0) s_carry += s_nt[blockDim.x];
    __syncthreads();
  }
  if (threadIdx.x == 0) *count = s_carry;
}

// ---------------------------------------------------------------------------
#ifndef MEP_GEMM_PAIR_STAGES
#define MEP_GEMM_PAIR_STAGES 5
#endif
constexpr int kStages2 = MEP_GEMM_PAIR_STAGES;  // ring depth of the CTA-pair kernel (32 KB stages)
constexpr int kStoreBox = 32 * 64 * 2;  // one epilogue warp's 32 rows x 64 columns of y, bf16: 4 KB
constexpr int kStaging = 4 * 2 * kStoreBox;  // two staging boxes per epilogue warp, 4 warps: 32 KB
constexpr int kSmemPair = 1024 /* alignment slack */ + kStages2 * (kABytes + 2 * kBBox) + kStaging + 256;
static_assert(kSmemPair <= 232448, "the CTA-pair ring must fit in 227 KB of shared memory");
struct GemmSmem {
  uint64_t full[kStages2], empty[kStages2], tfull[2], tempty[2], drain;
  uint32_t tmem;
  int abort;
  int count;
};

// ---------------------------------------------------------------------------
// CTA-pair kernel (cta_group::2). Clusters of two CTAs: CTA r of the pair
// takes tile 2p + r of a pair of adjacent tiles of one group.
// Each CTA stages its own 128x64 x tile and its half (128 columns) of the
// 256-column weight tile, so a stage is 32 KB per CTA and the ring is 6
// deep. Both CTAs' copies count on CTA 0's `full` barrier; one thread of CTA
// 0 issues the M=256 MMAs and multicasts every commit to both CTAs (stage
// free, accumulator ready). CTA 1's epilogue warps release an accumulator by
// arriving on CTA 0's `tempty` barrier (8 arrivals: 4 warps per CTA).
__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_pair(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_wh,
                const __grid_constant__ CUtensorMap map_ws, const int4* __restrict__ tiles,
                const int* __restrict__ count_ptr, int32_t* status, int E, int H, int Hp,
                __nv_bfloat16* __restrict__ y, int st32_flag,
                const __grid_constant__ CUtensorMap map_y) {
  constexpr int kSt = kStages2;
  const bool st32 = st32_flag != 0;
  constexpr int kBHalf = 2 * kBBox;  // 128 weight columns per CTA per stage
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gen_base = smem_raw + (base - raw);
  const uint32_t sa = base;
  const uint32_t sb = base + kSt * kABytes;
  const uint32_t sy = base + kSt * (kABytes + kBHalf);  // epilogue staging, 1024-byte aligned
  GemmSmem* S = reinterpret_cast<GemmSmem*>(gen_base + kSt * (kABytes + kBHalf) + kStaging);
  volatile int* abort_flag = &S->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = int(cluster_rank());
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSt; ++s) {
      mbar_init(smem_u32(&S->full[s]), 1);   // CTA 0: its producer's arrive + both CTAs' bytes
      mbar_init(smem_u32(&S->empty[s]), 1);  // CTA 0's multicast commit
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&S->tfull[a]), 1);
      mbar_init(smem_u32(&S->tempty[a]), 8);
    }
    mbar_init(smem_u32(&S->drain), 1);
    S->abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 1) {  // one warp of each CTA allocates the pair's TMEM together
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&S->tmem)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  pdl_wait();
  if (threadIdx.x == 0) S->count = read_status(status) != 0 ? 0 : *count_ptr;
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = S->tmem;
  const int nN = (Hp + kBN - 1) / kBN;
  const long long units = (long long)(S->count / 2) * nN;
  const long long u0 = blockIdx.x / 2, ustep = gridDim.x / 2;
  const int nk = H / kBK;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer (both CTAs) ----------------
      uint32_t it = 0;
      int last_round[kSt];
      for (int s = 0; s < kSt; ++s) last_round[s] = -1;
      bool ok = true;
      for (long long u = u0; ok && u < units; u += ustep) {
        const int4 t = tiles[(u / nN) * 2 + rank];
        const int n0 = int(u % nN) * kBN;
        const bool home = t.z < E;
        const CUtensorMap* wmap = home ? &map_wh : &map_ws;
        const int wrow = (home ? t.z : t.z - E) * H;
        const int left = (Hp - n0 + 63) / 64;
        const int nbox = left < 4 ? left : 4;  // 64-column boxes of the unit, both CTAs
        // each CTA's share of the boxes: two (N = 256), or one when at most
        // 128 columns remain and the MMAs run with N = 128
        const bool narrow = MEP_GEMM_NARROW_N && Hp - n0 <= 128;
        const int i0 = narrow ? rank : 2 * rank, i1 = narrow ? rank + 1 : 2 * rank + 2;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = int(it % kSt);
          const uint32_t round = it / kSt;
          if (!wait_phase(smem_u32(&S->empty[s]), (round & 1u) ^ 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          const uint32_t fb0 = map_to_rank(smem_u32(&S->full[s]), 0);
          if (leader) mbar_expect_tx(smem_u32(&S->full[s]), 2 * kABytes + nbox * kBBox);
          tma_load_2d_pair(sa + s * kABytes, &map_x, kb * kBK, t.x, fb0);
          for (int i = i0; i < nbox && i < i1; ++i)
            tma_load_2d_pair(sb + s * kBHalf + (i - i0) * kBBox, wmap, n0 + 64 * i,
                             wrow + kb * kBK, fb0);
          last_round[s] = int(round);
        }
      }
      // CTA 0: every copy of both CTAs has landed; both: every commit aimed
      // at this CTA's stage barriers has arrived
      for (int s = 0; s < kSt; ++s)
        if (last_round[s] >= 0) {
          if (leader)
            wait_phase(smem_u32(&S->full[s]), uint32_t(last_round[s]) & 1u, abort_flag, status,
                       false);
          wait_phase(smem_u32(&S->empty[s]), uint32_t(last_round[s]) & 1u, abort_flag, status,
                     false);
        }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (CTA 0 only) ----------------
      uint32_t it = 0, lt = 0;
      bool ok = true;
      for (long long u = u0; ok && u < units; u += ustep, ++lt) {
        const uint32_t a = lt & 1u, use = lt >> 1;
        if (!wait_phase(smem_u32(&S->tempty[a]), (use & 1u) ^ 1u, abort_flag, status)) break;
        tc_fence_after();
        const uint32_t d = tmem + a * kBN;
        const int n0 = int(u % nN) * kBN;
        const uint32_t idesc = MEP_GEMM_NARROW_N && Hp - n0 <= 128 ? kIdesc2n : kIdesc2;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = int(it % kSt);
          if (!wait_phase(smem_u32(&S->full[s]), (it / kSt) & 1u, abort_flag, status)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = sdesc(sa + s * kABytes + kk * 32, 16, 1024);
            const uint64_t bd =
                sdesc(sb + s * kBHalf + kk * 16 * 128, MEP_GEMM_B_LBO, MEP_GEMM_B_SBO);
            tc_mma2(d, ad, bd, (kb | kk) != 0 ? 1u : 0u, idesc);
          }
          tc_commit2_mc(smem_u32(&S->empty[s]), 3);
        }
        if (!ok) break;
        tc_commit2_mc(smem_u32(&S->tfull[a]), 3);
      }
      tc_commit2(smem_u32(&S->drain));
      wait_phase(smem_u32(&S->drain), 0u, abort_flag, status, false);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5 of both CTAs) ----------------
    // Warp q owns TMEM lanes (= tile rows) [32q, 32q + 32). When all 32 of
    // its rows are valid, each 64-column box goes TMEM -> registers -> bf16
    // -> shared memory (the 128-byte swizzled layout of the y map) -> one
    // bulk tensor store, alternating two staging boxes; otherwise each lane
    // stores its own row.
    const int q = warp & 3;
    const uint32_t stage0 = sy + (uint32_t)q * 2 * kStoreBox;
    uint32_t lt = 0, nbox = 0;
    for (long long u = u0; u < units; u += ustep, ++lt) {
      const uint32_t a = lt & 1u, use = lt >> 1;
      if (!wait_phase(smem_u32(&S->tfull[a]), use & 1u, abort_flag, status)) break;
      tc_fence_after();
      const int4 t = tiles[(u / nN) * 2 + rank];
      const int n0 = int(u % nN) * kBN;
      const int r = 32 * q + lane;
      const uint32_t ta = tmem + a * kBN + ((uint32_t)(32 * q) << 16);
      if (t.y >= 32 * q + 32) {
        for (int i = 0; i < kBN / 64 && n0 + 64 * i < Hp; ++i, ++nbox) {
          const uint32_t box = stage0 + (nbox & 1u) * kStoreBox;
          if (lane == 0) bulk_wait_read_1();  // the store that last used this box has read it
          __syncwarp();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int c = 2 * i + h;  // 32-column chunk
            if (n0 + 32 * c >= Hp) break;
            uint32_t v[32];
            tc_ld32_issue(ta + 32 * c, v);
            tc_ld_wait(v);
#pragma unroll
            for (int j = 0; j < 4; ++j) {  // 16-byte piece 4h + j of this row's 128 bytes
              const uint32_t off = (uint32_t)lane * 128u +
                                   ((uint32_t)((4 * h + j) ^ (lane & 7)) << 4);
              asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(box + off),
                           "r"(pack_bf16(v[8 * j + 0], v[8 * j + 1])),
                           "r"(pack_bf16(v[8 * j + 2], v[8 * j + 3])),
                           "r"(pack_bf16(v[8 * j + 4], v[8 * j + 5])),
                           "r"(pack_bf16(v[8 * j + 6], v[8 * j + 7]))
                           : "memory");
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) tma_store_2d(&map_y, n0 + 64 * i, t.x + 32 * q, box);
        }
      } else {
        const bool row_ok = r < t.y;  // padding tiles have no rows
        __nv_bfloat16* out = y + ((long long)t.x + r) * Hp + n0;
        for (int c = 0; c < kBN / 32 && n0 + 32 * c < Hp; ++c) {
          uint32_t v[32];
          tc_ld32_issue(ta + 32 * c, v);
          tc_ld_wait(v);
          if (row_ok) store_chunk(out + 32 * c, v, Hp - (n0 + 32 * c), st32);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(map_to_rank(smem_u32(&S->tempty[a]), 0));
    }
    if (lane == 0) bulk_wait_all();  // every bulk store of this warp has completed
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (threadIdx.x == 0 && read_status(status) != 0) {
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 100000ull) {
    }
  }
  cluster_sync();
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
}

// ---------------------------------------------------------------------------
// Self-test of the bounded wait: one thread waits on an mbarrier that nothing
// arrives at, with no copy or MMA in flight. The wait must give up after
// limit_ns and report MEP_ERR_TIMEOUT; *elapsed_ns gets the time it waited.
__global__ void k_wait_selftest(int32_t* status, unsigned long long limit_ns,
                                unsigned long long* elapsed_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0;
  mbar_init(smem_u32(&bar), 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const uint64_t t0 = globaltimer();
  const bool ok = wait_phase_slow(smem_u32(&bar), 0u, &abort_flag, status, false, limit_ns);
  *elapsed_ns = globaltimer() - t0;
  if (ok) set_status(status, MEP_ERR_INVALID_ARG);  // cannot happen: nothing arrives
}

// ---------------------------------------------------------------------------
// host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, looked up once (thread-safe static init).
EncodeTiledFn encode_fn() {
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
  }();
  return fn;
}

// 2D bf16 map over a row-major [rows, cols] matrix, box {64 columns, box_rows}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* ptr, unsigned long long rows, unsigned long long cols,
              unsigned box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {64, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// True when p is device (or managed) memory of the current device: the
// tensor maps are encoded over these pointers and the kernel's copies read
// and write through them, so memory of another GPU is refused on the host.
bool on_current_device(const void* p) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // the lookup failed: clear its (non-sticky) error
    return false;
  }
  return (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) && at.device == dev;
}

// Each group adds at most one partial tile and one padding tile.
long long max_tiles(int R, int S, int K, int E, int B) {
  return ((long long)R * S * K + kBM - 1) / kBM + 2LL * R * (E + B);
}

// Per-device grid size of one GEMM kernel, found once (thread-safe).
struct GridCache {
  std::mutex mu;
  int grid[64] = {};
};

// Launch a GEMM kernel as a persistent grid of clusters of CL CTAs: as many
// clusters as can be resident at once (a cluster of 2 needs two free SMs of
// one GPC), found once per device and kernel.
template <typename Kernel>
cudaError_t launch_gemm(Kernel kernel, int CL, int smem, GridCache& cache, cudaStream_t st,
                        const CUtensorMap& mx, const CUtensorMap& mh, const CUtensorMap& msl,
                        const int4* tiles, const int* count, int32_t* status, int E, int H,
                        int Hp, __nv_bfloat16* y, int st32, const CUtensorMap& my) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CL;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int grid = 0;
  {
    std::lock_guard<std::mutex> lock(cache.mu);
    if (cache.grid[dev] == 0) {
      int nclusters = 0;
      cfg.gridDim = dim3(sm_count() / CL * CL);
      const cudaError_t e = cudaOccupancyMaxActiveClusters(&nclusters, kernel, &cfg);
      if (e != cudaSuccess) return e;
      if (nclusters < 1) return cudaErrorInvalidConfiguration;
      cache.grid[dev] = (nclusters * CL < sm_count() ? nclusters : sm_count() / CL) * CL;
    }
    grid = cache.grid[dev];
  }
  cfg.gridDim = dim3(grid);
  return cudaLaunchKernelEx(&cfg, kernel, mx, mh, msl, tiles, count, status, E, H, Hp, y, st32, my);
}

}  // namespace
}  // namespace mep

using namespace mep;

extern "C" int mep_grouped_gemm_workspace_bytes(int R, int S, int K, int E, int B,
                                                size_t* bytes) {
  if (bytes == nullptr || R < 1 || S < 0 || K < 1 || E < 1 || B < 0) return MEP_ERR_INVALID_ARG;
  if (R > MEP_MAX_R || E > MEP_MAX_E || K > MEP_MAX_K || (long long)R * B > MEP_MAX_SLOTS)
    return MEP_ERR_INVALID_ARG;
  *bytes = 16 + 16 * (size_t)max_tiles(R, S, K, E, B);
  return MEP_OK;
}

extern "C" int mep_grouped_gemm(const mep_bf16* x, const int32_t* cu_seqlens,
                                const mep_bf16* w_home, const mep_bf16* w_slot, int32_t* status,
                                int R, int S, int K, int E, int B, int H, int Hp, void* ws,
                                size_t ws_bytes, mep_bf16* y, void* stream) {
  size_t need = 0;
  if (mep_grouped_gemm_workspace_bytes(R, S, K, E, B, &need) != MEP_OK) return MEP_ERR_INVALID_ARG;
  if (H < kBK || H % kBK != 0 || Hp < 8 || Hp % 8 != 0) return MEP_ERR_INVALID_ARG;
  const long long SK = (long long)S * K, rows = (long long)R * SK;
  if (rows > 0x7fffff00LL || (long long)E * H > 0x7fffffffLL ||
      (long long)R * B * H > 0x7fffffffLL)
    return MEP_ERR_INVALID_ARG;
  if (rows == 0) return MEP_OK;
  if (x == nullptr || cu_seqlens == nullptr || w_home == nullptr || y == nullptr ||
      ws == nullptr || ws_bytes < need || (B > 0 && w_slot == nullptr))
    return MEP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_home) || !aligned16(y) || !aligned16(ws) ||
      (B > 0 && !aligned16(w_slot)))
    return MEP_ERR_INVALID_ARG;
  if (!on_current_device(x) || !on_current_device(w_home) || !on_current_device(y) ||
      (B > 0 && !on_current_device(w_slot)))
    return MEP_ERR_INVALID_ARG;
  CUtensorMap mx, mh, msl, my;
  if (!make_map(&my, y, (unsigned long long)rows, (unsigned long long)Hp, 32) ||
      !make_map(&mx, x, (unsigned long long)rows, (unsigned long long)H, kBM) ||
      !make_map(&mh, w_home, (unsigned long long)E * H, (unsigned long long)Hp, kBK))
    return MEP_ERR_CUDA;
  if (B > 0) {
    if (!make_map(&msl, w_slot, (unsigned long long)R * B * H, (unsigned long long)Hp, kBK))
      return MEP_ERR_CUDA;
  } else {
    msl = mh;  // never read: every weight row is below E
  }
  int* count = static_cast<int*>(ws);
  int4* tiles = reinterpret_cast<int4*>(static_cast<char*>(ws) + 16);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t err = launch_pdl(k_gemm_tiles, dim3(1), dim3(kTileThreads), 0, st, cu_seqlens, R,
                               E, B, int(SK), kPair, status, tiles, count);
  if (err != cudaSuccess) return MEP_ERR_CUDA;
  __nv_bfloat16* yb = reinterpret_cast<__nv_bfloat16*>(y);
  const int st32 =
      MEP_GEMM_ST32 && Hp % 16 == 0 && (reinterpret_cast<uintptr_t>(y) & 31u) == 0 ? 1 : 0;
  static GridCache cache;
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(k_gemm_pair), kSmemPair))
    return MEP_ERR_CUDA;
  err = launch_gemm(k_gemm_pair, kPair, kSmemPair, cache, st, mx, mh, msl, tiles, count, status, E,
                    H, Hp, yb, st32, my);
  return err == cudaSuccess ? MEP_OK : MEP_ERR_CUDA;
}

extern "C" int mep_wait_selftest(int32_t* status, int64_t limit_ns, uint64_t* elapsed_ns,
                                 void* stream) {
  if (status == nullptr || elapsed_ns == nullptr || limit_ns < 0 || limit_ns > 10000000000LL)
    return MEP_ERR_INVALID_ARG;
  k_wait_selftest<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      status, (unsigned long long)limit_ns, reinterpret_cast<unsigned long long*>(elapsed_ns));
  return cudaGetLastError() == cudaSuccess ? MEP_OK : MEP_ERR_CUDA;
}
