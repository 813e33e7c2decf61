// plan.cu -- routing histogram, online planner and destination rows (mep_plan).
//
// Source: "月之暗面开源MoonEP：面向MoE训练的专家并行通信库", sections 核心技术
// (every rank receives exactly S*K tokens; redundant experts are planned
// online from the current router output, on the GPU, with no host sync) and
// 内存契约与权重布局 (E/R home rows per rank, B slot rows, cu_seqlens[E+B]).
// maxvio and T_e: same page, section 解决的核心问题.
//
// Three launches (four for large tile tables), all asynchronous on the
// caller's stream; all but the first use programmatic dependent launch, so
// each starts while its predecessor drains and waits (griddepcontrol.wait)
// only before reading it:
//   k_hist     grid over tiles of <= 2048 assignments: per-tile expert counts
//              (shared-memory atomics) and routing checks, one token per
//              thread.
//   k_gsum     (large tile tables only) one CTA per group of consecutive
//              tiles: the group's per-expert sums, so that the planner reads
//              Gs x E group sums instead of every tile's counts; it rewrites
//              each tile's counts as the tile's prefix within its group.
//   k_plan     one CTA: tile (or group) counts -> T_e and per-group prefixes
//              (16-byte column loads; without k_gsum it rewrites the tiles'
//              in-group prefixes itself), home-first keep, overflow pour into
//              deficits, slot table, then cu_seqlens and the row bases in
//              closed form (one parallel pass).
//   k_offsets  grid over the same tiles: before its wait, from the routing
//              alone, each assignment's rank among the tile's assignments of
//              its expert (warp prefix + rank inside the warp: up to K = 8
//              from per-warp expert masks, one token per thread
//              (k_offsets_tok); beyond, from __match_any_sync); after it, the
//              tile's base per expert (group prefix + in-group prefix) and
//              the planner's tables map it to its destination row.
// The planner's rule is home-first: a rank keeps, in expert order, at most
// S*K of its home experts' tokens; the overflow segments, in expert order,
// fill the under-loaded ranks' deficits in rank order, one slot per piece.

#include <climits>

#include "mep_common.cuh"

namespace mep {
namespace {

constexpr int kTileThreads = 256;            // k_hist / k_offsets block size (8 warps)
constexpr int kTileWarps = kTileThreads / 32;
constexpr int kTileAssign = 2048;            // assignments per tile (upper bound)
constexpr int kWarpIters = kTileAssign / (32 * kTileWarps);  // 8 iterations per warp
#ifndef MEP_PLAN_THREADS
#define MEP_PLAN_THREADS 1024
#endif
constexpr int kPlanThreads = MEP_PLAN_THREADS;  // k_plan block size
#ifndef MEP_PLAN_SCAN_GROUPS
#define MEP_PLAN_SCAN_GROUPS 64
#endif
constexpr int kMaxScanGroups = MEP_PLAN_SCAN_GROUPS;  // tile groups in k_plan's prefix pass
#ifndef MEP_PLAN_PRESUM_GROUPS
#define MEP_PLAN_PRESUM_GROUPS 16
#endif
// groups when k_gsum forms them: fewer, longer groups shorten the planner's
// scan
constexpr int kPresumGroups = MEP_PLAN_PRESUM_GROUPS;
constexpr int kPartInts = 8192;              // k_plan shared ints for group sums
#ifndef MEP_PLAN_GSUM_MIN_INTS
#define MEP_PLAN_GSUM_MIN_INTS 32768  // tile-count table size (ints) from which k_gsum runs
#endif
#ifndef MEP_PLAN_RANK_WARPS
#define MEP_PLAN_RANK_WARPS 1  // keep / overflow by one warp per rank where E/R <= 32 and R <= 32
#endif
#ifndef MEP_PLAN_WARP_SCAN_MAX_E
#define MEP_PLAN_WARP_SCAN_MAX_E 128
#endif

constexpr int kTokMaxK = 8;                  // k_offsets ranks one token per thread up to this K
// tokens per tile: one per thread up to K = 8 (256 tokens); beyond, as many
// as fit 2048 assignments. A multiple of 4, so that every tile starts on a
// 16-byte boundary of topk_idx.
inline int tile_tokens(int K) { return K <= kTokMaxK ? kTileThreads : (kTileAssign / K) & ~3; }

struct PlanWs {
  int* blockhist;    // [nblk, E] tile counts, rewritten as each tile's exclusive
                     // prefix within its group (count of e in the group's earlier tiles)
  int* groupbase;    // [Gs, E] count of e in all tiles before group g (Gs <= kMaxScanGroups)
  int* groupsum;     // [Gs, E] count of e in group g (k_gsum; large tile tables only)
  int* blockerr;     // [nblk]
  int* etab;         // [E][4] per expert: tokens kept on the home row, global row of
                     // the home row's first token, first piece (pieces are grouped
                     // by expert), number of pieces; one 16-byte load in k_offsets
  int* piece_lo;     // [E+R] first list index covered by the piece
  int* piece_base;   // [E+R] global row of the piece's first token
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t carve(PlanWs* ws, char* base, int nblk, int R, int E) {
  size_t off = 0;
  auto take = [&](int** p, size_t n) {
    if (ws) *p = reinterpret_cast<int*>(base + off);
    off += align256(n * sizeof(int));
  };
  PlanWs dummy;
  PlanWs* w = ws ? ws : &dummy;
  take(&w->blockhist, size_t(nblk) * E);
  take(&w->groupbase, size_t(kMaxScanGroups) * E);
  take(&w->groupsum, size_t(kMaxScanGroups) * E);
  take(&w->blockerr, size_t(nblk > 0 ? nblk : 1));
  take(&w->etab, size_t(4) * E);
  take(&w->piece_lo, size_t(E) + R);
  take(&w->piece_base, size_t(E) + R);
  return off;
}

// A token's K <= 8 expert ids (topk_idx row) into v[0, K): 16-byte loads
// when rows start on 16-byte boundaries (K % 4 == 0), 8-byte loads when on
// 8-byte ones, else one id at a time.
__device__ __forceinline__ void load_token_ids(const int32_t* row, int K, int (&v)[8]) {
  if ((K & 3) == 0) {
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (4 * q < K) {
        const int4 x = __ldg(reinterpret_cast<const int4*>(row) + q);
        v[4 * q] = x.x;
        v[4 * q + 1] = x.y;
        v[4 * q + 2] = x.z;
        v[4 * q + 3] = x.w;
      }
  } else if ((K & 1) == 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (2 * q < K) {
        const int2 x = __ldg(reinterpret_cast<const int2*>(row) + q);
        v[2 * q] = x.x;
        v[2 * q + 1] = x.y;
      }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (k < K) v[k] = __ldg(row + k);
  }
}

// ---------------------------------------------------------------------------
// k_hist: tile counts and routing checks. Thread tt owns token t0 + tt (and
// t0 + tt + 256, ...): it loads the token's K expert ids, checks each is in
// [0, E) and differs from the earlier ones, and counts them with one
// shared-memory atomic each. (Aggregating a warp's equal ids first -- one
// __match_any_sync per k, one atomic per group of lanes -- measured about
// 2 us slower per plan on every workload, the hot-expert stress routing
// included; so did forming the group sums in clusters of 8 or 16 tiles over
// distributed shared memory instead of in k_gsum.)
__global__ void __launch_bounds__(kTileThreads)
    k_hist(const int32_t* __restrict__ topk_idx, int N, int K, int E, int tok_per_tile,
           PlanWs ws) {
  pdl_launch_dependents();
  extern __shared__ int s_cnt[];  // [E]
  __shared__ int s_err;
  const int blk = blockIdx.x;
  const int t0 = blk * tok_per_tile;
  const int ntok = min(tok_per_tile, N - t0);
  if (threadIdx.x == 0) s_err = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  __syncthreads();

  bool bad = false;
  for (int tt = threadIdx.x; tt < ntok; tt += blockDim.x) {
    const int32_t* row = topk_idx + (size_t(t0) + tt) * K;
    if (K <= 8) {
      int v[8];
      load_token_ids(row, K, v);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k >= K) break;
        bool ok = v[k] >= 0 && v[k] < E;
#pragma unroll
        for (int k2 = 0; k2 < k; ++k2) ok = ok && (v[k2] != v[k]);
        if (ok) atomicAdd(&s_cnt[v[k]], 1);
        else bad = true;
      }
    } else {
      for (int k = 0; k < K; ++k) {
        const int e = __ldg(row + k);
        bool ok = e >= 0 && e < E;
        for (int k2 = 0; k2 < k && ok; ++k2) ok = __ldg(row + k2) != e;
        if (ok) atomicAdd(&s_cnt[e], 1);
        else bad = true;
      }
    }
  }
  if (bad) s_err = MEP_ERR_BAD_ROUTING;
  __syncthreads();
  int* out = ws.blockhist + size_t(blk) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) out[e] = s_cnt[e];
  if (threadIdx.x == 0) ws.blockerr[blk] = s_err;
}

// ---------------------------------------------------------------------------
// k_plan: the single-CTA planner.
struct PlanArgs {
  int nblk, R, S, K, E, B;
  int fallback;          // pieces beyond B take the expert's own row instead of failing
  int presummed;         // k_gsum ran: read the group sums, not every tile's counts
  int Gs, tpg;           // tile groups (tile_groups()) and tiles per group
  int32_t* counts;       // [E]
  int32_t* cu;           // [R, E+B]
  int32_t* slot_expert;  // [R, B]
  int32_t* status;
  PlanWs ws;
};

__device__ __noinline__ void plan_fail(const PlanArgs& a, int code, bool zero_counts) {
  const int G = a.E + a.B;
  for (int i = threadIdx.x; i < a.R * G; i += blockDim.x) a.cu[i] = 0;
  for (int i = threadIdx.x; i < a.R * a.B; i += blockDim.x) a.slot_expert[i] = -1;
  if (zero_counts)
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) a.counts[e] = 0;
  if (threadIdx.x == 0) *a.status = code;
}

template <int W> struct Vec;
template <> struct Vec<1> {
  using T = int;
  static __device__ __forceinline__ int get(const int& v, int) { return v; }
  static __device__ __forceinline__ int make(const int* s) { return s[0]; }
};
template <> struct Vec<4> {
  using T = int4;
  static __device__ __forceinline__ int get(const int4& v, int j) {
    return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
  }
  static __device__ __forceinline__ int4 make(const int* s) {
    return make_int4(s[0], s[1], s[2], s[3]);
  }
};

// Column c of tiles [b0, b1): adds their counts to s and rewrites each tile's
// counts as its prefix within the range (the sum of the earlier tiles). The
// loads of a batch of NB tiles all go out before any of their stores: each
// store writes the array the next load reads, so a load-store-load order
// would wait one L2 round trip per tile.
template <int W, int NB>
__device__ __forceinline__ void prefix_tiles(typename Vec<W>::T* h, int nc, int c, int b0, int b1,
                                             int (&s)[W]) {
  using V = typename Vec<W>::T;
  for (int b = b0; b < b1; b += NB) {
    V v[NB];
#pragma unroll
    for (int i = 0; i < NB; ++i)
      if (b + i < b1) v[i] = __ldcg(h + size_t(b + i) * nc + c);
#pragma unroll
    for (int i = 0; i < NB; ++i)
      if (b + i < b1) {
        h[size_t(b + i) * nc + c] = Vec<W>::make(s);
#pragma unroll
        for (int j = 0; j < W; ++j) s[j] += Vec<W>::get(v[i], j);
      }
  }
}

// Tiles are split into Gs groups of tpg consecutive tiles (tile_groups()).
// tile_group_sums: T_e, and for every group g the count of e in all tiles
// before g (groupbase). While summing a group's tiles (when k_gsum has not
// already), it rewrites each tile's counts as the tile's prefix within the
// group; a k_offsets CTA adds that row to its group's base. Columns are W
// experts wide; thread (g, c) owns group g of column c.
// Row pitch of the shared group sums: odd, so that the column writes of
// tile_group_sums spread over 8 banks; a single group needs no padding.
__host__ __device__ inline int part_pitch(int Gs) {
  return Gs == 1 ? 1 : ((Gs & 1) ? Gs + 2 : Gs + 1);
}

// The most groups (<= max_groups <= kMaxScanGroups, <= nblk) whose E rows of
// part_pitch ints fit kPartInts; E <= MEP_MAX_E = kPartInts / 2 always fits
// one group.
inline void tile_groups(int nblk, int E, int max_groups, int* Gs, int* tpg) {
  int g = nblk < max_groups ? nblk : max_groups;
  while (g > 1 && E * part_pitch(g) > kPartInts) --g;
  if (g < 1) g = 1;
  *tpg = nblk > 0 ? (nblk + g - 1) / g : 1;
  // only the groups that hold tiles (97 tiles in groups of 2: 49, not 64)
  *Gs = nblk > 0 ? (nblk + *tpg - 1) / *tpg : 1;
}

// Also collects k_hist's error words: their loads go out with the counts,
// and the lowest failing tile lands in *s_errblk (initialised before the
// call) by the end.
template <int W>
__device__ void tile_group_sums(const PlanArgs& a, int* sPart, int* sT, int* s_errblk) {
  using V = typename Vec<W>::T;
  const int E = a.E, nblk = a.nblk, nthr = blockDim.x, tid = threadIdx.x;
  const int nc = E / W;
  const int Gs = a.Gs, tpg = a.tpg;
  const int P = part_pitch(Gs);
  const int err0 = tid < nblk ? __ldcg(a.ws.blockerr + tid) : 0;  // in flight with the counts
  if (a.presummed) {
    // k_gsum already summed each group: Gs x E ints, one load each
    const V* gsum = reinterpret_cast<const V*>(a.ws.groupsum);
    for (int x = tid; x < Gs * nc; x += nthr) {
      const int g = x / nc, c = x - g * nc;
      const V v = __ldcg(gsum + x);
#pragma unroll
      for (int j = 0; j < W; ++j) sPart[(c * W + j) * P + g] = Vec<W>::get(v, j);
    }
  } else {
    V* h = reinterpret_cast<V*>(a.ws.blockhist);
    for (int x = tid; x < Gs * nc; x += nthr) {
      const int g = x / nc, c = x - g * nc;
      const int b0 = min(nblk, g * tpg), b1 = min(nblk, b0 + tpg);
      int s[W];
#pragma unroll
      for (int j = 0; j < W; ++j) s[j] = 0;
      prefix_tiles<W, 4>(h, nc, c, b0, b1, s);
#pragma unroll
      for (int j = 0; j < W; ++j) sPart[(c * W + j) * P + g] = s[j];
    }
  }
  __syncthreads();
  {
    int bad = err0 != 0 ? tid : INT_MAX;
    for (int b = tid + nthr; b < nblk; b += nthr)
      if (bad == INT_MAX && __ldcg(a.ws.blockerr + b) != 0) bad = b;
    if (bad != INT_MAX) atomicMin(s_errblk, bad);
  }
  // one thread per expert: exclusive scan over its Gs <= 64 group sums. The
  // rows have odd pitch P, so a warp's 32 experts read 32 different banks;
  // groupbase is group-major, so a warp's writes of one group coalesce (and
  // so do k_offsets' reads). (Splitting an expert's groups over several
  // lanes measured slower: its group-major writes no longer coalesce.)
  for (int e = tid; e < E; e += nthr) {
    const int* row = sPart + e * P;
    int run = 0;
#pragma unroll 8
    for (int g = 0; g < Gs; ++g) {
      const int v = row[g];
      a.ws.groupbase[g * E + e] = run;
      run += v;
    }
    sT[e] = run;
    a.counts[e] = run;
  }
  __syncthreads();
}

// E % 4 != 0: scalar columns, out of line (see keep_warp0).
__device__ __noinline__ void tile_group_sums_scalar(const PlanArgs& a, int* sPart, int* sT,
                                                    int* s_errblk) {
  tile_group_sums<1>(a, sPart, sT, s_errblk);
}

// k_gsum: CTA g sums the tile counts of its group of tpg consecutive tiles,
// W experts per thread (all of a column's tile loads in flight together),
// into groupsum[g][e].
template <int W>
__global__ void __launch_bounds__(kTileThreads)
    k_gsum(int* __restrict__ blockhist, int nblk, int E, int tpg, int* __restrict__ groupsum) {
  pdl_wait();  // k_hist's counts
  pdl_launch_dependents();
  using V = typename Vec<W>::T;
  const int nc = E / W, g = blockIdx.x;
  const int b0 = min(nblk, g * tpg), b1 = min(nblk, b0 + tpg);
  V* h = reinterpret_cast<V*>(blockhist);
  V* out = reinterpret_cast<V*>(groupsum) + size_t(g) * nc;
  for (int c = threadIdx.x; c < nc; c += blockDim.x) {
    int s[W];
#pragma unroll
    for (int j = 0; j < W; ++j) s[j] = 0;
    prefix_tiles<W, 16>(h, nc, c, b0, b1, s);
    int t[4] = {0, 0, 0, 0};
#pragma unroll
    for (int j = 0; j < W; ++j) t[j] = s[j];
    out[c] = Vec<W>::make(t);
  }
}

// Three exclusive block scans in one pass (out_i may alias in_i; out_i[n]
// gets the total): one round of warp scans and one pair of barriers for all
// three. s_w holds >= 3 * 33 ints. Ends with __syncthreads().
__device__ void block_excl_scan3(const int* in0, int* out0, const int* in1, int* out1,
                                 const int* in2, int* out2, int n, int* s_w) {
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = (nthr + 31) >> 5;
  const int per = (n + nthr - 1) / nthr;
  const int beg = min(n, tid * per), end = min(n, beg + per);
  int l0 = 0, l1 = 0, l2 = 0;
  for (int i = beg; i < end; ++i) {
    l0 += in0[i];
    l1 += in1[i];
    l2 += in2[i];
  }
  const int i0 = warp_incl_scan(l0), i1 = warp_incl_scan(l1), i2 = warp_incl_scan(l2);
  if (lane == 31) {
    s_w[warp] = i0;
    s_w[33 + warp] = i1;
    s_w[66 + warp] = i2;
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int q = 0; q < 3; ++q) {
      const int v = lane < nwarps ? s_w[33 * q + lane] : 0;
      const int vi = warp_incl_scan(v);
      s_w[33 * q + lane] = vi - v;
      if (lane == 31) s_w[33 * q + 32] = vi;
    }
  }
  __syncthreads();
  int r0 = s_w[warp] + i0 - l0, r1 = s_w[33 + warp] + i1 - l1, r2 = s_w[66 + warp] + i2 - l2;
  for (int i = beg; i < end; ++i) {
    const int v0 = in0[i], v1 = in1[i], v2 = in2[i];
    out0[i] = r0;
    out1[i] = r1;
    out2[i] = r2;
    r0 += v0;
    r1 += v1;
    r2 += v2;
  }
  if (tid == 0) {
    out0[n] = s_w[32];
    out1[n] = s_w[65];
    out2[n] = s_w[98];
  }
  __syncthreads();
}

// Exclusive scan of a short array by warp 0 (out may alias in; out[n] =
// total). Ends with __syncthreads().
__device__ void warp0_excl_scan(const int* in, int* out, int n) {
  if ((threadIdx.x >> 5) == 0) {
    const int lane = threadIdx.x & 31;
    int carry = 0;
    for (int i0 = 0; i0 < n; i0 += 32) {
      const int i = i0 + lane;
      const int v = i < n ? in[i] : 0;
      const int incl = warp_incl_scan(v);
      if (i < n) out[i] = carry + incl - v;
      carry += __shfl_sync(MEP_FULL_MASK, incl, 31);
    }
    if (lane == 0) out[n] = carry;
  }
  __syncthreads();
}

// Shared-memory arrays of k_plan, carved from its dynamic shared memory.
struct PlanSmem {
  int *sT, *sPre, *sKeep, *sOv, *sOst, *sOlist, *sFlag, *sPcBeg, *sPcCnt, *sPlen, *sPart, *sDef,
      *sDst, *sNp, *sPex, *sQ0, *sKpre;
};
__device__ __forceinline__ PlanSmem plan_smem(int E, int R) {
  extern __shared__ int smem[];
  const int EP = E + 1, RP = R + 1;
  PlanSmem P;
  P.sT = smem;                    // [E+1]
  P.sPre = P.sT + EP;             // [E+1]
  P.sKeep = P.sPre + EP;          // [E+1]
  P.sOv = P.sKeep + EP;           // [E+1]
  P.sOst = P.sOv + EP;            // [E+1]
  P.sOlist = P.sOst + EP;         // [E+1]
  P.sFlag = P.sOlist + EP;        // [E+1] overflow flags, then their numbering
  P.sPcBeg = P.sFlag + EP;        // [E+1]
  P.sPcCnt = P.sPcBeg + EP;       // [E+1]
  P.sPlen = P.sPcCnt + EP;        // [E+R] piece lengths, by global piece index
  P.sPart = P.sPlen + E + R;      // [kPartInts] group sums, then the running sum of keep
  P.sDef = P.sPart + kPartInts;   // [R+1]
  P.sDst = P.sDef + RP;           // [R+1]
  P.sNp = P.sDst + RP;            // [R+1]
  P.sPex = P.sNp + RP;            // [R+1]
  P.sQ0 = P.sPex + RP;            // [R+1] first overflow segment of each rank
  P.sKpre = P.sPart;              // [E+1] exclusive prefix of keep, total at E
  return P;
}

// The keep / overflow / deficit phase for shapes the one-warp-per-rank pass
// does not cover. They are kept out of line, with the failure path and the
// inference-overflow row walk below, so that the path the common shapes take
// is one short stretch of code. (Measured about even against the inlined
// form; running the planner twice in one CTA showed that instruction fetch
// is not what its time goes to.)
// Up to 128 experts: warp 0, one pass over chunks of 32 experts (three warp
// scans per chunk, no block barrier).
__device__ __noinline__ void keep_warp0(const PlanArgs& a) {
  const int E = a.E, R = a.R, per = E / R, SK = a.S * a.K;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const PlanSmem P = plan_smem(E, R);
  int *sT = P.sT, *sPre = P.sPre, *sKeep = P.sKeep, *sOv = P.sOv, *sOst = P.sOst,
      *sOlist = P.sOlist, *sFlag = P.sFlag, *sDef = P.sDef, *sDst = P.sDst, *sKpre = P.sKpre;
  if (warp == 0) {
    int cT = 0, cO = 0, cF = 0, cK = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int T = e < E ? sT[e] : 0;
      const int iT = warp_incl_scan(T);
      if (e < E) sPre[e] = cT + iT - T;
      cT += __shfl_sync(MEP_FULL_MASK, iT, 31);
      __syncwarp();  // sPre of this chunk visible to the whole warp
      int ov = 0;
      if (e < E) {
        const int r = e / per;
        const int kp = max(0, min(T, SK - (sPre[e] - sPre[r * per])));
        ov = T - kp;
        sKeep[e] = kp;
        sOv[e] = ov;
        a.ws.etab[4 * e] = kp;
      }
      const int iO = warp_incl_scan(ov);
      if (e < E) sOst[e] = cO + iO - ov;
      cO += __shfl_sync(MEP_FULL_MASK, iO, 31);
      const int kp = e < E ? T - ov : 0;
      const int iK = warp_incl_scan(kp);
      if (e < E) sKpre[e] = cK + iK - kp;
      cK += __shfl_sync(MEP_FULL_MASK, iK, 31);
      const int f = ov > 0 ? 1 : 0;
      const int iF = warp_incl_scan(f);
      if (f) sOlist[cF + iF - 1] = e;
      cF += __shfl_sync(MEP_FULL_MASK, iF, 31);
    }
    if (lane == 0) {
      sPre[E] = cT;
      sOst[E] = cO;
      sFlag[E] = cF;
      sKpre[E] = cK;
    }
    __syncwarp();
    // deficits S*K - load_r (rank order) and their exclusive running sum
    int cD = 0;
    for (int r0 = 0; r0 < R; r0 += 32) {
      const int r = r0 + lane;
      const int d = r < R ? max(0, SK - (sPre[(r + 1) * per] - sPre[r * per])) : 0;
      const int iD = warp_incl_scan(d);
      if (r < R) {
        sDef[r] = d;
        sDst[r] = cD + iD - d;
      }
      cD += __shfl_sync(MEP_FULL_MASK, iD, 31);
    }
    if (lane == 0) sDst[R] = cD;
  }
  __syncthreads();
}

// Beyond: block-wide scans (faster on GB300 from E = 256 on).
__device__ __noinline__ void keep_blocks(const PlanArgs& a, int* s_warp) {
  const int E = a.E, R = a.R, per = E / R, SK = a.S * a.K;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const PlanSmem P = plan_smem(E, R);
  int *sT = P.sT, *sPre = P.sPre, *sKeep = P.sKeep, *sOv = P.sOv, *sOst = P.sOst,
      *sOlist = P.sOlist, *sFlag = P.sFlag, *sDef = P.sDef, *sDst = P.sDst, *sKpre = P.sKpre;
  block_excl_scan(sT, sPre, E, s_warp, true);
  for (int e = tid; e < E; e += nthr) {
    const int r = e / per;
    const int before = sPre[e] - sPre[r * per];
    const int kp = max(0, min(sT[e], SK - before));
    sKeep[e] = kp;
    sOv[e] = sT[e] - kp;
    sFlag[e] = sOv[e] > 0 ? 1 : 0;
    a.ws.etab[4 * e] = kp;
  }
  __syncthreads();
  block_excl_scan3(sOv, sOst, sFlag, sFlag, sKeep, sKpre, E, s_warp);
  for (int e = tid; e < E; e += nthr)
    if (sOv[e] > 0) sOlist[sFlag[e]] = e;
  for (int r = tid; r < R; r += nthr)
    sDef[r] = max(0, SK - (sPre[(r + 1) * per] - sPre[r * per]));
  __syncthreads();
  warp0_excl_scan(sDef, sDst, R);
}

// Inference overflow present (pieces beyond B sit in home rows): cu_seqlens
// and the row bases by one warp per rank walking its rows in chunks of 32.
// Row j of rank r: home rows keep their kept count, slot rows E + b hold
// piece b < B, and pieces b >= B sit in the expert's own row e, found by a
// binary search over the rank's remaining pieces, whose experts ascend with
// b. g = the piece, or -1. Out of line (see keep_warp0).
__device__ __noinline__ void rows_with_overflow(const PlanArgs& a) {
  const int E = a.E, R = a.R, B = a.B, per = E / R, SK = a.S * a.K, G = E + B;
  const PlanSmem P = plan_smem(E, R);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int *sKeep = P.sKeep, *sOlist = P.sOlist, *sPlen = P.sPlen, *sNp = P.sNp, *sPex = P.sPex,
      *sQ0 = P.sQ0;
  auto row_count = [&](int r, int j, int& g) -> int {
    g = -1;
    const int np = sNp[r];
    if (j < E) {
      if (j / per == r) return sKeep[j];
      if (np > B) {
        const int q0 = sQ0[r];
        int lo = B, hi = np;
        while (lo < hi) {
          const int m = (lo + hi) >> 1;
          if (sOlist[q0 + m] < j) lo = m + 1; else hi = m;
        }
        if (lo < np && sOlist[q0 + lo] == j) {
          g = sPex[r] + lo;
          return sPlen[g];
        }
      }
      return 0;
    }
    if (j < G && j - E < min(np, B)) {
      g = sPex[r] + (j - E);
      return sPlen[g];
    }
    return 0;
  };
  auto write_row = [&](int r, int j, int c, int g, int incl_end) {
    a.cu[size_t(r) * G + j] = incl_end;
    const int start = r * SK + incl_end - c;
    if (j < E && j / per == r) a.ws.etab[4 * j + 1] = start;
    else if (g >= 0) a.ws.piece_base[g] = start;
  };
  for (int r = warp; r < R; r += nwarps) {
    int carry = 0;
    for (int j0 = 0; j0 < G; j0 += 32) {
      const int j = j0 + lane;
      int g;
      const int c = j < G ? row_count(r, j, g) : 0;
      const int incl = warp_incl_scan(c);
      if (j < G) write_row(r, j, c, g, carry + incl);
      carry += __shfl_sync(MEP_FULL_MASK, incl, 31);
    }
  }
}

// The arguments are a __grid_constant__ parameter: the out-of-line helpers
// read them in place, with no per-thread copy.
__global__ void __launch_bounds__(kPlanThreads) k_plan(const __grid_constant__ PlanArgs a) {
  pdl_wait();                // k_hist's counts and error words (k_gsum's group sums)
  // k_offsets starts now and ranks its tile (from the routing alone) while
  // this CTA plans. (Releasing it before the wait, while k_hist still runs,
  // measured 1.2-1.8 us slower at E = 64 and no faster at E = 256.)
  pdl_launch_dependents();
  const int E = a.E, R = a.R, B = a.B;
  const int per = E / R;
  const int SK = a.S * a.K;
  const int G = E + B;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
  const PlanSmem P = plan_smem(E, R);
  int *sT = P.sT, *sKeep = P.sKeep, *sOv = P.sOv, *sOst = P.sOst, *sOlist = P.sOlist,
      *sFlag = P.sFlag, *sPcBeg = P.sPcBeg, *sPcCnt = P.sPcCnt, *sPlen = P.sPlen,
      *sPart = P.sPart, *sDef = P.sDef, *sDst = P.sDst, *sNp = P.sNp, *sPex = P.sPex,
      *sQ0 = P.sQ0;
  __shared__ int s_warp[3 * 33];
  __shared__ int s_errblk, s_cap, s_over;

  if (tid == 0) {  // ordered before every use by the barriers in tile_group_sums
    s_errblk = INT_MAX;
    s_cap = 0;
    s_over = 0;
  }
  // 1. T_e and the per-group prefixes of the tile counts; with them, the
  //    routing errors k_hist found (lowest tile wins)
  if ((E & 3) == 0) tile_group_sums<4>(a, sPart, sT, &s_errblk);
  else tile_group_sums_scalar(a, sPart, sT, &s_errblk);
  if (s_errblk != INT_MAX) {
    plan_fail(a, a.ws.blockerr[s_errblk], true);
    return;
  }

  // 2. home-first keep: the count of e's earlier home experts is a
  //    difference of the running sum of T; then
  // 3. overflow segments (expert order) and deficits (rank order) on one
  //    line. Where E/R <= 32 and R <= 32, one warp per rank (below);
  //    otherwise, up to 128 experts, warp 0 does both in one pass over
  //    chunks of 32 experts (three warp scans per chunk, no block barrier),
  //    and beyond, block-wide scans (faster on GB300 from E = 256 on).
  // (the group sums are consumed: sPart now holds the running sum of keep)
  int* sKpre = sPart;  // [E+1] exclusive prefix of keep, total at E
  if (MEP_PLAN_RANK_WARPS && per <= 32 && R <= nwarps) {
    // Warp r holds rank r's home experts, one per lane: the keep, overflow,
    // flag and keep prefixes inside the rank are warp scans, and the rank's
    // load gives its deficit. After one block barrier every rank's warp scans
    // the R rank totals itself and adds its own offsets (warp 0 also the
    // deficits' running sum): two block barriers in all.
    const int r = warp, e = r * per + lane;
    const bool in = r < R && lane < per;
    int ov = 0, f = 0, kp = 0, exO = 0, exF = 0, exK = 0;
    if (r < R) {
      const int T = in ? sT[e] : 0;
      const int iT = warp_incl_scan(T);
      kp = in ? max(0, min(T, SK - (iT - T))) : 0;
      ov = T - kp;
      f = ov > 0 ? 1 : 0;
      const int iO = warp_incl_scan(ov), iF = warp_incl_scan(f), iK = warp_incl_scan(kp);
      exO = iO - ov;
      exF = iF - f;
      exK = iK - kp;
      if (in) {
        sKeep[e] = kp;
        sOv[e] = ov;
        a.ws.etab[4 * e] = kp;
      }
      if (lane == 31) {
        s_warp[r] = iO;
        s_warp[33 + r] = iF;
        s_warp[66 + r] = iK;
        sDef[r] = max(0, SK - iT);  // iT at lane 31: the rank's load
      }
    }
    __syncthreads();
    if (r < R) {
      const int vO = lane < R ? s_warp[lane] : 0;
      const int vF = lane < R ? s_warp[33 + lane] : 0;
      const int vK = lane < R ? s_warp[66 + lane] : 0;
      const int iO = warp_incl_scan(vO), iF = warp_incl_scan(vF), iK = warp_incl_scan(vK);
      const int bO = __shfl_sync(MEP_FULL_MASK, iO - vO, r);  // this rank's exclusive offsets
      const int bF = __shfl_sync(MEP_FULL_MASK, iF - vF, r);
      const int bK = __shfl_sync(MEP_FULL_MASK, iK - vK, r);
      if (in) {
        sOst[e] = bO + exO;
        if (f) sOlist[bF + exF] = e;
        sKpre[e] = bK + exK;
      }
      if (r == 0) {
        const int d = lane < R ? sDef[lane] : 0;
        const int iD = warp_incl_scan(d);
        if (lane < R) sDst[lane] = iD - d;
        if (lane == 31) {  // the totals
          sDst[R] = iD;
          sOst[E] = iO;
          sFlag[E] = iF;
          sKpre[E] = iK;
        }
      }
    }
    __syncthreads();
  } else if (E <= MEP_PLAN_WARP_SCAN_MAX_E) {
    keep_warp0(a);
  } else {
    keep_blocks(a, s_warp);
  }
  const int nov = sFlag[E];

  // 4. pieces of each under-loaded rank: the overflow segments that meet
  //    [Dst_r, Dst_r + d_r), in expert order, one slot each. First count
  //    them (and find the first segment), then number them globally in rank
  //    order, then write them.
  for (int e = tid; e < E; e += nthr) {  // per-expert piece tables, filled below
    sPcBeg[e] = INT_MAX;
    sPcCnt[e] = 0;
  }
  // Rank r's pieces: the segments tile the overflow line in order, so the
  // ones meeting [lo, hi) are those from the first ending after lo up to
  // (not including) the first starting at or after hi: two binary searches.
  auto count_pieces = [&](int r, int& q0) -> int {
    q0 = 0;
    const int d = sDef[r];
    if (d <= 0) return 0;
    const int lo = sDst[r], hi = lo + d;
    int q1 = nov;
    while (q0 < q1) {
      const int m = (q0 + q1) >> 1;
      const int e = sOlist[m];
      if (sOst[e] + sOv[e] > lo) q1 = m; else q0 = m + 1;
    }
    int q2 = q0, q3 = nov;
    while (q2 < q3) {
      const int m = (q2 + q3) >> 1;
      if (sOst[sOlist[m]] >= hi) q3 = m; else q2 = m + 1;
    }
    return q2 - q0;
  };
  if (R <= 32) {
    // warp 0, one rank per lane: count, flag, and number the pieces (a warp
    // scan) with no block barrier in between
    if (warp == 0) {
      int q0 = 0;
      const int np = lane < R ? count_pieces(lane, q0) : 0;
      if (__any_sync(MEP_FULL_MASK, np > B) && lane == 0) {
        if (!a.fallback) s_cap = 1;
        s_over = 1;  // inference: pieces beyond B sit in home rows
      }
      const int incl = warp_incl_scan(np);
      if (lane < R) {
        sNp[lane] = np;
        sQ0[lane] = q0;
        sPex[lane] = incl - np;
      }
      if (lane == 31) sPex[R] = incl;  // pieces in all
    }
    __syncthreads();
  } else {
    for (int r = tid; r < R; r += nthr) {
      int q0;
      const int np = count_pieces(r, q0);
      if (np > B) {
        if (!a.fallback) s_cap = 1;
        s_over = 1;
      }
      sNp[r] = np;
      sQ0[r] = q0;
    }
    __syncthreads();
    warp0_excl_scan(sNp, sPex, R);  // sPex[R]: pieces in all
  }
  if (s_cap) {
    plan_fail(a, MEP_ERR_CAPACITY, false);
    return;
  }
  // slot table, one thread per (rank, slot): the rank's b-th piece's expert,
  // or -1 (pieces beyond B, inference only, have no slot)
  for (int i = tid; i < R * B; i += nthr) {
    const int r = i / B, b = i - r * B;
    a.slot_expert[i] = b < sNp[r] ? sOlist[sQ0[r] + b] : -1;
  }
  // pieces, one thread each; its rank is the last r with sPex[r] <= g
  // (empty ranks repeat their successor's start, so the last one is right)
  const int npieces = min(sPex[R], E + R);  // <= overflow experts + deficit ranks - 1
  for (int g = tid; g < npieces; g += nthr) {
    int lo = 0, hi = R;
    while (hi - lo > 1) {
      const int m = (lo + hi) >> 1;
      if (sPex[m] <= g) lo = m; else hi = m;
    }
    const int r = lo, b = g - sPex[r];
    const int e = sOlist[sQ0[r] + b];
    const int os = sOst[e], oe = os + sOv[e];
    const int dlo = sDst[r], dhi = dlo + sDef[r];
    const int st = max(os, dlo), en = min(oe, dhi);
    a.ws.piece_lo[g] = sKeep[e] + (st - os);
    sPlen[g] = en - st;
    atomicMin(&sPcBeg[e], g);
    atomicAdd(&sPcCnt[e], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += nthr) {
    a.ws.etab[4 * e + 2] = sPcCnt[e] ? sPcBeg[e] : 0;
    a.ws.etab[4 * e + 3] = sPcCnt[e];
  }

  // 5. cu_seqlens; also the global first row of every home row and piece.
  if (!s_over) {
    // Every piece sits in a slot row (no inference overflow), so every entry
    // has a closed form and all R x (E+B) are written in one parallel pass.
    // Rank r keeps SK - d_r tokens on its home rows (their running sum is a
    // difference of the keep prefix); slot piece b covers [max(os, lo),
    // min(oe, lo + d_r)) of the overflow line, lo the rank's start on it, so
    // it starts at SK - d_r + (max(os, lo) - lo) in the rank's buffer.
    for (int i = tid; i < R * G; i += nthr) {
      const int r = i / G, j = i - r * G;
      const int s0 = r * per, d = sDef[r];
      int c;
      if (j < E) {
        c = j < s0 ? 0 : sKpre[min(j + 1, s0 + per)] - sKpre[s0];
        if (j >= s0 && j < s0 + per) a.ws.etab[4 * j + 1] = r * SK + sKpre[j] - sKpre[s0];
      } else if (j - E < sNp[r]) {
        const int b = j - E, e = sOlist[sQ0[r] + b];
        const int lo = sDst[r], os = sOst[e], oe = os + sOv[e];
        c = SK - d + (min(oe, lo + d) - lo);
        a.ws.piece_base[sPex[r] + b] = r * SK + SK - d + (max(os, lo) - lo);
      } else {
        c = SK;
      }
      a.cu[size_t(r) * G + j] = c;
    }
    if (tid == 0) *a.status = MEP_OK;
    return;
  }
  rows_with_overflow(a);
  if (tid == 0) *a.status = MEP_OK;
}

// ---------------------------------------------------------------------------
// k_offsets: destination rows. Two forms share the tables below: up to K = 8
// one token per thread (k_offsets_tok), beyond that a tile of up to 2048
// assignments ranked warp by warp (k_offsets).

// After the planner: per expert, with this tile's base gb (the count of e in
// all earlier tiles: its group's base from the planner plus the tile's
// prefix within the group) folded in. A kept token's row is home_base + gb +
// rel, for rel < keep - gb (one 8-byte shared load on the common path); the
// rest go through the expert's pieces, whose tables sit in shared memory when
// they fit (pieces_smem), else are read from the workspace.
struct RowTables {
  const int2* fast;   // [E] {home_base + gb, keep - gb}
  const int2* slow;   // [E] {gb, first piece | pieces << 16}
  const int* plo;     // [E+R] first list index covered by each piece
  const int* pbase;   // [E+R] global row of each piece's first token
};

__device__ __forceinline__ RowTables load_row_tables(int* tab, int* s_pc, int pieces_smem, int E,
                                                     int R, int g, int blk, const PlanWs& ws) {
  int2* s_fast = reinterpret_cast<int2*>(tab);
  int2* s_slow = s_fast + E;
  const int4* etab = reinterpret_cast<const int4*>(ws.etab);
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int gb = __ldcg(ws.groupbase + size_t(g) * E + e) +
                   __ldcg(ws.blockhist + size_t(blk) * E + e);
    const int4 t = __ldcg(etab + e);
    s_fast[e] = make_int2(t.y + min(gb, t.x), t.x - gb);  // (no kept token left: unused base)
    s_slow[e] = make_int2(gb, t.z | (t.w << 16));
  }
  if (pieces_smem)
    for (int q = threadIdx.x; q < E + R; q += blockDim.x) {
      s_pc[q] = __ldcg(ws.piece_lo + q);
      s_pc[E + R + q] = __ldcg(ws.piece_base + q);
    }
  return RowTables{s_fast, s_slow, pieces_smem ? s_pc : ws.piece_lo,
                   pieces_smem ? s_pc + E + R : ws.piece_base};
}

// Before the wait: ask L2 for the lines load_row_tables reads after it. A
// prefetch returns no value (nothing written by an earlier kernel is read
// before the wait); it warms the address translation and starts the fetch.
__device__ __forceinline__ void prefetch_row_tables(int pieces_smem, int E, int R, int g, int blk,
                                                    const PlanWs& ws, const int32_t* status) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    prefetch_l2(ws.groupbase + size_t(g) * E + e);
    prefetch_l2(ws.blockhist + size_t(blk) * E + e);
    prefetch_l2(ws.etab + 4 * e);
  }
  if (pieces_smem)
    for (int q = threadIdx.x; q < E + R; q += blockDim.x) {
      prefetch_l2(ws.piece_lo + q);
      prefetch_l2(ws.piece_base + q);
    }
  if (threadIdx.x == 0 && status != nullptr) prefetch_l2(status);
}

// Row of the assignment of expert e with rank rel among the tile's
// assignments of e.
__device__ __forceinline__ int dest_row(const RowTables& T, int e, int rel) {
  const int2 f = T.fast[e];
  if (rel < f.y) return f.x + rel;
  const int2 sl = T.slow[e];
  const int i = sl.x + rel;  // index of the token in expert e's list
  // the expert's pieces are consecutive and their first list indices
  // ascend: the last piece starting at or before i holds the token
  int p = sl.y & 0xffff, hi = p + (sl.y >> 16) - 1;
  while (p < hi) {
    const int m = (p + hi + 1) >> 1;
    if (T.plo[m] <= i) p = m; else hi = m - 1;
  }
  return T.pbase[p] + (i - T.plo[p]);
}

// K <= 8, one token per thread (tiles of 256 tokens). A token never holds an
// expert twice (the planner reports bad routing otherwise, and then nothing
// is written), so an assignment's rank among its warp's assignments of the
// same expert is the number of earlier lanes holding that expert: each lane
// sets its bit in a per-warp mask of every expert it holds (shared-memory
// atomicOr, order-free), and the rank is the population count of the mask
// below the lane. The per-warp counts (population counts of the masks)
// become exclusive offsets within the tile, as in the tile form below.
// out_vec: the widest store of a token's K rows the alignment of dst_pos and
// K allow (4, 2 or 1 ints).
__global__ void __launch_bounds__(kTileThreads)
    k_offsets_tok(const int32_t* __restrict__ topk_idx, int N, int K, int E, int R, int tpg,
                  int pieces_smem, int out_vec, PlanWs ws, const int32_t* __restrict__ status,
                  int32_t* __restrict__ dst_pos) {
  extern __shared__ int smem[];
  unsigned* s_mask = reinterpret_cast<unsigned*>(smem);  // [kTileWarps, E]; then the row tables
  int* s_pc = smem + kTileWarps * E;                    // piece tables, when they fit
  const int blk = blockIdx.x, tt = threadIdx.x;
  const int lane = tt & 31, warp = tt >> 5;
  const size_t t = size_t(blk) * kTileThreads + tt;
  const bool has = t < size_t(N);
  // Up to the wait, only the routing (an input) is read.
  int v[kTokMaxK];
#pragma unroll
  for (int k = 0; k < kTokMaxK; ++k) v[k] = -1;
  if (has) load_token_ids(topk_idx + t * K, K, v);
  for (int i = tt; i < kTileWarps * E; i += blockDim.x) s_mask[i] = 0;
  __syncthreads();
  unsigned* wm = s_mask + warp * E;
#pragma unroll
  for (int k = 0; k < kTokMaxK; ++k)
    if (k < K && v[k] >= 0 && v[k] < E) atomicOr(&wm[v[k]], 1u << lane);
  __syncthreads();
  int rel[kTokMaxK];
#pragma unroll
  for (int k = 0; k < kTokMaxK; ++k)
    rel[k] = k < K && v[k] >= 0 && v[k] < E ? __popc(wm[v[k]] & lanemask_lt()) : 0;
  __syncthreads();
  for (int e = tt; e < E; e += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kTileWarps; ++w) {
      const int c = __popc(s_mask[w * E + e]);
      s_mask[w * E + e] = unsigned(run);
      run += c;
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kTokMaxK; ++k)
    if (k < K && v[k] >= 0 && v[k] < E) rel[k] += int(wm[v[k]]);
  prefetch_row_tables(pieces_smem, E, R, blk / tpg, blk, ws, status);
  __syncthreads();  // the masks' space is reused below

  pdl_wait();  // the planner's tables and status
  pdl_launch_dependents();
  const int st = status != nullptr ? __ldcg(status) : 0;
  const RowTables T = load_row_tables(smem, s_pc, pieces_smem, E, R, blk / tpg, blk, ws);
  if (st != 0) return;  // uniform: one status word
  __syncthreads();
  if (!has) return;
  // status 0: every id is in [0, E) and distinct within the token
  int row[kTokMaxK];
#pragma unroll
  for (int k = 0; k < kTokMaxK; ++k)
    if (k < K) row[k] = dest_row(T, v[k], rel[k]);
  int32_t* out = dst_pos + t * K;
  if (out_vec == 4) {
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (4 * q < K)
        reinterpret_cast<int4*>(out)[q] =
            make_int4(row[4 * q], row[4 * q + 1], row[4 * q + 2], row[4 * q + 3]);
  } else if (out_vec == 2) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (2 * q < K) reinterpret_cast<int2*>(out)[q] = make_int2(row[2 * q], row[2 * q + 1]);
  } else {
#pragma unroll
    for (int k = 0; k < kTokMaxK; ++k)
      if (k < K) out[k] = row[k];
  }
}

// K > 8: a tile of up to 2048 assignments.
__global__ void __launch_bounds__(kTileThreads)
    k_offsets(const int32_t* __restrict__ topk_idx, int N, int K, int E, int R,
              int tok_per_tile, int tpg, int pieces_smem, PlanWs ws,
              const int32_t* __restrict__ status, int32_t* __restrict__ dst_pos) {
  extern __shared__ int smem[];
  int* s_idx = smem;                          // [kTileAssign]
  int* s_wcnt = smem + kTileAssign;           // [kTileWarps, E]; after the wait, the row tables
  int* s_pc = s_wcnt + kTileWarps * E;        // piece tables, when they fit (pieces_smem)
  const int blk = blockIdx.x;
  const int t0 = blk * tok_per_tile;
  const int ntok = min(tok_per_tile, N - t0);
  const int na = ntok * K;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // Everything up to the wait depends only on the routing (an input, complete
  // before k_hist started), so it overlaps the histogram and the planner:
  // stage the tile, then rank each assignment among the tile's assignments
  // of the same expert. Nothing an earlier kernel of the plan writes is read
  // before the wait.
  {
    const int32_t* g = topk_idx + size_t(t0) * K;
    const int nv = na >> 2;
    const int4* g4 = reinterpret_cast<const int4*>(g);
    int4* s4 = reinterpret_cast<int4*>(s_idx);
    for (int i = threadIdx.x; i < nv; i += blockDim.x) s4[i] = __ldg(g4 + i);
    for (int i = (nv << 2) + threadIdx.x; i < na; i += blockDim.x) s_idx[i] = __ldg(g + i);
  }
  for (int i = threadIdx.x; i < kTileWarps * E; i += blockDim.x) s_wcnt[i] = 0;
  __syncthreads();

  // Warp w owns the contiguous assignment range [wbeg, wend) of the tile,
  // so (warp, iteration, lane) order is the flattened (token, k) order.
  // Ids outside [0, E) are skipped here; the planner then reports bad
  // routing and the kernel returns after the wait without writing.
  const int chunk = (((na + kTileWarps - 1) / kTileWarps) + 31) & ~31;
  const int wbeg = min(na, warp * chunk), wend = min(na, wbeg + chunk);
  int* wc = s_wcnt + warp * E;
  int loc[kWarpIters];
#pragma unroll
  for (int j = 0; j < kWarpIters; ++j) {
    loc[j] = 0;
    const int a = wbeg + j * 32 + lane;
    if (wbeg + j * 32 < wend) {          // warp-uniform
      const int e = a < wend ? s_idx[a] : -1;
      const bool in = e >= 0 && e < E;
      const unsigned m = __ballot_sync(MEP_FULL_MASK, in);
      int cur = 0;
      unsigned peers = 0;
      if (in) {
        peers = __match_any_sync(m, e);
        cur = wc[e];
        loc[j] = cur + __popc(peers & lanemask_lt());
      }
      __syncwarp();
      if (in && lane == __ffs(peers) - 1) wc[e] = cur + __popc(peers);
      __syncwarp();
    }
  }
  __syncthreads();

  // Each warp's counts become exclusive offsets within the tile; then each
  // assignment's expert and tile-relative offset go to registers.
  const int g = blk / tpg;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < kTileWarps; ++w) {
      const int v = s_wcnt[w * E + e];
      s_wcnt[w * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  int ej[kWarpIters], rel[kWarpIters];
#pragma unroll
  for (int j = 0; j < kWarpIters; ++j) {
    const int a = wbeg + j * 32 + lane;
    const int e = a < wend ? s_idx[a] : -1;
    const bool in = e >= 0 && e < E;  // bad ids: the planner's status stops us below
    ej[j] = in ? e : 0;
    rel[j] = in ? wc[e] + loc[j] : 0;
  }
  prefetch_row_tables(pieces_smem, E, R, g, blk, ws, status);
  __syncthreads();  // s_wcnt is reused below

  pdl_wait();                           // the planner's tables and status
  pdl_launch_dependents();
  const int st = status != nullptr ? __ldcg(status) : 0;
  const RowTables T = load_row_tables(s_wcnt, s_pc, pieces_smem, E, R, g, blk, ws);
  if (st != 0) return;                  // uniform: one status word
  __syncthreads();
  int32_t* out = dst_pos + size_t(t0) * K;
#pragma unroll
  for (int j = 0; j < kWarpIters; ++j) {
    const int a = wbeg + j * 32 + lane;
    if (a < wend) out[a] = dest_row(T, ej[j], rel[j]);
  }
}

}  // namespace
}  // namespace mep

using namespace mep;

static int plan_check(int R, int S, int K, int E, int B) {
  if (R < 1 || R > MEP_MAX_R || S < 0 || K < 1 || K > MEP_MAX_K || E < 1 || E > MEP_MAX_E ||
      B < 0 || E % R != 0 || K > E)
    return MEP_ERR_INVALID_ARG;
  if ((long long)R * B > MEP_MAX_SLOTS) return MEP_ERR_INVALID_ARG;
  if ((long long)R * S * K > INT_MAX) return MEP_ERR_INVALID_ARG;
  return MEP_OK;
}

static int plan_nblk(int R, int S, int K) {
  const long long N = (long long)R * S;
  const int tpt = tile_tokens(K);
  return int((N + tpt - 1) / tpt);
}

extern "C" int mep_plan_workspace_bytes(int R, int S, int K, int E, int B, size_t* bytes) {
  if (bytes == nullptr) return MEP_ERR_INVALID_ARG;
  const int rc = plan_check(R, S, K, E, B);
  if (rc != MEP_OK) return rc;
  *bytes = carve(nullptr, nullptr, plan_nblk(R, S, K), R, E);
  return MEP_OK;
}

// Tile groups of the planner's prefix pass and whether k_gsum forms them:
// beyond 128 KB of tile counts, the group sums are formed by Gs CTAs in
// parallel rather than inside the one planner CTA.
static void plan_groups(int nblk, int E, int* Gs, int* tpg, int* presum) {
  const bool big = (long long)nblk * E >= MEP_PLAN_GSUM_MIN_INTS;
  tile_groups(nblk, E, big ? kPresumGroups : kMaxScanGroups, Gs, tpg);
  *presum = big && *Gs > 1 ? 1 : 0;
}

extern "C" int mep_plan_kernel_count(int R, int S, int K, int E, int B, int* count) {
  if (count == nullptr) return MEP_ERR_INVALID_ARG;
  const int rc = plan_check(R, S, K, E, B);
  if (rc != MEP_OK) return rc;
  const int nblk = plan_nblk(R, S, K);
  int Gs, tpg, presum;
  plan_groups(nblk, E, &Gs, &tpg, &presum);
  *count = (nblk > 0 ? 2 : 0) + presum + 1;  // k_hist, k_offsets; k_gsum; k_plan
  return MEP_OK;
}

static int plan_launch(const int32_t* topk_idx, int R, int S, int K, int E, int B, int fallback,
                       void* workspace, size_t workspace_bytes, int32_t* expert_counts,
                       int32_t* cu_seqlens, int32_t* slot_expert, int32_t* dst_pos,
                       int32_t* status, void* stream) {
  int rc = plan_check(R, S, K, E, B);
  if (rc != MEP_OK) return rc;
  const int N = R * S;
  const int nblk = plan_nblk(R, S, K);
  if (workspace == nullptr || expert_counts == nullptr || cu_seqlens == nullptr ||
      status == nullptr || (B > 0 && slot_expert == nullptr) ||
      (N > 0 && (topk_idx == nullptr || dst_pos == nullptr)))
    return MEP_ERR_INVALID_ARG;
  if (!aligned16(workspace) || (topk_idx && !aligned16(topk_idx))) return MEP_ERR_INVALID_ARG;
  const size_t need = carve(nullptr, nullptr, nblk, R, E);
  if (workspace_bytes < need) return MEP_ERR_INVALID_ARG;
  PlanWs ws;
  carve(&ws, static_cast<char*>(workspace), nblk, R, E);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int tpt = tile_tokens(K);

  const int hist_smem = E * int(sizeof(int));
  // k_offsets keeps its tile (K > 8), per-warp counters and per-expert
  // tables in shared memory, and the piece tables too when all of it fits
  const bool tok = K <= kTokMaxK;
  const int offs_base = ((tok ? 0 : kTileAssign) + kTileWarps * E) * int(sizeof(int));
  const int offs_pieces = 2 * (E + R) * int(sizeof(int));
  const int pieces_smem = offs_base + offs_pieces <= 220 * 1024 ? 1 : 0;
  const int offs_smem = offs_base + (pieces_smem ? offs_pieces : 0);
  const int npart = kPartInts;
  const int plan_smem = int(sizeof(int)) * (9 * (E + 1) + (E + R) + npart + 5 * (R + 1));
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(k_hist), hist_smem) ||
      set_max_dynamic_smem(tok ? reinterpret_cast<const void*>(k_offsets_tok)
                               : reinterpret_cast<const void*>(k_offsets),
                           offs_smem) ||
      set_max_dynamic_smem(reinterpret_cast<const void*>(k_plan), plan_smem))
    return MEP_ERR_CUDA;

  if (nblk > 0) k_hist<<<nblk, kTileThreads, hist_smem, st>>>(topk_idx, N, K, E, tpt, ws);
  int Gs, tpg, presum;
  plan_groups(nblk, E, &Gs, &tpg, &presum);
  if (presum) {
    const cudaError_t e =
        (E & 3) == 0
            ? launch_pdl(k_gsum<4>, dim3(Gs), dim3(kTileThreads), 0, st,
                         ws.blockhist, nblk, E, tpg, ws.groupsum)
            : launch_pdl(k_gsum<1>, dim3(Gs), dim3(kTileThreads), 0, st,
                         ws.blockhist, nblk, E, tpg, ws.groupsum);
    if (e != cudaSuccess) return MEP_ERR_CUDA;
  }
  PlanArgs pa{nblk,          R,          S,           K,      E,  B, fallback, presum, Gs, tpg,
              expert_counts, cu_seqlens, slot_expert, status, ws};
  if (launch_pdl(k_plan, dim3(1), dim3(kPlanThreads), plan_smem, st, pa) != cudaSuccess)
    return MEP_ERR_CUDA;
  if (nblk > 0) {
    cudaError_t e;
    if (tok) {
      const uintptr_t d = reinterpret_cast<uintptr_t>(dst_pos);
      const int out_vec = (K & 3) == 0 && (d & 15) == 0 ? 4 : (K & 1) == 0 && (d & 7) == 0 ? 2 : 1;
      e = launch_pdl(k_offsets_tok, dim3(nblk), dim3(kTileThreads), offs_smem, st, topk_idx, N, K,
                     E, R, tpg, pieces_smem, out_vec, ws, static_cast<const int32_t*>(status),
                     dst_pos);
    } else {
      e = launch_pdl(k_offsets, dim3(nblk), dim3(kTileThreads), offs_smem, st, topk_idx, N, K, E,
                     R, tpt, tpg, pieces_smem, ws, static_cast<const int32_t*>(status), dst_pos);
    }
    if (e != cudaSuccess) return MEP_ERR_CUDA;
  }
  return cudaGetLastError() == cudaSuccess ? MEP_OK : MEP_ERR_CUDA;
}

extern "C" int mep_plan(const int32_t* topk_idx, int R, int S, int K, int E, int B,
                        void* workspace, size_t workspace_bytes, int32_t* expert_counts,
                        int32_t* cu_seqlens, int32_t* slot_expert, int32_t* dst_pos,
                        int32_t* status, void* stream) {
  return plan_launch(topk_idx, R, S, K, E, B, 0, workspace, workspace_bytes, expert_counts,
                     cu_seqlens, slot_expert, dst_pos, status, stream);
}

extern "C" int mep_plan_remote_fallback(const int32_t* topk_idx, int R, int S, int K, int E, int B,
                                        void* workspace, size_t workspace_bytes,
                                        int32_t* expert_counts, int32_t* cu_seqlens,
                                        int32_t* slot_expert, int32_t* dst_pos, int32_t* status,
                                        void* stream) {
  return plan_launch(topk_idx, R, S, K, E, B, 1, workspace, workspace_bytes, expert_counts,
                     cu_seqlens, slot_expert, dst_pos, status, stream);
}
