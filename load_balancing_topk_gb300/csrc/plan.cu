// plan.cu -- routing histogram, online planner and destination rows (mep_plan).
//
// Source: "月之暗面开源MoonEP：面向MoE训练的专家并行通信库", sections 核心技术
// (every rank receives exactly S*K tokens; redundant experts are planned
// online from the current router output, on the GPU, with no host sync) and
// 内存契约与权重布局 (E/R home rows per rank, B slot rows, cu_seqlens[E+B]).
// maxvio and T_e: same page, section 解决的核心问题.
//
// Three launches, all asynchronous on the caller's stream:
//   k_hist     grid over tiles of assignments: per-tile expert counts
//              (warp-aggregated with __match_any_sync) and routing checks.
//   k_plan     one CTA: tile counts -> T_e and per-tile exclusive prefixes,
//              home-first keep, overflow pour into deficits, slot table,
//              cu_seqlens, and the per-expert row bases used by k_offsets.
//   k_offsets  grid over the same tiles: each assignment's index in its
//              expert's token-ordered list (tile prefix + warp prefix + rank
//              inside the warp), mapped to its destination row.
// The planner's rule is home-first: a rank keeps, in expert order, at most
// S*K of its home experts' tokens; the overflow segments, in expert order,
// fill the under-loaded ranks' deficits in rank order, one slot per piece.

#include <climits>

#include "mep_common.cuh"

namespace mep {
namespace {

constexpr int kTileThreads = 256;            // k_hist / k_offsets block size (8 warps)
constexpr int kTileWarps = kTileThreads / 32;
constexpr int kTileAssign = 4096;            // assignments per tile (upper bound)
constexpr int kWarpIters = kTileAssign / (32 * kTileWarps);  // 16 iterations per warp
constexpr int kPlanThreads = 1024;           // k_plan block size

// tokens per tile: as many as fit 4096 assignments, a multiple of 4 so that
// every tile starts on a 16-byte boundary of topk_idx.
inline int tile_tokens(int K) { return (kTileAssign / K) & ~3; }

struct PlanWs {
  int* blockhist;    // [nblk, E] tile counts, rewritten as tile exclusive prefixes
  int* blockerr;     // [nblk]
  int* keep;         // [E] tokens kept on the home row
  int* home_base;    // [E] global row of the home row's first token
  int* pc_begin;     // [E] first piece of the expert (pieces are grouped by expert)
  int* pc_count;     // [E]
  int* piece_lo;     // [E+R] first list index covered by the piece
  int* piece_base;   // [E+R] global row of the piece's first token
  int* piece_expert; // [E+R]
  int* slot_lo;      // [R*B]
  int* slot_len;     // [R*B]
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

size_t carve(PlanWs* ws, char* base, int nblk, int R, int E, int B) {
  size_t off = 0;
  auto take = [&](int** p, size_t n) {
    if (ws) *p = reinterpret_cast<int*>(base + off);
    off += align256(n * sizeof(int));
  };
  PlanWs dummy;
  PlanWs* w = ws ? ws : &dummy;
  take(&w->blockhist, size_t(nblk) * E);
  take(&w->blockerr, size_t(nblk > 0 ? nblk : 1));
  take(&w->keep, E);
  take(&w->home_base, E);
  take(&w->pc_begin, E);
  take(&w->pc_count, E);
  take(&w->piece_lo, size_t(E) + R);
  take(&w->piece_base, size_t(E) + R);
  take(&w->piece_expert, size_t(E) + R);
  take(&w->slot_lo, size_t(R) * (B > 0 ? B : 1));
  take(&w->slot_len, size_t(R) * (B > 0 ? B : 1));
  return off;
}

// Stage one tile of topk_idx into shared memory (16-byte loads; the tile
// start is 16-byte aligned, the tail is loaded element by element).
__device__ __forceinline__ void stage_tile(const int32_t* __restrict__ g, int na, int* s_idx) {
  const int nv = na >> 2;
  const int4* g4 = reinterpret_cast<const int4*>(g);
  int4* s4 = reinterpret_cast<int4*>(s_idx);
  for (int i = threadIdx.x; i < nv; i += blockDim.x) s4[i] = __ldg(g4 + i);
  for (int i = (nv << 2) + threadIdx.x; i < na; i += blockDim.x) s_idx[i] = __ldg(g + i);
}

// ---------------------------------------------------------------------------
// k_hist: tile counts and routing checks.
__global__ void __launch_bounds__(kTileThreads)
    k_hist(const int32_t* __restrict__ topk_idx, int N, int K, int E, int tok_per_tile,
           PlanWs ws) {
  extern __shared__ int smem[];
  int* s_idx = smem;                 // [kTileAssign]
  int* s_cnt = smem + kTileAssign;   // [E]
  __shared__ int s_err;
  const int blk = blockIdx.x;
  const int t0 = blk * tok_per_tile;
  const int ntok = min(tok_per_tile, N - t0);
  const int na = ntok * K;
  if (threadIdx.x == 0) s_err = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_cnt[e] = 0;
  stage_tile(topk_idx + size_t(t0) * K, na, s_idx);
  __syncthreads();

  const int lane = threadIdx.x & 31;
  bool bad = false;
  for (int a0 = 0; a0 < na; a0 += blockDim.x) {
    const int a = a0 + threadIdx.x;
    const bool in = a < na;
    int e = in ? s_idx[a] : -1;
    bool ok = in && e >= 0 && e < E;
    if (ok) {
      const int t = a / K, k = a - t * K;
      for (int k2 = 0; k2 < k; ++k2)
        if (s_idx[t * K + k2] == e) ok = false;
    }
    if (in && !ok) bad = true;
    const unsigned m = __ballot_sync(MEP_FULL_MASK, ok);
    if (ok) {
      const unsigned peers = __match_any_sync(m, e);
      if (lane == __ffs(peers) - 1) atomicAdd(&s_cnt[e], __popc(peers));
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
  int32_t* counts;       // [E]
  int32_t* cu;           // [R, E+B]
  int32_t* slot_expert;  // [R, B]
  int32_t* status;
  PlanWs ws;
};

__device__ void plan_fail(const PlanArgs& a, int code, bool zero_counts) {
  const int G = a.E + a.B;
  for (int i = threadIdx.x; i < a.R * G; i += blockDim.x) a.cu[i] = 0;
  for (int i = threadIdx.x; i < a.R * a.B; i += blockDim.x) a.slot_expert[i] = -1;
  if (zero_counts)
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) a.counts[e] = 0;
  if (threadIdx.x == 0) *a.status = code;
}

__global__ void __launch_bounds__(kPlanThreads) k_plan(PlanArgs a) {
  extern __shared__ int smem[];
  const int E = a.E, R = a.R, B = a.B, nblk = a.nblk;
  const int per = E / R;
  const int SK = a.S * a.K;
  const int G = E + B;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
  const int EP = E + 1, RP = R + 1;
  const int npart = max(nthr, E);
  int* sT = smem;                // [E+1]
  int* sPre = sT + EP;           // [E+1]
  int* sKeep = sPre + EP;        // [E]
  int* sOv = sKeep + E;          // [E+1]
  int* sOst = sOv + EP;          // [E+1]
  int* sOlist = sOst + EP;       // [E]
  int* sPcBeg = sOlist + E;      // [E]
  int* sPcCnt = sPcBeg + E;      // [E]
  int* sPart = sPcCnt + E;       // [max(nthr, E)]
  int* sLoad = sPart + npart;    // [R+1]
  int* sDef = sLoad + RP;        // [R+1]
  int* sDst = sDef + RP;         // [R+1]
  int* sNp = sDst + RP;          // [R+1]
  int* sPex = sNp + RP;          // [R+1]
  __shared__ int s_warp[33];
  __shared__ int s_errblk, s_cap, s_nov;

  // 0. routing errors found by k_hist (lowest tile wins)
  if (tid == 0) {
    s_errblk = INT_MAX;
    s_cap = 0;
  }
  __syncthreads();
  for (int b = tid; b < nblk; b += nthr)
    if (a.ws.blockerr[b] != 0) atomicMin(&s_errblk, b);
  __syncthreads();
  if (s_errblk != INT_MAX) {
    plan_fail(a, a.ws.blockerr[s_errblk], true);
    return;
  }

  // 1. T_e and exclusive prefixes over tiles, in place. Thread (g, e) owns
  //    tiles [g*nblk/Gs, (g+1)*nblk/Gs) of expert e.
  const int Gs = (E >= nthr) ? 1 : nthr / E;
  for (int x = tid; x < Gs * E; x += nthr) {
    const int g = x / E, e = x - g * E;
    const int b0 = int((long long)g * nblk / Gs), b1 = int((long long)(g + 1) * nblk / Gs);
    const int* h = a.ws.blockhist + e;
    int s = 0;
#pragma unroll 8
    for (int b = b0; b < b1; ++b) s += h[size_t(b) * E];
    sPart[x] = s;
  }
  __syncthreads();
  for (int e = tid; e < E; e += nthr) {
    int run = 0;
    for (int g = 0; g < Gs; ++g) {
      const int v = sPart[g * E + e];
      sPart[g * E + e] = run;
      run += v;
    }
    sT[e] = run;
    a.counts[e] = run;
  }
  __syncthreads();
  for (int x = tid; x < Gs * E; x += nthr) {
    const int g = x / E, e = x - g * E;
    const int b0 = int((long long)g * nblk / Gs), b1 = int((long long)(g + 1) * nblk / Gs);
    int* h = a.ws.blockhist + e;
    int run = sPart[x];
#pragma unroll 8
    for (int b = b0; b < b1; ++b) {
      const int v = h[size_t(b) * E];
      h[size_t(b) * E] = run;
      run += v;
    }
  }

  // 2. home loads and home-first keep
  block_excl_scan(sT, sPre, E, s_warp, true);
  for (int e = tid; e < E; e += nthr) {
    const int r = e / per;
    const int before = sPre[e] - sPre[r * per];   // earlier home experts of r
    const int kp = max(0, min(sT[e], SK - before));
    sKeep[e] = kp;
    sOv[e] = sT[e] - kp;
    a.ws.keep[e] = kp;
  }
  for (int r = tid; r < R; r += nthr) {
    const int load = sPre[(r + 1) * per] - sPre[r * per];
    sLoad[r] = load;
    sDef[r] = max(0, SK - load);
  }
  __syncthreads();

  // 3. overflow segments (expert order) and deficits (rank order) on one line
  block_excl_scan(sOv, sOst, E, s_warp, true);
  for (int e = tid; e < E; e += nthr) sPre[e] = sOv[e] > 0 ? 1 : 0;
  __syncthreads();
  block_excl_scan(sPre, sPre, E, s_warp, true);
  for (int e = tid; e < E; e += nthr)
    if (sOv[e] > 0) sOlist[sPre[e]] = e;
  if (tid == 0) s_nov = sPre[E];
  block_excl_scan(sDef, sDst, R, s_warp, true);

  // 4. pieces of each under-loaded rank: the overflow segments that meet
  //    [Dst_r, Dst_r + d_r), in expert order, one slot each.
  const int nov = s_nov;
  for (int r = tid; r < R; r += nthr) {
    int np = 0;
    const int d = sDef[r];
    if (d > 0) {
      const int lo = sDst[r], hi = lo + d;
      int q0 = 0, q1 = nov;  // first q whose segment ends after lo
      while (q0 < q1) {
        const int m = (q0 + q1) >> 1;
        const int e = sOlist[m];
        if (sOst[e] + sOv[e] > lo) q1 = m; else q0 = m + 1;
      }
      for (int q = q0; q < nov; ++q) {
        const int e = sOlist[q];
        const int os = sOst[e], oe = os + sOv[e];
        const int s = max(os, lo), en = min(oe, hi);
        if (s >= en) break;
        if (np >= B) {
          s_cap = 1;
          break;
        }
        a.slot_expert[r * B + np] = e;
        a.ws.slot_lo[r * B + np] = sKeep[e] + (s - os);
        a.ws.slot_len[r * B + np] = en - s;
        ++np;
        if (en < oe) break;
      }
    }
    for (int b = np; b < B; ++b) {
      a.slot_expert[r * B + b] = -1;
      a.ws.slot_lo[r * B + b] = 0;
      a.ws.slot_len[r * B + b] = 0;
    }
    sNp[r] = np;
  }
  __syncthreads();
  if (s_cap) {
    plan_fail(a, MEP_ERR_CAPACITY, false);
    return;
  }

  // 5. global piece numbering: rank order (= expert order along the line)
  block_excl_scan(sNp, sPex, R, s_warp, true);
  for (int e = tid; e < E; e += nthr) {
    sPcBeg[e] = INT_MAX;
    sPcCnt[e] = 0;
  }
  __syncthreads();
  for (int r = tid; r < R; r += nthr) {
    for (int b = 0; b < sNp[r]; ++b) {
      const int g = sPex[r] + b;
      if (g >= E + R) break;  // cannot happen: pieces <= overflow experts + deficit ranks - 1
      const int e = a.slot_expert[r * B + b];
      a.ws.piece_lo[g] = a.ws.slot_lo[r * B + b];
      a.ws.piece_expert[g] = e;
      atomicMin(&sPcBeg[e], g);
      atomicAdd(&sPcCnt[e], 1);
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += nthr) {
    a.ws.pc_begin[e] = sPcCnt[e] ? sPcBeg[e] : 0;
    a.ws.pc_count[e] = sPcCnt[e];
  }

  // 6. cu_seqlens, one warp per rank; also the global first row of every
  //    home row and piece.
  for (int r = warp; r < R; r += nwarps) {
    int carry = 0;
    const int np = sNp[r];
    for (int j0 = 0; j0 < G; j0 += 32) {
      const int j = j0 + lane;
      int c = 0;
      if (j < E) c = (j / per == r) ? sKeep[j] : 0;
      else if (j < G) c = a.ws.slot_len[r * B + (j - E)];
      const int incl = warp_incl_scan(c);
      if (j < G) {
        a.cu[size_t(r) * G + j] = carry + incl;
        const int start = r * SK + carry + incl - c;
        if (j < E) {
          if (j / per == r) a.ws.home_base[j] = start;
        } else if (j - E < np) {
          a.ws.piece_base[sPex[r] + (j - E)] = start;
        }
      }
      carry += __shfl_sync(MEP_FULL_MASK, incl, 31);
    }
  }
  if (tid == 0) *a.status = MEP_OK;
}

// ---------------------------------------------------------------------------
// k_offsets: destination rows.
__global__ void __launch_bounds__(kTileThreads)
    k_offsets(const int32_t* __restrict__ topk_idx, int N, int K, int E, int tok_per_tile,
              PlanWs ws, const int32_t* __restrict__ status, int32_t* __restrict__ dst_pos) {
  if (read_status(status) != 0) return;
  extern __shared__ int smem[];
  int* s_idx = smem;                    // [kTileAssign]
  int* s_wcnt = smem + kTileAssign;     // [kTileWarps, E]
  const int blk = blockIdx.x;
  const int t0 = blk * tok_per_tile;
  const int ntok = min(tok_per_tile, N - t0);
  const int na = ntok * K;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kTileWarps * E; i += blockDim.x) s_wcnt[i] = 0;
  stage_tile(topk_idx + size_t(t0) * K, na, s_idx);
  __syncthreads();

  // Warp w owns the contiguous assignment range [wbeg, wend) of the tile,
  // so (warp, iteration, lane) order is the flattened (token, k) order.
  const int chunk = (((na + kTileWarps - 1) / kTileWarps) + 31) & ~31;
  const int wbeg = min(na, warp * chunk), wend = min(na, wbeg + chunk);
  int* wc = s_wcnt + warp * E;
  int loc[kWarpIters];
#pragma unroll
  for (int j = 0; j < kWarpIters; ++j) {
    loc[j] = 0;
    const int a = wbeg + j * 32 + lane;
    if (wbeg + j * 32 < wend) {          // warp-uniform
      const bool in = a < wend;
      const int e = in ? s_idx[a] : -1;
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
  // per expert: exclusive prefix over warps, on top of the tile's prefix
  const int* tile_pre = ws.blockhist + size_t(blk) * E;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = tile_pre[e];
#pragma unroll
    for (int w = 0; w < kTileWarps; ++w) {
      const int v = s_wcnt[w * E + e];
      s_wcnt[w * E + e] = run;
      run += v;
    }
  }
  __syncthreads();
  int32_t* out = dst_pos + size_t(t0) * K;
#pragma unroll
  for (int j = 0; j < kWarpIters; ++j) {
    const int a = wbeg + j * 32 + lane;
    if (a < wend) {
      const int e = s_idx[a];
      const int i = wc[e] + loc[j];     // index of the token in expert e's list
      const int kp = __ldg(ws.keep + e);
      int row;
      if (i < kp) {
        row = __ldg(ws.home_base + e) + i;
      } else {
        const int p0 = __ldg(ws.pc_begin + e), pn = __ldg(ws.pc_count + e);
        int p = p0;
        for (int q = p0 + 1; q < p0 + pn; ++q)
          if (__ldg(ws.piece_lo + q) <= i) p = q;
        row = __ldg(ws.piece_base + p) + (i - __ldg(ws.piece_lo + p));
      }
      out[a] = row;
    }
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
  *bytes = carve(nullptr, nullptr, plan_nblk(R, S, K), R, E, B);
  return MEP_OK;
}

extern "C" int mep_plan(const int32_t* topk_idx, int R, int S, int K, int E, int B,
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
  const size_t need = carve(nullptr, nullptr, nblk, R, E, B);
  if (workspace_bytes < need) return MEP_ERR_INVALID_ARG;
  PlanWs ws;
  carve(&ws, static_cast<char*>(workspace), nblk, R, E, B);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int tpt = tile_tokens(K);

  const int hist_smem = (kTileAssign + E) * int(sizeof(int));
  const int offs_smem = (kTileAssign + kTileWarps * E) * int(sizeof(int));
  const int npart = kPlanThreads > E ? kPlanThreads : E;
  const int plan_smem = int(sizeof(int)) * (9 * (E + 1) + npart + 5 * (R + 1));
  if (set_max_dynamic_smem(reinterpret_cast<const void*>(k_hist), hist_smem) ||
      set_max_dynamic_smem(reinterpret_cast<const void*>(k_offsets), offs_smem) ||
      set_max_dynamic_smem(reinterpret_cast<const void*>(k_plan), plan_smem))
    return MEP_ERR_CUDA;

  if (nblk > 0) k_hist<<<nblk, kTileThreads, hist_smem, st>>>(topk_idx, N, K, E, tpt, ws);
  PlanArgs pa{nblk, R, S, K, E, B, expert_counts, cu_seqlens, slot_expert, status, ws};
  k_plan<<<1, kPlanThreads, plan_smem, st>>>(pa);
  if (nblk > 0)
    k_offsets<<<nblk, kTileThreads, offs_smem, st>>>(topk_idx, N, K, E, tpt, ws, status, dst_pos);
  return cudaGetLastError() == cudaSuccess ? MEP_OK : MEP_ERR_CUDA;
}
