/*
 * oracle.c -- plain, slow, CPU restatement of the dynamic-redundant-expert
 * hot path. TEST INFRASTRUCTURE ONLY: the tests, the package's smoke check
 * and the benchmark's CPU-baseline leg call it; the library never does.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Sources (web pages about MoonEP; cited below by the short tag in brackets):
 *   [umios]   "月之暗面开源MoonEP：面向MoE训练的专家并行通信库"
 *             sections 解决的核心问题 (problem, maxvio), 核心技术 (S*K invariant,
 *             planner, fused permute/unpermute, static shapes),
 *             内存契约与权重布局 (E/R home rows, [E+B] rows, cu_seqlens[E+B],
 *             B rule, fp32 [E+B,H,H'] grads, [R,B,H,H'] view, reduce_grad).
 *   [interestana] "Moonshot AI Open-Sources MoonEP for Expert Parallelism",
 *             paragraphs 2-3 (maxvio, invariant, redundant experts).
 *   [valhalla] "Valhalla 静态工程审阅 #004｜MoonshotAI MoonEP 源码证据驱动评测",
 *             section 2 项目背景 (every rank processes exactly S x K tokens).
 *
 * The pages give the planner only as "online planning ... near-optimal GPU
 * kernel". This oracle takes the home-first reading of it, step by step:
 *   1. validate the routing;
 *   2. T_e = number of (token, k) assignments to expert e, and L_e the
 *      ascending list of tokens routed to e;
 *   3. home(e) = e / (E/R)  ([umios] 内存契约: E/R rows per rank, in order);
 *   4. keep: each rank keeps, in expert order, at most S*K of its home
 *      experts' tokens, lowest token index first; the rest of each list is an
 *      overflow segment;
 *   5. pour: the overflow segments, concatenated in expert order, fill the
 *      deficits S*K - load_r of the under-loaded ranks in rank order; every
 *      piece (expert e, rank r, list range [lo, hi)) takes the next free
 *      redundant slot b of rank r; needing more than B slots is an error;
 *   6. groups: rank r's rows j in [0, E+B) hold c[r][j] tokens (home rows of
 *      r keep their kept count, other home rows 0, slot rows their piece);
 *      cu_seqlens[r][j] is the inclusive running sum (so the last entry is
 *      S*K, the invariant of [umios] 核心技术);
 *   7. positions: assignment (t, k) of expert e at list index i lands in
 *      rank r's static S*K buffer at row cu[r][j] - c[r][j] + offset;
 *   8. dispatch copies hidden[t] there; 9. combine sums the K rows back with
 *      fp32 fused multiply-adds in k order, rounded to bf16 (nearest-even);
 *  10. reduce_grad adds the slot gradients of each expert to its home
 *      gradient in (rank, slot) order and zeroes every consumed slot
 *      ([umios] 内存契约与权重布局, last paragraph).
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -o liboracle.so oracle.c -lm
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Oracle status values (own numbering; the tests map them by name). */
#define ORC_OK 0
#define ORC_BAD_ARG (-1)
#define ORC_BAD_ROUTING 1
#define ORC_CAPACITY 2

/* ------------------------------------------------------------------------ */
/* maxvio = max_e (T_e / T_bar) - 1 with T_bar = R*S*K / E, the count every
 * expert would get under perfect balance ([umios] 解决的核心问题;
 * [interestana] paragraph 2). Computed in double. */
double orc_maxvio(const int32_t* counts, int E, int R, int S, int K) {
  double tbar = (double)R * (double)S * (double)K / (double)E;
  double mx = 0.0;
  int e;
  if (E <= 0 || tbar <= 0.0) return 0.0;
  for (e = 0; e < E; ++e) {
    double v = (double)counts[e] / tbar;
    if (e == 0 || v > mx) mx = v;
  }
  return mx - 1.0;
}

/* Step 1: every index in [0, E), the K indices of a token distinct. */
int orc_validate(const int32_t* idx, int64_t N, int K, int E) {
  int64_t t;
  int k, k2;
  for (t = 0; t < N; ++t) {
    for (k = 0; k < K; ++k) {
      int32_t e = idx[t * K + k];
      if (e < 0 || e >= E) return ORC_BAD_ROUTING;
      for (k2 = 0; k2 < k; ++k2)
        if (idx[t * K + k2] == e) return ORC_BAD_ROUTING;
    }
  }
  return ORC_OK;
}

/* Step 2, first half: T_e. */
void orc_counts(const int32_t* idx, int64_t N, int K, int E, int32_t* counts) {
  int64_t a;
  memset(counts, 0, sizeof(int32_t) * (size_t)E);
  for (a = 0; a < N * (int64_t)K; ++a) counts[idx[a]] += 1;
}

typedef struct {
  int e;      /* expert */
  int r;      /* receiving rank */
  int b;      /* slot on that rank; -1: the expert's own row e (fallback) */
  int64_t lo; /* first list index of e covered */
  int64_t hi; /* one past the last */
} orc_piece;

/*
 * The whole plan: steps 1-7. Outputs (caller-allocated):
 *   counts[E], cu[R*(E+B)], slot_expert[R*B], slot_lo[R*B], slot_len[R*B],
 *   dst_pos[N*K]; n_pieces_out[1] (may be NULL).
 * On ORC_BAD_ROUTING / ORC_CAPACITY: slot_expert = -1, cu = 0, slot_lo =
 * slot_len = 0, dst_pos untouched; counts hold T_e for the capacity case.
 */
static int plan_impl(const int32_t* idx, int R, int S, int K, int E, int B, int fallback,
                     int32_t* counts, int32_t* cu, int32_t* slot_expert,
                     int32_t* slot_lo, int32_t* slot_len, int32_t* dst_pos,
                     int32_t* n_pieces_out) {
  const int64_t N = (int64_t)R * S;
  const int64_t A = N * K;
  const int64_t SK = (int64_t)S * K;
  const int G = E + B;
  int per, r, e, j, b, st;
  int64_t t, a;
  int64_t *load = NULL, *keep = NULL, *fill = NULL, *listpos = NULL;
  int* nslot = NULL;
  orc_piece* pieces = NULL;
  int npieces = 0;
  int64_t* c = NULL;

  if (R <= 0 || S < 0 || K <= 0 || E <= 0 || B < 0 || E % R != 0 || K > E)
    return ORC_BAD_ARG;
  per = E / R;

  for (j = 0; j < R * B; ++j) {
    slot_expert[j] = -1;
    slot_lo[j] = 0;
    slot_len[j] = 0;
  }
  for (j = 0; j < R * G; ++j) cu[j] = 0;
  if (n_pieces_out) *n_pieces_out = 0;

  /* 1. validate */
  st = orc_validate(idx, N, K, E);
  if (st != ORC_OK) {
    memset(counts, 0, sizeof(int32_t) * (size_t)E);
    return st;
  }

  /* 2. counts T_e and each assignment's index i in L_e. L_e is built by
   * walking tokens in ascending order, so the running count of e at the
   * moment (t, k) is met is exactly t's index in L_e. */
  memset(counts, 0, sizeof(int32_t) * (size_t)E);
  listpos = (int64_t*)malloc(sizeof(int64_t) * (size_t)(A > 0 ? A : 1));
  fill = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  for (t = 0; t < N; ++t) {
    int k;
    for (k = 0; k < K; ++k) {
      e = idx[t * K + k];
      listpos[t * K + k] = fill[e];
      fill[e] += 1;
    }
  }
  for (e = 0; e < E; ++e) counts[e] = (int32_t)fill[e];

  /* 3. home loads */
  load = (int64_t*)calloc((size_t)R, sizeof(int64_t));
  for (e = 0; e < E; ++e) load[e / per] += counts[e];

  /* 4. keep, home-first, in expert order within each rank */
  keep = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  for (r = 0; r < R; ++r) {
    int64_t budget = SK;
    for (e = r * per; e < (r + 1) * per; ++e) {
      int64_t k_e = counts[e] < budget ? counts[e] : budget;
      keep[e] = k_e;
      budget -= k_e;
    }
  }

  /* 5. pour the overflow (expert order) into deficits (rank order) */
  pieces = (orc_piece*)malloc(sizeof(orc_piece) * (size_t)(E + R + 1));
  nslot = (int*)calloc((size_t)R, sizeof(int));
  {
    int oe = 0;             /* current overflow expert */
    int64_t opos = 0;       /* next list index of oe still to place */
    /* advance to the first expert that overflows */
    while (oe < E && keep[oe] >= counts[oe]) ++oe;
    if (oe < E) opos = keep[oe];
    for (r = 0; r < R; ++r) {
      int64_t need = SK - load[r];
      while (need > 0) {
        int64_t avail, take;
        if (oe >= E) { /* cannot happen when the counts sum to R*S*K */
          st = ORC_BAD_ROUTING;
          goto fail;
        }
        avail = counts[oe] - opos;
        take = avail < need ? avail : need;
        b = nslot[r];
        if (b >= B && fallback) {
          b = -1; /* no slot left: rank r reads expert oe's home weights (row oe) */
        } else if (b >= B) {
          st = ORC_CAPACITY;
          goto fail;
        }
        pieces[npieces].e = oe;
        pieces[npieces].r = r;
        pieces[npieces].b = b;
        pieces[npieces].lo = opos;
        pieces[npieces].hi = opos + take;
        ++npieces;
        if (b >= 0) nslot[r] = b + 1;
        opos += take;
        need -= take;
        if (opos == counts[oe]) {
          ++oe;
          while (oe < E && keep[oe] >= counts[oe]) ++oe;
          if (oe < E) opos = keep[oe];
        }
      }
    }
  }

  /* 6. group sizes and inclusive cumulative ends */
  c = (int64_t*)calloc((size_t)R * (size_t)G, sizeof(int64_t));
  for (e = 0; e < E; ++e) c[(int64_t)(e / per) * G + e] = keep[e];
  for (j = 0; j < npieces; ++j) {
    if (pieces[j].b < 0) { /* fallback piece: row e of the receiving rank */
      c[(int64_t)pieces[j].r * G + pieces[j].e] = pieces[j].hi - pieces[j].lo;
      continue;
    }
    c[(int64_t)pieces[j].r * G + E + pieces[j].b] = pieces[j].hi - pieces[j].lo;
    slot_expert[pieces[j].r * B + pieces[j].b] = pieces[j].e;
    slot_lo[pieces[j].r * B + pieces[j].b] = (int32_t)pieces[j].lo;
    slot_len[pieces[j].r * B + pieces[j].b] = (int32_t)(pieces[j].hi - pieces[j].lo);
  }
  for (r = 0; r < R; ++r) {
    int64_t run = 0;
    for (j = 0; j < G; ++j) {
      run += c[(int64_t)r * G + j];
      cu[(int64_t)r * G + j] = (int32_t)run;
    }
  }

  /* 7. destination rows */
  for (a = 0; a < A; ++a) {
    int64_t i = listpos[a];
    int64_t off, start;
    e = idx[a];
    if (i < keep[e]) {
      r = e / per;
      j = e;
      off = i;
    } else {
      int p, found = -1;
      for (p = 0; p < npieces; ++p)
        if (pieces[p].e == e && pieces[p].lo <= i && i < pieces[p].hi) found = p;
      /* found >= 0 always: the pieces of e cover [keep_e, T_e) */
      r = pieces[found].r;
      j = pieces[found].b >= 0 ? E + pieces[found].b : e;
      off = i - pieces[found].lo;
    }
    start = cu[(int64_t)r * G + j] - c[(int64_t)r * G + j];
    dst_pos[a] = (int32_t)((int64_t)r * SK + start + off);
  }
  if (n_pieces_out) *n_pieces_out = npieces;
  st = ORC_OK;
  goto done;

fail:
  for (j = 0; j < R * B; ++j) {
    slot_expert[j] = -1;
    slot_lo[j] = 0;
    slot_len[j] = 0;
  }
  for (j = 0; j < R * G; ++j) cu[j] = 0;
  npieces = 0;
done:
  free(c);
  free(nslot);
  free(pieces);
  free(keep);
  free(load);
  free(fill);
  free(listpos);
  return st;
}

/* Training reading: more than B pieces on a rank is a capacity error. */
int orc_plan(const int32_t* idx, int R, int S, int K, int E, int B,
             int32_t* counts, int32_t* cu, int32_t* slot_expert,
             int32_t* slot_lo, int32_t* slot_len, int32_t* dst_pos,
             int32_t* n_pieces_out) {
  return plan_impl(idx, R, S, K, E, B, 0, counts, cu, slot_expert, slot_lo, slot_len, dst_pos,
                   n_pieces_out);
}

/* Inference reading ([umios] 内存契约与权重布局: inference may use B = 3-4;
 * when more remote experts are needed, their home rank's weights are read
 * through the symmetric mapping): a rank's pieces beyond its B slots are not
 * an error; such a piece of expert e takes row e (a [0, E) row, served by the
 * home weights) of the receiving rank. The first B pieces of a rank, in pour
 * order, keep slots 0..B-1. */
int orc_plan_fallback(const int32_t* idx, int R, int S, int K, int E, int B,
                      int32_t* counts, int32_t* cu, int32_t* slot_expert,
                      int32_t* slot_lo, int32_t* slot_len, int32_t* dst_pos,
                      int32_t* n_pieces_out) {
  return plan_impl(idx, R, S, K, E, B, 1, counts, cu, slot_expert, slot_lo, slot_len, dst_pos,
                   n_pieces_out);
}

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32 from the IEEE-754 binary16-brain layout: a bf16 value is the
 * top 16 bits of a binary32. Narrowing rounds to nearest, ties to even. */
static float orc_bf16_to_f32(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

uint16_t orc_f32_to_bf16(float f) {
  uint32_t u, low, keep_hi;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0)
    return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays NaN (quiet) */
  keep_hi = u >> 16;
  low = u & 0xFFFFu;
  if (low > 0x8000u || (low == 0x8000u && (keep_hi & 1u))) keep_hi += 1u;
  return (uint16_t)keep_hi;
}

/* Step 8, dispatch ([umios] 核心技术, fused permute): buf[dst_pos[t,k]] = hidden[t]. */
void orc_dispatch(const uint16_t* hidden, const int32_t* dst_pos, int64_t N, int K,
                  int64_t H, uint16_t* buf) {
  int64_t t, h;
  int k;
  for (t = 0; t < N; ++t)
    for (k = 0; k < K; ++k) {
      int64_t row = dst_pos[t * K + k];
      for (h = 0; h < H; ++h) buf[row * H + h] = hidden[t * H + h];
    }
}

/* Step 9, combine ([umios] 核心技术, fused unpermute), for a list of tokens:
 * out[t,h] = bf16( sum_k w[t,k] * y[dst_pos[t,k], h] ), accumulated in fp32
 * from 0 with fmaf in k order. tokens == NULL means all N tokens in order
 * and out is [N, H]; otherwise out is [n_tok, H]. */
void orc_combine(const uint16_t* y, const float* w, const int32_t* dst_pos,
                 const int64_t* tokens, int64_t n_tok, int K, int64_t H,
                 uint16_t* out) {
  int64_t i, h;
  int k;
  for (i = 0; i < n_tok; ++i) {
    int64_t t = tokens ? tokens[i] : i;
    for (h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (k = 0; k < K; ++k) {
        int64_t row = dst_pos[t * K + k];
        acc = fmaf(w[t * K + k], orc_bf16_to_f32(y[row * H + h]), acc);
      }
      out[i * H + h] = orc_f32_to_bf16(acc);
    }
  }
}

/* Step 10, reduce_grad ([umios] 内存契约与权重布局): for every expert e and
 * element, home[e] += slot[r][b] over the slots with slot_expert[r][b] == e,
 * in ascending (r, b) order; then every consumed slot (slot_expert != -1) is
 * zeroed. home is [E, HHp], slot is [R*B, HHp], both fp32.
 * Returns ORC_BAD_ROUTING (and changes nothing) if an entry of slot_expert
 * is neither -1 nor in [0, E). */
int orc_reduce_grad(const int32_t* slot_expert, int E, int R, int B, int64_t HHp,
                    float* home, float* slot) {
  int e, s;
  int64_t i;
  for (s = 0; s < R * B; ++s)
    if (slot_expert[s] < -1 || slot_expert[s] >= E) return ORC_BAD_ROUTING;
  for (e = 0; e < E; ++e) {
    float* hrow = home + (int64_t)e * HHp;
    for (s = 0; s < R * B; ++s) {
      const float* srow;
      if (slot_expert[s] != e) continue;
      srow = slot + (int64_t)s * HHp;
      for (i = 0; i < HHp; ++i) hrow[i] = hrow[i] + srow[i];
    }
  }
  for (s = 0; s < R * B; ++s)
    if (slot_expert[s] != -1) memset(slot + (int64_t)s * HHp, 0, sizeof(float) * (size_t)HHp);
  return ORC_OK;
}

/* Array form of the bf16 narrowing above (for pinning it in the tests). */
void orc_f32_to_bf16_array(const float* x, int64_t n, uint16_t* out) {
  int64_t i;
  for (i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(x[i]);
}

/* Replica weight prefetch ([umios] 核心技术: the weights of the planned
 * redundant experts are fetched before expert compute; 内存契约与权重布局:
 * rows [E, E+B) of each rank's [E+B, H, H'] weight tensor are local prefetch
 * slots). For every slot with slot_expert[r][b] = e != -1, slot[r][b] is a
 * byte copy of home[e]; unused slots are not touched. home is [E, nbytes],
 * slot is [R*B, nbytes]. Returns ORC_BAD_ROUTING (and copies nothing) if an
 * entry is neither -1 nor in [0, E). */
int orc_prefetch(const int32_t* slot_expert, int E, int R, int B, int64_t nbytes,
                 const uint8_t* home, uint8_t* slot) {
  int s;
  for (s = 0; s < R * B; ++s)
    if (slot_expert[s] < -1 || slot_expert[s] >= E) return ORC_BAD_ROUTING;
  for (s = 0; s < R * B; ++s)
    if (slot_expert[s] >= 0)
      memcpy(slot + (int64_t)s * nbytes, home + (int64_t)slot_expert[s] * nbytes, (size_t)nbytes);
  return ORC_OK;
}

/* Backward of the fused permute (dispatch): dispatch copies hidden[t] to the
 * K rows dst_pos[t, k], so dhidden[t, h] = sum_k dbuf[dst_pos[t, k], h]. The
 * pages give no backward arithmetic ([umios] 核心技术 names the fused
 * permute/unpermute only); this library's reading mirrors combine: fp32 from
 * 0, one add per k in k order, round to nearest-even bf16. */
void orc_dispatch_backward(const uint16_t* dbuf, const int32_t* dst_pos, int64_t N, int K,
                           int64_t H, uint16_t* dhidden) {
  int64_t t, h;
  int k;
  for (t = 0; t < N; ++t)
    for (h = 0; h < H; ++h) {
      float acc = 0.0f;
      for (k = 0; k < K; ++k) acc = acc + orc_bf16_to_f32(dbuf[(int64_t)dst_pos[t * K + k] * H + h]);
      dhidden[t * H + h] = orc_f32_to_bf16(acc);
    }
}

/* Backward of the weighted unpermute (combine): out[t] = sum_k w[t,k] *
 * y[dst_pos[t,k]], so
 *   dy[dst_pos[t,k], h] = w[t,k] * dout[t,h]   (an fp32 product, then nearest-
 *                                               even bf16, this library's reading)
 *   dw[t,k] = sum_h dout[t,h] * y[dst_pos[t,k], h]
 * dw is the plain definition, accumulated in double: every product of two
 * bf16 values is exact in double, so the result is the dot product to
 * within double rounding. */
void orc_combine_backward(const uint16_t* dout, const uint16_t* y, const float* w,
                          const int32_t* dst_pos, int64_t N, int K, int64_t H, uint16_t* dy,
                          double* dw) {
  int64_t t, h;
  int k;
  for (t = 0; t < N; ++t)
    for (k = 0; k < K; ++k) {
      const int64_t row = dst_pos[t * K + k];
      const float wk = w[t * K + k];
      double acc = 0.0;
      for (h = 0; h < H; ++h) {
        const float d = orc_bf16_to_f32(dout[t * H + h]);
        const float p = wk * d;
        dy[row * H + h] = orc_f32_to_bf16(p);
        acc += (double)d * (double)orc_bf16_to_f32(y[row * H + h]);
      }
      dw[t * K + k] = acc;
    }
}

/* Grouped expert product over the static buffer ([umios] 内存契约与权重布局:
 * one grouped GEMM per projection consumes a single [E+B, H, H'] weight
 * tensor, rows [0, E) the experts' own weights and rows [E, E+B) the rank's
 * prefetch slots, and cu_seqlens[E+B] says which of its rows are active).
 * Rank r's buffer rows [r*SK, (r+1)*SK) hold the groups j = 0..E+B-1 back to
 * back: group j is rows [cu[r][j-1], cu[r][j]) of that block (cu[r][-1] = 0).
 * Its weight W_j is w_home[j] for j < E and w_slot[r][j-E] for j >= E, and
 *   y[row, n] = sum_h x[row, h] * W_j[h, n],
 * summed in h order in double (every bf16 x bf16 product is exact there) and
 * returned in double: the caller picks the rounding. rows == NULL means all
 * R*SK rows in order, else the n_rows listed; y is [n_rows, Hp].
 * Returns ORC_BAD_ARG, writing nothing, if a cu row is not nondecreasing
 * from >= 0 to SK or a listed row is out of range. */
int orc_grouped_gemm(const uint16_t* x, const int32_t* cu, const uint16_t* w_home,
                     const uint16_t* w_slot, int R, int64_t SK, int E, int B, int64_t H,
                     int64_t Hp, const int64_t* rows, int64_t n_rows, double* y) {
  const int G = E + B;
  int r, j;
  int64_t q, h, n;
  for (r = 0; r < R; ++r) {
    int32_t prev = 0;
    for (j = 0; j < G; ++j) {
      if (cu[(int64_t)r * G + j] < prev) return ORC_BAD_ARG;
      prev = cu[(int64_t)r * G + j];
    }
    if (prev != SK) return ORC_BAD_ARG;
  }
  for (q = 0; q < n_rows; ++q) {
    const int64_t row = rows ? rows[q] : q;
    if (row < 0 || row >= (int64_t)R * SK) return ORC_BAD_ARG;
  }
  for (q = 0; q < n_rows; ++q) {
    const int64_t row = rows ? rows[q] : q;
    const int64_t i = row % SK;
    const uint16_t* W;
    double* out = y + q * Hp;
    r = (int)(row / SK);
    j = 0; /* the group holding local row i: the first j whose end exceeds i */
    while (cu[(int64_t)r * G + j] <= i) ++j;
    W = j < E ? w_home + (int64_t)j * H * Hp : w_slot + ((int64_t)r * B + (j - E)) * H * Hp;
    for (n = 0; n < Hp; ++n) out[n] = 0.0;
    for (h = 0; h < H; ++h) {
      const double xv = (double)orc_bf16_to_f32(x[row * H + h]);
      const uint16_t* wrow = W + h * Hp;
      for (n = 0; n < Hp; ++n) out[n] += xv * (double)orc_bf16_to_f32(wrow[n]);
    }
  }
  return ORC_OK;
}
