/*
 * mep.h -- C ABI of the GB300 (sm_103a) dynamic-redundant-expert hot path.
 *
 * Four steps of one MoE layer, for R "ranks" that are partitions of one
 * GPU's memory:
 *   mep_plan        routing histogram + online planner + destination rows
 *   mep_dispatch    fused permute into the static [R, S*K, H] buffer
 *   mep_combine     fused weighted unpermute back to [R*S, H]
 *   mep_reduce_grad redundant-slot gradients folded into home gradients
 *   mep_prefetch    redundant experts' weights copied into their slots
 *   mep_dispatch_backward / mep_combine_backward   the two permutes' gradients
 *   mep_grouped_gemm  the grouped expert product that consumes the buffer
 *   mep_plan_remote_fallback / mep_plan_static_scratch   planner variants
 *   mep_wait_selftest  the kernels' bounded wait, run on a barrier that never completes
 *
 * Sources (web pages about MoonEP, cited by title and section):
 *   "月之暗面开源MoonEP：面向MoE训练的专家并行通信库" -- sections
 *     解决的核心问题 (maxvio), 核心技术 (every rank receives exactly S*K
 *     tokens; redundant experts planned online from the router output;
 *     fused permute/unpermute into preset expert-grouped positions of a fixed
 *     S*K buffer; static shapes remove the per-layer host sync) and
 *     内存契约与权重布局 (rows [0,E) hold E/R home experts per rank, rows
 *     [E,E+B) are B prefetch slots; cu_seqlens[E+B]; fp32 gradients with the
 *     slot rows in a separate reduce buffer viewed as [R,B,H,H']; reduce_grad
 *     accumulates the slots into the home gradient and zeroes consumed slots).
 *   "Moonshot AI Open-Sources MoonEP for Expert Parallelism" -- paragraphs
 *     2 and 3 (maxvio; the S*K invariant; redundant-expert gradients are
 *     reduced back to their home ranks).
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     allocates nothing, keeps no state between calls and never synchronises
 *     the host. Work is enqueued on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream) and runs asynchronously.
 *   - Tensors are dense, row-major, and must start on a 16-byte boundary.
 *   - bf16 data is passed as 16-bit bit patterns (mep_bf16).
 *   - The int return value reports only the checks made on the host before
 *     anything is enqueued (MEP_ERR_INVALID_ARG) and launch failures
 *     (MEP_ERR_CUDA). Errors that depend on device data are written to the
 *     device word `status` (int32, written by mep_plan, read by the others);
 *     a step that finds *status != 0 on entry does nothing. No kernel traps
 *     or asserts.
 */
#ifndef MEP_H
#define MEP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MEP_API __attribute__((visibility("default")))
#else
#define MEP_API
#endif

typedef uint16_t mep_bf16;

/* Return / status codes. */
#define MEP_OK 0
#define MEP_ERR_INVALID_ARG 1   /* host check failed: null pointer, bad size, misalignment */
#define MEP_ERR_CUDA 2          /* a CUDA launch or attribute call failed */
#define MEP_ERR_BAD_ROUTING 3   /* device: an expert index out of [0,E) or repeated in a token's row */
#define MEP_ERR_CAPACITY 4      /* device: some rank needs more than B redundant slots */
#define MEP_ERR_BAD_POSITION 5  /* device: a dst_pos entry outside [0, R*S*K) */
#define MEP_ERR_BAD_SLOT_MAP 6  /* device: a slot_expert entry outside [-1, E) */
#define MEP_ERR_TIMEOUT 7       /* device: a bounded pipeline wait inside mep_grouped_gemm gave up */
#define MEP_ERR_BAD_SEQLENS 8   /* device: a cu_seqlens row decreases, is negative or does not end at S*K */

/* Size limits checked on the host. */
#define MEP_MAX_E 4096     /* experts */
#define MEP_MAX_R 1024     /* ranks */
#define MEP_MAX_K 64       /* experts per token */
#define MEP_MAX_SLOTS 32768 /* R * B */

/* Library version, (major << 16) | minor. */
MEP_API int mep_version(void);

/* Human-readable name of a return / status code (static string). */
MEP_API const char* mep_status_string(int code);

/*
 * mep_plan_workspace_bytes -- device scratch that mep_plan needs for these
 * sizes (per-block histograms, planner tables). Writes it to *bytes.
 * Returns MEP_ERR_INVALID_ARG for sizes mep_plan would reject.
 */
MEP_API int mep_plan_workspace_bytes(int R, int S, int K, int E, int B, size_t* bytes);

/*
 * mep_plan_kernel_count -- number of kernels one mep_plan (or
 * mep_plan_remote_fallback) call enqueues for these sizes. Writes it to
 * *count. For launch accounting only: nothing is enqueued.
 * Returns MEP_ERR_INVALID_ARG for sizes mep_plan would reject.
 */
MEP_API int mep_plan_kernel_count(int R, int S, int K, int E, int B, int* count);

/*
 * mep_plan -- routing histogram, online planner and destination rows.
 *
 * Problem ("月之暗面开源MoonEP：面向MoE训练的专家并行通信库", 解决的核心问题 and
 * 核心技术): N = R*S tokens, token t belongs to source rank t / S, and routes
 * to the K experts topk_idx[t, 0..K-1]. Expert e's home rank is e / (E/R)
 * (内存契约与权重布局: E/R rows per rank). After planning, every rank
 * receives exactly S*K (token, expert) assignments.
 *
 * Planner (this library's reading of the pages' "online planning"): T_e =
 * number of assignments to e; each rank keeps, in expert order, at most S*K
 * of its home experts' tokens (lowest token index first); the remaining
 * overflow segments, concatenated in expert order, are poured into the
 * deficits S*K - load_r of under-loaded ranks in rank order; each piece
 * occupies the rank's next free redundant slot b (0, 1, ...).
 *
 * Inputs:
 *   topk_idx   int32 [R*S, K]   expert ids, each in [0, E), distinct per row
 *   R, S, K, E, B               ranks, tokens per rank, experts per token,
 *                               experts (E % R == 0, K <= E), slots per rank
 *   workspace  device scratch of >= mep_plan_workspace_bytes(...) bytes
 * Outputs (all written in full on success):
 *   expert_counts int32 [E]          T_e
 *   cu_seqlens    int32 [R, E+B]     inclusive running ends of rank r's rows:
 *                                    row j holds rows [cu[r][j-1], cu[r][j]) of
 *                                    rank r's buffer (cu[r][-1] := 0); rows
 *                                    [0,E) are home experts (non-home rows are
 *                                    empty), rows [E,E+B) redundant slots;
 *                                    cu[r][E+B-1] == S*K
 *   slot_expert   int32 [R, B]       expert held by each slot, -1 if unused
 *   dst_pos       int32 [R*S, K]     row of the static [R*S*K, H] buffer that
 *                                    assignment (t,k) goes to; a permutation
 *                                    of [0, R*S*K); inside a group tokens are
 *                                    in ascending token order
 *   status        int32 [1]          MEP_OK, MEP_ERR_BAD_ROUTING or
 *                                    MEP_ERR_CAPACITY (always written)
 * On MEP_ERR_BAD_ROUTING / MEP_ERR_CAPACITY the device outputs are:
 * slot_expert all -1, cu_seqlens all 0, dst_pos unspecified; expert_counts
 * holds T_e for a capacity error and 0 for a routing error.
 * Host returns: MEP_OK, MEP_ERR_INVALID_ARG, MEP_ERR_CUDA.
 */
MEP_API int mep_plan(const int32_t* topk_idx, int R, int S, int K, int E, int B,
             void* workspace, size_t workspace_bytes,
             int32_t* expert_counts, int32_t* cu_seqlens, int32_t* slot_expert,
             int32_t* dst_pos, int32_t* status, void* stream);

/*
 * mep_plan_remote_fallback -- mep_plan under the inference reading of the
 * slot budget ("月之暗面开源MoonEP：面向MoE训练的专家并行通信库", 内存契约与权重
 * 布局: inference may use B = 3-4; when a rank needs more remote experts than
 * it has slots, their home rank's weights are read through the symmetric
 * mapping, slower but correct). A rank's first B pieces, in pour order, take
 * slots 0..B-1 as in mep_plan; every further piece of expert e takes row e
 * (a [0, E) row, served by e's home weights) of the receiving rank, so a
 * rank's non-home rows can be non-empty. MEP_ERR_CAPACITY never occurs.
 * Arguments, outputs, workspace and the other errors are those of mep_plan;
 * with enough slots the two plans are identical.
 */
MEP_API int mep_plan_remote_fallback(const int32_t* topk_idx, int R, int S, int K, int E, int B,
                                     void* workspace, size_t workspace_bytes,
                                     int32_t* expert_counts, int32_t* cu_seqlens,
                                     int32_t* slot_expert, int32_t* dst_pos, int32_t* status,
                                     void* stream);

/*
 * mep_prefetch -- copy the planned redundant experts' weights into their
 * slots ("月之暗面开源MoonEP：面向MoE训练的专家并行通信库", 核心技术: the
 * redundant experts' weights are prefetched before expert compute;
 * 内存契约与权重布局: rows [E, E+B) of each rank's [E+B, H, H'] weight tensor
 * are local prefetch slots):
 *   slot_w[r][b][:] = home_w[slot_expert[r][b]][:]  for every slot != -1,
 * a byte copy; unused slots are not touched. Any element type.
 *   slot_expert  int32 [R, B]           from mep_plan (or any map into [-1, E))
 *   expert_bytes int64                  bytes of one expert matrix (H*H'*elem), % 16 == 0,
 *                                       below 32 GiB (expert_bytes / 16 < 2^31 - 256)
 *   home_w       [E, expert_bytes]      home experts' weights (read only)
 *   slot_w       [R, B, expert_bytes]   slot weights (written); must not overlap home_w
 *   status       int32 [1]              read on entry (nonzero: no-op); set to
 *                                       MEP_ERR_BAD_SLOT_MAP (nothing copied) if an
 *                                       entry is outside [-1, E). May be NULL.
 * Host returns: MEP_OK, MEP_ERR_INVALID_ARG, MEP_ERR_CUDA.
 */
MEP_API int mep_prefetch(const int32_t* slot_expert, int E, int R, int B, int64_t expert_bytes,
                         const void* home_w, void* slot_w, int32_t* status, void* stream);

/*
 * mep_plan_static_scratch -- mep_plan without a caller-supplied workspace.
 * (The pages have no counterpart: this is an allocation-free variant of the
 * same planner for callers that cannot allocate device memory, such as a
 * host program that reaches the GPU only through this ABI, or a runtime whose
 * device memory belongs to one pool allocator that every allocation must go
 * through.)
 *
 * Arguments, outputs, status values and errors are those of mep_plan. The
 * scratch is a fixed array of MEP_PLAN_STATIC_SCRATCH_BYTES compiled into the
 * library; every GPU that loads the library keeps it until the process exits.
 *   - Sizes whose mep_plan_workspace_bytes exceeds
 *     MEP_PLAN_STATIC_SCRATCH_BYTES are rejected with MEP_ERR_INVALID_ARG
 *     before anything is enqueued.
 *   - No cudaMalloc, cudaFree or allocating library call is made.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and caches it with
 *     the id of the current CUDA context; make that first call before any
 *     stream capture. A call in a new context of the device (after
 *     cudaDeviceReset) looks the address up again: after a reset, make one
 *     call before any capture again. MEP_ERR_CUDA if the lookup fails.
 *   - All calls on a device share the one array and it keeps the last call's
 *     contents (each call writes every scratch byte it later reads, so no
 *     clearing is needed). Calls that overlap on the GPU -- on different
 *     streams, or from several host threads without ordering -- race on it:
 *     order them on one stream.
 */
#define MEP_PLAN_STATIC_SCRATCH_BYTES (4u << 20) /* 4 MiB per device */
MEP_API int mep_plan_static_scratch(const int32_t* topk_idx, int R, int S, int K, int E, int B,
                                    int32_t* expert_counts, int32_t* cu_seqlens,
                                    int32_t* slot_expert, int32_t* dst_pos, int32_t* status,
                                    void* stream);

/*
 * mep_dispatch -- fused permute ("月之暗面开源MoonEP：面向MoE训练的专家并行通信库",
 * 核心技术, 零拷贝与静态形状): buf[dst_pos[t,k], :] = hidden[t, :] for every
 * token t and k, a bit copy into the fixed [R, S*K, H] buffer.
 *   hidden   bf16 [R*S, H]     H % 8 == 0 (rows are whole 16-byte vectors)
 *   dst_pos  int32 [R*S, K]    from mep_plan
 *   status   int32 [1]         read on entry (nonzero: no-op); set to
 *                              MEP_ERR_BAD_POSITION if an entry is out of
 *                              range (that row is skipped). May be NULL.
 *   buf      bf16 [R*S*K, H]   output; must not overlap hidden
 * Host returns: MEP_OK, MEP_ERR_INVALID_ARG, MEP_ERR_CUDA.
 */
MEP_API int mep_dispatch(const mep_bf16* hidden, const int32_t* dst_pos, int32_t* status,
                 int R, int S, int K, int H, mep_bf16* buf, void* stream);

/*
 * mep_combine -- fused weighted unpermute (same section):
 *   out[t, h] = bf16_rn( sum_{k=0..K-1} topk_w[t,k] * y[dst_pos[t,k], h] )
 * accumulated in fp32 from 0 with one fused multiply-add per k, in k order,
 * then rounded to nearest-even bf16.
 *   y        bf16 [R*S*K, H]   expert outputs in the static buffer layout
 *                              (may be the dispatch buffer itself)
 *   topk_w   fp32 [R*S, K]     routing weights, used as given
 *   dst_pos  int32 [R*S, K]    from mep_plan
 *   status   int32 [1]         as for mep_dispatch; may be NULL
 *   out      bf16 [R*S, H]     output; must not overlap y
 * Host returns: MEP_OK, MEP_ERR_INVALID_ARG, MEP_ERR_CUDA.
 */
MEP_API int mep_combine(const mep_bf16* y, const float* topk_w, const int32_t* dst_pos,
                int32_t* status, int R, int S, int K, int H, mep_bf16* out,
                void* stream);

/*
 * mep_dispatch_backward -- gradient of mep_dispatch: dispatch copies
 * hidden[t] to the K rows dst_pos[t, k], so
 *   dhidden[t, h] = bf16_rn( sum_{k=0..K-1} dbuf[dst_pos[t,k], h] )
 * accumulated in fp32 from 0, one add per k in k order. (The pages name the
 * fused permute/unpermute, "月之暗面开源MoonEP：面向MoE训练的专家并行通信库",
 * 核心技术, but give no backward arithmetic; this is the same reading as
 * combine's.)
 *   dbuf     bf16 [R*S*K, H]   gradient of the dispatch buffer
 *   dst_pos  int32 [R*S, K]    from mep_plan
 *   status   int32 [1]         as for mep_dispatch; may be NULL
 *   dhidden  bf16 [R*S, H]     output; must not overlap dbuf
 * Host returns: MEP_OK, MEP_ERR_INVALID_ARG, MEP_ERR_CUDA.
 */
MEP_API int mep_dispatch_backward(const mep_bf16* dbuf, const int32_t* dst_pos, int32_t* status,
                                  int R, int S, int K, int H, mep_bf16* dhidden, void* stream);

/*
 * mep_combine_backward -- gradients of mep_combine (same section):
 *   dy[dst_pos[t,k], h] = bf16_rn( fp32(topk_w[t,k] * dout[t,h]) )
 *   dw[t, k]            = sum_h dout[t,h] * y[dst_pos[t,k], h]   (fp32)
 * Every bf16 x bf16 product is exact in fp32; the dw sum is accumulated in
 * fp32 (per lane, then across a warp), so it matches the exact dot product to
 * within (n + 5) * 2^-24 * sum_h |dout[t,h] * y[dst_pos[t,k],h]|, where
 * n = ceil(H / (32 c)) * c is the longest per-lane chain, c = 16 when
 * H % 16 == 0 and 8 otherwise (the bf16 elements per column vector).
 *   dout     bf16 [R*S, H]     gradient of combine's output
 *   y        bf16 [R*S*K, H]   combine's input (expert outputs)
 *   topk_w   fp32 [R*S, K]     routing weights
 *   dst_pos  int32 [R*S, K]    from mep_plan
 *   status   int32 [1]         as for mep_dispatch; may be NULL
 *   dy       bf16 [R*S*K, H]   output, every row written; must not overlap y or dout
 *   dw       fp32 [R*S, K]     output
 * Host returns: MEP_OK, MEP_ERR_INVALID_ARG, MEP_ERR_CUDA.
 */
MEP_API int mep_combine_backward(const mep_bf16* dout, const mep_bf16* y, const float* topk_w,
                                 const int32_t* dst_pos, int32_t* status, int R, int S, int K,
                                 int H, mep_bf16* dy, float* dw, void* stream);

/*
 * mep_reduce_grad -- fold redundant-slot gradients into home gradients
 * ("月之暗面开源MoonEP：面向MoE训练的专家并行通信库", 内存契约与权重布局, gradient
 * paragraph): for every expert e and element i,
 *   home_grad[e][i] += slot_grad[r][b][i]  over the slots with
 *                      slot_expert[r][b] == e, in ascending (r, b) order,
 * then slot_grad[r][b][:] = 0 for every slot with slot_expert[r][b] != -1.
 * Unused slots (-1) are not touched.
 *   slot_expert int32 [R, B]          from mep_plan (or any map into [-1, E))
 *   E, R, B                           sizes
 *   HHp         int64                 elements per expert matrix (H * H')
 *   home_grad   fp32 [E, HHp]         in/out, 16-byte aligned
 *   slot_grad   fp32 [R, B, HHp]      in/out, 16-byte aligned; must not overlap
 *                                     home_grad (32-byte alignment of both and
 *                                     HHp % 8 == 0 select 32-byte accesses)
 *   status      int32 [1]             read on entry (nonzero: no-op); set to
 *                                     MEP_ERR_BAD_SLOT_MAP (nothing changed)
 *                                     if an entry is outside [-1, E). May be NULL.
 * Host returns: MEP_OK, MEP_ERR_INVALID_ARG (also for a misaligned buffer),
 * MEP_ERR_CUDA.
 */
MEP_API int mep_reduce_grad(const int32_t* slot_expert, int E, int R, int B, int64_t HHp,
                    float* home_grad, float* slot_grad, int32_t* status, void* stream);

/*
 * mep_grouped_gemm -- the grouped expert product over the static buffer
 * ("月之暗面开源MoonEP：面向MoE训练的专家并行通信库", 内存契约与权重布局: one
 * grouped GEMM per expert projection consumes a single [E+B, H, H'] weight
 * tensor -- rows [0, E) the experts' own weights, rows [E, E+B) the rank's
 * prefetch slots -- and cu_seqlens[E+B] says which buffer rows each weight
 * row serves). For rank r, group j spans rows [cu[r][j-1], cu[r][j]) of the
 * rank's block [r*S*K, (r+1)*S*K) of x (cu[r][-1] = 0), and
 *   y[row, n] = bf16_rn( sum_h x[row, h] * W_j[h, n] ),
 *   W_j = w_home[j] for j < E,  w_slot[r][j - E] for j >= E,
 * with the sum accumulated in fp32 by the tensor cores (tcgen05, order
 * unspecified). Rows of an inference plan's overflow (mep_plan_remote_fallback)
 * sit in home rows j < E of a non-home rank and so read w_home[j] directly.
 *   x          bf16 [R*S*K, H]       the dispatch buffer (or any rows so grouped)
 *   cu_seqlens int32 [R, E+B]        inclusive group ends, from mep_plan
 *   w_home     bf16 [E, H, H']       experts' weights
 *   w_slot     bf16 [R, B, H, H']    prefetch slots (mep_prefetch); may be NULL when B == 0
 *   status     int32 [1]             read on entry (nonzero: no-op); set to
 *                                    MEP_ERR_BAD_SEQLENS (y untouched) for a
 *                                    malformed cu_seqlens row, or MEP_ERR_TIMEOUT
 *                                    if a pipeline wait gives up. May be NULL.
 *   H          multiple of 64;  Hp (= H') multiple of 8
 *   ws         device workspace of at least mep_grouped_gemm_workspace_bytes
 *              (the tile table, rebuilt by every call)
 *   y          bf16 [R*S*K, H']      output, every row written; must not overlap
 *              the inputs
 * Host returns: MEP_OK, MEP_ERR_INVALID_ARG (sizes, null pointers, alignment:
 * every tensor 16-byte aligned; x, w_home, w_slot and y must be device memory
 * of the current device, since the kernel's tensor-core operands are copied
 * through tensor maps encoded over them), MEP_ERR_CUDA.
 */
MEP_API int mep_grouped_gemm_workspace_bytes(int R, int S, int K, int E, int B, size_t* bytes);
MEP_API int mep_grouped_gemm(const mep_bf16* x, const int32_t* cu_seqlens, const mep_bf16* w_home,
                             const mep_bf16* w_slot, int32_t* status, int R, int S, int K, int E,
                             int B, int H, int Hp, void* ws, size_t ws_bytes, mep_bf16* y,
                             void* stream);

/*
 * mep_wait_selftest -- exercises the bounded wait that every pipeline wait
 * of mep_grouped_gemm uses: one GPU thread waits on a barrier that nothing
 * completes, with no copy or tensor-core operation in flight. After about
 * limit_ns nanoseconds the wait gives up and writes MEP_ERR_TIMEOUT to
 * *status (device int32; set only if it was 0); *elapsed_ns (device uint64)
 * receives the nanoseconds it waited. For tests of the failure path: the GPU
 * context stays usable.
 *   limit_ns   0 .. 10^10
 * Host returns: MEP_OK, MEP_ERR_INVALID_ARG (null pointer, limit out of range),
 * MEP_ERR_CUDA.
 */
MEP_API int mep_wait_selftest(int32_t* status, int64_t limit_ns, uint64_t* elapsed_ns,
                              void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MEP_H */
