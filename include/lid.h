/*
 * lid.h -- C ABI of the GB300 (sm_103a) lightning-indexer top-k library.
 *
 * The operation (DeepSeek-V4-Flash lightning indexer):
 *
 *   I[t,s] = sum_h w[t,h] * max(0, sum_d q[t,h,d] * k[s,d]) + mask[t,s]
 *
 * and, for every query row t, the top_k keys s of largest I[t,s].
 * Sources: "Eval bug: DeepSeek-V4-Flash lightning-indexer materialises a
 * ctx-proportional (4 GiB/layer) score buffer" (llama.cpp issue 25468),
 * root-cause comment: lid_kq = mul_mat(indexer_k, indexer_q) -> relu ->
 * * weights -> sum_rows -> lid_score -> + mask -> lid_top_k (top 512);
 * same issue, fused-op comment: the fused op takes q, k and the weights;
 * fairydreaming/llama.cpp PR 2, API-change note: the fused op's scale
 * factors were removed and an f16 mask was added; "deepseek v4 support"
 * (llama.cpp PR 22378), collapse-Q revert commit: the per-query formula.
 *
 * The library never forms the n_q x n_kv score matrix (the 4 GiB per layer
 * buffer of the issue): scores live in tensor memory and registers only, a
 * running top-k per query is kept in shared memory, and a split of the keys
 * over CTAs is merged either inside the same (cooperative) launch, where the
 * CTAs agree on a certified bound on each query's top_k-th score and rank the
 * few keys above it, or from O(n_q * splits * top_k) partial lists by a
 * second kernel.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Layouts are row-major, last index contiguous:
 *   q         [n_q][H][D]   16-bit floats (bf16 for lid_topk, f16 for
 *                           lid_topk_f16), 16-byte aligned
 *   k         [n_kv][D]     same type as q, 16-byte aligned
 *   w         [n_q][H]      f32
 *   mask      [n_q][n_kv]   f16 bit patterns, added to the score (0 or -inf
 *                           in the method; any finite value is simply
 *                           added); NULL means all zero
 *   out_idx   [n_q][top_k]  int32
 *   out_score [n_q][top_k]  f32, the value I[t,s] of each returned key
 * Device entry points take device pointers and a cudaStream_t passed as
 * void* (NULL = the legacy default stream); they are asynchronous with
 * respect to the host. The caller owns every buffer.
 *
 * Output order: each row is sorted by score descending, ties by key index
 * ascending; +0 and -0 compare equal; -inf is an ordinary value that ranks
 * below every finite score. When n_kv < top_k, slots j >= n_kv hold
 * (-1, -inf).
 *
 * Supported set: H in {8, 16, 32, 64}, D in {64, 128}, 1 <= top_k <= 2048,
 * 0 <= n_kv <= 2^31 - 1, 0 <= n_q with n_q * H <= 2^31 - 1. Other values
 * return LID_ERR_UNSUPPORTED. q, k, w, mask must hold finite values, except
 * for -inf (and +inf) in the mask.
 *
 * Errors: every error the host can detect (null or misaligned pointer, bad
 * sizes, unsupported H / D / top_k, no sm_103 device) is returned before
 * anything is launched, and the outputs are left untouched. A CUDA error
 * from a launch returns LID_ERR_CUDA. Each bounded device-side wait that
 * runs out records a code that lid_device_error() returns.
 *
 * Memory: when the keys are split over CTAs the call needs a workspace of
 * lid_plan's workspace_bytes (never n_q x n_kv: 1 KiB of barrier counters,
 * then about n_q * splits * top_k * 8 bytes of per-split lists for a merge
 * kernel, or about n_q * (44 KiB + splits * 64 + 8 KiB) bytes for the
 * one-launch path, lid_options.path); otherwise none. lid_topk_ws takes it
 * from the caller, lid_topk_static from a fixed static array; every other
 * device entry point allocates it stream-ordered on the caller's stream from
 * a memory pool the library creates per device, which keeps its memory
 * mapped between calls (inside a stream capture: cudaMallocAsync, i.e. a
 * graph memory node), and then keeps the one-launch path's barrier counters
 * in a static device array of slots that each launch leaves at zero: eager
 * calls use the slot of their stream, found by the stream's ID
 * (cudaStreamGetId, which no later stream reuses, so two streams that can
 * run at the same time never share a slot), and a call recorded into a
 * graph a slot of its own (a graph instantiated twice must not run its two
 * instances at the same time). Past 256 streams or 768 recorded calls the
 * counters move to the workspace, zeroed by a memset on the stream. Cached
 * per-device state (the pool, the static arrays' addresses) is tied to the
 * device's context and looked up again after a device reset.
 *
 * Launches: every kernel is launched as a programmatic dependent of the work
 * before it on the stream (programmatic stream serialization). It touches no
 * global memory before that work has finished (griddepcontrol.wait), so only
 * its set-up overlaps the previous kernel's tail.
 */
#ifndef LID_H
#define LID_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LID_OK = 0,
    LID_ERR_INVALID_ARG = 1,
    LID_ERR_UNSUPPORTED = 2,
    LID_ERR_OOM = 3,
    LID_ERR_CUDA = 4,
    LID_ERR_DEVICE_TIMEOUT = 5,
    LID_ERR_SCRATCH_TOO_SMALL = 6
} lid_status;

typedef enum { LID_DTYPE_BF16 = 0, LID_DTYPE_F16 = 1, LID_DTYPE_E4M3 = 2 } lid_dtype;

/* Tuning and test overrides for lid_topk_ex; zero-initialise for defaults. */
typedef struct lid_options {
    int force_splits;  /* 0: planned; else number of key splits (clamped to [1, key tiles]) */
    int force_qg;      /* 0: planned; else queries per CTA (power of two, H*qg in [16, 256]) */
    int force_kstages; /* 0: planned; else number of K pipeline stages (2..8) */
    int fault_inject;  /* 0: none; 1: the workspace allocation fails (returns LID_ERR_OOM);
                          2: each scoring CTA's epilogue waits on a barrier nothing
                          completes, gives up after ~2 ms (4M cycles), records code 3
                          for lid_device_error() and the CTA exits cleanly (outputs
                          are then unspecified);
                          3: (one-launch path only) the first group barrier waits for
                          one CTA more than the group has, gives up after ~2 ms,
                          records code 4 and every CTA exits cleanly */
    /* Optional cudaEvent_t handles (as void*) recorded on the stream right
       before and right after the scoring kernel, to time it alone. */
    void *ev_score_begin;
    void *ev_score_end;
    int path;          /* how split keys are merged. 0: planned (one launch wherever
                          the keys are split, every CTA of a query group fits on the
                          GPU at once and force_splits is 0); 1: per-split top-k lists
                          in the workspace and a second (merge) kernel; 2: one
                          cooperative launch whose CTAs agree on each query's bound
                          through group barriers (LID_ERR_UNSUPPORTED where the
                          shape does not allow it); 3: as 2, but never the
                          single-query kernel (lid_plan_info.fused) */
    int early_tiles;   /* 0: planned; else (one-launch path with one query per CTA) the
                          tiles a CTA streams before it publishes the certificates that
                          the query's bound comes from (clamped to [1, tiles per split]) */
    int plan_ranges;   /* lid_plan only: 1, the plan of the per-row range forms
                          (lid_topk_ranges, and lid_topk_ws / lid_topk_e4m3 given
                          row_lo / row_hi); 0, lid_topk_ex's. The calls themselves
                          ignore it. */
    int reserved;
} lid_options;

/* What lid_topk_ex would run for a shape (filled by lid_plan). */
typedef struct lid_plan_info {
    int qg;               /* queries per CTA */
    int n_groups;         /* ceil(n_q / qg) */
    int splits;           /* key splits per query group */
    int tiles_per_split;  /* 128-key tiles per split */
    int kstages;          /* K pipeline stages in shared memory */
    int acc_stages;       /* accumulator buffers in tensor memory */
    int cap;              /* candidate-buffer capacity per query (keys) */
    int threads;          /* threads per CTA of the scoring kernel */
    int smem_bytes;       /* dynamic shared memory per CTA */
    int fused;            /* 0: no split or per-split lists + a merge kernel; 1: splits merged
                             inside the one (cooperative) scoring launch; 2: the same by the
                             single-query kernel (one query per CTA, every key of a CTA in its
                             candidate buffer: the decode shape) */
    int64_t workspace_bytes; /* stream-ordered workspace per call */
} lid_plan_info;

/*
 * Top-k of the lightning-indexer score, bf16 q and k. Arguments as in the
 * conventions above. Returns a lid_status.
 */
int lid_topk(const void *q, const void *k, const float *w, const void *mask,
             int64_t n_q, int64_t n_kv, int H, int D, int top_k,
             int32_t *out_idx, float *out_score, void *stream);

/* Same as lid_topk with f16 q and k. */
int lid_topk_f16(const void *q, const void *k, const float *w, const void *mask,
                 int64_t n_q, int64_t n_kv, int H, int D, int top_k,
                 int32_t *out_idx, float *out_score, void *stream);

/* lid_topk / lid_topk_f16 selected by dtype (LID_DTYPE_BF16 or LID_DTYPE_F16;
   LID_DTYPE_E4M3 returns LID_ERR_INVALID_ARG: see lid_topk_e4m3), with
   options (may be NULL). */
int lid_topk_ex(const void *q, const void *k, const float *w, const void *mask,
                int64_t n_q, int64_t n_kv, int H, int D, int top_k,
                int32_t *out_idx, float *out_score, void *stream, int dtype,
                const lid_options *opt);

/*
 * lid_topk_ex with the mask given as one visible key range per query instead
 * of a dense f16 mask: row t sees keys row_lo[t] <= s < row_hi[t] (clamped to
 * [0, n_kv]); every other key scores -inf, exactly as with a dense mask of 0
 * on the range and -inf elsewhere (the pages' causal mask is the range
 * [0, pos + 1); the multi-sequence decode's is each sequence's key range).
 * No mask is read, and when every row of a CTA's query group sees at least
 * top_k keys, the CTA streams only the tiles that the group's ranges touch.
 * This form is not on the pages; it computes the same result without the
 * n_q x n_kv mask.
 *
 * row_lo, row_hi: device arrays of n_q int32, 4-byte aligned (NULL with
 * n_q > 0 returns LID_ERR_INVALID_ARG). By default a call with
 * n_q <= 8 plans one query per CTA (opt->force_qg overrides): right for rows
 * with disjoint ranges; rows sharing one range read its keys once per row.
 */
int lid_topk_ranges(const void *q, const void *k, const float *w,
                    const int32_t *row_lo, const int32_t *row_hi,
                    int64_t n_q, int64_t n_kv, int H, int D, int top_k,
                    int32_t *out_idx, float *out_score, void *stream, int dtype,
                    const lid_options *opt);

/*
 * The indexer with quantised operands: q and k as 8-bit floating point codes
 * (OCP E4M3, the variant without infinities: 1 sign, 4 exponent bits with
 * bias 7, 3 fraction bits, maximum 448; codes 0x7F and 0xFF are NaN and
 * outside the contract) with one f32 scale per row. Element values are
 *
 *   q[t,h,d] = q_scale[t,h] * e4m3(q8[t,h,d]),   k[s,d] = k_scale[s] * e4m3(k8[s,d])
 *
 * and the result is the lightning-indexer top-k of those values, as in the
 * conventions above. Sources: "llama.cpp DeepSeek v4 Flash experimental
 * inference", section "Plan: Implement CUDA Kernels for DeepSeek v4 (DSV4)
 * Operations", kernel 3 (dsv4_fp8_kv_quantize: rows quantised to E4M3 against
 * their amax); "deepseek v4 support" (llama.cpp PR 22378), batched-prefill
 * commit (the indexer's queries are quantised on its scoring path). The
 * quantiser itself (choosing scales and codes) is the caller's.
 *
 *   q8       [n_q][H][D] uint8 codes, 16-byte aligned
 *   q_scale  [n_q][H]    f32, finite and >= 0, 4-byte aligned
 *   k8       [n_kv][D]   uint8 codes, 16-byte aligned
 *   k_scale  [n_kv]      f32, finite and >= 0, 4-byte aligned
 *   w, mask, out_idx, out_score, stream, opt: as for lid_topk_ex
 *   row_lo, row_hi: NULL (use mask), or visible key ranges as for
 *            lid_topk_ranges (mask must then be NULL)
 *
 * Only D = 128 is supported (LID_ERR_UNSUPPORTED otherwise): a 128-element
 * row of codes is one 128-byte swizzle span of the operand layout. The scales
 * must be non-negative because the kernel applies them outside the ReLU:
 * w * relu(qs * ks * x) = (w * qs) * ks * relu(x) for qs, ks >= 0. The plan
 * (lid_plan) and the workspace are those of the 16-bit form of the shape.
 */
int lid_topk_e4m3(const void *q8, const float *q_scale, const void *k8, const float *k_scale,
                  const float *w, const void *mask, const int32_t *row_lo, const int32_t *row_hi,
                  int64_t n_q, int64_t n_kv, int H, int D, int top_k,
                  int32_t *out_idx, float *out_score, void *stream, const lid_options *opt);

/*
 * Host-buffer form: q, k, w, mask, out_idx and out_score are HOST pointers
 * (pinned memory gives the fastest copies). The call allocates device
 * staging, copies the inputs in, runs lid_topk_ex on `stream`, copies the
 * results out, releases the staging and synchronises `stream` before it
 * returns (the copies in run as lid_topk_host_async below describes). The
 * alignment rules for q and k do not apply. Argument errors return before
 * anything is enqueued.
 */
int lid_topk_host(const void *q, const void *k, const float *w, const void *mask,
                  int64_t n_q, int64_t n_kv, int H, int D, int top_k,
                  int32_t *out_idx, float *out_score, void *stream, int dtype);

/*
 * lid_topk_host without the final synchronisation: the call enqueues its work
 * and returns. The input copies run on a copy stream of the library's own,
 * which does not wait for earlier work on `stream`; the kernels, the result
 * copies and the release of the device staging follow on `stream`. So the
 * inputs must hold their values when the call is made and stay unchanged, and
 * out_idx / out_score hold the result, once `stream` has reached this call's
 * end. With pinned host buffers successive calls on one stream overlap one
 * call's input copies with the previous call's kernels, and the kernels run
 * one after another. A call's input copies wait for the end of the call two
 * before it (on any stream), so at most three calls' staging is allocated at
 * once. Inside a stream capture everything is recorded on `stream`. Same
 * arguments, results and errors as lid_topk_host; on an error return, work
 * already enqueued may still be running, so synchronise the stream before
 * reusing the host buffers.
 */
int lid_topk_host_async(const void *q, const void *k, const float *w, const void *mask,
                        int64_t n_q, int64_t n_kv, int H, int D, int top_k,
                        int32_t *out_idx, float *out_score, void *stream, int dtype);
/* (dtype LID_DTYPE_BF16 or LID_DTYPE_F16 for lid_topk_host, lid_topk_ranges
   and lid_topk_static; LID_DTYPE_E4M3 returns LID_ERR_INVALID_ARG) */

/*
 * Every form above with a caller-owned workspace, for callers that keep the
 * workspace themselves (to capture a call in a CUDA graph without memory
 * nodes, or to allocate nothing per call): q / k are bf16 or f16 (dtype
 * LID_DTYPE_BF16 / LID_DTYPE_F16, q_scale and k_scale ignored) or E4M3 codes
 * with their scales (LID_DTYPE_E4M3, as for lid_topk_e4m3); either a dense
 * mask or visible key ranges (as for lid_topk_ranges; both NULL: no mask);
 * other arguments as for lid_topk_ex.
 *
 * workspace: device memory of at least lid_plan's workspace_bytes for the
 * shape and options (for ranges with n_q <= 8 pass force_qg = max(1, 16 / H)
 * to lid_plan), 256-byte aligned, whose first 1024 bytes are zero before the
 * first call that uses it (e.g. from cudaMemset once); every call leaves them
 * zero again, so the same workspace serves any later call of any shape that
 * fits. A shape that needs no workspace accepts NULL. Too small (or NULL when
 * some is needed): LID_ERR_SCRATCH_TOO_SMALL before anything is launched.
 * The library allocates nothing and keeps no state for this call; two calls
 * that may run at the same time on the GPU must not share a workspace.
 * (The pages have no counterpart: this is a deployment form of the same
 * computation.)
 */
int lid_topk_ws(const void *q, const float *q_scale, const void *k, const float *k_scale,
                const float *w, const void *mask, const int32_t *row_lo, const int32_t *row_hi,
                int64_t n_q, int64_t n_kv, int H, int D, int top_k,
                int32_t *out_idx, float *out_score, void *workspace, int64_t workspace_bytes,
                void *stream, int dtype, const lid_options *opt);

/*
 * lid_topk_ex without allocating: for callers that cannot allocate device
 * memory while a step runs -- e.g. an engine that reserves all device memory
 * up front under its own allocator, or a latency-critical path that may not
 * risk an allocation failing or stalling mid-step. (The method on the pages
 * has no counterpart; this is a deployment variant of the same computation.)
 *
 * Same arguments and results as lid_topk_ex with default options, dtype as
 * lid_dtype. When the keys are split over CTAs, the workspace (lid_plan's
 * workspace_bytes: the one-launch path's counters, certificates and gathered
 * candidates, or the per-split lists) lives in one fixed array of 8 MiB in
 * device memory that the library defines statically; every device that loads
 * the library holds it until the process exits. Shapes that need more return
 * LID_ERR_SCRATCH_TOO_SMALL before anything is launched. Nothing else is
 * allocated.
 *
 * The first call on a device looks up the array's device address (with that
 * device current); make that first call before any stream capture on it (a
 * first call inside a capture returns LID_ERR_INVALID_ARG and launches
 * nothing). All calls share the array and it keeps the last call's contents:
 * each call writes every entry before reading it, except the one-launch
 * path's barrier counters in the array's first 1024 bytes, which are zero
 * when the library loads and which every launch leaves at zero. Calls that
 * may overlap on the GPU -- different streams, or different host threads --
 * race on it and must be serialised by the caller.
 */
int lid_topk_static(const void *q, const void *k, const float *w, const void *mask,
                    int64_t n_q, int64_t n_kv, int H, int D, int top_k,
                    int32_t *out_idx, float *out_score, void *stream, int dtype);

/* Fill *info with the launch plan lid_topk_ex would use for a shape on the
 * current device (opt->plan_ranges = 1: the plan of the per-row range forms,
 * which for n_q <= 8 put one row per CTA and give its candidate buffer more
 * of the shared memory). */
int lid_plan(int64_t n_q, int64_t n_kv, int H, int D, int top_k,
             const lid_options *opt, lid_plan_info *info);

/*
 * Sparse attention over the selected latent rows: the consumer of the top-k.
 * "Eval bug: DeepSeek-V4-Flash lightning-indexer ..." (llama.cpp issue 25468),
 * root-cause comment: the top-512 selection feeds the attention of the CSA
 * layers; "deepseek v4 support" (llama.cpp PR 22378), batched-prefill commit:
 * Q*K^T -> softmax -> *V over the MLA latent KV (512 wide), slots masked to
 * -inf contributing nothing. For each query row t and head h, over
 *   J = { j : 0 <= idx[t,j] < n_kv and (sel_score == NULL or sel_score[t,j] != -inf) }
 *   s_j = sum_d qa[t,h,d] * kv[idx[t,j],d]
 *   out[t,h,:] = sum_{j in J} exp(scale*s_j) kv[idx[t,j],:] / sum_{j in J} exp(scale*s_j)
 *   lse[t,h]   = log sum_{j in J} exp(scale*s_j)
 * and out = 0, lse = -inf when J is empty. Keys and values are the same rows.
 * idx / sel_score are exactly lid_topk's out_idx / out_score (its (-1, -inf)
 * padding and masked selections drop out); any other list of row indices
 * works too (repeated indices count once per occurrence).
 *
 *   qa        [n_q][Ha][Dc]  bf16 or f16 (dtype), the queries in the latent
 *                            space, 16-byte aligned
 *   kv        [n_kv][Dc]     same type, 16-byte aligned (may be NULL if n_kv = 0)
 *   idx       [n_q][top_k]   int32
 *   sel_score [n_q][top_k]   f32 or NULL
 *   out       [n_q][Ha][Dc]  f32, 16-byte aligned
 *   lse       [n_q][Ha]      f32 (natural log)
 *   scale     the softmax scale (finite; 1/sqrt(192) or whatever the model uses)
 * Supported: Dc = 512, Ha in {16, 32, 64, 128}, 1 <= top_k <= 2048; others
 * LID_ERR_UNSUPPORTED. Products are exact, sums fp32, the softmax weights are
 * rounded to the input type for the weighted sum of the rows. Two kernels:
 * a tensor-core (tcgen05) kernel with 64 heads per CTA, planned when there
 * are many (query, 64-head) pairs, and a warp-level MMA kernel that splits
 * heads and selections finer for few queries (lid_attn_options.path).
 *
 * When a query's selections are split over CTAs (lid_sparse_attn_plan's
 * splits > 1: few queries), the partial results need workspace_bytes of
 * workspace: from the caller (workspace, workspace_bytes; 256-byte aligned,
 * no initial contents) or, with workspace NULL, stream-ordered from the
 * library's pool as for lid_topk. Too small: LID_ERR_SCRATCH_TOO_SMALL.
 * Errors are returned before anything is launched, outputs untouched.
 */
typedef struct lid_attn_options {
    int force_splits;       /* 0: planned; else splits of each query's selections
                               (clamped to [1, chunks]: ceil(top_k / 64) on path 1,
                               ceil(top_k / 128) on path 2) */
    int force_head_groups;  /* (path 1) 0: planned; else groups of 16 heads per CTA: 1, 2
                               or 4, dividing Ha / 16 (else LID_ERR_INVALID_ARG) */
    int path;               /* 0: planned; 1: the warp-level MMA kernel (any supported Ha);
                               2: the tensor-core kernel (tcgen05, 64 heads per CTA: Ha a
                               multiple of 64 and n_kv > 0, else LID_ERR_UNSUPPORTED) */
    int reserved;
} lid_attn_options;

typedef struct lid_attn_plan_info {
    int path;                /* 1: warp-level MMA kernel, 2: tensor-core kernel */
    int head_groups;         /* groups of 16 heads per CTA */
    int splits;              /* CTAs per (query, head block) */
    int keys_per_split;      /* selections per split (a multiple of 64) */
    int64_t ctas;            /* CTAs of the main kernel */
    int64_t workspace_bytes; /* 0 when splits == 1 */
} lid_attn_plan_info;

int lid_sparse_attn(const void *qa, const void *kv, const int32_t *idx, const float *sel_score,
                    int64_t n_q, int64_t n_kv, int Ha, int Dc, int top_k, float scale,
                    float *out, float *lse, void *workspace, int64_t workspace_bytes,
                    void *stream, int dtype, const lid_attn_options *opt);

int lid_sparse_attn_plan(int64_t n_q, int64_t n_kv, int Ha, int Dc, int top_k,
                         const lid_attn_options *opt, lid_attn_plan_info *info);

/*
 * The first device-side error code recorded since the last reset (0 = none;
 * 1/2/3 = a bounded wait of the load / MMA / epilogue role ran out).
 * Synchronous: it waits for all work on the device. reset != 0 clears it.
 */
int lid_device_error(int reset);

/*
 * Text of the last CUDA error that made a call on this host thread return
 * LID_ERR_CUDA ("no error" if none). Static storage; do not free.
 */
const char *lid_last_cuda_error(void);

/* Static description of a lid_status value. */
const char *lid_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* LID_H */
