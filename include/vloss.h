/*
 * libvloss: fused per-token losses over rows of vocabulary logits (GB300, sm_103a).
 *
 * One row of fp32 logits s (length V) per token.  Each row gets one
 * max / log-sum-exp reduction, m = max_j s_j, lnS = ln sum_j exp(s_j - m),
 * lse = m + lnS, from which the entry points below produce:
 *
 *   cross-entropy   loss = lse - s[label],  gradient scale * (softmax(s) - onehot(label))
 *                   (aprender-train 0.36.0, entrenar/autograd/wgpu_cross_entropy.rs:
 *                    module doc, forward_async, read_loss, backward);
 *   top-k KL        loss = sum_q p_q (ln p_q - (s[id_q] - lse)),
 *                   gradient coef * (softmax(s) - p_T), p_T the teacher's top-k
 *                   probabilities scattered onto their ids
 *                   (cortiq-engine 0.8.21, src/gpu_wgpu/train_head.rs: module doc, kl_rows);
 *   teacher top-k   the k largest logits, descending, ties to the lower id, with
 *                   probabilities renormalised over the k (train_head.rs: topk_rows);
 *   acc_add         a += b, the sum of per-slice partials (train_head.rs: acc_add, head_kl).
 *
 * Conventions shared by every entry point:
 *
 *  - Pointers are DEVICE pointers owned by the caller, except where a comment says
 *    otherwise.  The library allocates no memory and keeps no pointer after return.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 *    stream).  They never synchronise and never read results back; argument errors
 *    are detected on the host and returned before anything is launched.
 *  - Logits are row-major fp32: row t starts at logits + t * ld; `ld >= V` is the
 *    row stride in elements.  Any alignment of `logits` and any `ld` is accepted
 *    (the kernels stream the 16-byte-aligned body of each row with bulk copies and
 *    handle up to 3 leading and 3 trailing elements with plain loads).
 *  - A vocabulary slice is the column range [col0, col0 + ncols) of every row;
 *    in-place entry points write exactly that range of rows [0, ntok) and nothing else.
 *  - The loss window [loss_start, loss_end), 0 <= loss_start <= loss_end <= ntok,
 *    selects the tokens that count (CEForwardParams / CEBackwardParams of the
 *    cross-entropy page).  Rows outside it get loss 0 and an all-zero gradient.
 *  - Labels and teacher ids are uint32.  A label or id >= V is a data error: it is
 *    counted into *err (when err is not NULL) with atomicAdd, its term is left out,
 *    and a CE loss with a bad label is NaN.  No kernel traps.
 *  - Row statistics `stats` are pairs (m, lnS) per row, [ntok][2] fp32.  They carry the
 *    log-sum-exp of a row between calls more precisely than lse itself: m is exact and
 *    lnS is small exactly when the row is peaked, so the softmax of a later sliced pass
 *    keeps full fp32 accuracy.  Passing only lse costs up to half an ulp of lse in the
 *    exponent of every softmax value.
 *  - A wait inside a kernel that exceeds about two seconds (a bug, never a normal
 *    condition) ends that kernel early with its outputs incomplete and sets a flag
 *    that vl_watchdog_flag() reports.
 */
#ifndef VLOSS_H
#define VLOSS_H

#include <stdint.h>

#if defined(__GNUC__)
#define VL_API __attribute__((visibility("default")))
#else
#define VL_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum vl_status {
    VL_OK = 0,
    VL_EINVAL = 1,        /* bad argument: NULL where required, size or window out of range */
    VL_ELAUNCH = 2,       /* a CUDA call failed; vl_last_error_string() says which */
    VL_EUNSUPPORTED = 3   /* valid request beyond this build's limits (e.g. k > VL_KL_KMAX) */
} vl_status;

/* Limits of this build. */
#define VL_KL_KMAX 1024      /* teacher support per row for vl_kl_topk_inplace */
#define VL_TOPK_KMAX 2048    /* k of vl_topk_rows (the page's bound for topk_rows) */
#define VL_MAX_COLS 0x7FFF0000LL   /* longest row V (2^31 - 2^16): rows are indexed with 32-bit ints */
#define VL_TOPK_NOALLOC_BYTES (32ll << 20)   /* fixed scratch of vl_topk_rows_noalloc (32 MiB a device) */

/* Library version, major * 10000 + minor * 100 + patch. */
VL_API int vl_version(void);

/* Static text for a status code. */
VL_API const char* vl_status_string(vl_status s);

/* Text of the last error raised on the calling host thread ("" if none). */
VL_API const char* vl_last_error_string(void);

/*
 * Cross-entropy forward (wgpu_cross_entropy.rs: module doc "loss = -logits[label] +
 * logsumexp(logits)", forward_async, read_loss).  Reads logits rows [0, ntok), columns
 * [0, V); writes for every row lse[t] (and stats[t] when not NULL), and loss[t] =
 * lse[t] - s_t[label_t] inside the window, 0 outside.  mean (nullable, one float) gets
 * sum of loss over the window / (loss_end - loss_start), 0 for an empty window, as
 * read_loss computes it.
 *   logits [ntok][ld] fp32 (read only)   labels [ntok] u32   loss [ntok] fp32
 *   lse [ntok] fp32 (nullable)           stats [ntok][2] fp32 (nullable)
 *   mean: one fp32 (nullable)            err: one int32 counter (nullable)
 */
VL_API vl_status vl_ce_fwd(const float* logits, int64_t ld, int64_t ntok, int64_t V,
                    const uint32_t* labels, int64_t loss_start, int64_t loss_end,
                    float* loss, float* lse, float* stats, float* mean,
                    int32_t* err, void* stream);

/*
 * Cross-entropy backward in place over a vocabulary slice (wgpu_cross_entropy.rs:
 * backward, "logits[i] = (softmax(logits)[i] - one_hot(label)[i]) * scale").  For rows in
 * the window, columns j in [col0, col0 + ncols):
 *     logits[t][j] = scale * (exp(s_t,j - lse_t) - [j == label_t]),
 * rows outside the window are zeroed.  The page fixes scale = 1 / max(1, window); here it
 * is the caller's argument.  The row statistics come from `stats` when not NULL, else from
 * `lse` (one of them is required).  loss_part (nullable) gets, per row, the slice's share
 * of the CE loss: lse - s[label] when the label lies in the slice and the row is in the
 * window, else 0.
 */
VL_API vl_status vl_ce_bwd_inplace(float* logits, int64_t ld, int64_t ntok, int64_t V,
                            int64_t col0, int64_t ncols, const uint32_t* labels,
                            const float* lse, const float* stats,
                            int64_t loss_start, int64_t loss_end, float scale,
                            float* loss_part, int32_t* err, void* stream);

/*
 * Cross-entropy forward and backward in one pass over each row: the row is read from
 * HBM once and the gradient written once.  Outputs as vl_ce_fwd, then logits rows are
 * overwritten as vl_ce_bwd_inplace does with col0 = 0, ncols = V.
 */
VL_API vl_status vl_ce_fused(float* logits, int64_t ld, int64_t ntok, int64_t V,
                      const uint32_t* labels, int64_t loss_start, int64_t loss_end,
                      float scale, float* loss, float* lse, float* stats, float* mean,
                      int32_t* err, void* stream);

/*
 * Top-k distillation KL with the gradient written in place (train_head.rs: module doc,
 * kl_rows; the float64 loop of head_kl_matches_host).  Per row t in the window:
 *     loss[t]     = sum over q with p_q > 0 and col0 <= id_q < col0 + ncols of
 *                   p_q * (ln p_q - (s[id_q] - lse_t))
 *     logits[t][j] = (coef + ce_coef) * exp(s_j - lse_t)
 *                    - coef * sum_{q: id_q = j} p_q - ce_coef * [j == label_t]
 * for j in [col0, col0 + ncols).  Rows outside the window: loss 0, slice zeroed.
 *   tid [ntok][k] u32, tp [ntok][k] fp32: the teacher's top-k ids and probabilities,
 *     taken as given (sum p = 1 is the caller's precondition; repeated ids add up).
 *   coef: the KL gradient coefficient (the page passes gscale / total).
 *   Row statistics: from stats_in when not NULL, else lse_in when not NULL, else
 *     computed here over the full row, which then requires col0 = 0 and ncols = V.
 *   labels (nullable) with ce_coef folds the CE gradient of the same row into this pass;
 *     the loss output stays the KL alone.  labels == NULL or ce_coef == 0: KL only.
 *   loss [ntok] fp32: the KL, or the slice's part of it for a slice (add the parts of
 *     all slices with vl_acc_add).
 * k must satisfy 1 <= k <= VL_KL_KMAX.
 */
VL_API vl_status vl_kl_topk_inplace(float* logits, int64_t ld, int64_t ntok, int64_t V,
                             int64_t col0, int64_t ncols,
                             const uint32_t* tid, const float* tp, int64_t k, float coef,
                             int64_t loss_start, int64_t loss_end,
                             const float* lse_in, const float* stats_in,
                             const uint32_t* labels, float ce_coef,
                             float* loss, int32_t* err, void* stream);

/*
 * Cross-entropy and top-k distillation KL of the same rows in one pass (the loss step of
 * train_head.rs head_kl -- one kl_rows over whole rows -- with the CE of
 * wgpu_cross_entropy.rs): each row is read from HBM once and its combined gradient is
 * written once, in place.  For rows t in the window:
 *     logits[t][j] = (coef + ce_coef) * exp(s_j - lse_t) - coef * sum_{q: id_q = j} p_q
 *                    - ce_coef * [j == label_t]
 *     kl_loss[t]   = sum over q with p_q > 0 of p_q * (ln p_q - (s[id_q] - lse_t))
 *     ce_loss[t]   = lse_t - s_t[label_t]  (NaN for a label >= V, counted in *err)
 * Rows outside the window: both losses 0, gradient row zeroed, lse and stats not written.
 * lse and stats (nullable) as vl_ce_fwd for the rows in the window; ce_mean (nullable) is
 * the mean of ce_loss over the window (as read_loss).  Long rows are split over a
 * thread-block cluster whose CTAs exchange their row statistics and loss parts through
 * distributed shared memory.
 *   labels [ntok] u32, tid [ntok][k] u32, tp [ntok][k] fp32 (as vl_kl_topk_inplace),
 *   kl_loss [ntok] fp32, ce_loss [ntok] fp32.  1 <= k <= VL_KL_KMAX.
 */
VL_API vl_status vl_ce_kl_fused(float* logits, int64_t ld, int64_t ntok, int64_t V,
                         const uint32_t* labels, const uint32_t* tid, const float* tp, int64_t k,
                         float coef, float ce_coef, int64_t loss_start, int64_t loss_end,
                         float* kl_loss, float* ce_loss, float* lse, float* stats, float* ce_mean,
                         int32_t* err, void* stream);

/*
 * bf16 logits (the page keeps f16 activations beside f32 logits, train_head.rs: Head,
 * head_kl's cvt / cvt_cols): the same five calls over rows of bf16 logits, given as
 * their 16-bit patterns (the upper half of an fp32).  Each row is read as bf16, every
 * maximum, sum, logarithm and exponential is taken in fp32, and each gradient element
 * is rounded to bf16 (nearest even) once, when it is written in place; losses, lse and
 * stats are fp32 as above.  Arguments, outputs and errors as in the fp32 calls; rows
 * may start at any 2-byte boundary, with any ld >= V.  Half the bytes of a row per pass.
 */
VL_API vl_status vl_ce_fwd_bf16(const uint16_t* logits, int64_t ld, int64_t ntok, int64_t V,
                    const uint32_t* labels, int64_t loss_start, int64_t loss_end,
                    float* loss, float* lse, float* stats, float* mean,
                    int32_t* err, void* stream);
VL_API vl_status vl_ce_bwd_inplace_bf16(uint16_t* logits, int64_t ld, int64_t ntok, int64_t V,
                            int64_t col0, int64_t ncols, const uint32_t* labels,
                            const float* lse, const float* stats,
                            int64_t loss_start, int64_t loss_end, float scale,
                            float* loss_part, int32_t* err, void* stream);
VL_API vl_status vl_ce_fused_bf16(uint16_t* logits, int64_t ld, int64_t ntok, int64_t V,
                      const uint32_t* labels, int64_t loss_start, int64_t loss_end,
                      float scale, float* loss, float* lse, float* stats, float* mean,
                      int32_t* err, void* stream);
VL_API vl_status vl_kl_topk_inplace_bf16(uint16_t* logits, int64_t ld, int64_t ntok, int64_t V,
                             int64_t col0, int64_t ncols,
                             const uint32_t* tid, const float* tp, int64_t k, float coef,
                             int64_t loss_start, int64_t loss_end,
                             const float* lse_in, const float* stats_in,
                             const uint32_t* labels, float ce_coef,
                             float* loss, int32_t* err, void* stream);
VL_API vl_status vl_ce_kl_fused_bf16(uint16_t* logits, int64_t ld, int64_t ntok, int64_t V,
                         const uint32_t* labels, const uint32_t* tid, const float* tp, int64_t k,
                         float coef, float ce_coef, int64_t loss_start, int64_t loss_end,
                         float* kl_loss, float* ce_loss, float* lse, float* stats, float* ce_mean,
                         int32_t* err, void* stream);

/*
 * Teacher top-k per row (train_head.rs: topk_rows): ids[t][q], q < k, are the columns of
 * the k largest logits of row t in descending order of value, ties broken by the lower
 * column (-0.0 equals +0.0); probs[t][q] = exp(s[ids[q]] - s[ids[0]]) / sum over the k.
 * The selection is exact (the page's per-thread best-8 is not).  Rows outside the window
 * are not written.  1 <= k <= min(V, VL_TOPK_KMAX).  NaN is a data error: a NaN value is
 * never selected, each row in the window that holds one adds 1 to *err (when err is not
 * NULL), and a row with fewer than k other values gets id 0xFFFFFFFF and probability 0
 * at the positions it cannot fill.  +-inf are ordinary values.
 * Time depends on the data: long rows are filtered with a threshold estimated from their
 * first 3840 columns, and a row for which fewer than k values reach it (one sorted in
 * descending order, for instance) is read a second time; the result is exact either way.
 *   ids [ntok][k] u32, probs [ntok][k] fp32, err: one int32 counter (nullable).
 *   workspace (nullable), workspace_bytes: device memory owned by the caller, 16-byte
 *     aligned, no initial contents needed.  Rows of 30720 to 2^20 columns with k up to
 *     about 6% of V are then streamed by one kernel whose filter warps write each row's
 *     candidates to the workspace while its finish warps order the previous row; the rare
 *     row it cannot settle goes to the exact kernel.  vl_topk_workspace_bytes gives the
 *     size for one CTA per SM of the current device; a smaller workspace that still holds
 *     one CTA's candidate regions runs fewer CTAs, and one below that (or none) has each
 *     row selected and ordered by the single exact kernel.  Same results either way.
 *     Calls that share a workspace must not overlap on the GPU.
 */
VL_API vl_status vl_topk_rows(const float* logits, int64_t ld, int64_t ntok, int64_t V, int64_t k,
                       int64_t loss_start, int64_t loss_end,
                       uint32_t* ids, float* probs, int32_t* err,
                       void* workspace, int64_t workspace_bytes, void* stream);

/*
 * vl_topk_rows for callers that cannot allocate device memory.  No counterpart on the
 * pages: it is the same selection, with its scratch taken from a fixed array in the
 * library instead of a workspace the caller passes.  It serves code that has no way to
 * get device memory at the point of the call: a custom memory pool or allocator hook that
 * calls into this library and must not re-enter the allocator, a latency-bound path that
 * may not risk an allocation (or its failure) there, or an embedded runtime with no device
 * allocator.  Results equal those of vl_topk_rows.
 *   The scratch is one array of VL_TOPK_NOALLOC_BYTES (32 MiB) that every device which
 *   loads the library holds until the process exits.  Rows of 30720 to 2^20 columns use
 *   it (shorter or longer rows need no scratch).  A call takes at most as many rows of
 *   the window as the array holds candidate regions and row list for (millions at
 *   V = 128256; 97 at V = 2^20 and k = 2048 on a 152-SM device); a larger window is
 *   rejected with VL_EUNSUPPORTED and a message that gives the limit (split it into calls).
 *   The first call on a device looks up the array's device address there (with that
 *   device current); make that first call before any stream capture.
 *   Every call shares the one array, which keeps the last call's contents (what must start
 *   at zero is cleared on the stream by each call); calls that overlap on the GPU -- on
 *   two streams, or from two host threads -- race on it and give wrong results.
 */
VL_API vl_status vl_topk_rows_noalloc(const float* logits, int64_t ld, int64_t ntok, int64_t V, int64_t k,
                               int64_t loss_start, int64_t loss_end,
                               uint32_t* ids, float* probs, int32_t* err, void* stream);

/*
 * Bytes of workspace with which vl_topk_rows streams ntok rows of V columns on one CTA per
 * SM of the current device (256 CTAs when no device is present): two sets of candidate
 * regions per CTA (about 60 KB at k = 256, 130 KB at k = 2048 for V = 128256) and 4 bytes a
 * row; 0 when rows of that length and k do not use a workspace (rows shorter than 30720 or
 * longer than 2^20 columns, or k above about 6% of V).
 */
VL_API int64_t vl_topk_workspace_bytes(int64_t ntok, int64_t V, int64_t k);

/*
 * Windowed mean of per-row losses (wgpu_cross_entropy.rs: read_loss, which sums the
 * losses and divides by loss_end - loss_start): *mean = sum of loss[loss_start, loss_end)
 * / (loss_end - loss_start), 0 for an empty window.  The same reduction as the mean
 * output of vl_ce_fwd / vl_ce_fused (a fixed-order double-float sum, so the result does
 * not depend on the launch), for losses produced piecewise, e.g. by calls over chunks of
 * the rows.  loss [ntok] fp32 (read only), mean: one fp32.
 */
VL_API vl_status vl_window_mean(const float* loss, int64_t ntok, int64_t loss_start, int64_t loss_end,
                                float* mean, void* stream);

/*
 * The frozen vocabulary head around the row losses, on chunks of rows so that the
 * [ntok][V] logits are never held whole (cortiq-engine train_head.rs: topk, head_kl).
 * hidden [ntok][hs] and w [V][hs] are bf16 (16-bit patterns), row-major, 16-byte
 * aligned, hs a multiple of 8.  Per chunk, logits = hidden . w^T with bf16 inputs and
 * fp32 accumulation and output (cuBLASLt: a plain dense GEMM), then this library's
 * kernels.  Everything stays on the stream: no host readback between chunks.
 * workspace: caller-owned device memory, 16-byte aligned, no initial contents needed;
 * the call takes as many rows per chunk as it holds (at least one row:
 * vl_*_workspace_bytes(1, ...)).  Calls that share a workspace must not overlap.
 *
 * vl_teacher_topk: ids/probs of the rows [loss_start, loss_end) as vl_topk_rows over the
 *   logits (the teacher's top-k, train_head.rs topk).
 * vl_head_kl: the student's head step (train_head.rs head_kl): per row, the CE + top-k
 *   KL losses and gradient of vl_ce_kl_fused over the logits (window, coef, ce_coef as
 *   there), the gradient rounded to bf16 (the page's cvt_cols), and
 *   dx[t] = dx_scale * sum_j g[t][j] * w[j]  (the page's mm(wt, ..., 1/gscale)),
 *   fp32 [ntok][hs], 16-byte aligned; rows outside the window get dx = 0.  ce_mean
 *   (nullable): the windowed mean of ce_loss.  wt (nullable): the transposed weight
 *   plane [hs][V] bf16, 16-byte aligned, as the page keeps for this GEMM; with it (and V
 *   a multiple of 8) both GEMMs run on the tensor-core kernel of vl_gemm_bf16_tn, without
 *   it the dx GEMM reads w through cuBLASLt.
 */
/*
 * The head's GEMM on the 5th-generation tensor cores: D[M][N] = alpha * A[M][K] . B[N][K]^T,
 * A and B bf16 (16-bit patterns), row-major, 16-byte aligned, K a multiple of 8; D fp32,
 * row-major with stride ldd >= N.  fp32 accumulation in tensor memory (tcgen05.mma fed by
 * TMA).  Logits are hidden . W^T; the backward dlogits . wt^T with the transposed weight
 * plane wt (train_head.rs keeps one per slice for that GEMM).
 */
VL_API vl_status vl_gemm_bf16_tn(const uint16_t* A, const uint16_t* B, float* D, int64_t M, int64_t N, int64_t K,
                          int64_t ldd, float alpha, void* stream);

VL_API int64_t vl_teacher_topk_workspace_bytes(int64_t rows, int64_t V, int64_t k);
VL_API vl_status vl_teacher_topk(const uint16_t* hidden, int64_t hs, const uint16_t* w, int64_t V, int64_t ntok,
                          int64_t k, int64_t loss_start, int64_t loss_end, uint32_t* ids, float* probs,
                          int32_t* err, void* workspace, int64_t workspace_bytes, void* stream);
VL_API int64_t vl_head_kl_workspace_bytes(int64_t rows, int64_t V);
VL_API vl_status vl_head_kl(const uint16_t* hidden, int64_t hs, const uint16_t* w, const uint16_t* wt, int64_t V,
                     int64_t ntok,
                     const uint32_t* labels, const uint32_t* tid, const float* tp, int64_t k, float coef,
                     float ce_coef, float dx_scale, int64_t loss_start, int64_t loss_end, float* dx,
                     float* kl_loss, float* ce_loss, float* ce_mean, int32_t* err, void* workspace,
                     int64_t workspace_bytes, void* stream);

/*
 * a[i] = a[i] + b[i] for 0 <= i < n, fp32, bit-exact (train_head.rs: acc_add, which adds a
 * later vocabulary slice's partial to the first one's).  a and b may not overlap unless
 * a == b.
 */
VL_API vl_status vl_acc_add(float* a, const float* b, int64_t n, void* stream);

/*
 * Test hook for the failure path (no counterpart on the pages).  Arms the next row-engine
 * launch (vl_ce_fwd, vl_ce_bwd_inplace, vl_ce_fused, vl_kl_topk_inplace) made from the
 * calling host thread: CTA 0 of that launch stops issuing its row tiles at body tile
 * number withhold_tile (counted over the CTA's tiles in issue order), and every wait of
 * the launch gives up after wait_cycles SM cycles instead of about two seconds.  The
 * consumers' wait for the missing tile then runs out: the kernel raises the watchdog
 * flag, lets the copies already issued land, and returns with that CTA's outputs
 * incomplete; the other CTAs' rows are unaffected.  Nothing faults or hangs.
 * 1000 <= wait_cycles <= 4e9.  The setting is used once, then cleared.
 */
VL_API vl_status vl_test_inject_wait_timeout(int64_t withhold_tile, int64_t wait_cycles);

/*
 * Reads (and with clear != 0 resets) the flag that a kernel wait timed out on `device`.
 * Synchronous: it waits for the device to finish its work.  Returns -1 if the read fails.
 */
VL_API int vl_watchdog_flag(int device, int clear);

#ifdef __cplusplus
}
#endif

#endif /* VLOSS_H */
