/*
 * kvc.h -- C ABI of the B300 (sm_103a) KV-cache compression hot path.
 *
 * One transformer layer's KV cache goes through four steps:
 *   score   -> a per-(unit, kv head, token) importance score (attention mass
 *              or maximum, KVzip+, linear or two-layer surrogate),
 *   select  -> a budget (global top-k across heads, per-head top-k, or a
 *              fixed threshold) that always keeps the sink and recent tokens,
 *   compact -> a gather of the kept K/V rows into one variable-length cache,
 *   decode  -> varlen decode attention over that cache (the consumer), plus a
 *              fidelity probe against full-cache attention.
 * Variants of the cache: group-quantised rows (kvc_quantize_rows,
 * kvc_decode_attn_q8), VECTOR's keys-for-all / values-for-some routing
 * (kvc_vector_*, kvc_decode_attn_vector), and decode-time threshold pruning
 * (kvc_gather_scores, kvc_decode_prune).
 *
 * Sources, cited by page title and section:
 *   [Sculpt] "KVSculpt: KV Cache Compression as Distillation"
 *   [VECTOR] "A Simple Plug-in for Improving Eviction-Based KV Cache Compression"
 *   [KVTC]   "KV Cache Transform Coding for Compact Storage in LLM Inference"
 *   [KVzap]  "KVzap: Fast, Adaptive, and Faithful KV Cache Pruning"
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers owned by the caller unless stated.  The
 *    library never allocates or frees device memory; steps that need scratch
 *    take a caller-provided workspace whose size a *_workspace() query gives.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream).  Nothing synchronises except
 *    kvc_device_status().
 *  - Tensors are dense, row-major, innermost dimension last.  Index names:
 *    U = independent units (batch x layers), Hq / Hkv = query / kv heads,
 *    G = Hq / Hkv (query head h reads kv head h / G), T = cached tokens,
 *    W = observation window, d = head dim.  Flat head index i = u*Hkv + g.
 *  - Return value: KVC_OK, or a negative kvc_status.  Argument errors are
 *    found on the host before any launch and leave every output untouched.
 *    Conditions only the device can see (a row index beyond a capacity, a
 *    bounded wait that gave up) are recorded in a per-device status word that
 *    kvc_device_status() returns and clears; the kernel skips the bad access
 *    and finishes.
 *  - Thread safety: calls on different streams may overlap if their output
 *    and workspace buffers are disjoint.
 */
#ifndef KVC_H_
#define KVC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum kvc_dtype { KVC_F32 = 0, KVC_BF16 = 1 };

enum kvc_status {
  KVC_OK = 0,
  KVC_ERR_INVALID = -1,      /* bad argument (null pointer, size, range)           */
  KVC_ERR_UNSUPPORTED = -2,  /* valid but not implemented (dtype, head dim, size)  */
  KVC_ERR_WORKSPACE = -3,    /* workspace smaller than the *_workspace() query     */
  KVC_ERR_CUDA = -4,         /* a CUDA launch or attribute call failed             */
  KVC_ERR_TIMEOUT = -5,      /* device: a bounded wait gave up                     */
  KVC_ERR_RANGE = -6         /* device: an index fell outside a stated capacity    */
};

enum kvc_select_mode {
  KVC_SEL_GLOBAL_TOPK = 0,   /* one budget per unit shared by its kv heads         */
  KVC_SEL_THRESHOLD = 1,     /* keep iff score >= tau                              */
  KVC_SEL_PER_HEAD = 2       /* one budget per (unit, kv head)                     */
};

/* Library version (major*10000 + minor*100 + patch). */
int kvc_version(void);

/* Static text for a status code; never NULL. */
const char* kvc_status_string(int status);

/*
 * Synchronises `stream`, then returns the first device-side error recorded
 * on the current device since the last call (KVC_OK if none) and clears it.
 * Returns KVC_ERR_CUDA if the synchronisation itself failed.
 */
int kvc_device_status(void* stream);

/* ------------------------------------------------------------------ score */

/* Bytes of workspace kvc_score_attn needs for these sizes (0 if none). */
size_t kvc_score_attn_workspace(int U, int Hq, int Hkv, int T, int W, int d, int dtype);

/*
 * Attention-mass score of every cached token ([Sculpt] §1 and [VECTOR]
 * "Énoncé du Problème": eviction ranks tokens by the attention they receive;
 * [KVzap] §2.1: a token's score is built from the attention weight it
 * receives; [Sculpt] §2B: the log-sum-exp normaliser of the attention row).
 *
 * For unit u, kv head g, query head h in g and window row w:
 *   s[(h,w),t]   = scale * f[u,h] * <q_win[u,h,w,:], k[u,g,t,:]>
 *                  (if causal, only t <= T - W + w: window row w is the
 *                   query at position T - W + w)
 *   scores[u,g,t] = sum over h in g, w < W of softmax_t(s[(h,w),:])[t]
 *
 * q_win      [U, Hq, W, d]  dtype
 * k          [U, Hkv, T, d] dtype
 * head_scale [U, Hq] fp32 temperature factor f, or NULL for all ones; every
 *            entry must be finite and > 0 (a kernel that meets another value
 *            records KVC_ERR_INVALID in the device status word and the scores
 *            of that call are unspecified)
 * scores     [U, Hkv, T] fp32 (written)
 * Requires 1 <= W <= T, Hq % Hkv == 0, d in {64, 128}, finite scale > 0.
 * dtype KVC_BF16 at d = 128 with G*W in {128, 256} runs on the tensor cores
 * (tcgen05, TMEM accumulators, TMA); every other supported shape runs on the
 * SIMT path.  Each unit of scores sums to G*W per kv head (rows are softmaxes).
 */
int kvc_score_attn(const void* q_win, const void* k, int dtype,
                   int U, int Hq, int Hkv, int T, int W, int d,
                   float scale, const float* head_scale, int causal,
                   float* scores, void* workspace, size_t workspace_bytes,
                   void* stream);

/* Aggregation of a token's attention weights over the G*W window rows. */
typedef enum {
  KVC_AGG_SUM = 0,   /* attention mass (kvc_score_attn)                     */
  KVC_AGG_MAX = 1    /* largest attention weight received from any row      */
} kvc_aggregation;

/*
 * kvc_score_attn with the aggregation over the window rows chosen.
 * KVC_AGG_SUM is kvc_score_attn; KVC_AGG_MAX gives
 *   scores[u,g,t] = max over h in g, w < W of softmax_t(s[(h,w),:])[t]
 * ([KVzap] §2.1: KVzip scores a token by the largest attention weight it
 * receives; the KVzip+ normalisation by value and hidden-state norms needs
 * model weights and is not applied here).  Same arguments, layouts,
 * workspace, limits and paths as kvc_score_attn; aggregation outside the
 * enum is KVC_ERR_INVALID.  Each max score lies in (0, 1].
 */
int kvc_score_attn_agg(const void* q_win, const void* k, int dtype,
                       int U, int Hq, int Hkv, int T, int W, int d,
                       float scale, const float* head_scale, int causal,
                       int aggregation, float* scores,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * Linear surrogate score ([KVzap] §2.2: a linear map from the hidden state
 * h_t in R^{Dh} to one score per kv head):
 *   scores[u,g,t] = bias[g] + sum_j hidden[u,t,j] * weight[j,g]
 * hidden [U, T, Dh] dtype; weight [Dh, Hkv] dtype; bias [Hkv] fp32 or NULL;
 * scores [U, Hkv, T] fp32.  Accumulates in fp32.  Requires Dh % 8 == 0,
 * 1 <= Hkv <= 8 and a 16-byte aligned hidden.  Many rows stream through a
 * persistent grid with the weight in shared memory; up to 1024 rows (e.g. the
 * new token of each sequence in a decode step), or a weight too large for
 * shared memory, take one CTA per row with the weight read from L2.
 */
int kvc_score_linear(const void* hidden, const void* weight, const float* bias,
                     int dtype, int U, int T, int Dh, int Hkv,
                     float* scores, void* stream);

/* Bytes of workspace kvc_score_kvzip_plus needs: the value norms
 * [U, Hq, T] fp32 (rounded up to 256 bytes), then the scoring pass's own
 * workspace (as kvc_score_attn_workspace). */
size_t kvc_score_kvzip_plus_workspace(int U, int Hq, int Hkv, int T, int W);

/*
 * KVzip+ score ([KVzap] §2.1): the largest attention weight a token receives
 * from the window rows, each weighted by the token's value contribution to
 * the residual stream over the row's hidden-state norm.  The printed formula
 * divides a_ji by ||W_O v_i|| / ||h_j||; the text and the normalisation it
 * cites weight by the contribution, which is what this computes:
 *   scores[u,g,t] = max_{h in g, w} p[(h,w), t] * ||W_O^h v_t|| / hnorm[u,w]
 * with p the row softmax of kvc_score_attn (same scale, head_scale and
 * causal mask) and ||W_O^h v_t|| = sqrt(v_t^T gram[h] v_t), gram[h] =
 * W_O^h^T W_O^h the d x d Gram matrix of the output projection's slice for
 * query head h (model weights, formed offline).
 * q_win [U, Hq, W, d], k, v [U, Hkv, T, d], gram [Hq, d, d] dtype (KVC_BF16,
 * d = 128, 16-byte aligned); hnorm [U, W] fp32 (> 0); scores [U, Hkv, T]
 * fp32.  The value norms run on warp-level bf16 MMAs; the scoring pass is
 * the tensor-core scorer of kvc_score_attn in a KVzip+ mode when G*W is 128
 * or 256 and W is a multiple of G*W / 4 (a quarter of the rows lies inside
 * one query head), else the SIMT pass (fp32).
 */
int kvc_score_kvzip_plus(const void* q_win, const void* k, const void* v, const void* gram,
                         const float* hnorm, int dtype, int U, int Hq, int Hkv, int T, int W,
                         int d, float scale, const float* head_scale, int causal, float* scores,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Bytes of workspace kvc_score_mlp needs: the first-layer weight transposed
 * to [Dm', Dh] bf16, Dm' = Dm rounded up to 32 (to 64 when Dm > 512), rounded
 * up to 256 bytes.  0 for a non-positive Dh or Dm. */
size_t kvc_score_mlp_workspace(int Dh, int Dm);

/*
 * Two-layer surrogate score ([KVzap] §2.2, the MLP variant: hidden width
 * Dh / 8 with a GELU):
 *   z[u,t,m]     = b1[m] + sum_j hidden[u,t,j] * w1[j,m]
 *   scores[u,g,t] = b2[g] + sum_m GELU(z[u,t,m]) * w2[m,g],
 *   GELU(z) = z (1 + erf(z / sqrt 2)) / 2.
 * hidden [U, T, Dh], w1 [Dh, Dm], w2 [Dm, Hkv] dtype (KVC_BF16); b1 [Dm],
 * b2 [Hkv] fp32 or NULL; scores [U, Hkv, T] fp32.  The first layer runs on
 * the tensor cores (bf16 products, fp32 accumulation in TMEM); each z is
 * rounded to bf16 when the epilogue takes it out of TMEM, and bias, GELU and
 * the second layer accumulate in fp32.  Two launches: w1 transposed into the
 * workspace, then the fused kernel (up to 512 columns of z per pass over the
 * hidden states; Dm > 512 takes two passes).
 * Requires Dh % 8 == 0, Dm % 8 == 0, Dm <= 1024, 1 <= Hkv <= 8, 16-byte
 * aligned hidden and w1, a 256-byte aligned workspace of
 * kvc_score_mlp_workspace(Dh, Dm) bytes.
 */
int kvc_score_mlp(const void* hidden, const void* w1, const float* b1, const void* w2,
                  const float* b2, int dtype, int U, int T, int Dh, int Dm, int Hkv,
                  float* scores, void* workspace, size_t workspace_bytes, void* stream);

/* ----------------------------------------------------------------- select */

/* Bytes of workspace kvc_select needs (currently 0 for every mode). */
size_t kvc_select_workspace(int U, int Hkv, int T, int mode);

/*
 * Budget selection ([KVzap] §2.3: fixed budget "keep exactly x%" or a fixed
 * threshold tau with the w most recent tokens always kept; [KVTC] §2A and
 * [Sculpt] §2A: sinks and the recent window are never compressed; [Sculpt]
 * §2D: heads of one layer end up with different budgets).
 *
 * Protected set P = {t < n_sink} U {t >= T - n_recent}, kept in every head.
 *  GLOBAL_TOPK: per unit, B = floor(keep_ratio * (Hkv*T)) computed in IEEE
 *    double; B_eff = min(max(B, Hkv*|P|), Hkv*T).  The unit keeps P in every
 *    head plus the B_eff - Hkv*|P| highest non-protected (g, t), ordered by
 *    (score desc, t asc, g asc); -0 == +0; NaN ranks below -inf.
 *  PER_HEAD: the same inside each head with B_eff = min(max(head_budget[i],
 *    |P|), T).
 *  THRESHOLD: keep t iff t in P or scores[u,g,t] >= tau (NaN never kept).
 *
 * scores      [U, Hkv, T] fp32
 * head_budget [U*Hkv] int32 (PER_HEAD only, else ignored / may be NULL)
 * kept_idx    [U*Hkv, T] int32 (written): row i holds counts[i] ascending
 *             token indices; entries past counts[i] are left untouched.
 * counts      [U*Hkv] int32 (written)
 * offsets     [U*Hkv + 1] int64 (written): exclusive prefix sum of counts.
 * Requires 0 <= keep_ratio <= 1 (GLOBAL_TOPK), n_sink, n_recent >= 0,
 * Hkv*T <= 2^24 per selection pool (GLOBAL_TOPK pools a unit's heads;
 * pooling several layers of a sequence is a matter of passing them as its
 * heads) and U*Hkv <= 2^24, else KVC_ERR_UNSUPPORTED; at most 512 heads per
 * GLOBAL_TOPK pool.  A pool is selected by one thread-block cluster of up
 * to 16 CTAs; pools of up to 8 heads whose keys fit the cluster's shared
 * memory (about 370 K keys on a B300) keep them on chip, larger ones re-read
 * the scores from global memory in each pass.
 * Selection decisions are taken on the fp32 bits of the scores, so the
 * result is exact and deterministic.
 */
int kvc_select(const float* scores, int U, int Hkv, int T, int mode,
               double keep_ratio, float tau, const int32_t* head_budget,
               int n_sink, int n_recent,
               int32_t* kept_idx, int32_t* counts, int64_t* offsets,
               void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------- compact */

/*
 * Gather-compaction of the kept rows into one variable-length cache
 * ([Sculpt] §1: eviction keeps a subset of the original pairs).  Head i owns
 * rows [start[i], start[i] + counts[i] + slack_per_head) of kc / vc with
 *   start[i] = offsets[i] + i * slack_per_head,
 *   kc[start[i] + j, :] = k[u, g, kept_idx[i, j], :]  (same for v), j < counts[i].
 * Slack rows are not written: decode appends new tokens there.
 *
 * k, v     [U, Hkv, T, d] dtype (a byte copy: any dtype of the enum), in
 *          device memory or in pinned host memory mapped at the same address
 *          (cudaHostAlloc under unified addressing): the kernel then reads
 *          only the kept rows across the bus (a cache held on the host need
 *          not be copied whole to be compacted).  Host memory the device
 *          cannot read is refused with KVC_ERR_INVALID before any launch.
 * kept_idx [U*Hkv, T] int32, counts [U*Hkv] int32, offsets [U*Hkv+1] int64
 *          as written by kvc_select.
 * kc, vc   [capacity_rows, d] dtype; capacity_rows must be at least
 *          offsets[U*Hkv] + U*Hkv*slack_per_head (the device checks every
 *          row and records KVC_ERR_RANGE instead of writing past it).
 * The device also checks the offsets against counts and T: a row j of head
 * i with j < 0 or j >= T is never looked up (its index would lie outside
 * row i of kept_idx), and one with j >= counts[i] (offsets that disagree
 * with counts), or with a kept index outside [0, T), is skipped; each is
 * recorded as KVC_ERR_RANGE.  An offsets total outside [0, U*Hkv*T] copies
 * nothing and records KVC_ERR_RANGE.
 * start    [U*Hkv] int64 (written), len [U*Hkv] int32 (written = counts).
 * Requires d * element size to be a multiple of 16 bytes and 16-byte aligned
 * k, v, kc, vc.
 */
int kvc_compact(const void* k, const void* v, int dtype, int U, int Hkv, int T, int d,
                const int32_t* kept_idx, const int32_t* counts, const int64_t* offsets,
                int slack_per_head, void* kc, void* vc, int64_t capacity_rows,
                int64_t* start, int32_t* len, void* stream);

/* Bytes of workspace kvc_select_compact uses to hand a single pool's
 * decision from the selection to the emission (0: it then runs kvc_select
 * and kvc_compact as they are). */
size_t kvc_select_compact_workspace(int U, int Hkv, int T, int mode);

/*
 * kvc_select followed by kvc_compact on the same arguments, with the same
 * outputs bit for bit (kept_idx, counts, offsets, start, len and the
 * compacted rows of kc / vc) and the same argument rules and error
 * behaviour.  A launch with one selection pool (GLOBAL_TOPK with U = 1, or
 * one head) given at least kvc_select_compact_workspace() bytes of
 * workspace ends the selection once the threshold is known and lets one
 * kernel, a CTA per (token range, head), decide each token again from that
 * threshold, write its index and copy its K / V rows (no separate pass over
 * the kept indices, one launch and one dependent round trip fewer).  Other
 * launches, or a smaller workspace, run the two calls back to back.
 */
int kvc_select_compact(const float* scores, int U, int Hkv, int T, int mode,
                       double keep_ratio, float tau, const int32_t* head_budget,
                       int n_sink, int n_recent,
                       const void* k, const void* v, int dtype, int d, int slack_per_head,
                       void* kc, void* vc, int64_t capacity_rows,
                       int32_t* kept_idx, int32_t* counts, int64_t* offsets,
                       int64_t* start, int32_t* len,
                       void* workspace, size_t workspace_bytes, void* stream);

/* ----------------------------------------------------------------- decode */

/* Bytes of workspace kvc_decode_attn needs when no head holds more than
 * max_len rows (counting the appended one). */
size_t kvc_decode_workspace(int U, int Hq, int Hkv, int d, int max_len, int dtype);

/*
 * One decode step of varlen attention over a compressed cache, GQA
 * ([KVzap] §2.3: pruning sits after attention and works in decode; [Sculpt]
 * §2B: output and log-sum-exp of the attention row).
 *
 * If k_new and v_new are non-NULL they are appended first: row
 * start[i] + len[i] of kc / vc receives k_new[u,g,:] / v_new[u,g,:] and
 * len[i] grows by one (the caller reserved that slack row).  Then, with
 * L = len[i] after the append and rows j < L of head i:
 *   lse[u,h] = log sum_j exp(scale * <q[u,h,:], kc[start[i]+j,:]>)
 *   out[u,h,:] = sum_j exp(scale * <q, kc_j> - lse[u,h]) * vc[start[i]+j,:]
 * A head with L = 0 gets out = 0 and lse = -inf.
 *
 * q      [U, Hq, d] dtype; k_new, v_new [U, Hkv, d] dtype or both NULL
 * kc, vc pool rows [*, d] dtype; start [U*Hkv] int64; len [U*Hkv] int32
 *        (read, and incremented when appending)
 * max_len upper bound on any len[i] after the append (sizes the split-K
 *        grid; rows beyond it are reported as KVC_ERR_RANGE and ignored)
 * out    [U, Hq, d] dtype (written, fp32 accumulate, round-to-nearest-even)
 * lse    [U, Hq] fp32 natural-log log-sum-exp, or NULL
 * Requires d in {64, 128}, G <= 8.
 */
int kvc_decode_attn(const void* q, void* kc, void* vc, const int64_t* start, int32_t* len,
                    const void* k_new, const void* v_new, int dtype,
                    int U, int Hq, int Hkv, int d, int max_len, float scale,
                    void* out, float* lse, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * Group-quantised copy of cache rows ([KVTC] §2B: coefficients quantised in
 * groups that share a scale and an offset, after the Microscaling formats;
 * applied here to the compacted K / V rows themselves).  For every row and
 * group of 32 consecutive elements, in IEEE fp32:
 *   lo    = fp16(min(group))                        (round to nearest even)
 *   scale = fp16((max(group) - lo) / 255)
 *   code  = clamp(rint((x - lo) / scale), 0, 255)    (0 for the group if scale == 0)
 * x      [rows, d] dtype (KVC_BF16, d in {64, 128}; values inside the fp16
 *        range; rows past the heads' lengths may hold anything)
 * codes  [rows, d] uint8 (written), params [rows, d / 32] pairs of fp16
 *        (scale, lo) (written).
 */
int kvc_quantize_rows(const void* x, int dtype, int64_t rows, int d,
                      uint8_t* codes, void* params, void* stream);

/*
 * kvc_decode_attn over a group-quantised pool: kq / vq are the codes and
 * kp / vp the (scale, lo) pairs of K and V as kvc_quantize_rows writes them
 * (same row indexing as kc / vc, 16-byte aligned).  Every cached row is
 * dequantised in the kernel (code * scale + lo, rounded once to fp16), which
 * streams 144 instead of 256 bytes per row and tensor; the dot products take
 * the queries and the softmax weights as fp16 (exact for bf16 queries of
 * magnitude 2^-14 .. 65504) and accumulate in fp32; k_new / v_new are
 * attended exactly and appended quantised (codes and pair of row
 * start[i] + len[i]).  dtype KVC_BF16, d = 128, Hq / Hkv <= 8; same
 * workspace (kvc_decode_workspace), start / len semantics and status word as
 * kvc_decode_attn.
 */
int kvc_decode_attn_q8(const void* q, uint8_t* kq, void* kp, uint8_t* vq, void* vp,
                       const int64_t* start, int32_t* len,
                       const void* k_new, const void* v_new,
                       int dtype, int U, int Hq, int Hkv, int d, int max_len,
                       float scale, void* out, float* lse,
                       void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------- decode-time pruning */

/* Most pools one kvc_decode_prune call moves (K and V rows, or the codes and
 * (scale, lo) pairs of a quantised K and V). */
#define KVC_PRUNE_MAX_POOLS 4

/*
 * Per-row scores of a compacted cache, the array kvc_decode_prune reads:
 * rscore[start[i] + j] = scores[u, g, kept_idx[i, j]] for j < counts[i],
 * i = u*Hkv + g ([KVzap] §2.3: a token's score decides whether it stays).
 * scores [U, Hkv, T] fp32 (as kvc_score_attn / kvc_score_linear write them);
 * kept_idx, counts as kvc_select writes them; start as kvc_compact writes it;
 * rscore [capacity_rows] fp32 (written at the kept rows only).  An index
 * outside [0, T) or a row at or beyond capacity_rows is skipped and reported
 * as KVC_ERR_RANGE in the status word.
 */
int kvc_gather_scores(const float* scores, int U, int Hkv, int T, const int32_t* kept_idx,
                      const int32_t* counts, const int64_t* start, float* rscore,
                      int64_t capacity_rows, void* stream);

/*
 * Decode-time threshold pruning ([KVzap] §2.3: the `window` most recent
 * tokens are always kept, a token whose score is below tau is dropped, and
 * the pruning runs after attention, in decoding as in prefilling).
 *
 * Call it after a decode step that appended one token per head (so len[i]
 * counts the new row, start[i] + len[i] - 1).  A head's rows are in token
 * order; rows [0, len - window) have been judged, the last `window` rows are
 * the window.  Per head i:
 *   1. rscore[start[i] + len[i] - 1] = s_new[i]  (the new token's score);
 *   2. e = len[i] - window - 1 is the row of the token that just left the
 *      window; if e >= n_sink and !(rscore[start[i] + e] >= tau) (fp32; a NaN
 *      score is dropped), rows e+1 .. len[i]-1 of every pool and of rscore
 *      move down by one row and len[i] shrinks by one.
 * Rows at or beyond the new len[i] are left unspecified.
 *
 * pools     HOST array of n_pools (1 .. KVC_PRUNE_MAX_POOLS) device pointers,
 *           16-byte aligned, each indexed by pool row; row_bytes HOST array of
 *           their row sizes (multiples of 16 bytes): e.g. {kc, vc} with
 *           {2d, 2d} for bf16 pools, {kq, kp, vq, vp} with {d, d/8, d, d/8}
 *           for quantised ones
 * rscore    [capacity_rows] fp32 per-row scores (kvc_gather_scores)
 * start     [n_heads] int64; len [n_heads] int32 (read, decremented on a drop)
 * s_new     [n_heads] fp32 scores of the appended tokens (e.g. kvc_score_linear
 *           on the new hidden states with T = 1)
 * window >= 1, n_sink >= 0, tau not NaN, capacity_rows = rows of every pool.
 * A head with start[i] + len[i] > capacity_rows is skipped and reported as
 * KVC_ERR_RANGE.  No workspace; one CTA per head.
 */
int kvc_decode_prune(void* const* pools, const int* row_bytes, int n_pools, float* rscore,
                     const int64_t* start, int32_t* len, const float* s_new, int n_heads,
                     int window, int n_sink, float tau, int64_t capacity_rows, void* stream);

/*
 * The same pruning with the window kept as a ring ([KVzap] §2.3, as
 * kvc_decode_prune): a head's rows are not kept in token order, so a drop
 * moves one row instead of the window's.  The window (a head's last `window`
 * appended rows) is a FIFO of row indices (relative to start[i]):
 * ring[i*window + t % window] holds the entry appended at step counter t
 * (-1: no row).  Call it after a decode step with counter t_new (any counter
 * that grows by one per step, the same for every head) appended row
 * len[i] - 1.  Per head i, with s = t_new % window and e = ring[i*window + s]
 * the row that leaves the window:
 *   - e < n_sink (no row, or a sink: the sinks are a head's first rows and
 *     never move) or rscore[start[i] + e] >= tau (fp32; a NaN score goes):
 *     the row stays; rscore[start[i] + len[i] - 1] = s_new[i] and
 *     ring[i*window + s] = len[i] - 1;
 *   - otherwise row len[i] - 1 of every pool moves into row e,
 *     rscore[start[i] + e] = s_new[i], ring[i*window + s] = e and len[i]
 *     shrinks by one.
 * The rows a head holds and their scores are those kvc_decode_prune gives,
 * in another order.  Arguments as kvc_decode_prune, plus ring [n_heads,
 * window] int32 (read and written; set up by kvc_prune_ring_init) and
 * t_new >= 0.  An e >= len[i] - 1 is reported as KVC_ERR_RANGE and the row
 * stays.  No workspace; one warp per head.
 */
int kvc_decode_prune_ring(void* const* pools, const int* row_bytes, int n_pools, float* rscore,
                          const int64_t* start, int32_t* len, int32_t* ring, int64_t t_new,
                          const float* s_new, int n_heads, int window, int n_sink, float tau,
                          int64_t capacity_rows, void* stream);

/*
 * The ring of kvc_decode_prune_ring for heads whose last `window` rows are
 * their window in append order (a compaction, or kvc_decode_prune's layout):
 * the entry of counter t_next - window + k is row len[i] - window + k
 * (k < window; -1 where that row would be negative), t_next = the counter of
 * the next decode step.  len [n_heads] int32; ring [n_heads, window] int32
 * (written).
 */
int kvc_prune_ring_init(const int32_t* len, int n_heads, int window, int64_t t_next,
                        int32_t* ring, void* stream);

/* ------------------------------------------------ VECTOR three-way routing */

/*
 * VECTOR ("A Simple Plug-in for Improving Eviction-Based KV Cache
 * Compression", Méthodologie : VECTOR): the base eviction selects a widened
 * pool of 1 - p_c + p_a of the tokens (kvc_select, e.g. global top-k); every
 * pool token keeps its key; the 2 p_a pool tokens whose values an offline OLS
 * predictor W rebuilds best from their keys (v ~ W k) drop their values; the
 * rest keep K and V.  W is [Hkv, d, d] bf16, row = output dimension.  The
 * pages rotate keys back before the reconstruction (RoPE); caches without a
 * rotary encoding need no rotation, which is what these calls assume.
 *
 * Step 2, the reconstruction error as a selection key: for pool position
 * j < counts[i] of head i = u*Hkv + g holding token t = kept_idx[i, j],
 *   key[u, g, j] = -sum_x (v[u,g,t,x] - sum_y W[g,x,y] k[u,g,t,y])^2
 * (fp32 accumulation of bf16 products), and key = NaN for protected tokens
 * (t < n_sink or t >= T - n_recent: their values stay exact) and for
 * positions j >= counts[i].  A global top-k of `key` (kvc_select, mode
 * KVC_SEL_GLOBAL_TOPK, no protection, a budget of at most the non-protected
 * pool tokens) then picks the lowest-error positions of each unit, in
 * (error asc, position asc, head asc) order.
 * k, v [U, Hkv, T, d] bf16, d = 128, 16-byte aligned; W as above; key
 * [U, Hkv, T] fp32 (written in full).
 */
int kvc_vector_residual(const void* k, const void* v, const void* W, int dtype, int U, int Hkv,
                        int T, int d, const int32_t* kept_idx, const int32_t* counts,
                        int n_sink, int n_recent, float* key, void* stream);

/*
 * Step 3's choice of the approximated tokens, reading only the pool's
 * positions: per unit u, the n_approx positions of highest key among
 * positions j < counts[u*Hkv + g] of its heads g, ranked by (key desc,
 * position asc, head asc), NaN below every number.  Positions at or past a
 * head's count are neither read as candidates nor chosen; when n_approx
 * exceeds the candidates, every candidate is chosen.  With the keys of
 * kvc_vector_residual and an n_approx of at most the pool's non-protected
 * tokens (the pages' budgets), no NaN key is chosen and the result equals
 * kvc_select(key, KVC_SEL_GLOBAL_TOPK) with no protected set and a budget of
 * n_approx, which sweeps all Hkv * T positions.
 * key [U, Hkv, T] fp32 (16-byte aligned rows take bulk copies); counts
 * [U*Hkv] int32 (the pool's, from kvc_select); outputs as kvc_select's:
 * approx_pos [U*Hkv, T] (the first approx_counts[i] entries of row i,
 * ascending), approx_counts [U*Hkv], approx_offsets [U*Hkv + 1].
 * Errors: KVC_ERR_INVALID for NULL pointers, non-positive sizes or n_approx
 * outside [0, Hkv*T]; KVC_ERR_UNSUPPORTED for more than 8 heads per unit or
 * a pool beyond 2^24 positions.  Device-side counts are clamped to [0, T].
 */
int kvc_vector_select(const float* key, int U, int Hkv, int T, const int32_t* counts,
                      int64_t n_approx, int32_t* approx_pos, int32_t* approx_counts,
                      int64_t* approx_offsets, void* stream);

/*
 * Step 3 as a cache layout.  Head i keeps the K rows of all counts[i] pool
 * tokens and the V rows of the exact ones:
 *   kc rows [kstart_i, kstart_i + counts_i + slack): the approximated tokens
 *     (pool positions approx_pos[i, 0..approx_counts[i]), ascending) first,
 *     then the exact tokens in pool order;
 *   vc rows [vstart_i, vstart_i + counts_i - approx_counts_i + slack): the
 *     exact tokens' values;
 *   kstart_i = offsets[i] + i*slack, vstart_i = offsets[i] - approx_offsets[i]
 *   + i*slack; klen[i] = counts[i]; napprox[i] = approx_counts[i].
 * kept_idx / counts / offsets: the pool (kvc_select); approx_pos /
 * approx_counts / approx_offsets: the global top-k of the residual keys
 * (kvc_select on kvc_vector_residual's output).  Byte copies; a row beyond
 * kc_rows / vc_rows or an index out of range is skipped and reported as
 * KVC_ERR_RANGE.  bf16, d = 128, 16-byte aligned pools.
 */
int kvc_vector_compact(const void* k, const void* v, int dtype, int U, int Hkv, int T, int d,
                       const int32_t* kept_idx, const int32_t* counts, const int64_t* offsets,
                       const int32_t* approx_pos, const int32_t* approx_counts,
                       const int64_t* approx_offsets, int slack_per_head, void* kc,
                       int64_t kc_rows, void* vc, int64_t vc_rows, int64_t* kstart,
                       int32_t* klen, int64_t* vstart, int32_t* napprox, void* stream);

/* Bytes of workspace kvc_decode_attn_vector needs when no head holds more
 * than max_len keys (counting the appended one). */
size_t kvc_decode_vector_workspace(int U, int Hq, int Hkv, int d, int max_len);

/*
 * One decode step over a VECTOR cache.  Head i holds klen[i] keys at
 * kc[kstart[i]..]; the value of key row j is W[g] kc[kstart[i] + j] for
 * j < napprox[i] (rebuilt) and vc[vstart[i] + j - napprox[i]] otherwise.  If
 * k_new / v_new are given they are appended as an exact row (kc row
 * kstart[i] + klen[i], vc row vstart[i] + klen[i] - napprox[i]) and klen[i]
 * grows by one.  Output and log-sum-exp as kvc_decode_attn.  The rebuilt
 * values are never formed row by row: the approximated rows' attention
 * weights are applied to their keys, and W[g] once per query head to that
 * sum (the same result up to rounding order).  bf16, d = 128,
 * Hq / Hkv <= 8, 16-byte aligned q, kc, vc and W.
 */
int kvc_decode_attn_vector(const void* q, void* kc, void* vc, const int64_t* kstart,
                           int32_t* klen, const int64_t* vstart, const int32_t* napprox,
                           const void* W, const void* k_new, const void* v_new, int dtype, int U,
                           int Hq, int Hkv, int d, int max_len, float scale, void* out,
                           float* lse, void* workspace, size_t workspace_bytes, void* stream);

/*
 * kvc_decode_attn without a workspace, for callers that cannot allocate
 * device memory (a plug-in inside a host engine that owns every allocation
 * and offers no workspace; a caller whose device-memory budget is fixed at
 * start-up).  The pages have no counterpart: this is an interface choice.
 *
 * Same arguments, semantics and results as kvc_decode_attn, minus the
 * workspace.  The split-K scratch is a fixed array of
 * KVC_DECODE_NOALLOC_SCRATCH_BYTES in the library's device memory, held on
 * every GPU where the library's device code has been loaded until the process
 * exits.  The call itself allocates and frees nothing.
 *  - Limit: sizes with kvc_decode_workspace(U, Hq, Hkv, d, max_len, dtype) >
 *    KVC_DECODE_NOALLOC_SCRATCH_BYTES are refused with KVC_ERR_WORKSPACE
 *    before any CUDA call (e.g. 64 x 8 kv heads, G = 4, d = 128 fit up to
 *    max_len = 15360).
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current.  With CUDA's lazy
 *    module loading (the default) that lookup is also what loads the module
 *    and so reserves the array on that device: the first call can fail with
 *    KVC_ERR_CUDA when the device's memory is already committed.  Make the
 *    first call on each device at start-up, before the caller commits its
 *    device memory and before any stream capture.
 *  - All calls on a device share the array: calls whose kernels can overlap
 *    on the GPU race and must be serialised by the caller.  The array keeps
 *    the last call's contents; nothing in it needs clearing, since each step
 *    writes every record it reads.
 */
#define KVC_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/* The scratch size of kvc_decode_attn_noalloc in bytes (a constant). */
size_t kvc_decode_noalloc_scratch_bytes(void);

int kvc_decode_attn_noalloc(const void* q, void* kc, void* vc, const int64_t* start,
                            int32_t* len, const void* k_new, const void* v_new, int dtype,
                            int U, int Hq, int Hkv, int d, int max_len, float scale,
                            void* out, float* lse, void* stream);

/*
 * Fidelity probe of a compressed cache against the full one, per (unit, q
 * head) ([Sculpt] §4 measures fidelity as a KL divergence):
 *   rel_err = ||out_comp - out_full||_2 / ||out_full||_2 (0/0 -> 0)
 *   kl      = KL(p_comp || p_full) = lse_full - lse_comp
 * (the second identity holds because the compressed rows are a subset of
 * the full rows; it equals -log of the attention mass the full softmax puts
 * on the kept rows).
 * out_* [n, d] dtype; lse_* [n] fp32; rel_err, kl [n] fp32 (written).
 */
int kvc_fidelity(const void* out_comp, const void* out_full,
                 const float* lse_comp, const float* lse_full, int dtype,
                 int n, int d, float* rel_err, float* kl, void* stream);

/* -------------------------------------------------------------- self-test */

/*
 * Runs one kernel whose bounded wait is made to run out: it waits on an
 * mbarrier nothing arrives on, gives up after timeout_ns nanoseconds,
 * records KVC_ERR_TIMEOUT in the device status word and returns.  Lets a
 * test check the timeout path of the kernels' waits without hanging a GPU.
 */
int kvc_selftest_wait_timeout(uint64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H_ */
