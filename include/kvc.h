/*
 * kvc.h -- C ABI of libkvc: attention-score-driven prompt KV-cache
 * compression on one GB300 GPU (sm_103a).
 *
 * The method, in the pages' terms:
 *  1. Observation-window scoring (SnapKV; blog post "ZigZagKV, KVCache 80%
 *     compression near-lossless", section "SnapKV"): the last W prompt
 *     tokens' queries attend to all T prompt keys; each KV head's attention
 *     rows are averaged over its window rows and its GQA query heads into one
 *     importance value per token.  Attention is softmax(Q K^T / sqrt(D))
 *     ("ThinK: Thinner Key Cache by Query-Driven Pruning", section "Method
 *     details").
 *  2. ZigZagKV budgets (same blog post, sections "ZigZagKV's new
 *     observations" and "ZigZagKV space allocation"): each head's MBA is the
 *     fewest tokens whose scores reach 90% of the attention mass; a layer's
 *     LMBA is the mean over its heads; the total budget is split across
 *     layers in proportion to LMBA with a per-layer floor.
 *  3. Selection (same post, sections "SnapKV" and "ZigZagKV token
 *     selection"): each head keeps its layer's budget of highest-scoring
 *     prefix tokens plus every window token; the kept K/V rows are gathered
 *     into a compacted cache.
 *  4. ThinK magnitude pruning (ThinK page, "Magnitude-based pruning"): keep
 *     floor((1-lambda) D) key channels per head with the largest l2 norm over
 *     the kept prefix rows; window (recent) rows are not pruned ("Implementation
 *     of THINK").
 *
 * Conventions (all entry points):
 *  - Every tensor argument is a DEVICE pointer owned by the caller,
 *    contiguous in the layout stated below (kvc_compress_host alone takes
 *    its prompt in pinned host memory).  No call allocates device memory;
 *    scratch lives in a caller-provided workspace of kvc_workspace_size()
 *    bytes, zeroed once with kvc_workspace_init() (kvc_score_noalloc alone
 *    uses a fixed array inside the library).
 *  - Work is enqueued on `stream` and is asynchronous.  Argument errors are
 *    detected on the host before anything is launched and returned as a
 *    negative kvc_status; kvc_last_error() then holds a message.
 *  - Data-dependent errors found by a kernel (a score outside [0,1], a
 *    budget larger than k_max, an output buffer too small, a pipeline wait
 *    that timed out) are OR-ed into a status word inside the workspace and
 *    read back with kvc_workspace_status().  Launch failures return
 *    KVC_ERR_CUDA.
 *  - Calls sharing one workspace must be ordered on one stream; distinct
 *    workspaces may run concurrently.
 *
 * Layouts (row-major, innermost last):
 *  q_obs   [L][H_q][W][D]   window queries; query head h belongs to KV head
 *                           h / (H_q / H_kv)
 *  k, v    [L][H_kv][T][D]  prompt keys / values; window = last W positions
 *  scores  [L][H_kv][T]     fp32, sums to 1 per head
 *  mba     [L][H_kv]        int32
 *  budget  [L]              int32, prefix tokens kept per head of layer l
 *  idx     [L][H_kv][k_max] int32, ascending kept prefix positions; entries
 *                           at and after n_l = min(budget[l], T-W) untouched
 *  k_out, v_out             packed: layer l holds [H_kv][n_l + W][D] (kept
 *                           rows ascending, then the W window rows); layer l
 *                           starts at row H_kv * sum_{l'<l} (n_l' + W)
 *  chan    [L][H_kv][keep]  int32, ascending kept key channels
 *  k_pruned packed: layer l holds [H_kv][n_l][keep], starting at element
 *                           H_kv * keep * sum_{l'<l} n_l'
 */
#ifndef KVC_H
#define KVC_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KVC_OK = 0,
    KVC_ERR_INVALID_ARG = -1,  /* bad shape, pointer, size or alignment */
    KVC_ERR_UNSUPPORTED = -2,  /* valid request the library cannot serve */
    KVC_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed */
    KVC_ERR_TIMEOUT = -4,      /* reserved: a device wait gave up */
    KVC_ERR_WORKSPACE = -5     /* workspace missing or smaller than required */
} kvc_status;

typedef enum { KVC_F32 = 0, KVC_BF16 = 1 } kvc_dtype;

/* Device status bits, OR-ed into the workspace status word by kernels. */
#define KVC_DEV_TIMEOUT      0x1u  /* a pipeline wait exceeded its limit */
#define KVC_DEV_BAD_SCORE    0x2u  /* a score was negative, NaN or > 1, or
                                      the scores of a head summed above 16 */
#define KVC_DEV_BAD_BUDGET   0x4u  /* min(budget[l], T-W) exceeded k_max or
                                      budget[l] was negative; clamped */
#define KVC_DEV_OUT_CAPACITY 0x8u  /* packed output larger than the buffer;
                                      rows past the end were not written */
#define KVC_DEV_INVARIANT    0x10u /* bounds-checking builds only (compiled with
                                      KVC_DEBUG_BOUNDS): an output invariant
                                      failed -- kept or compacted indices not
                                      strictly ascending or outside [0, T-W),
                                      an MBA outside [0, T], budgets not summing
                                      to min(total, L (T-W)) or outside
                                      [floor, T-W], kept channels not strictly
                                      ascending or outside [0, D).  The check
                                      records the bit and the kernel goes on; it
                                      never traps. */

typedef struct {
    int32_t n_layers;    /* L >= 1 */
    int32_t n_q_heads;   /* H_q >= 1, a multiple of H_kv */
    int32_t n_kv_heads;  /* H_kv >= 1 */
    int32_t head_dim;    /* D, 1..256 (tensor-core path: 64 or 128, bf16) */
    int32_t seq_len;     /* T > W */
    int32_t window;      /* W >= 1, observation window = last W tokens */
    int32_t dtype;       /* kvc_dtype of q_obs, k, v */
} kvc_shape;

/* Bytes of workspace the calls below need for `shape` on the CURRENT device
 * (the score pass splits work by the device's SM count).  Returns 0 for an
 * invalid shape.  k_max is accepted for future use and may be 0. */
size_t kvc_workspace_size(const kvc_shape *shape, int32_t k_max);

/* Zero the workspace (status word included).  Call once after allocating
 * it; kernels only OR bits into the status word afterwards. */
int kvc_workspace_init(void *ws, size_t ws_bytes, cudaStream_t stream);

/* Synchronise `stream` and return the device status word of `ws` (the OR of
 * KVC_DEV_* bits since the last kvc_workspace_init) in *status. */
int kvc_workspace_status(const void *ws, size_t ws_bytes, uint32_t *status,
                         cudaStream_t stream);

/* a1 -- observation-window scores (SnapKV scoring, causal inside the window,
 * GQA-averaged):
 *   scores[l][k][j] = 1/(G W) * sum_{g<G, i<W} softmax_j( q_{kG+g,i} . k_j / sqrt(D) )
 * with row i (position T-W+i) seeing keys j <= T-W+i only; scores of keys a
 * row cannot see are zero for that row.  Computed with fp32 accumulation;
 * bf16 inputs with D in {64,128} and G*W <= 512 run on the tcgen05 tensor
 * cores, everything else on a CUDA-core fp32 path.  q_obs and k must be
 * 16-byte aligned.  Uses the workspace for per-row softmax statistics.
 * The tensor-core kernels are persistent: one 2-CTA cluster per SM pair,
 * ~216 KB of shared memory and all 512 TMEM columns of every SM they run on;
 * other work on the device shares the SMs only between their launches.
 * Every device wait is bounded (1 s): a wait that runs out sets
 * KVC_DEV_TIMEOUT and the kernel returns.  The environment variable
 * KVC_TEST_SKIP_ARRIVE=1 (tests only) withholds one arrival in the first
 * tensor-core pass to exercise that path. */
int kvc_score(const kvc_shape *shape, const void *q_obs, const void *k, float *scores,
              void *ws, size_t ws_bytes, cudaStream_t stream);

/* kvc_score for callers that cannot allocate device memory (no counterpart in
 * the method pages; it exists for integration only).  Some hosts give a
 * plugin just its input and output buffers -- no workspace -- and forbid
 * cudaMalloc because their own allocator already holds the device memory
 * and an allocation would synchronise the device mid-schedule.  This call
 * computes exactly what kvc_score computes, with the same shape rules, the
 * same kernel choice (KVC_SCORE_IMPL included) and the same kernels, but
 * keeps its scratch in a fixed 8 MiB array inside the library's device memory
 * (held by every GPU that loads the library until the process exits).
 * Shapes whose scratch exceeds 8 MiB return KVC_ERR_UNSUPPORTED (the 32K and
 * 128K Llama-3-8B-shaped prompts need 2.5 MiB).  dev_status is an
 * optional 4-byte-aligned DEVICE uint32 that is zeroed and then receives the
 * KVC_DEV_* bits (misaligned: KVC_ERR_INVALID_ARG).  With dev_status NULL the
 * bits go to a word inside the array that no call reads back, so device-side
 * errors (a timed-out wait) cannot be observed: callers that need them pass
 * a word of their own.  The first call on each device
 * looks up the array's device address (cudaGetSymbolAddress) and should be
 * made outside any stream capture.  All calls share the array: calls that
 * overlap on the GPU race and give undefined scores, so order them on one
 * stream.  Allocates nothing. */
int kvc_score_noalloc(const kvc_shape *shape, const void *q_obs, const void *k, float *scores,
                      uint32_t *dev_status, cudaStream_t stream);

/* Optional variant of a1 -- Keyformer scores ("Keyformer: KV Cache reduction
 * through key tokens selection": Gumbel noise zeta is added to the logits
 * x = q.k / sqrt(D) and a temperature tau softens the softmax,
 * f = softmax((x + zeta) / tau); the most recent tokens are kept and the
 * remaining budget goes to the highest-scoring older tokens).  Same layouts,
 * workspace and two-pass structure as kvc_score, with
 *   scores[l][k][j] = 1/(G W) sum over window rows r that see j of
 *                     softmax_j((x_rj + zeta_rj) / tau),
 * zeta_rj = -ln(-ln u), u = (b + 1/2) 2^-24 where b is the top 24 bits of
 * word 0 of Philox4x32-10 at counter (j, r, l*H_kv + k, 0) and key
 * (seed & 0xffffffff, seed >> 32); r = g*W + w is the row within the unit.
 * The page sets tau to infinity in the prompt phase, which would make every
 * score equal; here tau is a parameter in (0, 1e30].  The window is the
 * recent part that compaction always keeps; pass the scores to
 * kvc_mba_budget / kvc_topk_select for the older part.  bf16 inputs with D in
 * {64,128} and G*W <= 512 run on the tcgen05 tensor cores (the noise drawn in
 * the epilogue), everything else on a CUDA-core fp32 path; both draw the same
 * numbers.  On the tensor-core path q_obs and k must be 16-byte aligned. */
int kvc_score_keyformer(const kvc_shape *shape, const void *q_obs, const void *k, uint64_t seed,
                        double tau, float *scores, void *ws, size_t ws_bytes, cudaStream_t stream);

/* The default path (kvc_score -> kvc_mba_budget -> kvc_topk_select ->
 * kvc_compact) for a prompt whose Q_obs, K and V live in HOST memory, the
 * pages have no counterpart (it is how the path is fed from a host).  The
 * copy of K is pipelined against the scoring: copy_stream moves Q_obs, then
 * K one layer at a time into the caller's device staging buffers q_dev / k_dev
 * (layouts as for kvc_score), and every layer is scored on `stream` as soon
 * as its keys have landed; V is never copied -- kvc_compact reads only the
 * kept rows through the device's mapping of v_host.  q_host and k_host must
 * be pinned (page-locked) for the copies to be asynchronous; v_host must be
 * pinned and mapped for the device (cudaHostAlloc, or cudaHostRegister with
 * cudaHostRegisterMapped), else KVC_ERR_INVALID_ARG.  copy_stream must differ
 * from stream.  Outputs, capacities and the workspace are those of the four
 * calls it makes (see them); the call is asynchronous on both streams, and
 * the host buffers must stay valid until `stream` has finished.  A call's
 * copies wait only for the compaction of the previous call on the same
 * staging buffers (their last read), so reading the outputs back overlaps
 * with the next prompt's copies.  Events: one per layer plus two, per staging
 * buffer k_dev and device, created on first use and kept (up to 64 idle sets;
 * beyond that the least recently used idle set is destroyed after the host
 * has waited for its last call).  Calls with distinct staging buffers may run
 * concurrently from any threads; a call whose k_dev is in use by a call still
 * being issued on another thread returns KVC_ERR_INVALID_ARG. */
int kvc_compress_host(const kvc_shape *shape, const void *q_host, const void *k_host,
                      const void *v_host, void *q_dev, void *k_dev, uint32_t mass_num,
                      uint32_t mass_den, int64_t total_budget, int32_t layer_floor, int32_t k_max,
                      float *scores, int32_t *mba, int32_t *budget, int32_t *idx, void *k_out,
                      void *v_out, int64_t out_rows, void *ws, size_t ws_bytes, cudaStream_t stream,
                      cudaStream_t copy_stream);

/* a2 + a3 -- ZigZagKV budgets.
 * mba[l][k] = smallest m with mass_den * (sum of the m largest u) >=
 *             mass_num * (sum of all u), u_j = floor(scores[l][k][j] * 2^56),
 *             over all T tokens (0 for an all-zero head);
 * budget[l] = layer_floor + largest-remainder share of
 *             (total_budget - L*layer_floor) by S_l = sum_k mba[l][k]
 *             (equal shares if every S_l is 0), remainder ties to the lower
 *             layer, then capped at T-W with the excess re-split over the
 *             layers still below T-W until none exceeds it.  If total_budget
 *             >= L*(T-W) every layer gets T-W.
 * Requires 0 <= layer_floor <= T-W, total_budget >= L*layer_floor,
 * 0 < mass_den, mass_num <= mass_den, L <= 1024 (KVC_ERR_UNSUPPORTED
 * otherwise).  Scores must lie in [0,1] (-0.0 counts as 0) and sum to at
 * most 16 per head (KVC_DEV_BAD_SCORE otherwise).  One launch: the last
 * head to finish computes the budgets, counting finished heads in a word of
 * the workspace header that is zero between calls (kvc_workspace_init zeroes
 * it), so the workspace of a call in flight must not serve another. */
int kvc_mba_budget(const kvc_shape *shape, const float *scores, uint32_t mass_num,
                   uint32_t mass_den, int64_t total_budget, int32_t layer_floor,
                   int32_t *mba, int32_t *budget, void *ws, size_t ws_bytes,
                   cudaStream_t stream);

/* a4 -- per-head top-K of the prefix.  For head (l,k) keep
 * n_l = min(max(budget[l],0), T-W) prefix positions j < T-W with the largest
 * scores, ties to the lower position, written ascending to idx[l][k][0..n_l).
 * budget is a DEVICE array (e.g. from kvc_mba_budget, or filled by the
 * caller with a uniform SnapKV budget).  n_l > k_max sets KVC_DEV_BAD_BUDGET
 * and keeps only k_max. */
int kvc_topk_select(const kvc_shape *shape, const float *scores, const int32_t *budget,
                    int32_t k_max, int32_t *idx, void *ws, size_t ws_bytes,
                    cudaStream_t stream);

/* Optional variant of a3/a4 -- per-head budgets inside a layer (blog post
 * "ZigZagKV, KVCache 80% compression near-lossless": memory should follow
 * how many tokens each attention head needs, and in "ZigZagKV token
 * selection" each head's K follows its quota).  For every layer l the
 * H_kv * min(max(budget[l],0), T-W) prefix tokens are split over its heads in
 * proportion to mba[l][k] by the largest-remainder rule (ties to the lower
 * head, equal shares if the layer's MBAs are all zero, no per-head minimum),
 * each head capped at T-W with the excess re-split over the uncapped heads.
 * mba [L][H_kv] and budget [L] are DEVICE arrays (kvc_mba_budget's
 * outputs); head_budget [L][H_kv] int32 is written.  H_kv <= 1024. */
int kvc_head_budget(const kvc_shape *shape, const int32_t *mba, const int32_t *budget,
                    int32_t *head_budget, void *ws, size_t ws_bytes, cudaStream_t stream);

/* kvc_topk_select with one budget per head: head (l,k) keeps
 * min(max(head_budget[l][k],0), T-W) positions (device array [L][H_kv]). */
int kvc_topk_select_heads(const kvc_shape *shape, const float *scores, const int32_t *head_budget,
                          int32_t k_max, int32_t *idx, void *ws, size_t ws_bytes,
                          cudaStream_t stream);

/* Optional variant of a4 -- threshold selection with the recent window (the
 * ZigZagKV post, section "SnapKV": scores above a threshold mark the
 * important tokens; "NVIDIA AI presents KVzap": low-score entries are dropped
 * and a sliding window of recent tokens is kept, so every head keeps as many
 * tokens as its context needs).  Per head, every prefix position j < T-W
 * with scores[l][k][j] >= tau (fp32 compare) is written ascending to
 * idx[l][k][0..); counts[l][k] (int32, device) receives how many there are.
 * At most k_max are written; a head with more sets KVC_DEV_BAD_BUDGET.
 * tau must not be NaN.  Pass idx/counts to kvc_compact_heads. */
int kvc_threshold_select(const kvc_shape *shape, const float *scores, float tau, int32_t k_max,
                         int32_t *idx, int32_t *counts, void *ws, size_t ws_bytes,
                         cudaStream_t stream);

/* kvc_compact with one count per head: head (l,k) contributes
 * n = min(max(counts[l][k],0), T-W, k_max) rows idx[l][k][0..n), then its W
 * window rows; heads follow each other in (l, k) order, so head (l,k) starts
 * at row sum over earlier heads of (n + W).  counts is a DEVICE array
 * [L][H_kv] (kvc_head_budget's or kvc_threshold_select's output). */
int kvc_compact_heads(const kvc_shape *shape, const void *k, const void *v, const int32_t *idx,
                      const int32_t *counts, int32_t k_max, void *k_out, void *v_out,
                      int64_t out_rows, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Optional step before a4 -- SnapKV pooling of the prefix scores (blog post
 * "ZigZagKV, KVCache 80% compression near-lossless", section "SnapKV": the
 * scores are pooled in 1D so that a kept token's neighbours are kept with
 * it; the post gives neither the kernel's size nor its type).  For every
 * head and prefix position j < T-W, over the in-range positions
 * t in [max(0, j-kernel/2), min(T-W-1, j+kernel/2)]:
 *   mode 0: pooled[j] = their mean (sum / their count, not / kernel);
 *   mode 1: pooled[j] = their maximum.
 * Window positions are copied unchanged.  kernel must be odd, 1..255
 * (above 255: KVC_ERR_UNSUPPORTED); each mean is summed left to right in
 * fp32.  pooled has the layout of scores and must not alias it; pass it to
 * kvc_topk_select in place of scores (MBA stays on the raw scores).  The
 * workspace is only validated (header size), not used. */
int kvc_pool_scores(const kvc_shape *shape, const float *scores, int32_t kernel, int32_t mode,
                    float *pooled, void *ws, size_t ws_bytes, cudaStream_t stream);

/* a5 -- compaction.  Gathers, for every head, rows idx[l][k][0..n_l) and then
 * the W window rows T-W..T-1 of k and v into k_out / v_out (packed layout
 * above).  out_rows is the capacity of each output in rows of D elements;
 * the rows needed are H_kv * sum_l (n_l + W).  k, v, k_out and v_out must be
 * 16-byte aligned. */
int kvc_compact(const kvc_shape *shape, const void *k, const void *v, const int32_t *idx,
                const int32_t *budget, int32_t k_max, void *k_out, void *v_out,
                int64_t out_rows, void *ws, size_t ws_bytes, cudaStream_t stream);

/* a6 -- ThinK magnitude pruning of the compacted keys.  keep =
 * kvc_keep_channels(lambda, D).  Per head: M_d = sum over its n_l kept
 * prefix rows of k_out[r][d]^2 (accumulated in a float-float pair, about 44
 * significant bits), the `keep` channels with the largest M_d (ties to the
 * lower d) are written ascending to chan, and those channels of the prefix
 * rows are copied to k_pruned (packed layout above; pruned_elems is its
 * capacity in elements).  Window rows stay full width in k_out. */
int kvc_channel_prune(const kvc_shape *shape, const void *k_out, const int32_t *budget,
                      double lambda, int32_t *chan, void *k_pruned, int64_t pruned_elems,
                      void *ws, size_t ws_bytes, cudaStream_t stream);

/* Optional variant of a6 -- ThinK's query-driven key-channel criterion
 * ("ThinK: Thinner Key Cache by Query-Driven Pruning", sections "Greedy
 * algorithm" and "Observation window": channel j scores the Frobenius norm of
 * Q[-S_obs:, j] K[:, j]^T).  Same outputs and layouts as kvc_channel_prune;
 * channels are ranked by (sum over the window query rows of q[d]^2) *
 * (sum over the n_l kept prefix rows of k_out[r][d]^2) -- the square of that
 * norm -- instead of the key magnitude alone.  With grouped-query attention
 * the query column of KV head k stacks the W window rows of its G query heads
 * (q_obs [L][H_q][W][D], dtype of the shape).  Both sums are float-float
 * (about 44 significant bits); ties go to the lower channel. */
int kvc_channel_prune_query(const kvc_shape *shape, const void *q_obs, const void *k_out,
                            const int32_t *budget, double lambda, int32_t *chan, void *k_pruned,
                            int64_t pruned_elems, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Optional variant of a6 for the VALUE cache -- THINKV ("ThinK: Thinner Key
 * Cache by Query-Driven Pruning", appendix "Value cache pruning strategy":
 * channel j of a head's value cache scores the norm of column j of the window
 * queries' attention output, || softmax(Q_obs K^T / sqrt(D)) V[:, j] ||, and
 * the top floor((1-lambda) D) channels are kept).  Per head (l, k):
 *   value_scores[l][k][j] = sum over the G*W window rows r of o_r[j]^2,
 *   o_r = sum over the keys t row r sees (t <= T-W+w, as in kvc_score) of
 *         softmax_t(q_r . k_t / sqrt(D)) v_t
 * (the squared norm; rows stack the KV head's G query heads); the `keep`
 * channels with the largest value_scores (ties to the lower channel) are
 * written ascending to chan [L][H_kv][keep] and copied out of the n_l kept
 * prefix rows of v_out (kvc_compact's packed values) into v_pruned, packed
 * like k_pruned (layer l: [H_kv][n_l][keep]); window rows stay full width in
 * v_out.  q_obs, k, v are the full prompt tensors of kvc_score (16-byte
 * aligned); value_scores is an optional DEVICE output [L][H_kv][D] fp32
 * (NULL: kept in the workspace).  The call recomputes the window rows'
 * softmax normalisers itself (the first half of kvc_score's work) and then
 * forms o on the tensor cores for bf16 with head_dim 128 and G*W <= 512
 * (each probability as the sum of two bf16 terms, about 16 significant bits;
 * fp32 accumulation), on the CUDA cores in fp32 otherwise; the workspace is
 * kvc_workspace_size()'s.  Same as kvc_channel_prune_value_ex with flags 0. */
int kvc_channel_prune_value(const kvc_shape *shape, const void *q_obs, const void *k,
                            const void *v, const void *v_out, const int32_t *budget, double lambda,
                            float *value_scores, int32_t *chan, void *v_pruned,
                            int64_t pruned_elems, void *ws, size_t ws_bytes, cudaStream_t stream);

/* kvc_channel_prune_value with flags.  KVC_VALUE_REUSE_SCORE_STATS: take the
 * window rows' softmax normalisers from the workspace, where the most recent
 * kvc_score on it over the same shape, q_obs and k (and the same kernel
 * choice, on the same device) left them, instead of recomputing them -- one
 * pass of the score's two fewer when THINKV follows the default path.  The
 * library keeps a host-side record per workspace of the last such call (per
 * process; replaced by the next kvc_score or kvc_channel_prune_value on the
 * workspace, dropped by kvc_score_keyformer and kvc_workspace_init, whose
 * statistics differ) and returns KVC_ERR_INVALID_ARG, launching nothing, when
 * there is none that matches.  The caller guarantees that q_obs and k were not
 * rewritten since and that the kvc_score work is ordered before this call on
 * the device (the same stream, or an event).  Results are identical to the
 * call without the flag.  Other flag bits: KVC_ERR_INVALID_ARG. */
#define KVC_VALUE_REUSE_SCORE_STATS 0x1u
int kvc_channel_prune_value_ex(const kvc_shape *shape, const void *q_obs, const void *k,
                               const void *v, const void *v_out, const int32_t *budget,
                               double lambda, float *value_scores, int32_t *chan, void *v_pruned,
                               int64_t pruned_elems, uint32_t flags, void *ws, size_t ws_bytes,
                               cudaStream_t stream);

/* floor((1 - lambda) * head_dim) computed in double; 0 if lambda is outside
 * [0,1). */
int32_t kvc_keep_channels(double lambda, int32_t head_dim);

const char *kvc_status_string(int status);

/* Message for the last error returned on the calling thread ("" if none). */
const char *kvc_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KVC_H */
