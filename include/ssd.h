/*
 * ssd.h -- C ABI of the GB300 (sm_103a) speculation-round library.
 *
 * One batched round of speculative-speculative decoding with the Saguaro
 * algorithm, as the following web pages describe it:
 *   [A] 機器之心 article "全球最強推理引擎還快2倍，斯坦福、普林斯頓破解大模型串行魔咒",
 *       section "SSD 如何實現草擬與驗證并行？".
 *   [B] technical summary "超越传统SD：SSD框架全异步解码实现4.7倍平均加速",
 *       sections "投机解码的瓶颈与 SSD 的核心机制", "Saguaro 算法：解决异步推测的三大挑战"
 *       (part 1 "验证结果预测与缓存拓扑优化", part 2 "操纵残差分布", part 3
 *       "大 Batch 下的退避策略") and
 *       "工程优化与系统表现".
 * The pages' formulas did not survive extraction; where a call fills a gap
 * the reading is stated at the call.
 *
 * Conventions shared by every call
 * --------------------------------
 * Memory.   Every pointer is caller-owned DEVICE memory unless marked "host".
 *           The library allocates nothing: calls that need scratch take a
 *           caller-provided workspace `ws` of at least the size the matching
 *           *_workspace_size() call returns.
 * Streams.  Every call only enqueues work on stream `s` (0 = legacy default)
 *           and returns without synchronising.
 * Errors.   Arguments that can be checked on the host are checked before any
 *           launch; a failed check returns SSD_ERR_INVALID_ARG (meaningless
 *           argument), SSD_ERR_UNSUPPORTED (valid but outside the supported
 *           shapes/alignments) or SSD_ERR_WORKSPACE (workspace too small) and
 *           launches nothing.  A launch failure returns SSD_ERR_CUDA.  Data
 *           problems only the device can see set bits (SSD_FLAG_*) in the
 *           caller's `status` word with an atomic OR and take the documented
 *           path; no kernel traps or asserts.  The library never clears
 *           `status`: the caller zeroes it before the calls it wants to watch.
 * Logits.   [B, K+1, V] per tensor, element (b, r, i) at
 *           base + b*seq_stride + r*row_stride + i (strides in elements);
 *           row r holds position j = r + 1.  dtype fp32 or bf16.  The base
 *           address and both strides (in bytes) must be multiples of 16;
 *           V may be any positive size.  Supported: 0 <= K <= 16,
 *           0 <= F_k <= min(V, 256), 1 <= V, and rows of at most 128
 *           chunks of 32 KiB (V*elem <= 4 MiB: V <= 2^21 in bf16).
 * Temperature T >= 0; T = 0 is the greedy limit (one-hot distributions at the
 *           argmax, lowest index on ties).  Saguaro's C must lie in (0, 1].
 * Uniforms  are inputs (the caller draws them, e.g. from a counter-based
 *           generator); each must lie in [0, 1).
 * Draws     use the inverse CDF in vocabulary order: the smallest i with
 *           sum_{k<=i} w_k > u * sum_k w_k.
 * Ties      between equal logits rank the lower index first (argmax, top-F).
 */
#ifndef SSD_GB300_H
#define SSD_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *ssd_stream_t; /* a cudaStream_t */

typedef enum {
  SSD_OK = 0,
  SSD_ERR_INVALID_ARG = 1,
  SSD_ERR_UNSUPPORTED = 2,
  SSD_ERR_WORKSPACE = 3,
  SSD_ERR_CUDA = 4
} ssd_status_t;

typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype_t;

/* status-word bits (device uint32[1], OR-ed by kernels) */
#define SSD_FLAG_BAD_TOKEN 1u     /* a draft token outside [0, V): that test rejects       */
#define SSD_FLAG_ZERO_RESIDUAL 2u /* residual without mass: the bonus is drawn from p_{a+1} */
#define SSD_FLAG_WAIT_TIMEOUT 4u  /* a bounded on-device wait gave up; outputs are invalid  */
#define SSD_FLAG_BAD_OUTCOME 8u   /* lookup: accept count outside [0, K]: treated as a miss */
#define SSD_FLAG_BAD_TREE 16u     /* attention: parent[m] outside [-1, m-1]: path ends there */
#define SSD_FLAG_BAD_BLOCK 32u    /* attention: block id outside [0, num_blocks): keys hidden */
#define SSD_FLAG_BAD_PREFIX 64u   /* attention: prefix_len < 0 or prefix_len + N > 16 maxb:  */
                                  /* keys past the block table are hidden                   */
#define SSD_FLAG_BAD_HISTORY 128u /* backup: hist_len outside [0, hist_stride]: taken as 0  */
#define SSD_FLAG_BAD_RATE 256u    /* plan: p_hit outside [0, 1] or e_hit < 0 / not finite:  */
                                  /* clamped into [0, 1], taken as 0                        */

/* Human-readable name of a status code (static string). */
const char *ssd_status_string(ssd_status_t st);

/*
 * Fan-out split of a speculation budget over depths k = 0..K [B, part 1: the
 * optimal F_k follows a truncated geometric series; more branches at shallow
 * depths].  Reading: weights r^k, F_k = max(1, floor(budget r^k / sum_j r^j));
 * a shortfall is handed out one unit at a time by descending fractional part
 * (ties: smaller k), an excess taken from the largest F_k > 1 (ties: larger k).
 * budget >= K+1, 0 < r <= 1, 0 <= K <= 16.  F_out: host int32[K+1].
 * Host-only; returns SSD_ERR_INVALID_ARG on bad arguments.
 */
ssd_status_t ssd_fanout_split(int budget, int K, double r, int32_t *F_out);

/*
 * Workspace bytes the vocabulary calls (ssd_saguaro_sample, ssd_verify,
 * ssd_predict_outcomes, ssd_round) need for B sequences of K+1 rows of V
 * logits of type dt with fan-out F (host int32[K+1]).  Returns 0 for
 * unsupported arguments.  The workspace needs no initialisation: a
 * verification call publishes each pair's record through 64-bit ready words
 * in it (a fixed 64-bit value, never written by anything else) and sets them
 * back to 0 before it completes.  Calls that share a workspace must not
 * overlap on the GPU.
 */
size_t ssd_workspace_size(int B, int K, int V, ssd_dtype_t dt, const int32_t *F);

/*
 * Saguaro draft sampling sigma_{F,C} [B, part 2 "操纵残差分布": the draft's
 * most likely tokens are down-weighted by C so that, when C shrinks, the
 * residual puts more mass on them and the bonus token tends to land in the
 * cache].  Reading: for position j = 1..K, S_j = the top-F_{j-1} tokens of
 * draft row j by raw logit; q_j = softmax(z^d_j / T);
 *   q'_j(i) = q_j(i) c_i / (1 - (1 - C) sum_{k in S_j} q_j(k)),  c_i = C on S_j, 1 off it;
 *   d_j = inverse-CDF draw from q'_j with u_draft[b, j-1].
 * draft: logits as above (rows 0..K-1 are read).  u_draft: [B, K] fp32.
 * d_out: [B, K] int32.  qd_out: [B, K] fp32 = q'_j(d_j), or NULL.
 */
ssd_status_t ssd_saguaro_sample(const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                                int64_t row_stride, int B, int K, int V, const int32_t *F,
                                float C, float T, const float *u_draft, int32_t *d_out,
                                float *qd_out, uint32_t *status, void *ws, size_t ws_bytes,
                                ssd_stream_t s);

/*
 * Lossless verification of K draft tokens per sequence [A: the target checks
 * the K draft tokens in one parallel pass, accepts a prefix of them and
 * samples one bonus token after the accepted ones, so the output follows the
 * target distribution exactly; B: the residual distribution "p_target -
 * p_draft"].  Reading: p_j = softmax(z^t_j / T); q'_j = sigma_{F_{j-1},C}(q_j)
 * (the distribution the draft sampled from, see ssd_saguaro_sample);
 *   for j = 1..K: accept d_j iff u_acc[b, j-1] * q'_j(d_j) < p_j(d_j);
 *   stop at the first rejection; a = number accepted;
 *   a < K: bonus ~ max(0, p_{a+1} - q'_{a+1}) renormalised (u_bonus[b]); a
 *          residual without mass draws from p_{a+1} and sets ZERO_RESIDUAL;
 *   a = K: bonus ~ p_{K+1}.
 * target, draft: logits (same dtype and strides).  d: [B, K] int32 (an id
 * outside [0, V) sets BAD_TOKEN and rejects).  u_acc: [B, K]; u_bonus: [B].
 * Outputs: accept_len [B]; out_tokens [B, K+1] = d_1..d_a, bonus, then -1;
 * bonus [B]; accept_prob [B, K] = P(u q' < p) = min(1, p/q') for every j (1
 * when q' = 0 < p, 0 when p = q' = 0 or d_j is invalid), or NULL; resid_mass
 * [B] = total mass of the residual used (1 after full acceptance), or NULL.
 * near_ties [1] (or NULL): the number of near-ties is ADDED to it (like
 * status, the caller zeroes it).  A near-tie is a decision that fp32 and
 * exact arithmetic may take differently, counted so that a caller can report
 * how many of its outcomes rest on one: an acceptance test actually taken (positions 1..a+1) with |u - p/q'| < 1e-6, or an
 * inverse-CDF draw whose target u*W lies within 1e-6*W of an edge of the
 * chosen token's bin (including the draws the kernel resolves by its
 * rounding fallback).  Greedy (T = 0) decisions are exact and never count.
 */
ssd_status_t ssd_verify(const void *target, const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                        int64_t row_stride, int B, int K, int V, const int32_t *F, float C, float T,
                        const int32_t *d, const float *u_acc, const float *u_bonus,
                        int32_t *accept_len, int32_t *out_tokens, int32_t *bonus,
                        float *accept_prob, float *resid_mass, uint32_t *near_ties,
                        uint32_t *status, void *ws, size_t ws_bytes, ssd_stream_t s);

/*
 * Verification-outcome prediction [A: the draft predicts the bonus token from
 * its most likely logits; B part 1: the outcome space has ~V^K points, so a
 * budget is spread as fan-out F_k over depths].  For depth k = 0..K the guesses
 * are the top-F_k tokens of draft row k+1 (value descending, index ascending):
 * guess[b, off_k + i], off_k = F_0 + ... + F_{k-1}; guess_q = q_{k+1} of each
 * guess (softmax(z / T); one-hot at T = 0), or NULL.
 */
ssd_status_t ssd_predict_outcomes(const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                                  int64_t row_stride, int B, int K, int V, const int32_t *F,
                                  float T, int32_t *guess, float *guess_q, uint32_t *status,
                                  void *ws, size_t ws_bytes, ssd_stream_t s);

/*
 * ssd_verify without a caller workspace.  For callers that cannot allocate
 * device memory themselves -- for example a plugin running inside another
 * framework that owns every device allocation and forbids new ones in its
 * execution path, or a plain C program linked only against this library with
 * no allocator of its own -- this entry point takes its scratch from a fixed
 * array compiled into the library (ssd_verify_noalloc_max_bytes() bytes,
 * 8 MiB; one copy on every GPU that loads the library, kept until the process
 * exits).  The pages describe no such variant; it exists only for those
 * callers.  Arguments, outputs and semantics are those of ssd_verify; the
 * caller still provides every input and output buffer.
 *   - Allocates nothing: no cudaMalloc / cudaFree / allocating library call.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture on the device.
 *   - Argument errors map exactly as in ssd_verify; a batch whose scratch
 *     (ssd_workspace_size) exceeds the array then returns SSD_ERR_WORKSPACE
 *     and launches nothing.
 *   - Every call shares the one array, and it keeps the previous call's
 *     contents (nothing in it needs to start at zero: each call writes every
 *     scratch record before reading it).  Calls whose work overlaps on the GPU
 *     (different streams, or different host threads) race on it: serialise
 *     them, e.g. on one stream.
 */
size_t ssd_verify_noalloc_max_bytes(void);
ssd_status_t ssd_verify_noalloc(const void *target, const void *draft, ssd_dtype_t dt,
                                int64_t seq_stride, int64_t row_stride, int B, int K, int V,
                                const int32_t *F, float C, float T, const int32_t *d,
                                const float *u_acc, const float *u_bonus, int32_t *accept_len,
                                int32_t *out_tokens, int32_t *bonus, float *accept_prob,
                                float *resid_mass, uint32_t *near_ties, uint32_t *status,
                                ssd_stream_t s);

/*
 * Speculation-cache lookup keyed by the verification outcome (a, b) [B,
 * "投机解码的瓶颈与 SSD 的核心机制": once verification returns, one cache lookup
 * decides whether pre-speculated tokens are ready].  Hit iff bonus b is among
 * the F_a guesses of depth a: slot[b] = off_a + rank, else -1.  next_tokens
 * [B, K] = payload[b, slot, 0..K-1] on a hit and -1 on a miss (NULL to skip;
 * payload [B, sumF, K] may then be NULL).  hits[0] = number of hits (written,
 * not accumulated).  An accept count outside [0, K] is a miss (BAD_OUTCOME).
 */
ssd_status_t ssd_cache_lookup(const int32_t *guess, const int32_t *payload, int B, int K,
                              const int32_t *F, const int32_t *accept_len, const int32_t *bonus,
                              int32_t *slot, int32_t *next_tokens, uint32_t *hits,
                              uint32_t *status, ssd_stream_t s);

/*
 * The whole round in one call: Saguaro sampling of d_1..d_K, verification,
 * outcome prediction and cache lookup, with every logit row read from HBM
 * once.  Equivalent to ssd_saguaro_sample -> ssd_verify ->
 * ssd_predict_outcomes -> ssd_cache_lookup on the same arguments; every
 * output pointer except the required d_out, accept_len, out_tokens, bonus may
 * be NULL (guess is needed when slot, next_tokens or hits is given).
 * near_ties counts as in ssd_verify, plus the K Saguaro draws of d_1..d_K.
 */
ssd_status_t ssd_round(const void *target, const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                       int64_t row_stride, int B, int K, int V, const int32_t *F, float C, float T,
                       const float *u_draft, const float *u_acc, const float *u_bonus,
                       const int32_t *payload, int32_t *d_out, float *qd_out, int32_t *accept_len,
                       int32_t *out_tokens, int32_t *bonus, float *accept_prob, float *resid_mass,
                       int32_t *guess, float *guess_q, int32_t *slot, int32_t *next_tokens,
                       uint32_t *hits, uint32_t *near_ties, uint32_t *status, void *ws,
                       size_t ws_bytes, ssd_stream_t s);

/*
 * ssd_round for back-to-back rounds of independent batches: its statistics
 * pass may start while the kernels of the previous call on the stream are
 * still finishing (their verification tail is a chain of dependent steps at
 * low occupancy), so consecutive rounds overlap.  Arguments, outputs and
 * semantics are those of ssd_round.  The caller guarantees that nothing this
 * call reads or writes -- logits, uniforms, payload, outputs, status and the
 * workspace -- is written or read by the kernel launched just before it on
 * the stream (e.g. the previous round runs on other buffers and the logits
 * were produced earlier).  A round's own kernels still run in order.
 */
ssd_status_t ssd_round_pipelined(const void *target, const void *draft, ssd_dtype_t dt,
                                 int64_t seq_stride, int64_t row_stride, int B, int K, int V,
                                 const int32_t *F, float C, float T, const float *u_draft,
                                 const float *u_acc, const float *u_bonus, const int32_t *payload,
                                 int32_t *d_out, float *qd_out, int32_t *accept_len,
                                 int32_t *out_tokens, int32_t *bonus, float *accept_prob,
                                 float *resid_mass, int32_t *guess, float *guess_q, int32_t *slot,
                                 int32_t *next_tokens, uint32_t *hits, uint32_t *near_ties,
                                 uint32_t *status, void *ws, size_t ws_bytes, ssd_stream_t s);

/*
 * Exact analytics of a round, before any uniform is drawn [B,
 * "投机解码的瓶颈与 SSD 的核心机制": the acceptance rate alpha; B, "Saguaro 算法"
 * part 1: the chance that the bonus token lands among the cached guesses is
 * what the fan-out is chosen for].  With the logit rows fixed, a draft token
 * d_j ~ q'_j is accepted with probability sum_i min(p_j(i), q'_j(i)), so per
 * sequence b (arguments as in ssd_round; F also names the guess lists):
 *   alpha    [B, K]  = sum_i min(p_j(i), q'_j(i))                 (or NULL)
 *   resid_w  [B, K]  = W_j = sum_i max(0, p_j(i) - q'_j(i))        (or NULL)
 *   p_accept [B, K+1]: P(a = k) = prod_{j<=k} alpha_j * W_{k+1}, P(a = K) = prod alpha_j
 *   hit_mass [B, K+1]: P(bonus among the F_k guesses of depth k | a = k); the
 *            bonus follows r_{k+1} / W_{k+1} (p_{k+1} when W_{k+1} = 0) for
 *            k < K and p_{K+1} for k = K                         (or NULL)
 *   hit_rate [B] = sum_k P(a = k) hit_mass_k  (the exact cache hit rate)
 *   exp_tokens [B] = sum_k P(a = k) (k + 1)  (tokens emitted per round)
 * All fp32.  T = 0 gives the greedy limit (alpha_j = 1 when both argmaxes
 * agree).  The statistics pass reads every row once; the sums of min and
 * max(0, p - q') then read the K row pairs again (from L2 when the batch
 * fits).  The fan-out may then be re-split with ssd_fanout_split(budget, K,
 * r) at a measured ratio, e.g. the batch's mean alpha.
 */
ssd_status_t ssd_round_analytics(const void *target, const void *draft, ssd_dtype_t dt,
                                 int64_t seq_stride, int64_t row_stride, int B, int K, int V,
                                 const int32_t *F, float C, float T, float *alpha, float *resid_w,
                                 float *p_accept, float *hit_mass, float *hit_rate,
                                 float *exp_tokens, uint32_t *status, void *ws, size_t ws_bytes,
                                 ssd_stream_t s);

/*
 * Timing hook for profiling: while set (both non-NULL cudaEvent_t handles),
 * every vocabulary call records `before` and `after` on its stream around its
 * HBM statistics pass (the dominant kernel), so a caller can time that kernel
 * inside a real round with cudaEventElapsedTime.  Process-wide, not
 * thread-safe; pass NULL, NULL to clear.  Returns SSD_ERR_INVALID_ARG when
 * exactly one handle is NULL.  Not part of the method: diagnostics only.
 */
ssd_status_t ssd_set_timing_events(void *before, void *after);

/*
 * Work trace for profiling: while set, every vocabulary call writes, for each
 * CTA of its kernels, eight 64-bit words into `buf` (device memory): first
 * the statistics kernel's CTAs (grid order: chunk, row slot, sequence), then
 * the pair kernel's (sequence-major, one per row pair), then the residual
 * kernel's.  Word 0 = (SM << 48 | kind << 40 | sequence << 20 | index), kind
 * 0 statistics (index: row slot * chunks + chunk), 1 pair (index: position),
 * 2 residual unit (index: unit); words 1-7 = %globaltimer marks in ns (0 =
 * not reached): start, after the wait for the previous kernel, then per
 * kind -- pair: records staged, rows merged, draw of d done, top-F done,
 * end; residual: records read, unit pass done, ticket taken, bonus drawn,
 * end (statistics CTAs mark only their start; the pair kernel's wait mark
 * shows when the statistics grid has completed).  Calls whose CTAs do not
 * fit in `bytes`, or with more than 65535 sequences, write nothing.
 * Process-wide, not thread-safe; NULL clears.  Diagnostics only.
 */
ssd_status_t ssd_set_trace(void *buf, size_t bytes);

/*
 * Tree-masked decode attention over a paged bf16 KV cache, so that the draft
 * decodes every branch of the speculation tree in one forward pass [B,
 * "工程优化与系统表现": a custom sparse attention mask].
 *   q [B, Nq, Hq, d] bf16; k_cache, v_cache [num_blocks, Hkv, 16, d] bf16
 *   (a block holds 16 consecutive positions of one KV head); block_table
 *   [B, maxb] int32; prefix_len [B] int32; parent [B, N] int32 (-1 = the
 *   prefix end).  Node m of sequence b sits at logical position
 *   prefix_len[b] + m (its K/V already in the cache); query row i is node
 *   N - Nq + i.  Row i of head h attends to every prefix position and to the
 *   nodes on its ancestor-or-self path, reading KV head h / (Hq / Hkv):
 *     out = softmax(scale * q k^T + mask) v   (fp32 accumulation, bf16 out),
 *     lse = natural log-sum-exp of the visible scores (fp32 [B, Nq, Hq], or NULL).
 * Supported: d in {64, 128}, Hq % Hkv == 0, Hq / Hkv <= 16, 1 <= Nq <= N <= 128,
 * prefix_len[b] + N <= 16 * maxb.  parent[m] outside [-1, m-1] ends the path
 * (BAD_TREE); a block id outside [0, num_blocks) hides its keys (BAD_BLOCK);
 * prefix_len[b] < 0 or prefix_len[b] + N > 16 * maxb sets BAD_PREFIX and the
 * keys past the table stay hidden (a negative prefix counts as 0).
 * Workspace: ssd_attention_workspace_size() bytes (256-byte aligned) let a
 * long key range be split across CTAs and merged afterwards.  ws may be NULL
 * or short: the keys are then not split, which gives the same result but can
 * be many times slower when few query rows meet a long prefix.
 */
size_t ssd_attention_workspace_size(int B, int Nq, int Hq, int Hkv, int d, int max_prefix);
ssd_status_t ssd_branch_attention(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_table, int maxb, int64_t num_blocks,
                                  const int32_t *prefix_len, const int32_t *parent, int B, int N,
                                  int Nq, int Hq, int Hkv, int d, float scale, void *out,
                                  float *lse, uint32_t *status, void *ws, size_t ws_bytes,
                                  ssd_stream_t s);

/*
 * Speculation-cache fill by branch decode [B, "投机解码的瓶颈与 SSD 的核心机制": while
 * the target verifies, the draft pre-speculates a continuation for every
 * predicted outcome (k, guess); "工程优化与系统表现": all F_k branches are
 * decoded in one forward pass with a custom sparse attention mask].
 * Reading (the pages give no step loop): a branch is one cache slot s
 * (0 <= s < S = sum_k F_k, slot-ordered as in ssd_cache_lookup); its chain
 * starts at the guessed bonus token and grows by one token per decode step
 * t = 0..Kp-1.  The Kp drawn tokens are the slot's payload: the next round's
 * draft tokens d_1..d_Kp, so step t draws with sigma_{F_t, C} (draft position
 * j uses F_{j-1}, as in ssd_saguaro_sample).  One step is
 *   ssd_kv_append     (the fed tokens' key/value rows into the paged cache),
 *   ssd_branch_attention (queries: the fed nodes; parent: the branch tree),
 *   the draft's other layers (not part of this library), then
 *   ssd_fill_sample   (the next token of every branch, into payload[:, :, t]).
 *
 * ssd_fill_sample: logits [B, S, V] (row (b, s) at logits + (b*S + s) *
 * branch_stride elements; fp32 or bf16; 16-byte aligned base and stride);
 * every row is drawn as ssd_saguaro_sample draws one draft position, with
 * F = F_t and the uniform u[b, s]: tokens [B, S] (required), q_out [B, S] =
 * q'(token) (or NULL), and payload [B, S, Kp] column t (or NULL).  Workspace:
 * ssd_workspace_size(B*S, 1, V, dt, {F_t, 0}) bytes.  Limits as in
 * ssd_saguaro_sample; B*S < 2^31.
 */
ssd_status_t ssd_fill_sample(const void *logits, ssd_dtype_t dt, int64_t branch_stride, int B, int S,
                             int V, int F_t, float C, float T, const float *u, int t, int Kp,
                             int32_t *tokens, float *q_out, int32_t *payload, uint32_t *status,
                             void *ws, size_t ws_bytes, ssd_stream_t s);

/*
 * ssd_kv_append: k_new, v_new [B, S, Hkv, d] bf16 (the rows of the S tokens
 * fed this step) go to the paged caches [num_blocks, Hkv, 16, d] (the layout
 * of ssd_branch_attention) at logical position pos = prefix_len[b] + node0 + i
 * of sequence b: page block_table[b, pos / 16], slot pos % 16.  node0 is the
 * tree index of the step's first node (node m sits at prefix_len + m, as in
 * ssd_branch_attention).  A negative prefix or a position past the table sets
 * BAD_PREFIX, a page id outside [0, num_blocks) sets BAD_BLOCK; that row is
 * not written.  d a multiple of 8, at most 256; 16-byte aligned pointers.
 * One thread per 16-byte piece.
 */
ssd_status_t ssd_kv_append(const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                           const int32_t *block_table, int maxb, int64_t num_blocks,
                           const int32_t *prefix_len, int node0, int B, int S, int Hkv, int d,
                           uint32_t *status, ssd_stream_t s);

/*
 * Token-tree verification with several candidates per node [A, closing
 * paragraph: combining SSD with token-tree speculation is named as future
 * work; B, "投机解码的瓶颈与 SSD 的核心机制" and "Saguaro 算法" part 2: the
 * single-chain acceptance rule and the residual p_target - p_draft].
 * Reading (the pages give no tree rule): the children of a node were drawn
 * independently from the draft's q at that node; they are tested in index
 * order against r, which starts as p and becomes the normalised residual
 * max(0, r - q) / sum max(0, r - q) after each rejection; an accepted child
 * continues the walk from it; when no child is accepted the bonus is drawn
 * from r (inverse CDF, u_bonus).  The emitted tokens then follow the target
 * exactly, as in single-chain verification.
 *   logits  [B, N+1, V] per tensor (layout and alignment as for ssd_verify):
 *           row 0 the distributions after the prefix (the root), row m+1 those
 *           after tree node m;  p = softmax(target / T), q = softmax(draft / T)
 *           (T = 0: one-hot at the argmax, lowest index on ties).
 *   parent  [B, N] int32 in [-1, m-1] (-1: the root); tokens [B, N];
 *   u_acc   [B, N]: the uniform of node m's test (u * q(x) < r(x) accepts);
 *   u_bonus [B].
 * Outputs: accept_len [B] (accepted nodes), path [B, N] (their indices in
 * order, then -1), bonus [B], out_tokens [B, N+1] (the accepted tokens, the
 * bonus, then -1; or NULL), resid_mass [B] (the W of the last residual taken
 * at the final node, 1 when its r is p; or NULL).  A parent outside [-1, m-1]
 * sets BAD_TREE (that node is nobody's child); a token outside [0, V) sets
 * BAD_TOKEN (that child is skipped); a residual without mass sets
 * ZERO_RESIDUAL (r stays).  Supported: N <= 256, V * elem <= 512 KiB.
 * One thread-block cluster of ceil(V*elem / 64 KiB) CTAs per sequence; each
 * visited node's two rows are read from HBM once.
 */
ssd_status_t ssd_tree_verify(const void *target, const void *draft, ssd_dtype_t dt, int64_t seq_stride,
                             int64_t row_stride, int B, int N, int V, float T, const int32_t *parent,
                             const int32_t *tokens, const float *u_acc, const float *u_bonus,
                             int32_t *accept_len, int32_t *path, int32_t *bonus, int32_t *out_tokens,
                             float *resid_mass, uint32_t *status, ssd_stream_t s);

/*
 * Miss fallback [B, "Saguaro 算法" part 3 "大 Batch 下的退避策略": a sequence
 * whose outcome missed the speculation cache falls back to synchronous
 * speculation with a backup speculator, and one miss holds up the whole batch
 * for the backup's latency; beyond a batch size set by the hit rate and the
 * latencies a backup of almost no latency (random tokens or an n-gram model)
 * is the better choice].
 *
 * ssd_ngram_backup: the n-gram backup for the sequences that missed.  Reading
 * (the pages name the backup only): history row b is hist[b*hist_stride ..
 * + hist_len[b]) (int32 token ids, positions 0..L-1), s = its last n tokens;
 * the latest earlier occurrence m (the largest m with m + n <= L - 1 and
 * h[m..m+n) = s) proposes next_tokens[b, t] = h[m + n + t] for t < K while
 * m + n + t < L; every other position, and every position when s occurs
 * nowhere earlier or L < n + 1, takes the random-token backup
 * floor(u_rand[b, t] * V) (exactly: ((uint64)(u * 2^24) * V) >> 24; u is
 * clamped into [0, 1)).  n = 0 gives the random-token backup alone.
 *   slot [B]        the cache lookup's slot: rows with slot[b] >= 0 are hits
 *                   and are left untouched (NULL: every row missed).
 *   plan_best       device int32[1] from ssd_fallback_plan, or NULL: when it
 *                   equals random_option the history is not searched (the
 *                   random-token backup alone), so the policy runs without a
 *                   host round trip.
 *   next_tokens [B, K]  written for missed rows (the cache lookup writes -1
 *                   there).  match_pos [B] (or NULL) = m, -1 without a match,
 *                   -2 for a hit.
 * Supported: 0 <= n <= 32, 0 <= K <= 1024, V >= 1, hist_stride <= 2^30
 * (hist and hist_len may be NULL when n = 0; u_rand [B, K] fp32).  A copied
 * token outside [0, V) sets BAD_TOKEN and takes the random token instead;
 * hist_len[b] outside [0, hist_stride] sets BAD_HISTORY and counts as 0.
 * One CTA per sequence; a missed sequence scans its history backwards in
 * chunks of 4096 positions and stops at the first chunk holding a match.
 */
ssd_status_t ssd_ngram_backup(const int32_t *hist, int64_t hist_stride, const int32_t *hist_len,
                              int B, int n, int K, int V, const int32_t *slot,
                              const float *u_rand, const int32_t *plan_best, int random_option,
                              int32_t *next_tokens, int32_t *match_pos, uint32_t *status,
                              ssd_stream_t s);

/*
 * ssd_fallback_plan: the batch-level speedup model and the backup choice.
 * Reading (the pages' formula did not survive extraction; restated from [B,
 * "投机解码的瓶颈与 SSD 的核心机制"]: the primary speculator drafts for the
 * predicted outcomes while the target verifies, so a round whose outcome hits
 * costs max(T_v, T_p); a miss falls back to synchronous speculation with
 * backup o and holds the batch up for T_b[o]).  With independent hits of
 * probability p_hit[b] (e.g. ssd_round_analytics' hit_rate) and expected
 * tokens e_hit[b] per round after a hit (e.g. its exp_tokens), for each of the
 * nopt backups o (T_b[o] its latency, e_miss[o] the expected tokens of a round
 * after a miss):
 *   time[o]       = max(T_v, T_p) + (1 - prod_b p_hit[b]) * T_b[o]
 *   tokens[o]     = sum_b (p_hit[b] e_hit[b] + (1 - p_hit[b]) e_miss[o])
 *   throughput[o] = tokens[o] / time[o]
 *   speedup[o]    = throughput[o] / (sum_b e_hit[b] / (T_p + T_v))  (against
 *                   synchronous speculation with the primary)
 *   best[0]       = the o of largest throughput (lowest index on ties)
 * p_hit, e_hit: device fp32 [B]; T_v, T_p, T_b[nopt], e_miss[nopt]: host fp64
 * (times in any one unit); outputs device fp64 [nopt] and int32[1], each may
 * be NULL.  Sums and the product are taken in fp64.  Requires B >= 1,
 * 1 <= nopt <= 8, T_v, T_p >= 0 with T_v + T_p > 0, T_b and e_miss finite and
 * >= 0 (else SSD_ERR_INVALID_ARG / SSD_ERR_UNSUPPORTED).
 */
ssd_status_t ssd_fallback_plan(const float *p_hit, const float *e_hit, int B, double T_v,
                               double T_p, int nopt, const double *T_b, const double *e_miss,
                               double *time, double *tokens, double *throughput, double *speedup,
                               int32_t *best, uint32_t *status, ssd_stream_t s);

#ifdef __cplusplus
}
#endif

#endif /* SSD_GB300_H */
