/*
 * specverify.h -- C ABI of the GB300 speculative-decoding verification library.
 *
 * The library turns target and draft logits into verified tokens (token-level and block
 * verification, also with the vocabulary split across ranks, or straight from hidden states
 * through an output projection), drafts a block with DSpark's Markov head, and schedules how much
 * of each drafted block to verify.  Every call is one or more hand-written CUDA kernels for sm_103a launched on the
 * caller's stream.
 *
 * Conventions for every entry point
 *   - Pointers marked DEVICE are device pointers owned by the caller; HOST pointers are read
 *     synchronously during the call.  The library allocates no memory and keeps no state between
 *     calls.  Scratch memory is the caller's `workspace` (DEVICE, 256-byte aligned), sized by the
 *     matching *_workspace_bytes query; its contents need no initialisation and are clobbered.
 *     (spec_verify_token_noalloc is the one exception: its scratch is a fixed array inside the
 *     library.)
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are asynchronous: they
 *     return after launching; outputs are valid once the stream reaches that point.
 *   - Argument errors (bad sizes, NULL required pointers, misaligned rows, a too-small workspace)
 *     return SV_ERR_INVALID / SV_ERR_UNSUPPORTED synchronously and launch nothing.
 *   - Data errors found on the device (token id outside [0, V), NaN or +inf logits, an all -inf
 *     row, q(x) = 0 for the drafted token x, a drafted length outside [0, max_draft_len]) are
 *     written to the optional DEVICE word `status` (reset to SV_OK by each call; the first error
 *     found is kept).  Outputs are then undefined.  `status` is NULL -> data errors go unreported.
 *   - A device-side wait that exceeds its bound writes SV_ERR_TIMEOUT to `status`.
 *   - Logits may hold -inf (masked tokens); such tokens are never emitted.
 *   - Rows are `ld` elements apart; the row base addresses must be 16-byte aligned, i.e. the logit
 *     pointers 16-byte aligned and ld * sizeof(element) a multiple of 16.  V itself is arbitrary.
 *
 * Random numbers: uniforms come from Philox4x32-10 (Salmon et al., SC'11, "Parallel Random
 * Numbers: As Easy as 1, 2, 3") with key (lo32(seed), hi32(seed)); block(g, tag) is the output
 * for counter (g, position, lo32(request id), tag << 24 | (hi32(request id) & 0xFFFFFF)).
 * Every uniform is u = (n + 0.5) * 2^-23 for a 23-bit n (never 0 or 1):
 *   - the ACCEPT draw of a position: n = word 0 of block(0, ACCEPT) >> 9;
 *   - race entry v (vocabulary index) under tag T: n = (h << 7) | f, with h the 16-bit half v & 1
 *     (0: low) of word (v >> 1) & 3 of block(v >> 3, T) -- one block per 8 entries -- and f the
 *     top 7 bits of word v & 3 of block(v >> 2, T + 4).
 * Tags: DRAFT 0, ACCEPT 1, RESID 2, BONUS 3.  Positions are 1-based: drafted tokens at 1..gamma,
 * the bonus row at gamma + 1.
 * Every sample is an exponential race: x = argmax_x log w(x) - log(-log u_x), which draws x with
 * probability w(x) / sum(w) without a normalisation pass; equal keys go to the lower index.
 *
 * Sources (web pages, by title and section):
 *   "Speculative Decoding: The Same Distribution, Twice as Fast" §3 "The loop", §4 "The rule that
 *     makes it exact" (accept with min(1, p/q); correction from max(0, p - q) renormalised).
 *   "How much does a token cost", "On Speculative Sampling" (the same rule; Panels A-C) and "Block
 *     verification" (running target-to-draft ratio capped at one; longest passing prefix).
 *   "DeepSeek DSpark 详解" §03 (Markov head: a rank-256 low-rank transition from the previous
 *     sampled token corrects the parallel backbone's logits, left to right) and §04 (confidence
 *     head, prefix survival = product of conditional acceptance probabilities, sequential
 *     temperature scaling, maximise expected accepted tokens x SPS(B), early stop).
 *   "DSpark: DeepSeek's bet on speed that doesn't betray quality", "Verifying only what matters".
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID = 1,      /* invalid argument (returned synchronously) */
  SV_ERR_UNSUPPORTED = 2,  /* valid but unsupported argument (returned synchronously) */
  SV_ERR_CUDA = 3,         /* a CUDA runtime call failed (returned synchronously) */
  SV_ERR_BAD_INPUT = 4,    /* data error found on the device (written to *status) */
  SV_ERR_TIMEOUT = 5       /* a bounded device-side wait expired (written to *status) */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Largest drafted length per request accepted by the verify calls and the Markov head. */
#define SV_MAX_DRAFT_LEN 64

/* Human-readable name of a status code (static string). */
const char* sv_status_string(sv_status status);

/* Library build identifier (static string), e.g. for logs. */
const char* sv_version(void);

/* Failure-detection self test.  Runs one of the bounded device-side waits the kernels use on a
 * condition that never comes true -- which = 0: an mbarrier phase no thread completes; which = 1:
 * a shared-memory request-number word no thread publishes -- with a limit of `limit_us`
 * microseconds (1 .. 1000000) instead of the kernels' one second.  The wait gives up, writes
 * SV_ERR_TIMEOUT to the DEVICE word `status` (required; reset first) and the kernel returns, so the
 * context stays usable.  No page has a counterpart: it checks the library's own safety net. */
sv_status sv_selftest_wait(int32_t which, int32_t limit_us, int32_t* status, void* stream);

/* Kernel timing (diagnostic, off by default).  While enabled on the calling host thread, every
 * spec_verify_token / spec_verify_block call records CUDA events on its stream around each of its
 * kernels: [0] row streaming (all passes), [1] acceptance decisions, [2] correction / bonus race.
 * sv_profile_read waits for the events of the last profiled call and returns the three durations
 * in milliseconds.  The events belong to the library (created on first use, one set per host
 * thread); nothing is recorded while profiling is disabled.  A spec_verify_lmhead call records
 * [0] the statistics GEMM, [1] the decisions, [2] the race GEMM and the outputs. */
sv_status sv_profile_enable(int enable);
sv_status sv_profile_read(float* ms_out /* HOST [3] */);

/* ---------------------------------------------------------------------------------------------
 * Verification.
 *
 * Layout (all DEVICE unless noted).  Request r (0 <= r < B) drafted gamma_r = draft_len[r]
 * tokens.  Its target rows are target_row0[r] + 0 .. gamma_r (row i-1 scores position i, row
 * gamma_r is the bonus row) and its draft rows draft_row0[r] + 0 .. gamma_r - 1, all in units of
 * rows of `ld` elements of `dtype`.  Its drafted token at position i is
 * draft_tokens[draft_row0[r] + i - 1] (the token array is indexed like the draft rows).
 * `max_draft_len` (HOST value) bounds every gamma_r and sizes the workspace.
 * request_ids (nullable, [B] uint64): the request id that keys the uniforms; NULL means r.
 *
 * Outputs: accepted_len[B] = tau_r; out_tokens[B * out_ld] (out_ld >= max_draft_len + 1) holds
 * x_1 .. x_tau, then the correction (or bonus) token, then -1; correction_token[B] (nullable) the
 * last emitted token.
 * ------------------------------------------------------------------------------------------- */

/* Workspace bytes needed by spec_verify_token / spec_verify_block / spec_sample_draft. */
size_t spec_verify_workspace_bytes(int32_t B, int32_t max_draft_len, int64_t V, sv_dtype dtype);

/* Token-level speculative sampling ("Speculative Decoding: The Same Distribution, Twice as Fast"
 * §4; "How much does a token cost", "On Speculative Sampling").  For i = 1..gamma_r:
 * rho_i = p_i(x_i) / q_i(x_i) with p_i = softmax(target row i), q_i = softmax(draft row i);
 * accept iff u_i < rho_i (u_i: ACCEPT tag, position i).  tau = (first rejected i) - 1, or gamma_r.
 * On a rejection the correction is raced from max(p_{tau+1} - q_{tau+1}, 0) (RESID tag, position
 * tau + 1; if that residual is empty to working precision, from p_{tau+1} with the same
 * uniforms); otherwise the bonus token is raced from p_{gamma+1} (BONUS tag, position gamma + 1).
 * accept_ratio (nullable, indexed like draft_tokens): min(1, rho_i) for EVERY drafted position. */
sv_status spec_verify_token(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                            int64_t V, int64_t ld, const int64_t* target_row0,
                            const int64_t* draft_row0, const int32_t* draft_len,
                            int32_t max_draft_len, const int32_t* draft_tokens, int32_t B,
                            uint64_t seed, const uint64_t* request_ids, int32_t* accepted_len,
                            int32_t* out_tokens, int64_t out_ld, int32_t* correction_token,
                            float* accept_ratio, int32_t* status, void* workspace,
                            size_t workspace_bytes, void* stream);

/* Block verification ("How much does a token cost", "Block verification": the running ratio
 * starts at one, is multiplied by p/q at every drafted token and capped at one after every step;
 * all prefixes are checked and the longest passing one is kept; its acceptance thresholds and
 * correction sampling are those of Sun et al. 2024, "Block Verification Accelerates Speculative
 * Decoding", whose two-token toy the page reproduces):
 *   rho_0 = 1, rho_i = min(1, rho_{i-1} p_i(x_i) / q_i(x_i))
 *   R_i = sum_x max(rho_i p_{i+1}(x) - q_{i+1}(x), 0) for i < gamma
 *   h_i = R_i / (R_i + 1 - rho_i) for i < gamma (1 if the denominator is 0), h_gamma = rho_gamma
 *   tau = max{i : eta_i <= h_i} or 0 (eta_i: ACCEPT tag, position i)
 *   tau < gamma: correction raced from max(rho_tau p_{tau+1} - q_{tau+1}, 0) (RESID, tau + 1)
 *   tau = gamma: bonus raced from p_{gamma+1} (BONUS, gamma + 1).
 * running_ratio, h_threshold (nullable, indexed like draft_tokens): rho_i and h_i. */
sv_status spec_verify_block(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                            int64_t V, int64_t ld, const int64_t* target_row0,
                            const int64_t* draft_row0, const int32_t* draft_len,
                            int32_t max_draft_len, const int32_t* draft_tokens, int32_t B,
                            uint64_t seed, const uint64_t* request_ids, int32_t* accepted_len,
                            int32_t* out_tokens, int64_t out_ld, int32_t* correction_token,
                            float* running_ratio, float* h_threshold, int32_t* status,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Draft tokens sampled from q ("Speculative Decoding: The Same Distribution, Twice as Fast" §3
 * step 1, the drafter's own sampling): for every request r and i = 1..gamma_r,
 * draft_tokens[draft_row0[r] + i - 1] = race sample of softmax(draft row draft_row0[r] + i - 1)
 * with the DRAFT tag at position i.  Layout and workspace as for spec_verify_token. */
sv_status spec_sample_draft(const void* draft_logits, sv_dtype dtype, int64_t V, int64_t ld,
                            const int64_t* draft_row0, const int32_t* draft_len,
                            int32_t max_draft_len, int32_t B, uint64_t seed,
                            const uint64_t* request_ids, int32_t* draft_tokens, int32_t* status,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Token-level verification that allocates nothing and takes no workspace (the pages have no
 * counterpart: this is a packaging variant of spec_verify_token for callers that cannot allocate
 * device memory, e.g. a plugin handed only its input and output buffers by an engine that owns all
 * device memory, or a serving loop that must not call cudaMalloc because it can synchronise the
 * device).  Arguments, results and data-error reporting are those of spec_verify_token.
 * Scratch memory is a fixed array of SV_NOALLOC_SCRATCH_BYTES inside the library, held by every
 * GPU that loads the library until the process exits; calls whose
 * spec_verify_workspace_bytes(B, max_draft_len, V, dtype) exceeds it return SV_ERR_UNSUPPORTED.
 * The first call in each CUDA context (the current device's primary context, or a context the
 * caller made current) looks up the array's device address (cudaGetSymbolAddress) and caches it
 * by the context's id, so a device reset or a new context gets a fresh lookup; make that first
 * call before any stream capture.  Every call shares the one array and clears the counters it
 * needs before use, so calls that overlap on the GPU (other streams or other host threads) race
 * on it and produce undefined results. */
#define SV_NOALLOC_SCRATCH_BYTES (8u << 20)
sv_status spec_verify_token_noalloc(const void* target_logits, const void* draft_logits,
                                    sv_dtype dtype, int64_t V, int64_t ld,
                                    const int64_t* target_row0, const int64_t* draft_row0,
                                    const int32_t* draft_len, int32_t max_draft_len,
                                    const int32_t* draft_tokens, int32_t B, uint64_t seed,
                                    const uint64_t* request_ids, int32_t* accepted_len,
                                    int32_t* out_tokens, int64_t out_ld,
                                    int32_t* correction_token, float* accept_ratio,
                                    int32_t* status, void* stream);

/* ---------------------------------------------------------------------------------------------
 * Token-level verification with the vocabulary split across ranks (tensor parallelism over the
 * vocabulary, as in the vocabulary-parallel serving of "How much does a token cost",
 * "Experiments").  A rank holds columns [v_off, v_off + Vs) of every logit row (v_off a multiple
 * of 8; V_total the whole vocabulary); rows, tokens and layout are those of spec_verify_token
 * with V = Vs, and draft tokens are global vocabulary ids.  Softmax statistics merge across shards
 * by log-sum-exp and the exponential race keys every entry by its global index, so the result
 * equals spec_verify_token's over the whole vocabulary.  A round is four calls and two exchanges
 * that the caller makes between ranks (all-gathers, in rank = shard order):
 *   spec_verify_shard_stats   per drafted row pair (request r, position i at r * max_draft_len +
 *                             i - 1): row_stats DEVICE fp32 [B * max_draft_len][4] = this shard's
 *                             (m_t, s_t, m_d, s_d), m in log2 units (max * log2 e), s = sum of
 *                             2^(x log2 e - m); token_logits DEVICE fp32 [B * max_draft_len][2] =
 *                             the drafted token's target and draft logits if the shard holds it,
 *                             -inf otherwise.  Workspace: spec_verify_workspace_bytes(B,
 *                             max_draft_len, Vs, dtype).
 *   -- all-gather both arrays over the shards: [n_shards][rows][4] and [n_shards][rows][2]
 *   spec_verify_shard_merge   the shards' statistics merged in shard order, the token logits of
 *                             the shard that holds each token (the same on every rank).
 *   spec_verify_shard_race    every request decided as spec_verify_token does (accepted_len[B],
 *                             accept_ratio as there), then this shard's race of the correction
 *                             (or bonus) row: winners DEVICE uint64 [B][2] = the shard's best
 *                             (order-preserving key bits << 32 | ~global index), and, when the
 *                             shard holds no positive residual entry, its best for the race over p
 *                             with the same uniforms (else 0).
 *   -- all-gather winners: [n_shards][B][2]
 *   spec_verify_shard_finish  the largest winner over the shards (the race over p's if no shard
 *                             had a residual entry, as spec_verify_token falls back) and the
 *                             outputs out_tokens / correction_token of spec_verify_token.
 * Each call resets `status` and reports data errors as spec_verify_token does. */
sv_status spec_verify_shard_stats(const void* target_logits, const void* draft_logits,
                                  sv_dtype dtype, int64_t Vs, int64_t ld, int64_t v_off,
                                  int64_t V_total, const int64_t* target_row0,
                                  const int64_t* draft_row0, const int32_t* draft_len,
                                  int32_t max_draft_len, const int32_t* draft_tokens, int32_t B,
                                  float* row_stats, float* token_logits, int32_t* status,
                                  void* workspace, size_t workspace_bytes, void* stream);
sv_status spec_verify_shard_merge(const float* row_stats_all, const float* token_logits_all,
                                  int32_t n_shards, int64_t rows, float* row_stats,
                                  float* token_logits, void* stream);
sv_status spec_verify_shard_race(const void* target_logits, const void* draft_logits,
                                 sv_dtype dtype, int64_t Vs, int64_t ld, int64_t v_off,
                                 int64_t V_total, const int64_t* target_row0,
                                 const int64_t* draft_row0, const int32_t* draft_len,
                                 int32_t max_draft_len, const int32_t* draft_tokens, int32_t B,
                                 uint64_t seed, const uint64_t* request_ids,
                                 const float* row_stats, const float* token_logits,
                                 int32_t* accepted_len, float* accept_ratio, uint64_t* winners,
                                 int32_t* status, void* workspace, size_t workspace_bytes,
                                 void* stream);
sv_status spec_verify_shard_finish(const uint64_t* winners_all, int32_t n_shards, int32_t B,
                                   const int32_t* accepted_len, const int64_t* draft_row0,
                                   const int32_t* draft_tokens, int32_t* out_tokens,
                                   int64_t out_ld, int32_t* correction_token, int32_t* status,
                                   void* stream);

/* Token-level verification from hidden states ("How much does a token cost", "The Role of
 * Arithmetic Intensity": a projection of Q input rows of width H by an [H, W] weight makes the
 * Q x W logits).  The target's logit row i is target_hidden row i times W^T and the draft's logit
 * row i is draft_hidden row i times W^T: the draft scores its tokens through the same output
 * projection as the target.  The logits are computed on the tensor cores (bf16 products, fp32
 * sums) and folded as they are produced; none is written to memory.  Given those logits the call
 * decides and samples exactly as spec_verify_token does on stored logits (same Philox streams,
 * same outputs, same data-error reporting), the logits being the fp32 sums rather than stored
 * values.
 *   target_hidden / draft_hidden  DEVICE bf16, row stride ldh elements (multiple of 8, >= H); the
 *                                 rows of request r are target_row0[r] + 0 .. gamma_r and
 *                                 draft_row0[r] + 0 .. gamma_r - 1, as for the logit rows of
 *                                 spec_verify_token.
 *   W                             DEVICE bf16 [V][ldw] (ldw multiple of 8, >= H): row v is token
 *                                 v's output vector.
 *   H                             hidden size, a multiple of 64.
 *   recomputed                    DEVICE [1] (nullable): how many requests' correction tokens
 *                                 needed the second pass (below); the rest were settled by the
 *                                 candidates the first pass kept.
 * Two passes over W at most.  The first computes every logit once: the softmax statistics and,
 * per position, the few entries that can win the correction or bonus race; the second recomputes
 * the two rows of only those requests whose candidates cannot prove their winner, and is skipped
 * (an empty launch) when there are none.  Both passes race with the same uniforms, so they draw
 * the same token unless two keys lie within their rounding of each other.
 * All DEVICE pointers 16-byte aligned; SV_ERR_UNSUPPORTED otherwise, or for V above 2^31 - 256.
 * The workspace (DEVICE, 256-byte aligned) holds a copy of the hidden rows in GEMM order and the
 * per-tile partials: spec_verify_lmhead_workspace_bytes(B, max_draft_len, V, H) bytes, 0 for sizes
 * the call rejects. */
size_t spec_verify_lmhead_workspace_bytes(int32_t B, int32_t max_draft_len, int64_t V, int64_t H);
sv_status spec_verify_lmhead(const void* target_hidden, const void* draft_hidden, int64_t ldh,
                             const void* W, int64_t ldw, int64_t H, int64_t V,
                             const int64_t* target_row0, const int64_t* draft_row0,
                             const int32_t* draft_len, int32_t max_draft_len,
                             const int32_t* draft_tokens, int32_t B, uint64_t seed,
                             const uint64_t* request_ids, int32_t* accepted_len,
                             int32_t* out_tokens, int64_t out_ld, int32_t* correction_token,
                             float* accept_ratio, int32_t* recomputed, int32_t* status,
                             void* workspace, size_t workspace_bytes, void* stream);

/* ---------------------------------------------------------------------------------------------
 * DSpark draft side.
 * ------------------------------------------------------------------------------------------- */

/* Workspace bytes needed by dspark_markov_draft: one race partial per (request, CTA) and a
 * [K][B] table of published race bounds; 0 for sizes the call rejects. */
size_t dspark_markov_workspace_bytes(int32_t B, int32_t K, int64_t V, int32_t R);

/* Markov-head drafting ("DeepSeek DSpark 详解" §03; "How much does a token cost", "DSpark
 * Architecture"): x_0 = anchor_token[b]; for k = 1..K, left to right,
 *   z_k = bf16( backbone_k + U[x_{k-1}] . W )      (bf16 operands, fp32 accumulation)
 *   x_k = argmax_v z_k(v) - log(-log u_v)           (DRAFT tag, position k)
 *   conf_k = 1 / (1 + exp(-conf_scores[b][k] / sts_T[k]))   (sequential temperature scaling)
 * backbone_logits: DEVICE bf16 [B][K][V], row (b, k) at (b * K + k) * ldb elements;
 * U: DEVICE bf16 [V][R] (row stride R); Wt: DEVICE bf16 [V][R], the factor W [R][V] stored
 * transposed (Wt[v][j] = W[j][v], row stride ldw >= R) so that both GEMM operands are K-major;
 * anchor_token: DEVICE int32 [B]; conf_scores: DEVICE fp32 [B][K]; sts_T: DEVICE fp32 [K].
 * R must be 256 (SV_ERR_UNSUPPORTED otherwise); 1 <= K <= SV_MAX_DRAFT_LEN.
 * Outputs: draft_tokens DEVICE int32 [B][K]; draft_logits_out (nullable) DEVICE bf16 [B][K][V]
 * with row stride ldz -- the exact rows the tokens were sampled from, to be passed to verify;
 * row_stats (nullable) fp32 [B][K][2] = (max z, log-sum-exp z); conf_out (nullable) fp32 [B][K].
 * request_ids as for verify.  ldb, ldw, ldz: multiples of 8 elements; backbone_logits, U, Wt
 * and draft_logits_out 16-byte aligned; workspace 256-byte aligned, at least
 * dspark_markov_workspace_bytes(B, K, V, R) bytes, owned by the caller and free again once the
 * stream has passed this call.  conf_out needs conf_scores and sts_T.  An out-of-range anchor or
 * a row of z without a finite maximum (or holding NaN / +inf) writes SV_ERR_BAD_INPUT to status
 * and drafts token 0 there.  All work is queued on `stream`; nothing is allocated. */
sv_status dspark_markov_draft(const void* backbone_logits, int64_t ldb, const void* U,
                              const void* Wt, int64_t ldw, const int32_t* anchor_token,
                              const float* conf_scores, const float* sts_T, int32_t B, int32_t K,
                              int64_t V, int32_t R, uint64_t seed, const uint64_t* request_ids,
                              int32_t* draft_tokens, void* draft_logits_out, int64_t ldz,
                              float* row_stats, float* conf_out, int32_t* status,
                              void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes needed by dspark_schedule. */
size_t dspark_schedule_workspace_bytes(int32_t N, int32_t K);

/* Hardware-aware prefix scheduler ("DeepSeek DSpark 详解" §04; "DSpark: DeepSeek's bet on speed
 * that doesn't betray quality", "Verifying only what matters"):
 *   S[i][k] = c[i][1] * ... * c[i][k]  (sequential binary32 products, k <= max_len[i])
 *   extendable prefixes (i, k) sorted by S descending, then k ascending, then i ascending;
 *   F = floor(S * 2^40); T(b) = N * 2^40 + (sum of F over the first b);
 *   f(b) = (double) T(b) * 2^-40 * sps[N + b];
 *   admit while f(b + 1) > f(b) and N + b + 1 <= B_max, stopping at the first non-increase.
 * cond_accept: DEVICE fp32 [N][K] in [0, 1] (calibrated conditional acceptance probabilities);
 * max_len: DEVICE int32 [N] in [0, K] (nullable -> K); sps: DEVICE fp64 [B_max + 1], engine steps
 * per second at B verification rows (one row per request plus admitted drafts).
 * Outputs: sel_len DEVICE int32 [N] (drafts to verify per request); survival (nullable) fp32
 * [N][K] (0 past max_len); total_rows DEVICE int32 [1] = N + b; objective DEVICE fp64 [1] = f(b).
 * Supported sizes: N * K <= 16384, N <= B_max. */
sv_status dspark_schedule(const float* cond_accept, const int32_t* max_len, int32_t N, int32_t K,
                          const double* sps, int32_t B_max, int32_t* sel_len, float* survival,
                          int32_t* total_rows, double* objective, int32_t* status,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Stopping rules of the scheduler.
 *   SV_STOP_FIRST_DROP  admit while f still rises and stop at its first non-increase (DSpark's early
 *                       stop; "DeepSeek DSpark 详解" §04, "DSpark: DeepSeek's bet on speed...").
 *   SV_STOP_ARGMAX      the budget with the highest expected tokens per unit time over every
 *                       admissible budget b = 0 .. min(items, B_max - N), the smallest b among
 *                       equals (vLLM's choice in "How much does a token cost", "Adaptive
 *                       verification").
 *   SV_STOP_FIXED_DEPTH one depth k for every request (min(k, max_len) drafts each), deepened while
 *                       the next depth still raises f -- the marginal-slot condition of "How much
 *                       does a token cost", "Our own simple cost model" (slot k + 1 pays when its
 *                       survival mass exceeds L_k (C_{k+1} - C_k) / C_k, C the step time) -- and
 *                       stays within B_max.  total_rows and objective are those of that depth. */
typedef enum { SV_STOP_FIRST_DROP = 0, SV_STOP_ARGMAX = 1, SV_STOP_FIXED_DEPTH = 2 } sv_stop_rule;

/* dspark_schedule with a choice of stopping rule (`rule`, an sv_stop_rule); the order, the fixed
 * point sums and f(b) are those of dspark_schedule, and so are the arguments, outputs, errors and
 * workspace (dspark_schedule_workspace_bytes).  dspark_schedule is rule SV_STOP_FIRST_DROP. */
sv_status dspark_schedule_rule(const float* cond_accept, const int32_t* max_len, int32_t N,
                               int32_t K, const double* sps, int32_t B_max, int32_t rule,
                               int32_t* sel_len, float* survival, int32_t* total_rows,
                               double* objective, int32_t* status, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Asynchronous scheduling with confidences from two rounds before ("DeepSeek Boosts Inference
 * Speed by 85%", "The Third Ace": at production speed the scheduler cannot wait for the current
 * step's confidence, so it schedules with the predictions of two steps before, and the admission
 * never depends on the token it admits; "DSpark: DeepSeek's bet on speed that doesn't betray
 * quality", "Verifying only what matters": the same, for the reference capacity).
 * conf_ring: DEVICE fp32 [depth][N][K], depth >= 3, a ring of confidence-head outputs: round t's
 * predictions go to slot t % depth (for instance dspark_markov_draft's conf_out pointed there).
 * Round t (>= 0) is scheduled with slot (t - 2) % depth, the predictions made two rounds before
 * for request slot i and position k; the first two rounds, which have none, with cond_prior
 * (DEVICE fp32 [N][K], for instance dspark_acceptance_update's estimates).  The scheduling itself
 * -- stopping rule, order, fixed-point sums, arguments, outputs, errors, workspace -- is
 * dspark_schedule_rule's.  The call reads nothing written for rounds t and t - 1, so it can run on
 * a stream that waits only for round t - 2's confidence head, concurrently with round t's draft. */
sv_status dspark_schedule_async(const float* conf_ring, int32_t depth, int64_t round,
                                const float* cond_prior, const int32_t* max_len, int32_t N,
                                int32_t K, const double* sps, int32_t B_max, int32_t rule,
                                int32_t* sel_len, float* survival, int32_t* total_rows,
                                double* objective, int32_t* status, void* workspace,
                                size_t workspace_bytes, void* stream);

/* Per-position acceptance learned while serving ("How much does a token cost", "Adaptive
 * verification": a drafter without a confidence head gets a per-position trust level estimated
 * from the tokens verification accepted).  One verified round: request i verified its first
 * sel_len[i] drafted tokens and accepted the first accepted_len[i] (DEVICE int32 [N] each, the
 * scheduler's and the verifier's outputs).  Position k (1-based) was reached iff
 * k <= min(accepted + 1, verified), accepted iff k <= accepted; the counts decay by `decay`
 * (in [0, 1]; 1 keeps every round) before the round is added:
 *   trials[k]  = decay * trials[k]  + #{i : k <= min(accepted_i + 1, verified_i)}
 *   accepts[k] = decay * accepts[k] + #{i : k <= accepted_i}
 *   alpha[k]   = (float) ((accepts[k] + prior_a) / (trials[k] + prior_a + prior_b))
 * the posterior mean of the conditional acceptance probability under a Beta(prior_a, prior_b)
 * prior (prior_a, prior_b > 0).  trials, accepts: DEVICE fp64 [K], read and updated in place (the
 * caller zeroes them once); alpha: DEVICE fp32 [K]; cond_accept_out (nullable): DEVICE fp32 [N][K],
 * every row set to alpha -- the next round's dspark_schedule input for a drafter without a
 * confidence head.  1 <= K < 4096 (K = 0: nothing to do).  A request with inconsistent lengths
 * (accepted > verified, verified outside [0, K]) is skipped and SV_ERR_BAD_INPUT written to
 * `status`.  No workspace. */
sv_status dspark_acceptance_update(const int32_t* sel_len, const int32_t* accepted_len, int32_t N,
                                   int32_t K, double decay, double prior_a, double prior_b,
                                   double* trials, double* accepts, float* alpha,
                                   float* cond_accept_out, int32_t* status, void* stream);

/* Sequential temperature scaling of the confidence head ("DeepSeek Boosts Inference Speed by 85%",
 * "The Second Ace"; "DeepSeek DSpark 详解" §04): one temperature T_k per draft position, dividing
 * the confidence logit (argmax-preserving), fitted to verified outcomes.  The samples of position k
 * (1-based) are the requests that reached it, k <= min(accepted_len + 1, sel_len); the label is 1
 * when k <= accepted_len.  Fit (a reading: the pages give no rule): `iters` Newton steps on the
 * negative log-likelihood of sigma(s / T_k) in beta = 1 / T_k from beta = 1, each clamped to
 * [beta_min, beta_max]; the logistic in binary32, the sums in binary64.  Expected calibration error
 * over `nbins` (1..256) equal-width confidence bins: sum over bins of |sum (label - confidence)|,
 * over the sample count, at T = 1 (ece_raw_out) and at the fit (ece_fit_out).
 * scores: DEVICE fp32 [N][K] confidence logits; sel_len, accepted_len: DEVICE int32 [N].
 * Outputs (DEVICE, per position): T_out fp32 [K]; nll_out fp64 [K] (mean loss at the fit),
 * ece_raw_out, ece_fit_out fp64 [K], count_out int32 [K] -- all but T_out nullable.
 * Inconsistent lengths: the request is skipped and SV_ERR_BAD_INPUT written to `status`.
 * One CTA per position; no workspace. */
sv_status dspark_sts_fit(const float* scores, const int32_t* sel_len, const int32_t* accepted_len,
                         int32_t N, int32_t K, int32_t iters, double beta_min, double beta_max,
                         int32_t nbins, float* T_out, double* nll_out, double* ece_raw_out,
                         double* ece_fit_out, int32_t* count_out, int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
