/*
 * oracle.h -- CPU oracle for speculative-decoding verification and DSpark drafting.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, double-precision C restatement of what the
 * method computes.  Only the test suite, the package smoke check and the CPU-baseline leg of the
 * benchmark may load it.  The CUDA library shares no code, header, table or constant with it; the
 * two meet only through seeded synthetic inputs.
 *
 * Sources (web pages, cited by title and section):
 *   [SD]  "Speculative Decoding: The Same Distribution, Twice as Fast" (derpx06.online explainer)
 *         §3 "The loop", §4 "The rule that makes it exact", §5 "What decides the speedup",
 *         §6 "A worked example".
 *   [TC]  "How much does a token cost" (blog.luminal.com), sections "On Speculative Sampling",
 *         "Block verification", "Adaptive verification", "DSpark Architecture".
 *   [DS]  "DeepSeek DSpark 详解" (zskr.cn), §03 (semi-autoregressive head, Markov head rank 256),
 *         §04 (confidence head, prefix survival, sequential temperature scaling, SPS(B) scheduler,
 *         early stop).
 *   [AI]  "DSpark: DeepSeek's bet on speed that doesn't betray quality" (aitalk.it), sections
 *         "A drafter that learns to doubt itself" and "Verifying only what matters".
 *   [KC]  "DeepSeek Boosts Inference Speed by 85%" (kongchang.com), "The First Ace" (Markov head),
 *         "The Second Ace" (confidence head, temperature scaling), "The Third Ace" (scheduler).
 *   Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3",
 *         SC'11 (the counter-based generator the uniforms come from; not on the pages).
 *   Block thresholds: Sun, Mendlovic, Leviathan, Aharoni, Beirami, Ro, Suresh, "Block
 *         Verification Accelerates Speculative Decoding" (2024) -- the method [TC] "Block
 *         verification" describes and whose toy example it reproduces.
 *
 * Conventions shared by every call:
 *   - Logit rows are float arrays (bf16 inputs are widened exactly by the caller); all arithmetic
 *     on them is double.  p = softmax(target row), q = softmax(draft row), temperature 1.
 *   - Positions are 1-based: drafted tokens sit at positions 1..gamma, the bonus row at gamma+1.
 *   - Random uniforms: orc_uniform() for scalar draws (the ACCEPT test), orc_race_uniform() for
 *     the entries of a race.  Tags: DRAFT 0, ACCEPT 1, RESID 2, BONUS 3.
 *   - Exponential race: to sample x with probability w(x)/sum(w), take argmax_x log w(x) - log E_x,
 *     E_x = -log u_x (Exp(1) variables); equal keys resolve to the lowest index; w(x)=0 never wins.
 *
 * Parity unpinned: the bit layout of the Philox counter and the uniform conversion are readings
 * (nothing on the pages fixes them); the generator itself is pinned against a library Philox.
 */
#ifndef SPECVERIFY_ORACLE_H
#define SPECVERIFY_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_TAG_DRAFT = 0, ORC_TAG_ACCEPT = 1, ORC_TAG_RESID = 2, ORC_TAG_BONUS = 3 };

/* Added to a race's tag for the stream that holds the low bits of its uniforms. */
enum { ORC_TAG_FINE = 4 };

/* Result codes of the oracle calls. */
enum {
  ORC_OK = 0,
  ORC_ERR_ARGS = 1,       /* a size or pointer argument is invalid */
  ORC_ERR_TOKEN = 2,      /* a drafted token id is outside [0, V) */
  ORC_ERR_NAN = 3,        /* a logit row holds NaN or +inf, or is entirely -inf */
  ORC_ERR_ZERO_Q = 4      /* the draft gave probability 0 to its own drafted token */
};

/* Which race produced the emitted token. */
enum { ORC_RACE_RESIDUAL = 0, ORC_RACE_BONUS = 1, ORC_RACE_RESIDUAL_EMPTY = 2 };

/* ---- random numbers --------------------------------------------------------------------- */

/* Philox4x32-10 block function (Salmon et al., SC'11): 10 rounds of the 4x32 Philox S-box with
 * multipliers 0xD2511F53, 0xCD9E8D57 and the Weyl key schedule 0x9E3779B9, 0xBB67AE85. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* One 32-bit random word for (seed, request, position, tag, vocab index v):
 *   key     = (lo32(seed), hi32(seed))
 *   counter = (v >> 2, pos, lo32(req), (tag << 24) | (hi32(req) & 0xFFFFFF))
 *   word    = output word number (v & 3). */
uint32_t orc_random_word(uint64_t seed, uint64_t req, uint32_t pos, uint32_t tag, uint64_t v);

/* Uniform in (0,1): u = ((word >> 9) + 0.5) * 2^-23.  Exact in float and double, never 0 or 1. */
double orc_uniform(uint64_t seed, uint64_t req, uint32_t pos, uint32_t tag, uint64_t v);

/* The uniform of race entry v, on the same grid as orc_uniform (23 bits, n + 0.5 over 2^23):
 *   n = (h << 7) | f, where
 *   h = 16-bit half (v & 1) (0: low, 1: high) of word (v >> 1) & 3 of the block at counter
 *       (v >> 3, pos, lo32(req), (tag << 24) | (hi32(req) & 0xFFFFFF)) -- one block per 8 entries;
 *   f = orc_random_word(seed, req, pos, tag + ORC_TAG_FINE, v) >> 25.
 * n is uniform on [0, 2^23) because h and f are independent uniform bit fields. */
double orc_race_uniform(uint64_t seed, uint64_t req, uint32_t pos, uint32_t tag, uint64_t v);

/* ---- closed forms --------------------------------------------------------------------- */

/* Row statistics of softmax: *M = max_x row[x], *S = sum_x exp(row[x] - M).  Returns ORC_ERR_NAN
 * for NaN / +inf entries or an all -inf row. */
int orc_row_stats(const float* row, int64_t V, double* M, double* S);

/* Per-token acceptance rate alpha = sum_x min(p(x), q(x)) for two logit rows ([SD] §5; [TC] "On
 * Speculative Sampling": the accepted proposals carry exactly the overlap mass). */
double orc_overlap(const float* target_row, const float* draft_row, int64_t V);

/* Expected words per round (1 - alpha^(gamma+1)) / (1 - alpha) ([SD] §5); gamma+1 at alpha = 1. */
double orc_expected_words(double alpha, int gamma);

/* Speedup of the worked example ([SD] §6): expected words / (1 + gamma * c). */
double orc_speedup(double alpha, int gamma, double c);

/* ---- sampling ---------------------------------------------------------------------------- */

/* Exponential-race sample from softmax(row) with uniforms (seed, req, pos, tag, v):
 * argmax_x log p(x) - log(-log u_x).  *margin (nullable) = best key minus second-best key. */
int orc_sample_race(const float* row, int64_t V, uint64_t seed, uint64_t req, uint32_t pos,
                    uint32_t tag, int32_t* token, double* margin);

/* Draft tokens sampled from q for a batch laid out like the verify calls: for request r and
 * i = 1..draft_len[r], token[draft_row0[r] + i - 1] = race sample of draft row draft_row0[r]+i-1
 * with the DRAFT tag at position i.  request_ids nullable (then request id = r). */
int orc_sample_draft_batch(const float* draft, int64_t V, int64_t ld, const int64_t* draft_row0,
                           const int32_t* draft_len, int32_t B, uint64_t seed,
                           const uint64_t* request_ids, int32_t* draft_tokens);

/* ---- verification -------------------------------------------------------------------------- */

/* Per-request diagnostics, so that near-ties can be counted rather than silently passed. */
typedef struct {
  int32_t accepted_len;      /* tau */
  int32_t correction;        /* the emitted residual / bonus token */
  int32_t race_kind;         /* ORC_RACE_* */
  int32_t status;            /* ORC_* */
  double decision_margin;    /* min |u_i - threshold_i| over the decisions that were taken */
  double race_margin;        /* best minus second-best race key of the race that was run */
} orc_verify_result;

/* Token-level verification of one request ([SD] §3-§4, [TC] "On Speculative Sampling").
 * target: (gamma+1) rows of V floats (row stride ld); draft: gamma rows; tokens: gamma ids.
 * Walk i = 1..gamma: rho_i = p_i(x_i) / q_i(x_i); accept iff u_i < rho_i (ACCEPT tag, pos i).
 * At the first rejection sample the correction from max(p_i - q_i, 0) (RESID tag, pos i) and stop;
 * if all are accepted sample the bonus token from p_{gamma+1} (BONUS tag, pos gamma+1).
 * accept_ratio (nullable, gamma entries) receives min(1, rho_i) for EVERY drafted position. */
/* Race over one vocabulary shard, columns [v_off, v_off + Vs) of a row pair, with the row's
 * whole-vocabulary statistics (natural log: M = max, S = sum exp(x - M)); uniforms keyed by the
 * global index.  Best key and global index out ("How much does a token cost", "Experiments"). */
int orc_race_shard(const float* trow, const float* drow, int64_t Vs, int64_t v_off, int resid,
                   double w, double Mt, double St, double Md, double Sd, uint64_t seed,
                   uint64_t req, uint32_t pos, uint32_t tag, double* key, int64_t* index);

/* Logits of hidden-state rows through an output projection ("How much does a token cost", "The
 * Role of Arithmetic Intensity"): logits[i][v] = sum_j hidden[i][j] W[v][j] in binary64, rounded
 * once to binary32.  hidden [rows][H], W [V][H], logits [rows][V]. */
int orc_lmhead_logits(const float* hidden, const float* W, int64_t rows, int64_t H, int64_t V,
                      float* logits);

int orc_verify_token_request(const float* target, const float* draft, int64_t V, int64_t ld,
                             const int32_t* tokens, int32_t gamma, uint64_t seed, uint64_t req,
                             double* accept_ratio, orc_verify_result* res);

/* Block verification of one request ([TC] "Block verification"; thresholds of Sun et al. 2024):
 *   rho_0 = 1, rho_i = min(1, rho_{i-1} * p_i(x_i) / q_i(x_i))
 *   R_i = sum_x max(rho_i p_{i+1}(x) - q_{i+1}(x), 0)            (i < gamma)
 *   h_i = R_i / (R_i + 1 - rho_i) (i < gamma; 1 when the denominator is 0),  h_gamma = rho_gamma
 *   tau = max{ i in 1..gamma : eta_i <= h_i }, or 0 when none passes (eta_i: ACCEPT tag, pos i)
 *   tau < gamma: correction from max(rho_tau p_{tau+1} - q_{tau+1}, 0) (RESID tag, pos tau+1)
 *   tau = gamma: bonus from p_{gamma+1} (BONUS tag, pos gamma+1).
 * rho_out, h_out nullable, gamma entries each. */
int orc_verify_block_request(const float* target, const float* draft, int64_t V, int64_t ld,
                             const int32_t* tokens, int32_t gamma, uint64_t seed, uint64_t req,
                             double* rho_out, double* h_out, orc_verify_result* res);

/* Batched wrappers laid out like the C-ABI calls: request r owns target rows
 * target_row0[r] .. target_row0[r] + draft_len[r] and draft rows draft_row0[r] ..
 * draft_row0[r] + draft_len[r] - 1; its drafted tokens are draft_tokens[draft_row0[r] + i - 1].
 * Outputs: accepted_len[B], out_tokens[B * out_ld] (x_1..x_tau, correction, then -1),
 * correction[B], per-draft-row arrays indexed like draft_tokens (nullable), results[B]
 * (nullable).  request_ids nullable (then r).  block != 0 selects block verification, in which
 * case ratio_out receives rho_i and h_out receives h_i; otherwise ratio_out receives min(1, p/q). */
int orc_verify_batch(int block, const float* target, const float* draft, int64_t V, int64_t ld,
                     const int64_t* target_row0, const int64_t* draft_row0,
                     const int32_t* draft_len, const int32_t* draft_tokens, int32_t B,
                     uint64_t seed, const uint64_t* request_ids, int32_t* accepted_len,
                     int32_t* out_tokens, int64_t out_ld, int32_t* correction, double* ratio_out,
                     double* h_out, orc_verify_result* results);

/* ---- DSpark draft side -------------------------------------------------------------------- */

/* Round a double to the nearest bfloat16 (ties to even) and return its 16-bit pattern. */
uint16_t orc_bf16_round(double x);

/* Sequential temperature scaling of a confidence logit ([KC] "The Second Ace", [DS] §04):
 * conf = 1 / (1 + exp(-s / T)). */
double orc_sts_confidence(double s, double T);

/* Markov-head drafting of one request ([DS] §03, [TC] "DSpark Architecture", [KC] "The First
 * Ace"): x_0 = anchor; for k = 1..K
 *   z_k(v) = bf16( backbone_k(v) + sum_{j<R} U[x_{k-1}][j] * W[j][v] )   (sum in double, one rounding)
 *   x_k    = argmax_v z_k(v) - log(-log u_v)                           (DRAFT tag, position k)
 *   conf_k = 1 / (1 + exp(-scores_k / T_k)).
 * backbone: K rows of V floats (stride ldb); U: V rows of R floats; W: R rows of V floats.
 * forced_prev (nullable, K entries): teacher forcing -- step k uses forced_prev[k-1] as x_{k-1}
 * instead of the oracle's own previous sample.  Outputs (all nullable except x_out):
 * z_out K*V bf16 patterns, x_out K tokens, stats_out K*2 (max z, log-sum-exp z), conf_out K,
 * margin_out K race margins. */
int orc_markov_draft_request(const float* backbone, int64_t ldb, const float* U, const float* W,
                             int32_t anchor, const float* scores, const float* T, int32_t K,
                             int64_t V, int32_t R, uint64_t seed, uint64_t req,
                             const int32_t* forced_prev, uint16_t* z_out, int32_t* x_out,
                             double* stats_out, double* conf_out, double* margin_out);

/* Hardware-aware prefix scheduler ([DS] §04, [AI] "Verifying only what matters", [KC] "The
 * Third Ace"):
 *   S[i][k] = c[i][1] * ... * c[i][k] as a sequential float (binary32) product, k = 1..max_len[i]
 *   items (i, k) sorted by S descending, then k ascending, then i ascending
 *   F(i, k) = floor(S[i][k] * 2^40) (int64);  T(b) = N * 2^40 + sum of F over the first b items
 *   f(b) = (double) T(b) * 2^-40 * sps[N + b]
 *   admit items while f(b + 1) > f(b) and N + b + 1 <= B_max; stop at the first non-increase.
 * sel_len[i] = admitted items of request i; survival (nullable) N*K floats (0 past max_len);
 * *total_rows = N + b; *objective = f(b). */
int orc_schedule(const float* cond_accept, const int32_t* max_len, int32_t N, int32_t K,
                 const double* sps, int32_t B_max, int32_t* sel_len, float* survival,
                 int32_t* total_rows, double* objective);

/* Stopping rules of the scheduler.  FIRST_DROP: the rule above (DSpark's early stop).  ARGMAX: the
 * budget with the highest expected tokens per unit time over every admissible budget, vLLM's choice
 * in [TC] "Adaptive verification" (each budget filled with the positions most likely to survive,
 * the best one kept): b* = the smallest b in 0..min(items, B_max - N) with f(b) = max f.  The order,
 * F, T and f are the same as above. */
enum { ORC_STOP_FIRST_DROP = 0, ORC_STOP_ARGMAX = 1, ORC_STOP_FIXED_DEPTH = 2 };
/* FIXED_DEPTH: the fixed-depth cost model of [TC] "Our own simple cost model" -- every request
 * verifies the same number k of drafts (min(k, max_len[i])), and one more slot is worth adding only
 * while it raises the expected tokens per unit time: with L_k = expected tokens (the guaranteed one
 * plus the survivals up to depth k) and C_k = the step time at the rows of depth k, slot k + 1 pays
 * when its survival exceeds L_k (C_{k+1} - C_k) / C_k, i.e. when f(k + 1) > f(k) with
 * f(k) = T(k) 2^-40 sps[B(k)], T(k) = N 2^40 + sum of F up to depth k, B(k) = N + sum of
 * min(k, max_len).  The depth is the first k where the next one does not pay (or would exceed
 * B_max); sel_len[i] = min(k, max_len[i]). */
int orc_schedule_rule(const float* cond_accept, const int32_t* max_len, int32_t N, int32_t K,
                      const double* sps, int32_t B_max, int32_t rule, int32_t* sel_len,
                      float* survival, int32_t* total_rows, double* objective);

/* Asynchronous scheduling ("DeepSeek Boosts Inference Speed by 85%", "The Third Ace"; "DSpark:
 * DeepSeek's bet on speed that doesn't betray quality", "Verifying only what matters"): the
 * scheduler of round t uses the confidence predictions made two rounds before, so its admission
 * never depends on the token it admits.  conf_rounds [rounds][N][K] holds each round's predictions;
 * round t is scheduled by orc_schedule_rule with conf_rounds[t - 2] when t >= 2, with prior [N][K]
 * for rounds 0 and 1 (no prediction is two rounds old yet). */
int orc_schedule_async(const float* conf_rounds, int64_t round, const float* prior,
                       const int32_t* max_len, int32_t N, int32_t K, const double* sps,
                       int32_t B_max, int32_t rule, int32_t* sel_len, float* survival,
                       int32_t* total_rows, double* objective);

/* Per-position acceptance learned while serving ([TC] "Adaptive verification": a drafter without a
 * confidence head gets a per-position trust level estimated from the tokens verification
 * accepted).  Request i verified its first sel_len[i] drafted tokens and accepted the first
 * accepted_len[i] (0 <= accepted <= verified <= K).  Position k (1-based) was reached when every
 * earlier token was accepted, k <= min(accepted + 1, verified), and accepted when k <= accepted.
 * Reading: the counts decay by `decay` in [0, 1] before a round is added, and the estimate of the
 * conditional acceptance probability is the posterior mean under a Beta(prior_a, prior_b) prior:
 *   trials[k]  = decay * trials[k]  + #{i : k <= min(accepted_i + 1, verified_i)}
 *   accepts[k] = decay * accepts[k] + #{i : k <= accepted_i}
 *   alpha[k]   = (float) ((accepts[k] + prior_a) / (trials[k] + prior_a + prior_b))
 * trials, accepts: K doubles, updated in place; alpha: K floats.  A request with inconsistent
 * lengths is skipped and ORC_ERR_NAN returned. */
int orc_acceptance_update(const int32_t* sel_len, const int32_t* accepted_len, int32_t N,
                          int32_t K, double decay, double prior_a, double prior_b, double* trials,
                          double* accepts, float* alpha);

/* Sequential temperature scaling ([KC] "The Second Ace", [DS] §04: one temperature per draft
 * position divides the confidence head's logit, argmax-preserving, fitted until the stated
 * confidences match the observed acceptance; the calibration error is the expected calibration
 * error, ECE).  The samples of position k (1-based) are the requests that reached it (every earlier
 * drafted token accepted and k verified: k <= min(accepted_len + 1, sel_len)); the label is 1 when
 * k <= accepted_len.  scores: N*K floats, the confidence logits s.
 * Reading (the pages give no fitting rule): the standard temperature-scaling fit -- minimise the
 * negative log-likelihood of sigma(s / T_k) -- by `iters` Newton steps in beta = 1 / T from beta = 1,
 * each clamped to [beta_min, beta_max], in binary64; ECE over `nbins` equal-width confidence bins:
 * sum over bins of |sum of (label - confidence)| / n_k.
 * Outputs per position: T_out (float), nll_out (mean NLL at the fit), ece_raw_out (T = 1),
 * ece_fit_out, count_out (n_k); all but T_out nullable.  Inconsistent lengths: request skipped,
 * ORC_ERR_NAN returned. */
int orc_sts_fit(const float* scores, const int32_t* sel_len, const int32_t* accepted_len,
                int32_t N, int32_t K, int32_t iters, double beta_min, double beta_max,
                int32_t nbins, float* T_out, double* nll_out, double* ece_raw_out,
                double* ece_fit_out, int32_t* count_out);

#ifdef __cplusplus
}
#endif

#endif
