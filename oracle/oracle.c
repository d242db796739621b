/*
 * oracle.c -- CPU oracle (test infrastructure only; see oracle.h for the sources and conventions).
 *
 * Plain loops in double.  No blocking, no fusion, no reordering beyond what each definition says,
 * so that every function can be read against the passage it cites.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- random numbers --------------------------------------------------------------------- */

/* Philox4x32-10 (Salmon et al., SC'11, section 3.3 "Philox"): each round multiplies the even
 * counter words by the two round constants, swaps the halves and xors the key; the key advances
 * by the Weyl constants between rounds. */
void orc_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    uint64_t prod0 = (uint64_t)0xD2511F53u * (uint64_t)c0;
    uint64_t prod1 = (uint64_t)0xCD9E8D57u * (uint64_t)c2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t n0 = hi1 ^ c1 ^ k0;
    uint32_t n1 = lo1;
    uint32_t n2 = hi0 ^ c3 ^ k1;
    uint32_t n3 = lo0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

/* The Philox block at counter (group, pos, lo32(req), tag << 24 | hi32(req) & 0xFFFFFF). */
static void random_block(uint64_t seed, uint64_t req, uint32_t pos, uint32_t tag, uint32_t group,
                         uint32_t out[4]) {
  uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
  uint32_t ctr[4] = {group, pos, (uint32_t)(req & 0xFFFFFFFFu),
                     (tag << 24) | ((uint32_t)(req >> 32) & 0xFFFFFFu)};
  orc_philox4x32_10(ctr, key, out);
}

uint32_t orc_random_word(uint64_t seed, uint64_t req, uint32_t pos, uint32_t tag, uint64_t v) {
  uint32_t out[4];
  random_block(seed, req, pos, tag, (uint32_t)(v >> 2), out);
  return out[v & 3u];
}

double orc_uniform(uint64_t seed, uint64_t req, uint32_t pos, uint32_t tag, uint64_t v) {
  uint32_t w = orc_random_word(seed, req, pos, tag, v);
  return ((double)(w >> 9) + 0.5) * ldexp(1.0, -23);
}

/* Race entries: 16 high bits from a block shared by 8 entries, 7 low bits from the FINE stream. */
double orc_race_uniform(uint64_t seed, uint64_t req, uint32_t pos, uint32_t tag, uint64_t v) {
  uint32_t blk[4];
  random_block(seed, req, pos, tag, (uint32_t)(v >> 3), blk);
  uint32_t word = blk[(v >> 1) & 3u];
  uint32_t h = (v & 1u) ? (word >> 16) : (word & 0xFFFFu);
  uint32_t f = orc_random_word(seed, req, pos, tag + ORC_TAG_FINE, v) >> 25;
  return ((double)((h << 7) | f) + 0.5) * ldexp(1.0, -23);
}

/* -log(E) for the exponential variable E = -log(u) of one race entry. */
static double race_noise(uint64_t seed, uint64_t req, uint32_t pos, uint32_t tag, uint64_t v) {
  double u = orc_race_uniform(seed, req, pos, tag, v);
  double E = -log(u);
  return -log(E);
}

/* ---- closed forms --------------------------------------------------------------------- */

int orc_row_stats(const float* row, int64_t V, double* M, double* S) {
  if (V <= 0) return ORC_ERR_ARGS;
  double m = -INFINITY;
  for (int64_t x = 0; x < V; ++x) {
    double t = row[x];
    if (isnan(t) || (isinf(t) && t > 0)) return ORC_ERR_NAN;
    if (t > m) m = t;
  }
  if (isinf(m)) return ORC_ERR_NAN; /* every entry is -inf: no distribution */
  double s = 0.0;
  for (int64_t x = 0; x < V; ++x) s += exp((double)row[x] - m);
  *M = m;
  *S = s;
  return ORC_OK;
}

/* p(x) for a row with statistics (M, S). */
static double prob(const float* row, int64_t x, double M, double S) {
  return exp((double)row[x] - M) / S;
}

double orc_overlap(const float* target_row, const float* draft_row, int64_t V) {
  double Mt, St, Md, Sd;
  if (orc_row_stats(target_row, V, &Mt, &St) != ORC_OK) return NAN;
  if (orc_row_stats(draft_row, V, &Md, &Sd) != ORC_OK) return NAN;
  double a = 0.0;
  for (int64_t x = 0; x < V; ++x) {
    double p = prob(target_row, x, Mt, St), q = prob(draft_row, x, Md, Sd);
    a += p < q ? p : q;
  }
  return a;
}

double orc_expected_words(double alpha, int gamma) {
  if (alpha == 1.0) return (double)gamma + 1.0;
  return (1.0 - pow(alpha, (double)gamma + 1.0)) / (1.0 - alpha);
}

double orc_speedup(double alpha, int gamma, double c) {
  return orc_expected_words(alpha, gamma) / (1.0 + (double)gamma * c);
}

/* ---- races ------------------------------------------------------------------------------ */

/* Running best / second-best of an exponential race; ties go to the lowest index because
 * entries are offered in increasing index order and only a strictly larger key replaces. */
typedef struct {
  double best, second;
  int64_t arg;
} race_t;

static void race_init(race_t* r) {
  r->best = -INFINITY;
  r->second = -INFINITY;
  r->arg = -1;
}

static void race_offer(race_t* r, double key, int64_t x) {
  if (key > r->best) {
    r->second = r->best;
    r->best = key;
    r->arg = x;
  } else if (key > r->second) {
    r->second = key;
  }
}

static double race_margin(const race_t* r) {
  if (isinf(r->second)) return INFINITY;
  return r->best - r->second;
}

/* Race over p = softmax(row): key = log p(x) - log E_x. */
static void race_softmax(const float* row, int64_t V, double M, double S, uint64_t seed,
                         uint64_t req, uint32_t pos, uint32_t tag, race_t* r) {
  race_init(r);
  for (int64_t x = 0; x < V; ++x) {
    double p = prob(row, x, M, S);
    if (!(p > 0.0)) continue;
    race_offer(r, log(p) + race_noise(seed, req, pos, tag, (uint64_t)x), x);
  }
}

int orc_sample_race(const float* row, int64_t V, uint64_t seed, uint64_t req, uint32_t pos,
                    uint32_t tag, int32_t* token, double* margin) {
  double M, S;
  int st = orc_row_stats(row, V, &M, &S);
  if (st != ORC_OK) return st;
  race_t r;
  race_softmax(row, V, M, S, seed, req, pos, tag, &r);
  *token = (int32_t)r.arg;
  if (margin) *margin = race_margin(&r);
  return ORC_OK;
}

int orc_sample_draft_batch(const float* draft, int64_t V, int64_t ld, const int64_t* draft_row0,
                           const int32_t* draft_len, int32_t B, uint64_t seed,
                           const uint64_t* request_ids, int32_t* draft_tokens) {
  if (B < 0 || V <= 0 || ld < V) return ORC_ERR_ARGS;
  for (int32_t r = 0; r < B; ++r) {
    uint64_t req = request_ids ? request_ids[r] : (uint64_t)r;
    for (int32_t i = 1; i <= draft_len[r]; ++i) {
      int64_t row = draft_row0[r] + i - 1;
      int st = orc_sample_race(draft + row * ld, V, seed, req, (uint32_t)i, ORC_TAG_DRAFT,
                               &draft_tokens[row], NULL);
      if (st != ORC_OK) return st;
    }
  }
  return ORC_OK;
}

/* Race over one vocabulary shard, columns [v_off, v_off + Vs) of a row pair, with the row's
 * whole-vocabulary statistics: weight w p(x) - q(x) when resid (else p(x)), the key of column x
 * keyed by the uniform of its global index v_off + x.  Returns the shard's best key and its global
 * index (-1 if no entry carries weight).  The shards' best keys combine by maximum (lowest index
 * among equals) into the race over the whole row ("How much does a token cost", "Experiments":
 * vocabulary-parallel serving). */
int orc_race_shard(const float* trow, const float* drow, int64_t Vs, int64_t v_off, int resid,
                   double w, double Mt, double St, double Md, double Sd, uint64_t seed,
                   uint64_t req, uint32_t pos, uint32_t tag, double* key, int64_t* index) {
  race_t r;
  race_init(&r);
  for (int64_t x = 0; x < Vs; ++x) {
    double weight = resid ? w * prob(trow, x, Mt, St) - prob(drow, x, Md, Sd)
                          : prob(trow, x, Mt, St);
    if (!(weight > 0.0)) continue;
    race_offer(&r, log(weight) + race_noise(seed, req, pos, tag, (uint64_t)(v_off + x)),
               v_off + x);
  }
  *key = r.best;
  *index = r.arg;
  return ORC_OK;
}

/* ---- logits from hidden states ------------------------------------------------------------- */

/* The output projection ("How much does a token cost", "The Role of Arithmetic Intensity": inputs
 * [Q, H] times weights [H, W] give the Q x W logits): logits[i][v] = sum_j hidden[i][j] W[v][j],
 * the products and their sum in binary64, rounded once to binary32. */
int orc_lmhead_logits(const float* hidden, const float* W, int64_t rows, int64_t H, int64_t V,
                      float* logits) {
  if (rows < 0 || H <= 0 || V <= 0) return ORC_ERR_ARGS;
  for (int64_t i = 0; i < rows; ++i)
    for (int64_t v = 0; v < V; ++v) {
      double acc = 0.0;
      for (int64_t j = 0; j < H; ++j) acc += (double)hidden[i * H + j] * (double)W[v * H + j];
      logits[i * V + v] = (float)acc;
    }
  return ORC_OK;
}

/* ---- verification -------------------------------------------------------------------------- */

static int check_tokens(const int32_t* tokens, int32_t gamma, int64_t V) {
  for (int32_t i = 0; i < gamma; ++i)
    if (tokens[i] < 0 || (int64_t)tokens[i] >= V) return ORC_ERR_TOKEN;
  return ORC_OK;
}

/* Statistics of target rows 1..gamma+1 and draft rows 1..gamma (index i-1). */
static int all_stats(const float* target, const float* draft, int64_t V, int64_t ld,
                     int32_t gamma, double* Mt, double* St, double* Md, double* Sd) {
  for (int32_t i = 0; i <= gamma; ++i) {
    int st = orc_row_stats(target + (int64_t)i * ld, V, &Mt[i], &St[i]);
    if (st != ORC_OK) return st;
  }
  for (int32_t i = 0; i < gamma; ++i) {
    int st = orc_row_stats(draft + (int64_t)i * ld, V, &Md[i], &Sd[i]);
    if (st != ORC_OK) return st;
  }
  return ORC_OK;
}

/* Ratio p_i(x_i) / q_i(x_i) of drafted position i (1-based). */
static int token_ratio(const float* target, const float* draft, int64_t ld, const int32_t* tokens,
                       int32_t i, const double* Mt, const double* St, const double* Md,
                       const double* Sd, double* rho) {
  const float* trow = target + (int64_t)(i - 1) * ld;
  const float* drow = draft + (int64_t)(i - 1) * ld;
  int32_t x = tokens[i - 1];
  double p = prob(trow, x, Mt[i - 1], St[i - 1]);
  double q = prob(drow, x, Md[i - 1], Sd[i - 1]);
  if (!(q > 0.0)) return ORC_ERR_ZERO_Q;
  *rho = p / q;
  return ORC_OK;
}

/* Race over the residual max(w * p(x) - q(x), 0) of one row pair (w = 1 for token-level,
 * w = rho_tau for block verification).  Falls back to a race over p with the same uniforms when
 * the residual is empty after rounding (p and q equal to working precision). */
static void race_residual(const float* trow, const float* drow, int64_t V, double w, double Mt,
                          double St, double Md, double Sd, uint64_t seed, uint64_t req,
                          uint32_t pos, race_t* r, int32_t* kind) {
  race_init(r);
  for (int64_t x = 0; x < V; ++x) {
    double res = w * prob(trow, x, Mt, St) - prob(drow, x, Md, Sd);
    if (!(res > 0.0)) continue;
    race_offer(r, log(res) + race_noise(seed, req, pos, ORC_TAG_RESID, (uint64_t)x), x);
  }
  *kind = ORC_RACE_RESIDUAL;
  if (r->arg < 0) {
    race_softmax(trow, V, Mt, St, seed, req, pos, ORC_TAG_RESID, r);
    *kind = ORC_RACE_RESIDUAL_EMPTY;
  }
}

int orc_verify_token_request(const float* target, const float* draft, int64_t V, int64_t ld,
                             const int32_t* tokens, int32_t gamma, uint64_t seed, uint64_t req,
                             double* accept_ratio, orc_verify_result* res) {
  memset(res, 0, sizeof(*res));
  res->accepted_len = -1;
  res->correction = -1;
  if (gamma < 0 || V <= 0 || ld < V) return res->status = ORC_ERR_ARGS;
  int st = check_tokens(tokens, gamma, V);
  if (st != ORC_OK) return res->status = st;

  double* stats = (double*)malloc(sizeof(double) * 4 * ((size_t)gamma + 1));
  double *Mt = stats, *St = stats + gamma + 1, *Md = stats + 2 * (gamma + 1),
         *Sd = stats + 3 * (gamma + 1);
  st = all_stats(target, draft, V, ld, gamma, Mt, St, Md, Sd);
  if (st != ORC_OK) {
    free(stats);
    return res->status = st;
  }

  /* min(1, p/q) for every drafted position (acceptance-rate monitoring output). */
  double* rho = (double*)malloc(sizeof(double) * ((size_t)gamma + 1));
  for (int32_t i = 1; i <= gamma; ++i) {
    st = token_ratio(target, draft, ld, tokens, i, Mt, St, Md, Sd, &rho[i]);
    if (st != ORC_OK) {
      free(rho);
      free(stats);
      return res->status = st;
    }
    if (accept_ratio) accept_ratio[i - 1] = rho[i] < 1.0 ? rho[i] : 1.0;
  }

  /* Walk left to right; stop at the first rejection ([SD] §3 step 3, §4). */
  res->decision_margin = INFINITY;
  int32_t tau = gamma;
  for (int32_t i = 1; i <= gamma; ++i) {
    double u = orc_uniform(seed, req, (uint32_t)i, ORC_TAG_ACCEPT, 0);
    double m = fabs(u - rho[i]);
    if (m < res->decision_margin) res->decision_margin = m;
    if (!(u < rho[i])) {
      tau = i - 1;
      break;
    }
  }

  race_t r;
  if (tau < gamma) {
    /* Correction from p'(x) = max(0, p - q) / sum max(0, p - q) of the rejected position. */
    int32_t i = tau + 1;
    race_residual(target + (int64_t)(i - 1) * ld, draft + (int64_t)(i - 1) * ld, V, 1.0,
                  Mt[i - 1], St[i - 1], Md[i - 1], Sd[i - 1], seed, req, (uint32_t)i, &r,
                  &res->race_kind);
  } else {
    /* All gamma accepted: the (gamma+1)-th word comes from the target's own next row. */
    race_softmax(target + (int64_t)gamma * ld, V, Mt[gamma], St[gamma], seed, req,
                 (uint32_t)(gamma + 1), ORC_TAG_BONUS, &r);
    res->race_kind = ORC_RACE_BONUS;
  }
  res->accepted_len = tau;
  res->correction = (int32_t)r.arg;
  res->race_margin = race_margin(&r);
  free(rho);
  free(stats);
  return res->status = ORC_OK;
}

int orc_verify_block_request(const float* target, const float* draft, int64_t V, int64_t ld,
                             const int32_t* tokens, int32_t gamma, uint64_t seed, uint64_t req,
                             double* rho_out, double* h_out, orc_verify_result* res) {
  memset(res, 0, sizeof(*res));
  res->accepted_len = -1;
  res->correction = -1;
  if (gamma < 0 || V <= 0 || ld < V) return res->status = ORC_ERR_ARGS;
  int st = check_tokens(tokens, gamma, V);
  if (st != ORC_OK) return res->status = st;

  double* stats = (double*)malloc(sizeof(double) * 6 * ((size_t)gamma + 1));
  double *Mt = stats, *St = stats + gamma + 1, *Md = stats + 2 * (gamma + 1),
         *Sd = stats + 3 * (gamma + 1), *rho = stats + 4 * (gamma + 1),
         *h = stats + 5 * (gamma + 1);
  st = all_stats(target, draft, V, ld, gamma, Mt, St, Md, Sd);
  if (st != ORC_OK) {
    free(stats);
    return res->status = st;
  }

  /* Running target-to-draft ratio, capped at one after every step. */
  rho[0] = 1.0;
  for (int32_t i = 1; i <= gamma; ++i) {
    double ratio;
    st = token_ratio(target, draft, ld, tokens, i, Mt, St, Md, Sd, &ratio);
    if (st != ORC_OK) {
      free(stats);
      return res->status = st;
    }
    double next = rho[i - 1] * ratio;
    rho[i] = next < 1.0 ? next : 1.0;
    if (rho_out) rho_out[i - 1] = rho[i];
  }

  /* Acceptance thresholds: h_i = R_i / (R_i + 1 - rho_i) for i < gamma, h_gamma = rho_gamma. */
  for (int32_t i = 1; i <= gamma; ++i) {
    if (i < gamma) {
      const float* trow = target + (int64_t)i * ld; /* row i+1 */
      const float* drow = draft + (int64_t)i * ld;
      double R = 0.0;
      for (int64_t x = 0; x < V; ++x) {
        double d = rho[i] * prob(trow, x, Mt[i], St[i]) - prob(drow, x, Md[i], Sd[i]);
        if (d > 0.0) R += d;
      }
      double den = R + 1.0 - rho[i];
      h[i] = den > 0.0 ? R / den : 1.0;
    } else {
      h[i] = rho[i];
    }
    if (h_out) h_out[i - 1] = h[i];
  }

  /* Longest passing prefix. */
  res->decision_margin = INFINITY;
  int32_t tau = 0;
  for (int32_t i = 1; i <= gamma; ++i) {
    double eta = orc_uniform(seed, req, (uint32_t)i, ORC_TAG_ACCEPT, 0);
    double m = fabs(eta - h[i]);
    if (m < res->decision_margin) res->decision_margin = m;
    if (eta <= h[i]) tau = i;
  }

  race_t r;
  if (tau < gamma) {
    int32_t i = tau + 1;
    race_residual(target + (int64_t)(i - 1) * ld, draft + (int64_t)(i - 1) * ld, V, rho[tau],
                  Mt[i - 1], St[i - 1], Md[i - 1], Sd[i - 1], seed, req, (uint32_t)i, &r,
                  &res->race_kind);
  } else {
    race_softmax(target + (int64_t)gamma * ld, V, Mt[gamma], St[gamma], seed, req,
                 (uint32_t)(gamma + 1), ORC_TAG_BONUS, &r);
    res->race_kind = ORC_RACE_BONUS;
  }
  res->accepted_len = tau;
  res->correction = (int32_t)r.arg;
  res->race_margin = race_margin(&r);
  free(stats);
  return res->status = ORC_OK;
}

int orc_verify_batch(int block, const float* target, const float* draft, int64_t V, int64_t ld,
                     const int64_t* target_row0, const int64_t* draft_row0,
                     const int32_t* draft_len, const int32_t* draft_tokens, int32_t B,
                     uint64_t seed, const uint64_t* request_ids, int32_t* accepted_len,
                     int32_t* out_tokens, int64_t out_ld, int32_t* correction, double* ratio_out,
                     double* h_out, orc_verify_result* results) {
  if (B < 0 || V <= 0 || ld < V) return ORC_ERR_ARGS;
  int first_err = ORC_OK;
  for (int32_t r = 0; r < B; ++r) {
    uint64_t req = request_ids ? request_ids[r] : (uint64_t)r;
    int32_t gamma = draft_len[r];
    const int32_t* tokens = draft_tokens + draft_row0[r];
    orc_verify_result res;
    double* ratio = ratio_out ? ratio_out + draft_row0[r] : NULL;
    int st;
    if (out_ld < (int64_t)gamma + 1) {
      st = ORC_ERR_ARGS;
      memset(&res, 0, sizeof(res));
      res.status = st;
      res.accepted_len = res.correction = -1;
    } else if (block) {
      st = orc_verify_block_request(target + target_row0[r] * ld, draft + draft_row0[r] * ld, V,
                                    ld, tokens, gamma, seed, req, ratio,
                                    h_out ? h_out + draft_row0[r] : NULL, &res);
    } else {
      st = orc_verify_token_request(target + target_row0[r] * ld, draft + draft_row0[r] * ld, V,
                                    ld, tokens, gamma, seed, req, ratio, &res);
    }
    if (st != ORC_OK && first_err == ORC_OK) first_err = st;
    if (accepted_len) accepted_len[r] = res.accepted_len;
    if (correction) correction[r] = res.correction;
    if (out_tokens) {
      int32_t* row = out_tokens + (int64_t)r * out_ld;
      for (int64_t j = 0; j < out_ld; ++j) row[j] = -1;
      if (st == ORC_OK) {
        for (int32_t j = 0; j < res.accepted_len; ++j) row[j] = tokens[j];
        row[res.accepted_len] = res.correction;
      }
    }
    if (results) results[r] = res;
  }
  return first_err;
}

/* ---- DSpark draft side -------------------------------------------------------------------- */

uint16_t orc_bf16_round(double x) {
  if (isnan(x)) return 0x7FC0u;
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double ax = fabs(x);
  if (isinf(ax)) return (uint16_t)(sign | 0x7F80u);
  if (ax == 0.0) return sign;
  int e;
  frexp(ax, &e);           /* 2^(e-1) <= ax < 2^e */
  int E = e - 1;
  if (E < -126) E = -126;  /* subnormal bfloat16 values share the spacing 2^-133 */
  double quantum = ldexp(1.0, E - 7); /* 7 stored fraction bits */
  double r = nearbyint(ax / quantum) * quantum; /* default rounding mode: ties to even */
  float f = (float)r;      /* exact for every bfloat16 value; 2^128 and above become inf */
  uint32_t bits;
  memcpy(&bits, &f, sizeof(bits));
  return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

static double bf16_value(uint16_t h) {
  uint32_t bits = (uint32_t)h << 16;
  float f;
  memcpy(&f, &bits, sizeof(f));
  return (double)f;
}

double orc_sts_confidence(double s, double T) { return 1.0 / (1.0 + exp(-s / T)); }

int orc_markov_draft_request(const float* backbone, int64_t ldb, const float* U, const float* W,
                             int32_t anchor, const float* scores, const float* T, int32_t K,
                             int64_t V, int32_t R, uint64_t seed, uint64_t req,
                             const int32_t* forced_prev, uint16_t* z_out, int32_t* x_out,
                             double* stats_out, double* conf_out, double* margin_out) {
  if (K < 0 || V <= 0 || R <= 0 || ldb < V || !x_out) return ORC_ERR_ARGS;
  double* z = (double*)malloc(sizeof(double) * (size_t)V);
  int32_t prev = anchor;
  for (int32_t k = 1; k <= K; ++k) {
    if (forced_prev) prev = forced_prev[k - 1];
    if (prev < 0 || (int64_t)prev >= V) {
      free(z);
      return ORC_ERR_TOKEN;
    }
    const float* brow = backbone + (int64_t)(k - 1) * ldb;
    const float* urow = U + (int64_t)prev * R;
    /* z_k = bf16(backbone_k + U[x_{k-1}] . W), one rounding of the exact-in-double sum. */
    for (int64_t v = 0; v < V; ++v) {
      double acc = 0.0;
      for (int32_t j = 0; j < R; ++j) acc += (double)urow[j] * (double)W[(int64_t)j * V + v];
      uint16_t h = orc_bf16_round((double)brow[v] + acc);
      if (z_out) z_out[(int64_t)(k - 1) * V + v] = h;
      z[v] = bf16_value(h);
    }
    /* Sample x_k from softmax(z_k) by the exponential race on the logits (DRAFT tag). */
    race_t r;
    race_init(&r);
    double M = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
      if (isnan(z[v]) || (isinf(z[v]) && z[v] > 0)) {
        free(z);
        return ORC_ERR_NAN;
      }
      if (z[v] > M) M = z[v];
    }
    if (isinf(M)) {
      free(z);
      return ORC_ERR_NAN;
    }
    double S = 0.0;
    for (int64_t v = 0; v < V; ++v) {
      S += exp(z[v] - M);
      if (isinf(z[v])) continue;
      race_offer(&r, z[v] + race_noise(seed, req, (uint32_t)k, ORC_TAG_DRAFT, (uint64_t)v), v);
    }
    x_out[k - 1] = (int32_t)r.arg;
    if (stats_out) {
      stats_out[2 * (k - 1)] = M;
      stats_out[2 * (k - 1) + 1] = M + log(S);
    }
    if (conf_out) conf_out[k - 1] = orc_sts_confidence(scores[k - 1], T[k - 1]);
    if (margin_out) margin_out[k - 1] = race_margin(&r);
    prev = (int32_t)r.arg;
  }
  free(z);
  return ORC_OK;
}

/* ---- scheduler ---------------------------------------------------------------------------- */

typedef struct {
  float S;
  int32_t k, i;
} sched_item;

static int item_order(const void* a, const void* b) {
  const sched_item* x = (const sched_item*)a;
  const sched_item* y = (const sched_item*)b;
  if (x->S != y->S) return x->S > y->S ? -1 : 1; /* survival descending */
  if (x->k != y->k) return x->k < y->k ? -1 : 1; /* shorter prefix first */
  if (x->i != y->i) return x->i < y->i ? -1 : 1; /* lower request index first */
  return 0;
}

int orc_schedule_rule(const float* cond_accept, const int32_t* max_len, int32_t N, int32_t K,
                      const double* sps, int32_t B_max, int32_t rule, int32_t* sel_len,
                      float* survival, int32_t* total_rows, double* objective) {
  if (N < 0 || K < 0 || B_max < N || !sel_len || !total_rows || !objective) return ORC_ERR_ARGS;
  if (rule != ORC_STOP_FIRST_DROP && rule != ORC_STOP_ARGMAX && rule != ORC_STOP_FIXED_DEPTH)
    return ORC_ERR_ARGS;
  int64_t n_items = 0;
  for (int32_t i = 0; i < N; ++i) {
    if (max_len[i] < 0 || max_len[i] > K) return ORC_ERR_ARGS;
    n_items += max_len[i];
  }
  sched_item* items = (sched_item*)malloc(sizeof(sched_item) * (size_t)(n_items > 0 ? n_items : 1));
  int64_t n = 0;
  for (int32_t i = 0; i < N; ++i) {
    float S = 1.0f;
    for (int32_t k = 1; k <= K; ++k) {
      float c = cond_accept[(int64_t)i * K + (k - 1)];
      if (k <= max_len[i]) {
        if (!(c >= 0.0f && c <= 1.0f)) {
          free(items);
          return ORC_ERR_NAN;
        }
        S = S * c; /* prefix survival: product of conditional acceptance probabilities */
        items[n].S = S;
        items[n].k = k;
        items[n].i = i;
        ++n;
      }
      if (survival) survival[(int64_t)i * K + (k - 1)] = k <= max_len[i] ? S : 0.0f;
    }
    sel_len[i] = 0;
  }
  const double two40 = ldexp(1.0, 40);
  if (rule == ORC_STOP_FIXED_DEPTH) {
    /* one depth k for every request (min(k, max_len) drafts each): T(k) = N + sum of survivals up
       to depth k, B(k) = N + sum of min(k, max_len); stop at the first k whose next depth does not
       raise f, or whose next depth would exceed B_max */
    int64_t Tk = (int64_t)N << 40, Bk = N;
    double f = (double)Tk * ldexp(1.0, -40) * sps[N];
    int32_t depth = 0;
    for (int32_t k = 1; k <= K; ++k) {
      int64_t Tn = Tk, Bn = Bk;
      for (int32_t i = 0; i < N; ++i) {
        if (k > max_len[i]) continue;
        float S = 1.0f;
        for (int32_t j = 1; j <= k; ++j) S = S * cond_accept[(int64_t)i * K + (j - 1)];
        Tn += (int64_t)floor((double)S * two40);
        Bn += 1;
      }
      if (Bn > (int64_t)B_max || Bn == Bk) break;
      double fn = (double)Tn * ldexp(1.0, -40) * sps[Bn];
      if (!(fn > f)) break;
      Tk = Tn;
      Bk = Bn;
      f = fn;
      depth = k;
    }
    for (int32_t i = 0; i < N; ++i) sel_len[i] = depth < max_len[i] ? depth : max_len[i];
    *total_rows = (int32_t)Bk;
    *objective = f;
    free(items);
    return ORC_OK;
  }
  qsort(items, (size_t)n_items, sizeof(sched_item), item_order);

  int64_t Tb = (int64_t)N << 40; /* one guaranteed token per request, in 2^-40 units */
  double f = (double)Tb * ldexp(1.0, -40) * sps[N];
  int64_t b = 0;
  if (rule == ORC_STOP_FIRST_DROP) {
    while (b < n_items && (int64_t)N + b + 1 <= (int64_t)B_max) {
      int64_t F = (int64_t)floor((double)items[b].S * two40);
      int64_t Tn = Tb + F;
      double fn = (double)Tn * ldexp(1.0, -40) * sps[N + b + 1];
      if (!(fn > f)) break; /* early stop: never look past the first non-increase */
      Tb = Tn;
      f = fn;
      ++b;
    }
  } else {
    /* every admissible budget b = 0 .. min(items, B_max - N); the largest f(b), the smallest b
       among equals */
    const int64_t b_lim = n_items < (int64_t)B_max - N ? n_items : (int64_t)B_max - N;
    double best = f;
    for (int64_t j = 1; j <= b_lim; ++j) {
      Tb += (int64_t)floor((double)items[j - 1].S * two40);
      double fj = (double)Tb * ldexp(1.0, -40) * sps[N + j];
      if (fj > best) {
        best = fj;
        b = j;
      }
    }
    f = best;
  }
  for (int64_t j = 0; j < b; ++j) sel_len[items[j].i] += 1;
  *total_rows = (int32_t)(N + b);
  *objective = f;
  free(items);
  return ORC_OK;
}

int orc_schedule(const float* cond_accept, const int32_t* max_len, int32_t N, int32_t K,
                 const double* sps, int32_t B_max, int32_t* sel_len, float* survival,
                 int32_t* total_rows, double* objective) {
  return orc_schedule_rule(cond_accept, max_len, N, K, sps, B_max, ORC_STOP_FIRST_DROP, sel_len,
                           survival, total_rows, objective);
}

/* ---- asynchronous scheduling: predictions from two rounds before ------------------------------ */

int orc_schedule_async(const float* conf_rounds, int64_t round, const float* prior,
                       const int32_t* max_len, int32_t N, int32_t K, const double* sps,
                       int32_t B_max, int32_t rule, int32_t* sel_len, float* survival,
                       int32_t* total_rows, double* objective) {
  if (round < 0) return ORC_ERR_ARGS;
  const float* cond = round >= 2 ? conf_rounds + (size_t)(round - 2) * (size_t)N * (size_t)K : prior;
  return orc_schedule_rule(cond, max_len, N, K, sps, B_max, rule, sel_len, survival, total_rows,
                           objective);
}

/* ---- online per-position acceptance ----------------------------------------------------------- */

int orc_acceptance_update(const int32_t* sel_len, const int32_t* accepted_len, int32_t N,
                          int32_t K, double decay, double prior_a, double prior_b, double* trials,
                          double* accepts, float* alpha) {
  if (N < 0 || K < 0 || !trials || !accepts || !alpha) return ORC_ERR_ARGS;
  if (!(decay >= 0.0 && decay <= 1.0) || !(prior_a > 0.0) || !(prior_b > 0.0)) return ORC_ERR_ARGS;
  if (N > 0 && (!sel_len || !accepted_len)) return ORC_ERR_ARGS;
  int bad = 0;
  for (int32_t k = 1; k <= K; ++k) {
    /* position k was reached by request i when every earlier drafted token was accepted and k was
       verified: k <= min(accepted + 1, verified); it was accepted when k <= accepted */
    int64_t reached = 0, taken = 0;
    for (int32_t i = 0; i < N; ++i) {
      const int32_t s = sel_len[i], a = accepted_len[i];
      if (s < 0 || s > K || a < 0 || a > s) {
        bad = 1;
        continue;
      }
      const int32_t last = a + 1 < s ? a + 1 : s;
      if (k <= last) ++reached;
      if (k <= a) ++taken;
    }
    trials[k - 1] = decay * trials[k - 1] + (double)reached;
    accepts[k - 1] = decay * accepts[k - 1] + (double)taken;
    /* posterior mean of the conditional acceptance probability under a Beta(prior_a, prior_b)
       prior */
    alpha[k - 1] = (float)((accepts[k - 1] + prior_a) / (trials[k - 1] + prior_a + prior_b));
  }
  return bad ? ORC_ERR_NAN : ORC_OK;
}

/* ---- sequential temperature scaling: fit and calibration error ------------------------------ */

static double logistic(double x) { return 1.0 / (1.0 + exp(-x)); }

/* log(1 + exp(x)) without overflow */
static double softplus(double x) { return x > 0.0 ? x + log1p(exp(-x)) : log1p(exp(x)); }

int orc_sts_fit(const float* scores, const int32_t* sel_len, const int32_t* accepted_len,
                int32_t N, int32_t K, int32_t iters, double beta_min, double beta_max,
                int32_t nbins, float* T_out, double* nll_out, double* ece_raw_out,
                double* ece_fit_out, int32_t* count_out) {
  if (N < 0 || K < 0 || iters < 0 || nbins <= 0 || !T_out) return ORC_ERR_ARGS;
  if (!(beta_min > 0.0) || !(beta_max >= beta_min)) return ORC_ERR_ARGS;
  if (N > 0 && (!scores || !sel_len || !accepted_len)) return ORC_ERR_ARGS;
  int bad = 0;
  for (int32_t i = 0; i < N; ++i) {
    const int32_t s = sel_len[i], a = accepted_len[i];
    if (s < 0 || s > K || a < 0 || a > s) bad = 1;
  }
  double* bin_gap = (double*)malloc(sizeof(double) * (size_t)nbins);
  for (int32_t k = 1; k <= K; ++k) {
    /* the samples of position k: requests that reached it (every earlier drafted token accepted,
       k verified); the label says whether it was accepted */
    int32_t n = 0;
    for (int32_t i = 0; i < N; ++i) {
      const int32_t s = sel_len[i], a = accepted_len[i];
      if (s < 0 || s > K || a < 0 || a > s) continue;
      if (k <= (a + 1 < s ? a + 1 : s)) ++n;
    }
    /* Newton's method on the convex negative log-likelihood in beta = 1 / T:
         NLL(beta) = sum_i softplus(-(2 y_i - 1) beta s_i)
         g = sum_i (sigma(beta s_i) - y_i) s_i,  H = sum_i sigma(beta s_i) (1 - sigma(beta s_i)) s_i^2
       starting from beta = 1, each step clamped to [beta_min, beta_max] */
    double beta = 1.0;
    for (int32_t t = 0; t < iters; ++t) {
      double g = 0.0, H = 0.0;
      for (int32_t i = 0; i < N; ++i) {
        const int32_t s = sel_len[i], a = accepted_len[i];
        if (s < 0 || s > K || a < 0 || a > s) continue;
        if (!(k <= (a + 1 < s ? a + 1 : s))) continue;
        const double x = (double)scores[(int64_t)i * K + (k - 1)];
        const double y = k <= a ? 1.0 : 0.0;
        const double q = logistic(beta * x);
        g += (q - y) * x;
        H += q * (1.0 - q) * x * x;
      }
      if (!(H > 0.0)) break;
      double nb = beta - g / H;
      if (nb < beta_min) nb = beta_min;
      if (nb > beta_max) nb = beta_max;
      beta = nb;
    }
    T_out[k - 1] = (float)(1.0 / beta);
    /* the fitted loss and the expected calibration error (equal-width bins over [0, 1]:
       sum over bins of |sum (label - confidence)|, over the samples) before and after */
    double nll = 0.0;
    for (int pass = 0; pass < 2; ++pass) {
      const double b = pass == 0 ? 1.0 : beta;
      for (int32_t j = 0; j < nbins; ++j) bin_gap[j] = 0.0;
      for (int32_t i = 0; i < N; ++i) {
        const int32_t s = sel_len[i], a = accepted_len[i];
        if (s < 0 || s > K || a < 0 || a > s) continue;
        if (!(k <= (a + 1 < s ? a + 1 : s))) continue;
        const double x = (double)scores[(int64_t)i * K + (k - 1)];
        const double y = k <= a ? 1.0 : 0.0;
        const double q = logistic(b * x);
        int32_t bin = (int32_t)floor(q * nbins);
        if (bin >= nbins) bin = nbins - 1;
        if (bin < 0) bin = 0;
        bin_gap[bin] += y - q;
        if (pass == 1) nll += softplus(-(2.0 * y - 1.0) * b * x);
      }
      double ece = 0.0;
      for (int32_t j = 0; j < nbins; ++j) ece += fabs(bin_gap[j]);
      ece = n > 0 ? ece / n : 0.0;
      if (pass == 0 && ece_raw_out) ece_raw_out[k - 1] = ece;
      if (pass == 1 && ece_fit_out) ece_fit_out[k - 1] = ece;
    }
    if (nll_out) nll_out[k - 1] = n > 0 ? nll / n : 0.0;
    if (count_out) count_out[k - 1] = n;
  }
  free(bin_gap);
  return bad ? ORC_ERR_NAN : ORC_OK;
}
