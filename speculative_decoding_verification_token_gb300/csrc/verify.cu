// verify.cu -- block verification and draft sampling from q (token-level verification is in
// token.cu).
//
// Block verification ("How much does a token cost", "Block verification") is one kernel: one
// CTA per request (a persistent grid when requests outnumber the SMs), the stream ring's producer
// / consumer layout.  The CTA walks its request's row pairs in order, each pair's statistics pass
// from HBM followed by its residual pass re-read from L2, decides the request (thresholds h_i, the
// longest passing prefix), then streams the correction (or bonus) row through the same ring and
// runs the exponential race over it.
// Draft sampling ("Speculative Decoding: The Same Distribution, Twice as Fast" §3 step 1) races
// every drafted row from its own softmax, one row split into contiguous shares over a few CTAs.
// The allocation-free token-level entry point closes the file.
#include <mutex>

#include <cuda.h>

#include "verify_common.cuh"

namespace sv {

constexpr int kRaceSplitMax = 8;                 // CTAs (row shares) per race job, many jobs
constexpr int kRaceSplitFew = 16;                // the same when one wave holds every share
constexpr int kRaceCtasPerSm = 4;                // resident race CTAs per SM (launch bounds)
constexpr uint32_t kRaceShareMax = 64 * 1024;    // largest row share staged in shared memory

// ---------------------------------------------------------------------------------------------
// block: one CTA per request -- statistics, running ratios, residual masses and the decision
// ---------------------------------------------------------------------------------------------
// Block verification needs, for every i < gamma, the residual mass
//   R_i = sum_x max(rho_i p_{i+1}(x) - q_{i+1}(x), 0),
// which depends on the normalisers of row pair i + 1 and on rho_i, i.e. on every earlier pair.
// The CTA walks its request's row pairs in order: the statistics pass of pair j streams it from
// HBM, and the residual pass over pair j (with rho_{j-1}) follows at once, re-reading the pair
// from L2 (about half a megabyte per CTA in flight at V = 129280).
// The threshold h_i = R_i / (R_i + 1 - rho_i) never exceeds rho_i, because R_i <= rho_i, so a
// position whose uniform eta_i exceeds rho_i fails whatever R_i is: unless the caller asks for
// every h_i, the residual pass runs only for positions with eta_i <= rho_i.  The decision is the
// same either way.
struct BlockParams {
  const uint8_t* target;
  const uint8_t* draft;
  int64_t V, ld;
  const int64_t* target_row0;
  const int64_t* draft_row0;
  const int32_t* draft_len;
  const int32_t* draft_tokens;
  int32_t B, gmax;
  uint64_t seed;
  const uint64_t* request_ids;
  float* rho_out;  // rho_i per drafted row (nullable)
  float* h_out;    // h_i per drafted row (nullable; non-null computes every R_i)
  int32_t* accepted_len;
  int32_t* out_tokens;
  int64_t out_ld;
  int32_t* correction_token;
  VerifyWs ws;
  int32_t* status;
};

enum : int32_t { kSegStats = 0, kSegResid = 1, kSegEnd = 2, kSegExit = 3, kSegRace = 4 };

struct BlockMeta {
  int32_t kind;  // kSeg*
  int32_t row;   // row pair j of the request (1-based)
  int32_t last;  // this stage closes its segment
  int32_t len;   // elements of the slice
  int32_t bulk;  // elements brought by the bulk copies (the rest is read from global)
  int32_t seg;   // running segment number of this CTA (selects the merge buffer)
  int32_t r;     // request
  uint32_t seq;  // running request number of this CTA (1, 2, ...)
  int64_t e0;    // first vocabulary index of the slice
  const uint8_t* trow;
  const uint8_t* drow;
};

constexpr int kBlockRows = SV_MAX_DRAFT_LEN + 1;

struct BlockState {  // the request in flight, in shared memory
  float4 norm[kBlockRows];       // (m_t, s_t, m_d, s_d) of row pair j, m in log2 units
  float rho[kBlockRows];         // rho_j
  float eta[kBlockRows];         // eta_j (ACCEPT uniform of position j)
  float R[kBlockRows];           // R_i, the residual mass over pair i + 1
  int32_t cand[kBlockRows];      // R_i is needed: eta_i <= rho_i and i < gamma
  uint32_t norm_seq[kBlockRows]; // request number whose norm[j] is published
  uint32_t rho_seq[kBlockRows];  // request number whose rho[j], eta[j], cand[j] are published
  float dep[kRedBufs][kConsumerWarps][4];
  int32_t count[kRedBufs];       // warps that have deposited a segment
  int32_t bad;                   // data error seen in the request in flight
  RaceDesc desc;                 // the decision: tau, residual or bonus, gap
  uint32_t desc_seq;             // request number whose desc is published
  uint32_t race_k0;              // key_order of the best exact key of the race so far (0: none)
};

template <typename E>
__device__ void block_producer(const BlockParams& p, uint8_t* ring, uint64_t* full,
                               uint64_t* empty, BlockMeta* meta, BlockState* bs) {
  constexpr int32_t kSE = kRowBytes / esize<E>();
  uint32_t n = 0;   // stages issued so far
  int32_t seg = 0;  // segments issued so far
  uint32_t seq = 0;
  auto acquire = [&](uint32_t& stage) {
    stage = n % kRing;
    return n < kRing || mbar_wait(&empty[stage], ((n / kRing) - 1) & 1, p.status);
  };
  // every slice of one row pair, as one segment
  auto issue_pair = [&](int32_t kind, int32_t r, int32_t j) {
    const uint8_t* trow = row_ptr<E>(p.target, p.target_row0[r] + (j - 1), p.ld);
    const uint8_t* drow = row_ptr<E>(p.draft, p.draft_row0[r] + (j - 1), p.ld);
    for (int64_t e0 = 0; e0 < p.V; e0 += kSE) {
      uint32_t stage;
      if (!acquire(stage)) return false;
      BlockMeta m;
      m.kind = kind;
      m.row = j;
      m.last = e0 + kSE >= p.V;
      m.len = static_cast<int32_t>(p.V - e0 < kSE ? p.V - e0 : kSE);
      const uint32_t bulk_bytes = (uint32_t(m.len) * esize<E>()) & ~15u;
      m.bulk = static_cast<int32_t>(bulk_bytes / esize<E>());
      m.seg = seg;
      m.r = r;
      m.seq = seq;
      m.e0 = e0;
      m.trow = trow;
      m.drow = drow;
      meta[stage] = m;
      uint8_t* dst = ring + size_t(stage) * 2 * kRowBytes;
      fence_proxy_async();
      mbar_expect_tx(&full[stage], 2 * bulk_bytes);
      if (bulk_bytes) {
        bulk_g2s(dst, trow + e0 * esize<E>(), bulk_bytes, &full[stage]);
        bulk_g2s(dst + kRowBytes, drow + e0 * esize<E>(), bulk_bytes, &full[stage]);
      }
      ++n;
    }
    ++seg;
    return true;
  };
  // the correction (or bonus) row of the decided request: row pair tau + 1, or target row gamma + 1
  auto issue_race = [&](int32_t r, const RaceDesc& d) {
    const uint8_t* trow = row_ptr<E>(p.target, p.target_row0[r] + d.tau, p.ld);
    const uint8_t* drow = d.resid ? row_ptr<E>(p.draft, p.draft_row0[r] + d.tau, p.ld) : nullptr;
    for (int64_t e0 = 0; e0 < p.V; e0 += kSE) {
      uint32_t stage;
      if (!acquire(stage)) return false;
      BlockMeta m;
      m.kind = kSegRace;
      m.row = d.tau + 1;
      m.last = e0 + kSE >= p.V;
      m.len = static_cast<int32_t>(p.V - e0 < kSE ? p.V - e0 : kSE);
      const uint32_t bulk_bytes = (uint32_t(m.len) * esize<E>()) & ~15u;
      m.bulk = static_cast<int32_t>(bulk_bytes / esize<E>());
      m.seg = seg;
      m.r = r;
      m.seq = seq;
      m.e0 = e0;
      m.trow = trow;
      m.drow = drow;
      meta[stage] = m;
      uint8_t* dst = ring + size_t(stage) * 2 * kRowBytes;
      fence_proxy_async();
      mbar_expect_tx(&full[stage], (drow ? 2 : 1) * bulk_bytes);
      if (bulk_bytes) {
        bulk_g2s(dst, trow + e0 * esize<E>(), bulk_bytes, &full[stage]);
        if (drow) bulk_g2s(dst + kRowBytes, drow + e0 * esize<E>(), bulk_bytes, &full[stage]);
      }
      ++n;
    }
    ++seg;
    return true;
  };
  auto issue_marker = [&](int32_t kind, int32_t r) {
    uint32_t stage;
    if (!acquire(stage)) return false;
    BlockMeta m = {};
    m.kind = kind;
    m.last = 1;
    m.seg = seg;
    m.r = r;
    m.seq = seq;
    meta[stage] = m;
    mbar_arrive(&full[stage]);
    ++n;
    ++seg;
    return true;
  };
  for (int32_t r = blockIdx.x; r < p.B; r += gridDim.x) {
    ++seq;
    const int32_t g = clamp_gamma(p.draft_len[r], p.gmax);
    for (int32_t j = 1; j <= g; ++j) {
      if (!issue_pair(kSegStats, r, j)) return;
      if (j >= 2) {
        // R_{j-1}, over pair j, is needed when eta_{j-1} <= rho_{j-1} or every h is asked for
        if (!wait_seq(&bs->rho_seq[j - 1], seq, p.status)) return;
        if ((p.h_out || bs->cand[j - 1]) && !issue_pair(kSegResid, r, j)) return;
      }
    }
    if (!issue_marker(kSegEnd, r)) return;
    if (!wait_seq(&bs->desc_seq, seq, p.status)) return;
    const RaceDesc d = bs->desc;
    if (!issue_race(r, d)) return;
  }
  issue_marker(kSegExit, -1);
}

// One pair of residual entries: the positive part of rho p - q, written (up to the per-row factor
// rho / s_t) as 2^(t log2e - m_t) (1 - exp(y)) with y = min((d - t) + gap, 0).  1 - exp(y) is kept
// accurate relative to itself: near 0 by the Taylor series of -expm1 to degree 6 (truncation below
// 5e-8 relative for |y| <= 1/4), further out as 1 - 2^(y log2e).  Entries with y >= 0 add 0.
__device__ __forceinline__ float2 resid_pair(float2 acc, float2 t, float2 d, float2 gap,
                                             float2 nmt) {
  float2 y = add2(fma2(t, splat2(-1.f), d), gap);
  y.x = fminf(y.x, 0.f);
  y.y = fminf(y.y, 0.f);
  const float2 e = exp2_2(fma2(t, splat2(kLog2e), nmt));
  const float2 big = fma2(exp2_2(mul2(y, splat2(kLog2e))), splat2(-1.f), splat2(1.f));
  float2 s = splat2(-1.f / 720.f);
  s = fma2(s, y, splat2(-1.f / 120.f));
  s = fma2(s, y, splat2(-1.f / 24.f));
  s = fma2(s, y, splat2(-1.f / 6.f));
  s = fma2(s, y, splat2(-0.5f));
  s = fma2(s, y, splat2(-1.f));
  s = mul2(s, y);
  const float2 om = make_float2(y.x > -0.25f ? s.x : big.x, y.y > -0.25f ? s.y : big.y);
  return fma2(e, om, acc);
}

template <typename E>
__device__ __forceinline__ float2 resid_vec(float2 acc, const uint4& a, const uint4& b,
                                            float2 gap, float2 nmt) {
  if constexpr (Elem<E>::kPerVec == 8) {
    acc = resid_pair(acc, bf16x2_f2(a.x), bf16x2_f2(b.x), gap, nmt);
    acc = resid_pair(acc, bf16x2_f2(a.y), bf16x2_f2(b.y), gap, nmt);
    acc = resid_pair(acc, bf16x2_f2(a.z), bf16x2_f2(b.z), gap, nmt);
    acc = resid_pair(acc, bf16x2_f2(a.w), bf16x2_f2(b.w), gap, nmt);
  } else {
    acc = resid_pair(acc, make_float2(__uint_as_float(a.x), __uint_as_float(a.y)),
                     make_float2(__uint_as_float(b.x), __uint_as_float(b.y)), gap, nmt);
    acc = resid_pair(acc, make_float2(__uint_as_float(a.z), __uint_as_float(a.w)),
                     make_float2(__uint_as_float(b.z), __uint_as_float(b.w)), gap, nmt);
  }
  return acc;
}

// The decision of request r, by one warp once every segment of the request is merged: thresholds
// h_i, the accepted length tau = max{i : eta_i <= h_i} (0 if none), the race descriptor.
template <typename E>
__device__ void block_decide(const BlockParams& p, int32_t r, uint32_t seq, BlockState* bs) {
  if ((threadIdx.x & 31) != 0) return;
  const int32_t graw = p.draft_len[r];
  const int32_t g = clamp_gamma(graw, p.gmax);
  int32_t tau = 0;
  for (int32_t i = 1; i <= g; ++i) {
    float h;
    if (i == g) {
      h = bs->rho[i];
    } else if (p.h_out || bs->cand[i]) {
      const float den = bs->R[i] + (1.f - bs->rho[i]);
      h = den > 0.f ? bs->R[i] / den : 1.f;
    } else {
      h = -1.f;  // eta_i > rho_i >= h_i: position i fails whatever R_i is
    }
    const int64_t row = p.draft_row0[r] + (i - 1);
    if (p.h_out) p.h_out[row] = h;
    if (p.rho_out) p.rho_out[row] = bs->rho[i];
    if (bs->eta[i] <= h) tau = i;
  }
  RaceDesc d;
  d.tau = tau;
  d.resid = tau < g;
  d.gap = d.resid ? resid_gap(bs->norm[tau + 1], tau > 0 ? logf(bs->rho[tau]) : 0.f) : 0.f;
  d.pad = 0;
  if (graw != g || bs->bad) report(p.status, SV_ERR_BAD_INPUT);
  bs->bad = 0;
  bs->desc = d;
  bs->race_k0 = 0u;
  publish_seq(&bs->desc_seq, seq);  // the producer may stream the race's row now
}

// ---- the correction (or bonus) race of a decided request, streamed through the ring ----------

// Offers entry e (logit t, draft logit d, Philox word w) to this thread's race if its noise can lift
// it to the bound (gate constant c = 23 - K0 log2e; see gate_threshold).
__device__ __forceinline__ void race_offer_td(const RaceSpec& rs, int64_t e, float t, float d,
                                              uint32_t w, float c, float& bk, int32_t& bi) {
  if (!(gate_m(w) <= gate_threshold(t, c))) return;
  if (!race_active(rs, t, d)) return;
  const float k = race_key(rs, t, d, race_noise(uniform_of(w)));
  if (race_better(k, int32_t(e), bk, bi)) {
    bk = k;
    bi = int32_t(e);
  }
}

// Exact key of entry e (-inf if it carries no weight).
__device__ __forceinline__ float race_exact_td(const RaceSpec& rs, int64_t e, float t, float d) {
  if (!race_active(rs, t, d)) return -INFINITY;
  const uint4 b = stream_block(rs.st, static_cast<uint32_t>(e >> 2));
  return race_key(rs, t, d, race_noise(uniform_of(word_of(b, static_cast<uint32_t>(e & 3)))));
}

// Seed of one stage: the exact key of this thread's largest-logit entry among its whole vectors.
template <typename E>
__device__ float race_stage_seed(const RaceSpec& rs, const uint4* vt, const uint4* vd, int nvec,
                                 int64_t e0, int tid, int32_t& idx) {
  constexpr int kPer = Elem<E>::kPerVec;
  float bt = -INFINITY;
  int bv = -1;
  for (int v = tid; v < nvec; v += kConsumers) {
    const float m = vec_max<E>(vt[v]);
    if (m > bt) {
      bt = m;
      bv = v;
    }
  }
  idx = -1;
  if (bv < 0) return -INFINITY;
  float x[8], y[8];
  Elem<E>::unpack(vt[bv], x);
  if (rs.resid) Elem<E>::unpack(vd[bv], y);
  int q0 = 0;
#pragma unroll
  for (int q = kPer - 1; q >= 0; --q)
    if (x[q] == bt) q0 = q;
  const int64_t e = e0 + int64_t(bv) * kPer + q0;
  idx = int32_t(e);
  return race_exact_td(rs, e, bt, rs.resid ? y[q0] : 0.f);
}

// Main pass of one stage against the bound K0: vectors whose largest logit cannot reach K0 are
// skipped before any Philox; the others are gated by their largest Philox word, then entry by
// entry (the race kernel's gate, with the draft logits at hand in the stage).
template <typename E>
__device__ void race_stage_main(const RaceSpec& rs, const uint4* vt, const uint4* vd, int nvec,
                                int32_t len, int64_t e0, const uint8_t* trow,
                                const uint8_t* drow, int tid, float K0, float& bk, int32_t& bi) {
  constexpr int kPer = Elem<E>::kPerVec;
  const float floor_t = K0 - kMaxNoise;
  const float c = 23.0f - K0 * kLog2e;
  for (int v = tid; v < nvec; v += kConsumers) {
    const uint4 a = vt[v];
    const float tmax = vec_max<E>(a);
    if (!(tmax >= floor_t)) continue;
    const int64_t e = e0 + int64_t(v) * kPer;  // a multiple of kPer: whole Philox blocks
    const uint4 b0 = stream_block(rs.st, static_cast<uint32_t>(e >> 2));
    const uint4 b1 = kPer == 8 ? stream_block(rs.st, static_cast<uint32_t>(e >> 2) + 1) : b0;
    const uint32_t wmax = max(max(max(b0.x, b0.y), max(b0.z, b0.w)),
                              max(max(b1.x, b1.y), max(b1.z, b1.w)));
    if (gate_m(wmax) > gate_threshold(tmax, c)) continue;
    float x[8], y[8];
    Elem<E>::unpack(a, x);
    if (rs.resid) Elem<E>::unpack(vd[v], y);
    const uint32_t w[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int q = 0; q < kPer; ++q)
      race_offer_td(rs, e + q, x[q], rs.resid ? y[q] : 0.f, w[q], c, bk, bi);
  }
  for (int i = nvec * kPer + tid; i < len; i += kConsumers) {  // ragged tail, from global memory
    const int64_t e = e0 + i;
    const float t = Elem<E>::load(trow, e);
    if (!(t >= floor_t)) continue;
    const float d = rs.resid ? Elem<E>::load(drow, e) : 0.f;
    const uint4 b = stream_block(rs.st, static_cast<uint32_t>(e >> 2));
    race_offer_td(rs, e, t, d, word_of(b, static_cast<uint32_t>(e & 3)), c, bk, bi);
  }
}

// The race's winner and the request's outputs, by the warp that merged the race; a residual with
// no positive entry left (p and q agree to working precision) is drawn from p with the same
// uniforms, by this warp over the whole row.
template <typename E>
__device__ void block_finish(const BlockParams& p, const BlockMeta& m, const RaceSpec& rs,
                             const RaceDesc& d, int32_t y) {
  const int lane = threadIdx.x & 31;
  if (y < 0 && rs.resid) {
    RaceSpec fb = rs;
    fb.resid = false;
    float bk = -INFINITY;
    int32_t bi = -1;
    for (int64_t e = lane; e < p.V; e += 32) {
      const float t = Elem<E>::load(m.trow, e);
      const float k = race_exact_td(fb, e, t, 0.f);
      if (k > -INFINITY && race_better(k, int32_t(e), bk, bi)) {
        bk = k;
        bi = int32_t(e);
      }
    }
    warp_race(bk, bi);
    y = bi;
  }
  int32_t* out = p.out_tokens + size_t(m.r) * p.out_ld;
  for (int64_t q = lane; q < p.out_ld; q += 32) {
    int32_t v = -1;
    if (q < d.tau) v = p.draft_tokens[p.draft_row0[m.r] + q];
    else if (q == d.tau) v = y;
    out[q] = v;
  }
  if (lane == 0) {
    if (y < 0) report(p.status, SV_ERR_BAD_INPUT);  // the row carries no probability at all
    p.accepted_len[m.r] = d.tau;
    if (p.correction_token) p.correction_token[m.r] = y;
  }
}

template <typename E>
__device__ void block_consumer(const BlockParams& p, const uint8_t* ring, uint64_t* full,
                               uint64_t* empty, const BlockMeta* meta, BlockState* bs) {
  constexpr int kPer = Elem<E>::kPerVec;
  constexpr int kFull = int(kRowBytes / 16) / kConsumers;
  static_assert(kFull * kConsumers * 16 == int(kRowBytes), "stage not a whole multiple");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float mt = kM2Empty, st = 0.f, md = kM2Empty, sd = 0.f;
  float2 acc = make_float2(0.f, 0.f);
  float2 gap = splat2(0.f), nmt = splat2(0.f);
  float A = 0.f;
  int32_t cur_seg = -1;
  RaceSpec rs{};  // the race of the request in flight
  float bk = -INFINITY;
  int32_t bi = -1;
  for (uint32_t n = 0;; ++n) {
    const uint32_t stage = n % kRing;
    if (!mbar_wait(&full[stage], (n / kRing) & 1, p.status)) return;
    const BlockMeta m = meta[stage];
    if (m.kind == kSegExit) return;
    const uint4* vt = reinterpret_cast<const uint4*>(ring + size_t(stage) * 2 * kRowBytes);
    const uint4* vd = vt + kRowBytes / 16;
    const int nvec = m.bulk / kPer;
    const bool whole = m.bulk == int32_t(kRowBytes / esize<E>());
    if (m.kind == kSegStats) {
      if (whole) {
        uint4 a[kFull], b[kFull];
#pragma unroll
        for (int u = 0; u < kFull; ++u) a[u] = vt[tid + u * kConsumers];
#pragma unroll
        for (int u = 0; u < kFull; ++u) b[u] = vd[tid + u * kConsumers];
        if constexpr (kPer == 8) {
          ms2_fold_vecs_bf16<kFull>(mt, st, a);
          ms2_fold_vecs_bf16<kFull>(md, sd, b);
        } else {
          ms2_fold_vecs_f32<kFull>(mt, st, a);
          ms2_fold_vecs_f32<kFull>(md, sd, b);
        }
      } else {
        for (int v = tid; v < nvec; v += kConsumers) {
          if constexpr (kPer == 8) {
            ms2_vec_bf16(mt, st, vt[v]);
            ms2_vec_bf16(md, sd, vd[v]);
          } else {
            ms2_vec_f32(mt, st, vt[v]);
            ms2_vec_f32(md, sd, vd[v]);
          }
        }
        for (int e = m.bulk + tid; e < m.len; e += kConsumers) {
          ms2_one(mt, st, Elem<E>::load(m.trow, m.e0 + e));
          ms2_one(md, sd, Elem<E>::load(m.drow, m.e0 + e));
        }
      }
    } else if (m.kind == kSegResid) {
      if (m.seg != cur_seg) {
        // first stage of the residual pass over pair j: rho_{j-1} p_j(x) = A 2^(t log2e - m_t)
        // with A = rho_{j-1} / s_t, and q_j(x) / (rho_{j-1} p_j(x)) = exp((d - t) + gap)
        int32_t ok = 1;
        if (lane == 0)
          ok = wait_seq(&bs->norm_seq[m.row], m.seq, p.status) &&
               wait_seq(&bs->rho_seq[m.row - 1], m.seq, p.status);
        if (!__shfl_sync(0xffffffffu, ok, 0)) return;
        __syncwarp();
        const float4 nm = bs->norm[m.row];
        const float rho_prev = bs->rho[m.row - 1];
        A = rho_prev / nm.y;
        gap = splat2(resid_gap(nm, logf(rho_prev)));
        nmt = splat2(-nm.x);
        cur_seg = m.seg;
      }
      if (whole) {
        uint4 a[kFull], b[kFull];
#pragma unroll
        for (int u = 0; u < kFull; ++u) a[u] = vt[tid + u * kConsumers];
#pragma unroll
        for (int u = 0; u < kFull; ++u) b[u] = vd[tid + u * kConsumers];
#pragma unroll
        for (int u = 0; u < kFull; ++u) acc = resid_vec<E>(acc, a[u], b[u], gap, nmt);
      } else {
        for (int v = tid; v < nvec; v += kConsumers) acc = resid_vec<E>(acc, vt[v], vd[v], gap, nmt);
        for (int e = m.bulk + tid; e < m.len; e += kConsumers) {
          const float2 t = make_float2(Elem<E>::load(m.trow, m.e0 + e), -INFINITY);
          const float2 d = make_float2(Elem<E>::load(m.drow, m.e0 + e), -INFINITY);
          acc = resid_pair(acc, t, d, gap, nmt);
        }
      }
    } else if (m.kind == kSegRace) {
      if (m.seg != cur_seg) {
        // first stage of the request's race: its stream, then a bound from this stage's seeds
        int32_t ok = 1;
        if (lane == 0) ok = wait_seq(&bs->desc_seq, m.seq, p.status);
        if (!__shfl_sync(0xffffffffu, ok, 0)) return;
        __syncwarp();
        const RaceDesc d = bs->desc;
        const uint64_t req = p.request_ids ? p.request_ids[m.r] : uint64_t(m.r);
        rs.resid = d.resid != 0;
        rs.gap = d.gap;
        rs.st = make_stream(p.seed, req, uint32_t(d.tau + 1), rs.resid ? kTagResid : kTagBonus);
        cur_seg = m.seg;
        int32_t si;
        const float sk = race_stage_seed<E>(rs, vt, vd, nvec, m.e0, tid, si);
        bk = sk > -INFINITY ? sk : -INFINITY;
        bi = sk > -INFINITY ? si : -1;
        const float wk = warp_max(sk);
        if (lane == 0 && wk > -INFINITY) atomicMax(&bs->race_k0, key_order(wk));
        __syncwarp();
      }
      // the bound: the best exact key any warp has published (each an entry of this row, so never
      // above the winner's key); a warp that reads it before the others publish gates more loosely
      const float K0 = fmaxf(warp_max(bk),
                             key_from_order(*reinterpret_cast<volatile uint32_t*>(&bs->race_k0)));
      race_stage_main<E>(rs, vt, vd, nvec, m.len, m.e0, m.trow, m.drow, tid, K0, bk, bi);
      const float wk = warp_max(bk);
      if (lane == 0 && wk > K0) atomicMax(&bs->race_k0, key_order(wk));
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (!m.last) continue;

    // segment complete: each warp leaves its result; the last warp to do so merges
    const int buf = m.seg % kRedBufs;
    if (m.kind == kSegStats) {
      warp_ms2(mt, st);
      warp_ms2(md, sd);
    } else if (m.kind == kSegResid) {
      st = warp_sum(acc.x + acc.y);
    } else if (m.kind == kSegRace) {
      warp_race(bk, bi);
      mt = bk;
      st = __int_as_float(bi);
    }
    int32_t last = 0;
    if (lane == 0) {
      bs->dep[buf][warp][0] = mt;
      bs->dep[buf][warp][1] = st;
      bs->dep[buf][warp][2] = md;
      bs->dep[buf][warp][3] = sd;
      __threadfence_block();
      last = atomicAdd(&bs->count[buf], 1) == kConsumerWarps - 1;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      __threadfence_block();
      if (m.kind == kSegStats) {
        float a = kM2Empty, b = 0.f, c = kM2Empty, d = 0.f;
        if (lane < kConsumerWarps) {
          a = bs->dep[buf][lane][0];
          b = bs->dep[buf][lane][1];
          c = bs->dep[buf][lane][2];
          d = bs->dep[buf][lane][3];
        }
        warp_ms2(a, b);
        warp_ms2(c, d);
        if (lane == 0) {
          const int32_t j = m.row;
          const float4 nm = make_float4(a, b, c, d);
          bs->norm[j] = nm;
          publish_seq(&bs->norm_seq[j], m.seq);  // the residual pass over pair j may start
          // ratio p_j(x_j) / q_j(x_j) and the running ratio rho_j = min(1, rho_{j-1} ratio)
          const int64_t drow = p.draft_row0[m.r] + (j - 1);
          const int32_t x = p.draft_tokens[drow];
          float tx = 0.f, dx = 0.f;
          if (x >= 0 && int64_t(x) < p.V) {
            tx = Elem<E>::load(m.trow, x);
            dx = Elem<E>::load(m.drow, x);
          }
          bool bad = false;
          const float ratio = row_ratio(nm, x, p.V, tx, dx, bad);
          if (bad) bs->bad = 1;
          float rho_prev = 1.f;  // on an expired wait the status word already says so
          if (j > 1) rho_prev = wait_seq(&bs->rho_seq[j - 1], m.seq, p.status) ? bs->rho[j - 1] : 0.f;
          const float rho = rho_prev > 0.f ? fminf(1.f, rho_prev * ratio) : 0.f;
          const uint64_t req = p.request_ids ? p.request_ids[m.r] : uint64_t(m.r);
          const float eta =
              uniform_of(stream_block(make_stream(p.seed, req, j, kTagAccept), 0).x);
          const int32_t g = clamp_gamma(p.draft_len[m.r], p.gmax);
          bs->rho[j] = rho;
          bs->eta[j] = eta;
          bs->cand[j] = j < g && eta <= rho;
          publish_seq(&bs->rho_seq[j], m.seq);
        }
      } else if (m.kind == kSegResid) {
        float a = lane < kConsumerWarps ? bs->dep[buf][lane][1] : 0.f;
        a = warp_sum(a);
        if (lane == 0) bs->R[m.row - 1] = a * A;
      } else if (m.kind == kSegRace) {
        float k = -INFINITY;
        int32_t i = -1;
        if (lane < kConsumerWarps) {
          k = bs->dep[buf][lane][0];
          i = __float_as_int(bs->dep[buf][lane][1]);
        }
        warp_race(k, i);
        block_finish<E>(p, m, rs, bs->desc, i);
      } else {
        block_decide<E>(p, m.r, m.seq, bs);
      }
      __syncwarp();
      if (lane == 0) bs->count[buf] = 0;
    }
    mt = kM2Empty;
    st = 0.f;
    md = kM2Empty;
    sd = 0.f;
    acc = make_float2(0.f, 0.f);
    bk = -INFINITY;
    bi = -1;
  }
}

template <typename E>
__global__ void __launch_bounds__(kStreamThreads, 1) block_kernel(BlockParams p) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kRing], empty[kRing];
  __shared__ BlockMeta meta[kRing];
  __shared__ BlockState bs;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int k = 0; k < kRing; ++k) {
      mbar_init(&full[k], 1);
      mbar_init(&empty[k], kConsumerWarps);
    }
    for (int k = 0; k < kRedBufs; ++k) bs.count[k] = 0;
    for (int k = 0; k < kBlockRows; ++k) {
      bs.norm_seq[k] = 0u;
      bs.rho_seq[k] = 0u;
    }
    bs.bad = 0;
    bs.desc_seq = 0u;
    bs.race_k0 = 0u;
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == kConsumerWarps) {
    if ((threadIdx.x & 31) == 0) block_producer<E>(p, ring, full, empty, meta, &bs);
  } else {
    block_consumer<E>(p, ring, full, empty, meta, &bs);
  }
}

// ---------------------------------------------------------------------------------------------
// sample: CL CTAs per drafted row -- the drafted token raced from q (DRAFT tag)
// ---------------------------------------------------------------------------------------------
struct SampleParams {
  const uint8_t* draft;
  int64_t V, ld;
  const int64_t* draft_row0;
  const int32_t* draft_len;
  int32_t B, gmax, CL;      // requests, largest drafted length, CTAs (row shares) per row
  uint64_t seed;
  const uint64_t* request_ids;
  int32_t* sampled_tokens;  // indexed like the draft rows
  RaceSlot* slots;          // one per (request, position), zeroed before the launch
  int32_t* status;
  int32_t stage_share;      // the launch provides dynamic shared memory for the row share
};

template <typename E>
__global__ void __launch_bounds__(kThreads, kRaceCtasPerSm) sample_kernel(SampleParams p) {
  extern __shared__ __align__(128) uint8_t share_sm[];  // this CTA's share of the row (staged)
  __shared__ uint64_t share_bar;
  __shared__ float red_k[kWarps];
  __shared__ int32_t red_i[kWarps];
  __shared__ int32_t s_last;
  __shared__ int32_t s_winner;
  __shared__ float s_k0;
  const int tid = threadIdx.x;
  const int32_t job = blockIdx.x / p.CL;
  const int32_t part = blockIdx.x - job * p.CL;  // this CTA's share of the job's row
  const int32_t r = job / p.gmax;
  const int32_t pos = job - r * p.gmax + 1;
  const int32_t g = p.draft_len[r];
  if (g < 0 || g > p.gmax) {
    if (tid == 0 && part == 0 && pos == 1) report(p.status, SV_ERR_BAD_INPUT);
    return;
  }
  if (pos > g) return;
  RaceSpec rs;
  rs.resid = false;
  rs.gap = 0.f;
  const int64_t sample_row = p.draft_row0[r] + (pos - 1);
  const uint8_t* trow = row_ptr<E>(p.draft, sample_row, p.ld);
  const uint64_t req = p.request_ids ? p.request_ids[r] : uint64_t(r);
  rs.st = make_stream(p.seed, req, pos, kTagDraft);

  // this CTA's share of the row: a contiguous range, a whole number of 16-byte vectors long
  constexpr int32_t kPer = Elem<E>::kPerVec;
  const int64_t share = (p.V + int64_t(p.CL) * kPer - 1) / (int64_t(p.CL) * kPer) * kPer;
  const int64_t lo = min(p.V, int64_t(part) * share);
  const int64_t hi = min(p.V, lo + share);

  // stage the share's whole 16-byte vectors in shared memory with one bulk copy (shares too
  // large for it are read from global memory); a ragged tail is read from global memory
  const uint32_t vec_bytes = static_cast<uint32_t>(((hi - lo) * esize<E>()) & ~int64_t(15));
  const bool staged = p.stage_share && vec_bytes > 0;
  if (tid == 0 && staged) {
    mbar_init(&share_bar, 1);
    fence_barrier_init();
    mbar_expect_tx(&share_bar, vec_bytes);
    bulk_g2s(share_sm, trow + lo * esize<E>(), vec_bytes, &share_bar);
  }
  __syncthreads();
  const uint4* gsrc = reinterpret_cast<const uint4*>(trow + lo * esize<E>());

  // seed: the best exact key among the threads' largest-logit entries, raised to the best seed
  // the row's other shares have published so far -- a lower bound on the winning key, against
  // which the main pass gates.  It reads the share from global memory (L2) while the bulk copy
  // stages it for the main pass.
  RaceSlot* slot = p.slots + job;
  float seed = seed_range<E>(rs, gsrc, trow, nullptr, lo, int32_t(hi - lo));
  if (staged) mbar_wait(&share_bar, 0, p.status);
  const uint4* vsrc = staged ? reinterpret_cast<const uint4*>(share_sm) : gsrc;
  seed = block_max(seed, red_k);
  if (tid == 0) {
    const uint32_t prev = atomicMax(&slot->k0, key_order(seed));
    s_k0 = fmaxf(seed, key_from_order(prev));
  }
  __syncthreads();
  const float K0 = s_k0;

  // main pass: only entries whose logit and noise can reach K0 are keyed
  float bk = -INFINITY;
  int32_t bi = -1;
  if (staged) race_range<E>(rs, vsrc, trow, nullptr, lo, int32_t(hi - lo), K0, bk, bi);
  else race_range<E, kBatchGlobal>(rs, vsrc, trow, nullptr, lo, int32_t(hi - lo), K0, bk, bi);
  block_race(bk, bi, red_k, red_i);

  // combine the shares: a 64-bit max over (order-preserving key bits, ~index), so equal keys go
  // to the lower index; the last share to arrive writes the token
  if (tid == 0) {
    if (bi >= 0) atomicMax(&slot->best, race_pack(bk, bi));
    // release: this share's maximum before its count; acquire (last share): every share's
    s_last = atom_add_acq_rel(&slot->count, 1u) == uint32_t(p.CL - 1);
  }
  __syncthreads();
  if (!s_last) return;
  if (tid == 0) {
    const unsigned long long best = atomicAdd(&slot->best, 0ull);
    s_winner = best ? race_unpack_index(best) : -1;
    if (s_winner < 0) report(p.status, SV_ERR_BAD_INPUT);  // the row carries no probability
    p.sampled_tokens[sample_row] = s_winner;
  }
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
// CTAs per sampled row for rows of S 16 KB slices: each owns one contiguous share of the row.
// Shares per row: as many as one wave of resident sampler CTAs holds (up to kRaceSplitFew), so
// that every row's shares run at once and no CTA pays the seed and combine latencies twice; at
// least one share per row (then several waves).
static int32_t race_split(int32_t S, int64_t jobs) {
  int32_t cl = kRaceSplitMax;
  const int sms = device_sm_count();
  if (sms > 0 && jobs > 0) {
    const int64_t slots = int64_t(sms) * kRaceCtasPerSm;
    cl = int32_t(std::max<int64_t>(1, std::min<int64_t>(kRaceSplitFew, slots / jobs)));
  }
  return std::max(1, std::min(cl, S));
}

// One CTA per request while the requests fit on the SMs (one CTA per SM), else a persistent grid.
template <typename E>
static sv_status launch_block(const BlockParams& bp, cudaStream_t stream) {
  const void* kfn = reinterpret_cast<const void*>(&block_kernel<E>);
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kStreamSmem)) !=
      cudaSuccess)
    return SV_ERR_CUDA;
  const int sms = device_sm_count();
  if (sms <= 0) return SV_ERR_CUDA;
  const unsigned grid = unsigned(std::min<int64_t>(bp.B, sms));
  block_kernel<E><<<grid, kStreamThreads, kStreamSmem, stream>>>(bp);
  return SV_OK;
}

template <typename E>
static sv_status run_block(const CommonArgs& a, const int64_t* target_row0,
                           const int64_t* draft_row0, const int32_t* draft_len,
                           const int32_t* draft_tokens, uint64_t seed,
                           const uint64_t* request_ids, int32_t* accepted_len,
                           int32_t* out_tokens, int64_t out_ld, int32_t* correction_token,
                           float* rho_out, float* h_out, int32_t* status, cudaStream_t stream) {
  const int32_t C = chunks_of(a.V, esize<E>());
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  BlockParams bp;
  bp.target = static_cast<const uint8_t*>(a.target);
  bp.draft = static_cast<const uint8_t*>(a.draft);
  bp.V = a.V;
  bp.ld = a.ld;
  bp.target_row0 = target_row0;
  bp.draft_row0 = draft_row0;
  bp.draft_len = draft_len;
  bp.draft_tokens = draft_tokens;
  bp.B = a.B;
  bp.gmax = a.gmax;
  bp.seed = seed;
  bp.request_ids = request_ids;
  bp.rho_out = rho_out;
  bp.h_out = h_out;
  bp.accepted_len = accepted_len;
  bp.out_tokens = out_tokens;
  bp.out_ld = out_ld;
  bp.correction_token = correction_token;
  bp.ws = verify_layout(a.ws, a.B, a.gmax, C);
  bp.status = status;
  profile_mark(0, stream);
  const sv_status st = launch_block<E>(bp, stream);
  if (st != SV_OK) return st;
  profile_mark(1, stream);
  profile_mark(2, stream);
  profile_mark(3, stream);  // the block kernel draws the correction itself
  return launch_status(cudaGetLastError());
}

template <typename E>
static sv_status run_sample(const CommonArgs& a, const int64_t* draft_row0,
                            const int32_t* draft_len, uint64_t seed, const uint64_t* request_ids,
                            int32_t* draft_tokens, int32_t* status, cudaStream_t stream) {
  const int32_t S = slices_of(a.V, esize<E>());
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  SampleParams sp = {};
  sp.draft = static_cast<const uint8_t*>(a.draft);
  sp.V = a.V;
  sp.ld = a.ld;
  sp.draft_row0 = draft_row0;
  sp.draft_len = draft_len;
  sp.B = a.B;
  sp.gmax = a.gmax;
  sp.seed = seed;
  sp.request_ids = request_ids;
  sp.sampled_tokens = draft_tokens;
  sp.status = status;
  sp.slots = verify_layout(a.ws, a.B, a.gmax, chunks_of(a.V, esize<E>())).slots;
  const int64_t jobs = int64_t(a.B) * a.gmax;
  if (jobs == 0) return SV_OK;
  if (cudaMemsetAsync(sp.slots, 0, sizeof(RaceSlot) * size_t(jobs), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  sp.CL = race_split(S, jobs);
  // the kernel's share: ceil(V / (CL * kPer)) whole vectors
  constexpr int64_t kPer = Elem<E>::kPerVec;
  const int64_t share_bytes = (sp.V + sp.CL * kPer - 1) / (sp.CL * kPer) * 16;
  sp.stage_share = share_bytes <= int64_t(kRaceShareMax);
  const size_t smem = sp.stage_share ? size_t(share_bytes) : 0;
  if (cudaFuncSetAttribute(sample_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kRaceShareMax)) != cudaSuccess)
    return SV_ERR_CUDA;
  sample_kernel<E><<<unsigned(jobs * sp.CL), kThreads, smem, stream>>>(sp);
  return launch_status(cudaGetLastError());
}

}  // namespace sv

using namespace sv;

extern "C" size_t spec_verify_workspace_bytes(int32_t B, int32_t max_draft_len, int64_t V,
                                              sv_dtype dtype) {
  if (B < 0 || max_draft_len < 0 || max_draft_len > SV_MAX_DRAFT_LEN || V <= 0) return 0;
  if (dtype != SV_F32 && dtype != SV_BF16) return 0;
  return verify_ws_bytes(B, max_draft_len, V, elem_bytes(dtype));
}

extern "C" sv_status spec_verify_block(const void* target_logits, const void* draft_logits,
                                       sv_dtype dtype, int64_t V, int64_t ld,
                                       const int64_t* target_row0, const int64_t* draft_row0,
                                       const int32_t* draft_len, int32_t max_draft_len,
                                       const int32_t* draft_tokens, int32_t B, uint64_t seed,
                                       const uint64_t* request_ids, int32_t* accepted_len,
                                       int32_t* out_tokens, int64_t out_ld,
                                       int32_t* correction_token, float* running_ratio,
                                       float* h_threshold, int32_t* status, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  CommonArgs a{target_logits, draft_logits, dtype, V, ld, B, max_draft_len, workspace,
               workspace_bytes};
  sv_status st = check_common(a, true);
  if (st != SV_OK) return st;
  if (B == 0) return SV_OK;
  if (!target_row0 || !draft_len || !accepted_len || !out_tokens) return SV_ERR_INVALID;
  if (max_draft_len > 0 && (!draft_row0 || !draft_tokens)) return SV_ERR_INVALID;
  if (out_ld < int64_t(max_draft_len) + 1) return SV_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SV_BF16)
    return run_block<bf16_tag>(a, target_row0, draft_row0, draft_len, draft_tokens, seed,
                               request_ids, accepted_len, out_tokens, out_ld, correction_token,
                               running_ratio, h_threshold, status, s);
  return run_block<float>(a, target_row0, draft_row0, draft_len, draft_tokens, seed, request_ids,
                          accepted_len, out_tokens, out_ld, correction_token, running_ratio,
                          h_threshold, status, s);
}

extern "C" sv_status spec_sample_draft(const void* draft_logits, sv_dtype dtype, int64_t V,
                                       int64_t ld, const int64_t* draft_row0,
                                       const int32_t* draft_len, int32_t max_draft_len, int32_t B,
                                       uint64_t seed, const uint64_t* request_ids,
                                       int32_t* draft_tokens, int32_t* status, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  CommonArgs a{nullptr, draft_logits, dtype, V, ld, B, max_draft_len, workspace, workspace_bytes};
  sv_status st = check_common(a, false);
  if (st != SV_OK) return st;
  if (B == 0 || max_draft_len == 0) return SV_OK;
  if (!draft_row0 || !draft_len || !draft_tokens) return SV_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SV_BF16)
    return run_sample<bf16_tag>(a, draft_row0, draft_len, seed, request_ids, draft_tokens, status,
                                s);
  return run_sample<float>(a, draft_row0, draft_len, seed, request_ids, draft_tokens, status, s);
}

// ---------------------------------------------------------------------------------------------
// spec_verify_token_noalloc: token-level verification with scratch memory owned by the library.
//
// Some callers cannot allocate device memory at all: a plugin that is handed only its input and
// output buffers by a host engine that owns every device allocation, or a serving loop that must
// not call cudaMalloc because a device allocation can implicitly synchronise the device.  For
// them the scratch memory of the verify kernels lives in the file-scope array below, which every
// GPU that loads this library holds until the process exits.
// ---------------------------------------------------------------------------------------------
namespace sv {

constexpr size_t kNoAllocScratchBytes = SV_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Unique id of the CUDA context current on the calling thread, or 0 if there is none yet or the
// driver cannot be asked.  The two driver calls are reached through the runtime's entry-point
// query, so the library needs no link against the driver library.  Context ids are never reused
// within a process, unlike context handles.
static unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_noalloc_scratch in the current context.  In host code the array's name is
// a host-side stand-in, not a device address, so the address is looked up with the context
// current and cached by context id: a device reset or another context (a driver-API context of
// an engine, say) gets a lookup of its own instead of a stale address.  Without a context id
// (no driver entry points) every call looks the address up again.
static sv_status noalloc_scratch_address(void** out) {
  constexpr int kSlots = 64;
  static std::mutex mu;
  static unsigned long long ids[kSlots] = {};
  static void* addr[kSlots] = {};
  static int next = 0;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = current_context_id();
  if (id != 0)
    for (int k = 0; k < kSlots; ++k)
      if (ids[k] == id) {
        *out = addr[k];
        return SV_OK;
      }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
    return SV_ERR_CUDA;
  id = current_context_id();  // the lookup made the runtime's context current if none was
  if (id != 0) {
    ids[next] = id;
    addr[next] = p;
    next = (next + 1) % kSlots;
  }
  *out = p;
  return SV_OK;
}

}  // namespace sv

extern "C" sv_status spec_verify_token_noalloc(
    const void* target_logits, const void* draft_logits, sv_dtype dtype, int64_t V, int64_t ld,
    const int64_t* target_row0, const int64_t* draft_row0, const int32_t* draft_len,
    int32_t max_draft_len, const int32_t* draft_tokens, int32_t B, uint64_t seed,
    const uint64_t* request_ids, int32_t* accepted_len, int32_t* out_tokens, int64_t out_ld,
    int32_t* correction_token, float* accept_ratio, int32_t* status, void* stream) {
  const size_t need = spec_verify_workspace_bytes(B, max_draft_len, V, dtype);
  if (need == 0) return SV_ERR_INVALID;
  if (need > sv::kNoAllocScratchBytes) return SV_ERR_UNSUPPORTED;  // batch too large for it
  void* scratch = nullptr;
  const sv_status st = sv::noalloc_scratch_address(&scratch);
  if (st != SV_OK) return st;
  // The verify kernels never read scratch they have not written earlier in the same call; the
  // only counters (race tickets) are cleared by the call's first kernel before the race kernel
  // runs.
  return spec_verify_token(target_logits, draft_logits, dtype, V, ld, target_row0, draft_row0,
                           draft_len, max_draft_len, draft_tokens, B, seed, request_ids,
                           accepted_len, out_tokens, out_ld, correction_token, accept_ratio,
                           status, scratch, sv::kNoAllocScratchBytes, stream);
}
