// verify_kernels.cuh -- the kernels token-level verification (token.cu) and block verification
// (block.cu) share:
//   stream  persistent, warp-specialised CTAs (one per SM): a producer warp walks this CTA's
//           items -- a chunk of one (request, position) row pair -- and feeds a three-deep ring of
//           32 KB shared-memory stages with bulk copies; sixteen consumer warps fold every staged
//           element into log2-domain softmax statistics; the last warp to finish an item merges
//           the warps' results into one partial per (row pair, chunk), so no consumer ever waits
//           on another.  Positions are walked highest first, so the early positions -- where the
//           first rejection and hence the correction race most often fall -- are read last and
//           are still in L2 when the later kernels read them again.
//   race    up to 16 CTAs per request.  Each first decides its request (token level: it folds the
//           partials of the request's rows into the row normalisers and the ratios p(x)/q(x),
//           draws the uniforms and finds the first rejection; block level: it reads the running
//           ratios, uniforms and residual masses the block kernels left and finds the longest
//           passing prefix).  It then stages its contiguous share of the correction (or bonus) row
//           in shared memory with one bulk copy and runs the exponential race of the share, pruned
//           against the best seed key any share has published; the shares combine through one
//           64-bit atomic max per request and the last share to finish writes the outputs.  It is
//           launched as a programmatic dependent of the kernel before it, so its launch overlaps
//           that kernel's tail.
//   finish  the partial race winners of a request folded into its outputs (vocabulary shards,
//           and the tiles of the race over recomputed logits in lmhead.cu).
// Everything here has internal linkage: each file that includes it compiles its own copy.
#pragma once

#include "verify_common.cuh"

namespace sv {
namespace {

constexpr int kRaceSplitMax = 8;                 // CTAs (row shares) per race job, many jobs
constexpr int kRaceSplitFew = 16;                // the same when one wave holds every share
constexpr int kRaceCtasPerSm = 4;                // resident race CTAs per SM (launch bounds)
constexpr uint32_t kRaceShareMax = 64 * 1024;    // largest row share staged in shared memory

// ---------------------------------------------------------------------------------------------
// stream: producer / consumer ring over (row pair, chunk) items
// ---------------------------------------------------------------------------------------------
struct StreamParams {
  const uint8_t* target;
  const uint8_t* draft;
  int64_t V, ld;
  const int64_t* target_row0;
  const int64_t* draft_row0;
  const int32_t* draft_len;
  int32_t B, gmax, C;
  VerifyWs ws;
  int32_t* status;
  int32_t clear_status;  // this launch resets the call's status word (see stream_kernel)
  int32_t* zero_words;   // nullable: counters of the kernels that follow, zeroed by block 0
  int32_t n_zero;
  int32_t* claim;        // nullable: the tail's item counter (dynamic claims), zeroed by block 0
  unsigned long long* claim_ready;  // block 0 stores call_id here once the counter is zeroed
  unsigned long long call_id;       // unique to this launch
};

// The items of the last kDynRounds rounds are claimed one at a time from a counter instead of
// dealt out round-robin, so that the SMs that stream faster take more of the tail.
constexpr int kDynRounds = 2;

struct StageMeta {
  int32_t unit;   // r * gmax + (i - 1); -1 marks the end of the stream
  int32_t chunk;
  int32_t last;   // this stage closes its item
  int32_t len;    // elements of the slice
  int32_t bulk;   // elements brought by the bulk copies (the rest is read from global)
  int32_t item;   // running item number of this CTA (selects the merge buffer)
  int64_t e0;     // first vocabulary index of the slice
  const uint8_t* trow;
  const uint8_t* drow;
};

template <typename E>
__device__ void stream_producer(const StreamParams& p, uint8_t* ring, uint64_t* full,
                                uint64_t* empty, StageMeta* meta) {
  constexpr int32_t kSE = kRowBytes / esize<E>();
  const int64_t per_pos = int64_t(p.B) * p.C;
  const int64_t n_items = int64_t(p.gmax) * per_pos;
  uint32_t n = 0;      // stages issued so far
  int32_t issued = 0;  // items issued so far
  // items [0, n_static) round-robin, the rest claimed; the first claim waits (bounded) until block
  // 0 has zeroed the counter for this launch
  const int64_t n_dyn = p.claim ? min(n_items, int64_t(gridDim.x) * kDynRounds) : 0;
  const int64_t n_static = n_items - n_dyn;
  bool ready = false;
  auto next_item = [&](int64_t after) -> int64_t {  // after < 0: this CTA's first item
    if (after < n_static) {
      const int64_t s = after < 0 ? int64_t(blockIdx.x) : after + gridDim.x;
      if (s < n_static) return s;
    }
    if (n_dyn == 0) return n_items;
    if (!ready) {
      const uint64_t t0 = global_ns();
      while (ld_acquire_u64(p.claim_ready) != p.call_id) {
        if (global_ns() - t0 > kWaitLimitNs) {
          report(p.status, SV_ERR_TIMEOUT);
          return n_items;
        }
        __nanosleep(64);
      }
      ready = true;
    }
    return n_static + atomicAdd(p.claim, 1);
  };
  for (int64_t item = next_item(-1); item < n_items;) {
    const int64_t cur = item;
    const int32_t i = p.gmax - static_cast<int32_t>(cur / per_pos);  // highest position first
    const int64_t rem = cur % per_pos;
    const int32_t r = static_cast<int32_t>(rem / p.C);
    const int32_t c = static_cast<int32_t>(rem % p.C);
    if (i > clamp_gamma(p.draft_len[r], p.gmax)) {  // request r drafted fewer tokens
      item = next_item(cur);
      continue;
    }
    const int32_t unit = r * p.gmax + (i - 1);
    const uint8_t* trow = row_ptr<E>(p.target, p.target_row0[r] + (i - 1), p.ld);
    const uint8_t* drow = row_ptr<E>(p.draft, p.draft_row0[r] + (i - 1), p.ld);
    const int64_t ie0 = int64_t(c) * kSE * kStagesPerItem;
    const int64_t iend = p.V - ie0 < int64_t(kSE) * kStagesPerItem ? p.V
                                                                    : ie0 + int64_t(kSE) * kStagesPerItem;
    for (int64_t e0 = ie0; e0 < iend; e0 += kSE) {
      const uint32_t stage = n % kRing;
      if (n >= kRing && !mbar_wait(&empty[stage], ((n / kRing) - 1) & 1, p.status)) return;
      StageMeta m;
      m.unit = unit;
      m.chunk = c;
      m.last = e0 + kSE >= iend;
      m.item = issued;
      m.e0 = e0;
      m.len = static_cast<int32_t>(iend - e0 < kSE ? iend - e0 : kSE);
      const uint32_t bulk_bytes = (uint32_t(m.len) * esize<E>()) & ~15u;
      m.bulk = static_cast<int32_t>(bulk_bytes / esize<E>());
      m.trow = trow;
      m.drow = drow;
      meta[stage] = m;
      uint8_t* dst = ring + size_t(stage) * 2 * kRowBytes;
      fence_proxy_async();
      mbar_expect_tx(&full[stage], 2 * bulk_bytes);
      if (bulk_bytes) {
        bulk_g2s(dst, trow + m.e0 * esize<E>(), bulk_bytes, &full[stage]);
        bulk_g2s(dst + kRowBytes, drow + m.e0 * esize<E>(), bulk_bytes, &full[stage]);
      }
      ++n;
    }
    ++issued;
    item = next_item(cur);  // claimed after this item's copies are under way
  }
  // end-of-stream marker
  const uint32_t stage = n % kRing;
  if (n >= kRing && !mbar_wait(&empty[stage], ((n / kRing) - 1) & 1, p.status)) return;
  meta[stage].unit = -1;
  mbar_arrive(&full[stage]);
}

struct MergeSlots {
  float v[kRedBufs][kConsumerWarps][4];
  int32_t count[kRedBufs];
};

template <typename E>
__device__ void stream_consumer(const StreamParams& p, const uint8_t* ring, uint64_t* full,
                                uint64_t* empty, const StageMeta* meta, MergeSlots* ms) {
  constexpr int kPer = Elem<E>::kPerVec;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float mt = kM2Empty, st = 0.f, md = kM2Empty, sd = 0.f;
  for (uint32_t n = 0;; ++n) {
    const uint32_t stage = n % kRing;
    if (!mbar_wait(&full[stage], (n / kRing) & 1, p.status)) return;
    const StageMeta m = meta[stage];
    if (m.unit < 0) return;
    const uint4* vt = reinterpret_cast<const uint4*>(ring + size_t(stage) * 2 * kRowBytes);
    const uint4* vd = vt + kRowBytes / 16;
    const int nvec = m.bulk / kPer;
    if (m.bulk == int32_t(kRowBytes / esize<E>())) {
      // full stage: every consumer thread holds kFull vectors of each row
      constexpr int kFull = int(kRowBytes / 16) / kConsumers;
      static_assert(kFull * kConsumers * 16 == int(kRowBytes), "stage not a whole multiple");
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
#pragma unroll 2
      for (int v = tid; v < nvec; v += kConsumers) {
        const uint4 a = vt[v], b = vd[v];
        if constexpr (kPer == 8) {
          ms2_vec_bf16(mt, st, a);
          ms2_vec_bf16(md, sd, b);
        } else {
          ms2_vec_f32(mt, st, a);
          ms2_vec_f32(md, sd, b);
        }
      }
      for (int e = m.bulk + tid; e < m.len; e += kConsumers) {
        ms2_one(mt, st, Elem<E>::load(m.trow, m.e0 + e));
        ms2_one(md, sd, Elem<E>::load(m.drow, m.e0 + e));
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    if (!m.last) continue;
    // item complete: each warp leaves its result; the last warp to do so merges and writes
    const int buf = m.item % kRedBufs;
    warp_ms2(mt, st);
    warp_ms2(md, sd);
    int32_t last = 0;
    if (lane == 0) {
      ms->v[buf][warp][0] = mt;
      ms->v[buf][warp][1] = st;
      ms->v[buf][warp][2] = md;
      ms->v[buf][warp][3] = sd;
      __threadfence_block();
      last = atomicAdd(&ms->count[buf], 1) == kConsumerWarps - 1;
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (last) {
      __threadfence_block();
      const size_t slot = size_t(m.unit) * p.C + m.chunk;
      float a = kM2Empty, b = 0.f, c = kM2Empty, d = 0.f;
      if (lane < kConsumerWarps) {
        a = ms->v[buf][lane][0];
        b = ms->v[buf][lane][1];
        c = ms->v[buf][lane][2];
        d = ms->v[buf][lane][3];
      }
      warp_ms2(a, b);
      warp_ms2(c, d);
      if (lane == 0) __stcg(&p.ws.partials[slot], make_float4(a, b, c, d));
      if (lane == 0) ms->count[buf] = 0;
    }
    mt = kM2Empty;
    st = 0.f;
    md = kM2Empty;
    sd = 0.f;
  }
}

template <typename E>
__global__ void __launch_bounds__(kStreamThreads, 1) stream_kernel(StreamParams p) {
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ uint64_t full[kRing], empty[kRing];
  __shared__ StageMeta meta[kRing];
  __shared__ MergeSlots ms;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int k = 0; k < kRing; ++k) {
      mbar_init(&full[k], 1);
      mbar_init(&empty[k], kConsumerWarps);
    }
    for (int k = 0; k < kRedBufs; ++k) ms.count[k] = 0;
    fence_barrier_init();
  }
  // the race kernel that follows may launch now (it waits for this grid's results itself)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == 0) {  // the race's per-request slots start empty
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) p.ws.slots[i] = RaceSlot{0ull, 0u, 0u};
    // The call's status word starts at SV_OK.  This kernel reports nothing but an expired wait,
    // a second after its start, and the race kernel that follows waits for this grid before it
    // reports anything, so clearing the word here orders it before every report of the call.
    if (threadIdx.x == 0 && p.clear_status && p.status) *p.status = SV_OK;
    if (threadIdx.x < p.n_zero) p.zero_words[threadIdx.x] = 0;
    if (threadIdx.x == 0 && p.claim) {  // the counter, then (release) this launch's id
      *p.claim = 0;
      st_release_u64(p.claim_ready, p.call_id);
    }
  }
  __syncthreads();
  if (warp == kConsumerWarps) {
    if ((threadIdx.x & 31) == 0) stream_producer<E>(p, ring, full, empty, meta);
  } else {
    stream_consumer<E>(p, ring, full, empty, meta, &ms);
  }
}

// ---------------------------------------------------------------------------------------------
// decide (token-level): per-request combination of the row statistics and the acceptance test
// ---------------------------------------------------------------------------------------------
struct DecideParams {
  const uint8_t* target;
  const uint8_t* draft;
  int64_t V, ld;
  const int64_t* target_row0;
  const int64_t* draft_row0;
  const int32_t* draft_len;
  const int32_t* draft_tokens;
  int32_t B, gmax, C;
  uint64_t seed;
  const uint64_t* request_ids;
  float* ratio_out;  // min(1, p/q) per drafted row (nullable)
  VerifyWs ws;
  int32_t* status;
  const float2* tok;  // nullable: the drafted tokens' (target, draft) logits per row pair, for a
                      // vocabulary shard that may not hold them (V is then the whole vocabulary)
};

// Drafted token x of position i of request r and its target and draft logits (lane 0 of a warp).
template <typename E>
__device__ __forceinline__ void fetch_drafted(const DecideParams& p, int32_t r, int32_t i,
                                              int32_t& x, float& tx, float& dx) {
  const int64_t drow = p.draft_row0[r] + (i - 1);
  x = p.draft_tokens[drow];
  tx = dx = 0.f;
  if (x >= 0 && int64_t(x) < p.V) {
    if (p.tok) {
      const float2 v = p.tok[size_t(r) * p.gmax + (i - 1)];
      tx = v.x;
      dx = v.y;
    } else {
      tx = Elem<E>::load(row_ptr<E>(p.target, p.target_row0[r] + (i - 1), p.ld), x);
      dx = Elem<E>::load(row_ptr<E>(p.draft, drow, p.ld), x);
    }
  }
}

// The decision of request r by one CTA.  `writer`: this CTA writes the call's ratio outputs and
// the status word; `s_desc` receives the race descriptor and `s_tok` the drafted tokens (position
// i at i - 1) in shared memory.  Every thread of the CTA must call it.  `dep_wait`: the caller is a programmatic dependent that has not yet waited
// for the previous kernel (whose row partials this reads); the call's own inputs -- the ACCEPT
// uniforms, each warp's first drafted token and its two logits -- are fetched before the wait.
template <typename E>
__device__ __noinline__ void decide_body(const DecideParams& p, int32_t r, bool writer,
                                         RaceDesc* s_desc, int32_t* s_tok, bool dep_wait) {
  __shared__ float s_ratio[SV_MAX_DRAFT_LEN + 1];
  __shared__ float s_u[SV_MAX_DRAFT_LEN + 1];
  __shared__ float4 s_norm[SV_MAX_DRAFT_LEN + 1];
  __shared__ int32_t s_bad;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t graw = p.draft_len[r];
  const int32_t g = clamp_gamma(graw, p.gmax);
  const uint64_t req = p.request_ids ? p.request_ids[r] : uint64_t(r);
  // uniforms u_i (ACCEPT tag, position i), one thread each
  for (int i = tid + 1; i <= g; i += kThreads)
    s_u[i] = uniform_of(stream_block(make_stream(p.seed, req, i, kTagAccept), 0).x);
  int32_t x0 = -1;
  float tx0 = 0.f, dx0 = 0.f;
  if (lane == 0 && warp + 1 <= g) fetch_drafted<E>(p, r, warp + 1, x0, tx0, dx0);
  if (dep_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0) s_bad = (graw != g) ? SV_ERR_BAD_INPUT : 0;
  __syncthreads();

  // row normalisers and the drafted token's ratio, one warp per row
  for (int i = warp + 1; i <= g; i += kWarps) {
    const int32_t unit = r * p.gmax + (i - 1);
    // lane 0 has the drafted token and its two logits (fetched now past the first row)
    int32_t x = x0;
    float tx = tx0, dx = dx0;
    if (lane == 0 && i != warp + 1) fetch_drafted<E>(p, r, i, x, tx, dx);
    float mt = kM2Empty, st = 0.f, md = kM2Empty, sd = 0.f;
    for (int c = lane; c < p.C; c += 32) {
      const float4 q = __ldcg(&p.ws.partials[size_t(unit) * p.C + c]);
      ms2_merge(mt, st, q.x, q.y);
      ms2_merge(md, sd, q.z, q.w);
    }
    warp_ms2(mt, st);
    warp_ms2(md, sd);
    if (lane == 0) {
      bool bad = false;
      const float ratio = row_ratio(make_float4(mt, st, md, sd), x, p.V, tx, dx, bad);
      if (bad) s_bad = SV_ERR_BAD_INPUT;
      s_ratio[i] = ratio;
      s_norm[i] = make_float4(mt, st, md, sd);
      s_tok[i - 1] = x;
    }
  }
  __syncthreads();

  if (tid == 0) {
    if (writer && s_bad) report(p.status, s_bad);
    int32_t tau = g;  // walk left to right, stop at the first rejection
    for (int i = 1; i <= g; ++i)
      if (!(s_u[i] < s_ratio[i])) {
        tau = i - 1;
        break;
      }
    RaceDesc d;
    d.tau = tau;
    d.resid = tau < g;
    d.gap = d.resid ? resid_gap(s_norm[tau + 1], 0.f) : 0.f;
    d.pad = 0;
    *s_desc = d;
  }
  if (writer && p.ratio_out)
    for (int i = tid + 1; i <= g; i += kThreads)
      p.ratio_out[p.draft_row0[r] + (i - 1)] = fminf(1.f, s_ratio[i]);
}

// ---------------------------------------------------------------------------------------------
// race: CL CTAs per request -- its decision, then the correction / bonus token
// ---------------------------------------------------------------------------------------------
// h_i = R_i / (R_i + 1 - rho_i) (1 if the denominator is 0), R_i the sum of its residual
// partials in share order -- the one order every reader of them uses.
__device__ __forceinline__ float block_threshold(const float* rpart, int32_t CLr, float rho) {
  float R = 0.f;
  for (int32_t s = 0; s < CLr; ++s) R += __ldcg(rpart + s);
  const float den = R + (1.f - rho);
  return den > 0.f ? R / den : 1.f;
}

// What block verification's prep and residual kernels leave in the workspace for the decision.
struct BlockDecideParams {
  const float4* norm;    // [units] row-pair normalisers (m_t, s_t, m_d, s_d), log2 domain
  const float* rho;      // [units] running ratio rho_i
  const float* eta;      // [units] ACCEPT uniform eta_i
  const int32_t* cand;   // [units] slot of (r, i), -1 if R_i was not computed
  const float* rpart;    // [slots * CLr] residual mass partials, one per (slot, share)
  int32_t CLr;           // residual shares per row
  float* rho_out;        // nullable, per drafted row
  float* h_out;          // nullable, per drafted row
};

struct RaceParams {
  const uint8_t* target;
  const uint8_t* draft;
  int64_t V, ld;
  const int64_t* target_row0;
  const int64_t* draft_row0;
  const int32_t* draft_tokens;
  int32_t B, gmax, S, CL;  // 16 KB slices per row, CTAs (row shares) per request
  uint64_t seed;
  const uint64_t* request_ids;
  int32_t* accepted_len;
  int32_t* out_tokens;
  int64_t out_ld;
  int32_t* correction_token;
  VerifyWs ws;
  int32_t* status;
  int32_t stage_share;      // the launch provides dynamic shared memory for the row share
  int64_t v_off;            // vocabulary index of column 0 (a vocabulary shard; 0 otherwise)
  unsigned long long* winners;  // nullable: a shard's race, [B][2] packed winners, not outputs
  DecideParams dp;          // token-level decision
  BlockDecideParams bd;     // block decision
};

// The block decision of request r by warp 0 of a race CTA, from the running ratios, uniforms and
// residual-mass partials in the workspace: h_i = R_i / (R_i + 1 - rho_i) for the positions whose
// R_i was computed, h_gamma = rho_gamma, h_i below every uniform for the rest (eta_i > rho_i >= h_i
// fails whatever R_i is, and positions below a passing one were not evaluated); tau = the highest
// passing position, or 0.  `writer`: this CTA writes the per-row outputs.
__device__ void block_decide_warp(const RaceParams& p, int32_t r, bool writer, RaceDesc* s_desc,
                                  int32_t* s_tok) {
  const int lane = threadIdx.x & 31;
  const BlockDecideParams& b = p.bd;
  const int32_t g = clamp_gamma(p.dp.draft_len[r], p.gmax);
  const int64_t d0 = g > 0 ? p.draft_row0[r] : 0;
  int32_t tau = 0;
  for (int32_t base = 0; base < g; base += 32) {
    const int32_t i = base + lane + 1;
    bool pass = false;
    if (i <= g) {
      const int32_t unit = r * p.gmax + i - 1;
      const float rho = b.rho[unit];
      float h;
      if (i == g) {
        h = rho;
      } else {
        const int32_t c = b.cand[unit];
        if (c >= 0) {
          h = block_threshold(b.rpart + size_t(c) * b.CLr, b.CLr, rho);
        } else {
          // eta_i > rho_i >= h_i: position i fails whatever R_i is; or a higher position passed
          // already, so position i cannot be the longest passing prefix
          h = -1.f;
        }
      }
      pass = b.eta[unit] <= h;
      if (writer && b.h_out) b.h_out[d0 + i - 1] = h;
      if (writer && b.rho_out) b.rho_out[d0 + i - 1] = rho;
      s_tok[i - 1] = p.draft_tokens[d0 + i - 1];
    }
    const uint32_t m = __ballot_sync(0xffffffffu, pass);
    if (m) tau = base + 32 - __clz(m);  // the highest passing position so far
  }
  if (lane == 0) {
    RaceDesc d;
    d.tau = tau;
    d.resid = tau < g;
    d.gap = 0.f;
    if (d.resid) {
      const float lnw = tau > 0 ? logf(b.rho[r * p.gmax + tau - 1]) : 0.f;
      d.gap = resid_gap(b.norm[r * p.gmax + tau], lnw);
    }
    d.pad = 0;
    *s_desc = d;
  }
}

template <typename E, bool kBlock>
__global__ void __launch_bounds__(kThreads, kRaceCtasPerSm) race_kernel(RaceParams p) {
  extern __shared__ __align__(128) uint8_t share_sm[];  // this CTA's share of the row (staged)
  __shared__ uint64_t share_bar;
  __shared__ float red_k[kWarps];
  __shared__ int32_t red_i[kWarps];
  __shared__ int32_t s_last;
  __shared__ int32_t s_winner;
  __shared__ float s_k0;
  __shared__ RaceDesc s_desc;
  __shared__ int32_t s_tok[SV_MAX_DRAFT_LEN];  // the request's drafted tokens (decided here)
  const int tid = threadIdx.x;
  const int32_t r = blockIdx.x / p.CL;
  const int32_t part = blockIdx.x - r * p.CL;  // this CTA's share of the request's row
  if constexpr (kBlock) {
    // launched as a programmatic dependent of the residual kernel: wait for its results
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x < 32) block_decide_warp(p, r, part == 0, &s_desc, s_tok);
  } else {
    // launched as a programmatic dependent of the stream kernel: the decision waits for its
    // results inside decide_body, after fetching the call's own inputs
    decide_body<E>(p.dp, r, part == 0, &s_desc, s_tok, true);
  }
  __syncthreads();
  const RaceDesc d = s_desc;
  const int32_t tau = d.tau;
  RaceSpec rs;
  rs.resid = d.resid != 0;
  rs.gap = d.gap;
  const uint8_t* trow = row_ptr<E>(p.target, p.target_row0[r] + tau, p.ld);
  const uint8_t* drow = rs.resid ? row_ptr<E>(p.draft, p.draft_row0[r] + tau, p.ld) : nullptr;
  const uint64_t req = p.request_ids ? p.request_ids[r] : uint64_t(r);
  rs.st = make_stream(p.seed, req, uint32_t(tau + 1), rs.resid ? kTagResid : kTagBonus);
  rs.off = p.v_off;

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
  // the request's other shares have published so far -- a lower bound on the winning key,
  // against which the main pass gates.  It reads the share from global memory (L2) while the bulk
  // copy stages it for the main pass.
  RaceSlot* slot = p.ws.slots + r;
  float seed = seed_range<E>(rs, gsrc, trow, drow, lo, int32_t(hi - lo));
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
  if (staged) race_range<E>(rs, vsrc, trow, drow, lo, int32_t(hi - lo), K0, bk, bi);
  else race_range<E, kBatchGlobal>(rs, vsrc, trow, drow, lo, int32_t(hi - lo), K0, bk, bi);
  block_race(bk, bi, red_k, red_i);

  // combine the shares: a 64-bit max over (order-preserving key bits, ~index), so equal keys go
  // to the lower index; the last share to arrive writes the request's outputs
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
  }
  __syncthreads();
  int32_t y = s_winner;
  if (p.winners) {
    // a vocabulary shard: this shard's winner with its global index, and -- if the shard holds no
    // positive residual entry -- the shard's winner of the race over p with the same uniforms,
    // which the request takes if no shard holds one (the residual is then empty everywhere)
    unsigned long long fb_best = 0ull;
    if (y < 0 && rs.resid) {
      RaceSpec fb = rs;
      fb.resid = false;
      float k;
      int32_t yf;
      race_row_global<E>(fb, trow, nullptr, p.V, red_k, red_i, k, yf);
      if (yf >= 0) fb_best = race_pack(k, int32_t(p.v_off + yf));
    }
    if (tid == 0) {
      const unsigned long long best = atomicAdd(&slot->best, 0ull);
      p.winners[2 * size_t(r)] =
          best ? race_pack(key_from_order(uint32_t(best >> 32)), int32_t(p.v_off + y)) : 0ull;
      p.winners[2 * size_t(r) + 1] = fb_best;
      p.accepted_len[r] = tau;
    }
    return;
  }
  if (y < 0 && rs.resid) {
    // residual empty to working precision (p and q agree): draw from p with the same uniforms
    RaceSpec fb = rs;
    fb.resid = false;
    float k;
    race_row_global<E>(fb, trow, nullptr, p.V, red_k, red_i, k, y);
  }
  int32_t* out = p.out_tokens + size_t(r) * p.out_ld;
  for (int64_t q = tid; q < p.out_ld; q += kThreads) {
    int32_t v = -1;
    if (q < tau) v = s_tok[q];
    else if (q == tau) v = y;
    out[q] = v;
  }
  if (tid == 0) {
    if (y < 0) report(p.status, SV_ERR_BAD_INPUT);  // the row carries no probability at all
    p.accepted_len[r] = tau;
    if (p.correction_token) p.correction_token[r] = y;
  }
}

// ---------------------------------------------------------------------------------------------
// host side: launches shared by both verification calls
// ---------------------------------------------------------------------------------------------
// CTAs per race job for rows of S 16 KB slices: each owns one contiguous share of the row.
// Shares per job: as many as one wave of resident race CTAs holds (up to kRaceSplitFew), so that
// every job's shares run at once and no CTA pays the decide, seed and combine latencies twice; at
// least one share per job (then several waves).
static int32_t race_split(int32_t S, int64_t jobs) {
  int32_t cl = kRaceSplitMax;
  const int sms = device_sm_count();
  if (sms > 0 && jobs > 0) {
    const int64_t slots = int64_t(sms) * kRaceCtasPerSm;
    cl = int32_t(std::max<int64_t>(1, std::min<int64_t>(kRaceSplitFew, slots / jobs)));
  }
  return std::max(1, std::min(cl, S));
}

template <typename E>
static sv_status launch_stream(const StreamParams& sp, cudaStream_t stream) {
  const void* kfn = reinterpret_cast<const void*>(&stream_kernel<E>);
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kStreamSmem)) !=
      cudaSuccess)
    return SV_ERR_CUDA;
  const int64_t items = int64_t(sp.gmax) * sp.B * sp.C;
  if (items == 0) return SV_OK;
  const int sms = device_sm_count();
  if (sms <= 0) return SV_ERR_CUDA;
  const unsigned grid = unsigned(std::min<int64_t>(items, sms));
  stream_kernel<E><<<grid, kStreamThreads, kStreamSmem, stream>>>(sp);
  return SV_OK;
}

template <typename E, bool kBlock>
static sv_status launch_race(RaceParams rp, cudaStream_t stream) {
  const int64_t jobs = rp.B;
  if (jobs == 0) return SV_OK;
  rp.CL = race_split(rp.S, jobs);
  // the kernel's share: ceil(V / (CL * kPer)) whole vectors, staged in shared memory unless it is
  // too large, or unless staging would leave too few resident CTAs for one wave of every share
  constexpr int64_t kPer = Elem<E>::kPerVec;
  auto share_of = [&](int32_t cl) { return (rp.V + cl * kPer - 1) / (cl * kPer) * 16; };
  int64_t share_bytes = share_of(rp.CL);
  rp.stage_share = share_bytes <= int64_t(kRaceShareMax);
  const int sms = device_sm_count();
  const int smem_sm = device_smem_per_sm();
  if (rp.stage_share && sms > 0 && smem_sm > 0) {
    const int64_t per_sm = std::min<int64_t>(kRaceCtasPerSm, smem_sm / (share_bytes + 4096));
    if (jobs * rp.CL > int64_t(sms) * per_sm && jobs * rp.CL <= int64_t(sms) * kRaceCtasPerSm)
      rp.stage_share = false;
  }
  if (!rp.stage_share && sms > 0 && jobs * rp.CL <= int64_t(sms) * kRaceCtasPerSm) {
    // one wave of shares that cannot all be staged: twice as many shares, half as large (staged
    // if they fit) beat it -- 128 jobs of V = 129280 bf16, 4 -> 8 shares: 0.148 -> 0.144 ms per
    // block-verification call; 512 jobs, 1 -> 2 shares: the race of a scheduled round 102 -> 98 us
    const int32_t cl2 = std::min<int32_t>(std::min<int32_t>(rp.S, kRaceSplitFew), 2 * rp.CL);
    if (cl2 > rp.CL) {
      rp.CL = cl2;
      share_bytes = share_of(cl2);
      rp.stage_share = share_bytes <= int64_t(kRaceShareMax);
    }
  }
  const size_t smem = rp.stage_share ? size_t(share_bytes) : 0;
  if (cudaFuncSetAttribute(race_kernel<E, kBlock>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kRaceShareMax)) != cudaSuccess)
    return SV_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(jobs * rp.CL));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return launch_status(cudaLaunchKernelEx(&cfg, race_kernel<E, kBlock>, rp));
}

// ---------------------------------------------------------------------------------------------
// finish: partial race winners -> outputs
// ---------------------------------------------------------------------------------------------
// The largest of n partial race winners per request -- the largest of the race over p if no
// partial had a residual entry -- and the request's outputs.  winners_all is [n][B][2] packed
// results (race_pack; 0: none), the residual (or bonus) winner first, the race over p second.
// With `pending` set, a request whose pending[r] is 0 was decided before: its packed winner is
// decided[r] and winners_all is not read for it.  One thread per request.
template <int kDummy = 0>
__global__ void winners_finish_kernel(const unsigned long long* winners_all, int32_t n,
                                      int32_t B, const int32_t* accepted_len,
                                      const int64_t* draft_row0, const int32_t* draft_tokens,
                                      int32_t* out_tokens, int64_t out_ld,
                                      int32_t* correction_token, int32_t* status,
                                      const int32_t* pending = nullptr,
                                      const unsigned long long* decided = nullptr) {
  // launched as a programmatic dependent or not: the wait is a no-op in the second case
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int32_t r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= B) return;
  unsigned long long best = 0ull, fb = 0ull;
  if (pending && !pending[r]) {
    best = decided[r];
  } else {
    for (int32_t k = 0; k < n; ++k) {
      best = max(best, winners_all[(size_t(k) * B + r) * 2]);
      fb = max(fb, winners_all[(size_t(k) * B + r) * 2 + 1]);
    }
  }
  if (!best) best = fb;
  const int32_t y = best ? race_unpack_index(best) : -1;
  if (y < 0) report(status, SV_ERR_BAD_INPUT);  // the row carries no probability at all
  const int32_t tau = accepted_len[r];
  int32_t* out = out_tokens + size_t(r) * out_ld;
  for (int64_t q = 0; q < out_ld; ++q) {
    int32_t v = -1;
    if (q < tau) v = draft_tokens[draft_row0[r] + q];
    else if (q == tau) v = y;
    out[q] = v;
  }
  if (correction_token) correction_token[r] = y;
}

}  // namespace
}  // namespace sv
