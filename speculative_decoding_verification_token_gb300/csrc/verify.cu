// verify.cu -- token-level and block verification, and draft sampling from q.
//
// Token-level verification is two kernels on the caller's stream:
//   stream  persistent, warp-specialised CTAs (one per SM): a producer warp walks this CTA's
//           items -- a chunk of one (request, position) row pair -- and feeds a three-deep ring of
//           32 KB shared-memory stages with bulk copies; sixteen consumer warps fold every staged
//           element into log2-domain softmax statistics; the last warp to finish an item merges
//           the warps' results into one partial per (row pair, chunk), so no consumer ever waits
//           on another.  Positions are walked highest first, so the early positions -- where the
//           first rejection and hence the correction race most often fall -- are read last and
//           are still in L2 when the race reads them again.
//   race    up to 8 CTAs per request.  Each first decides its request: it folds the partials of
//           the request's rows into the row normalisers and the ratios p(x)/q(x), draws the
//           uniforms and finds the first rejection.  It then stages its contiguous share of the
//           correction (or bonus) row in shared memory with one bulk copy and runs the exponential
//           race of the share, pruned against the best seed key any share has published; the
//           shares combine through one 64-bit atomic max per request and the last share to finish
//           writes the outputs.  It is launched as a programmatic dependent of the stream kernel,
//           so its launch overlaps the stream's tail.
// Block verification is block -> race: the block kernel (one CTA per request, the same producer /
// consumer ring) walks the request's row pairs in order, each pair's statistics pass from HBM
// followed by its residual pass re-read from L2, and decides the request; the race kernel then
// draws its correction or bonus token.
#include <algorithm>
#include <mutex>

#include <cuda.h>

#include "race.cuh"
#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kStreamThreads = kConsumers + 32;  // + one producer warp
constexpr uint32_t kRowBytes = 32768;            // bytes of one row in one stream stage
constexpr int kStagesPerItem = 2;                // stages of one item (one merge per item)
constexpr uint32_t kItemBytes = kStagesPerItem * kRowBytes;
constexpr int kRing = 3;                         // stages of 2 x kRowBytes (target + draft)
constexpr int kRedBufs = 4;                      // items a consumer warp may run ahead, plus one
constexpr size_t kStreamSmem = size_t(kRing) * 2 * kRowBytes;
constexpr int kRaceSplitMax = 8;                 // CTAs (row shares) per race job, many jobs
constexpr int kRaceSplitFew = 16;                // the same when one wave holds every share
constexpr int kRaceCtasPerSm = 4;                // resident race CTAs per SM (launch bounds)
constexpr uint32_t kRaceShareMax = 64 * 1024;    // largest row share staged in shared memory

struct RaceDesc {  // per request, written by decide, read by race
  int32_t tau;
  int32_t resid;   // 1: correction from the residual of row pair tau+1; 0: bonus row
  float gap;       // log of q / (w p) at d = t: (m_t - m_d) ln 2 + log(s_t / (w s_d))
  int32_t pad;
};

struct RaceSlot {                 // per race job: the shares' combined winner
  unsigned long long best;        // race_pack(key, index); 0: no candidate yet
  uint32_t count;                 // shares finished
  uint32_t k0;                    // key_order of the best seed key published so far (0: none)
};

struct VerifyWs {
  float4* partials;  // [units * C] (m_t, s_t, m_d, s_d), m in log2 units (token-level)
  RaceDesc* desc;    // [B] (block)
  RaceSlot* slots;   // [units]: verify uses B of them, the sampler one per drafted row
  size_t total;
};

static inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static inline int32_t slices_of(int64_t V, int esz) {
  const int64_t per = kSliceBytes / esz;
  return static_cast<int32_t>((V + per - 1) / per);
}

// Stream items (chunks) per row: up to kStagesPerItem stages of kRowBytes each.
static inline int32_t chunks_of(int64_t V, int esz) {
  const int64_t per = kItemBytes / esz;
  return static_cast<int32_t>((V + per - 1) / per);
}

static VerifyWs verify_layout(void* base, int32_t B, int32_t gmax, int32_t C) {
  VerifyWs w;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* q = p + off;
    off = align256(off + bytes);
    return q;
  };
  const size_t Bn = size_t(B > 0 ? B : 1);
  const size_t units = Bn * size_t(gmax > 0 ? gmax : 1);
  w.partials = reinterpret_cast<float4*>(take(sizeof(float4) * units * size_t(C)));
  w.desc = reinterpret_cast<RaceDesc*>(take(sizeof(RaceDesc) * Bn));
  w.slots = reinterpret_cast<RaceSlot*>(take(sizeof(RaceSlot) * units));
  w.total = off;
  return w;
}

__device__ __forceinline__ int32_t clamp_gamma(int32_t g, int32_t gmax) {
  return (g < 0 || g > gmax) ? 0 : g;
}

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
};

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
  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int32_t i = p.gmax - static_cast<int32_t>(item / per_pos);  // highest position first
    const int64_t rem = item % per_pos;
    const int32_t r = static_cast<int32_t>(rem / p.C);
    const int32_t c = static_cast<int32_t>(rem % p.C);
    if (i > clamp_gamma(p.draft_len[r], p.gmax)) continue;  // request r drafted fewer tokens
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
};

// p_j(x)/q_j(x) of the drafted token x from the row pair's statistics nm = (m_t, s_t, m_d, s_d)
// (log2 domain) and the two logits of x; `bad` flags a data error: an all -inf row (its sum is
// 0), a NaN or +inf logit (the sum is NaN), x out of range, or q(x) = 0.
__device__ __forceinline__ float row_ratio(float4 nm, int32_t x, int64_t V, float tx, float dx,
                                           bool& bad) {
  bad = !(nm.y > 0.f && nm.y < INFINITY && nm.w > 0.f && nm.w < INFINITY);
  if (x < 0 || int64_t(x) >= V) {
    bad = true;
    return 0.f;
  }
  if (!(dx > -INFINITY)) bad = true;  // q(x) = 0: x cannot have been proposed
  // p(x)/q(x) = 2^((t_x log2e - m_t) - (d_x log2e - m_d)) s_d / s_t
  return exp2f(fmaf(tx, kLog2e, -nm.x) - fmaf(dx, kLog2e, -nm.z)) * (nm.w / nm.y);
}

// log of q(x) / (w p(x)) at d = t for the row pair's statistics nm and lnw = log w:
// (m_t - m_d) ln 2 + log(s_t / s_d) - log w, so that q(x) / (w p(x)) = exp((d - t) + gap).
__device__ __forceinline__ float resid_gap(float4 nm, float lnw) {
  return (nm.x - nm.z) * kLn2 + logf(nm.y / nm.w) - lnw;
}

// Drafted token x of position i of request r and its target and draft logits (lane 0 of a warp).
template <typename E>
__device__ __forceinline__ void fetch_drafted(const DecideParams& p, int32_t r, int32_t i,
                                              int32_t& x, float& tx, float& dx) {
  const int64_t drow = p.draft_row0[r] + (i - 1);
  x = p.draft_tokens[drow];
  tx = dx = 0.f;
  if (x >= 0 && int64_t(x) < p.V) {
    tx = Elem<E>::load(row_ptr<E>(p.target, p.target_row0[r] + (i - 1), p.ld), x);
    dx = Elem<E>::load(row_ptr<E>(p.draft, drow, p.ld), x);
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
  // the race kernel that follows may launch now (it waits for this grid's results itself)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (blockIdx.x == 0)  // the race's per-request slots start empty
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) p.ws.slots[i] = RaceSlot{0ull, 0u, 0u};
  __syncthreads();
  if (warp == kConsumerWarps) {
    if ((threadIdx.x & 31) == 0) block_producer<E>(p, ring, full, empty, meta, &bs);
  } else {
    block_consumer<E>(p, ring, full, empty, meta, &bs);
  }
}

// ---------------------------------------------------------------------------------------------
// race: CL CTAs per job -- the correction / bonus token of a request (verify), or one drafted
// token (sampler)
// ---------------------------------------------------------------------------------------------
struct RaceParams {
  const uint8_t* target;  // verify: target logits; sampler: the draft logits
  const uint8_t* draft;
  int64_t V, ld;
  const int64_t* target_row0;
  const int64_t* draft_row0;
  const int32_t* draft_len;
  const int32_t* draft_tokens;
  int32_t B, gmax, S, CL;  // 16 KB slices per row, CTAs (row shares) per job
  int32_t sampler;
  uint64_t seed;
  const uint64_t* request_ids;
  int32_t* accepted_len;
  int32_t* out_tokens;
  int64_t out_ld;
  int32_t* correction_token;
  int32_t* sampled_tokens;  // sampler output, indexed like the draft rows
  VerifyWs ws;
  int32_t* status;
  int32_t fused;            // token-level verify: decide in this kernel (dp), rank 0 writing
  int32_t stage_share;      // the launch provides dynamic shared memory for the row share
  DecideParams dp;
};

template <typename E>
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
  const int32_t job = blockIdx.x / p.CL;
  const int32_t part = blockIdx.x - job * p.CL;  // this CTA's share of the job's row
  // launched as a programmatic dependent of the previous kernel: wait for its results (the
  // token-level decision waits inside decide_body, after fetching the call's own inputs)
  const bool decide_here = !p.sampler && p.fused;
  if (!decide_here) asm volatile("griddepcontrol.wait;" ::: "memory");

  // resolve the job
  bool active = true;
  RaceSpec rs;
  const uint8_t* trow;
  const uint8_t* drow = nullptr;
  int32_t r, tau = 0, pos;
  int64_t sample_row = 0;
  if (!p.sampler) {
    r = job;
    if (p.fused) {
      decide_body<E>(p.dp, r, part == 0, &s_desc, s_tok, true);
      __syncthreads();
    }
    const RaceDesc d = p.fused ? s_desc : p.ws.desc[r];
    tau = d.tau;
    rs.resid = d.resid != 0;
    rs.gap = d.gap;
    pos = tau + 1;
    trow = row_ptr<E>(p.target, p.target_row0[r] + tau, p.ld);
    if (rs.resid) drow = row_ptr<E>(p.draft, p.draft_row0[r] + tau, p.ld);
  } else {
    r = job / p.gmax;
    pos = job - r * p.gmax + 1;
    const int32_t g = p.draft_len[r];
    if (g < 0 || g > p.gmax) {
      if (tid == 0 && part == 0 && pos == 1) report(p.status, SV_ERR_BAD_INPUT);
      active = false;
    } else if (pos > g) {
      active = false;
    }
    rs.resid = false;
    rs.gap = 0.f;
    sample_row = p.draft_row0[r] + (pos - 1);
    trow = row_ptr<E>(p.target, active ? sample_row : 0, p.ld);
  }
  const uint64_t req = p.request_ids ? p.request_ids[r] : uint64_t(r);
  rs.st = make_stream(p.seed, req, pos, p.sampler ? kTagDraft : (rs.resid ? kTagResid : kTagBonus));

  // this CTA's share of the row: a contiguous range, a whole number of 16-byte vectors long
  constexpr int32_t kPer = Elem<E>::kPerVec;
  const int64_t share = (p.V + int64_t(p.CL) * kPer - 1) / (int64_t(p.CL) * kPer) * kPer;
  const int64_t lo = min(p.V, int64_t(part) * share);
  const int64_t hi = min(p.V, lo + share);

  // stage the share's whole 16-byte vectors in shared memory with one bulk copy (shares too
  // large for it are read from global memory); a ragged tail is read from global memory
  const uint32_t vec_bytes = static_cast<uint32_t>(((hi - lo) * esize<E>()) & ~int64_t(15));
  const bool staged = p.stage_share && active && vec_bytes > 0;
  if (tid == 0 && staged) {
    mbar_init(&share_bar, 1);
    fence_barrier_init();
    mbar_expect_tx(&share_bar, vec_bytes);
    bulk_g2s(share_sm, trow + lo * esize<E>(), vec_bytes, &share_bar);
  }
  __syncthreads();
  const uint4* gsrc = reinterpret_cast<const uint4*>(trow + lo * esize<E>());

  // seed: the best exact key among the threads' largest-logit entries, raised to the best seed
  // the job's other shares have published so far -- a lower bound on the winning key, against
  // which the main pass gates.  It reads the share from global memory (L2) while the bulk copy
  // stages it for the main pass.
  RaceSlot* slot = p.ws.slots + job;
  float seed = active ? seed_range<E>(rs, gsrc, trow, drow, lo, int32_t(hi - lo)) : -INFINITY;
  if (staged) mbar_wait(&share_bar, 0, p.status);
  const uint4* vsrc = staged ? reinterpret_cast<const uint4*>(share_sm) : gsrc;
  seed = block_max(seed, red_k);
  if (tid == 0) {
    const uint32_t prev = active ? atomicMax(&slot->k0, key_order(seed)) : 0u;
    s_k0 = fmaxf(seed, key_from_order(prev));
  }
  __syncthreads();
  const float K0 = s_k0;

  // main pass: only entries whose logit and noise can reach K0 are keyed
  float bk = -INFINITY;
  int32_t bi = -1;
  if (active) {
    if (staged) race_range<E>(rs, vsrc, trow, drow, lo, int32_t(hi - lo), K0, bk, bi);
    else race_range<E, kBatchGlobal>(rs, vsrc, trow, drow, lo, int32_t(hi - lo), K0, bk, bi);
  }
  block_race(bk, bi, red_k, red_i);

  // combine the shares: a 64-bit max over (order-preserving key bits, ~index), so equal keys go
  // to the lower index; the last share to arrive writes the job's outputs
  if (tid == 0) {
    if (bi >= 0) atomicMax(&slot->best, race_pack(bk, bi));
    // release: this share's maximum before its count; acquire (last share): every share's
    s_last = atom_add_acq_rel(&slot->count, 1u) == uint32_t(p.CL - 1);
  }
  __syncthreads();
  if (!s_last || !active) return;
  if (tid == 0) {
    const unsigned long long best = atomicAdd(&slot->best, 0ull);
    s_winner = best ? race_unpack_index(best) : -1;
  }
  __syncthreads();
  int32_t y = s_winner;
  if (y < 0 && rs.resid) {
    // residual empty to working precision (p and q agree): draw from p with the same uniforms
    RaceSpec fb = rs;
    fb.resid = false;
    float k;
    race_row_global<E>(fb, trow, nullptr, p.V, red_k, red_i, k, y);
  }
  if (!p.sampler) {
    int32_t* out = p.out_tokens + size_t(r) * p.out_ld;
    for (int64_t q = tid; q < p.out_ld; q += kThreads) {
      int32_t v = -1;
      if (q < tau) v = p.fused ? s_tok[q] : p.draft_tokens[p.draft_row0[r] + q];
      else if (q == tau) v = y;
      out[q] = v;
    }
  }
  if (tid == 0) {
    if (y < 0) report(p.status, SV_ERR_BAD_INPUT);  // the row carries no probability at all
    if (!p.sampler) {
      p.accepted_len[r] = tau;
      if (p.correction_token) p.correction_token[r] = y;
    } else {
      p.sampled_tokens[sample_row] = y;
    }
  }
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
static size_t verify_ws_bytes(int32_t B, int32_t gmax, int64_t V, int esz) {
  return verify_layout(nullptr, B, gmax, chunks_of(V, esz)).total;
}

struct CommonArgs {
  const void* target;
  const void* draft;
  sv_dtype dtype;
  int64_t V, ld;
  int32_t B, gmax;
  void* ws;
  size_t ws_bytes;
};

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

static sv_status check_common(const CommonArgs& a, bool need_target) {
  if (a.dtype != SV_F32 && a.dtype != SV_BF16) return SV_ERR_INVALID;
  if (a.V <= 0 || a.ld < a.V || a.B < 0) return SV_ERR_INVALID;
  if (a.gmax < 0 || a.gmax > SV_MAX_DRAFT_LEN) return SV_ERR_INVALID;
  if (a.V >= (int64_t(1) << 31)) return SV_ERR_UNSUPPORTED;
  if (!a.draft && a.gmax > 0) return SV_ERR_INVALID;
  if (need_target && !a.target) return SV_ERR_INVALID;
  const int esz = elem_bytes(a.dtype);
  if ((a.ld * esz) % 16 != 0) return SV_ERR_UNSUPPORTED;
  if ((a.target && !aligned16(a.target)) || (a.draft && !aligned16(a.draft)))
    return SV_ERR_UNSUPPORTED;
  if (!a.ws || !aligned256(a.ws)) return SV_ERR_INVALID;
  if (a.ws_bytes < verify_ws_bytes(a.B, a.gmax, a.V, esz)) return SV_ERR_INVALID;
  return SV_OK;
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
static sv_status launch_race(RaceParams rp, int64_t jobs, cudaStream_t stream) {
  if (jobs == 0) return SV_OK;
  rp.CL = race_split(rp.S, jobs);
  // the kernel's share: ceil(V / (CL * kPer)) whole vectors
  constexpr int64_t kPer = Elem<E>::kPerVec;
  const int64_t share_bytes = (rp.V + rp.CL * kPer - 1) / (rp.CL * kPer) * 16;
  rp.stage_share = share_bytes <= int64_t(kRaceShareMax);
  const size_t smem = rp.stage_share ? size_t(share_bytes) : 0;
  if (cudaFuncSetAttribute(race_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
  return launch_status(cudaLaunchKernelEx(&cfg, race_kernel<E>, rp));
}

template <typename E>
static sv_status run_verify(bool block, const CommonArgs& a, const int64_t* target_row0,
                            const int64_t* draft_row0, const int32_t* draft_len,
                            const int32_t* draft_tokens, uint64_t seed,
                            const uint64_t* request_ids, int32_t* accepted_len,
                            int32_t* out_tokens, int64_t out_ld, int32_t* correction_token,
                            float* ratio_out, float* h_out, int32_t* status,
                            cudaStream_t stream) {
  const int32_t S = slices_of(a.V, esize<E>());
  const int32_t C = chunks_of(a.V, esize<E>());
  const VerifyWs ws = verify_layout(a.ws, a.B, a.gmax, C);
  // token-level verification with rows to stream clears the status word in its first kernel
  const bool stream_clears = !block && int64_t(a.gmax) * a.B * C > 0;
  if (status && !stream_clears &&
      cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return SV_ERR_CUDA;

  const uint8_t* target = static_cast<const uint8_t*>(a.target);
  const uint8_t* draft = static_cast<const uint8_t*>(a.draft);
  DecideParams dp = {};
  sv_status st;
  if (!block) {
    StreamParams sp = {};
    sp.target = target;
    sp.draft = draft;
    sp.V = a.V;
    sp.ld = a.ld;
    sp.target_row0 = target_row0;
    sp.draft_row0 = draft_row0;
    sp.draft_len = draft_len;
    sp.B = a.B;
    sp.gmax = a.gmax;
    sp.C = C;
    sp.ws = ws;
    sp.status = status;
    sp.clear_status = stream_clears ? 1 : 0;
    profile_mark(0, stream);
    st = launch_stream<E>(sp, stream);
    if (st != SV_OK) return st;
    if (a.gmax == 0 &&  // no stream launch: the race slots are zeroed here instead
        cudaMemsetAsync(ws.slots, 0, sizeof(RaceSlot) * size_t(a.B), stream) != cudaSuccess)
      return SV_ERR_CUDA;
    profile_mark(1, stream);  // the race kernel decides (no kernel in between)
    dp.target = target;
    dp.draft = draft;
    dp.V = a.V;
    dp.ld = a.ld;
    dp.target_row0 = target_row0;
    dp.draft_row0 = draft_row0;
    dp.draft_len = draft_len;
    dp.draft_tokens = draft_tokens;
    dp.B = a.B;
    dp.gmax = a.gmax;
    dp.C = C;
    dp.seed = seed;
    dp.request_ids = request_ids;
    dp.ratio_out = ratio_out;
    dp.ws = ws;
    dp.status = status;
  } else {
    BlockParams bp;
    bp.target = target;
    bp.draft = draft;
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
    bp.rho_out = ratio_out;
    bp.h_out = h_out;
    bp.accepted_len = accepted_len;
    bp.out_tokens = out_tokens;
    bp.out_ld = out_ld;
    bp.correction_token = correction_token;
    bp.ws = ws;
    bp.status = status;
    profile_mark(0, stream);
    st = launch_block<E>(bp, stream);
    if (st != SV_OK) return st;
    profile_mark(1, stream);
    profile_mark(2, stream);
    profile_mark(3, stream);  // the block kernel draws the correction itself
    return launch_status(cudaGetLastError());
  }
  profile_mark(2, stream);

  RaceParams rp = {};
  rp.target = target;
  rp.draft = draft;
  rp.V = a.V;
  rp.ld = a.ld;
  rp.target_row0 = target_row0;
  rp.draft_row0 = draft_row0;
  rp.draft_len = draft_len;
  rp.draft_tokens = draft_tokens;
  rp.B = a.B;
  rp.gmax = a.gmax;
  rp.S = S;
  rp.sampler = 0;
  rp.seed = seed;
  rp.request_ids = request_ids;
  rp.accepted_len = accepted_len;
  rp.out_tokens = out_tokens;
  rp.out_ld = out_ld;
  rp.correction_token = correction_token;
  rp.ws = ws;
  rp.status = status;
  rp.fused = block ? 0 : 1;
  rp.dp = dp;
  st = launch_race<E>(rp, a.B, stream);
  if (st != SV_OK) return st;
  profile_mark(3, stream);
  return launch_status(cudaGetLastError());
}

template <typename E>
static sv_status run_sample(const CommonArgs& a, const int64_t* draft_row0,
                            const int32_t* draft_len, uint64_t seed, const uint64_t* request_ids,
                            int32_t* draft_tokens, int32_t* status, cudaStream_t stream) {
  const int32_t S = slices_of(a.V, esize<E>());
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  RaceParams rp = {};
  rp.target = static_cast<const uint8_t*>(a.draft);
  rp.V = a.V;
  rp.ld = a.ld;
  rp.draft_row0 = draft_row0;
  rp.draft_len = draft_len;
  rp.B = a.B;
  rp.gmax = a.gmax;
  rp.S = S;
  rp.sampler = 1;
  rp.seed = seed;
  rp.request_ids = request_ids;
  rp.sampled_tokens = draft_tokens;
  rp.status = status;
  rp.ws = verify_layout(a.ws, a.B, a.gmax, chunks_of(a.V, esize<E>()));
  const int64_t jobs = int64_t(a.B) * a.gmax;
  if (jobs > 0 &&
      cudaMemsetAsync(rp.ws.slots, 0, sizeof(RaceSlot) * size_t(jobs), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  return launch_race<E>(rp, jobs, stream);
}

}  // namespace sv

using namespace sv;

extern "C" size_t spec_verify_workspace_bytes(int32_t B, int32_t max_draft_len, int64_t V,
                                              sv_dtype dtype) {
  if (B < 0 || max_draft_len < 0 || max_draft_len > SV_MAX_DRAFT_LEN || V <= 0) return 0;
  if (dtype != SV_F32 && dtype != SV_BF16) return 0;
  return verify_ws_bytes(B, max_draft_len, V, elem_bytes(dtype));
}

static sv_status verify_entry(bool block, const void* target_logits, const void* draft_logits,
                              sv_dtype dtype, int64_t V, int64_t ld, const int64_t* target_row0,
                              const int64_t* draft_row0, const int32_t* draft_len,
                              int32_t max_draft_len, const int32_t* draft_tokens, int32_t B,
                              uint64_t seed, const uint64_t* request_ids, int32_t* accepted_len,
                              int32_t* out_tokens, int64_t out_ld, int32_t* correction_token,
                              float* ratio_out, float* h_out, int32_t* status, void* workspace,
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
    return run_verify<bf16_tag>(block, a, target_row0, draft_row0, draft_len, draft_tokens, seed,
                                request_ids, accepted_len, out_tokens, out_ld, correction_token,
                                ratio_out, h_out, status, s);
  return run_verify<float>(block, a, target_row0, draft_row0, draft_len, draft_tokens, seed,
                           request_ids, accepted_len, out_tokens, out_ld, correction_token,
                           ratio_out, h_out, status, s);
}

extern "C" sv_status spec_verify_token(const void* target_logits, const void* draft_logits,
                                       sv_dtype dtype, int64_t V, int64_t ld,
                                       const int64_t* target_row0, const int64_t* draft_row0,
                                       const int32_t* draft_len, int32_t max_draft_len,
                                       const int32_t* draft_tokens, int32_t B, uint64_t seed,
                                       const uint64_t* request_ids, int32_t* accepted_len,
                                       int32_t* out_tokens, int64_t out_ld,
                                       int32_t* correction_token, float* accept_ratio,
                                       int32_t* status, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  return verify_entry(false, target_logits, draft_logits, dtype, V, ld, target_row0, draft_row0,
                      draft_len, max_draft_len, draft_tokens, B, seed, request_ids, accepted_len,
                      out_tokens, out_ld, correction_token, accept_ratio, nullptr, status,
                      workspace, workspace_bytes, stream);
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
  return verify_entry(true, target_logits, draft_logits, dtype, V, ld, target_row0, draft_row0,
                      draft_len, max_draft_len, draft_tokens, B, seed, request_ids, accepted_len,
                      out_tokens, out_ld, correction_token, running_ratio, h_threshold, status,
                      workspace, workspace_bytes, stream);
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
