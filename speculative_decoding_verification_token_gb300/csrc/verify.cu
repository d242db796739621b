// verify.cu -- token-level and block verification, and draft sampling from q.
//
// One verify call is a short chain of kernels on the caller's stream:
//   plan    1 CTA: orders the (request, position) row pairs by position (highest first), clears the
//           tickets, resets the status word.
//   stream  persistent CTAs read every drafted row pair once from HBM in 16 KB slices (bulk copies
//           into a two-stage shared-memory ring) and fold each slice into online softmax
//           statistics.  The CTA that finishes the last slice of a row pair combines the slices
//           into the row normalisers and the ratio p(x)/q(x) of its drafted token; in block mode
//           the last row of a request also yields the running capped ratios rho_i.
//   resid   (block verification only) the same stream over row pairs 2..gamma computes the
//           residual masses R_{i-1} = sum_x max(rho_{i-1} p_i(x) - q_i(x), 0).
//   final   one CTA per (request, slice) decides the accepted length and runs the exponential race
//           of the correction (or bonus) row on its slice; the CTA that finishes last for a request
//           picks the winner and writes the request's outputs.
// Row pairs are streamed highest position first, so the early positions -- where the first
// rejection, and therefore the correction race, most often falls -- are the most recently read
// when the final kernel reads them again.
#include <algorithm>
#include <mutex>

#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

struct RowInfo {  // one (request, position) row pair
  float ct;       // log normaliser of the target row: max + log(sum exp(t - max))
  float cd;       // log normaliser of the draft row
  float ratio;    // p(x)/q(x) of the drafted token x
  float rho;      // block verification: running capped ratio rho_i
};

struct VerifyWs {
  int32_t* hdr;       // [0] = number of row-pair units
  int32_t* cnt;       // [gmax + 1]: cnt[i] = #requests with gamma >= i (i >= 1)
  int32_t* base;      // [gmax + 1]: index of the first unit of position i (positions descending)
  int32_t* perm;      // [B] requests by decreasing gamma
  int32_t* tickets;   // start of the ticket block cleared by the plan kernel
  int32_t* tick_a;    // [B * gmax] slices of a row pair streamed
  int32_t* tick_r;    // [B * gmax] slices of a residual mass streamed
  int32_t* tick_req;  // [B] rows of a request combined (block)
  int32_t* tick_f;    // [B] slices of the final race done
  int32_t n_tickets;
  float4* partials;   // [B * gmax * S] (m_t, s_t, m_d, s_d) per slice
  RowInfo* rows;      // [B * gmax]
  float4* norms;      // [B * gmax] (m_t, s_t, m_d, s_d) of the whole row pair
  float* rpart;       // [B * gmax * S] residual mass per slice
  float* rmass;       // [B * gmax] R_{i-1} stored at unit (r, i)
  int2* race;         // [B * S] (key bits, index) per slice of the final race
  size_t total;
};

static inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static VerifyWs verify_layout(void* base, int32_t B, int32_t gmax, int32_t S) {
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
  w.hdr = reinterpret_cast<int32_t*>(take(16));
  w.cnt = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (gmax + 2)));
  w.base = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * (gmax + 2)));
  w.perm = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * Bn));
  w.n_tickets = static_cast<int32_t>(2 * units + 2 * Bn);
  w.tickets = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * size_t(w.n_tickets)));
  w.tick_a = w.tickets;
  w.tick_r = w.tick_a + units;
  w.tick_req = w.tick_r + units;
  w.tick_f = w.tick_req + Bn;
  w.partials = reinterpret_cast<float4*>(take(sizeof(float4) * units * S));
  w.rows = reinterpret_cast<RowInfo*>(take(sizeof(RowInfo) * units));
  w.norms = reinterpret_cast<float4*>(take(sizeof(float4) * units));
  w.rpart = reinterpret_cast<float*>(take(sizeof(float) * units * S));
  w.rmass = reinterpret_cast<float*>(take(sizeof(float) * units));
  w.race = reinterpret_cast<int2*>(take(sizeof(int2) * Bn * S));
  w.total = off;
  return w;
}

static inline int32_t slices_of(int64_t V, int esize) {
  const int64_t per = kSliceBytes / esize;
  return static_cast<int32_t>((V + per - 1) / per);
}

__device__ __forceinline__ int32_t clamp_gamma(int32_t g, int32_t gmax) {
  return (g < 0 || g > gmax) ? 0 : g;
}

// ---------------------------------------------------------------------------------------------
// plan
// ---------------------------------------------------------------------------------------------
struct PlanParams {
  const int32_t* draft_len;
  int32_t B, gmax;
  VerifyWs ws;
  int32_t* status;
};

__global__ void __launch_bounds__(1024) plan_kernel(PlanParams p) {
  __shared__ int32_t hist[SV_MAX_DRAFT_LEN + 2];
  __shared__ int32_t start[SV_MAX_DRAFT_LEN + 2];
  const int tid = threadIdx.x;
  if (tid == 0 && p.status) *p.status = SV_OK;
  for (int i = tid; i < SV_MAX_DRAFT_LEN + 2; i += blockDim.x) hist[i] = 0;
  for (int32_t i = tid; i < p.ws.n_tickets; i += blockDim.x) p.ws.tickets[i] = 0;
  __syncthreads();
  for (int r = tid; r < p.B; r += blockDim.x) {
    const int32_t g = p.draft_len[r];
    if (g < 0 || g > p.gmax) report(p.status, SV_ERR_BAD_INPUT);
    atomicAdd(&hist[clamp_gamma(g, p.gmax)], 1);
  }
  __syncthreads();
  if (tid == 0) {
    int32_t acc = 0;
    for (int g = p.gmax; g >= 0; --g) {  // slots of requests sorted by decreasing gamma
      start[g] = acc;
      acc += hist[g];
    }
    int32_t ge = 0, units = 0;
    for (int i = p.gmax; i >= 1; --i) {
      ge += hist[i];
      p.ws.cnt[i] = ge;
      p.ws.base[i] = units;
      units += ge;
    }
    p.ws.cnt[0] = 0;
    p.ws.base[0] = units;
    p.ws.hdr[0] = units;
  }
  __syncthreads();
  for (int r = tid; r < p.B; r += blockDim.x) {
    const int slot = atomicAdd(&start[clamp_gamma(p.draft_len[r], p.gmax)], 1);
    p.ws.perm[slot] = r;
  }
}

// ---------------------------------------------------------------------------------------------
// stream: statistics pass and residual-mass pass
// ---------------------------------------------------------------------------------------------
struct StreamParams {
  const uint8_t* target;
  const uint8_t* draft;
  int64_t V, ld;
  const int64_t* target_row0;
  const int64_t* draft_row0;
  const int32_t* draft_len;
  const int32_t* draft_tokens;
  int32_t B, gmax, S;
  int32_t block;       // block verification: also produce running ratios
  int32_t resid_pass;  // this launch streams row pairs 2..gamma for R_{i-1}
  VerifyWs ws;
  int32_t* status;
};

struct SliceMeta {
  int32_t unit, r, i, s;
  int32_t len, bulk_elems;
  int64_t trow, drow;
};

template <typename E>
constexpr int esize() {
  return 16 / Elem<E>::kPerVec;
}

template <typename E>
__device__ __forceinline__ const uint8_t* row_ptr(const uint8_t* base, int64_t row, int64_t ld) {
  return base + row * ld * esize<E>();
}

// Locate item `item` (unit, slice) and start the bulk copies of its two row slices.
template <typename E>
__device__ __forceinline__ void issue_slice(const StreamParams& p, int32_t item, uint8_t* buf_t,
                                            uint8_t* buf_d, uint64_t* bar, SliceMeta* meta) {
  constexpr int32_t kSE = kSliceBytes / esize<E>();
  const int32_t u = item / p.S;
  const int32_t s = item - u * p.S;
  int32_t i = p.gmax;
  while (u >= p.ws.base[i] + p.ws.cnt[i]) --i;
  const int32_t r = p.ws.perm[u - p.ws.base[i]];
  SliceMeta m;
  m.unit = r * p.gmax + (i - 1);
  m.r = r;
  m.i = i;
  m.s = s;
  const int64_t e0 = int64_t(s) * kSE;
  m.len = static_cast<int32_t>((p.V - e0 < int64_t(kSE) ? p.V - e0 : int64_t(kSE)));
  const uint32_t bulk_bytes = (uint32_t(m.len) * esize<E>()) & ~15u;
  m.bulk_elems = static_cast<int32_t>(bulk_bytes / esize<E>());
  m.trow = p.target_row0[r] + (i - 1);
  m.drow = p.draft_row0[r] + (i - 1);
  *meta = m;
  mbar_expect_tx(bar, 2 * bulk_bytes);
  if (bulk_bytes) {
    bulk_g2s(buf_t, row_ptr<E>(p.target, m.trow, p.ld) + e0 * esize<E>(), bulk_bytes, bar);
    bulk_g2s(buf_d, row_ptr<E>(p.draft, m.drow, p.ld) + e0 * esize<E>(), bulk_bytes, bar);
  }
}

// Fold the S slice statistics of a row pair into its normalisers and the drafted token's ratio.
// One warp.
template <typename E>
__device__ void combine_unit(const StreamParams& p, const SliceMeta& m, int lane) {
  float mt = -INFINITY, st = 0.f, md = -INFINITY, sd = 0.f;
  const float4* part = p.ws.partials + size_t(m.unit) * p.S;
  for (int j = lane; j < p.S; j += 32) {
    const float4 q = __ldcg(part + j);
    ms_merge(mt, st, q.x, q.y);
    ms_merge(md, sd, q.z, q.w);
  }
  warp_ms(mt, st);
  warp_ms(md, sd);
  if (lane != 0) return;
  RowInfo ri;
  // an all -inf row has s = 0; NaN or +inf logits make s NaN
  bool bad = !(st > 0.f && st < INFINITY && sd > 0.f && sd < INFINITY);
  ri.ct = mt + logf(st);
  ri.cd = md + logf(sd);
  ri.ratio = 0.f;
  ri.rho = 0.f;
  const int32_t x = p.draft_tokens[m.drow];
  if (x < 0 || int64_t(x) >= p.V) {
    bad = true;
  } else {
    // p(x)/q(x) = exp((t_x - m_t) - (d_x - m_d)) * s_d / s_t: the max-shifted logits are exact
    // in binary32, so only the exponential and the two sums carry rounding
    const float tx = Elem<E>::load(row_ptr<E>(p.target, m.trow, p.ld), x);
    const float dx = Elem<E>::load(row_ptr<E>(p.draft, m.drow, p.ld), x);
    if (!(dx > -INFINITY)) bad = true;  // q(x) = 0: the drafter cannot have proposed x
    ri.ratio = expf((tx - mt) - (dx - md)) * (sd / st);
  }
  if (bad) report(p.status, SV_ERR_BAD_INPUT);
  __stcg(reinterpret_cast<float4*>(&p.ws.rows[m.unit]), make_float4(ri.ct, ri.cd, ri.ratio, 0.f));
  __stcg(&p.ws.norms[m.unit], make_float4(mt, st, md, sd));
}

// Block verification: running capped ratios rho_i = min(1, rho_{i-1} * ratio_i) of request r once
// all its rows are combined.  One warp.
__device__ void running_ratios(const StreamParams& p, int32_t r, int32_t gamma, int lane) {
  RowInfo* rows = p.ws.rows + size_t(r) * p.gmax;
  float a0 = lane < gamma ? __ldcg(&rows[lane].ratio) : 0.f;
  float a1 = lane + 32 < gamma ? __ldcg(&rows[lane + 32].ratio) : 0.f;
  float rho = 1.f;
  for (int i = 0; i < gamma; ++i) {
    const float a = __shfl_sync(0xffffffffu, i < 32 ? a0 : a1, i & 31);
    rho = rho > 0.f ? fminf(1.f, rho * a) : 0.f;
    if (lane == 0) __stcg(&rows[i].rho, rho);
  }
}

template <typename E>
__global__ void __launch_bounds__(kThreads) stream_kernel(StreamParams p) {
  constexpr int kPer = Elem<E>::kPerVec;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bars[2];
  __shared__ SliceMeta meta[2];
  __shared__ float red[kWarps][4];
  __shared__ int32_t s_last;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t n_units = p.resid_pass ? p.ws.base[1] : p.ws.hdr[0];
  const int32_t n_items = n_units * p.S;
  if (int32_t(blockIdx.x) >= n_items) return;

  uint8_t* const buf_t[2] = {smem, smem + 2 * kSliceBytes};
  uint8_t* const buf_d[2] = {smem + kSliceBytes, smem + 3 * kSliceBytes};
  if (tid == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_barrier_init();
    issue_slice<E>(p, blockIdx.x, buf_t[0], buf_d[0], &bars[0], &meta[0]);
  }
  __syncthreads();

  int j = 0;
  for (int32_t item = blockIdx.x; item < n_items; item += gridDim.x, ++j) {
    const int stage = j & 1;
    const int32_t next = item + gridDim.x;
    if (tid == 0 && next < n_items) {
      fence_proxy_async();
      issue_slice<E>(p, next, buf_t[stage ^ 1], buf_d[stage ^ 1], &bars[stage ^ 1],
                     &meta[stage ^ 1]);
    }
    const SliceMeta m = meta[stage];
    if (!mbar_wait(&bars[stage], (j >> 1) & 1, p.status)) {
      // the copy never completed (cannot happen with consistent byte counts); give the copies in
      // flight a last bounded chance to land before the CTA leaves
      mbar_wait(&bars[stage ^ 1], ((j + 1) >> 1) & 1, nullptr);
      return;
    }
    const uint4* vt = reinterpret_cast<const uint4*>(buf_t[stage]);
    const uint4* vd = reinterpret_cast<const uint4*>(buf_d[stage]);
    const int nvec = m.bulk_elems / kPer;
    const int64_t e0 = int64_t(m.s) * (kSliceBytes / esize<E>());
    const uint8_t* trow = row_ptr<E>(p.target, m.trow, p.ld);
    const uint8_t* drow = row_ptr<E>(p.draft, m.drow, p.ld);
    float o0, o1, o2, o3;

    if (!p.resid_pass) {
      float mt = -INFINITY, st = 0.f, md = -INFINITY, sd = 0.f;
#pragma unroll 2
      for (int v = tid; v < nvec; v += kThreads) {
        float x[kPer], y[kPer];
        Elem<E>::unpack(vt[v], x);
        Elem<E>::unpack(vd[v], y);
        ms_accumulate<kPer>(mt, st, x);
        ms_accumulate<kPer>(md, sd, y);
      }
      for (int e = m.bulk_elems + tid; e < m.len; e += kThreads) {
        float x = Elem<E>::load(trow, e0 + e);
        float y = Elem<E>::load(drow, e0 + e);
        ms_accumulate<1>(mt, st, &x);
        ms_accumulate<1>(md, sd, &y);
      }
      warp_ms(mt, st);
      warp_ms(md, sd);
      o0 = mt;
      o1 = st;
      o2 = md;
      o3 = sd;
    } else {
      // mass of max(rho_{i-1} p_i(x) - q_i(x), 0) over the slice.  Each positive entry is
      // written rho p (1 - exp(y)) with rho p = A exp(t - m_t), A = rho_{i-1} / s_t, and
      // y = log(q / (rho p)) = (d - t) + gap, gap = (m_t - m_d) + log(s_t / (rho_{i-1} s_d)):
      // the difference is then accurate relative to itself, not to rho p.
      const float4 nm = __ldcg(&p.ws.norms[m.unit]);
      const float rho_prev = __ldcg(&p.ws.rows[m.unit - 1].rho);
      const float A = rho_prev / nm.y;
      const float gap = (nm.x - nm.z) + (logf(nm.y / nm.w) - logf(rho_prev));  // +inf if rho = 0
      float acc = 0.f;
#pragma unroll 2
      for (int v = tid; v < nvec; v += kThreads) {
        float x[kPer], y[kPer];
        Elem<E>::unpack(vt[v], x);
        Elem<E>::unpack(vd[v], y);
#pragma unroll
        for (int q = 0; q < kPer; ++q) {
          const float yy = (y[q] - x[q]) + gap;
          if (yy < 0.f) acc += A * fast_exp2((x[q] - nm.x) * kLog2e) * one_minus_exp(yy);
        }
      }
      for (int e = m.bulk_elems + tid; e < m.len; e += kThreads) {
        const float x = Elem<E>::load(trow, e0 + e);
        const float y = Elem<E>::load(drow, e0 + e);
        const float yy = (y - x) + gap;
        if (yy < 0.f) acc += A * fast_exp2((x - nm.x) * kLog2e) * one_minus_exp(yy);
      }
      o0 = warp_sum(acc);
      o1 = o2 = o3 = 0.f;
    }
    if (lane == 0) {
      red[warp][0] = o0;
      red[warp][1] = o1;
      red[warp][2] = o2;
      red[warp][3] = o3;
    }
    __syncthreads();
    if (tid == 0) {
      int32_t ticket;
      if (!p.resid_pass) {
        float mt = red[0][0], st = red[0][1], md = red[0][2], sd = red[0][3];
        for (int w = 1; w < kWarps; ++w) {
          ms_merge(mt, st, red[w][0], red[w][1]);
          ms_merge(md, sd, red[w][2], red[w][3]);
        }
        __stcg(&p.ws.partials[size_t(m.unit) * p.S + m.s], make_float4(mt, st, md, sd));
        __threadfence();
        ticket = atomicAdd(&p.ws.tick_a[m.unit], 1);
      } else {
        float acc = 0.f;
        for (int w = 0; w < kWarps; ++w) acc += red[w][0];
        __stcg(&p.ws.rpart[size_t(m.unit) * p.S + m.s], acc);
        __threadfence();
        ticket = atomicAdd(&p.ws.tick_r[m.unit], 1);
      }
      s_last = ticket == p.S - 1;
    }
    __syncthreads();
    if (s_last && warp == 0) {
      __threadfence();
      if (!p.resid_pass) {
        combine_unit<E>(p, m, lane);
        if (p.block) {
          __threadfence();
          int32_t done = 0;
          if (lane == 0) done = atomicAdd(&p.ws.tick_req[m.r], 1);
          done = __shfl_sync(0xffffffffu, done, 0);
          const int32_t gamma = clamp_gamma(p.draft_len[m.r], p.gmax);
          if (done == gamma - 1) {
            __threadfence();
            running_ratios(p, m.r, gamma, lane);
          }
        }
      } else {
        const float* part = p.ws.rpart + size_t(m.unit) * p.S;
        float acc = 0.f;
        for (int q = lane; q < p.S; q += 32) acc += __ldcg(part + q);
        acc = warp_sum(acc);
        if (lane == 0) __stcg(&p.ws.rmass[m.unit], acc);
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------------------------
// exponential race over one staged slice
// ---------------------------------------------------------------------------------------------
// Residual entries: weight max(w p(x) - q(x), 0) = w p(x) (-expm1(y)), y = (d - t) + gap, so the
// key log(weight) - log(E) is, up to a per-row constant, t + log(-expm1(y)) - log(E) (entries with
// y >= 0 carry no weight).  Plain entries (bonus row, drafts, the empty-residual fallback): t -
// log(E).  In both cases key <= t + kMaxNoise, which lets an entry be skipped without drawing its
// uniform once some key above that bound is known.
struct RaceSpec {
  bool resid;
  float gap;
  Stream st;
};

__device__ __forceinline__ float race_key(const RaceSpec& rs, float t, float d, float noise) {
  if (!rs.resid) return t + noise;
  const float y = (d - t) + rs.gap;
  return t + __logf(one_minus_exp(y)) + noise;
}

__device__ __forceinline__ bool race_active(const RaceSpec& rs, float t, float d) {
  return rs.resid ? ((d - t) + rs.gap < 0.f) : (t > -INFINITY);
}

// Per-thread helper: uniform of vocabulary entry v, reusing the Philox block of its group of four.
struct BlockCache {
  uint32_t group = 0xFFFFFFFFu;
  uint4 words;
  __device__ __forceinline__ float noise(const Stream& st, int64_t v) {
    const uint32_t g = static_cast<uint32_t>(v >> 2);
    if (g != group) {
      group = g;
      words = stream_block(st, g);
    }
    return race_noise(uniform_of(word_of(words, static_cast<uint32_t>(v & 3))));
  }
};

// Race over elements [0, len) of a slice starting at vocabulary index e0: [0, bulk_elems) staged
// in shared memory (st_t, st_d), the tail read from the global rows.  Returns the CTA-wide winner
// in (key, idx) on every thread.  Two passes: a seed pass evaluates, per thread, the entry of
// largest logit (a cheap lower bound on the winning key), the main pass skips every entry whose
// bound t + kMaxNoise is below the best seed.
template <typename E>
__device__ void race_slice(const RaceSpec& rs, const uint8_t* st_t, const uint8_t* st_d,
                           const uint8_t* trow, const uint8_t* drow, int64_t e0, int32_t len,
                           int32_t bulk_elems, float* red_k, int32_t* red_i, float& out_key,
                           int32_t& out_idx) {
  constexpr int kPer = Elem<E>::kPerVec;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint4* vt = reinterpret_cast<const uint4*>(st_t);
  const uint4* vd = reinterpret_cast<const uint4*>(st_d);
  const int nvec = bulk_elems / kPer;

  // seed pass
  float bt = -INFINITY;
  int32_t be = -1;
  for (int v = tid; v < nvec; v += kThreads) {
    float x[kPer], y[kPer];
    Elem<E>::unpack(vt[v], x);
    if (rs.resid) Elem<E>::unpack(vd[v], y);
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const float d = rs.resid ? y[q] : 0.f;
      if (race_active(rs, x[q], d) && x[q] > bt) {
        bt = x[q];
        be = v * kPer + q;
      }
    }
  }
  for (int e = bulk_elems + tid; e < len; e += kThreads) {
    const float x = Elem<E>::load(trow, e0 + e);
    const float d = rs.resid ? Elem<E>::load(drow, e0 + e) : 0.f;
    if (race_active(rs, x, d) && x > bt) {
      bt = x;
      be = e;
    }
  }
  float seed_key = -INFINITY;
  BlockCache cache;
  if (be >= 0) {
    float x, d = 0.f;
    if (be < bulk_elems) {
      float xs[kPer], ys[kPer];
      Elem<E>::unpack(vt[be / kPer], xs);
      x = xs[be % kPer];
      if (rs.resid) {
        Elem<E>::unpack(vd[be / kPer], ys);
        d = ys[be % kPer];
      }
    } else {
      x = Elem<E>::load(trow, e0 + be);
      if (rs.resid) d = Elem<E>::load(drow, e0 + be);
    }
    seed_key = race_key(rs, x, d, cache.noise(rs.st, e0 + be));
  }
  seed_key = warp_max(seed_key);
  if (lane == 0) red_k[warp] = seed_key;
  __syncthreads();
  float K0 = red_k[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) K0 = fmaxf(K0, red_k[w]);
  __syncthreads();

  // main pass
  float bk = -INFINITY;
  int32_t bi = -1;
  const float floor_t = K0 - kMaxNoise;  // entries with t < floor_t cannot reach K0
  for (int v = tid; v < nvec; v += kThreads) {
    float x[kPer], y[kPer];
    Elem<E>::unpack(vt[v], x);
    float xm = x[0];
#pragma unroll
    for (int q = 1; q < kPer; ++q) xm = fmaxf(xm, x[q]);
    if (!(xm >= floor_t)) continue;
    if (rs.resid) Elem<E>::unpack(vd[v], y);
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const float d = rs.resid ? y[q] : 0.f;
      if (x[q] >= floor_t && race_active(rs, x[q], d)) {
        const int32_t e = v * kPer + q;
        const float k = race_key(rs, x[q], d, cache.noise(rs.st, e0 + e));
        if (race_better(k, int32_t(e0 + e), bk, bi)) {
          bk = k;
          bi = int32_t(e0 + e);
        }
      }
    }
  }
  for (int e = bulk_elems + tid; e < len; e += kThreads) {
    const float x = Elem<E>::load(trow, e0 + e);
    const float d = rs.resid ? Elem<E>::load(drow, e0 + e) : 0.f;
    if (x >= floor_t && race_active(rs, x, d)) {
      const float k = race_key(rs, x, d, cache.noise(rs.st, e0 + e));
      if (race_better(k, int32_t(e0 + e), bk, bi)) {
        bk = k;
        bi = int32_t(e0 + e);
      }
    }
  }
  warp_race(bk, bi);
  if (lane == 0) {
    red_k[warp] = bk;
    red_i[warp] = bi;
  }
  __syncthreads();
  float k = red_k[0];
  int32_t i = red_i[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w)
    if (race_better(red_k[w], red_i[w], k, i)) {
      k = red_k[w];
      i = red_i[w];
    }
  __syncthreads();
  out_key = k;
  out_idx = i;
}

// Race over a whole row read from global memory by one CTA (rare fallback paths).
template <typename E>
__device__ void race_row_global(const RaceSpec& rs, const uint8_t* trow, const uint8_t* drow,
                                int64_t V, float* red_k, int32_t* red_i, float& out_key,
                                int32_t& out_idx) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float bk = -INFINITY;
  int32_t bi = -1;
  BlockCache cache;
  for (int64_t e = tid; e < V; e += kThreads) {
    const float x = Elem<E>::load(trow, e);
    const float d = rs.resid ? Elem<E>::load(drow, e) : 0.f;
    if (!race_active(rs, x, d)) continue;
    const float k = race_key(rs, x, d, cache.noise(rs.st, e));
    if (race_better(k, int32_t(e), bk, bi)) {
      bk = k;
      bi = int32_t(e);
    }
  }
  warp_race(bk, bi);
  if (lane == 0) {
    red_k[warp] = bk;
    red_i[warp] = bi;
  }
  __syncthreads();
  float k = red_k[0];
  int32_t i = red_i[0];
  for (int w = 1; w < kWarps; ++w)
    if (race_better(red_k[w], red_i[w], k, i)) {
      k = red_k[w];
      i = red_i[w];
    }
  __syncthreads();
  out_key = k;
  out_idx = i;
}

// Stage elements [e0, e0 + len) of one or two rows into shared memory; returns the number of
// elements brought by bulk copies (the rest is read from global memory).
template <typename E>
__device__ int32_t stage_slice(const uint8_t* trow, const uint8_t* drow, int64_t e0, int32_t len,
                               uint8_t* st_t, uint8_t* st_d, uint64_t* bar, int32_t* status,
                               bool* ok) {
  const uint32_t bulk_bytes = (uint32_t(len) * esize<E>()) & ~15u;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    mbar_expect_tx(bar, bulk_bytes * (drow ? 2u : 1u));
    if (bulk_bytes) {
      bulk_g2s(st_t, trow + e0 * esize<E>(), bulk_bytes, bar);
      if (drow) bulk_g2s(st_d, drow + e0 * esize<E>(), bulk_bytes, bar);
    }
  }
  __syncthreads();
  *ok = mbar_wait(bar, 0, status);
  return static_cast<int32_t>(bulk_bytes / esize<E>());
}

// ---------------------------------------------------------------------------------------------
// final: decisions and the correction / bonus race
// ---------------------------------------------------------------------------------------------
struct FinalParams {
  const uint8_t* target;
  const uint8_t* draft;
  int64_t V, ld;
  const int64_t* target_row0;
  const int64_t* draft_row0;
  const int32_t* draft_len;
  const int32_t* draft_tokens;
  int32_t B, gmax, S, block;
  uint64_t seed;
  const uint64_t* request_ids;
  int32_t* accepted_len;
  int32_t* out_tokens;
  int64_t out_ld;
  int32_t* correction_token;
  float* ratio_out;  // token: min(1, p/q); block: rho_i
  float* h_out;      // block: h_i
  VerifyWs ws;
  int32_t* status;
};

template <typename E>
__global__ void __launch_bounds__(kThreads) final_kernel(FinalParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bar;
  __shared__ float s_ratio[SV_MAX_DRAFT_LEN + 1];
  __shared__ float s_rho[SV_MAX_DRAFT_LEN + 1];
  __shared__ float s_h[SV_MAX_DRAFT_LEN + 1];
  __shared__ float s_R[SV_MAX_DRAFT_LEN + 1];
  __shared__ int32_t s_tau;
  __shared__ float s_gap;
  __shared__ float red_k[kWarps];
  __shared__ int32_t red_i[kWarps];
  __shared__ int32_t s_last;

  constexpr int32_t kSE = kSliceBytes / esize<E>();
  const int tid = threadIdx.x;
  const int32_t r = blockIdx.x / p.S;
  const int32_t s = blockIdx.x - r * p.S;
  const int32_t gamma = clamp_gamma(p.draft_len[r], p.gmax);
  const uint64_t req = p.request_ids ? p.request_ids[r] : uint64_t(r);

  for (int i = tid; i < gamma; i += kThreads) {
    const float4 ri = __ldcg(reinterpret_cast<const float4*>(&p.ws.rows[size_t(r) * p.gmax + i]));
    s_ratio[i + 1] = ri.z;
    s_rho[i + 1] = ri.w;
    if (p.block && i + 1 < gamma) s_R[i + 1] = __ldcg(&p.ws.rmass[size_t(r) * p.gmax + i + 1]);
  }
  __syncthreads();
  if (tid == 0) {
    int32_t tau;
    float lnw = 0.f;
    if (!p.block) {
      // walk left to right, stop at the first rejection
      tau = gamma;
      for (int i = 1; i <= gamma; ++i) {
        const float u = uniform_of(stream_block(make_stream(p.seed, req, i, kTagAccept), 0).x);
        if (!(u < s_ratio[i])) {
          tau = i - 1;
          break;
        }
      }
    } else {
      // thresholds h_i, then the longest passing prefix
      tau = 0;
      for (int i = 1; i <= gamma; ++i) {
        float h;
        if (i < gamma) {
          const float den = s_R[i] + (1.f - s_rho[i]);
          h = den > 0.f ? s_R[i] / den : 1.f;
        } else {
          h = s_rho[i];
        }
        s_h[i] = h;
        const float eta = uniform_of(stream_block(make_stream(p.seed, req, i, kTagAccept), 0).x);
        if (eta <= h) tau = i;
      }
      lnw = tau > 0 ? logf(s_rho[tau]) : 0.f;
    }
    s_tau = tau;
    if (tau < gamma) {
      const float4 ri =
          __ldcg(reinterpret_cast<const float4*>(&p.ws.rows[size_t(r) * p.gmax + tau]));
      s_gap = (ri.x - lnw) - ri.y;  // (c_t - log w) - c_d
    } else {
      s_gap = 0.f;
    }
  }
  __syncthreads();
  const int32_t tau = s_tau;

  if (s == 0) {  // per-position outputs
    for (int i = tid; i < gamma; i += kThreads) {
      const int64_t drow = p.draft_row0[r] + i;
      if (!p.block) {
        if (p.ratio_out) p.ratio_out[drow] = fminf(1.f, s_ratio[i + 1]);
      } else {
        if (p.ratio_out) p.ratio_out[drow] = s_rho[i + 1];
        if (p.h_out) p.h_out[drow] = s_h[i + 1];
      }
    }
  }

  // the race of this request's correction or bonus row, restricted to slice s
  RaceSpec rs;
  rs.resid = tau < gamma;
  rs.gap = s_gap;
  rs.st = make_stream(p.seed, req, tau + 1, rs.resid ? kTagResid : kTagBonus);
  const uint8_t* trow = row_ptr<E>(p.target, p.target_row0[r] + tau, p.ld);
  const uint8_t* drow = rs.resid ? row_ptr<E>(p.draft, p.draft_row0[r] + tau, p.ld) : nullptr;
  const int64_t e0 = int64_t(s) * kSE;
  const int32_t len = static_cast<int32_t>((p.V - e0 < int64_t(kSE) ? p.V - e0 : int64_t(kSE)));
  bool ok;
  const int32_t bulk = stage_slice<E>(trow, drow, e0, len, smem, smem + kSliceBytes, &bar,
                                      p.status, &ok);
  if (!ok) return;
  float key;
  int32_t idx;
  race_slice<E>(rs, smem, smem + kSliceBytes, trow, drow, e0, len, bulk, red_k, red_i, key, idx);
  if (tid == 0) {
    __stcg(&p.ws.race[size_t(r) * p.S + s], make_int2(__float_as_int(key), idx));
    __threadfence();
    s_last = atomicAdd(&p.ws.tick_f[r], 1) == p.S - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // last slice of the request: pick the winner over the slices
  if (tid == 0) {
    float bk = -INFINITY;
    int32_t bi = -1;
    for (int q = 0; q < p.S; ++q) {
      const int2 c = __ldcg(&p.ws.race[size_t(r) * p.S + q]);
      if (race_better(__int_as_float(c.x), c.y, bk, bi)) {
        bk = __int_as_float(c.x);
        bi = c.y;
      }
    }
    red_i[0] = bi;
  }
  __syncthreads();
  int32_t y = red_i[0];
  __syncthreads();
  if (y < 0 && rs.resid) {
    // residual empty to working precision (p and q agree): draw from p with the same uniforms
    RaceSpec fb = rs;
    fb.resid = false;
    race_row_global<E>(fb, trow, nullptr, p.V, red_k, red_i, key, y);
  }
  if (tid == 0) {
    if (y < 0) report(p.status, SV_ERR_BAD_INPUT);  // the row carries no probability at all
    p.accepted_len[r] = tau;
    if (p.correction_token) p.correction_token[r] = y;
    int32_t* out = p.out_tokens + size_t(r) * p.out_ld;
    for (int64_t q = 0; q < p.out_ld; ++q) {
      int32_t v = -1;
      if (q < tau) v = p.draft_tokens[p.draft_row0[r] + q];
      else if (q == tau) v = y;
      out[q] = v;
    }
  }
}

// ---------------------------------------------------------------------------------------------
// draft sampling from q
// ---------------------------------------------------------------------------------------------
struct SampleParams {
  const uint8_t* draft;
  int64_t V, ld;
  const int64_t* draft_row0;
  const int32_t* draft_len;
  int32_t B, gmax, S;
  uint64_t seed;
  const uint64_t* request_ids;
  int32_t* draft_tokens;
  VerifyWs ws;
  int32_t* status;
};

template <typename E>
__global__ void __launch_bounds__(kThreads) sample_kernel(SampleParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ uint64_t bar;
  __shared__ float red_k[kWarps];
  __shared__ int32_t red_i[kWarps];
  __shared__ int32_t s_last;
  constexpr int32_t kSE = kSliceBytes / esize<E>();
  const int32_t s = blockIdx.x % p.S;
  const int32_t unit = blockIdx.x / p.S;
  const int32_t r = unit / p.gmax;
  const int32_t i = unit - r * p.gmax + 1;
  const int32_t g = p.draft_len[r];
  if (g < 0 || g > p.gmax) {
    if (threadIdx.x == 0 && i == 1 && s == 0) report(p.status, SV_ERR_BAD_INPUT);
    return;
  }
  if (i > g) return;
  const uint64_t req = p.request_ids ? p.request_ids[r] : uint64_t(r);
  RaceSpec rs;
  rs.resid = false;
  rs.gap = 0.f;
  rs.st = make_stream(p.seed, req, i, kTagDraft);
  const int64_t row = p.draft_row0[r] + (i - 1);
  const uint8_t* drow = row_ptr<E>(p.draft, row, p.ld);
  const int64_t e0 = int64_t(s) * kSE;
  const int32_t len = static_cast<int32_t>((p.V - e0 < int64_t(kSE) ? p.V - e0 : int64_t(kSE)));
  bool ok;
  const int32_t bulk = stage_slice<E>(drow, nullptr, e0, len, smem, nullptr, &bar, p.status, &ok);
  if (!ok) return;
  float key;
  int32_t idx;
  race_slice<E>(rs, smem, nullptr, drow, nullptr, e0, len, bulk, red_k, red_i, key, idx);
  if (threadIdx.x == 0) {
    __stcg(&p.ws.race[size_t(unit) * p.S + s], make_int2(__float_as_int(key), idx));
    __threadfence();
    s_last = atomicAdd(&p.ws.tick_a[unit], 1) == p.S - 1;
  }
  __syncthreads();
  if (!s_last || threadIdx.x != 0) return;
  __threadfence();
  float bk = -INFINITY;
  int32_t bi = -1;
  for (int q = 0; q < p.S; ++q) {
    const int2 c = __ldcg(&p.ws.race[size_t(unit) * p.S + q]);
    if (race_better(__int_as_float(c.x), c.y, bk, bi)) {
      bk = __int_as_float(c.x);
      bi = c.y;
    }
  }
  if (bi < 0) report(p.status, SV_ERR_BAD_INPUT);
  p.draft_tokens[row] = bi;
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
static size_t sample_race_bytes(int32_t B, int32_t gmax, int32_t S) {
  return align256(sizeof(int2) * size_t(B > 0 ? B : 1) * size_t(gmax > 0 ? gmax : 1) * S);
}

static size_t verify_ws_bytes(int32_t B, int32_t gmax, int64_t V, int esz) {
  const int32_t S = slices_of(V, esz);
  const size_t a = verify_layout(nullptr, B, gmax, S).total;
  // the sampler reuses the layout with a race buffer of one entry per (row, slice)
  return a + sample_race_bytes(B, gmax, S);
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
static sv_status run_verify(bool block, const CommonArgs& a, const int64_t* target_row0,
                            const int64_t* draft_row0, const int32_t* draft_len,
                            const int32_t* draft_tokens, uint64_t seed,
                            const uint64_t* request_ids, int32_t* accepted_len,
                            int32_t* out_tokens, int64_t out_ld, int32_t* correction_token,
                            float* ratio_out, float* h_out, int32_t* status,
                            cudaStream_t stream) {
  const int32_t S = slices_of(a.V, esize<E>());
  const VerifyWs ws = verify_layout(a.ws, a.B, a.gmax, S);

  PlanParams pp{draft_len, a.B, a.gmax, ws, status};
  plan_kernel<<<1, 1024, 0, stream>>>(pp);

  StreamParams sp;
  sp.target = static_cast<const uint8_t*>(a.target);
  sp.draft = static_cast<const uint8_t*>(a.draft);
  sp.V = a.V;
  sp.ld = a.ld;
  sp.target_row0 = target_row0;
  sp.draft_row0 = draft_row0;
  sp.draft_len = draft_len;
  sp.draft_tokens = draft_tokens;
  sp.B = a.B;
  sp.gmax = a.gmax;
  sp.S = S;
  sp.block = block ? 1 : 0;
  sp.ws = ws;
  sp.status = status;
  const size_t stream_smem = 4 * kSliceBytes;
  const void* kfn = reinterpret_cast<const void*>(&stream_kernel<E>);
  if (cudaFuncSetAttribute(kfn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(stream_smem)) !=
      cudaSuccess)
    return SV_ERR_CUDA;
  const int resident = resident_ctas(kfn, kThreads, stream_smem);
  if (resident <= 0) return SV_ERR_CUDA;
  const int64_t persistent = int64_t(resident) * device_sm_count();
  if (a.gmax > 0) {
    const int64_t items = int64_t(a.B) * a.gmax * S;
    sp.resid_pass = 0;
    stream_kernel<E><<<unsigned(std::min<int64_t>(items, persistent)), kThreads, stream_smem,
                       stream>>>(sp);
    if (block && a.gmax > 1) {
      const int64_t ritems = int64_t(a.B) * (a.gmax - 1) * S;
      sp.resid_pass = 1;
      stream_kernel<E><<<unsigned(std::min<int64_t>(ritems, persistent)), kThreads, stream_smem,
                         stream>>>(sp);
    }
  }

  FinalParams fp;
  fp.target = sp.target;
  fp.draft = sp.draft;
  fp.V = a.V;
  fp.ld = a.ld;
  fp.target_row0 = target_row0;
  fp.draft_row0 = draft_row0;
  fp.draft_len = draft_len;
  fp.draft_tokens = draft_tokens;
  fp.B = a.B;
  fp.gmax = a.gmax;
  fp.S = S;
  fp.block = block ? 1 : 0;
  fp.seed = seed;
  fp.request_ids = request_ids;
  fp.accepted_len = accepted_len;
  fp.out_tokens = out_tokens;
  fp.out_ld = out_ld;
  fp.correction_token = correction_token;
  fp.ratio_out = ratio_out;
  fp.h_out = h_out;
  fp.ws = ws;
  fp.status = status;
  final_kernel<E><<<unsigned(int64_t(a.B) * S), kThreads, 2 * kSliceBytes, stream>>>(fp);
  return launch_status(cudaGetLastError());
}

template <typename E>
static sv_status run_sample(const CommonArgs& a, const int64_t* draft_row0,
                            const int32_t* draft_len, uint64_t seed, const uint64_t* request_ids,
                            int32_t* draft_tokens, int32_t* status, cudaStream_t stream) {
  const int32_t S = slices_of(a.V, esize<E>());
  VerifyWs ws = verify_layout(a.ws, a.B, a.gmax, S);
  // the race buffer of the sampler holds one entry per (draft row, slice)
  ws.race = reinterpret_cast<int2*>(static_cast<uint8_t*>(a.ws) + ws.total);
  const size_t units = size_t(a.B) * a.gmax;
  if (cudaMemsetAsync(ws.tick_a, 0, sizeof(int32_t) * units, stream) != cudaSuccess)
    return SV_ERR_CUDA;
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  SampleParams sp{static_cast<const uint8_t*>(a.draft), a.V, a.ld, draft_row0, draft_len,
                  a.B, a.gmax, S, seed, request_ids, draft_tokens, ws, status};
  sample_kernel<E><<<unsigned(units * S), kThreads, kSliceBytes, stream>>>(sp);
  return launch_status(cudaGetLastError());
}

}  // namespace sv

using namespace sv;

extern "C" size_t spec_verify_workspace_bytes(int32_t B, int32_t max_draft_len, int64_t V,
                                              sv_dtype dtype) {
  if (B < 0 || max_draft_len < 0 || max_draft_len > SV_MAX_DRAFT_LEN || V <= 0) return 0;
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

// Device address of g_noalloc_scratch on the current device.  In host code the array's name is a
// host-side stand-in, not a device address, so the address is looked up once per device (with
// that device current) and cached.
static sv_status noalloc_scratch_address(void** out) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static void* addr[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return SV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return SV_ERR_CUDA;
    addr[dev] = p;
  }
  *out = addr[dev];
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
  // The plan kernel clears every counter of the scratch before the other kernels use it.
  return spec_verify_token(target_logits, draft_logits, dtype, V, ld, target_row0, draft_row0,
                           draft_len, max_draft_len, draft_tokens, B, seed, request_ids,
                           accepted_len, out_tokens, out_ld, correction_token, accept_ratio,
                           status, scratch, sv::kNoAllocScratchBytes, stream);
}
