// schedule.cu -- DSpark's hardware-aware prefix scheduler: three kernels on the caller's stream.
//
//   chunk  (one CTA per 32 requests)  one thread per request forms the survival products
//          S[i][k] = c[i][1] * ... * c[i][k] (sequential binary32) and one 64-bit key per
//          extendable prefix (i, k):
//            key = (~bits(S) << 32) | (k << 20) | i
//          ascending keys order prefixes by S descending, then k ascending, then i ascending (S >= 0,
//          whose bit patterns are monotone in the value).  S never grows with k, so each request's
//          keys form an ascending run; the CTA merges its runs pairwise in shared memory into one
//          sorted chunk.
//   rank   (every SM, a programmatic dependent of chunk)  each CTA stages the sorted chunks; the
//          rank of a key in the global order is its place in its own chunk plus one binary search
//          in every other chunk.  The rank places F = floor(S * 2^40) and the request in sorted
//          order.
//   admit  (one CTA, a programmatic dependent of rank)  an exclusive int64 scan of F in sorted
//          order gives T(b) = N * 2^40 + (sum of the first b values of F), exact and independent of
//          the summation order; f(b) = (double) T(b) * 2^-40 * sps[N + b]; the admitted count b* is
//          the first b with f(b + 1) <= f(b) (early stop; a min-reduction over b), or the smallest b
//          of largest f(b) (best budget), capped by the item count and by B_max; sel_len[i] counts
//          the prefixes of request i ranked below b* (prefix-closed by the ordering).
// The fixed-depth rule needs no ranking (depth kernel), and the per-position acceptance update is a
// kernel of its own.
#include <algorithm>
#include <cstdint>

#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

constexpr int kChunkThreads = 512;
constexpr int kChunkSlots = 512;  // keys per chunk (at least one request's K)
constexpr int kRankThreads = 512;
constexpr int kSchedThreads = 1024;
constexpr int kSchedWarps = kSchedThreads / 32;
constexpr int kSchedMaxItems = 16384;
constexpr double kTwo40 = 1099511627776.0;                   // 2^40
constexpr double kTwoM40 = 9.094947017729282379150390625e-13;  // 2^-40

struct ScheduleParams {
  const float* c;
  const int32_t* max_len;
  int32_t N, K;
  const double* sps;
  int32_t B_max;
  int32_t* sel_len;
  float* survival;
  int32_t* total_rows;
  double* objective;
  int32_t* status;
  int32_t rule;           // SV_STOP_FIRST_DROP or SV_STOP_ARGMAX
  int32_t R;              // requests per chunk
  int32_t CL;             // keys per chunk (R * K)
  int32_t n_chunks;       // ceil(N / R)
  uint64_t* chunk_keys;   // workspace [n_chunks][CL]: each chunk's keys, sorted
  long long* sorted_F;    // workspace [N * K]: F of the prefix of rank b, at b
  int32_t* sorted_req;    // workspace [N * K]: the request of the prefix of rank b, at b
  unsigned long long* depth_F;  // workspace [K] (fixed-depth rule): sum of F at depth k + 1
  unsigned long long* depth_n;  // workspace [K] (fixed-depth rule): requests reaching depth k + 1
};

static inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__device__ __forceinline__ long long fixed40(uint64_t key) {
  const float S = __uint_as_float(~static_cast<uint32_t>(key >> 32));
  return static_cast<long long>(floor(static_cast<double>(S) * kTwo40));
}

// binary32 estimates for the screen of the admission test, by bit manipulation (no binary64
// arithmetic): the mantissa is truncated, so the relative error is below 2^-23.
// x >= 0 (binary64): -1 when x lies outside the normal binary32 range (the screen then defers to
// binary64).
__device__ __forceinline__ float approx_f32(double x) {
  const unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(x));
  if (u == 0ull) return 0.f;
  const int e = int(u >> 52) - 1023;
  if ((u >> 63) || e < -126 || e > 127) return -1.f;
  return __uint_as_float((uint32_t(e + 127) << 23) | (uint32_t(u >> 29) & 0x7FFFFFu));
}

// T * 2^-40 for 0 <= T < 2^63 (T * 2^-40 then lies in the normal binary32 range, or is 0).
__device__ __forceinline__ float approx_f32_scaled40(long long T) {
  if (T <= 0) return 0.f;
  const int lz = __clzll(T);
  const unsigned long long norm = static_cast<unsigned long long>(T) << lz;  // leading bit at 63
  const int e = 63 - lz - 40;
  return __uint_as_float((uint32_t(e + 127) << 23) | (uint32_t(norm >> 40) & 0x7FFFFFu));
}

__device__ __forceinline__ int32_t clamp_len(const ScheduleParams& p, int32_t i) {
  const int32_t L = p.max_len ? p.max_len[i] : p.K;
  return (L < 0 || L > p.K) ? 0 : L;
}

// Number of entries of the ascending array a[0, n) below key (strict) or, with `upper`, not above
// it: a branch-free lower / upper bound.
__device__ __forceinline__ int32_t count_below(const uint64_t* a, int32_t n, uint64_t key,
                                               bool upper) {
  int32_t pos = 0;
  int32_t step = 1;
  while (step * 2 <= n) step *= 2;
  for (; step >= 1; step >>= 1)
    if (pos + step <= n) {
      const uint64_t v = a[pos + step - 1];
      if (v < key || (upper && v == key)) pos += step;
    }
  return pos;
}

// chunk: CTA c forms the keys of requests [c R, c R + R) -- one ascending run of K keys each, all
// ones past max_len -- and sorts them by merging the runs pairwise in shared memory (each key's
// place in the merged pair is its place in its own run plus its count in the partner run).
__global__ void __launch_bounds__(kChunkThreads) schedule_chunk_kernel(ScheduleParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t* buf[2] = {reinterpret_cast<uint64_t*>(smem),
                      reinterpret_cast<uint64_t*>(smem) + p.CL};
  const int tid = threadIdx.x;
  // the rank kernel may launch now (it waits for this grid's results itself)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // survival products and keys, one thread per request (its probabilities are read sixteen at a
  // time, ahead of the sequential products)
  for (int32_t t = tid; t < p.R; t += kChunkThreads) {
    const int32_t i = blockIdx.x * p.R + t;
    uint64_t* run = buf[0] + t * p.K;
    if (i >= p.N) {
      for (int32_t k = 0; k < p.K; ++k) run[k] = ~0ull;
      continue;
    }
    int32_t L = p.max_len ? p.max_len[i] : p.K;
    if (L < 0 || L > p.K) {
      report(p.status, SV_ERR_BAD_INPUT);
      L = 0;
    }
    const float* ci = p.c + size_t(i) * p.K;
    float S = 1.0f;
    for (int32_t k0 = 0; k0 < p.K; k0 += 16) {
      float cv[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) cv[u] = k0 + u < L ? __ldg(ci + k0 + u) : 0.0f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int32_t k = k0 + u + 1;
        if (k > p.K) break;
        float out = 0.0f;
        uint64_t key = ~0ull;
        if (k <= L) {
          const float c = cv[u];
          if (!(c >= 0.0f && c <= 1.0f)) report(p.status, SV_ERR_BAD_INPUT);
          S = __fmul_rn(S, c);
          out = S;
          const uint32_t bits = S == 0.0f ? 0u : __float_as_uint(S);  // -0 ranks as +0
          key = (uint64_t(~bits) << 32) | (uint64_t(k) << 20) | uint64_t(i);
        }
        run[k - 1] = key;
        if (p.survival) p.survival[size_t(i) * p.K + (k - 1)] = out;
        if (p.rule == SV_STOP_FIXED_DEPTH && k <= L) {  // exact integer sums per depth
          atomicAdd(&p.depth_F[k - 1], static_cast<unsigned long long>(fixed40(key)));
          atomicAdd(&p.depth_n[k - 1], 1ull);
        }
      }
    }
  }
  __syncthreads();

  // merge runs of length w pairwise until one run remains; all-ones keys are equal, so a key of a
  // left run counts the partner's keys below it and a key of a right run those not above it
  int src = 0;
  for (int32_t w = p.K; w < p.CL; w *= 2) {
    const uint64_t* in = buf[src];
    uint64_t* out = buf[src ^ 1];
    for (int32_t e = tid; e < p.CL; e += kChunkThreads) {
      const int32_t q = e / w;
      const int32_t pq = q ^ 1;
      const uint64_t key = in[e];
      const int32_t lo = min(q, pq) * w;
      const int32_t p0 = pq * w;
      const int32_t pn = min(p0 + w, p.CL) - p0;  // partner length (<= 0: no partner)
      const int32_t own = e - q * w;
      out[pn > 0 ? lo + own + count_below(in + p0, pn, key, (q & 1) != 0) : e] = key;
    }
    __syncthreads();
    src ^= 1;
  }
  uint64_t* dst = p.chunk_keys + size_t(blockIdx.x) * p.CL;
  for (int32_t e = tid; e < p.CL; e += kChunkThreads) dst[e] = buf[src][e];
}

// rank: every CTA stages all sorted chunks; the rank of a key is its place in its own chunk plus
// its count in each other chunk (groups of G lanes split the chunks of one key), and the rank
// places F = floor(S * 2^40) and the request in sorted order.
__global__ void __launch_bounds__(kRankThreads) schedule_rank_kernel(ScheduleParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t* keys = reinterpret_cast<uint64_t*>(smem);  // [n_chunks][CL]
  const int tid = threadIdx.x, lane = tid & 31;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the chunk kernel's results
  const int32_t total = p.n_chunks * p.CL;
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.chunk_keys);
    uint4* dst = reinterpret_cast<uint4*>(keys);
    for (int32_t v = tid; v < total / 2; v += kRankThreads) dst[v] = __ldcg(src + v);
    if ((total & 1) && tid == 0) keys[total - 1] = __ldcg(p.chunk_keys + total - 1);
  }
  __syncthreads();
  int32_t G = 1;  // lanes per key: a power of two, at most 32
  while (G < p.n_chunks && G < 32) G *= 2;
  const int32_t gl = lane & (G - 1);          // this lane within its group
  const int32_t groups = kRankThreads / G;    // keys in flight per CTA
  const int32_t per = (total + gridDim.x - 1) / gridDim.x;
  const int32_t e0 = blockIdx.x * per, e1 = min(total, e0 + per);
  for (int32_t base = e0; base < e1; base += groups) {
    const int32_t e = base + tid / G;
    const bool live = e < e1;
    const uint64_t key = live ? keys[e] : ~0ull;
    const int32_t own = e / p.CL;
    int32_t cnt = 0;
    if (key != ~0ull) {
      for (int32_t c = gl; c < p.n_chunks; c += G)
        cnt += c == own ? e - own * p.CL : count_below(keys + c * p.CL, p.CL, key, false);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      if (o < G) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    if (key != ~0ull && gl == 0) {
      p.sorted_F[cnt] = fixed40(key);
      p.sorted_req[cnt] = static_cast<int32_t>(key & 0xFFFFFu);
    }
  }
}

template <int KPT>
__global__ void __launch_bounds__(kSchedThreads) schedule_admit_kernel(ScheduleParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  int32_t* counts = reinterpret_cast<int32_t*>(smem);  // [N] admitted prefixes per request
  __shared__ long long warp_tot[kSchedWarps];
  __shared__ int32_t s_bstar;
  __shared__ int32_t s_items;
  __shared__ uint32_t s_fmax;            // argmax rule: largest binary32 estimate (bits)
  __shared__ unsigned long long s_fbest;  // argmax rule: largest exact f among candidates (bits)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    s_bstar = 0x7FFFFFFF;
    s_items = 0;
    s_fmax = 0u;
    s_fbest = 0ull;
  }
  for (int32_t i = tid; i < p.N; i += kSchedThreads) counts[i] = 0;
  __syncthreads();
  // inputs first (they do not depend on the rank kernel): the item count and this thread's SPS
  int32_t my_items = 0;
  for (int32_t i = tid; i < p.N; i += kSchedThreads) my_items += clamp_len(p, i);
  atomicAdd(&s_items, my_items);
  const int32_t b0 = tid * KPT;  // this thread owns ranks [b0, b0 + KPT)
  double sp[KPT + 1];
  const double* spb = p.sps + p.N + b0;
  if (KPT % 2 == 0 && p.N + b0 + KPT <= p.B_max &&
      (reinterpret_cast<uintptr_t>(spb) & 15u) == 0) {
#pragma unroll
    for (int j = 0; j + 1 < KPT; j += 2) {
      const double2 v = __ldg(reinterpret_cast<const double2*>(spb + j));
      sp[j] = v.x;
      sp[j + 1] = v.y;
    }
    sp[KPT] = __ldg(spb + KPT);
  } else {
#pragma unroll
    for (int j = 0; j <= KPT; ++j) sp[j] = p.N + b0 + j <= p.B_max ? p.sps[p.N + b0 + j] : 0.0;
  }
  __syncthreads();
  const int32_t n_items = s_items;
  // the rank kernel's results
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // exact prefix sums of F in sorted order
  long long F[KPT];
  int32_t req[KPT];
  long long run = 0;
  if (KPT % 2 == 0 && b0 + KPT <= n_items) {  // whole run: 16-byte loads (b0 a multiple of KPT)
#pragma unroll
    for (int j = 0; j + 1 < KPT; j += 2) {
      const longlong2 v = __ldcg(reinterpret_cast<const longlong2*>(p.sorted_F + b0 + j));
      F[j] = v.x;
      F[j + 1] = v.y;
    }
#pragma unroll
    for (int j = 0; j < KPT; ++j) req[j] = __ldcg(p.sorted_req + b0 + j);
  } else {
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const bool in = b0 + j < n_items;
      F[j] = in ? __ldcg(p.sorted_F + b0 + j) : 0;
      req[j] = in ? __ldcg(p.sorted_req + b0 + j) : -1;
    }
  }
#pragma unroll
  for (int j = 0; j < KPT; ++j) run += F[j];
  long long incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    long long w = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long t = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += t;
    }
    warp_tot[lane] = w;
  }
  __syncthreads();
  const long long base =
      (static_cast<long long>(p.N) << 40) + (warp > 0 ? warp_tot[warp - 1] : 0) + (incl - run);

  const int32_t b_lim = min(n_items, p.B_max - p.N);
  float spf[KPT + 1];
#pragma unroll
  for (int j = 0; j <= KPT; ++j) spf[j] = approx_f32(sp[j]);
  if (p.rule == SV_STOP_FIRST_DROP) {
    // first non-increase of f(b) = T(b) 2^-40 sps[N + b], b < b_lim.  A binary32 estimate of both
    // sides (relative error below 3e-7 each) settles every comparison whose sides differ by more
    // than 4e-6 relative; the rest are decided in binary64, exactly as defined.
    long long T = base;  // T(b0)
    float Tf = approx_f32_scaled40(T);
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const int32_t b = b0 + j;
      if (b < b_lim) {
        const long long Tn = T + F[j];
        const float Tnf = approx_f32_scaled40(Tn);
        const float ff = Tf * spf[j], fnf = Tnf * spf[j + 1];
        bool up;
        if (spf[j] >= 0.f && spf[j + 1] >= 0.f && fnf > ff * (1.0f + 4e-6f)) {
          up = true;
        } else if (spf[j] >= 0.f && spf[j + 1] >= 0.f && fnf < ff * (1.0f - 4e-6f)) {
          up = false;
        } else {
          const double f = static_cast<double>(T) * kTwoM40 * sp[j];
          const double fn = static_cast<double>(Tn) * kTwoM40 * sp[j + 1];
          up = fn > f;
        }
        if (!up) {
          atomicMin(&s_bstar, b);
          break;
        }
        T = Tn;
        Tf = Tnf;
      }
    }
  } else {
    // the largest f(b) over b = 0 .. b_lim, the smallest b among equals.  This thread owns the
    // budgets b0 + 1 .. b0 + KPT (and thread 0 also b = 0).  The binary32 estimates (relative
    // error below 3e-7) leave as candidates only budgets within 8e-6 of the largest estimate,
    // which always include the true maximum; the candidates compare in binary64.
    // budget b0 + j (j = 1 .. KPT) at index j, and b = 0 at index 0 on thread 0; an estimate of
    // -1 marks a budget out of range, `force` one whose SPS lies outside the binary32 range
    long long Tb[KPT + 1];
    float fe[KPT + 1];
    bool force[KPT + 1];
    Tb[0] = base;
    fe[0] = -1.f;
    force[0] = false;
    if (tid == 0) {
      force[0] = !(spf[0] >= 0.f);
      fe[0] = force[0] ? -1.f : approx_f32_scaled40(base) * spf[0];
    }
    long long T = base;
#pragma unroll
    for (int j = 1; j <= KPT; ++j) {
      T += F[j - 1];
      Tb[j] = T;
      const bool in = b0 + j <= b_lim;
      force[j] = in && !(spf[j] >= 0.f);
      fe[j] = in && !force[j] ? approx_f32_scaled40(T) * spf[j] : -1.f;
    }
    float m = -1.f;
#pragma unroll
    for (int j = 0; j <= KPT; ++j) m = fmaxf(m, fe[j]);
    m = warp_max(m);
    if (lane == 0 && m >= 0.f) atomicMax(&s_fmax, __float_as_uint(m));  // order-preserving for >= 0
    __syncthreads();
    const float cut = __uint_as_float(s_fmax) * (1.0f - 8e-6f);
    double fx[KPT + 1];
    bool cand[KPT + 1];
#pragma unroll
    for (int j = 0; j <= KPT; ++j) {
      cand[j] = force[j] || (fe[j] >= 0.f && fe[j] >= cut);
      fx[j] = cand[j] ? static_cast<double>(Tb[j]) * kTwoM40 * sp[j] : 0.0;
    }
#pragma unroll
    for (int j = 0; j <= KPT; ++j)  // f >= 0: the bit pattern orders as the value
      if (cand[j]) atomicMax(&s_fbest, static_cast<unsigned long long>(__double_as_longlong(fx[j])));
    __syncthreads();
    const double fbest = __longlong_as_double(static_cast<long long>(s_fbest));
#pragma unroll
    for (int j = 0; j <= KPT; ++j)
      if (cand[j] && fx[j] == fbest) {
        atomicMin(&s_bstar, j == 0 ? 0 : b0 + j);
        break;
      }
  }
  __syncthreads();
  const int32_t bstar = s_bstar == 0x7FFFFFFF ? max(b_lim, 0) : s_bstar;

  // admitted prefixes per request (a prefix of its run, by the ordering)
#pragma unroll
  for (int j = 0; j < KPT; ++j)
    if (b0 + j < bstar) atomicAdd(&counts[req[j]], 1);
  // T(b*): published by the thread owning rank b* - 1 (thread 0 for b* = 0)
  if (bstar == 0) {
    if (tid == 0) {
      *p.total_rows = p.N;
      *p.objective =
          static_cast<double>(static_cast<long long>(p.N) << 40) * kTwoM40 * p.sps[p.N];
    }
  } else if (bstar - 1 >= b0 && bstar - 1 < b0 + KPT) {
    long long Tq = base;
#pragma unroll
    for (int j = 0; j < KPT; ++j)
      if (b0 + j < bstar) Tq += F[j];
    *p.total_rows = p.N + bstar;
    *p.objective = static_cast<double>(Tq) * kTwoM40 * p.sps[p.N + bstar];
  }
  __syncthreads();
  for (int32_t i = tid; i < p.N; i += kSchedThreads) p.sel_len[i] = counts[i];
}

// The fixed-depth rule, one CTA: one depth k for every request (min(k, max_len) drafts each),
// deepened while f(k + 1) = T(k + 1) 2^-40 sps[B(k + 1)] exceeds f(k) and B(k + 1) <= B_max, from
// the chunk kernel's exact per-depth sums of F and request counts.
__global__ void __launch_bounds__(kSchedThreads) schedule_depth_kernel(ScheduleParams p) {
  __shared__ int32_t s_depth;
  const int tid = threadIdx.x;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the chunk kernel's sums
  if (tid == 0) {
    long long T = static_cast<long long>(p.N) << 40, B = p.N;
    double f = static_cast<double>(T) * kTwoM40 * p.sps[p.N];
    int32_t depth = 0;
    for (int32_t k = 1; k <= p.K; ++k) {
      const long long Tn = T + static_cast<long long>(__ldcg(p.depth_F + (k - 1)));
      const long long Bn = B + static_cast<long long>(__ldcg(p.depth_n + (k - 1)));
      if (Bn > p.B_max || Bn == B) break;
      const double fn = static_cast<double>(Tn) * kTwoM40 * p.sps[Bn];
      if (!(fn > f)) break;
      T = Tn;
      B = Bn;
      f = fn;
      depth = k;
    }
    *p.total_rows = static_cast<int32_t>(B);
    *p.objective = f;
    s_depth = depth;
  }
  __syncthreads();
  for (int32_t i = tid; i < p.N; i += kSchedThreads) p.sel_len[i] = min(s_depth, clamp_len(p, i));
}

// Launches `kernel` as a programmatic dependent of the previous kernel on `stream`.
template <typename... Args>
static cudaError_t launch_dependent(void (*kernel)(Args...), unsigned grid, int threads,
                                    size_t smem, cudaStream_t stream, Args... args) {
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

struct ChunkShape {
  int32_t R, CL, n_chunks;
};

static ChunkShape chunk_shape(int32_t N, int32_t K) {
  ChunkShape c;
  c.R = std::max(1, kChunkSlots / std::max(K, 1));
  c.CL = c.R * std::max(K, 1);
  c.n_chunks = std::max(1, (N + c.R - 1) / c.R);
  return c;
}

static size_t schedule_ws_bytes(int32_t N, int32_t K) {
  const ChunkShape c = chunk_shape(N, K);
  const size_t nk = size_t(std::max<int64_t>(int64_t(N) * K, 1));
  return align256(sizeof(uint64_t) * size_t(c.n_chunks) * size_t(c.CL)) +
         align256(sizeof(long long) * nk) + align256(sizeof(int32_t) * nk) +
         align256(2 * sizeof(unsigned long long) * size_t(std::max(K, 1)));
}

}  // namespace sv

using namespace sv;

extern "C" size_t dspark_schedule_workspace_bytes(int32_t N, int32_t K) {
  if (N < 0 || K < 0) return 0;
  return schedule_ws_bytes(N, K);
}

extern "C" sv_status dspark_schedule_rule(const float* cond_accept, const int32_t* max_len,
                                          int32_t N, int32_t K, const double* sps, int32_t B_max,
                                          int32_t rule, int32_t* sel_len, float* survival,
                                          int32_t* total_rows, double* objective, int32_t* status,
                                          void* workspace, size_t workspace_bytes, void* stream) {
  if (rule != SV_STOP_FIRST_DROP && rule != SV_STOP_ARGMAX && rule != SV_STOP_FIXED_DEPTH)
    return SV_ERR_INVALID;
  if (N < 0 || K < 0 || B_max < N) return SV_ERR_INVALID;
  if (!sel_len || !total_rows || !objective || !sps) return SV_ERR_INVALID;
  if (N > 0 && K > 0 && !cond_accept) return SV_ERR_INVALID;
  if (int64_t(N) * K > kSchedMaxItems || K >= 4096 || N >= (1 << 20)) return SV_ERR_UNSUPPORTED;
  if (!workspace || !aligned256(workspace) || workspace_bytes < schedule_ws_bytes(N, K))
    return SV_ERR_INVALID;
  const int32_t NK = N * K;
  const ChunkShape cs = chunk_shape(N, K);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const size_t keys_bytes = align256(sizeof(uint64_t) * size_t(cs.n_chunks) * size_t(cs.CL));
  const size_t f_bytes = align256(sizeof(long long) * size_t(NK > 0 ? NK : 1));
  ScheduleParams p;
  p.c = cond_accept;
  p.max_len = max_len;
  p.N = N;
  p.K = K;
  p.sps = sps;
  p.B_max = B_max;
  p.sel_len = sel_len;
  p.survival = survival;
  p.total_rows = total_rows;
  p.objective = objective;
  p.status = status;
  p.rule = rule;
  p.R = cs.R;
  p.CL = cs.CL;
  p.n_chunks = cs.n_chunks;
  p.chunk_keys = reinterpret_cast<uint64_t*>(ws);
  p.sorted_F = reinterpret_cast<long long*>(ws + keys_bytes);
  p.sorted_req = reinterpret_cast<int32_t*>(ws + keys_bytes + f_bytes);
  p.depth_F = reinterpret_cast<unsigned long long*>(
      ws + keys_bytes + f_bytes + align256(sizeof(int32_t) * size_t(NK > 0 ? NK : 1)));
  p.depth_n = p.depth_F + std::max(K, 1);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return SV_ERR_CUDA;
  const int sms = device_sm_count();
  const int smem_sm = device_smem_per_sm();
  if (sms <= 0 || smem_sm <= 0) return SV_ERR_CUDA;

  if (rule == SV_STOP_FIXED_DEPTH &&
      cudaMemsetAsync(p.depth_F, 0, 2 * sizeof(unsigned long long) * size_t(std::max(K, 1)), s) !=
          cudaSuccess)
    return SV_ERR_CUDA;
  profile_mark(0, s);
  // chunk: one CTA per chunk of R requests; double-buffered keys
  const size_t chunk_smem = 2 * sizeof(uint64_t) * size_t(cs.CL);
  cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(&schedule_chunk_kernel),
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       int(chunk_smem));
  if (e != cudaSuccess) return SV_ERR_CUDA;
  schedule_chunk_kernel<<<unsigned(cs.n_chunks), kChunkThreads, chunk_smem, s>>>(p);
  if (cudaGetLastError() != cudaSuccess) return SV_ERR_CUDA;
  if (rule == SV_STOP_FIXED_DEPTH) {  // no ranking: the depth kernel reads the per-depth sums
    profile_mark(1, s);
    profile_mark(2, s);
    e = launch_dependent(schedule_depth_kernel, 1, kSchedThreads, 0, s, p);
    profile_mark(3, s);
    return launch_status(e);
  }
  // rank: every SM (as many CTAs as fit), each staging all chunks
  const size_t rank_smem = sizeof(uint64_t) * size_t(cs.n_chunks) * size_t(cs.CL);
  const int per_sm = std::max(1, std::min(4, smem_sm / int(rank_smem + 2048)));
  const int64_t total = int64_t(cs.n_chunks) * cs.CL;
  const unsigned rank_grid = unsigned(std::max<int64_t>(
      1, std::min<int64_t>(int64_t(sms) * per_sm, (total + 63) / 64)));
  e = launch_dependent(schedule_rank_kernel, rank_grid, kRankThreads, rank_smem, s, p);
  if (e != cudaSuccess) return SV_ERR_CUDA;
  profile_mark(1, s);
  profile_mark(2, s);
  // admit: one CTA
  int32_t n_pad = kSchedThreads;
  while (n_pad < NK) n_pad <<= 1;
  const size_t admit_smem = std::max<size_t>(sizeof(int32_t) * size_t(N), 16);
  switch (n_pad / kSchedThreads) {
    case 1: e = launch_dependent(schedule_admit_kernel<1>, 1, kSchedThreads, admit_smem, s, p); break;
    case 2: e = launch_dependent(schedule_admit_kernel<2>, 1, kSchedThreads, admit_smem, s, p); break;
    case 4: e = launch_dependent(schedule_admit_kernel<4>, 1, kSchedThreads, admit_smem, s, p); break;
    case 8: e = launch_dependent(schedule_admit_kernel<8>, 1, kSchedThreads, admit_smem, s, p); break;
    default: e = launch_dependent(schedule_admit_kernel<16>, 1, kSchedThreads, admit_smem, s, p); break;
  }
  profile_mark(3, s);
  return launch_status(e);
}

extern "C" sv_status dspark_schedule(const float* cond_accept, const int32_t* max_len, int32_t N,
                                     int32_t K, const double* sps, int32_t B_max,
                                     int32_t* sel_len, float* survival, int32_t* total_rows,
                                     double* objective, int32_t* status, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  return dspark_schedule_rule(cond_accept, max_len, N, K, sps, B_max, SV_STOP_FIRST_DROP, sel_len,
                              survival, total_rows, objective, status, workspace,
                              workspace_bytes, stream);
}

// ---------------------------------------------------------------------------------------------
// dspark_schedule_async: round t scheduled with the confidences of round t - 2
// ---------------------------------------------------------------------------------------------
extern "C" sv_status dspark_schedule_async(const float* conf_ring, int32_t depth, int64_t round,
                                           const float* cond_prior, const int32_t* max_len,
                                           int32_t N, int32_t K, const double* sps,
                                           int32_t B_max, int32_t rule, int32_t* sel_len,
                                           float* survival, int32_t* total_rows,
                                           double* objective, int32_t* status, void* workspace,
                                           size_t workspace_bytes, void* stream) {
  if (depth < 3 || round < 0) return SV_ERR_INVALID;
  if (N > 0 && K > 0 && (!conf_ring || !cond_prior)) return SV_ERR_INVALID;
  // slot (t - 2) % depth holds the predictions made two rounds before; slots t % depth and
  // (t - 1) % depth, which rounds t and t - 1 write, are never read
  const float* cond = cond_prior;
  if (round >= 2) cond = conf_ring + size_t((round - 2) % depth) * size_t(N) * size_t(K);
  return dspark_schedule_rule(cond, max_len, N, K, sps, B_max, rule, sel_len, survival,
                              total_rows, objective, status, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------------------------------------
// dspark_acceptance_update: per-position acceptance counts from one verified round
// ---------------------------------------------------------------------------------------------
namespace sv {

constexpr int kAcceptThreads = 1024;

struct AcceptParams {
  const int32_t* sel_len;
  const int32_t* accepted_len;
  int32_t N, K;
  double decay, prior_a, prior_b;
  double* trials;
  double* accepts;
  float* alpha;
  float* cond_out;
  int32_t* status;
};

// One CTA.  Position k was reached by request i iff k <= min(accepted + 1, verified) and accepted
// iff k <= accepted, so both counts are suffix sums of two histograms (of min(accepted + 1,
// verified) and of accepted) built with shared-memory atomics.  Then one thread per position
// updates its counts and estimate, with the same binary64 operations and order as the definition
// (no fused multiply-add), and the estimates are broadcast to every request's row of cond_out.
__global__ void __launch_bounds__(kAcceptThreads) acceptance_kernel(AcceptParams p) {
  extern __shared__ __align__(16) int32_t hist[];  // [2][K + 1], then alpha [K] as floats
  int32_t* h_last = hist;
  int32_t* h_acc = hist + (p.K + 1);
  float* al = reinterpret_cast<float*>(hist + 2 * (p.K + 1));
  const int tid = threadIdx.x;
  for (int32_t k = tid; k < 2 * (p.K + 1); k += kAcceptThreads) hist[k] = 0;
  __syncthreads();
  for (int32_t i = tid; i < p.N; i += kAcceptThreads) {
    const int32_t s = p.sel_len[i], a = p.accepted_len[i];
    if (s < 0 || s > p.K || a < 0 || a > s) {
      report(p.status, SV_ERR_BAD_INPUT);
      continue;
    }
    atomicAdd(&h_last[min(a + 1, s)], 1);
    atomicAdd(&h_acc[a], 1);
  }
  __syncthreads();
  for (int32_t k = tid + 1; k <= p.K; k += kAcceptThreads) {
    int32_t reached = 0, taken = 0;
    for (int32_t j = k; j <= p.K; ++j) {
      reached += h_last[j];
      taken += h_acc[j];
    }
    const double t = __dadd_rn(__dmul_rn(p.decay, p.trials[k - 1]), static_cast<double>(reached));
    const double c = __dadd_rn(__dmul_rn(p.decay, p.accepts[k - 1]), static_cast<double>(taken));
    p.trials[k - 1] = t;
    p.accepts[k - 1] = c;
    const float e = __double2float_rn(
        __ddiv_rn(__dadd_rn(c, p.prior_a), __dadd_rn(__dadd_rn(t, p.prior_a), p.prior_b)));
    p.alpha[k - 1] = e;
    al[k - 1] = e;
  }
  if (!p.cond_out) return;
  __syncthreads();
  const int64_t NK = int64_t(p.N) * p.K;
  for (int64_t e = tid; e < NK; e += kAcceptThreads) p.cond_out[e] = al[e % p.K];
}

}  // namespace sv

extern "C" sv_status dspark_acceptance_update(const int32_t* sel_len,
                                              const int32_t* accepted_len, int32_t N, int32_t K,
                                              double decay, double prior_a, double prior_b,
                                              double* trials, double* accepts, float* alpha,
                                              float* cond_accept_out, int32_t* status,
                                              void* stream) {
  if (N < 0 || K <= 0 || K >= 4096) return K == 0 && N >= 0 ? SV_OK : SV_ERR_INVALID;
  if (!(decay >= 0.0 && decay <= 1.0) || !(prior_a > 0.0) || !(prior_b > 0.0))
    return SV_ERR_INVALID;
  if (!trials || !accepts || !alpha || (N > 0 && (!sel_len || !accepted_len)))
    return SV_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return SV_ERR_CUDA;
  AcceptParams p{sel_len, accepted_len, N, K, decay, prior_a, prior_b, trials, accepts, alpha,
                 cond_accept_out, status};
  const size_t smem = sizeof(int32_t) * size_t(2 * (K + 1)) + sizeof(float) * size_t(K);
  acceptance_kernel<<<1, kAcceptThreads, smem, s>>>(p);
  return launch_status(cudaGetLastError());
}
