// schedule.cu -- DSpark's hardware-aware prefix scheduler in one CTA.
//
//   1. the conditional acceptance probabilities are staged in shared memory (coalesced); survival
//      products S[i][k] = c[i][1] * ... * c[i][k] (sequential binary32, one thread per request)
//      and one 64-bit key per extendable prefix (i, k):
//        key = (~bits(S) << 32) | (k << 20) | i
//      ascending keys order prefixes by S descending, then k ascending, then i ascending (S >= 0,
//      whose bit patterns are monotone in the value); unused slots get the all-ones key;
//   2. bitonic sort of the keys, each thread holding a contiguous run of KPT keys in registers:
//      strides below KPT swap within a thread, strides below 32 KPT exchange through warp
//      shuffles, only the longer ones go through shared memory;
//   3. F = floor(S * 2^40) in sorted order (every thread sums its own run) and an exclusive int64
//      scan of the runs: T(b) = N * 2^40 + (sum of the first b values of F), exact and independent
//      of the summation order;
//   4. f(b) = (double) T(b) * 2^-40 * sps[N + b]; the admitted count b* is the first b with
//      f(b + 1) <= f(b) (early stop; a min-reduction over b), capped by the item count and by B_max;
//   5. sel_len[i] = admitted prefixes of request i (prefix-closed by the ordering), counted with
//      shared-memory atomics and written once.
#include <cstdint>

#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

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
  int32_t n_pad;  // 1024 * KPT >= N * K
  int32_t* sel_len;
  float* survival;
  int32_t* total_rows;
  double* objective;
  int32_t* status;
};

__device__ __forceinline__ long long fixed40(uint64_t key) {
  const float S = __uint_as_float(~static_cast<uint32_t>(key >> 32));
  return static_cast<long long>(floor(static_cast<double>(S) * kTwo40));
}

// Ascending bitonic sort of the n = kSchedThreads * KPT keys held as v[j] = element tid * KPT + j.
template <int KPT>
__device__ __forceinline__ void bitonic_sort(uint64_t (&v)[KPT], uint64_t* sm, int tid) {
  constexpr int n = kSchedThreads * KPT;
  for (int size = 2; size <= n; size <<= 1) {
    int stride = size >> 1;
    if (stride >= 32 * KPT) {
      // partners in other warps: through shared memory
#pragma unroll
      for (int j = 0; j < KPT; ++j) sm[tid * KPT + j] = v[j];
      __syncthreads();
      for (; stride >= 32 * KPT; stride >>= 1) {
        for (int t = tid; t < n / 2; t += kSchedThreads) {
          const int lo = 2 * t - (t & (stride - 1));
          const int hi = lo + stride;
          const bool up = (lo & size) == 0;
          const uint64_t a = sm[lo], b = sm[hi];
          if ((a > b) == up) {
            sm[lo] = b;
            sm[hi] = a;
          }
        }
        __syncthreads();
      }
#pragma unroll
      for (int j = 0; j < KPT; ++j) v[j] = sm[tid * KPT + j];
    }
    // partners in other lanes of this warp: element tid * KPT + j pairs with lane tid ^ (stride /
    // KPT), same j
    for (; stride >= KPT; stride >>= 1) {
      const int ts = stride / KPT;
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const uint64_t o = __shfl_xor_sync(0xffffffffu, v[j], ts);
        const int g = tid * KPT + j;
        const bool up = (g & size) == 0;
        const bool lower = (g & stride) == 0;
        v[j] = (lower == up) ? (v[j] < o ? v[j] : o) : (v[j] < o ? o : v[j]);
      }
    }
    // partners within this thread
#pragma unroll
    for (int s = KPT / 2; s >= 1; s /= 2) {
      if (s < size) {
#pragma unroll
        for (int j = 0; j < KPT; ++j) {
          if (j & s) continue;
          const bool up = ((tid * KPT + j) & size) == 0;
          const uint64_t a = v[j], b = v[j | s];
          if ((a > b) == up) {
            v[j] = b;
            v[j | s] = a;
          }
        }
      }
    }
  }
}

template <int KPT>
__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(ScheduleParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint64_t* keys = reinterpret_cast<uint64_t*>(smem);                       // [n_pad]
  float* cs = reinterpret_cast<float*>(smem + sizeof(uint64_t) * p.n_pad);  // [N * K], then
  int32_t* counts = reinterpret_cast<int32_t*>(cs);                          // [N] (reused)
  __shared__ long long warp_tot[kSchedWarps];
  __shared__ int32_t s_bstar;
  __shared__ int32_t s_items;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t NK = p.N * p.K;
  if (tid == 0) {
    if (p.status) *p.status = SV_OK;
    s_bstar = 0x7FFFFFFF;
    s_items = 0;
  }
  for (int32_t i = tid; i < p.n_pad; i += kSchedThreads) keys[i] = ~0ull;
  for (int32_t i = tid; i < NK; i += kSchedThreads) cs[i] = p.c[i];
  __syncthreads();

  // 1. survival products and keys
  int32_t my_items = 0;
  for (int32_t i = tid; i < p.N; i += kSchedThreads) {
    int32_t L = p.max_len ? p.max_len[i] : p.K;
    if (L < 0 || L > p.K) {
      report(p.status, SV_ERR_BAD_INPUT);
      L = 0;
    }
    float S = 1.0f;
    for (int32_t k = 1; k <= p.K; ++k) {
      float out = 0.0f;
      if (k <= L) {
        const float c = cs[i * p.K + (k - 1)];
        if (!(c >= 0.0f && c <= 1.0f)) report(p.status, SV_ERR_BAD_INPUT);
        S = __fmul_rn(S, c);
        out = S;
        const uint32_t bits = S == 0.0f ? 0u : __float_as_uint(S);  // -0 ranks as +0
        keys[i * p.K + (k - 1)] = (uint64_t(~bits) << 32) | (uint64_t(k) << 20) | uint64_t(i);
      }
      if (p.survival) p.survival[size_t(i) * p.K + (k - 1)] = out;
    }
    my_items += L;
  }
  atomicAdd(&s_items, my_items);
  __syncthreads();
  // per-request counts reuse the staged probabilities (N <= N * K whenever there are items)
  if (NK > 0)
    for (int32_t i = tid; i < p.N; i += kSchedThreads) counts[i] = 0;

  // 2. sort
  uint64_t v[KPT];
#pragma unroll
  for (int j = 0; j < KPT; ++j) v[j] = keys[tid * KPT + j];
  __syncthreads();
  bitonic_sort<KPT>(v, keys, tid);

  // 3. exact prefix sums of F in sorted order: this thread owns ranks [b0, b0 + KPT)
  const int32_t n_items = s_items;
  const int32_t b0 = tid * KPT;
  long long F[KPT];
  long long run = 0;
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    F[j] = b0 + j < n_items ? fixed40(v[j]) : 0;
    run += F[j];
  }
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

  // 4. first non-increase of f(b) = T(b) 2^-40 sps[N + b], b < b_lim
  const int32_t b_lim = min(n_items, p.B_max - p.N);
  double sp[KPT + 1];
#pragma unroll
  for (int j = 0; j <= KPT; ++j) sp[j] = b0 + j <= b_lim ? p.sps[p.N + b0 + j] : 0.0;
  long long T = base;  // T(b0)
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const int32_t b = b0 + j;
    if (b < b_lim) {
      const long long Tn = T + F[j];
      const double f = static_cast<double>(T) * kTwoM40 * sp[j];
      const double fn = static_cast<double>(Tn) * kTwoM40 * sp[j + 1];
      if (!(fn > f)) {
        atomicMin(&s_bstar, b);
        break;
      }
      T = Tn;
    }
  }
  __syncthreads();
  const int32_t bstar = s_bstar == 0x7FFFFFFF ? max(b_lim, 0) : s_bstar;

  // 5. admitted prefixes per request
#pragma unroll
  for (int j = 0; j < KPT; ++j)
    if (b0 + j < bstar) atomicAdd(&counts[static_cast<int32_t>(v[j] & 0xFFFFFu)], 1);
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
  for (int32_t i = tid; i < p.N; i += kSchedThreads) p.sel_len[i] = NK > 0 ? counts[i] : 0;
}

template <int KPT>
static cudaError_t launch_schedule(const ScheduleParams& p, size_t smem, cudaStream_t stream) {
  const void* fn = reinterpret_cast<const void*>(&schedule_kernel<KPT>);
  const cudaError_t e =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  schedule_kernel<KPT><<<1, kSchedThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace sv

using namespace sv;

extern "C" size_t dspark_schedule_workspace_bytes(int32_t N, int32_t K) {
  (void)N;
  (void)K;
  return 256;  // the scheduler works in shared memory
}

extern "C" sv_status dspark_schedule(const float* cond_accept, const int32_t* max_len, int32_t N,
                                     int32_t K, const double* sps, int32_t B_max,
                                     int32_t* sel_len, float* survival, int32_t* total_rows,
                                     double* objective, int32_t* status, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  (void)workspace;
  (void)workspace_bytes;
  if (N < 0 || K < 0 || B_max < N) return SV_ERR_INVALID;
  if (!sel_len || !total_rows || !objective || !sps) return SV_ERR_INVALID;
  if (N > 0 && K > 0 && !cond_accept) return SV_ERR_INVALID;
  if (int64_t(N) * K > kSchedMaxItems || K >= 4096 || N >= (1 << 20)) return SV_ERR_UNSUPPORTED;
  int32_t n_pad = kSchedThreads;
  while (n_pad < N * K) n_pad <<= 1;
  // keys, then the staged probabilities (reused for the per-request counts: N <= N * K whenever
  // there are items to admit)
  const size_t cs_bytes = sizeof(float) * size_t(int64_t(N) * K);
  const size_t smem = sizeof(uint64_t) * size_t(n_pad) + ((cs_bytes + 15) & ~size_t(15));
  ScheduleParams p{cond_accept, max_len, N, K, sps, B_max, n_pad, sel_len, survival, total_rows,
                   objective, status};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  switch (n_pad / kSchedThreads) {
    case 1: e = launch_schedule<1>(p, smem, s); break;
    case 2: e = launch_schedule<2>(p, smem, s); break;
    case 4: e = launch_schedule<4>(p, smem, s); break;
    case 8: e = launch_schedule<8>(p, smem, s); break;
    default: e = launch_schedule<16>(p, smem, s); break;
  }
  return launch_status(e);
}
