// schedule.cu -- DSpark's hardware-aware prefix scheduler in one CTA.
//
//   1. survival products S[i][k] = c[i][1] * ... * c[i][k] (sequential binary32, one thread per
//      request) and one 64-bit key per extendable prefix (i, k):
//        key = (~bits(S) << 32) | (k << 20) | i
//      ascending keys order prefixes by S descending, then k ascending, then i ascending (S >= 0,
//      whose bit patterns are monotone in the value); unused slots get the all-ones key;
//   2. bitonic sort of the keys in shared memory;
//   3. F = floor(S * 2^40) in sorted order and an inclusive int64 prefix scan: T(b) = N * 2^40 +
//      (sum of the first b values of F), exact and independent of the summation order;
//   4. f(b) = (double) T(b) * 2^-40 * sps[N + b]; the admitted count b* is the first b with
//      f(b + 1) <= f(b) (early stop; a min-reduction over b), capped by the item count and by B_max;
//   5. sel_len[i] = admitted prefixes of request i (prefix-closed by the ordering).
#include <cstdint>

#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

constexpr int kSchedThreads = 1024;
constexpr int kSchedMaxItems = 16384;

struct ScheduleParams {
  const float* c;
  const int32_t* max_len;
  int32_t N, K;
  const double* sps;
  int32_t B_max;
  int32_t n_pad;  // power of two >= N * K
  int32_t* sel_len;
  float* survival;
  int32_t* total_rows;
  double* objective;
  int32_t* status;
};

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(ScheduleParams p) {
  extern __shared__ __align__(16) uint64_t keys[];  // [n_pad]
  __shared__ long long warp_tot[kSchedThreads / 32];
  __shared__ int32_t s_bstar;
  __shared__ int32_t s_items;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    if (p.status) *p.status = SV_OK;
    s_bstar = 0x7FFFFFFF;
    s_items = 0;
  }
  for (int32_t i = tid; i < p.n_pad; i += kSchedThreads) keys[i] = ~0ull;
  for (int32_t i = tid; i < p.N; i += kSchedThreads) p.sel_len[i] = 0;
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
        const float c = p.c[size_t(i) * p.K + (k - 1)];
        if (!(c >= 0.0f && c <= 1.0f)) report(p.status, SV_ERR_BAD_INPUT);
        S = __fmul_rn(S, c);
        out = S;
        const uint32_t bits = S == 0.0f ? 0u : __float_as_uint(S);  // -0 ranks as +0
        keys[size_t(i) * p.K + (k - 1)] =
            (uint64_t(~bits) << 32) | (uint64_t(k) << 20) | uint64_t(i);
      }
      if (p.survival) p.survival[size_t(i) * p.K + (k - 1)] = out;
    }
    my_items += L;
  }
  atomicAdd(&s_items, my_items);
  __syncthreads();

  // 2. bitonic sort, ascending
  for (int32_t size = 2; size <= p.n_pad; size <<= 1) {
    for (int32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (int32_t t = tid; t < (p.n_pad >> 1); t += kSchedThreads) {
        const int32_t lo = 2 * t - (t & (stride - 1));
        const int32_t hi = lo + stride;
        const bool up = (lo & size) == 0;
        const uint64_t a = keys[lo], b = keys[hi];
        if ((a > b) == up) {
          keys[lo] = b;
          keys[hi] = a;
        }
      }
      __syncthreads();
    }
  }

  // 3. exact prefix sums of F in sorted order: each thread owns a contiguous run
  const int32_t n_items = s_items;
  const int32_t per = (p.n_pad + kSchedThreads - 1) / kSchedThreads;
  const int32_t b0 = tid * per;
  long long run = 0;
  for (int32_t j = 0; j < per; ++j) {
    const int32_t b = b0 + j;
    if (b < n_items) {
      const float S = __uint_as_float(~static_cast<uint32_t>(keys[b] >> 32));
      run += static_cast<long long>(floor(static_cast<double>(S) * 1099511627776.0));
    }
  }
  // exclusive scan of the per-thread totals
  long long incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < kSchedThreads / 32 ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += v;
    }
    if (lane < kSchedThreads / 32) warp_tot[lane] = w;
  }
  __syncthreads();
  const long long base = (static_cast<long long>(p.N) << 40) + (warp > 0 ? warp_tot[warp - 1] : 0) +
                         (incl - run);

  // 4. first non-increase of f(b) = T(b) 2^-40 sps[N + b], b < b_lim
  const int32_t b_lim = min(n_items, p.B_max - p.N);
  long long T = base;  // T(b0)
  int32_t first = 0x7FFFFFFF;
  for (int32_t j = 0; j < per; ++j) {
    const int32_t b = b0 + j;
    if (b >= b_lim) break;
    const float S = __uint_as_float(~static_cast<uint32_t>(keys[b] >> 32));
    const long long Tn = T + static_cast<long long>(floor(static_cast<double>(S) * 1099511627776.0));
    const double f = static_cast<double>(T) * 9.094947017729282379150390625e-13 * p.sps[p.N + b];
    const double fn =
        static_cast<double>(Tn) * 9.094947017729282379150390625e-13 * p.sps[p.N + b + 1];
    if (!(fn > f)) {
      first = b;
      break;
    }
    T = Tn;
  }
  if (first != 0x7FFFFFFF) atomicMin(&s_bstar, first);
  __syncthreads();
  const int32_t bstar = s_bstar == 0x7FFFFFFF ? max(b_lim, 0) : s_bstar;

  // 5. admitted prefixes per request
  for (int32_t b = tid; b < bstar; b += kSchedThreads)
    atomicAdd(&p.sel_len[static_cast<int32_t>(keys[b] & 0xFFFFFu)], 1);
  // T(b*): the thread owning rank b* - 1 (or b* for b* = 0) publishes it
  if (bstar == 0) {
    if (tid == 0) {
      *p.total_rows = p.N;
      *p.objective = static_cast<double>(static_cast<long long>(p.N) << 40) *
                     9.094947017729282379150390625e-13 * p.sps[p.N];
    }
  } else if (bstar - 1 >= b0 && bstar - 1 < b0 + per) {
    long long Tq = base;
    for (int32_t b = b0; b < bstar; ++b) {
      const float S = __uint_as_float(~static_cast<uint32_t>(keys[b] >> 32));
      Tq += static_cast<long long>(floor(static_cast<double>(S) * 1099511627776.0));
    }
    *p.total_rows = p.N + bstar;
    *p.objective = static_cast<double>(Tq) * 9.094947017729282379150390625e-13 * p.sps[p.N + bstar];
  }
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
  int32_t n_pad = 2;
  while (n_pad < N * K) n_pad <<= 1;
  const size_t smem = sizeof(uint64_t) * size_t(n_pad);
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(&schedule_kernel),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return SV_ERR_CUDA;
  ScheduleParams p{cond_accept, max_len, N, K, sps, B_max, n_pad, sel_len, survival, total_rows,
                   objective, status};
  schedule_kernel<<<1, kSchedThreads, smem, static_cast<cudaStream_t>(stream)>>>(p);
  return launch_status(cudaGetLastError());
}
