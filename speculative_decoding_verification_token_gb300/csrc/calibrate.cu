// calibrate.cu -- sequential temperature scaling of the confidence head: one temperature per draft
// position, fitted to verified outcomes, and the expected calibration error before and after.
//
// One CTA per position k.  Its samples are the requests that reached k (every earlier drafted
// token accepted, k verified: k <= min(accepted + 1, verified)); the label says whether k was
// accepted (k <= accepted).  Newton's method on the negative log-likelihood of sigma(beta s) in
// beta = 1 / T, from beta = 1, each step clamped to [beta_min, beta_max], stopping early once a step
// moves beta by less than 1e-9 of itself: every step sums
//   g = sum (sigma(beta s) - y) s   and   H = sum sigma(beta s) (1 - sigma(beta s)) s^2
// over the samples (logistic in binary32, from e^-|z| so that neither sigma nor 1 - sigma cancels;
// compensated binary32 sums per thread, then binary64 across the block).  The first 32768 samples
// of the position are staged in shared memory once, for every step and both error passes.  The
// expected calibration error bins the confidences into equal-width bins (per-warp binary32 bins,
// summed across warps in binary64) and sums |sum (y - sigma)| per bin over the sample count.
#include <algorithm>
#include <cstdint>

#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

constexpr int kStsThreads = 512;
constexpr int kStsWarps = kStsThreads / 32;
constexpr int kStsMaxBins = 256;
constexpr int32_t kStsStaged = 32768;  // samples of a position staged in shared memory

struct StsParams {
  const float* scores;  // [N][K]
  const int32_t* sel_len;
  const int32_t* accepted_len;
  int32_t N, K, iters;
  double beta_min, beta_max;
  int32_t nbins;
  float* T_out;         // [K]
  double* nll_out;      // [K] nullable
  double* ece_raw_out;  // [K] nullable
  double* ece_fit_out;  // [K] nullable
  int32_t* count_out;   // [K] nullable
  int32_t* status;
};

__device__ __forceinline__ float logistic_f(float x) { return 1.0f / (1.0f + expf(-x)); }

// sigma(z) and 1 - sigma(z), each without cancellation (from e^-|z|; the fast exponential and the
// rounded reciprocal keep both within a few units of the last place)
__device__ __forceinline__ void logistic_pair(float z, float& q, float& one_minus_q) {
  const float e = __expf(-fabsf(z));
  const float big = __frcp_rn(1.0f + e), small = e * big;
  q = z >= 0.0f ? big : small;
  one_minus_q = z >= 0.0f ? small : big;
}

// log(1 + e^x) without overflow
__device__ __forceinline__ float softplus_f(float x) {
  return x > 0.0f ? x + log1pf(expf(-x)) : log1pf(expf(x));
}

// Compensated (Kahan) binary32 accumulation: the running error of the sum is carried separately,
// so that thousands of terms keep close to binary32 accuracy relative to the total.
struct KahanF {
  float s = 0.0f, c = 0.0f;
  __device__ __forceinline__ void add(float v) {
    const float y = v - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
  }
  __device__ __forceinline__ double value() const {
    return static_cast<double>(s) - static_cast<double>(c);
  }
};

// Block-wide sum of two doubles; every thread receives them.
__device__ __forceinline__ void block_sum2(double& a, double& b, double (*red)[kStsWarps]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, o);
    b += __shfl_xor_sync(0xffffffffu, b, o);
  }
  if (lane == 0) {
    red[0][warp] = a;
    red[1][warp] = b;
  }
  __syncthreads();
  a = 0.0;
  b = 0.0;
#pragma unroll
  for (int w = 0; w < kStsWarps; ++w) {
    a += red[0][w];
    b += red[1][w];
  }
  __syncthreads();
}

// Sample i of position k: its score and label, or false when request i did not reach k (or its
// lengths are inconsistent).
__device__ __forceinline__ bool sts_sample(const StsParams& p, int32_t i, int32_t k, float& x,
                                           float& y) {
  const int32_t s = p.sel_len[i], a = p.accepted_len[i];
  if (s < 0 || s > p.K || a < 0 || a > s) return false;
  if (k > min(a + 1, s)) return false;
  x = p.scores[size_t(i) * p.K + (k - 1)];
  y = k <= a ? 1.0f : 0.0f;
  return true;
}

__global__ void __launch_bounds__(kStsThreads, 1) sts_kernel(StsParams p) {
  __shared__ double red[2][kStsWarps];
  __shared__ float wbins[kStsWarps][kStsMaxBins];  // per-warp bins (no contention across warps)
  const int32_t k = blockIdx.x + 1;
  const int tid = threadIdx.x;
  if (blockIdx.x == 0)
    for (int32_t i = tid; i < p.N; i += kStsThreads) {
      const int32_t s = p.sel_len[i], a = p.accepted_len[i];
      if (s < 0 || s > p.K || a < 0 || a > s) report(p.status, SV_ERR_BAD_INPUT);
    }
  // the position's first kStsStaged samples go to shared memory once: the score, and the label
  // (-1: request i did not reach position k)
  extern __shared__ __align__(16) uint8_t sts_smem[];
  const int32_t staged = min(p.N, kStsStaged);
  float* xs = reinterpret_cast<float*>(sts_smem);
  int8_t* ys = reinterpret_cast<int8_t*>(xs + staged);
  for (int32_t i = tid; i < staged; i += kStsThreads) {
    const int32_t sl = p.sel_len[i], a = p.accepted_len[i];
    const bool in = !(sl < 0 || sl > p.K || a < 0 || a > sl) && k <= min(a + 1, sl);
    xs[i] = in ? p.scores[size_t(i) * p.K + (k - 1)] : 0.0f;
    ys[i] = in ? int8_t(k <= a ? 1 : 0) : int8_t(-1);
  }
  __syncthreads();
  // Newton steps in beta = 1 / T
  double beta = 1.0;
  for (int32_t t = 0; t < p.iters; ++t) {
    KahanF gs, hs;
    const float bf = static_cast<float>(beta);
    auto term = [&](float x, bool y) {
      float q, q1;
      logistic_pair(bf * x, q, q1);
      const float r = y ? -q1 : q;  // sigma - y, accurate where sigma saturates
      gs.add(r * x);
      hs.add(q * q1 * x * x);
    };
    for (int32_t i = tid; i < staged; i += kStsThreads)
      if (ys[i] >= 0) term(xs[i], ys[i] > 0);
    for (int32_t i = staged + tid; i < p.N; i += kStsThreads) {
      float x, y;
      if (sts_sample(p, i, k, x, y)) term(x, y > 0.0f);
    }
    double g = gs.value(), H = hs.value();
    block_sum2(g, H, red);
    if (!(H > 0.0)) break;  // every thread sees the same sums
    const double nb = fmin(fmax(beta - g / H, p.beta_min), p.beta_max);
    const bool settled = fabs(nb - beta) <= 1e-9 * beta;  // converged (or pinned at a clamp)
    beta = nb;
    if (settled) break;
  }
  // the fitted loss, the sample count, and the calibration error before (beta = 1) and after
  double nll = 0.0, n = 0.0;
  for (int pass = 0; pass < 2; ++pass) {
    const float b = pass == 0 ? 1.0f : static_cast<float>(beta);
    for (int32_t j = tid; j < kStsWarps * p.nbins; j += kStsThreads)
      wbins[j / p.nbins][j % p.nbins] = 0.0f;
    __syncthreads();
    double loss = 0.0, cnt = 0.0;
    for (int32_t i = tid; i < p.N; i += kStsThreads) {
      float x, y;
      if (i < staged) {
        if (ys[i] < 0) continue;
        x = xs[i];
        y = float(ys[i]);
      } else if (!sts_sample(p, i, k, x, y)) {
        continue;
      }
      const float q = logistic_f(b * x);
      const int32_t bin = min(p.nbins - 1, max(0, static_cast<int32_t>(floorf(q * p.nbins))));
      atomicAdd(&wbins[tid >> 5][bin], y - q);
      if (pass == 1) loss += static_cast<double>(softplus_f(-(2.0f * y - 1.0f) * b * x));
      cnt += 1.0;
    }
    __syncthreads();
    double ece = 0.0;
    for (int32_t j = tid; j < p.nbins; j += kStsThreads) {
      double bsum = 0.0;
      for (int w = 0; w < kStsWarps; ++w) bsum += static_cast<double>(wbins[w][j]);
      ece += fabs(bsum);
    }
    block_sum2(ece, cnt, red);
    if (pass == 1) {
      double unused = 0.0;
      block_sum2(loss, unused, red);
      nll = loss;
    }
    n = cnt;
    if (tid == 0) {
      const double e = n > 0.0 ? ece / n : 0.0;
      if (pass == 0 && p.ece_raw_out) p.ece_raw_out[k - 1] = e;
      if (pass == 1 && p.ece_fit_out) p.ece_fit_out[k - 1] = e;
    }
  }
  if (tid == 0) {
    p.T_out[k - 1] = static_cast<float>(1.0 / beta);
    if (p.nll_out) p.nll_out[k - 1] = n > 0.0 ? nll / n : 0.0;
    if (p.count_out) p.count_out[k - 1] = static_cast<int32_t>(n);
  }
}

}  // namespace sv

using namespace sv;

extern "C" sv_status dspark_sts_fit(const float* scores, const int32_t* sel_len,
                                    const int32_t* accepted_len, int32_t N, int32_t K,
                                    int32_t iters, double beta_min, double beta_max,
                                    int32_t nbins, float* T_out, double* nll_out,
                                    double* ece_raw_out, double* ece_fit_out, int32_t* count_out,
                                    int32_t* status, void* stream) {
  if (N < 0 || K < 0 || iters < 0 || nbins <= 0 || nbins > kStsMaxBins) return SV_ERR_INVALID;
  if (!(beta_min > 0.0) || !(beta_max >= beta_min)) return SV_ERR_INVALID;
  if (!T_out || (N > 0 && (!scores || !sel_len || !accepted_len))) return SV_ERR_INVALID;
  if (K == 0) return SV_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return SV_ERR_CUDA;
  StsParams p{scores, sel_len, accepted_len, N, K, iters, beta_min, beta_max, nbins,
              T_out, nll_out, ece_raw_out, ece_fit_out, count_out, status};
  const size_t smem = size_t(std::min(N, kStsStaged)) * (sizeof(float) + 1) + 16;
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(&sts_kernel),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess)
    return SV_ERR_CUDA;
  sts_kernel<<<unsigned(K), kStsThreads, smem, s>>>(p);
  return launch_status(cudaGetLastError());
}
