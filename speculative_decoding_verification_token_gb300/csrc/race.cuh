// race.cuh -- the exponential race over a row (or a row pair for residuals) split across the CTAs
// of a thread-block cluster.
//
// The key of entry x is log w(x) - log E_x (E_x = -log u_x); the largest key wins, equal keys go to
// the lower index.  Residual entries (weight max(w p(x) - q(x), 0)) are written, up to a per-row
// constant, t + log(1 - exp(y)) - log E with y = (d - t) + gap; plain entries (a row sampled
// from its own softmax) t - log E.  Either way key <= t + noise with noise = -log(-log u).
//
// Each CTA of the cluster owns one contiguous 1/CL of the row and reads it twice from global
// memory (the rows were just streamed, so mostly from L2):
//   seed  every thread keys its entry of largest logit; the cluster shares the best such key K0
//         through distributed shared memory -- a lower bound on the winning key;
//   main  an entry can reach K0 only if its logit is within kMaxNoise of K0 (no uniform needed to
//         reject the rest) and, given its uniform, only if its noise reaches K0 - t (the noise gate,
//         an integer compare on the Philox word); the few entries that pass both are keyed exactly.
#pragma once

#include "sv_device.cuh"

namespace sv {

template <typename E>
__host__ __device__ constexpr int esize() {
  return 16 / Elem<E>::kPerVec;
}

template <typename E>
__device__ __forceinline__ const uint8_t* row_ptr(const uint8_t* base, int64_t row, int64_t ld) {
  return base + row * ld * esize<E>();
}

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

// Exact key of vocabulary entry e (reads the entry again; used on the rare survivors only).
template <typename E>
__device__ __noinline__ float exact_key(const RaceSpec& rs, const uint8_t* trow,
                                        const uint8_t* drow, int64_t e) {
  const float t = Elem<E>::load(trow, e);
  const float d = rs.resid ? Elem<E>::load(drow, e) : 0.f;
  const uint4 b = stream_block(rs.st, static_cast<uint32_t>(e >> 2));
  return race_key(rs, t, d, race_noise(uniform_of(word_of(b, static_cast<uint32_t>(e & 3)))));
}

// Noise gate.  An entry whose logit is delta below K0 reaches K0 only if its noise
// -log(-log u) >= delta, i.e. u >= exp(-exp(-delta)).  gate[k] is that threshold for
// delta = k / 4 as a bound on the 23-bit numerator (w >> 9) of u, lowered by 4 to absorb the
// binary32 rounding of the threshold: an entry with delta >= k / 4 + 0.01 and (w >> 9) < gate[k]
// cannot win.  (The 0.01 margin covers the binary32 rounding of the key itself.)
constexpr int kGateBuckets = 68;  // quarter nats up to the kMaxNoise floor

__device__ __forceinline__ void build_gate(uint32_t* gate) {
  for (int k = threadIdx.x; k < kGateBuckets; k += blockDim.x) {
    const float thr = expf(-expf(-0.25f * float(k)));
    const float num = floorf(thr * 8388608.0f) - 4.0f;
    gate[k] = num < 0.f ? 0u : static_cast<uint32_t>(num);
  }
}

__device__ __forceinline__ bool gate_passes(const uint32_t* gate, float K0, float t, uint32_t w) {
  const float delta = K0 - t;
  if (!(delta > 0.01f)) return true;
  const int k = min(static_cast<int>((delta - 0.01f) * 4.0f), kGateBuckets - 1);
  return (w >> 9) >= gate[k];
}

template <typename E>
__device__ __forceinline__ uint4 load_vec(const uint8_t* row, int64_t first_elem) {
  return __ldg(reinterpret_cast<const uint4*>(row + first_elem * esize<E>()));
}

constexpr int kBatch = 2;  // vectors whose loads each thread issues before using any

// Seed pass over vocabulary range [e0, e0 + len): this thread's active entry of largest logit.
template <typename E>
__device__ __forceinline__ void seed_range(const RaceSpec& rs, const uint8_t* trow,
                                           const uint8_t* drow, int64_t e0, int32_t len,
                                           float& bt, int64_t& be) {
  constexpr int kPer = Elem<E>::kPerVec;
  const int nvec = len / kPer;
  for (int v0 = threadIdx.x; v0 < nvec; v0 += kThreads * kBatch) {
    uint4 a[kBatch], b[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int v = v0 + u * kThreads;
      if (v < nvec) {
        a[u] = load_vec<E>(trow, e0 + int64_t(v) * kPer);
        if (rs.resid) b[u] = load_vec<E>(drow, e0 + int64_t(v) * kPer);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int v = v0 + u * kThreads;
      if (v >= nvec) break;
      const int64_t e = e0 + int64_t(v) * kPer;
      float x[kPer], y[kPer];
      Elem<E>::unpack(a[u], x);
      if (rs.resid) Elem<E>::unpack(b[u], y);
#pragma unroll
      for (int q = 0; q < kPer; ++q) {
        const float dq = rs.resid ? y[q] : 0.f;
        if (x[q] > bt && race_active(rs, x[q], dq)) {
          bt = x[q];
          be = e + q;
        }
      }
    }
  }
  for (int i = nvec * kPer + threadIdx.x; i < len; i += kThreads) {
    const float x = Elem<E>::load(trow, e0 + i);
    const float d = rs.resid ? Elem<E>::load(drow, e0 + i) : 0.f;
    if (x > bt && race_active(rs, x, d)) {
      bt = x;
      be = e0 + i;
    }
  }
}

// Main pass over [e0, e0 + len): exact keys for the entries that pass the floor and the gate.
template <typename E>
__device__ __forceinline__ void race_range(const RaceSpec& rs, const uint8_t* trow,
                                           const uint8_t* drow, int64_t e0, int32_t len,
                                           float floor_t, float K0, const uint32_t* gate,
                                           float& bk, int32_t& bi) {
  constexpr int kPer = Elem<E>::kPerVec;
  const int nvec = len / kPer;
  for (int v0 = threadIdx.x; v0 < nvec; v0 += kThreads * kBatch) {
    uint4 a[kBatch], b[kBatch];
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
      const int v = v0 + u * kThreads;
      if (v < nvec) {
        a[u] = load_vec<E>(trow, e0 + int64_t(v) * kPer);
        if (rs.resid) b[u] = load_vec<E>(drow, e0 + int64_t(v) * kPer);
      }
    }
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
    const int v = v0 + u * kThreads;
    if (v >= nvec) break;
    const int64_t e = e0 + int64_t(v) * kPer;
    float x[kPer], y[kPer];
    Elem<E>::unpack(a[u], x);
    float xm = x[0];
#pragma unroll
    for (int q = 1; q < kPer; ++q) xm = fmaxf(xm, x[q]);
    if (!(xm >= floor_t)) continue;
    if (rs.resid) Elem<E>::unpack(b[u], y);
    // e is a multiple of kPer (>= 4): the vector's words are whole Philox blocks
    const uint4 b0 = stream_block(rs.st, static_cast<uint32_t>(e >> 2));
    const uint4 b1 = kPer == 8 ? stream_block(rs.st, static_cast<uint32_t>(e >> 2) + 1) : b0;
    const uint32_t w[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    uint32_t mask = 0;
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const float dq = rs.resid ? y[q] : 0.f;
      if (x[q] >= floor_t && race_active(rs, x[q], dq) && gate_passes(gate, K0, x[q], w[q]))
        mask |= 1u << q;
    }
    while (mask) {
      const int q = __ffs(mask) - 1;
      mask &= mask - 1;
      const float k = exact_key<E>(rs, trow, drow, e + q);
      if (race_better(k, int32_t(e + q), bk, bi)) {
        bk = k;
        bi = int32_t(e + q);
      }
    }
    }
  }
  for (int i = nvec * kPer + threadIdx.x; i < len; i += kThreads) {
    const int64_t e = e0 + i;
    const float x = Elem<E>::load(trow, e);
    const float d = rs.resid ? Elem<E>::load(drow, e) : 0.f;
    if (!(x >= floor_t && race_active(rs, x, d))) continue;
    const uint4 b = stream_block(rs.st, static_cast<uint32_t>(e >> 2));
    if (!gate_passes(gate, K0, x, word_of(b, static_cast<uint32_t>(e & 3)))) continue;
    const float k = exact_key<E>(rs, trow, drow, e);
    if (race_better(k, int32_t(e), bk, bi)) {
      bk = k;
      bi = int32_t(e);
    }
  }
}

// CTA-wide winner (every thread receives it).
__device__ __forceinline__ void block_race(float& key, int32_t& idx, float* red_k,
                                           int32_t* red_i) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_race(key, idx);
  if (lane == 0) {
    red_k[warp] = key;
    red_i[warp] = idx;
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
  key = k;
  idx = i;
}

__device__ __forceinline__ float block_max(float v, float* red_k) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  if (lane == 0) red_k[warp] = v;
  __syncthreads();
  float m = red_k[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) m = fmaxf(m, red_k[w]);
  __syncthreads();
  return m;
}

// Race over a whole row by one CTA (rare fallback path; no pruning).
template <typename E>
__device__ void race_row_global(const RaceSpec& rs, const uint8_t* trow, const uint8_t* drow,
                                int64_t V, float* red_k, int32_t* red_i, float& out_key,
                                int32_t& out_idx) {
  float bk = -INFINITY;
  int32_t bi = -1;
  for (int64_t e = threadIdx.x; e < V; e += kThreads) {
    const float x = Elem<E>::load(trow, e);
    const float d = rs.resid ? Elem<E>::load(drow, e) : 0.f;
    if (!race_active(rs, x, d)) continue;
    const float k = exact_key<E>(rs, trow, drow, e);
    if (race_better(k, int32_t(e), bk, bi)) {
      bk = k;
      bi = int32_t(e);
    }
  }
  block_race(bk, bi, red_k, red_i);
  out_key = bk;
  out_idx = bi;
}

// ---- thread-block clusters --------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Read a 32-bit word at the same shared-memory offset in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t dsmem_load_u32(const void* local, uint32_t rank) {
  uint32_t remote, v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)),
               "r"(rank));
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(remote) : "memory");
  return v;
}

}  // namespace sv
