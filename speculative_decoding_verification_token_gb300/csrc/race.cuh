// race.cuh -- the exponential race over a row (or a row pair for residuals) split across CTAs.
//
// The key of entry x is log w(x) - log E_x (E_x = -log u_x); the largest key wins, equal keys go to
// the lower index.  Residual entries (weight max(w p(x) - q(x), 0)) are written, up to a per-row
// constant, t + log(1 - exp(y)) - log E with y = (d - t) + gap; plain entries (a row sampled
// from its own softmax) t - log E.  Either way key <= t + noise with noise = -log(-log u).
//
// Each CTA owns one contiguous 1/CL of the row; its 16-byte vectors come from `vsrc` -- the share
// staged in shared memory by one bulk copy, or the row itself in global memory -- and are read
// twice:
//   seed  every thread keys its entry of largest logit; the best such key of the CTA, raised to
//         the best that the job's other shares have published, is a lower bound K0 on the winning
//         key;
//   main  an entry can reach K0 only if its logit is within kMaxNoise of K0 (no uniform needed to
//         reject the rest) and, given the 16 high bits of its uniform, only if its noise can reach
//         K0 - t (the noise gate, tested for a whole 16-byte vector at once on the largest coarse
//         half of its block); the entries of the few vectors that pass are gated one by one, and
//         those that pass draw their low bits and are keyed exactly.
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
  int64_t off = 0;  // vocabulary index of the row's first entry (a vocabulary shard's offset, a
                    // multiple of 8); the uniforms are keyed by the global index off + e
};

__device__ __forceinline__ float race_key(const RaceSpec& rs, float t, float d, float noise) {
  if (!rs.resid) return t + noise;
  const float y = (d - t) + rs.gap;
  return t + __logf(one_minus_exp(y)) + noise;
}

__device__ __forceinline__ bool race_active(const RaceSpec& rs, float t, float d) {
  return rs.resid ? ((d - t) + rs.gap < 0.f) : (t > -INFINITY);
}

// Exact key of vocabulary entry e with logit t and coarse half h, or -inf if the entry carries no
// weight (reads the draft logit of a residual entry; used on the rare survivors only).
template <typename E>
__device__ __noinline__ float exact_key_h(const RaceSpec& rs, float t, const uint8_t* drow,
                                          int64_t e, uint32_t h) {
  const float d = rs.resid ? Elem<E>::load(drow, e) : 0.f;
  if (!race_active(rs, t, d)) return -INFINITY;
  return race_key(rs, t, d, race_noise(race_uniform_at(rs.st, uint64_t(e + rs.off), h)));
}

// The same, drawing the coarse half too.
template <typename E>
__device__ __noinline__ float exact_key_t(const RaceSpec& rs, float t, const uint8_t* drow,
                                          int64_t e) {
  const uint64_t v = uint64_t(e + rs.off);
  const uint4 b = stream_block(rs.st, static_cast<uint32_t>(v >> 3));
  return exact_key_h<E>(rs, t, drow, e, half_of(b, static_cast<uint32_t>(v & 7)));
}

template <typename E>
__device__ __forceinline__ float exact_key(const RaceSpec& rs, const uint8_t* trow,
                                           const uint8_t* drow, int64_t e) {
  return exact_key_t<E>(rs, Elem<E>::load(trow, e), drow, e);
}

// A race result as one 64-bit word whose unsigned order is the race order: the key's bits made
// order-preserving in the high half, the complemented index in the low half (equal keys: the
// lower index is larger).  0 is below every packed result.
__device__ __forceinline__ unsigned long long race_pack(float key, int32_t idx) {
  const uint32_t u = __float_as_uint(key);
  const uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(o) << 32) | static_cast<uint32_t>(~idx);
}

__device__ __forceinline__ int32_t race_unpack_index(unsigned long long packed) {
  return static_cast<int32_t>(~static_cast<uint32_t>(packed));
}

// Order-preserving bits of a key (the high half of race_pack) and back; 0 decodes to -inf.
__device__ __forceinline__ uint32_t key_order(float key) {
  const uint32_t u = __float_as_uint(key);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_from_order(uint32_t o) {
  if (o == 0) return -INFINITY;
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// Largest element of one 16-byte vector of logits.
template <typename E>
__device__ __forceinline__ float vec_max(const uint4& v);

template <>
__device__ __forceinline__ float vec_max<bf16_tag>(const uint4& v) {
  __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&v.x),
                             *reinterpret_cast<const __nv_bfloat162*>(&v.y));
  const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&v.z),
                                   *reinterpret_cast<const __nv_bfloat162*>(&v.w));
  a = __hmax2(a, b);
  const uint32_t ab = *reinterpret_cast<const uint32_t*>(&a);
  return fmaxf(__uint_as_float(ab << 16), __uint_as_float(ab & 0xFFFF0000u));
}

template <>
__device__ __forceinline__ float vec_max<float>(const uint4& v) {
  return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
               fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
}

// Noise gate.  key <= t + G with G = -log(-log u) <= -log(1 - u), and 1 - u > m 2^-23 with
// m = 0x7FFFFF - n for the uniform's 23-bit numerator n.  So an entry reaches the bound K only if
// m <= 2^23 e^(t - K) = 2^(t log2e + c), c = 23 - K log2e.  The coarse half h bounds m from
// below by gate_mh(h) whatever the low bits, so a whole 8-entry vector can hold such an entry only
// if gate_mh of its block's largest half is within the threshold of its largest logit: one Philox
// block, three SIMD maxima and one ex2 per vector reject almost every vector.  The factor 1.001
// covers the binary32 rounding of the threshold and of the keys.
__device__ __forceinline__ float gate_threshold(float t, float c) {
  return fast_exp2(fmaf(t, kLog2e, c)) * 1.001f;
}

constexpr int kSeedBatch = 8;  // vectors whose loads each thread issues before using any (seed)
constexpr int kBatch = 2;      // the same for the main pass over a staged share
constexpr int kBatchGlobal = 4;  // ... and over a share read from global memory

// Seed pass over vocabulary range [e0, e0 + len): the exact key of this thread's entry of largest
// logit (-inf if that entry carries no weight) -- a lower bound on the range's winning key.
template <typename E>
__device__ __forceinline__ float seed_range(const RaceSpec& rs, const uint4* vsrc,
                                            const uint8_t* trow, const uint8_t* drow, int64_t e0,
                                            int32_t len) {
  constexpr int kPer = Elem<E>::kPerVec;
  const int nvec = len / kPer;
  float bt = -INFINITY;
  int64_t bv = -1;  // first element of the vector holding bt
  for (int v0 = threadIdx.x; v0 < nvec; v0 += kThreads * kSeedBatch) {
    uint4 a[kSeedBatch];
#pragma unroll
    for (int u = 0; u < kSeedBatch; ++u) {
      const int v = v0 + u * kThreads;
      if (v < nvec) a[u] = vsrc[v];
    }
#pragma unroll
    for (int u = 0; u < kSeedBatch; ++u) {
      const int v = v0 + u * kThreads;
      if (v >= nvec) break;
      const float m = vec_max<E>(a[u]);
      if (m > bt) {
        bt = m;
        bv = e0 + int64_t(v) * kPer;
      }
    }
  }
  int64_t be = -1;
  if (bv >= 0) {
    float x[8];
    Elem<E>::unpack(vsrc[(bv - e0) / kPer], x);
#pragma unroll
    for (int q = kPer - 1; q >= 0; --q)
      if (x[q] == bt) be = bv + q;
  }
  for (int i = nvec * kPer + threadIdx.x; i < len; i += kThreads) {
    const float x = Elem<E>::load(trow, e0 + i);
    if (x > bt) {
      bt = x;
      be = e0 + i;
    }
  }
  return be >= 0 ? exact_key_t<E>(rs, bt, drow, be) : -INFINITY;
}

// Offers entry e, with logit t and coarse half h, to the race if it passes the gate.
template <typename E>
__device__ __forceinline__ void offer(const RaceSpec& rs, const uint8_t* trow,
                                      const uint8_t* drow, int64_t e, float t, uint32_t h,
                                      float c, float& bk, int32_t& bi) {
  if (!(gate_mh(h) <= gate_threshold(t, c))) return;
  const float k = exact_key_h<E>(rs, t, drow, e, h);
  if (k > -INFINITY && race_better(k, int32_t(e), bk, bi)) {
    bk = k;
    bi = int32_t(e);
  }
}

// Main pass over [e0, e0 + len) against the lower bound K0: only the target row is read; the
// draft row is touched for the few entries keyed exactly.
template <typename E, int NB = kBatch>
__device__ __forceinline__ void race_range(const RaceSpec& rs, const uint4* vsrc,
                                           const uint8_t* trow, const uint8_t* drow, int64_t e0,
                                           int32_t len, float K0, float& bk, int32_t& bi) {
  constexpr int kPer = Elem<E>::kPerVec;
  const float floor_t = K0 - kMaxNoise;  // no noise lifts a logit below this to K0
  const float c = 23.0f - K0 * kLog2e;
  const int nvec = len / kPer;
  for (int v0 = threadIdx.x; v0 < nvec; v0 += kThreads * NB) {
    uint4 a[NB];
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int v = v0 + u * kThreads;
      if (v < nvec) a[u] = vsrc[v];
    }
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int v = v0 + u * kThreads;
      if (v >= nvec) break;
      const int64_t e = e0 + int64_t(v) * kPer;
      const float tmax = vec_max<E>(a[u]);
      if (!(tmax >= floor_t)) continue;
      // e + off is a multiple of kPer (8 or 4): the vector's halves are one coarse block (8) or
      // its first or second pair of words (4)
      const uint64_t g = uint64_t(e + rs.off);
      uint4 b = stream_block(rs.st, static_cast<uint32_t>(g >> 3));
      if (kPer == 4) {
        const bool upper = (g & 4) != 0;
        b = make_uint4(upper ? b.z : b.x, upper ? b.w : b.y, 0u, 0u);
      }
      if (gate_mh(half_max(b)) > gate_threshold(tmax, c)) continue;
      float x[8];
      Elem<E>::unpack(a[u], x);
#pragma unroll
      for (int q = 0; q < kPer; ++q)
        offer<E>(rs, trow, drow, e + q, x[q], half_of(b, uint32_t(q)), c, bk, bi);
    }
  }
  for (int i = nvec * kPer + threadIdx.x; i < len; i += kThreads) {
    const int64_t e = e0 + i;
    const float x = Elem<E>::load(trow, e);
    if (!(x >= floor_t)) continue;
    const uint64_t g = uint64_t(e + rs.off);
    const uint4 b = stream_block(rs.st, static_cast<uint32_t>(g >> 3));
    offer<E>(rs, trow, drow, e, x, half_of(b, static_cast<uint32_t>(g & 7)), c, bk, bi);
  }
}

// CTA-wide winner (every thread receives it) of a CTA of NT threads.
template <int NT = kThreads>
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
  for (int w = 1; w < NT / 32; ++w)
    if (race_better(red_k[w], red_i[w], k, i)) {
      k = red_k[w];
      i = red_i[w];
    }
  __syncthreads();
  key = k;
  idx = i;
}

template <int NT = kThreads>
__device__ __forceinline__ float block_max(float v, float* red_k) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  if (lane == 0) red_k[warp] = v;
  __syncthreads();
  float m = red_k[0];
#pragma unroll
  for (int w = 1; w < NT / 32; ++w) m = fmaxf(m, red_k[w]);
  __syncthreads();
  return m;
}

// Race over a whole row by one CTA of NT threads (rare fallback path; no pruning).
template <typename E, int NT = kThreads>
__device__ void race_row_global(const RaceSpec& rs, const uint8_t* trow, const uint8_t* drow,
                                int64_t V, float* red_k, int32_t* red_i, float& out_key,
                                int32_t& out_idx) {
  float bk = -INFINITY;
  int32_t bi = -1;
  for (int64_t e = threadIdx.x; e < V; e += NT) {
    const float x = Elem<E>::load(trow, e);
    const float d = rs.resid ? Elem<E>::load(drow, e) : 0.f;
    if (!race_active(rs, x, d)) continue;
    const float k = exact_key<E>(rs, trow, drow, e);
    if (k > -INFINITY && race_better(k, int32_t(e), bk, bi)) {
      bk = k;
      bi = int32_t(e);
    }
  }
  block_race<NT>(bk, bi, red_k, red_i);
  out_key = bk;
  out_idx = bi;
}

}  // namespace sv
