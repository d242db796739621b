// sv_device.cuh -- device building blocks shared by the verification, drafting and scheduling
// kernels: the Philox4x32-10 counter generator, exponential-race keys, bulk-copy / mbarrier PTX,
// online softmax statistics and block reductions.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "specverify.h"

namespace sv {

constexpr int kThreads = 256;               // threads of every streaming CTA
constexpr int kWarps = kThreads / 32;
constexpr uint32_t kSliceBytes = 16384;     // one row slice staged in shared memory
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Upper bound of -log(E) over every uniform the generator can produce: the largest uniform is
// 1 - 2^-24, for which E = -log(u) ~ 5.96e-8 and -log(E) ~ 16.6355; the bound leaves room for
// rounding.  A race entry whose log-weight plus this bound is below the best key so far cannot win.
constexpr float kMaxNoise = 16.75f;

enum : uint32_t { kTagDraft = 0, kTagAccept = 1, kTagResid = 2, kTagBonus = 3 };

// Added to a race's tag for the stream that holds the low bits of its entries' uniforms.
constexpr uint32_t kTagFine = 4;

// ---- Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11, "Parallel Random Numbers: As Easy as
// 1, 2, 3", section 3.3): ten rounds of the 4x32 S-box; the round multipliers act on words 0 and
// 2, their high halves are xored with the odd words and the round key, and the key advances by the
// Weyl increments after every round.
__device__ __forceinline__ uint4 philox_block(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t m0 = 0xD2511F53u, m1 = 0xCD9E8D57u;
    const uint32_t hi0 = __umulhi(m0, c.x), lo0 = m0 * c.x;
    const uint32_t hi1 = __umulhi(m1, c.z), lo1 = m1 * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// One stream of uniforms: key (lo32(seed), hi32(seed)); the block of group g is the output for
// counter (g, pos, lo32(req), tag << 24 | hi32(req) & 0xFFFFFF).  A scalar draw (ACCEPT) reads
// word 0 of group 0; race entries use the layout below.
struct Stream {
  uint32_t k0, k1, pos, req_lo, hi;
};

__device__ __forceinline__ Stream make_stream(uint64_t seed, uint64_t req, uint32_t pos,
                                              uint32_t tag) {
  Stream s;
  s.k0 = static_cast<uint32_t>(seed);
  s.k1 = static_cast<uint32_t>(seed >> 32);
  s.pos = pos;
  s.req_lo = static_cast<uint32_t>(req);
  s.hi = (tag << 24) | (static_cast<uint32_t>(req >> 32) & 0xFFFFFFu);
  return s;
}

__device__ __forceinline__ uint4 stream_block(const Stream& s, uint32_t group) {
  return philox_block(make_uint4(group, s.pos, s.req_lo, s.hi), s.k0, s.k1);
}

__device__ __forceinline__ uint32_t word_of(const uint4& b, uint32_t lane) {
  return lane == 0 ? b.x : lane == 1 ? b.y : lane == 2 ? b.z : b.w;
}

// The uniform of a scalar draw from word w: u = ((w >> 9) + 1/2) * 2^-23, exact in binary32, inside
// (0, 1).
__device__ __forceinline__ float uniform_of(uint32_t w) {
  return (static_cast<float>(w >> 9) + 0.5f) * 1.1920928955078125e-07f;
}

// Race entries.  The uniform of vocabulary entry v is (n + 1/2) 2^-23 with n = (h << 7) | f:
//   h = 16-bit half (v & 1) (0: low) of word (v >> 1) & 3 of the block at counter v >> 3, so one
//       block serves 8 consecutive entries (the block at v >> 3 is the race's coarse block);
//   f = the top 7 bits of word v & 3 of the block at counter v >> 2 of the FINE stream (tag + 4),
//       drawn only for the few entries whose coarse half does not settle the noise gate.
__device__ __forceinline__ uint32_t half_of(const uint4& b, uint32_t j) {
  const uint32_t w = word_of(b, j >> 1);
  return (j & 1u) ? (w >> 16) : (w & 0xFFFFu);
}

__device__ __forceinline__ Stream fine_stream(Stream s) {
  s.hi += kTagFine << 24;
  return s;
}

// u = (((h << 7) | (fine_word >> 25)) + 1/2) * 2^-23, exact in binary32, inside (0, 1).
__device__ __forceinline__ float race_uniform(uint32_t h, uint32_t fine_word) {
  return (static_cast<float>((h << 7) | (fine_word >> 25)) + 0.5f) * 1.1920928955078125e-07f;
}

// The uniform of race entry v whose coarse half h is known: one FINE block.
__device__ __forceinline__ float race_uniform_at(const Stream& s, uint64_t v, uint32_t h) {
  const uint4 fb = stream_block(fine_stream(s), static_cast<uint32_t>(v >> 2));
  return race_uniform(h, word_of(fb, static_cast<uint32_t>(v & 3)));
}

// The largest of the 8 coarse halves of a block (SIMD 16-bit maxima).
__device__ __forceinline__ uint32_t half_max(const uint4& b) {
  const uint32_t m = __vmaxu2(__vmaxu2(b.x, b.y), __vmaxu2(b.z, b.w));
  return max(m & 0xFFFFu, m >> 16);
}

// Lower bound on m = 2^23 (1 - u) - 1/2 = 0x7FFFFF - n over the 128 uniforms that share the
// coarse half h: (0xFFFF - h) << 7, exact in binary32.
__device__ __forceinline__ float gate_mh(uint32_t h) {
  return static_cast<float>((0xFFFFu - h) << 7);
}

// -log(E) with E = -log(u) the exponential variable of a race entry.  Accurate logf: race winners
// have u close to 1, where E must keep its relative precision.
__device__ __forceinline__ float race_noise(float u) { return -logf(-logf(u)); }

// ---- ordering atomics ------------------------------------------------------------------------
// Add with acquire-release semantics at GPU scope: this thread's earlier writes are ordered before
// the add, and writes ordered before earlier adds on the same word are visible after it -- the
// ordering a "last one to arrive" count needs, without a sequentially consistent fence.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

// ---- status word ---------------------------------------------------------------------------
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status) atomicCAS(status, 0, code);
}

// ---- shared-memory addressing, mbarriers and bulk copies (PTX) ----------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Make barrier initialisation visible to the asynchronous (bulk-copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order earlier generic-proxy accesses of shared memory before later bulk copies into it.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Bulk copy global -> shared completing on `bar` (src, dst 16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Barrier `id` (1..15) over the first `nthreads` threads that reach it (a multiple of 32).
__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Every device-side wait gives up after this long, reports SV_ERR_TIMEOUT and lets its kernel wind
// down, so that a wait that can never end leaves the GPU usable.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Wait for phase `parity` of `bar` for at most `limit_ns`; on expiry report SV_ERR_TIMEOUT and give
// up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int32_t* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > limit_ns) {
      report(status, SV_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// 64-bit global loads with acquire and stores with release semantics at GPU scope.
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Wait until the request number in shared-memory word `w` reaches `seq`, for at most `limit_ns`;
// on expiry report SV_ERR_TIMEOUT and give up.
__device__ __forceinline__ bool wait_seq(const uint32_t* w, uint32_t seq, int32_t* status,
                                         uint64_t limit_ns = kWaitLimitNs) {
  const volatile uint32_t* v = w;
  if (int32_t(*v - seq) >= 0) {
    __threadfence_block();
    return true;
  }
  const uint64_t t0 = global_ns();
  while (int32_t(*v - seq) < 0) {
    if (global_ns() - t0 > limit_ns) {
      report(status, SV_ERR_TIMEOUT);
      return false;
    }
    __nanosleep(64);
  }
  __threadfence_block();
  return true;
}

__device__ __forceinline__ void publish_seq(uint32_t* w, uint32_t seq) {
  __threadfence_block();
  *reinterpret_cast<volatile uint32_t*>(w) = seq;
}

// ---- element access ---------------------------------------------------------------------------
template <typename E>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kPerVec = 4;
  __device__ static __forceinline__ float load(const void* base, int64_t i) {
    return __ldg(reinterpret_cast<const float*>(base) + i);
  }
  __device__ static __forceinline__ void unpack(const uint4& v, float* x) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
};

struct bf16_tag {};

template <>
struct Elem<bf16_tag> {
  static constexpr int kPerVec = 8;
  __device__ static __forceinline__ float load(const void* base, int64_t i) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(base) + i);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  __device__ static __forceinline__ void unpack(const uint4& v, float* x) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(w[j] << 16);
      x[2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
    }
  }
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 1 - exp(y) for y <= 0, accurate relative to the result: near 0 the Taylor series of -expm1,
// -y (1 + y/2! + y^2/3! + ... + y^7/8!) (truncation below 1.1e-8 relative for |y| <= 1/2); below
// -1/2 the difference 1 - 2^(y log2 e) keeps all but 1.4 bits of the result.
__device__ __forceinline__ float one_minus_exp(float y) {
  if (y > -0.5f) {
    float p = 2.48015873015873e-05f;           // 1/8!
    p = fmaf(p, y, 1.984126984126984e-04f);    // 1/7!
    p = fmaf(p, y, 1.388888888888889e-03f);    // 1/6!
    p = fmaf(p, y, 8.333333333333333e-03f);    // 1/5!
    p = fmaf(p, y, 4.166666666666666e-02f);    // 1/4!
    p = fmaf(p, y, 1.666666666666667e-01f);    // 1/3!
    p = fmaf(p, y, 0.5f);                      // 1/2!
    p = fmaf(p, y, 1.0f);
    return -y * p;
  }
  return 1.0f - fast_exp2(y * kLog2e);
}

// ---- online softmax statistics: (m, s) = (running max, sum of exp(x - m)) ----------------------
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) {  // both empty (all -inf so far)
    s = s + s2;           // keeps a NaN visible
    return;
  }
  s = s * fast_exp2((m - mn) * kLog2e) + s2 * fast_exp2((m2 - mn) * kLog2e);
  m = mn;
}

// Fold `n` values into (m, s): one rescale per increase of the maximum, one exp per value.
template <int N>
__device__ __forceinline__ void ms_accumulate(float& m, float& s, const float* x) {
  float cm = x[0];
#pragma unroll
  for (int j = 1; j < N; ++j) cm = fmaxf(cm, x[j]);
  float acc = 0.f;
  if (cm > m) {
    if (m != -INFINITY) s *= fast_exp2((m - cm) * kLog2e);
    m = cm;
  }
  if (m == -INFINITY) {
    // every value so far is -inf (contributes 0) unless one is NaN
#pragma unroll
    for (int j = 0; j < N; ++j)
      if (x[j] != x[j]) s = x[j];
    return;
  }
  // x - m is exact for bf16 inputs; scaling afterwards keeps the rounding relative to the
  // (small) shifted value instead of adding an absolute rounding of m * log2(e) to every term
#pragma unroll
  for (int j = 0; j < N; ++j) acc += fast_exp2((x[j] - m) * kLog2e);
  s += acc;
}

__device__ __forceinline__ void warp_ms(float& m, float& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    ms_merge(m, s, m2, s2);
  }
}

// ---- softmax statistics in the log2 domain: (m, s) with m a binary32 multiple of the row maximum
// times log2(e) and s = sum 2^(x log2(e) - m).  fma(x, log2e, -m) rounds once, relative to the
// (small) shifted value, so the reference point 2^m is exact and carries no rounding into the sum.
// m starts at kM2Empty (finite, below every real value): an all -inf stretch keeps s = 0 and a NaN
// or +inf logit turns s into NaN, which the combining step reports.
constexpr float kM2Empty = -1.0e30f;

__device__ __forceinline__ void ms2_merge(float& m, float& s, float m2, float s2) {
  const float mn = fmaxf(m, m2);
  s = s * fast_exp2(m - mn) + s2 * fast_exp2(m2 - mn);
  m = mn;
}

// Warp-wide (m, s): the common maximum first, then one rescale per lane and a plain sum.
__device__ __forceinline__ void warp_ms2(float& m, float& s) {
  float M = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  s *= fast_exp2(m - M);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  m = M;
}

// Fold one 16-byte vector of logits into (m, s): the vector maximum decides a (rare) rescale,
// then every element costs one fma, one ex2 and one add (summed as a tree).
__device__ __forceinline__ void ms2_fold(float& m, float& s, const float* x, float vmax, int n) {
  const float vm = vmax * kLog2e;
  if (vm > m) {
    s *= fast_exp2(m - vm);
    m = vm;
  }
  float e[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) e[j] = j < n ? fast_exp2(fmaf(x[j], kLog2e, -m)) : 0.f;
  s += ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
}

__device__ __forceinline__ void ms2_vec_bf16(float& m, float& s, const uint4& v) {
  __nv_bfloat162 a = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&v.x),
                             *reinterpret_cast<const __nv_bfloat162*>(&v.y));
  const __nv_bfloat162 b = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&v.z),
                                   *reinterpret_cast<const __nv_bfloat162*>(&v.w));
  a = __hmax2(a, b);
  const uint32_t ab = *reinterpret_cast<const uint32_t*>(&a);
  const float vmax = fmaxf(__uint_as_float(ab << 16), __uint_as_float(ab & 0xFFFF0000u));
  float x[8];
  Elem<bf16_tag>::unpack(v, x);
  ms2_fold(m, s, x, vmax, 8);
}

__device__ __forceinline__ void ms2_vec_f32(float& m, float& s, const uint4& v) {
  float x[8];
  Elem<float>::unpack(v, x);
  const float vmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
  ms2_fold(m, s, x, vmax, 4);
}

// ---- packed binary32 pairs: one fma / add instruction for two lanes, each rounded exactly as the
// scalar operation would be
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 splat2(float x) { return make_float2(x, x); }
// a packed bf16 pair (low half first) widened to binary32, exactly
__device__ __forceinline__ float2 bf16x2_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ float2 exp2_2(float2 a) {
  return make_float2(fast_exp2(a.x), fast_exp2(a.y));
}

// Fold N 16-byte vectors into (m, s): one maximum over all of them decides a (rare) rescale, then
// every element costs half a packed fma, one ex2 and half a packed add (summed as a tree).
template <int N>
__device__ __forceinline__ void ms2_fold_vecs_bf16(float& m, float& s, const uint4* v) {
  auto pair = [](uint32_t w) { return *reinterpret_cast<const __nv_bfloat162*>(&w); };
  __nv_bfloat162 mx = __hmax2(__hmax2(pair(v[0].x), pair(v[0].y)), __hmax2(pair(v[0].z), pair(v[0].w)));
#pragma unroll
  for (int u = 1; u < N; ++u)
    mx = __hmax2(mx, __hmax2(__hmax2(pair(v[u].x), pair(v[u].y)), __hmax2(pair(v[u].z), pair(v[u].w))));
  const uint32_t ab = *reinterpret_cast<const uint32_t*>(&mx);
  const float vm = fmaxf(__uint_as_float(ab << 16), __uint_as_float(ab & 0xFFFF0000u)) * kLog2e;
  if (vm > m) {
    s *= fast_exp2(m - vm);
    m = vm;
  }
  const float2 l2 = splat2(kLog2e), nm = splat2(-m);
  float2 tot = make_float2(0.f, 0.f);
#pragma unroll
  for (int u = 0; u < N; ++u) {
    const float2 e0 = exp2_2(fma2(bf16x2_f2(v[u].x), l2, nm));
    const float2 e1 = exp2_2(fma2(bf16x2_f2(v[u].y), l2, nm));
    const float2 e2 = exp2_2(fma2(bf16x2_f2(v[u].z), l2, nm));
    const float2 e3 = exp2_2(fma2(bf16x2_f2(v[u].w), l2, nm));
    tot = add2(tot, add2(add2(e0, e1), add2(e2, e3)));
  }
  s += tot.x + tot.y;
}

template <int N>
__device__ __forceinline__ void ms2_fold_vecs_f32(float& m, float& s, const uint4* v) {
  float mx = -INFINITY;
#pragma unroll
  for (int u = 0; u < N; ++u)
    mx = fmaxf(mx, fmaxf(fmaxf(__uint_as_float(v[u].x), __uint_as_float(v[u].y)),
                         fmaxf(__uint_as_float(v[u].z), __uint_as_float(v[u].w))));
  const float vm = mx * kLog2e;
  if (vm > m) {
    s *= fast_exp2(m - vm);
    m = vm;
  }
  const float2 l2 = splat2(kLog2e), nm = splat2(-m);
  float2 tot = make_float2(0.f, 0.f);
#pragma unroll
  for (int u = 0; u < N; ++u) {
    const float2 e0 = exp2_2(fma2(make_float2(__uint_as_float(v[u].x), __uint_as_float(v[u].y)), l2, nm));
    const float2 e1 = exp2_2(fma2(make_float2(__uint_as_float(v[u].z), __uint_as_float(v[u].w)), l2, nm));
    tot = add2(tot, add2(e0, e1));
  }
  s += tot.x + tot.y;
}

__device__ __forceinline__ void ms2_one(float& m, float& s, float x) {
  float xs[8] = {x, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  ms2_fold(m, s, xs, x, 1);
}

// Race winner: larger key wins, equal keys go to the lower index; idx < 0 means "none".
__device__ __forceinline__ bool race_better(float k2, int32_t i2, float k1, int32_t i1) {
  if (i2 < 0) return false;
  if (i1 < 0) return true;
  return k2 > k1 || (k2 == k1 && i2 < i1);
}

__device__ __forceinline__ void warp_race(float& key, int32_t& idx) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float k2 = __shfl_xor_sync(0xffffffffu, key, o);
    const int32_t i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    if (race_better(k2, i2, key, idx)) {
      key = k2;
      idx = i2;
    }
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace sv
