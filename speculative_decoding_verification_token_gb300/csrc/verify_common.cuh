// verify_common.cuh -- what token-level verification (token.cu) and block verification and draft
// sampling (verify.cu) share: the streaming ring's geometry, the per-request race descriptor and
// race slot, the workspace layout, the argument checks, and the arithmetic that turns a row pair's
// softmax statistics into the drafted token's ratio p(x)/q(x) and the residual's offset.
#pragma once

#include <algorithm>

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

struct RaceDesc {  // per request: the decision, read by the race
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

constexpr int32_t kResShareBytes = 16384;  // bytes of one row in one residual-mass task

// Block verification's per-request state between its kernels.  Residual masses are computed for
// "slots": round-1 slots [0, count[0]) are listed by the prep kernel, round-2 slots
// [units, units + count[1]) by the round-1 kernel.
struct BlockWs {
  float4* norm;    // [units] row-pair normalisers (m_t, s_t, m_d, s_d), log2 domain
  float* rho;      // [units] running ratio rho_i
  float* eta;      // [units] ACCEPT uniform eta_i
  int32_t* cand;   // [units] slot of (r, i), -1 if R_i is not computed
  int32_t* unit;   // [2 units] unit (r * gmax + i - 1) of each slot
  int32_t* done;   // [units] round-1 slots: shares finished
  int32_t* count;  // [2] slots listed for round 1 and round 2
  float* rpart;    // [2 units * CLr] residual mass partials, one per (slot, share)
  int32_t units;   // B * gmax: the first round-2 slot
  int32_t CLr;     // residual tasks (shares) per row
};

struct VerifyWs {
  float4* partials;  // [units * C] (m_t, s_t, m_d, s_d), m in log2 units
  RaceDesc* desc;    // [B]
  RaceSlot* slots;   // [units]: verify uses B of them, the sampler one per drafted row
  BlockWs blk;
  int32_t* claim;                   // the stream kernel's item counter
  unsigned long long* claim_ready;  // the launch's call id once the counter is zeroed
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

// Residual-mass tasks per row: one per kResShareBytes of the row.
static inline int32_t resid_shares_of(int64_t V, int esz) {
  const int64_t per = kResShareBytes / esz;
  return static_cast<int32_t>((V + per - 1) / per);
}

static inline VerifyWs verify_layout(void* base, int32_t B, int32_t gmax, int64_t V, int esz) {
  const int32_t C = chunks_of(V, esz);
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
  w.blk.CLr = resid_shares_of(V, esz);
  w.blk.units = static_cast<int32_t>(units);
  w.blk.norm = reinterpret_cast<float4*>(take(sizeof(float4) * units));
  w.blk.rho = reinterpret_cast<float*>(take(sizeof(float) * units));
  w.blk.eta = reinterpret_cast<float*>(take(sizeof(float) * units));
  w.blk.cand = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * units));
  w.blk.unit = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * 2 * units));
  w.blk.done = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * units));
  w.blk.count = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * 2));
  w.blk.rpart = reinterpret_cast<float*>(take(sizeof(float) * 2 * units * size_t(w.blk.CLr)));
  w.claim = reinterpret_cast<int32_t*>(take(sizeof(int32_t)));
  w.claim_ready = reinterpret_cast<unsigned long long*>(take(sizeof(unsigned long long)));
  w.total = off;
  return w;
}

static inline size_t verify_ws_bytes(int32_t B, int32_t gmax, int64_t V, int esz) {
  return verify_layout(nullptr, B, gmax, V, esz).total;
}

__device__ __forceinline__ int32_t clamp_gamma(int32_t g, int32_t gmax) {
  return (g < 0 || g > gmax) ? 0 : g;
}

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

// ---- host side ------------------------------------------------------------------------------
struct CommonArgs {
  const void* target;
  const void* draft;
  sv_dtype dtype;
  int64_t V, ld;
  int32_t B, gmax;
  void* ws;
  size_t ws_bytes;
};

static inline sv_status check_common(const CommonArgs& a, bool need_target) {
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

}  // namespace sv
