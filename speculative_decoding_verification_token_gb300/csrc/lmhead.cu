// lmhead.cu -- token-level verification from hidden states (spec_verify_lmhead).
//
// The target's and the draft's logits are the products of their hidden states with one output
// projection W [V][H] ("How much does a token cost", "The Role of Arithmetic Intensity": inputs
// [Q, H] times weights [H, W]).  They are computed on the tensor cores and folded as they leave
// the accumulators; no logit is ever written to memory.  Kernels on the caller's stream:
//   gather  the hidden rows of every request into the GEMM's A operand, two slots per position:
//           slot 2j holds target row j, slot 2j + 1 draft row j, 2 (gmax + 1) slots per request
//           (the slots a request does not use are never read back);
//   stats   persistent, warp-specialised tcgen05 GEMM, (128 slots) x (256 vocabulary columns) per
//           tile, K = H streamed in 64-element k-blocks:
//             warp 0      tensor-TMA loads of the slot block's and of W's k-blocks into a ring;
//             warp 1      tcgen05.mma (M = 128, N = 256, K = 16) into one of two TMEM
//                         accumulators;
//             warps 2-17  the epilogue, a lane quadrant (32 slots) and a column quarter each: the
//                         log2-domain softmax statistics of every slot and the drafted token's
//                         logit -- one (m_t, s_t, m_d, s_d) partial per (row pair, CTA) -- and the
//                         race candidates of every position: each target slot and its draft slot
//                         (neighbouring lanes) split the columns and keep the kLmCand entries of
//                         largest plain key a = t - log E (E the entry's exponential variable of
//                         the position's correction or bonus stream), with d - t beside each;
//   decide  one CTA per request: the row normalisers, p(x)/q(x), the ACCEPT uniforms and the first
//           rejection, exactly as token-level verification of stored logits decides; then the race
//           over the candidates of the rejected (or bonus) position.  Every entry a lane did not
//           keep has a plain key no larger than that lane's bound theta (its last kept key, or the
//           gate key shared by all lanes of the position that it was dropped against), and its
//           residual key a + log(1 - exp(d - t + gap)) is smaller still; so the candidates' winner
//           is the race's winner whenever its key exceeds every theta (always, for a bonus token).
//           Otherwise the request is queued and its two hidden rows are copied into a second A
//           operand;
//   race    the same GEMM over the queued requests' rows (128-column tiles; no work and an early
//           exit when the queue is empty): the epilogue pairs each target slot with its draft slot
//           and runs the exponential race on the recomputed logits, gated against a bound every
//           CTA of the request publishes;
//   finish  the outputs: the candidates' winner, or the folded partial winners of a queued request.
#include <algorithm>

#include "tc.cuh"
#include "tmap.h"
#include "verify_kernels.cuh"

namespace sv {
namespace {

constexpr int kLmRows = 128;                   // slots per M-block (UMMA M)
constexpr int kLmEpiWarps = 16;                // 4 lane quadrants x 4 column quarters
constexpr int kLmThreads = 32 * (2 + kLmEpiWarps);
constexpr uint32_t kLmABytes = kLmRows * 128;  // one 64-element k-block of the slot block: 16 KB
constexpr uint32_t kLmRingBytes = 196608;      // the operand ring
constexpr int kLmStatsN = 256;                 // vocabulary columns per tile, statistics GEMM
constexpr int kLmRaceN = 128;                  // the same, race GEMM
constexpr int kLmCand = 8;                     // race candidates kept per lane and position
constexpr int kLmParts = 8;                    // candidate partitions per (position, CTA):
                                               // 4 column quarters x 2 lanes of a slot pair

template <int kN>
struct LmShape {
  static constexpr uint32_t kBBytes = kN * 128;  // one k-block of W: kN rows x 64
  static constexpr uint32_t kStageBytes = kLmABytes + kBBytes;
  static constexpr int kStages = int(kLmRingBytes / kStageBytes);
  static constexpr int kCols = kN / 4;           // columns per epilogue warp and tile
  static constexpr uint32_t kTmemCols = 2 * kN;  // two accumulators
  static constexpr size_t kSmem = 1024 + size_t(kStages) * kStageBytes;
};

struct LmParams {
  int32_t n_mblocks, per_mblock, n_tiles;  // slot blocks, CTAs per slot block, vocabulary tiles
  int32_t kblocks;                         // H / 64
  int64_t V;
  int32_t B, gmax, slots;                  // slots per request: 2 (gmax + 1), or 2 for the race
  // statistics
  const int64_t* draft_row0;
  const int32_t* draft_len;
  const int32_t* draft_tokens;
  float4* partials;  // [B * gmax][per_mblock]: (m_t, s_t, m_d, s_d), log2 domain
  float2* tok;       // [B * gmax]: the drafted token's target and draft logits
  float4* cand;      // [B (gmax + 1)][per_mblock][kLmParts][kLmCand]: (a, d - t, index, 0)
  float* theta;      // [B (gmax + 1)][per_mblock][kLmParts]: bound on the dropped entries' a
  uint32_t* cpub;    // [B (gmax + 1)] largest last-kept key any lane has published (key_order)
  // race
  const RaceDesc* desc;          // [B]
  uint64_t seed;
  const uint64_t* request_ids;
  uint32_t* k0;                  // [B] best exact race key published so far (key_order; 0: none)
  unsigned long long* winners;   // [per_mblock][B][2] packed partial winners
  const int32_t* race_count;     // requests queued for the race GEMM
  const int32_t* race_list;      // [B] the queued requests, in queue order
  int32_t* status;
};

// The GEMM's waits: mbar_wait with a suspend-time hint, so that a waiting thread sleeps until the
// phase completes instead of polling, leaving the issue slots to the epilogue's arithmetic (0.407
// -> 0.397 ms per call at 64 x 5, V = 151936, H = 2560).  Bounded like mbar_wait: after
// kWaitLimitNs it reports SV_ERR_TIMEOUT and gives up.
__device__ __forceinline__ bool lm_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred P;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2, %3;\n\t"
      "selp.b32 %0, 1, 0, P;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool lm_wait(uint64_t* bar, uint32_t parity, int32_t* status) {
  if (lm_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!lm_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) {
      report(status, SV_ERR_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Copies of hidden rows: one warp per row, 16-byte vectors, four loads in flight per lane.
__device__ __forceinline__ void copy_row(uint8_t* dst, const uint8_t* src, int64_t bytes,
                                         int lane) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
  uint4* d = reinterpret_cast<uint4*>(dst);
  const int64_t n = bytes / 16;
  int64_t i = lane;
  for (; i + 96 < n; i += 128) {
    const uint4 a0 = __ldg(s + i), a1 = __ldg(s + i + 32), a2 = __ldg(s + i + 64),
                a3 = __ldg(s + i + 96);
    d[i] = a0;
    d[i + 32] = a1;
    d[i + 64] = a2;
    d[i + 96] = a3;
  }
  for (; i < n; i += 32) d[i] = __ldg(s + i);
}

constexpr int kGatherWarps = 8;

// Slot block of the statistics GEMM: request r's target row j into slot r S + 2j (j <= g), its
// draft row j into slot r S + 2j + 1 (j < g); one warp per (request, slot).  The first warp of
// each request also clears its published candidate bounds; block 0 clears the status and the race
// queue.
__global__ void __launch_bounds__(32 * kGatherWarps)
    lm_gather_kernel(const uint8_t* __restrict__ th, const uint8_t* __restrict__ dh, int64_t ldh,
                     int64_t H, const int64_t* __restrict__ target_row0,
                     const int64_t* __restrict__ draft_row0, const int32_t* __restrict__ draft_len,
                     int32_t B, int32_t gmax, uint8_t* __restrict__ A, uint32_t* cpub,
                     int32_t* race_count, int32_t* status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    *race_count = 0;
    if (status) *status = 0;
  }
  const int32_t per = 2 * gmax + 1;  // rows a request may have
  const int64_t w = int64_t(blockIdx.x) * kGatherWarps + (threadIdx.x >> 5);
  if (w >= int64_t(B) * per) return;
  const int32_t r = static_cast<int32_t>(w / per);
  const int32_t s = static_cast<int32_t>(w % per);
  if (s == 0)
    for (int32_t j = lane; j <= gmax; j += 32) cpub[size_t(r) * (gmax + 1) + j] = 0u;
  const int32_t g = clamp_gamma(draft_len[r], gmax);
  if (s >= 2 * g + 1) return;
  const int32_t j = s >> 1;
  const uint8_t* src = (s & 1) ? dh + (draft_row0[r] + j) * ldh * 2
                               : th + (target_row0[r] + j) * ldh * 2;
  copy_row(A + (int64_t(r) * 2 * (gmax + 1) + s) * H * 2, src, H * 2, lane);
}

struct KeyIdx {
  float key;
  int32_t idx;
};

__device__ __forceinline__ void offer_key(float k, int32_t e, KeyIdx& b) {
  if (race_better(k, e, b.key, b.idx)) {
    b.key = k;
    b.idx = e;
  }
}

// Exact keys of entry e (logits t, d; race uniform u): the race's own key into `best` (residual or
// bonus), and for a residual race the key of the race over p with the same uniform into `fb`.
__device__ __forceinline__ void key_entry(const RaceSpec& rs, float t, float d, float u,
                                          int32_t e, KeyIdx& best, KeyIdx& fb) {
  if (!(t > -INFINITY)) return;
  const float noise = race_noise(u);
  if (rs.resid) offer_key(t + noise, e, fb);
  if (race_active(rs, t, d)) offer_key(race_key(rs, t, d, noise), e, best);
}

// ---- race candidates: per lane, the kLmCand entries of largest plain key a = t - log E seen so
// far (unordered), with the position and key of the smallest.  The keys stay in registers; each
// entry's b = d - t and index sit in shared memory (bx[i * kBxStride], this lane's column of the
// block's candidate buffer), written only when an entry enters the list.  Equal keys may be kept
// either way: the decision only needs every dropped entry's key to be no larger than a bound.
constexpr int kBxStride = 32 * kLmEpiWarps;

struct CandList {
  float a[kLmCand];
  float amin;  // smallest kept key (-inf while the list is not full)
  int pmin;    // its position
  float2* bx;  // (b, index as float bits) of entry i at bx[i * kBxStride]
};

__device__ __forceinline__ void cand_init(CandList& c, float2* bx) {
  c.bx = bx;
#pragma unroll
  for (int i = 0; i < kLmCand; ++i) {
    c.a[i] = -INFINITY;
    c.bx[i * kBxStride] = make_float2(0.f, __int_as_float(-1));
  }
  c.amin = -INFINITY;
  c.pmin = 0;
}

// (a, b, e) replaces the smallest entry (the caller checked a > amin).
__device__ __forceinline__ void cand_insert(CandList& c, float a, float b, int32_t e) {
  c.bx[c.pmin * kBxStride] = make_float2(b, __int_as_float(e));
#pragma unroll
  for (int i = 0; i < kLmCand; ++i)
    if (i == c.pmin) c.a[i] = a;
  float m = c.a[0];
  int pm = 0;
#pragma unroll
  for (int i = 1; i < kLmCand; ++i)
    if (c.a[i] < m) {
      m = c.a[i];
      pm = i;
    }
  c.amin = m;
  c.pmin = pm;
}

// Offers 16 entries (columns e0 .. e0 + 15, e0 a multiple of 16) with target logits tt and draft
// logits dd, against the gate key G: an entry enters the list only if its plain key exceeds both
// the list's smallest key and G.  Its logit must then be within kMaxNoise of that bound, and the
// coarse half of its uniform must pass the noise gate of race.cuh (first for each 8 entries at
// once, on their coarse block's largest half); the few entries that pass are collected in a mask
// and keyed exactly afterwards, drawing their low bits in one (not unrolled) loop.
__device__ __forceinline__ void cand_offer16(CandList& c, const Stream& st, const float* tt,
                                             const float* dd, int64_t e0, float G) {
#pragma unroll
  for (int g8 = 0; g8 < 2; ++g8) {
    const float T = fmaxf(c.amin, G);
    float tm = tt[8 * g8];
#pragma unroll
    for (int q = 1; q < 8; ++q) tm = fmaxf(tm, tt[8 * g8 + q]);
    if (!(tm >= T - kMaxNoise)) continue;
    const float cg = 23.0f - T * kLog2e;
    const uint4 blk = stream_block(st, static_cast<uint32_t>((e0 >> 3) + g8));
    if (gate_mh(half_max(blk)) > gate_threshold(tm, cg)) continue;
    uint32_t surv = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float t = tt[8 * g8 + q];
      const uint32_t hq = half_of(blk, static_cast<uint32_t>(q));
      if (t > -INFINITY && gate_mh(hq) <= gate_threshold(t, cg)) surv |= 1u << q;
    }
#pragma unroll 1
    while (surv) {
      const uint32_t q = __ffs(surv) - 1;
      surv &= surv - 1;
      float t = 0.f, d = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k)
        if (uint32_t(k) == q) {
          t = tt[8 * g8 + k];
          d = dd[8 * g8 + k];
        }
      const int64_t e = e0 + 8 * g8 + q;
      const float u = race_uniform_at(st, static_cast<uint64_t>(e), half_of(blk, q));
      const float a = t + race_noise(u);
      if (a > c.amin && a > G) cand_insert(c, a, d - t, static_cast<int32_t>(e));
    }
  }
}

// The decision of request r (decide_body, on the statistics partials and the drafted tokens'
// logits the statistics GEMM left), then the race over the candidates of its correction (or
// bonus) position; a request the candidates cannot settle is queued for the race GEMM with its
// two rows: queue slot i <- target row tau (slot 2i) and draft row tau (slot 2i + 1), both copied
// from the statistics slot block.
struct LmDecideParams {
  DecideParams dp;
  const uint8_t* A1;
  uint8_t* A2;
  int64_t row_bytes;
  RaceDesc* desc;
  uint32_t* k0;
  int32_t* accepted_len;
  const float4* cand;
  const float* theta;
  int32_t C;                      // statistics CTAs per slot block
  unsigned long long* decided;    // [B] packed winner of a settled request
  int32_t* pending;               // [B] 1: queued for the race GEMM
  int32_t* race_count;
  int32_t* race_list;
};

__global__ void __launch_bounds__(kThreads) lm_decide_kernel(LmDecideParams p) {
  __shared__ RaceDesc s_desc;
  __shared__ int32_t s_tok[SV_MAX_DRAFT_LEN];
  __shared__ float red_k[kWarps];
  __shared__ int32_t red_i[kWarps];
  __shared__ int32_t s_slot;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the statistics GEMM's partials
  const int32_t r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  decide_body<float>(p.dp, r, true, &s_desc, s_tok, false);
  __syncthreads();
  const RaceDesc d = s_desc;
  const size_t u2 = size_t(r) * (p.dp.gmax + 1) + d.tau;
  const int32_t n_parts = p.C * kLmParts;
  const float4* cd = p.cand + u2 * n_parts * kLmCand;
  KeyIdx best = {-INFINITY, -1};
  auto offer_cand = [&](const float4& q) {
    const int32_t e = __float_as_int(q.z);
    if (e < 0) return;
    if (!d.resid) {
      offer_key(q.x, e, best);
    } else {
      const float y = q.y + d.gap;
      if (y < 0.f) offer_key(q.x + __logf(one_minus_exp(y)), e, best);
    }
  };
  const int32_t n_cand = n_parts * kLmCand;
  int32_t i = tid;
  for (; i + 3 * kThreads < n_cand; i += 4 * kThreads) {  // four loads in flight
    const float4 q0 = cd[i], q1 = cd[i + kThreads], q2 = cd[i + 2 * kThreads],
                 q3 = cd[i + 3 * kThreads];
    offer_cand(q0);
    offer_cand(q1);
    offer_cand(q2);
    offer_cand(q3);
  }
  for (; i < n_cand; i += kThreads) offer_cand(cd[i]);
  float bound = -INFINITY;  // largest plain key an unkept entry may have
  for (int32_t i = tid; i < n_parts; i += kThreads) bound = fmaxf(bound, p.theta[u2 * n_parts + i]);
  block_race<kThreads>(best.key, best.idx, red_k, red_i);
  bound = block_max<kThreads>(bound, red_k);
  // settled: a bonus (its winner has the largest plain key of all, which some partition kept), or
  // a residual winner above every unkept entry's plain key
  const bool settled = !d.resid || (best.idx >= 0 && best.key > bound);
  if (tid == 0) {
    p.desc[r] = d;
    p.accepted_len[r] = d.tau;
    p.pending[r] = settled ? 0 : 1;
    p.decided[r] = (settled && best.idx >= 0) ? race_pack(best.key, best.idx) : 0ull;
    if (!settled) {
      p.k0[r] = 0u;
      const int32_t i = atomicAdd(p.race_count, 1);
      p.race_list[i] = r;
      s_slot = i;
    }
  }
  __syncthreads();
  if (settled) return;
  const int32_t S = 2 * (p.dp.gmax + 1);
  if (warp < (d.resid ? 2 : 1))
    copy_row(p.A2 + (int64_t(2) * s_slot + warp) * p.row_bytes,
             p.A1 + (int64_t(r) * S + 2 * d.tau + warp) * p.row_bytes, p.row_bytes, lane);
}

template <int kN, bool kRace>
__global__ void __launch_bounds__(kLmThreads, 1)
    lm_gemm_kernel(const __grid_constant__ CUtensorMap map_a,
                   const __grid_constant__ CUtensorMap map_w, LmParams p) {
  using Sh = LmShape<kN>;
  constexpr int kStages = Sh::kStages;
  constexpr int kCols = Sh::kCols;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kStages], empty[kStages];
  __shared__ uint64_t acc_full[2], acc_empty[2];
  __shared__ uint32_t tmem_base;
  // the epilogue's candidate buffer ([kLmCand][kBxStride] float2), reused afterwards for the
  // merge of column quarters 1..3 into quarter 0 ([3][kLmRows] float4)
  __shared__ __align__(16) uint8_t epi_buf[kLmCand * kBxStride * sizeof(float2)];
  static_assert(sizeof(epi_buf) >= 3 * kLmRows * sizeof(float4), "merge area");
  float4 (*merge)[kLmRows] = reinterpret_cast<float4 (*)[kLmRows]>(epi_buf);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t mb = blockIdx.x % p.n_mblocks;
  const int32_t ci = blockIdx.x / p.n_mblocks;
  const int32_t m0 = mb * kLmRows;
  const int32_t n_my = ci < p.n_tiles ? (p.n_tiles - ci + p.per_mblock - 1) / p.per_mblock : 0;
  // programmatic dependent of the kernel before it (gather, resp. decide): its outputs are read
  // only after griddepcontrol.wait, which every CTA executes before it exits
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  int32_t queued = 0;  // race GEMM: requests in the queue (two slots each)
  if constexpr (kRace) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    queued = *reinterpret_cast<const volatile int32_t*>(p.race_count);
    if (m0 >= 2 * queued) return;  // the whole CTA: nothing allocated or initialised yet
  }

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&acc_full[a], 1);
      mbar_init(&acc_empty[a], kLmEpiWarps);
    }
    fence_barrier_init();
  }
  if (warp == 1) tc::tmem_alloc(&tmem_base, Sh::kTmemCols);
  if constexpr (!kRace) asm volatile("griddepcontrol.wait;" ::: "memory");  // the slot block
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    // ---- producer: for every tile, the k-blocks of the slot block and of W's columns
    if (lane == 0) {
      // the slot block is re-read for every tile: keep it in L2; W streams through once
      const uint64_t keep = tc::policy_evict_last(), once = tc::policy_evict_first();
      uint32_t it = 0;
      bool ok = true;
      for (int t = 0; t < n_my && ok; ++t) {
        const int32_t n = ci + t * p.per_mblock;
        for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t use = it / kStages;
          if (use > 0 && !lm_wait(&empty[s], (use - 1) & 1, p.status)) {
            ok = false;
            break;
          }
          uint8_t* st = ring + size_t(s) * Sh::kStageBytes;
          mbar_expect_tx(&full[s], Sh::kStageBytes);
          tc::tma_load_2d_hint(st, &map_a, kb * 64, m0, &full[s], keep);
          tc::tma_load_2d_hint(st + kLmABytes, &map_w, kb * 64, n * kN, &full[s], once);
        }
      }
    }
  } else if (warp == 1) {
    // ---- tensor-core issuer
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kLmRows, kN);
      uint32_t it = 0;
      bool ok = true;
      for (int t = 0; t < n_my && ok; ++t) {
        const int acc = t & 1;
        if (t >= 2 && !lm_wait(&acc_empty[acc], ((t >> 1) - 1) & 1, p.status)) break;
        tc::fence_after_sync();
        for (int kb = 0; kb < p.kblocks; ++kb, ++it) {
          const int s = it % kStages;
          if (!lm_wait(&full[s], (it / kStages) & 1, p.status)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a_base = smem_addr(ring + size_t(s) * Sh::kStageBytes);
          const uint32_t b_base = a_base + kLmABytes;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)  // 16 K-elements (32 bytes) per instruction
            tc::mma_bf16(tmem + acc * kN, tc::smem_desc_sw128(a_base + ks * 32),
                         tc::smem_desc_sw128(b_base + ks * 32), idesc, (kb | ks) != 0);
          tc::mma_commit(&empty[s]);
        }
        if (ok) tc::mma_commit(&acc_full[acc]);
      }
    }
  } else {
    // ---- epilogue: warp w reads TMEM lane quadrant q = w % 4 (slots m0 + 32q ..) and column
    // quarter h of every tile; thread (q, lane) owns slot m0 + 32q + lane.  A target slot and its
    // draft slot are neighbouring lanes (2i, 2i + 1).
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const uint32_t rl = 32 * q + lane;
    const int32_t R = m0 + static_cast<int32_t>(rl);
    const int32_t kind = R & 1;  // 0: target slot, 1: draft slot
    bool failed = false;

    if constexpr (!kRace) {
      const int32_t r = R / p.slots;
      const bool row_ok = r < p.B;
      const int32_t j = (R - r * p.slots) >> 1;  // 0-based position of the row pair
      int32_t x = -1;                            // drafted token of the pair, if any
      int32_t mode = 0;                          // 1: correction candidates, 2: bonus candidates
      uint64_t req = 0;
      if (row_ok) {
        const int32_t g = clamp_gamma(p.draft_len[r], p.gmax);
        if (j < g) {
          x = p.draft_tokens[p.draft_row0[r] + j];
          mode = 1;
        } else if (j == g) {
          mode = 2;
        }
        req = p.request_ids ? p.request_ids[r] : uint64_t(r);
      }
      const Stream st = make_stream(p.seed, req, static_cast<uint32_t>(j + 1),
                                    mode == 1 ? kTagResid : kTagBonus);
      // Candidate gate shared by every lane of the position (all CTAs): the largest last-kept key
      // any full list has published.  An entry below it is not needed from this lane either: its
      // plain key is no larger than that lane's bound, which the decision checks anyway.
      uint32_t* const cslot = mode ? p.cpub + size_t(r) * (p.gmax + 1) + j : nullptr;
      float G = -INFINITY;          // gate key read at the previous tile
      float gate_max = -INFINITY;   // largest gate key used
      float published = -INFINITY;  // the largest key this lane has published
      CandList cl;
      cand_init(cl, reinterpret_cast<float2*>(epi_buf) + (tid - 64));
      float m2 = kM2Empty, sum = 0.f, xl = 0.f;
      float xf = 0.f;  // 1: this CTA saw the drafted token's column
      for (int t = 0; t < n_my; ++t) {
        const int32_t n = ci + t * p.per_mblock;
        const int acc = t & 1;
        if (!failed && !lm_wait(&acc_full[acc], (t >> 1) & 1, p.status)) failed = true;
        __syncwarp();
        tc::fence_after_sync();
        gate_max = fmaxf(gate_max, G);
#pragma unroll
        for (int hh = 0; hh < kCols / 32; ++hh) {
          float v[32];
          tc::tmem_load32(tmem + (uint32_t(32 * q) << 16) + acc * kN + h * kCols + 32 * hh, v);
          if (hh == kCols / 32 - 1) {  // the accumulator is free once every column is loaded
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
          }
          const int64_t c0 = int64_t(n) * kN + h * kCols + 32 * hh;
          if (c0 + 32 > p.V) {  // the tile that crosses V: W's rows past V load as zeros
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (c0 + c >= p.V) v[c] = -INFINITY;
          }
          const int64_t dx = int64_t(x) - c0;
          if (dx >= 0 && dx < 32) {
            float val = v[0];
#pragma unroll
            for (int c = 1; c < 32; ++c)
              if (c == dx) val = v[c];
            xl = val;
            xf = 1.f;
          }
          // log2-domain statistics: one rescale per 32 columns, then 2^(v log2e - m2) each
          float tmax = v[0];
#pragma unroll
          for (int c = 1; c < 32; ++c) tmax = fmaxf(tmax, v[c]);
          const float vm = tmax * kLog2e;
          if (vm > m2) {
            sum *= fast_exp2(m2 - vm);
            m2 = vm;
          }
          const float2 l2 = splat2(kLog2e), nm = splat2(-m2);
          float2 tot = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < 32; c += 4) {
            const float2 e0 = exp2_2(fma2(make_float2(v[c], v[c + 1]), l2, nm));
            const float2 e1 = exp2_2(fma2(make_float2(v[c + 2], v[c + 3]), l2, nm));
            tot = add2(tot, add2(e0, e1));
          }
          sum += tot.x + tot.y;
          // race candidates: the target slot takes columns 0..15 of the 32, the draft slot
          // 16..31, each with both logits of its entries.  In place: afterwards v[0..15] holds the
          // target logits and v[16..31] the draft logits of this lane's 16 entries.
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float recv = __shfl_xor_sync(0xffffffffu, kind ? v[c] : v[16 + c], 1);
            if (kind)
              v[c] = recv;
            else
              v[16 + c] = recv;
          }
          if (mode) cand_offer16(cl, st, v, v + 16, c0 + (kind ? 16 : 0), G);
        }
        if (mode) {
          const float last = cl.amin;  // -inf until the list is full
          if (last > published && last > G) {
            atomicMax(cslot, key_order(last));
            published = last;
          }
          G = key_from_order(__ldcg(cslot));  // used from the next tile on
        }
      }
      if (mode) {
        const size_t pp = (size_t(r) * (p.gmax + 1) + j) * p.per_mblock + ci;
        const int part = h * 2 + kind;
        float4* dst = p.cand + (pp * kLmParts + part) * kLmCand;
#pragma unroll
        for (int i = 0; i < kLmCand; ++i) {
          const float2 bx = cl.bx[i * kBxStride];
          dst[i] = make_float4(cl.a[i], bx.x, bx.y, 0.f);
        }
        // every entry this lane did not keep has a plain key no larger than its last kept one or
        // than the gate key it was dropped against
        p.theta[pp * kLmParts + part] = fmaxf(cl.amin, gate_max);
      }
      named_sync(1, 32 * kLmEpiWarps);  // the candidate buffer becomes the merge area
      if (h > 0) merge[h - 1][rl] = make_float4(m2, sum, xl, xf);
      named_sync(1, 32 * kLmEpiWarps);
      if (h == 0) {
#pragma unroll
        for (int hh = 0; hh < 3; ++hh) {
          const float4 o = merge[hh][rl];
          ms2_merge(m2, sum, o.x, o.y);
          if (o.w != 0.f) {
            xl = o.z;
            xf = 1.f;
          }
        }
        const float pm = __shfl_xor_sync(0xffffffffu, m2, 1);
        const float ps = __shfl_xor_sync(0xffffffffu, sum, 1);
        const float pxl = __shfl_xor_sync(0xffffffffu, xl, 1);
        if (kind == 0 && row_ok && j < p.gmax) {
          const int32_t unit = r * p.gmax + j;
          p.partials[size_t(unit) * p.per_mblock + ci] = make_float4(m2, sum, pm, ps);
          if (xf != 0.f) p.tok[unit] = make_float2(xl, pxl);
        }
      }
    } else {
      // race: the target slot keys the first half of each warp's columns, the draft slot the
      // second half, each with both logits of its entries (one exchange per column)
      constexpr int kHalf = kCols / 2;
      const int32_t qi = R >> 1;  // queue slot
      const bool row_ok = qi < queued;
      const int32_t r = row_ok ? p.race_list[qi] : 0;
      RaceDesc d = {0, 0, 0.f, 0};
      if (row_ok) d = p.desc[r];
      RaceSpec rs;
      rs.resid = d.resid != 0;
      rs.gap = d.gap;
      const uint64_t req = row_ok ? (p.request_ids ? p.request_ids[r] : uint64_t(r)) : 0;
      rs.st = make_stream(p.seed, req, static_cast<uint32_t>(d.tau + 1),
                          rs.resid ? kTagResid : kTagBonus);
      uint32_t* const kslot = row_ok ? p.k0 + r : nullptr;
      uint32_t kpub = 0;
      float published = -INFINITY;
      KeyIdx best = {-INFINITY, -1}, fb = {-INFINITY, -1};
      bool seeded = false;
      for (int t = 0; t < n_my; ++t) {
        const int32_t n = ci + t * p.per_mblock;
        const int acc = t & 1;
        if (!failed && !lm_wait(&acc_full[acc], (t >> 1) & 1, p.status)) failed = true;
        __syncwarp();
        tc::fence_after_sync();
        float v[kCols];
#pragma unroll
        for (int c = 0; c < kCols; c += 32)
          tc::tmem_load32(tmem + (uint32_t(32 * q) << 16) + acc * kN + h * kCols + c, v + c);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[acc]);
        float tt[kHalf], dd[kHalf];
#pragma unroll
        for (int c = 0; c < kHalf; ++c) {
          const float recv = __shfl_xor_sync(0xffffffffu, kind ? v[c] : v[kHalf + c], 1);
          tt[c] = kind ? recv : v[c];
          dd[c] = kind ? v[kHalf + c] : recv;
        }
        if (!row_ok) continue;
        const int64_t e0 = int64_t(n) * kN + h * kCols + (kind ? kHalf : 0);  // multiple of 16
        if (e0 + kHalf > p.V) {
#pragma unroll
          for (int c = 0; c < kHalf; ++c)
            if (e0 + c >= p.V) tt[c] = -INFINITY;
        }
        if (!seeded) {
          // the first tile seeds the bound with the exact key of its largest logit
          float tm = tt[0], dm = dd[0];
          int cm = 0;
#pragma unroll
          for (int c = 1; c < kHalf; ++c)
            if (tt[c] > tm) {
              tm = tt[c];
              dm = dd[c];
              cm = c;
            }
          if (tm > -INFINITY) {
            const int64_t e = e0 + cm;
            const uint4 b = stream_block(rs.st, static_cast<uint32_t>(e >> 3));
            const uint32_t hm = half_of(b, static_cast<uint32_t>(e & 7));
            key_entry(rs, tm, dm, race_uniform_at(rs.st, static_cast<uint64_t>(e), hm),
                      static_cast<int32_t>(e), best, fb);
            seeded = true;
          }
        }
        // gate (race.cuh): an entry reaches the bound K only if its logit is within kMaxNoise
        // of K and the coarse half of its uniform passes the noise threshold (first for 8
        // entries at once); the survivors draw their low bits and are keyed exactly
        const float K = fmaxf(best.key, key_from_order(kpub));
        const float floor_t = K - kMaxNoise;
        const float cg = 23.0f - K * kLog2e;
#pragma unroll
        for (int g8 = 0; g8 < kHalf / 8; ++g8) {
          float tm = tt[8 * g8];
#pragma unroll
          for (int c = 1; c < 8; ++c) tm = fmaxf(tm, tt[8 * g8 + c]);
          if (!(tm >= floor_t)) continue;
          const uint4 b = stream_block(rs.st, static_cast<uint32_t>((e0 >> 3) + g8));
          if (gate_mh(half_max(b)) > gate_threshold(tm, cg)) continue;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float tv = tt[8 * g8 + c];
            const uint32_t hv = half_of(b, static_cast<uint32_t>(c));
            if (!(gate_mh(hv) <= gate_threshold(tv, cg))) continue;
            const int64_t e = e0 + 8 * g8 + c;
            key_entry(rs, tv, dd[8 * g8 + c], race_uniform_at(rs.st, static_cast<uint64_t>(e), hv),
                      static_cast<int32_t>(e), best, fb);
          }
        }
        const float kp = key_from_order(kpub);
        if (best.key > published && best.key > kp) {
          atomicMax(kslot, key_order(best.key));
          published = best.key;
        }
        kpub = __ldcg(kslot);  // consumed at the next tile
      }
      if (h > 0)
        merge[h - 1][rl] = make_float4(best.key, __int_as_float(best.idx), fb.key,
                                       __int_as_float(fb.idx));
      named_sync(1, 32 * kLmEpiWarps);
      if (h == 0) {
#pragma unroll
        for (int hh = 0; hh < 3; ++hh) {
          const float4 o = merge[hh][rl];
          offer_key(o.x, __float_as_int(o.y), best);
          offer_key(o.z, __float_as_int(o.w), fb);
        }
        const float bk = __shfl_xor_sync(0xffffffffu, best.key, 1);
        const int32_t bi = __shfl_xor_sync(0xffffffffu, best.idx, 1);
        const float fk = __shfl_xor_sync(0xffffffffu, fb.key, 1);
        const int32_t fi = __shfl_xor_sync(0xffffffffu, fb.idx, 1);
        offer_key(bk, bi, best);
        offer_key(fk, fi, fb);
        if (kind == 0 && row_ok) {
          unsigned long long* w = p.winners + (size_t(ci) * p.B + r) * 2;
          w[0] = best.idx >= 0 ? race_pack(best.key, best.idx) : 0ull;
          w[1] = fb.idx >= 0 ? race_pack(fb.key, fb.idx) : 0ull;
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, Sh::kTmemCols);
  }
}

// ---- host side --------------------------------------------------------------------------------
struct LmGeom {
  int32_t mb1, per1, tiles1;  // statistics GEMM: slot blocks, CTAs per block, vocabulary tiles
  int32_t mb2, per2, tiles2;  // race GEMM
};

bool lm_geom(int32_t B, int32_t gmax, int64_t V, LmGeom* g) {
  const int sms = device_sm_count();
  if (sms <= 0) return false;
  const int64_t slots1 = int64_t(B) * 2 * (gmax + 1);
  g->mb1 = static_cast<int32_t>((slots1 + kLmRows - 1) / kLmRows);
  g->tiles1 = static_cast<int32_t>((V + kLmStatsN - 1) / kLmStatsN);
  g->per1 = std::max(1, std::min(sms / std::max(1, g->mb1), g->tiles1));
  g->mb2 = static_cast<int32_t>((int64_t(2) * B + kLmRows - 1) / kLmRows);
  g->tiles2 = static_cast<int32_t>((V + kLmRaceN - 1) / kLmRaceN);
  g->per2 = std::max(1, std::min(sms / std::max(1, g->mb2), g->tiles2));
  return true;
}

struct LmWs {
  uint8_t* A1;            // [mb1 * 128][H] bf16
  uint8_t* A2;            // [mb2 * 128][H] bf16
  float4* partials;       // [B * gmax][per1]
  float2* tok;            // [B * gmax]
  RaceDesc* desc;         // [B]
  uint32_t* k0;           // [B]
  unsigned long long* winners;  // [per2][B][2]
  float4* cand;           // [B (gmax + 1)][per1][kLmParts][kLmCand]
  float* theta;           // [B (gmax + 1)][per1][kLmParts]
  unsigned long long* decided;  // [B]
  int32_t* pending;       // [B]
  int32_t* race_list;     // [B]
  int32_t* race_count;    // [1]
  uint32_t* cpub;         // [B (gmax + 1)]
  size_t total;
};

LmWs lm_layout(void* base, int32_t B, int32_t gmax, int64_t H, const LmGeom& g) {
  LmWs w;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    uint8_t* q = p + off;
    off = align256(off + bytes);
    return q;
  };
  const size_t units = size_t(B) * size_t(gmax > 0 ? gmax : 1);
  w.A1 = take(size_t(g.mb1) * kLmRows * size_t(H) * 2);
  w.A2 = take(size_t(g.mb2) * kLmRows * size_t(H) * 2);
  w.partials = reinterpret_cast<float4*>(take(sizeof(float4) * units * size_t(g.per1)));
  w.tok = reinterpret_cast<float2*>(take(sizeof(float2) * units));
  w.desc = reinterpret_cast<RaceDesc*>(take(sizeof(RaceDesc) * size_t(B)));
  w.k0 = reinterpret_cast<uint32_t*>(take(sizeof(uint32_t) * size_t(B)));
  w.winners = reinterpret_cast<unsigned long long*>(
      take(sizeof(unsigned long long) * 2 * size_t(B) * size_t(g.per2)));
  const size_t parts = size_t(B) * size_t(gmax + 1) * size_t(g.per1) * kLmParts;
  w.cand = reinterpret_cast<float4*>(take(sizeof(float4) * parts * kLmCand));
  w.theta = reinterpret_cast<float*>(take(sizeof(float) * parts));
  w.decided = reinterpret_cast<unsigned long long*>(take(sizeof(unsigned long long) * size_t(B)));
  w.pending = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * size_t(B)));
  w.race_list = reinterpret_cast<int32_t*>(take(sizeof(int32_t) * size_t(B)));
  w.race_count = reinterpret_cast<int32_t*>(take(sizeof(int32_t)));
  w.cpub = reinterpret_cast<uint32_t*>(take(sizeof(uint32_t) * size_t(B) * size_t(gmax + 1)));
  w.total = off;
  return w;
}

// A programmatic dependent launch: the kernel may start while the one before it finishes, and
// waits for it (griddepcontrol.wait) before touching its outputs.
template <typename... KArgs, typename... Args>
sv_status launch_pdl(void (*kernel)(KArgs...), int grid, int threads, size_t smem, cudaStream_t s,
                     Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return launch_status(cudaLaunchKernelEx(&cfg, kernel, args...));
}

template <int kN, bool kRace>
sv_status launch_lm_gemm(const CUtensorMap& map_a, const CUtensorMap& map_w, const LmParams& p,
                         cudaStream_t s) {
  using Sh = LmShape<kN>;
  auto* kern = lm_gemm_kernel<kN, kRace>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(Sh::kSmem)) != cudaSuccess)
    return SV_ERR_CUDA;
  return launch_pdl(kern, p.n_mblocks * p.per_mblock, kLmThreads, Sh::kSmem, s, map_a, map_w, p);
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" size_t spec_verify_lmhead_workspace_bytes(int32_t B, int32_t max_draft_len, int64_t V,
                                                     int64_t H) {
  LmGeom g;
  if (B <= 0 || max_draft_len < 0 || max_draft_len > SV_MAX_DRAFT_LEN || V <= 0 || H <= 0 ||
      !lm_geom(B, max_draft_len, V, &g))
    return 0;
  return lm_layout(nullptr, B, max_draft_len, H, g).total;
}

extern "C" sv_status spec_verify_lmhead(
    const void* target_hidden, const void* draft_hidden, int64_t ldh, const void* W, int64_t ldw,
    int64_t H, int64_t V, const int64_t* target_row0, const int64_t* draft_row0,
    const int32_t* draft_len, int32_t max_draft_len, const int32_t* draft_tokens, int32_t B,
    uint64_t seed, const uint64_t* request_ids, int32_t* accepted_len, int32_t* out_tokens,
    int64_t out_ld, int32_t* correction_token, float* accept_ratio, int32_t* recomputed,
    int32_t* status, void* workspace, size_t workspace_bytes, void* stream) {
  if (B < 0 || max_draft_len < 0 || max_draft_len > SV_MAX_DRAFT_LEN || V < 1 || H < 1)
    return SV_ERR_INVALID;
  if (H % 64 != 0 || V > (int64_t(1) << 31) - kLmStatsN) return SV_ERR_UNSUPPORTED;
  if (!target_hidden || !W || (max_draft_len > 0 && !draft_hidden)) return SV_ERR_INVALID;
  if (ldh < H || ldw < H) return SV_ERR_INVALID;
  if (ldh % 8 || ldw % 8 || !aligned16(target_hidden) || !aligned16(W) ||
      (draft_hidden && !aligned16(draft_hidden)))
    return SV_ERR_UNSUPPORTED;
  if (B == 0) return SV_OK;
  if (!target_row0 || !draft_len || !accepted_len || !out_tokens) return SV_ERR_INVALID;
  if (max_draft_len > 0 && (!draft_row0 || !draft_tokens)) return SV_ERR_INVALID;
  if (out_ld < int64_t(max_draft_len) + 1) return SV_ERR_INVALID;
  LmGeom g;
  if (!lm_geom(B, max_draft_len, V, &g)) return SV_ERR_CUDA;
  if (!workspace || !aligned256(workspace)) return SV_ERR_INVALID;
  const LmWs ws = lm_layout(workspace, B, max_draft_len, H, g);
  if (workspace_bytes < ws.total) return SV_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int32_t gmax = max_draft_len;

  // tensor maps: the two slot blocks [rows][H] and W [V][ldw], 64-element (128-byte) k-blocks
  CUtensorMap map_a1, map_a2, map_w1, map_w2;
  {
    const uint64_t dims[2] = {uint64_t(H), uint64_t(g.mb1) * kLmRows};
    const uint64_t strides[1] = {uint64_t(H) * 2};
    const uint32_t box[2] = {64, kLmRows};
    if (!make_map(&map_a1, ws.A1, 2, dims, strides, box)) return SV_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {uint64_t(H), uint64_t(g.mb2) * kLmRows};
    const uint64_t strides[1] = {uint64_t(H) * 2};
    const uint32_t box[2] = {64, kLmRows};
    if (!make_map(&map_a2, ws.A2, 2, dims, strides, box)) return SV_ERR_CUDA;
  }
  {
    const uint64_t dims[2] = {uint64_t(H), uint64_t(V)};
    const uint64_t strides[1] = {uint64_t(ldw) * 2};
    const uint32_t box1[2] = {64, kLmStatsN};
    const uint32_t box2[2] = {64, kLmRaceN};
    if (!make_map(&map_w1, W, 2, dims, strides, box1)) return SV_ERR_CUDA;
    if (!make_map(&map_w2, W, 2, dims, strides, box2)) return SV_ERR_CUDA;
  }

  profile_mark(0, s);
  const int64_t gather_warps = int64_t(B) * (2 * gmax + 1);
  lm_gather_kernel<<<unsigned((gather_warps + kGatherWarps - 1) / kGatherWarps),
                     32 * kGatherWarps, 0, s>>>(
      static_cast<const uint8_t*>(target_hidden), static_cast<const uint8_t*>(draft_hidden), ldh,
      H, target_row0, draft_row0, draft_len, B, gmax, ws.A1, ws.cpub, ws.race_count, status);
  sv_status st = launch_status(cudaGetLastError());
  if (st != SV_OK) return st;

  LmParams p = {};
  p.kblocks = static_cast<int32_t>(H / 64);
  p.V = V;
  p.B = B;
  p.gmax = gmax;
  p.draft_row0 = draft_row0;
  p.draft_len = draft_len;
  p.draft_tokens = draft_tokens;
  p.partials = ws.partials;
  p.tok = ws.tok;
  p.desc = ws.desc;
  p.seed = seed;
  p.request_ids = request_ids;
  p.k0 = ws.k0;
  p.winners = ws.winners;
  p.cand = ws.cand;
  p.theta = ws.theta;
  p.cpub = ws.cpub;
  p.race_count = ws.race_count;
  p.race_list = ws.race_list;
  p.status = status;
  {
    LmParams p1 = p;
    p1.n_mblocks = g.mb1;
    p1.per_mblock = g.per1;
    p1.n_tiles = g.tiles1;
    p1.slots = 2 * (gmax + 1);
    st = launch_lm_gemm<kLmStatsN, false>(map_a1, map_w1, p1, s);
    if (st != SV_OK) return st;
  }
  profile_mark(1, s);

  LmDecideParams dq = {};
  DecideParams& dp = dq.dp;
  dp.V = V;
  dp.target_row0 = target_row0;
  dp.draft_row0 = draft_row0;
  dp.draft_len = draft_len;
  dp.draft_tokens = draft_tokens;
  dp.B = B;
  dp.gmax = gmax;
  dp.C = g.per1;
  dp.seed = seed;
  dp.request_ids = request_ids;
  dp.ratio_out = accept_ratio;
  dp.ws.partials = ws.partials;
  dp.status = status;
  dp.tok = ws.tok;
  dq.A1 = ws.A1;
  dq.A2 = ws.A2;
  dq.row_bytes = H * 2;
  dq.desc = ws.desc;
  dq.k0 = ws.k0;
  dq.accepted_len = accepted_len;
  dq.cand = ws.cand;
  dq.theta = ws.theta;
  dq.C = g.per1;
  dq.decided = ws.decided;
  dq.pending = ws.pending;
  dq.race_count = ws.race_count;
  dq.race_list = ws.race_list;
  st = launch_pdl(lm_decide_kernel, B, kThreads, 0, s, dq);
  if (st != SV_OK) return st;
  profile_mark(2, s);

  {
    LmParams p2 = p;
    p2.n_mblocks = g.mb2;
    p2.per_mblock = g.per2;
    p2.n_tiles = g.tiles2;
    p2.slots = 2;
    st = launch_lm_gemm<kLmRaceN, true>(map_a2, map_w2, p2, s);
    if (st != SV_OK) return st;
  }
  st = launch_pdl(winners_finish_kernel<0>, (B + 127) / 128, 128, 0, s,
                  static_cast<const unsigned long long*>(ws.winners), g.per2, B,
                  static_cast<const int32_t*>(accepted_len), draft_row0, draft_tokens, out_tokens,
                  out_ld, correction_token, status, static_cast<const int32_t*>(ws.pending),
                  static_cast<const unsigned long long*>(ws.decided));
  if (st != SV_OK) return st;
  if (recomputed && cudaMemcpyAsync(recomputed, ws.race_count, sizeof(int32_t),
                                    cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return SV_ERR_CUDA;
  profile_mark(3, s);
  return launch_status(cudaGetLastError());
}
