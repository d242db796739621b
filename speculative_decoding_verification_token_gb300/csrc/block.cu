// block.cu -- block verification ("How much does a token cost", "Block verification": the
// running target-to-draft ratio starts at one, is capped at one after every step, every prefix is
// checked and the longest passing one kept; its thresholds and correction sampling are those of
// Sun et al. 2024, "Block Verification Accelerates Speculative Decoding").
//
// Four kernels on the caller's stream, each a programmatic dependent of the one before:
//   stream  the row-statistics stream of verify_kernels.cuh over every drafted row pair;
//   prep    one warp per request: the row normalisers, p_i(x_i)/q_i(x_i), the running ratios
//           rho_i = min(1, rho_{i-1} p_i(x_i)/q_i(x_i)) and the ACCEPT uniforms eta_i.  The
//           candidates are the positions i < gamma with eta_i <= rho_i (h_i <= rho_i, so no other
//           position can pass); since tau is the highest passing position they are tried from the
//           top, and the prep kernel lists for round 1 only the highest candidate of each request
//           whose position gamma fails (all of them when every h_i is asked for);
//   resid   two rounds, one CTA per row share of a listed position: R_i = sum_x max(rho_i
//           p_{i+1}(x) - q_{i+1}(x), 0), each share leaving a partial sum.  The last share of a
//           round-1 position forms h_i; if eta_i > h_i it lists the request's other candidates
//           for round 2;
//   race    verify_kernels.cuh's race in block mode: h_i = R_i / (R_i + 1 - rho_i), tau the
//           longest passing prefix, then the correction race over max(rho_tau p - q, 0) (or the
//           bonus race over the next target row).
#include "verify_kernels.cuh"

namespace sv {
namespace {

constexpr int kPrepWarps = 8;  // requests per prep CTA
constexpr int kResidCtasPerSm = 5;
constexpr int kResVecs = int(kResShareBytes / 16) / kThreads;  // vectors of a row per thread
static_assert(kResVecs * kThreads * 16 == int(kResShareBytes), "task not a whole multiple");

struct PrepParams {
  const uint8_t* target;
  const uint8_t* draft;
  int64_t V, ld;
  const int64_t* target_row0;
  const int64_t* draft_row0;
  const int32_t* draft_len;
  const int32_t* draft_tokens;
  int32_t B, gmax, C;
  uint64_t seed;
  const uint64_t* request_ids;
  int32_t all_rows;  // every h_i is asked for: list every i < gamma
  VerifyWs ws;
  int32_t* status;
};

// One warp per request.  Lane l takes positions l + 1, l + 33, ...: it merges its row pair's chunk
// partials into the normalisers and forms p(x)/q(x) of the drafted token and its uniform; lane 0
// then runs the running ratio along the positions (the order the definition fixes), and the lanes
// list their candidates (one atomic add per warp and row group).
template <typename E>
__global__ void __launch_bounds__(32 * kPrepWarps) block_prep_kernel(PrepParams p) {
  __shared__ float s_ratio[kPrepWarps][SV_MAX_DRAFT_LEN + 1];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the stream kernel's partials
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t r = blockIdx.x * kPrepWarps + warp;
  if (r >= p.B) return;
  const BlockWs& b = p.ws.blk;
  const int32_t graw = p.draft_len[r];
  const int32_t g = clamp_gamma(graw, p.gmax);
  const uint64_t req = p.request_ids ? p.request_ids[r] : uint64_t(r);
  const int64_t t0 = p.target_row0[r];
  const int64_t d0 = g > 0 ? p.draft_row0[r] : 0;
  bool bad = graw != g;
  for (int32_t i = lane + 1; i <= g; i += 32) {
    const int32_t unit = r * p.gmax + i - 1;
    const int32_t x = p.draft_tokens[d0 + i - 1];
    float tx = 0.f, dx = 0.f;
    if (x >= 0 && int64_t(x) < p.V) {
      tx = Elem<E>::load(row_ptr<E>(p.target, t0 + i - 1, p.ld), x);
      dx = Elem<E>::load(row_ptr<E>(p.draft, d0 + i - 1, p.ld), x);
    }
    float mt = kM2Empty, st = 0.f, md = kM2Empty, sd = 0.f;
    const float4* part = p.ws.partials + size_t(unit) * p.C;
    for (int32_t c = 0; c < p.C; ++c) {
      const float4 q = __ldcg(part + c);
      ms2_merge(mt, st, q.x, q.y);
      ms2_merge(md, sd, q.z, q.w);
    }
    const float4 nm = make_float4(mt, st, md, sd);
    bool bd;
    const float ratio = row_ratio(nm, x, p.V, tx, dx, bd);
    bad |= bd;
    b.norm[unit] = nm;
    b.eta[unit] = uniform_of(stream_block(make_stream(p.seed, req, i, kTagAccept), 0).x);
    s_ratio[warp][i] = ratio;
  }
  __syncwarp();
  if (lane == 0) {  // rho_i = min(1, rho_{i-1} ratio_i), left to right
    float rho = 1.f;
    for (int32_t i = 1; i <= g; ++i) {
      rho = rho > 0.f ? fminf(1.f, rho * s_ratio[warp][i]) : 0.f;
      s_ratio[warp][i] = rho;
    }
  }
  __syncwarp();
  // Candidates: positions i < gamma with eta_i <= rho_i (h_i <= rho_i, so the others fail whatever
  // R_i is).  tau is the highest passing position, so the positions are tried from the top: if
  // eta_gamma <= rho_gamma (h_gamma = rho_gamma) no residual mass is needed at all; otherwise round
  // 1 computes R of the highest candidate only, and round 2 the candidates below it if that one
  // fails.  When every h_i is asked for, round 1 computes them all.
  int32_t top = 0;  // highest candidate (top-down mode)
  for (int32_t base = 0; base < g; base += 32) {
    const int32_t i = base + lane + 1;
    bool cand = false;
    if (i <= g) {
      const int32_t unit = r * p.gmax + i - 1;
      const float rho = s_ratio[warp][i];
      b.rho[unit] = rho;
      b.cand[unit] = -1;
      cand = i < g && (p.all_rows || b.eta[unit] <= rho);
    }
    const uint32_t m = __ballot_sync(0xffffffffu, cand);
    if (m) top = base + 32 - __clz(m);
    if (p.all_rows) {  // list every candidate now
      int32_t first = 0;
      if (lane == 0 && m) first = atomicAdd(&b.count[0], __popc(m));
      first = __shfl_sync(0xffffffffu, first, 0);
      if (cand) {
        const int32_t slot = first + __popc(m & ((1u << lane) - 1u));
        b.cand[r * p.gmax + i - 1] = slot;
        b.unit[slot] = r * p.gmax + i - 1;
      }
    }
  }
  __syncwarp();  // the lanes' rho and cand stores before lane 0 reads and overwrites them
  if (!p.all_rows && lane == 0 && top > 0) {
    const int32_t unit_g = r * p.gmax + g - 1;
    if (!(b.eta[unit_g] <= b.rho[unit_g])) {  // position gamma fails: R_top decides next
      const int32_t slot = atomicAdd(&b.count[0], 1);
      const int32_t unit = r * p.gmax + top - 1;
      b.cand[unit] = slot;
      b.unit[slot] = unit;
      b.done[slot] = 0;
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) report(p.status, SV_ERR_BAD_INPUT);
}

// Residual terms of one 16-byte vector pair, in pairs of entries: max(a 2^(t log2e - m_t) -
// 2^(d log2e - m_d), 0) with a = rho s_d / s_t, i.e. s_d max(rho p(x) - q(x), 0).  Where rho p and q
// nearly cancel the difference loses its relative precision, but the sum R only needs absolute
// precision: each term carries the rounding of its two exponentials (ex2.approx, about 2^-22
// relative) and of the fma, so R (after the final 1 / s_d) is within about 3 * 2^-22 rho < 1e-6 of
// the exact residual mass.
__device__ __forceinline__ float2 resid_pair(float2 acc, float2 t, float2 d, float2 a,
                                             float2 nmt, float2 nmd) {
  const float2 et = exp2_2(fma2(t, splat2(kLog2e), nmt));
  const float2 ed = exp2_2(fma2(d, splat2(kLog2e), nmd));
  const float2 w = fma2(a, et, make_float2(-ed.x, -ed.y));
  return add2(acc, make_float2(fmaxf(w.x, 0.f), fmaxf(w.y, 0.f)));
}

template <typename E>
__device__ __forceinline__ float2 resid_vec(float2 acc, const uint4& t, const uint4& d, float2 a,
                                            float2 nmt, float2 nmd) {
  if constexpr (Elem<E>::kPerVec == 8) {
    acc = resid_pair(acc, bf16x2_f2(t.x), bf16x2_f2(d.x), a, nmt, nmd);
    acc = resid_pair(acc, bf16x2_f2(t.y), bf16x2_f2(d.y), a, nmt, nmd);
    acc = resid_pair(acc, bf16x2_f2(t.z), bf16x2_f2(d.z), a, nmt, nmd);
    acc = resid_pair(acc, bf16x2_f2(t.w), bf16x2_f2(d.w), a, nmt, nmd);
  } else {
    acc = resid_pair(acc, make_float2(__uint_as_float(t.x), __uint_as_float(t.y)),
                     make_float2(__uint_as_float(d.x), __uint_as_float(d.y)), a, nmt, nmd);
    acc = resid_pair(acc, make_float2(__uint_as_float(t.z), __uint_as_float(t.w)),
                     make_float2(__uint_as_float(d.z), __uint_as_float(d.w)), a, nmt, nmd);
  }
  return acc;
}

struct ResidParams {
  const uint8_t* target;
  const uint8_t* draft;
  int64_t V, ld;
  int32_t gmax;
  const int64_t* target_row0;
  const int64_t* draft_row0;
  int32_t top_down;  // round 1 lists the next candidates of the requests whose slot fails
  VerifyWs ws;
};

// Share s of slot c: one CTA.  Position i of request r (the slot's unit) needs R_i = sum_x
// max(rho_i p_{i+1}(x) - q_{i+1}(x), 0) over row pair i + 1.  Each thread loads its vectors of
// both rows before using any; the CTA's sum is the slot's partial for the share.
template <typename E>
__device__ void resid_share(const ResidParams& p, int32_t c, int32_t s, float* red) {
  constexpr int kPer = Elem<E>::kPerVec;
  const BlockWs& b = p.ws.blk;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int32_t unit = __ldcg(b.unit + c);
  const int32_t r = unit / p.gmax;
  const int32_t i = unit - r * p.gmax + 1;  // R_i: row pair i + 1, weight rho_i
  const float rho = __ldcg(b.rho + unit);
  const float4 nm = __ldcg(b.norm + unit + 1);
  const float2 a = splat2(rho * (nm.w / nm.y));
  const float2 nmt = splat2(-nm.x), nmd = splat2(-nm.z);
  const uint8_t* trow = row_ptr<E>(p.target, p.target_row0[r] + i, p.ld);
  const uint8_t* drow = row_ptr<E>(p.draft, p.draft_row0[r] + i, p.ld);
  const int64_t share = kResShareBytes / esize<E>();  // entries per task
  const int64_t lo = int64_t(s) * share;
  const int64_t hi = min(p.V, lo + share);
  const int32_t nvec = static_cast<int32_t>((hi - lo) / kPer);
  const uint4* vt = reinterpret_cast<const uint4*>(trow + lo * esize<E>());
  const uint4* vd = reinterpret_cast<const uint4*>(drow + lo * esize<E>());
  uint4 at[kResVecs], ad[kResVecs];
#pragma unroll
  for (int u = 0; u < kResVecs; ++u) {
    const int32_t v = tid + u * kThreads;
    if (v < nvec) {
      at[u] = __ldg(vt + v);
      ad[u] = __ldg(vd + v);
    }
  }
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int u = 0; u < kResVecs; ++u)
    if (tid + u * kThreads < nvec) acc = resid_vec<E>(acc, at[u], ad[u], a, nmt, nmd);
  for (int64_t e = lo + int64_t(nvec) * kPer + tid; e < hi; e += kThreads) {
    const float2 tt = make_float2(Elem<E>::load(trow, e), -INFINITY);
    const float2 dd = make_float2(Elem<E>::load(drow, e), -INFINITY);
    acc = resid_pair(acc, tt, dd, a, nmt, nmd);
  }
  const float sum = warp_sum(acc.x + acc.y);
  if (lane == 0) red[warp] = sum;
  __syncthreads();
  if (tid == 0) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) tot += red[w];
    b.rpart[size_t(c) * b.CLr + s] = tot / nm.w;
  }
}

// Round 1: one CTA per (slot, share) of the slots the prep kernel listed; CTAs past them exit.
// In top-down mode the last share of a slot forms h_i from the slot's partials; if eta_i > h_i the
// request's candidates below i are listed for round 2.
template <typename E>
__global__ void __launch_bounds__(kThreads, kResidCtasPerSm) block_resid1_kernel(ResidParams p) {
  __shared__ float red[kWarps];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the prep kernel's slots and state
  const BlockWs& b = p.ws.blk;
  const int64_t t = blockIdx.x;
  if (t >= int64_t(__ldcg(b.count)) * b.CLr) return;
  const int32_t c = static_cast<int32_t>(t / b.CLr);
  const int32_t s = static_cast<int32_t>(t - int64_t(c) * b.CLr);
  resid_share<E>(p, c, s, red);
  if (!p.top_down || threadIdx.x != 0) return;
  // release: this share's partial before its count; acquire (last share): every share's
  if (atom_add_acq_rel(reinterpret_cast<uint32_t*>(b.done + c), 1u) != uint32_t(b.CLr - 1)) return;
  const int32_t unit = __ldcg(b.unit + c);
  const float rho = __ldcg(b.rho + unit);
  if (__ldcg(b.eta + unit) <= block_threshold(b.rpart + size_t(c) * b.CLr, b.CLr, rho)) return;
  const int32_t r = unit / p.gmax;
  for (int32_t u = r * p.gmax; u < unit; ++u) {  // the candidates below, for round 2
    if (!(__ldcg(b.eta + u) <= __ldcg(b.rho + u))) continue;
    const int32_t slot = b.units + atomicAdd(&b.count[1], 1);
    b.cand[u] = slot;
    b.unit[slot] = u;
  }
}

// Round 2: every slot the round-1 kernel listed, CTAs walking the (slot, share) tasks.
template <typename E>
__global__ void __launch_bounds__(kThreads, kResidCtasPerSm) block_resid2_kernel(ResidParams p) {
  __shared__ float red[kWarps];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the round-1 kernel's slots
  const BlockWs& b = p.ws.blk;
  const int64_t n = int64_t(__ldcg(b.count + 1)) * b.CLr;
  for (int64_t t = blockIdx.x; t < n; t += gridDim.x) {
    const int32_t c = static_cast<int32_t>(t / b.CLr);
    resid_share<E>(p, b.units + c, static_cast<int32_t>(t - int64_t(c) * b.CLr), red);
    __syncthreads();
  }
}

template <typename E>
static sv_status run_block(const CommonArgs& a, const int64_t* target_row0,
                           const int64_t* draft_row0, const int32_t* draft_len,
                           const int32_t* draft_tokens, uint64_t seed,
                           const uint64_t* request_ids, int32_t* accepted_len,
                           int32_t* out_tokens, int64_t out_ld, int32_t* correction_token,
                           float* rho_out, float* h_out, int32_t* status, cudaStream_t stream) {
  const int32_t S = slices_of(a.V, esize<E>());
  const int32_t C = chunks_of(a.V, esize<E>());
  const VerifyWs ws = verify_layout(a.ws, a.B, a.gmax, a.V, esize<E>());
  const int sms = device_sm_count();
  if (sms <= 0) return SV_ERR_CUDA;
  const uint8_t* target = static_cast<const uint8_t*>(a.target);
  const uint8_t* draft = static_cast<const uint8_t*>(a.draft);
  // with rows to stream, the stream kernel clears the status word, the race slots and the
  // candidate count
  const bool stream_clears = int64_t(a.gmax) * a.B * C > 0;
  if (!stream_clears) {
    if ((status && cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess) ||
        cudaMemsetAsync(ws.slots, 0, sizeof(RaceSlot) * size_t(a.B), stream) != cudaSuccess ||
        cudaMemsetAsync(ws.blk.count, 0, 2 * sizeof(int32_t), stream) != cudaSuccess)
      return SV_ERR_CUDA;
  }
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;

  StreamParams sp = {};
  sp.target = target;
  sp.draft = draft;
  sp.V = a.V;
  sp.ld = a.ld;
  sp.target_row0 = target_row0;
  sp.draft_row0 = draft_row0;
  sp.draft_len = draft_len;
  sp.B = a.B;
  sp.gmax = a.gmax;
  sp.C = C;
  sp.ws = ws;
  sp.status = status;
  sp.clear_status = stream_clears ? 1 : 0;
  sp.claim = ws.claim;
  sp.claim_ready = ws.claim_ready;
  sp.call_id = next_call_id();
  sp.zero_words = ws.blk.count;  // the two rounds' slot counts
  sp.n_zero = 2;
  profile_mark(0, stream);
  sv_status st = launch_stream<E>(sp, stream);
  if (st != SV_OK) return st;
  profile_mark(1, stream);

  PrepParams pp = {};
  pp.target = target;
  pp.draft = draft;
  pp.V = a.V;
  pp.ld = a.ld;
  pp.target_row0 = target_row0;
  pp.draft_row0 = draft_row0;
  pp.draft_len = draft_len;
  pp.draft_tokens = draft_tokens;
  pp.B = a.B;
  pp.gmax = a.gmax;
  pp.C = C;
  pp.seed = seed;
  pp.request_ids = request_ids;
  pp.all_rows = h_out != nullptr;
  pp.ws = ws;
  pp.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((a.B + kPrepWarps - 1) / kPrepWarps));
  cfg.blockDim = dim3(32 * kPrepWarps);
  cfg.stream = stream;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, block_prep_kernel<E>, pp) != cudaSuccess) return SV_ERR_CUDA;

  ResidParams rp0 = {};
  rp0.target = target;
  rp0.draft = draft;
  rp0.V = a.V;
  rp0.ld = a.ld;
  rp0.gmax = a.gmax;
  rp0.target_row0 = target_row0;
  rp0.draft_row0 = draft_row0;
  rp0.top_down = h_out == nullptr;
  rp0.ws = ws;
  // round 1: one CTA per possible task (at most one slot per request in top-down mode); those past
  // the slots the prep kernel listed exit at once
  const int64_t slots1 = rp0.top_down ? int64_t(a.B) : int64_t(a.B) * std::max(0, a.gmax - 1);
  const int64_t tasks1 = slots1 * ws.blk.CLr;
  if (tasks1 >= (int64_t(1) << 31)) return SV_ERR_UNSUPPORTED;
  cfg.gridDim = dim3(unsigned(std::max<int64_t>(1, tasks1)));
  cfg.blockDim = dim3(kThreads);
  if (cudaLaunchKernelEx(&cfg, block_resid1_kernel<E>, rp0) != cudaSuccess) return SV_ERR_CUDA;
  // round 2 (top-down mode): every SM walks the listed tasks
  if (rp0.top_down && a.gmax > 2) {
    cfg.gridDim = dim3(unsigned(int64_t(sms) * kResidCtasPerSm));
    if (cudaLaunchKernelEx(&cfg, block_resid2_kernel<E>, rp0) != cudaSuccess) return SV_ERR_CUDA;
  }
  profile_mark(2, stream);

  RaceParams rp = {};
  rp.target = target;
  rp.draft = draft;
  rp.V = a.V;
  rp.ld = a.ld;
  rp.target_row0 = target_row0;
  rp.draft_row0 = draft_row0;
  rp.draft_tokens = draft_tokens;
  rp.B = a.B;
  rp.gmax = a.gmax;
  rp.S = S;
  rp.seed = seed;
  rp.request_ids = request_ids;
  rp.accepted_len = accepted_len;
  rp.out_tokens = out_tokens;
  rp.out_ld = out_ld;
  rp.correction_token = correction_token;
  rp.ws = ws;
  rp.status = status;
  rp.dp.draft_len = draft_len;
  rp.bd.norm = ws.blk.norm;
  rp.bd.rho = ws.blk.rho;
  rp.bd.eta = ws.blk.eta;
  rp.bd.cand = ws.blk.cand;
  rp.bd.rpart = ws.blk.rpart;
  rp.bd.CLr = ws.blk.CLr;
  rp.bd.rho_out = rho_out;
  rp.bd.h_out = h_out;
  st = launch_race<E, true>(rp, stream);
  if (st != SV_OK) return st;
  profile_mark(3, stream);
  return launch_status(cudaGetLastError());
}

}  // namespace
}  // namespace sv

using namespace sv;

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
  CommonArgs a{target_logits, draft_logits, dtype, V, ld, B, max_draft_len, workspace,
               workspace_bytes};
  sv_status st = check_common(a, true);
  if (st != SV_OK) return st;
  if (B == 0) return SV_OK;
  if (!target_row0 || !draft_len || !accepted_len || !out_tokens) return SV_ERR_INVALID;
  if (max_draft_len > 0 && (!draft_row0 || !draft_tokens)) return SV_ERR_INVALID;
  if (out_ld < int64_t(max_draft_len) + 1) return SV_ERR_INVALID;
  if (int64_t(B) * max_draft_len >= (int64_t(1) << 31)) return SV_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SV_BF16)
    return run_block<bf16_tag>(a, target_row0, draft_row0, draft_len, draft_tokens, seed,
                               request_ids, accepted_len, out_tokens, out_ld, correction_token,
                               running_ratio, h_threshold, status, s);
  return run_block<float>(a, target_row0, draft_row0, draft_len, draft_tokens, seed, request_ids,
                          accepted_len, out_tokens, out_ld, correction_token, running_ratio,
                          h_threshold, status, s);
}
