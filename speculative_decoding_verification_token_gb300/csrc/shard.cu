// shard.cu -- token-level verification with the vocabulary split across ranks (tensor
// parallelism over the vocabulary, as in the vocabulary-parallel serving of "How much does a
// token cost", "Experiments").  Rank k holds columns [v_off_k, v_off_k + Vs_k) of every logit row.
// Softmax statistics and exponential races both decompose over a split of the vocabulary:
//   - the statistics (m, s) of a row are the log-sum-exp merge of its shards' statistics;
//   - the race winner of a row is the largest of its shards' winners, every entry keyed with the
//     uniform of its global vocabulary index.
// So a round is four calls with two exchanges between ranks (the caller's all-gathers):
//   stats   this shard's statistics of every drafted row pair, and the drafted token's two logits
//           where the token lies in the shard (-inf otherwise);            -> exchange
//   merge   every rank merges the gathered statistics in shard order (the same result on every
//           rank) and takes the drafted tokens' logits from the shard that holds them;
//   race    every rank decides every request (identically) and races its shard of the correction
//           (or bonus) row; per request it leaves the shard's best (key, global index), and, if the
//           shard holds no positive residual entry, its best for the race over p;   -> exchange
//   finish  the largest winner over the shards (the race over p if no shard had a residual entry)
//           and the request's outputs.
#include "verify_kernels.cuh"

namespace sv {
namespace {

constexpr int kShardWarps = 8;

// Per drafted row pair: the chunk partials merged into the shard's statistics, and the drafted
// token's two logits if the shard holds the token (else -inf).  One warp per request.
struct ShardStatsParams {
  const uint8_t* target;
  const uint8_t* draft;
  int64_t Vs, ld, v_off;
  const int64_t* target_row0;
  const int64_t* draft_row0;
  const int32_t* draft_len;
  const int32_t* draft_tokens;
  int32_t B, gmax, C;
  const float4* partials;
  float4* stats;   // [B * gmax]
  float2* tok;     // [B * gmax]
  int32_t* status;
};

template <typename E>
__global__ void __launch_bounds__(32 * kShardWarps) shard_stats_kernel(ShardStatsParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the stream kernel's partials
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int32_t r = blockIdx.x * kShardWarps + warp;
  if (r >= p.B) return;
  const int32_t graw = p.draft_len[r];
  const int32_t g = clamp_gamma(graw, p.gmax);
  if (graw != g && lane == 0) report(p.status, SV_ERR_BAD_INPUT);
  for (int32_t i = lane + 1; i <= g; i += 32) {
    const int32_t unit = r * p.gmax + i - 1;
    float mt = kM2Empty, st = 0.f, md = kM2Empty, sd = 0.f;
    for (int32_t c = 0; c < p.C; ++c) {
      const float4 q = __ldcg(p.partials + size_t(unit) * p.C + c);
      ms2_merge(mt, st, q.x, q.y);
      ms2_merge(md, sd, q.z, q.w);
    }
    p.stats[unit] = make_float4(mt, st, md, sd);
    const int64_t drow = p.draft_row0[r] + (i - 1);
    const int64_t x = int64_t(p.draft_tokens[drow]) - p.v_off;
    float2 v = make_float2(-INFINITY, -INFINITY);
    if (x >= 0 && x < p.Vs)
      v = make_float2(Elem<E>::load(row_ptr<E>(p.target, p.target_row0[r] + (i - 1), p.ld), x),
                      Elem<E>::load(row_ptr<E>(p.draft, drow, p.ld), x));
    p.tok[unit] = v;
  }
}

// Shard statistics merged in shard order, drafted-token logits from the shard that has them.
__global__ void shard_merge_kernel(const float4* stats_all, const float2* tok_all, int32_t n,
                                   int64_t units, float4* stats_out, float2* tok_out) {
  const int64_t u = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (u >= units) return;
  float mt = kM2Empty, st = 0.f, md = kM2Empty, sd = 0.f;
  float2 tk = make_float2(-INFINITY, -INFINITY);
  for (int32_t k = 0; k < n; ++k) {
    const float4 q = stats_all[size_t(k) * units + u];
    ms2_merge(mt, st, q.x, q.y);
    ms2_merge(md, sd, q.z, q.w);
    const float2 v = tok_all[size_t(k) * units + u];
    tk.x = fmaxf(tk.x, v.x);
    tk.y = fmaxf(tk.y, v.y);
  }
  stats_out[u] = make_float4(mt, st, md, sd);
  tok_out[u] = tk;
}

bool shard_args_ok(const CommonArgs& a, int64_t v_off, int64_t V_total) {
  return v_off >= 0 && v_off % 8 == 0 && V_total >= v_off + a.V && V_total < (int64_t(1) << 31);
}

template <typename E>
sv_status run_shard_stats(const CommonArgs& a, int64_t v_off, const int64_t* target_row0,
                          const int64_t* draft_row0, const int32_t* draft_len,
                          const int32_t* draft_tokens, float* stats, float* tok, int32_t* status,
                          cudaStream_t stream) {
  const int32_t C = chunks_of(a.V, esize<E>());
  const VerifyWs ws = verify_layout(a.ws, a.B, a.gmax, a.V, esize<E>());
  const bool stream_clears = int64_t(a.gmax) * a.B * C > 0;
  if (status && !stream_clears &&
      cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  StreamParams sp = {};
  sp.target = static_cast<const uint8_t*>(a.target);
  sp.draft = static_cast<const uint8_t*>(a.draft);
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
  sv_status st = launch_stream<E>(sp, stream);
  if (st != SV_OK) return st;
  ShardStatsParams pp;
  pp.target = sp.target;
  pp.draft = sp.draft;
  pp.Vs = a.V;
  pp.ld = a.ld;
  pp.v_off = v_off;
  pp.target_row0 = target_row0;
  pp.draft_row0 = draft_row0;
  pp.draft_len = draft_len;
  pp.draft_tokens = draft_tokens;
  pp.B = a.B;
  pp.gmax = a.gmax;
  pp.C = C;
  pp.partials = ws.partials;
  pp.stats = reinterpret_cast<float4*>(stats);
  pp.tok = reinterpret_cast<float2*>(tok);
  pp.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((a.B + kShardWarps - 1) / kShardWarps));
  cfg.blockDim = dim3(32 * kShardWarps);
  cfg.stream = stream;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  return launch_status(cudaLaunchKernelEx(&cfg, shard_stats_kernel<E>, pp));
}

template <typename E>
sv_status run_shard_race(const CommonArgs& a, int64_t v_off, int64_t V_total,
                         const int64_t* target_row0, const int64_t* draft_row0,
                         const int32_t* draft_len, const int32_t* draft_tokens, uint64_t seed,
                         const uint64_t* request_ids, const float* stats, const float* tok,
                         int32_t* accepted_len, float* ratio_out, unsigned long long* winners,
                         int32_t* status, cudaStream_t stream) {
  const VerifyWs ws = verify_layout(a.ws, a.B, a.gmax, a.V, esize<E>());
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  if (cudaMemsetAsync(ws.slots, 0, sizeof(RaceSlot) * size_t(a.B), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  RaceParams rp = {};
  rp.target = static_cast<const uint8_t*>(a.target);
  rp.draft = static_cast<const uint8_t*>(a.draft);
  rp.V = a.V;
  rp.ld = a.ld;
  rp.target_row0 = target_row0;
  rp.draft_row0 = draft_row0;
  rp.draft_tokens = draft_tokens;
  rp.B = a.B;
  rp.gmax = a.gmax;
  rp.S = slices_of(a.V, esize<E>());
  rp.seed = seed;
  rp.request_ids = request_ids;
  rp.accepted_len = accepted_len;
  rp.ws = ws;
  rp.status = status;
  rp.v_off = v_off;
  rp.winners = winners;
  DecideParams& dp = rp.dp;
  dp.target = rp.target;
  dp.draft = rp.draft;
  dp.V = V_total;  // the drafted tokens are checked against the whole vocabulary
  dp.ld = a.ld;
  dp.target_row0 = target_row0;
  dp.draft_row0 = draft_row0;
  dp.draft_len = draft_len;
  dp.draft_tokens = draft_tokens;
  dp.B = a.B;
  dp.gmax = a.gmax;
  dp.C = 1;  // the merged statistics: one "partial" per row pair
  dp.seed = seed;
  dp.request_ids = request_ids;
  dp.ratio_out = ratio_out;
  dp.ws = ws;
  dp.ws.partials = const_cast<float4*>(reinterpret_cast<const float4*>(stats));
  dp.status = status;
  dp.tok = reinterpret_cast<const float2*>(tok);
  return launch_race<E, false>(rp, stream);
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status spec_verify_shard_stats(const void* target_logits, const void* draft_logits,
                                             sv_dtype dtype, int64_t Vs, int64_t ld,
                                             int64_t v_off, int64_t V_total,
                                             const int64_t* target_row0,
                                             const int64_t* draft_row0, const int32_t* draft_len,
                                             int32_t max_draft_len, const int32_t* draft_tokens,
                                             int32_t B, float* row_stats, float* token_logits,
                                             int32_t* status, void* workspace,
                                             size_t workspace_bytes, void* stream) {
  CommonArgs a{target_logits, draft_logits, dtype, Vs, ld, B, max_draft_len, workspace,
               workspace_bytes};
  sv_status st = check_common(a, true);
  if (st != SV_OK) return st;
  if (!shard_args_ok(a, v_off, V_total)) return SV_ERR_INVALID;
  if (B == 0 || max_draft_len == 0) return SV_OK;
  if (!target_row0 || !draft_row0 || !draft_len || !draft_tokens || !row_stats || !token_logits)
    return SV_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SV_BF16)
    return run_shard_stats<bf16_tag>(a, v_off, target_row0, draft_row0, draft_len, draft_tokens,
                                     row_stats, token_logits, status, s);
  return run_shard_stats<float>(a, v_off, target_row0, draft_row0, draft_len, draft_tokens,
                                row_stats, token_logits, status, s);
}

extern "C" sv_status spec_verify_shard_merge(const float* row_stats_all,
                                             const float* token_logits_all, int32_t n_shards,
                                             int64_t rows, float* row_stats,
                                             float* token_logits, void* stream) {
  if (n_shards < 1 || rows < 0) return SV_ERR_INVALID;
  if (rows == 0) return SV_OK;
  if (!row_stats_all || !token_logits_all || !row_stats || !token_logits) return SV_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  shard_merge_kernel<<<unsigned((rows + 255) / 256), 256, 0, s>>>(
      reinterpret_cast<const float4*>(row_stats_all),
      reinterpret_cast<const float2*>(token_logits_all), n_shards, rows,
      reinterpret_cast<float4*>(row_stats), reinterpret_cast<float2*>(token_logits));
  return launch_status(cudaGetLastError());
}

extern "C" sv_status spec_verify_shard_race(const void* target_logits, const void* draft_logits,
                                            sv_dtype dtype, int64_t Vs, int64_t ld, int64_t v_off,
                                            int64_t V_total, const int64_t* target_row0,
                                            const int64_t* draft_row0, const int32_t* draft_len,
                                            int32_t max_draft_len, const int32_t* draft_tokens,
                                            int32_t B, uint64_t seed, const uint64_t* request_ids,
                                            const float* row_stats, const float* token_logits,
                                            int32_t* accepted_len, float* accept_ratio,
                                            uint64_t* winners, int32_t* status, void* workspace,
                                            size_t workspace_bytes, void* stream) {
  CommonArgs a{target_logits, draft_logits, dtype, Vs, ld, B, max_draft_len, workspace,
               workspace_bytes};
  sv_status st = check_common(a, true);
  if (st != SV_OK) return st;
  if (!shard_args_ok(a, v_off, V_total)) return SV_ERR_INVALID;
  if (B == 0) return SV_OK;
  if (!target_row0 || !draft_len || !accepted_len || !winners) return SV_ERR_INVALID;
  if (max_draft_len > 0 && (!draft_row0 || !draft_tokens || !row_stats || !token_logits))
    return SV_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto* w = reinterpret_cast<unsigned long long*>(winners);
  if (dtype == SV_BF16)
    return run_shard_race<bf16_tag>(a, v_off, V_total, target_row0, draft_row0, draft_len,
                                    draft_tokens, seed, request_ids, row_stats, token_logits,
                                    accepted_len, accept_ratio, w, status, s);
  return run_shard_race<float>(a, v_off, V_total, target_row0, draft_row0, draft_len,
                               draft_tokens, seed, request_ids, row_stats, token_logits,
                               accepted_len, accept_ratio, w, status, s);
}

extern "C" sv_status spec_verify_shard_finish(const uint64_t* winners_all, int32_t n_shards,
                                              int32_t B, const int32_t* accepted_len,
                                              const int64_t* draft_row0,
                                              const int32_t* draft_tokens, int32_t* out_tokens,
                                              int64_t out_ld, int32_t* correction_token,
                                              int32_t* status, void* stream) {
  if (n_shards < 1 || B < 0 || out_ld < 1) return SV_ERR_INVALID;
  if (B == 0) return SV_OK;
  if (!winners_all || !accepted_len || !out_tokens) return SV_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return SV_ERR_CUDA;
  winners_finish_kernel<<<unsigned((B + 127) / 128), 128, 0, s>>>(
      reinterpret_cast<const unsigned long long*>(winners_all), n_shards, B, accepted_len,
      draft_row0, draft_tokens, out_tokens, out_ld, correction_token, status);
  return launch_status(cudaGetLastError());
}
