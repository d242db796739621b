// token.cu -- token-level verification ("Speculative Decoding: The Same Distribution, Twice as
// Fast" §3-§4; "How much does a token cost", "On Speculative Sampling").
//
// Two kernels on the caller's stream (verify_kernels.cuh): the stream kernel folds every drafted
// row pair into softmax-statistics partials; the race kernel, a programmatic dependent of it,
// decides each request (row normalisers, p(x)/q(x) of each drafted token, the ACCEPT uniforms,
// the first rejection) and races its correction token from max(p - q, 0), or its bonus token from
// the next target row when every draft was accepted.
#include "verify_kernels.cuh"

namespace sv {
namespace {

template <typename E>
static sv_status run_token(const CommonArgs& a, const int64_t* target_row0,
                           const int64_t* draft_row0, const int32_t* draft_len,
                           const int32_t* draft_tokens, uint64_t seed,
                           const uint64_t* request_ids, int32_t* accepted_len,
                           int32_t* out_tokens, int64_t out_ld, int32_t* correction_token,
                           float* ratio_out, int32_t* status, cudaStream_t stream) {
  const int32_t S = slices_of(a.V, esize<E>());
  const int32_t C = chunks_of(a.V, esize<E>());
  const VerifyWs ws = verify_layout(a.ws, a.B, a.gmax, a.V, esize<E>());
  // with rows to stream, the stream kernel clears the status word and the race slots
  const bool stream_clears = int64_t(a.gmax) * a.B * C > 0;
  if (status && !stream_clears &&
      cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  const uint8_t* target = static_cast<const uint8_t*>(a.target);
  const uint8_t* draft = static_cast<const uint8_t*>(a.draft);

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
  sp.zero_words = nullptr;
  sp.n_zero = 0;
  profile_mark(0, stream);
  sv_status st = launch_stream<E>(sp, stream);
  if (st != SV_OK) return st;
  if (!stream_clears &&  // no stream launch: the race slots are zeroed here instead
      cudaMemsetAsync(ws.slots, 0, sizeof(RaceSlot) * size_t(a.B), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  profile_mark(1, stream);  // the race kernel decides (no kernel in between)
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
  DecideParams& dp = rp.dp;
  dp.target = target;
  dp.draft = draft;
  dp.V = a.V;
  dp.ld = a.ld;
  dp.target_row0 = target_row0;
  dp.draft_row0 = draft_row0;
  dp.draft_len = draft_len;
  dp.draft_tokens = draft_tokens;
  dp.B = a.B;
  dp.gmax = a.gmax;
  dp.C = C;
  dp.seed = seed;
  dp.request_ids = request_ids;
  dp.ratio_out = ratio_out;
  dp.ws = ws;
  dp.status = status;
  st = launch_race<E, false>(rp, stream);
  if (st != SV_OK) return st;
  profile_mark(3, stream);
  return launch_status(cudaGetLastError());
}

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" sv_status spec_verify_token(const void* target_logits, const void* draft_logits,
                                       sv_dtype dtype, int64_t V, int64_t ld,
                                       const int64_t* target_row0, const int64_t* draft_row0,
                                       const int32_t* draft_len, int32_t max_draft_len,
                                       const int32_t* draft_tokens, int32_t B, uint64_t seed,
                                       const uint64_t* request_ids, int32_t* accepted_len,
                                       int32_t* out_tokens, int64_t out_ld,
                                       int32_t* correction_token, float* accept_ratio,
                                       int32_t* status, void* workspace, size_t workspace_bytes,
                                       void* stream) {
  CommonArgs a{target_logits, draft_logits, dtype, V, ld, B, max_draft_len, workspace,
               workspace_bytes};
  sv_status st = check_common(a, true);
  if (st != SV_OK) return st;
  if (B == 0) return SV_OK;
  if (!target_row0 || !draft_len || !accepted_len || !out_tokens) return SV_ERR_INVALID;
  if (max_draft_len > 0 && (!draft_row0 || !draft_tokens)) return SV_ERR_INVALID;
  if (out_ld < int64_t(max_draft_len) + 1) return SV_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SV_BF16)
    return run_token<bf16_tag>(a, target_row0, draft_row0, draft_len, draft_tokens, seed,
                               request_ids, accepted_len, out_tokens, out_ld, correction_token,
                               accept_ratio, status, s);
  return run_token<float>(a, target_row0, draft_row0, draft_len, draft_tokens, seed, request_ids,
                          accepted_len, out_tokens, out_ld, correction_token, accept_ratio,
                          status, s);
}
