// verify.cu -- draft sampling from q, the verification workspace query and the allocation-free
// token-level entry point (token-level verification is in token.cu, block verification in
// block.cu).
//
// Draft sampling ("Speculative Decoding: The Same Distribution, Twice as Fast" §3 step 1) races
// every drafted row from its own softmax, one row split into contiguous shares over a few CTAs.
// The allocation-free token-level entry point closes the file.
#include <mutex>

#include <cuda.h>

#include "verify_common.cuh"

namespace sv {

constexpr int kRaceSplitMax = 8;                 // CTAs (row shares) per race job, many jobs
constexpr int kRaceSplitFew = 16;                // the same when one wave holds every share
constexpr int kRaceCtasPerSm = 4;                // resident race CTAs per SM (launch bounds)
constexpr uint32_t kRaceShareMax = 64 * 1024;    // largest row share staged in shared memory

// ---------------------------------------------------------------------------------------------
// sample: CL CTAs per drafted row -- the drafted token raced from q (DRAFT tag)
// ---------------------------------------------------------------------------------------------
struct SampleParams {
  const uint8_t* draft;
  int64_t V, ld;
  const int64_t* draft_row0;
  const int32_t* draft_len;
  int32_t B, gmax, CL;      // requests, largest drafted length, CTAs (row shares) per row
  uint64_t seed;
  const uint64_t* request_ids;
  int32_t* sampled_tokens;  // indexed like the draft rows
  RaceSlot* slots;          // one per (request, position), zeroed before the launch
  int32_t* status;
  int32_t stage_share;      // the launch provides dynamic shared memory for the row share
};

template <typename E>
__global__ void __launch_bounds__(kThreads, kRaceCtasPerSm) sample_kernel(SampleParams p) {
  extern __shared__ __align__(128) uint8_t share_sm[];  // this CTA's share of the row (staged)
  __shared__ uint64_t share_bar;
  __shared__ float red_k[kWarps];
  __shared__ int32_t red_i[kWarps];
  __shared__ int32_t s_last;
  __shared__ int32_t s_winner;
  __shared__ float s_k0;
  const int tid = threadIdx.x;
  const int32_t job = blockIdx.x / p.CL;
  const int32_t part = blockIdx.x - job * p.CL;  // this CTA's share of the job's row
  const int32_t r = job / p.gmax;
  const int32_t pos = job - r * p.gmax + 1;
  const int32_t g = p.draft_len[r];
  if (g < 0 || g > p.gmax) {
    if (tid == 0 && part == 0 && pos == 1) report(p.status, SV_ERR_BAD_INPUT);
    return;
  }
  if (pos > g) return;
  RaceSpec rs;
  rs.resid = false;
  rs.gap = 0.f;
  const int64_t sample_row = p.draft_row0[r] + (pos - 1);
  const uint8_t* trow = row_ptr<E>(p.draft, sample_row, p.ld);
  const uint64_t req = p.request_ids ? p.request_ids[r] : uint64_t(r);
  rs.st = make_stream(p.seed, req, pos, kTagDraft);

  // this CTA's share of the row: a contiguous range, a whole number of 16-byte vectors long
  constexpr int32_t kPer = Elem<E>::kPerVec;
  const int64_t share = (p.V + int64_t(p.CL) * kPer - 1) / (int64_t(p.CL) * kPer) * kPer;
  const int64_t lo = min(p.V, int64_t(part) * share);
  const int64_t hi = min(p.V, lo + share);

  // stage the share's whole 16-byte vectors in shared memory with one bulk copy (shares too
  // large for it are read from global memory); a ragged tail is read from global memory
  const uint32_t vec_bytes = static_cast<uint32_t>(((hi - lo) * esize<E>()) & ~int64_t(15));
  const bool staged = p.stage_share && vec_bytes > 0;
  if (tid == 0 && staged) {
    mbar_init(&share_bar, 1);
    fence_barrier_init();
    mbar_expect_tx(&share_bar, vec_bytes);
    bulk_g2s(share_sm, trow + lo * esize<E>(), vec_bytes, &share_bar);
  }
  __syncthreads();
  const uint4* gsrc = reinterpret_cast<const uint4*>(trow + lo * esize<E>());

  // seed: the best exact key among the threads' largest-logit entries, raised to the best seed
  // the row's other shares have published so far -- a lower bound on the winning key, against
  // which the main pass gates.  It reads the share from global memory (L2) while the bulk copy
  // stages it for the main pass.
  RaceSlot* slot = p.slots + job;
  float seed = seed_range<E>(rs, gsrc, trow, nullptr, lo, int32_t(hi - lo));
  if (staged) mbar_wait(&share_bar, 0, p.status);
  const uint4* vsrc = staged ? reinterpret_cast<const uint4*>(share_sm) : gsrc;
  seed = block_max(seed, red_k);
  if (tid == 0) {
    const uint32_t prev = atomicMax(&slot->k0, key_order(seed));
    s_k0 = fmaxf(seed, key_from_order(prev));
  }
  __syncthreads();
  const float K0 = s_k0;

  // main pass: only entries whose logit and noise can reach K0 are keyed
  float bk = -INFINITY;
  int32_t bi = -1;
  if (staged) race_range<E>(rs, vsrc, trow, nullptr, lo, int32_t(hi - lo), K0, bk, bi);
  else race_range<E, kBatchGlobal>(rs, vsrc, trow, nullptr, lo, int32_t(hi - lo), K0, bk, bi);
  block_race(bk, bi, red_k, red_i);

  // combine the shares: a 64-bit max over (order-preserving key bits, ~index), so equal keys go
  // to the lower index; the last share to arrive writes the token
  if (tid == 0) {
    if (bi >= 0) atomicMax(&slot->best, race_pack(bk, bi));
    // release: this share's maximum before its count; acquire (last share): every share's
    s_last = atom_add_acq_rel(&slot->count, 1u) == uint32_t(p.CL - 1);
  }
  __syncthreads();
  if (!s_last) return;
  if (tid == 0) {
    const unsigned long long best = atomicAdd(&slot->best, 0ull);
    s_winner = best ? race_unpack_index(best) : -1;
    if (s_winner < 0) report(p.status, SV_ERR_BAD_INPUT);  // the row carries no probability
    p.sampled_tokens[sample_row] = s_winner;
  }
}

// ---------------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------------
// CTAs per sampled row for rows of S 16 KB slices: each owns one contiguous share of the row.
// Shares per row: as many as one wave of resident sampler CTAs holds (up to kRaceSplitFew), so
// that every row's shares run at once and no CTA pays the seed and combine latencies twice; at
// least one share per row (then several waves).
static int32_t race_split(int32_t S, int64_t jobs) {
  int32_t cl = kRaceSplitMax;
  const int sms = device_sm_count();
  if (sms > 0 && jobs > 0) {
    const int64_t slots = int64_t(sms) * kRaceCtasPerSm;
    cl = int32_t(std::max<int64_t>(1, std::min<int64_t>(kRaceSplitFew, slots / jobs)));
  }
  return std::max(1, std::min(cl, S));
}

template <typename E>
static sv_status run_sample(const CommonArgs& a, const int64_t* draft_row0,
                            const int32_t* draft_len, uint64_t seed, const uint64_t* request_ids,
                            int32_t* draft_tokens, int32_t* status, cudaStream_t stream) {
  const int32_t S = slices_of(a.V, esize<E>());
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  SampleParams sp = {};
  sp.draft = static_cast<const uint8_t*>(a.draft);
  sp.V = a.V;
  sp.ld = a.ld;
  sp.draft_row0 = draft_row0;
  sp.draft_len = draft_len;
  sp.B = a.B;
  sp.gmax = a.gmax;
  sp.seed = seed;
  sp.request_ids = request_ids;
  sp.sampled_tokens = draft_tokens;
  sp.status = status;
  sp.slots = verify_layout(a.ws, a.B, a.gmax, a.V, esize<E>()).slots;
  const int64_t jobs = int64_t(a.B) * a.gmax;
  if (jobs == 0) return SV_OK;
  if (cudaMemsetAsync(sp.slots, 0, sizeof(RaceSlot) * size_t(jobs), stream) != cudaSuccess)
    return SV_ERR_CUDA;
  sp.CL = race_split(S, jobs);
  // the kernel's share: ceil(V / (CL * kPer)) whole vectors
  constexpr int64_t kPer = Elem<E>::kPerVec;
  const int64_t share_bytes = (sp.V + sp.CL * kPer - 1) / (sp.CL * kPer) * 16;
  sp.stage_share = share_bytes <= int64_t(kRaceShareMax);
  const size_t smem = sp.stage_share ? size_t(share_bytes) : 0;
  if (cudaFuncSetAttribute(sample_kernel<E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(kRaceShareMax)) != cudaSuccess)
    return SV_ERR_CUDA;
  sample_kernel<E><<<unsigned(jobs * sp.CL), kThreads, smem, stream>>>(sp);
  return launch_status(cudaGetLastError());
}

}  // namespace sv

using namespace sv;

extern "C" size_t spec_verify_workspace_bytes(int32_t B, int32_t max_draft_len, int64_t V,
                                              sv_dtype dtype) {
  if (B < 0 || max_draft_len < 0 || max_draft_len > SV_MAX_DRAFT_LEN || V <= 0) return 0;
  if (dtype != SV_F32 && dtype != SV_BF16) return 0;
  return verify_ws_bytes(B, max_draft_len, V, elem_bytes(dtype));
}

extern "C" sv_status spec_sample_draft(const void* draft_logits, sv_dtype dtype, int64_t V,
                                       int64_t ld, const int64_t* draft_row0,
                                       const int32_t* draft_len, int32_t max_draft_len, int32_t B,
                                       uint64_t seed, const uint64_t* request_ids,
                                       int32_t* draft_tokens, int32_t* status, void* workspace,
                                       size_t workspace_bytes, void* stream) {
  CommonArgs a{nullptr, draft_logits, dtype, V, ld, B, max_draft_len, workspace, workspace_bytes};
  sv_status st = check_common(a, false);
  if (st != SV_OK) return st;
  if (B == 0 || max_draft_len == 0) return SV_OK;
  if (!draft_row0 || !draft_len || !draft_tokens) return SV_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dtype == SV_BF16)
    return run_sample<bf16_tag>(a, draft_row0, draft_len, seed, request_ids, draft_tokens, status,
                                s);
  return run_sample<float>(a, draft_row0, draft_len, seed, request_ids, draft_tokens, status, s);
}

// ---------------------------------------------------------------------------------------------
// spec_verify_token_noalloc: token-level verification with scratch memory owned by the library.
//
// Some callers cannot allocate device memory at all: a plugin that is handed only its input and
// output buffers by a host engine that owns every device allocation, or a serving loop that must
// not call cudaMalloc because a device allocation can implicitly synchronise the device.  For
// them the scratch memory of the verify kernels lives in the file-scope array below, which every
// GPU that loads this library holds until the process exits.
// ---------------------------------------------------------------------------------------------
namespace sv {

constexpr size_t kNoAllocScratchBytes = SV_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Unique id of the CUDA context current on the calling thread, or 0 if there is none yet or the
// driver cannot be asked.  The two driver calls are reached through the runtime's entry-point
// query, so the library needs no link against the driver library.  Context ids are never reused
// within a process, unlike context handles.
static unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_noalloc_scratch in the current context.  In host code the array's name is
// a host-side stand-in, not a device address, so the address is looked up with the context
// current and cached by context id: a device reset or another context (a driver-API context of
// an engine, say) gets a lookup of its own instead of a stale address.  Without a context id
// (no driver entry points) every call looks the address up again.
static sv_status noalloc_scratch_address(void** out) {
  constexpr int kSlots = 64;
  static std::mutex mu;
  static unsigned long long ids[kSlots] = {};
  static void* addr[kSlots] = {};
  static int next = 0;
  std::lock_guard<std::mutex> lock(mu);
  unsigned long long id = current_context_id();
  if (id != 0)
    for (int k = 0; k < kSlots; ++k)
      if (ids[k] == id) {
        *out = addr[k];
        return SV_OK;
      }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
    return SV_ERR_CUDA;
  id = current_context_id();  // the lookup made the runtime's context current if none was
  if (id != 0) {
    ids[next] = id;
    addr[next] = p;
    next = (next + 1) % kSlots;
  }
  *out = p;
  return SV_OK;
}

}  // namespace sv

extern "C" sv_status spec_verify_token_noalloc(
    const void* target_logits, const void* draft_logits, sv_dtype dtype, int64_t V, int64_t ld,
    const int64_t* target_row0, const int64_t* draft_row0, const int32_t* draft_len,
    int32_t max_draft_len, const int32_t* draft_tokens, int32_t B, uint64_t seed,
    const uint64_t* request_ids, int32_t* accepted_len, int32_t* out_tokens, int64_t out_ld,
    int32_t* correction_token, float* accept_ratio, int32_t* status, void* stream) {
  const size_t need = spec_verify_workspace_bytes(B, max_draft_len, V, dtype);
  if (need == 0) return SV_ERR_INVALID;
  if (need > sv::kNoAllocScratchBytes) return SV_ERR_UNSUPPORTED;  // batch too large for it
  void* scratch = nullptr;
  const sv_status st = sv::noalloc_scratch_address(&scratch);
  if (st != SV_OK) return st;
  // The verify kernels never read scratch they have not written earlier in the same call; the
  // only counters (race tickets) are cleared by the call's first kernel before the race kernel
  // runs.
  return spec_verify_token(target_logits, draft_logits, dtype, V, ld, target_row0, draft_row0,
                           draft_len, max_draft_len, draft_tokens, B, seed, request_ids,
                           accepted_len, out_tokens, out_ld, correction_token, accept_ratio,
                           status, scratch, sv::kNoAllocScratchBytes, stream);
}
