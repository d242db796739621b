// markov.cu -- DSpark Markov-head drafting (placeholder until the tcgen05 kernel lands).
#include "sv_host.h"

extern "C" size_t dspark_markov_workspace_bytes(int32_t B, int32_t K, int64_t V, int32_t R) {
  (void)B; (void)K; (void)V; (void)R;
  return 256;
}

extern "C" sv_status dspark_markov_draft(const void*, int64_t, const void*, const void*, int64_t,
                                         const int32_t*, const float*, const float*, int32_t,
                                         int32_t, int64_t, int32_t, uint64_t, const uint64_t*,
                                         int32_t*, void*, int64_t, float*, float*, int32_t*, void*,
                                         size_t, void*) {
  return SV_ERR_UNSUPPORTED;
}
