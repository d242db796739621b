// api.cu -- status strings, version and the host-side device queries used by every entry point.
#include <atomic>
#include <chrono>
#include <mutex>

#include "sv_device.cuh"
#include "sv_host.h"

namespace sv {

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sm_count[kMaxDevices] = {0};
int g_smem_per_sm[kMaxDevices] = {0};
}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

int device_smem_per_sm() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_smem_per_sm[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
        cudaSuccess)
      return 0;
    g_smem_per_sm[dev] = n;
  }
  return g_smem_per_sm[dev];
}

uint64_t next_call_id() {
  static std::atomic<uint64_t> counter{
      static_cast<uint64_t>(std::chrono::steady_clock::now().time_since_epoch().count()) *
          0xD1342543DE82EF95ull ^
      static_cast<uint64_t>(reinterpret_cast<uintptr_t>(&counter))};
  return counter.fetch_add(0x9E3779B97F4A7C15ull, std::memory_order_relaxed);
}

int resident_ctas(const void* kernel, int threads, size_t smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess)
    return 0;
  return n;
}

namespace {
struct ProfileState {
  bool enabled = false;
  bool created = false;
  cudaEvent_t ev[4];
};
thread_local ProfileState g_prof;
}  // namespace

void profile_mark(int k, cudaStream_t stream) {
  if (!g_prof.enabled || !g_prof.created) return;
  cudaEventRecord(g_prof.ev[k], stream);
}

}  // namespace sv

extern "C" sv_status sv_profile_enable(int enable) {
  sv::ProfileState& ps = sv::g_prof;
  if (enable && !ps.created) {
    for (int k = 0; k < 4; ++k)
      if (cudaEventCreate(&ps.ev[k]) != cudaSuccess) return SV_ERR_CUDA;
    ps.created = true;
  }
  ps.enabled = enable != 0;
  return SV_OK;
}

extern "C" sv_status sv_profile_read(float* ms_out) {
  sv::ProfileState& ps = sv::g_prof;
  if (!ms_out || !ps.created) return SV_ERR_INVALID;
  if (cudaEventSynchronize(ps.ev[3]) != cudaSuccess) return SV_ERR_CUDA;
  for (int k = 0; k < 3; ++k)
    if (cudaEventElapsedTime(&ms_out[k], ps.ev[k], ps.ev[k + 1]) != cudaSuccess) return SV_ERR_CUDA;
  return SV_OK;
}

extern "C" const char* sv_status_string(sv_status status) {
  switch (status) {
    case SV_OK: return "SV_OK";
    case SV_ERR_INVALID: return "SV_ERR_INVALID: invalid argument";
    case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED: unsupported argument";
    case SV_ERR_CUDA: return "SV_ERR_CUDA: CUDA runtime error";
    case SV_ERR_BAD_INPUT: return "SV_ERR_BAD_INPUT: invalid data found on the device";
    case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT: bounded device-side wait expired";
  }
  return "unknown sv_status";
}

extern "C" const char* sv_version(void) { return "specverify 0.1 (sm_103a)"; }

// ---------------------------------------------------------------------------------------------
// sv_selftest_wait: the bounded waits of the kernels, made to run out
// ---------------------------------------------------------------------------------------------
namespace sv {

// One warp.  which = 0: an mbarrier phase that no thread completes; which = 1: a shared-memory
// request-number word that no thread publishes.  Both use the waits every kernel uses, with the
// caller's limit, and must end with SV_ERR_TIMEOUT in `status`.
__global__ void selftest_wait_kernel(int32_t which, uint64_t limit_ns, int32_t* status) {
  __shared__ uint64_t bar;
  __shared__ uint32_t word;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    word = 0u;
  }
  __syncwarp();
  if (threadIdx.x != 0) return;
  if (which == 0) mbar_wait(&bar, 0, status, limit_ns);
  else wait_seq(&word, 1u, status, limit_ns);
}

}  // namespace sv

extern "C" sv_status sv_selftest_wait(int32_t which, int32_t limit_us, int32_t* status,
                                      void* stream) {
  if ((which != 0 && which != 1) || limit_us <= 0 || limit_us > 1000000 || !status)
    return SV_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return SV_ERR_CUDA;
  sv::selftest_wait_kernel<<<1, 32, 0, s>>>(which, uint64_t(limit_us) * 1000ull, status);
  return sv::launch_status(cudaGetLastError());
}
