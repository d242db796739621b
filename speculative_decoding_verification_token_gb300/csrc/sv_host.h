// sv_host.h -- host-side helpers shared by the entry points (argument checks, device queries).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "specverify.h"

namespace sv {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned256(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }

inline int elem_bytes(sv_dtype d) { return d == SV_BF16 ? 2 : 4; }

// Number of SMs of the current device (queried once per device).
int device_sm_count();

// Shared memory per SM of the current device, in bytes (queried once per device).
int device_smem_per_sm();

// Resident CTAs per SM of `kernel` with `smem` bytes of dynamic shared memory (0 on error).
int resident_ctas(const void* kernel, int threads, size_t smem);

// A fresh 64-bit value per call, distinct for every call of the process (an odd-stride counter
// from a time- and address-derived start): tags a launch's own writes in a reused workspace.
uint64_t next_call_id();

// Diagnostic kernel timing (sv_profile_enable): record event `k` (0..3) on `stream` if enabled.
void profile_mark(int k, cudaStream_t stream);

inline sv_status launch_status(cudaError_t e) {
  return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

}  // namespace sv
