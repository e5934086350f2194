// Host-side helpers shared by the library's translation units: error
// reporting through bwd_last_error() and launch checks.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "bwd.h"

namespace bwd {
namespace host {

// Records a printf-style message as this thread's last error and returns s.
bwd_status fail(bwd_status s, const char* fmt, ...);

// BWD_ERR_CUDA with the runtime's name and description of e.
bwd_status cuda_fail(cudaError_t e, const char* what);

// BWD_OK, or BWD_ERR_CUDA if the last launch on this thread failed.
bwd_status check_launch(const char* what);

// This thread's last error message ("" if none).
const char* last_error();

// Unique id of the current CUDA context (the driver's cuCtxGetId, unique for
// the life of the process).  Per-device state cached by the library (the
// uploaded code tables, kernel attributes) belongs to one context: after a
// cudaDeviceReset or a released primary context the id changes and the state
// is set up again.  Initialises the device's primary context if none is
// current.
bwd_status current_context_id(unsigned long long* id);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// p is a multiple of `bytes` (a power of two): element pointers must be
// aligned to their element size, or device accesses through them fault.
inline bool aligned_to(const void* p, uintptr_t bytes) { return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) == 0; }

}  // namespace host
}  // namespace bwd
