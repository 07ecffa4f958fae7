// trace.cuh -- optional per-role clock64 timeline of one CTA.
//
// Built only with -DNEA_TRACE (never in the default library): each traced
// role (one lane of one warp of the traced CTA) appends (clock64 << 8 | event)
// to a row of its own in a device array, with no atomics and no waits, so the
// timeline perturbs the kernel as little as possible.  The host reads the
// array back through the nea_trace_read_* function of the translation unit.
// Without NEA_TRACE every call compiles to nothing.
#pragma once
#include <cstdint>

namespace nea {

constexpr int kTraceRoles = 8;
constexpr int kTraceEvents = 2048;

#ifdef NEA_TRACE
struct Tracer {
  long long* row;
  int n;
  __device__ Tracer(long long* base, bool on, int role)
      : row(on ? base + static_cast<long long>(role) * kTraceEvents : nullptr), n(0) {}
  __device__ __forceinline__ void ev(int id) {
    if (row != nullptr && n < kTraceEvents) row[n++] = (clock64() << 8) | (id & 0xff);
  }
};
#else
struct Tracer {
  __device__ Tracer(long long*, bool, int) {}
  __device__ __forceinline__ void ev(int) {}
};
#endif

}  // namespace nea
