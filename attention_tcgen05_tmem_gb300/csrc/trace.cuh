// trace.cuh -- opt-in pipeline timeline tracing (build with -DATTN_TRACE).
//
// For the first kTraceCtas CTAs of a launch, one thread per role records the
// SM cycle counter at named points of iterations [kTraceFirst, kTraceFirst +
// kTraceIters) into a per-translation-unit device array; a host reader
// (ATTN_TRACE_READER) copies it out.  Roles: 0 producer, 1 MMA issuer,
// 2 first elementwise warpgroup, 3 second.  Without ATTN_TRACE every probe
// compiles to nothing.
#pragma once
#include <cstdint>

namespace attn {
constexpr int kTraceCtas = 4, kTraceRoles = 4, kTraceEvents = 8, kTraceIters = 64,
              kTraceFirst = 16;
}  // namespace attn

#ifdef ATTN_TRACE
static __device__ unsigned long long
    g_attn_trace[attn::kTraceCtas][attn::kTraceRoles][attn::kTraceEvents][attn::kTraceIters];
#define ATTN_TR(role, ev, it)                                                                    \
  do {                                                                                           \
    const int _i = (it)-attn::kTraceFirst;                                                       \
    if (blockIdx.x < attn::kTraceCtas && _i >= 0 && _i < attn::kTraceIters)                      \
      g_attn_trace[blockIdx.x][role][ev][_i] = clock64();                                        \
  } while (0)
#define ATTN_TRACE_READER(name)                                                                  \
  extern "C" int name(void* dst, size_t n) {                                                     \
    return (int)cudaMemcpyFromSymbol(dst, g_attn_trace, n < sizeof(g_attn_trace) ? n : sizeof(g_attn_trace)); \
  }                                                                                              \
  extern "C" int name##_clear() {                                                                \
    static unsigned long long z[attn::kTraceCtas][attn::kTraceRoles][attn::kTraceEvents][attn::kTraceIters]; \
    return (int)cudaMemcpyToSymbol(g_attn_trace, z, sizeof(z));                                  \
  }
#else
#define ATTN_TR(role, ev, it) \
  do {                        \
  } while (0)
#define ATTN_TRACE_READER(name)
#endif
