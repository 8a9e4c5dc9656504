// Phase timeline of the streaming executor, compiled in only with -DVP_PHASE_TRACE (the
// libverify_trace.so build); in the normal build every hook below is empty.
//
// For each phase p of a launch and each CTA, globaltimer stamps (ns): [0] phase start, [1] end of the
// activation staging, [2 + w] warp w done with its units, [18 + w] warp w done with its row blocks
// shared within the CTA, [35] (K-sliced phases) the cross-slice sums done, [34] grid barrier passed,
// [36] the staging's loads and row statistics done (before the conversion).  Two launch buffers alternate (the
// launch counter's parity), so the two launches of a verify pass keep both halves.
#pragma once
#include <cstdint>

#include "internal.h"

namespace vp {

constexpr int kTraceSlots = 37;

#ifdef VP_PHASE_TRACE
__device__ unsigned long long g_trace[2][kMaxPhases][kMaxGrid][kTraceSlots];
__device__ unsigned g_trace_launches;  // launches completed (the last CTA to leave counts)
// The launch buffer of this launch, read once per CTA at the start (VP_TRACE_INIT, followed by a
// barrier), so that a stamp is a timer read and a store that nothing waits for.
// It lives in the last word of the dynamic shared memory (the executor's misc area leaves it free).
__device__ __forceinline__ unsigned& trace_parity() {
  extern __shared__ __align__(128) uint8_t trace_smem[];
  return *reinterpret_cast<unsigned*>(trace_smem + kSmemBytes - sizeof(unsigned));
}
__device__ __forceinline__ void trace_stamp(int p, int slot) {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  g_trace[trace_parity()][p][blockIdx.x][slot] = t;
}
#define VP_TRACE(cond, p, slot)                   \
  do {                                            \
    if (cond) ::vp::trace_stamp((p), (slot));     \
  } while (0)
#define VP_TRACE_INIT()                                                                                \
  do {                                                                                                 \
    if (threadIdx.x == 0) ::vp::trace_parity() = *reinterpret_cast<volatile unsigned*>(&::vp::g_trace_launches) & 1u; \
  } while (0)
#define VP_TRACE_LAUNCH_DONE() atomicAdd(&::vp::g_trace_launches, 1u)
#else
#define VP_TRACE(cond, p, slot) ((void)0)
#define VP_TRACE_INIT() ((void)0)
#define VP_TRACE_LAUNCH_DONE() ((void)0)
#endif

}  // namespace vp
