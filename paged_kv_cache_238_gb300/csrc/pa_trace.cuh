// Optional per-warp timeline of the decode kernel, for profiling builds only.
//
// Compiled in only when PA_TRACE is defined (never in the library that build() makes): each
// warp's lane 0 writes %globaltimer stamps of the kernel's phases into a ring of the last
// kTraceLaunches launches, read back with pa_trace_read(). Without PA_TRACE every macro below
// expands to nothing.
#pragma once

#include <stdint.h>

#ifdef PA_TRACE
namespace pa {
constexpr int kTraceLaunches = 16;
constexpr int kTraceCtas = 160;
constexpr int kTraceWarps = 16;
constexpr int kTraceEvents = 32;
constexpr int kTraceWords = kTraceLaunches * kTraceCtas * kTraceWarps * kTraceEvents;
}  // namespace pa
#define PA_TRACE_DECL                          \
    __shared__ uint32_t pa_trace_launch_s;     \
    uint32_t pa_trace_launch = 0;
// Launch index: the CTAs of one launch all start before any CTA of the next one (a persistent
// grid of one CTA per SM), so the entry counter over the grid size numbers the launches.
#define PA_TRACE_BEGIN(counter)                                                      \
    do {                                                                             \
        if (threadIdx.x == 0) pa_trace_launch_s = atomicAdd(&(counter), 1u) / gridDim.x; \
        __syncthreads();                                                             \
        pa_trace_launch = pa_trace_launch_s;                                         \
    } while (0)
#define PA_TRACE_AT(buf, ev, val)                                                                    \
    do {                                                                                             \
        if ((threadIdx.x & 31) == 0 && blockIdx.x < pa::kTraceCtas && (threadIdx.x >> 5) < pa::kTraceWarps) \
            (buf)[((static_cast<uint64_t>(pa_trace_launch % pa::kTraceLaunches) * pa::kTraceCtas + blockIdx.x) * \
                       pa::kTraceWarps + (threadIdx.x >> 5)) * pa::kTraceEvents + (ev)] = (val);     \
    } while (0)
#define PA_TRACE_STAMP(buf, ev) PA_TRACE_AT(buf, ev, pa::global_timer_ns())
#else
#define PA_TRACE_DECL
#define PA_TRACE_BEGIN(counter) \
    do {                        \
    } while (0)
#define PA_TRACE_AT(buf, ev, val) \
    do {                          \
    } while (0)
#define PA_TRACE_STAMP(buf, ev) \
    do {                        \
    } while (0)
#endif
