// Optional per-block timeline stamps (%globaltimer, ns), compiled in only with
// -DGQA_TRACE; otherwise every macro expands to nothing.
#pragma once

#ifdef GQA_TRACE
#include <stdint.h>
namespace gqa {
constexpr int kTraceSlots = 1 << 16;
// One copy per translation unit that includes this header.
static __device__ unsigned long long g_trace[kTraceSlots][8];
}  // namespace gqa
#define GQA_TRACE_STAMP(block, k)                                                       \
    do {                                                                                \
        if ((block) < gqa::kTraceSlots) gqa::g_trace[(block)][(k)] = gqa::globaltimer(); \
    } while (0)
#define GQA_TRACE_VALUE(block, k, v)                                     \
    do {                                                                 \
        if ((block) < gqa::kTraceSlots) gqa::g_trace[(block)][(k)] = (v); \
    } while (0)
#else
#define GQA_TRACE_STAMP(block, k) \
    do {                          \
    } while (0)
#define GQA_TRACE_VALUE(block, k, v) \
    do {                             \
    } while (0)
#endif
