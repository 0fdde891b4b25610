// ring_schedule.h -- the load schedule of a staging ring whose bulk loads run
// `la` units ahead of the unit being consumed (the bf16 dispatch ring), as
// plain host/device functions, so that its bookkeeping -- in particular which
// loads may still be in flight when a wait gives up -- is checked on the CPU.
//
// Schedule over the n units of one CTA:
//   prologue:      load units 0 .. ring_prologue_loads(n, la) - 1;
//   iteration i:   if ring_issues_ahead(i, n, la), load unit i + la; then
//                  wait for unit i.
// When the wait of iteration i gives up, the loads of units
// i .. ring_issued_end(i, n, la) - 1 have been issued and none of them has
// been waited for: all of them must land before the CTA may exit.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define EP_HOST_DEVICE __host__ __device__
#else
#define EP_HOST_DEVICE
#endif

namespace ep {

EP_HOST_DEVICE constexpr int64_t ring_prologue_loads(int64_t n, int la) { return la < n ? la : n; }

EP_HOST_DEVICE constexpr bool ring_issues_ahead(int64_t i, int64_t n, int la) { return i + la < n; }

EP_HOST_DEVICE constexpr int64_t ring_issued_end(int64_t i, int64_t n, int la) {
    return i + la + 1 < n ? i + la + 1 : n;
}

}  // namespace ep
