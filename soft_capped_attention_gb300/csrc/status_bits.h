// Bits of the device status word (first word of the workspace).
#pragma once
#include <stdint.h>

namespace capattn {
constexpr uint32_t kStatusTimeoutBit = 1u;      // a kernel gave up on a bounded wait
constexpr uint32_t kStatusBadSegmentsBit = 2u;  // segment ids decrease along a batch row
constexpr uint32_t kStatusBadBoundsBit = 4u;    // ranker bounds outside 0 <= lo <= hi <= L
constexpr uint32_t kStatusRankerIdsBit = 8u;    // history / candidate ids of a row not contiguous
constexpr uint32_t kStatusBandBit = 16u;        // a visited tile pair outside the configuration's band
                                                // (no dX slot for it; an internal inconsistency)
}  // namespace capattn
