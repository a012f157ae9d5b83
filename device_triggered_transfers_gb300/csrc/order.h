// The builtin step-to-tile orders, compiled for host and device from one definition so that a
// schedule built on the host and the producer kernel that marks it cannot disagree ("Triggered
// Plans", section Model: pass the kernel's own mapping rather than a copy of it).
#pragma once

#include <cstdint>

#include "dtt.h"

#if defined(__CUDACC__)
#define DTT_HD __host__ __device__ __forceinline__
#else
#define DTT_HD inline
#endif

namespace dtt {

// Row-major: step s -> (s / tiles_n, s % tiles_n).
// Grouped: group_m tile rows at a time, swept column by column inside the group; the last
// group may hold fewer rows.
DTT_HD void tile_of(uint32_t kind, uint32_t group_m, uint64_t step, uint32_t tiles_m,
                    uint32_t tiles_n, uint32_t* tm, uint32_t* tn) {
    if (kind == DTT_ORDER_GROUPED && group_m > 0) {
        const uint64_t per_group = (uint64_t)group_m * tiles_n;
        const uint64_t g = step / per_group;
        const uint64_t m0 = g * group_m;
        const uint64_t left = tiles_m - m0;
        const uint64_t h = left < group_m ? left : group_m;
        const uint64_t w = step - g * per_group;
        *tm = (uint32_t)(m0 + w % h);
        *tn = (uint32_t)(w / h);
    } else {
        *tm = (uint32_t)(step / tiles_n);
        *tn = (uint32_t)(step % tiles_n);
    }
}

}  // namespace dtt
