// wmtp_ring.cuh -- the ring slot rule shared by the index and tree kernels.
//
// "Windowed-MTP" App. A: slot = ring_base(r) + logical position, with a ring
// of n_sink + W + d slots per request; §7: a tree of width k reserves
// n_sink + W + d*k.  Sinks are pinned on branch 0; every other position rolls
// over the W + d*k slots after them, each branch shifted by branch * d (side
// branches never use the shared sink slots).
#pragma once

#include <stdint.h>

namespace wmtp {

__device__ __forceinline__ int64_t ring_slot(int64_t base, int64_t p, int64_t branch,
                                             int64_t n_sink, int64_t window, int64_t depth,
                                             int64_t tree_k) {
    if (p < n_sink && branch == 0) return base + p;
    const int64_t m = window + depth * tree_k;
    int64_t r = (p - n_sink + branch * depth) % m;
    if (r < 0) r += m;
    return base + n_sink + r;
}

}  // namespace wmtp
