// The one TMA form that only the single-GPU multicast library uses: a 2-D
// tiled load issued by one CTA of a pair that lands at the same shared-memory
// offset in several CTAs of the cluster.  It is kept out of the default
// library: that library, which a process may load on each of several GPUs,
// issues no multicast load at all.  This library (libgemm_f16_nt_mcast.so) may
// multicast only within one GPU's own memory: its host code refuses operands
// that are not device memory of the current device, in a process that sees
// more than one GPU, before anything is enqueued.
#pragma once

#include <stdint.h>

namespace g16 {

// Loader hook of the kernel for clusters of two CTA pairs that share their A
// rows: the same-rank CTA of both pairs receives the half of A this CTA loads.
template <int CP>
struct McastA {
    static constexpr bool kAvailable = true;
    // `dst`: shared-memory offset in every CTA of `cta_mask`; each destination's
    // completion bytes go to the barrier at `bar`'s offset in the leader CTA of
    // that destination's pair.
    __device__ static __forceinline__ void load(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                                uint32_t bar, uint16_t cta_mask) {
        asm volatile(
            "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
            ".multicast::cluster [%0], [%1, {%2, %3}], [%4], %5;"
            :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "h"(cta_mask)
            : "memory");
    }
};

}  // namespace g16
