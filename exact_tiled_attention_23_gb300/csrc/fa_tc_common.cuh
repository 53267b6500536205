// fa_tc_common.cuh -- pieces shared by the tensor-core kernels: tcgen05
// instruction and shared-memory descriptors, and the bounded mbarrier wait.
#pragma once

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// tcgen05 instruction descriptor, kind::f16: A and B both bf16 (or both
// f16), fp32 accumulator.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, int a_mn_major, int b_mn_major,
                                                  bool f16 = false)
{
    return (1u << 4)                      // accumulator format: f32
         | ((f16 ? 0u : 1u) << 7)         // A format: f16 = 0, bf16 = 1
         | ((f16 ? 0u : 1u) << 10)        // B format: same as A
         | ((uint32_t)a_mn_major << 15)
         | ((uint32_t)b_mn_major << 16)
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand.
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;               // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;               // swizzle: 128 B
    return d;
}

// Per-CTA abort flag (shared memory) and the library status word that a
// give-up is recorded in.
struct Abort {
    volatile int *flag;
    uint32_t *status;
};

// Drains (waits that do not follow the abort flag) wait for copies and MMAs
// the CTA itself has in flight, which always end: they keep at least this
// budget whatever the caller's limit, so a CTA never exits, or frees TMEM,
// while its own copies or MMAs are still running.
constexpr uint64_t kDrainFloorNs = 1000000000ull;

// Bounded wait on phase `parity` of `bar`.  Returns false when the budget ran
// out (the status word records `site`) or, if `follow_abort`, as soon as
// another thread of the CTA has aborted.  Budgets below 100 us are checked on
// every probe, so that a short limit runs out as soon as it is exceeded.
__device__ __forceinline__ bool wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns,
                                             uint32_t site, Abort ab, bool follow_abort = true)
{
    if (ptx::mbar_test(bar, parity)) return true;
    if (!follow_abort && limit_ns < kDrainFloorNs) limit_ns = kDrainFloorNs;
    const uint32_t check_mask = limit_ns < 100000ull ? 0u : 63u;
    const uint64_t t0 = ptx::globaltimer_ns();
    uint32_t spins = 0;
    while (true) {
        if (ptx::mbar_test(bar, parity)) return true;
        if ((++spins & check_mask) == 0) {
            if (follow_abort && *ab.flag) return false;
            if (ptx::globaltimer_ns() - t0 > limit_ns) {
                atomicOr(ab.status, kStatusTimeout | (site << 8));
                *ab.flag = 1;
                return false;
            }
        }
    }
}


}  // namespace fa
