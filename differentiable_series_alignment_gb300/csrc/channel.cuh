// channel.cuh -- bounded waits on the tagged-slot channels between wavefront warps and strips.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace sdtw {

constexpr unsigned kFull = 0xffffffffu;

// The waits below spin on the value itself and look at the global status word and
// the clock only every kPollEvery retries: a global load per retry would put an
// L2 round trip between the producer's store and the consumer noticing it.
constexpr unsigned kPollEvery = 32;

// Bounded wait on a shared-memory counter (back-pressure of a ring). `seen` gets
// the count observed, so the caller can skip the next checks while its target
// stays at or below it. Warp-uniform result.
static __device__ __forceinline__ bool wait_smem(const volatile int* cnt, int target, const WaveParams& q, int& seen) {
    bool ok = true;
    int c = *cnt;
    if (c < target) {
        unsigned long long t0 = 0;
        for (unsigned it = 1; (c = *cnt) < target; ++it) {
            if ((it % kPollEvery) == 0) {
                if (t0 == 0) t0 = global_ns();
                if (ld_volatile_global(q.status) != 0) { ok = false; break; }
                if (global_ns() - t0 > q.wait_ns) { atomicOr(q.status, kStatusTimeout); ok = false; break; }
                __nanosleep(32);
            }
        }
    }
    seen = __shfl_sync(kFull, c, 0);
    return __shfl_sync(kFull, ok, 0);
}

// wait_smem for a warp whose wait is off the critical path: sleeps between tests so
// that it leaves the issue slots of its scheduler to the DP warp there.
static __device__ __forceinline__ bool wait_smem_sleep(const volatile int* cnt, int target, const WaveParams& q,
                                                       int& seen, unsigned ns) {
    bool ok = true;
    int c = *cnt;
    if (c < target) {
        const unsigned long long t0 = global_ns();
        while ((c = *cnt) < target) {
            __nanosleep(ns);
            if (ld_volatile_global(q.status) != 0) { ok = false; break; }
            if (global_ns() - t0 > q.wait_ns) { atomicOr(q.status, kStatusTimeout); ok = false; break; }
        }
    }
    seen = __shfl_sync(kFull, c, 0);
    return __shfl_sync(kFull, ok, 0);
}

// Wait until every lane's slot (or pair of slots) carries its expected tag,
// reloading the lanes that do not yet. want == 0 marks a lane with nothing to
// check. Bounded; warp-uniform result.
template <int NS>
static __device__ __forceinline__ bool validate(Slot (&cur)[NS], const Slot* src, unsigned want, const WaveParams& q) {
    bool mine = true;
#pragma unroll
    for (int k = 0; k < NS; ++k) mine = mine && (want == 0u || cur[k].tag == want);
    if (__all_sync(kFull, mine)) return true;
    unsigned long long t0 = 0;
    for (unsigned it = 1;; ++it) {
        if (!mine) {
#pragma unroll
            for (int k = 0; k < NS; ++k) cur[k] = slot_load(src + k);
            mine = true;
#pragma unroll
            for (int k = 0; k < NS; ++k) mine = mine && (cur[k].tag == want);
        }
        if (__all_sync(kFull, mine)) return true;
        if ((it % kPollEvery) == 0) {
            if (t0 == 0) t0 = global_ns();
            bool bad = ld_volatile_global(q.status) != 0;
            if (!bad && global_ns() - t0 > q.wait_ns) { atomicOr(q.status, kStatusTimeout); bad = true; }
            if (__any_sync(kFull, bad)) return false;
            __nanosleep(20);
        }
    }
}

}  // namespace sdtw
