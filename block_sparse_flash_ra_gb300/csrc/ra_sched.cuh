// ra_sched.cuh -- work-unit scheduling helpers shared by the persistent
// tensor-core kernels: snake round-robin over a longest-first unit order,
// bounded drain waits and the scalar merge math.
#pragma once

#include "ra_device.cuh"

namespace ra {

// Snake order over rounds of G units: round r gives CTA c the unit r*G + c
// (even r) or r*G + G-1-c (odd r).
__device__ __forceinline__ int unit_index(int round, int cta, int G)
{
    return round * G + ((round & 1) ? (G - 1 - cta) : cta);
}

// Wait used only while tearing down after an abort: bounded, ignores the
// abort flag.
__device__ __forceinline__ bool wait_drain(uint64_t *bar, uint32_t parity, uint64_t ns)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > ns) return false;
    }
    return true;
}

__device__ __forceinline__ float sigmoid_f(float x)
{
    if (x >= 0.f) return 1.f / (1.f + expf(-x));
    const float e = expf(x);
    return e / (1.f + e);
}

__device__ __forceinline__ float softplus_f(float x)
{
    return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}

constexpr uint64_t kDrainNs = 100000000ull; // 100 ms

} // namespace ra
