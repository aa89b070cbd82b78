// watchdog.cuh -- bounded mbarrier waits for the standalone kernels (GEMM, row softmax).
// A wait that outlives its limit records a site in the translation unit's status word,
// raises the CTA's abort flag and returns false; the caller then drains and exits.
#pragma once
#include <cstdint>

#include "ptx.cuh"

namespace fa {

__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             uint64_t timeout_ns, uint32_t site, unsigned int *status,
                                             bool check_abort = true)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1; it < (1u << 30); ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 31u) == 0) {
            if (check_abort && *abort_flag) return false;
            if (globaltimer_ns() - t0 > timeout_ns) break;
        }
    }
    *abort_flag = 1;
    atomicCAS(status, 0u, 1u | (site << 8));
    atomicOr(status, 1u);
    return false;
}

// Hardware tanh (MUFU), maximum relative error about 2^-11 -- below the 16-bit output rounding.
__device__ __forceinline__ float tanh_approx(float x)
{
    float y;
    asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

} // namespace fa
