// selftest.cuh -- a device check of the pipeline-wait bound, without a fault.
//
// Every wait of the prefill and decode kernels goes through mbar_wait: it gives
// up after kWaitLimitNs, records a timeout in the device status word, raises the
// CTA's abort flag, and returns false, so that a lost arrival ends the kernel with
// an error the host can read instead of hanging the GPU.  This kernel exercises
// exactly that path on barriers nothing ever arrives on:
//   warp 0 waits on barrier 0; its wait runs out after kWaitLimitNs, records the
//          timeout and raises the abort flag;
//   warp 1 starts its own wait on barrier 1 half a second later, so its own bound
//          would end it half a second after warp 0's; it must leave on the flag
//          instead, at about the moment warp 0 gives up.
// out[2w] = 1 if warp w's wait returned true (it must not), out[2w + 1] = the
// nanoseconds warp w spent from the kernel's start to the end of its wait.
#pragma once

#include "ptx.cuh"

namespace attn07 {

constexpr unsigned long long kSelftestStaggerNs = 500000000ull;  // 0.5 s

__global__ void __launch_bounds__(64, 1)
selftest_wait_timeout_kernel(unsigned *status, unsigned long long *out) {
    __shared__ __align__(8) uint64_t bars[2];
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars[0]), 1);
        mbar_init(smem_u32(&bars[1]), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) == 0) {
        const unsigned long long t0 = globaltimer();
        if (warp == 1) {
            // bounded: ends after kSelftestStaggerNs
            while (globaltimer() - t0 < kSelftestStaggerNs) {
            }
        }
        const bool ok = mbar_wait(smem_u32(&bars[warp]), 0u, status,
                                  reinterpret_cast<volatile int *>(&abort_flag));
        out[2 * warp] = ok ? 1ull : 0ull;
        out[2 * warp + 1] = globaltimer() - t0;
    }
}

}  // namespace attn07
