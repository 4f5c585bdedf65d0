// hbm_read.cuh -- the read ceiling of a launch: a kernel that only streams
// `bytes` of global memory into shared memory, with the launch structure of
// the GEMM kernels (one CTA per SM, a producer warp issuing bulk copies into
// a ring of stages, programmatic dependent launch, equal contiguous shares).
// Timing it on a weight matrix's byte count, back to back like the GEMMs,
// gives the rate a kernel of that size can reach at all, fixed launch costs
// included; the GEMMs are reported as a fraction of it.
#pragma once

#include "w4a16_stream.cuh"

namespace sv {

constexpr int HR_STAGE = 32768;     // bytes per stage
constexpr int HR_NST = 6;           // stages

// One warp issues the copies; one warp waits for each stage, folds one word
// of it into a checksum (so the data is used) and frees the stage.
__global__ void __launch_bounds__(64, 1) hbm_read_kernel(const uint8_t *src, unsigned long long bytes,
                                                         uint32_t *sink, int *err)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + HR_NST * HR_STAGE);
    uint64_t *empty = full + HR_NST;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // this CTA's share, in 16-byte chunks
    const unsigned long long chunks = bytes / 16;
    const unsigned long long c0 = chunks * blockIdx.x / gridDim.x, c1 = chunks * (blockIdx.x + 1) / gridDim.x;
    const unsigned long long beg = c0 * 16, end = c1 * 16;
    const int n = static_cast<int>((end - beg + HR_STAGE - 1) / HR_STAGE);
    if (threadIdx.x == 0) {
        for (int s = 0; s < HR_NST; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), 1);
        }
        fence_barrier_init();
    }
    __syncthreads();
    pdl_launch_dependents();
    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            for (int i = 0; i < n; ++i) {
                const int s = i % HR_NST;
                if (i >= HR_NST && !mbar_wait_bounded(smem_addr(&empty[s]), static_cast<uint32_t>(((i / HR_NST) & 1) ^ 1),
                                                     WAIT_LIMIT_NS))
                    atomicOr(err, 2);
                const unsigned long long off = beg + static_cast<unsigned long long>(i) * HR_STAGE;
                const uint32_t len = static_cast<uint32_t>(end - off < HR_STAGE ? end - off : HR_STAGE);
                mbar_arrive_expect_tx(smem_addr(&full[s]), len);
                bulk_g2s(smem_addr(smem + s * HR_STAGE), src + off, len, smem_addr(&full[s]), pol);
            }
            // do not leave while a copy may still be landing
            for (int i = n - (n < HR_NST ? n : HR_NST); i < n; ++i)
                if (!mbar_wait_bounded(smem_addr(&full[i % HR_NST]), static_cast<uint32_t>((i / HR_NST) & 1),
                                       WAIT_LIMIT_AFTER_ERR_NS))
                    atomicOr(err, 2);
        }
        return;
    }
    uint32_t acc = 0;
    for (int i = 0; i < n; ++i) {
        const int s = i % HR_NST;
        if (!mbar_wait_bounded(smem_addr(&full[s]), static_cast<uint32_t>((i / HR_NST) & 1), WAIT_LIMIT_NS))
            atomicOr(err, 2);
        if (lane == 0) {
            acc ^= *reinterpret_cast<const uint32_t *>(smem + s * HR_STAGE);
            mbar_arrive(smem_addr(&empty[s]));
        }
    }
    pdl_wait_prior();               // the output may be read by the previous kernel
    if (lane == 0) sink[blockIdx.x] = acc;
}

}  // namespace sv
