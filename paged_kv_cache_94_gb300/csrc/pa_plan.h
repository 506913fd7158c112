// Equal split of a line of W positions over G = min(grid, W) parts, shared
// by host and device code: part c owns [floor(c*W/G), floor((c+1)*W/G)).
// The decode kernels apply it to a cost-weighted line of their items (blocks
// plus a fixed charge per (sequence, kv head), pa_decode.cuh).
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define PA_HD __host__ __device__ __forceinline__
#else
#define PA_HD inline
#endif

namespace pa {

// CTAs that take part: never more than there are items, so that every
// participating CTA owns at least one item.
PA_HD int64_t plan_ctas(int64_t grid, int64_t W) { return grid < W ? grid : W; }

// First item of CTA c (G = plan_ctas(grid, W)). In 32-bit arithmetic when
// W * G fits (every product below is at most W * G): same result, cheaper
// division on the device.
PA_HD int64_t plan_lo(int64_t c, int64_t W, int64_t G)
{
    if (W * G <= (int64_t)0xFFFFFFFF)
        return (int64_t)((uint32_t)c * (uint32_t)W / (uint32_t)G);
    return c * W / G;
}

// The CTA that owns item x (0 <= x < W): the largest c with plan_lo(c) <= x,
// i.e. ceil((x+1)*G/W) - 1.
PA_HD int64_t plan_owner(int64_t x, int64_t W, int64_t G)
{
    if (W * G <= (int64_t)0xFFFFFFFF)
        return (int64_t)((((uint32_t)x + 1u) * (uint32_t)G - 1u) / (uint32_t)W);
    return ((x + 1) * G - 1) / W;
}

} // namespace pa
