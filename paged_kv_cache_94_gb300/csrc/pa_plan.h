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

// First item of CTA c (G = plan_ctas(grid, W)).
PA_HD int64_t plan_lo(int64_t c, int64_t W, int64_t G) { return c * W / G; }

// The CTA that owns item x (0 <= x < W): the largest c with plan_lo(c) <= x,
// i.e. ceil((x+1)*G/W) - 1.
PA_HD int64_t plan_owner(int64_t x, int64_t W, int64_t G) { return ((x + 1) * G - 1) / W; }

} // namespace pa
