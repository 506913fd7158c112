// Compiled multi-query decode kernels: int4 K/V, head dim 128, NQ new tokens per
// sequence (2, 4 or 8) for group sizes g with g * NQ <= 16.
#include "pa_decode_quant_mq.cuh"

// Warps per CTA, ring stages per warp, resident CTAs per SM and blocks per
// ring item (as the single-query kernels; overridable for a tuning sweep).
#ifndef PA_INT4_D128_MQ_NW
#define PA_INT4_D128_MQ_NW 4
#endif
#ifndef PA_INT4_D128_MQ_STAGES
#define PA_INT4_D128_MQ_STAGES 3
#endif
#ifndef PA_INT4_D128_MQ_MINB
#define PA_INT4_D128_MQ_MINB 3
#endif
#ifndef PA_INT4_D128_MQ_BPI
#define PA_INT4_D128_MQ_BPI 2
#endif

namespace pa {

const DecodeKernel *find_decode_kernel_int4_mq_d128(int group, int nq)
{
    return pick_quant_mq<4, 128, PA_INT4_D128_MQ_NW, PA_INT4_D128_MQ_STAGES, PA_INT4_D128_MQ_MINB,
                         PA_INT4_D128_MQ_BPI>(group, nq);
}

} // namespace pa
