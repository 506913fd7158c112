// Compiled multi-query decode kernels: bf16 K/V, head dim 128 and 64, NQ new
// tokens per sequence (2, 4 or 8) for group sizes g with g * NQ <= 16.
#include "pa_decode_kernel.cuh"

// Warps per CTA and ring stages per warp (as the single-query kernels; 16
// query rows keep four warps at head dim 128 for the merge slices' room).
#ifndef PA_BF16_MQ_D128_NW
#define PA_BF16_MQ_D128_NW 8
#endif
#ifndef PA_BF16_MQ_D128_NW_R16
#define PA_BF16_MQ_D128_NW_R16 4
#endif
#ifndef PA_BF16_MQ_D128_STAGES
#define PA_BF16_MQ_D128_STAGES 2
#endif
#ifndef PA_BF16_MQ_D128_STAGES_R16
#define PA_BF16_MQ_D128_STAGES_R16 2
#endif
#ifndef PA_BF16_MQ_D64_NW
#define PA_BF16_MQ_D64_NW 4
#endif
#ifndef PA_BF16_MQ_D64_STAGES
#define PA_BF16_MQ_D64_STAGES 6
#endif

namespace pa {
namespace {

template <class Pol>
size_t smem_of(int num_seqs)
{
    return Pol::Layout::bytes(num_seqs);
}

template <class Pol>
cudaError_t launch_of(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int grid,
                      size_t smem, cudaStream_t stream)
{
    return launch_decode<Pol, 0>(tk, tv, p, grid, smem, stream);
}

template <int D, int G, int NQ>
using Pol = Bf16Policy<D, G * NQ,
                       D == 128 ? (G * NQ >= 16 ? PA_BF16_MQ_D128_NW_R16 : PA_BF16_MQ_D128_NW)
                                : PA_BF16_MQ_D64_NW,
                       D == 128 ? (G * NQ >= 16 ? PA_BF16_MQ_D128_STAGES_R16 : PA_BF16_MQ_D128_STAGES)
                                : PA_BF16_MQ_D64_STAGES,
                       NQ>;

template <int D, int G, int NQ>
const DecodeKernel kEntry = {reinterpret_cast<const void *>(&decode_kernel<Pol<D, G, NQ>>),
                             Pol<D, G, NQ>::NW * 32, &smem_of<Pol<D, G, NQ>>,
                             &launch_of<Pol<D, G, NQ>>};

template <int D>
const DecodeKernel *pick(int group, int nq)
{
    switch (group * 16 + nq) {
    case 1 * 16 + 2: return &kEntry<D, 1, 2>;
    case 1 * 16 + 4: return &kEntry<D, 1, 4>;
    case 1 * 16 + 8: return &kEntry<D, 1, 8>;
    case 2 * 16 + 2: return &kEntry<D, 2, 2>;
    case 2 * 16 + 4: return &kEntry<D, 2, 4>;
    case 2 * 16 + 8: return &kEntry<D, 2, 8>;
    case 4 * 16 + 2: return &kEntry<D, 4, 2>;
    case 4 * 16 + 4: return &kEntry<D, 4, 4>;
    case 8 * 16 + 2: return &kEntry<D, 8, 2>;
    default: return nullptr;
    }
}

} // namespace

const DecodeKernel *find_decode_kernel_bf16_mq(int d_h, int group, int nq)
{
    return d_h == 128 ? pick<128>(group, nq) : d_h == 64 ? pick<64>(group, nq) : nullptr;
}

} // namespace pa
