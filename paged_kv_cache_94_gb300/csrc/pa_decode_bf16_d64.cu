// Compiled decode kernels: bf16 K/V, head dim 64, group sizes 1..16.
#include "pa_decode_kernel.cuh"

// Warps per CTA and ring stages per warp (overridable when building for a
// tuning sweep).
#ifndef PA_BF16_D64_NW
#define PA_BF16_D64_NW 4
#endif
#ifndef PA_BF16_D64_STAGES
#define PA_BF16_D64_STAGES 6
#endif

namespace pa {
namespace {

template <class Pol>
size_t smem_of(int num_seqs)
{
    return Pol::Layout::bytes(num_seqs);
}

template <class Pol, int PASS = 0>
cudaError_t launch_of(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int grid,
                      size_t smem, cudaStream_t stream)
{
    return launch_decode<Pol, PASS>(tk, tv, p, grid, smem, stream);
}

template <int G>
using Pol = Bf16Policy<64, G, PA_BF16_D64_NW, PA_BF16_D64_STAGES>;

template <int G>
const DecodeKernel kEntry = {reinterpret_cast<const void *>(&decode_kernel<Pol<G>>),
                             Pol<G>::NW * 32, &smem_of<Pol<G>>, &launch_of<Pol<G>>};

// Shared-prefix decode, one launch: group units (the query rows of
// up to kShareMembers(G) sequences, G heads each, share every K/V tile) and
// then every sequence's remaining blocks.
template <int G>
const DecodeKernel kPrefix = {
    reinterpret_cast<const void *>(&decode_kernel<Pol<G * kShareMembers(G)>, 2>),
    Pol<G * kShareMembers(G)>::NW * 32, &smem_of<Pol<G * kShareMembers(G)>>,
    &launch_of<Pol<G * kShareMembers(G)>, 2>};

} // namespace

const DecodeKernel *find_prefix_kernel_bf16_d64(int group)
{
    switch (group) {
    case 1: return &kPrefix<1>;
    case 2: return &kPrefix<2>;
    case 4: return &kPrefix<4>;
    case 8: return &kPrefix<8>;
    default: return nullptr;
    }
}

const DecodeKernel *find_decode_kernel_bf16_d64(int group)
{
    switch (group) {
    case 1: return &kEntry<1>;
    case 2: return &kEntry<2>;
    case 4: return &kEntry<4>;
    case 8: return &kEntry<8>;
    case 16: return &kEntry<16>;
    default: return nullptr;
    }
}

} // namespace pa
