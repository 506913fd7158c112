// Compiled decode kernels: int4 K/V, head dim 128, group sizes 1..16.
#include "pa_decode_kernel.cuh"

// Warps per CTA, ring stages per warp and the resident CTAs per SM the
// register budget targets (overridable when building for a tuning sweep).
#ifndef PA_INT4_D128_NW
#define PA_INT4_D128_NW 4
#endif
#ifndef PA_INT4_D128_MINB
#define PA_INT4_D128_MINB 3
#endif
#ifndef PA_INT4_D128_TMA
#define PA_INT4_D128_TMA 0 // 1: TMA boxes instead of per-lane 16-byte copies
#endif
#ifndef PA_INT4_D128_SHARE_TMA
#define PA_INT4_D128_SHARE_TMA PA_INT4_D128_TMA
#endif
#ifndef PA_INT4_D128_BPI
#define PA_INT4_D128_BPI 2 // blocks per ring item
#endif
#ifndef PA_INT4_D128_STAGES
#define PA_INT4_D128_STAGES 2
#endif

// The shared-prefix kernel keeps a GQ = g * members merge area per warp, so
// its ring uses one-block items to leave room for the same CTAs per SM.
#ifndef PA_INT4_D128_SHARE_BPI
#define PA_INT4_D128_SHARE_BPI 1
#endif
#ifndef PA_INT4_D128_SHARE_NW
#define PA_INT4_D128_SHARE_NW PA_INT4_D128_NW
#endif
#ifndef PA_INT4_D128_SHARE_MINB
#define PA_INT4_D128_SHARE_MINB PA_INT4_D128_MINB
#endif
#ifndef PA_INT4_D128_SHARE_STAGES
#define PA_INT4_D128_SHARE_STAGES 6
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
using Pol = QuantMmaPolicy<4, 128, G, PA_INT4_D128_NW, PA_INT4_D128_STAGES,
                           (G >= 16 ? 1 : PA_INT4_D128_MINB), // g = 16 needs its registers
                           PA_INT4_D128_BPI, 1, PA_INT4_D128_TMA != 0>;

template <int G>
const DecodeKernel kEntry = {reinterpret_cast<const void *>(&decode_kernel<Pol<G>>),
                             Pol<G>::NW * 32, &smem_of<Pol<G>>, &launch_of<Pol<G>>};

// Shared-prefix decode, one launch: group units (the query rows of
// up to kShareMembers(G) sequences, G heads each, share every K/V tile) and
// then every sequence's remaining blocks.
template <int G>
using PolShare = QuantMmaPolicy<4, 128, G, PA_INT4_D128_SHARE_NW, PA_INT4_D128_SHARE_STAGES,
                                (G >= 16 ? 1 : PA_INT4_D128_SHARE_MINB), PA_INT4_D128_SHARE_BPI, 1,
                                PA_INT4_D128_SHARE_TMA != 0>;

template <int G>
const DecodeKernel kPrefix = {
    reinterpret_cast<const void *>(&decode_kernel<PolShare<G * kShareMembers(G)>, 2>),
    PolShare<G * kShareMembers(G)>::NW * 32, &smem_of<PolShare<G * kShareMembers(G)>>,
    &launch_of<PolShare<G * kShareMembers(G)>, 2>};

} // namespace

const DecodeKernel *find_prefix_kernel_int4_d128(int group)
{
    switch (group) {
    case 1: return &kPrefix<1>;
    case 2: return &kPrefix<2>;
    case 4: return &kPrefix<4>;
    case 8: return &kPrefix<8>;
    default: return nullptr;
    }
}

const DecodeKernel *find_decode_kernel_int4_d128(int group)
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
