// Compiled head-group decode kernels for INT8 pools: head dim 128 and 64,
// group sizes 1..16, and the shared-prefix launch for groups 1..8.
#include "pa_decode_hg.cuh"

// Consumer warps per CTA (a multiple of 4; the head group is at most the
// largest power of two dividing it).
#ifndef PA_HG_INT8_NC
#define PA_HG_INT8_NC 12
#endif

namespace pa {
namespace {

constexpr int NC = PA_HG_INT8_NC;

template <int D, int GQ>
size_t hg_smem(int stages, int stage_bytes, int hg, int num_seqs)
{
    return HgSmem<D, GQ, NC>(stages, stage_bytes, hg).bytes(num_seqs);
}

template <class Pol, int PASS>
cudaError_t hg_launch(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int grid,
                      size_t smem, cudaStream_t stream)
{
    return launch_decode_hg<Pol, PASS, NC>(tk, tv, p, grid, smem, stream);
}

template <int D, int GQ>
using Pol = QuantMmaPolicy<8, D, GQ, NC, 1, 1, 1, 1, false>;

template <int D, int GQ, int PASS>
const HgKernel kHg = {reinterpret_cast<const void *>(&decode_hg_kernel<Pol<D, GQ>, PASS, NC>),
                      (NC + 1) * 32, NC, Pol<D, GQ>::TILE, &hg_smem<D, GQ>,
                      &hg_launch<Pol<D, GQ>, PASS>};

template <int D>
const HgKernel *pick(int group, bool share)
{
    if (share) {
        switch (group) {
        case 1: return &kHg<D, kShareMembers(1), 2>;
        case 2: return &kHg<D, 2 * kShareMembers(2), 2>;
        case 4: return &kHg<D, 4 * kShareMembers(4), 2>;
        case 8: return &kHg<D, 8 * kShareMembers(8), 2>;
        default: return nullptr;
        }
    }
    switch (group) {
    case 1: return &kHg<D, 1, 0>;
    case 2: return &kHg<D, 2, 0>;
    case 4: return &kHg<D, 4, 0>;
    case 8: return &kHg<D, 8, 0>;
    case 16: return &kHg<D, 16, 0>;
    default: return nullptr;
    }
}

} // namespace

const HgKernel *find_hg_kernel_int8(int d_h, int group, bool share)
{
    return d_h == 128 ? pick<128>(group, share) : d_h == 64 ? pick<64>(group, share) : nullptr;
}

} // namespace pa
