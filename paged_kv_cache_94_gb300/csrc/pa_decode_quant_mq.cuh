// Multi-query decode kernels on quantised pools (INT8 or INT4 codes): the
// NQ new tokens of a sequence attend causally over one read of each K/V tile,
// their G * NQ query rows on the tensor cores' N side (G * NQ <= 16). Each
// translation unit that includes this compiles one (BITS, D) family.
#pragma once

#include "pa_decode_kernel.cuh"

namespace pa {
namespace {

template <class Pol>
size_t mq_smem_of(int num_seqs)
{
    return Pol::Layout::bytes(num_seqs);
}

template <class Pol>
cudaError_t mq_launch_of(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p,
                         int grid, size_t smem, cudaStream_t stream)
{
    return launch_decode<Pol, 0>(tk, tv, p, grid, smem, stream);
}

// NW warps, S ring stages, BPI blocks per item, MINB resident CTAs per SM
// (16 query rows need their registers: one).
template <int BITS, int D, int G, int NQ, int NW, int S, int MINB, int BPI>
using MqPol = QuantMmaPolicy<BITS, D, G * NQ, NW, S, (G * NQ >= 16 ? 1 : MINB), BPI, NQ>;

template <int BITS, int D, int G, int NQ, int NW, int S, int MINB, int BPI>
const DecodeKernel kMqEntry = {
    reinterpret_cast<const void *>(&decode_kernel<MqPol<BITS, D, G, NQ, NW, S, MINB, BPI>>),
    MqPol<BITS, D, G, NQ, NW, S, MINB, BPI>::NW * 32,
    &mq_smem_of<MqPol<BITS, D, G, NQ, NW, S, MINB, BPI>>,
    &mq_launch_of<MqPol<BITS, D, G, NQ, NW, S, MINB, BPI>>};

template <int BITS, int D, int NW, int S, int MINB, int BPI>
const DecodeKernel *pick_quant_mq(int group, int nq)
{
    switch (group * 16 + nq) {
    case 1 * 16 + 2: return &kMqEntry<BITS, D, 1, 2, NW, S, MINB, BPI>;
    case 1 * 16 + 4: return &kMqEntry<BITS, D, 1, 4, NW, S, MINB, BPI>;
    case 1 * 16 + 8: return &kMqEntry<BITS, D, 1, 8, NW, S, MINB, BPI>;
    case 2 * 16 + 2: return &kMqEntry<BITS, D, 2, 2, NW, S, MINB, BPI>;
    case 2 * 16 + 4: return &kMqEntry<BITS, D, 2, 4, NW, S, MINB, BPI>;
    case 2 * 16 + 8: return &kMqEntry<BITS, D, 2, 8, NW, S, MINB, BPI>;
    case 4 * 16 + 2: return &kMqEntry<BITS, D, 4, 2, NW, S, MINB, BPI>;
    case 4 * 16 + 4: return &kMqEntry<BITS, D, 4, 4, NW, S, MINB, BPI>;
    case 8 * 16 + 2: return &kMqEntry<BITS, D, 8, 2, NW, S, MINB, BPI>;
    default: return nullptr;
    }
}

} // namespace
} // namespace pa
