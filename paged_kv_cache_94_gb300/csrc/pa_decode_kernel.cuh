// The decode kernel template and its two compute policies.
//
//  Bf16Policy: K/V tiles in bf16; the g-wide contractions run on the tensor
//              cores with mma.sync m16n8k16 (bf16 in, fp32 accumulate):
//                S^T[16 tok][8 heads] = K[16 tok][D] . Q^T[D][8 heads]
//                O^T[D][8 heads]     += V^T[D][16 tok] . P^T[16 tok][8 heads]
//              Tokens sit on the M side, so the query group only pads N to 8;
//              P^T is moved from the accumulator layout to the B-operand
//              layout with movmatrix.
//  QuantMmaPolicy (pa_decode_quant.cuh): K/V tiles as INT8 or packed INT4
//              codes plus an fp32 scale per row ("kv-cache-guide"
//              (guijiagi.com) §4.2, dequantize_kv: x = code * scale); codes
//              become exact fp16 values and both contractions run as mma.sync
//              f16. The K scale multiplies the score, the V scale the softmax
//              weight.
#pragma once

#include "pa_decode.cuh"

namespace pa {

// L2 policy of the K/V tile loads: evict_first (the KV stream is read once;
// measured faster than evict_normal on every bf16 workload, and no slower on
// the shared-prefix INT8 one).
#ifndef PA_KV_EVICT_FIRST
#define PA_KV_EVICT_FIRST 1
#endif

// The running softmax base moves only when a tile's max exceeds it by more
// than this (log2 units): softmax weights stay <= 2^8 between rescales.
constexpr float kRescaleLog2 = 8.0f;

// Multi-query causal mask on one 16x8 score tile (rows: tokens gid, gid+8 of
// the block; columns: query rows nt*8 + 2*t4 + e). Query row v belongs to new
// token i = v / (GQ/NQ), which sees the block's first rem - (NQ-1-i) tokens,
// rem = ctx - (the block's first position), not clamped to the block.
template <int GQ, int NQ>
__device__ __forceinline__ void causal_mask(float (&sc)[4], int nt, int gid, int t4, int rem)
{
    constexpr int G = GQ / NQ;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int i = (nt * 8 + 2 * t4 + e) / G;
        const int vis = rem - (NQ - 1 - i);
        if (gid >= vis)
            sc[e] = -INFINITY;
        if (gid + 8 >= vis)
            sc[e + 2] = -INFINITY;
    }
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// ---------------------------------------------------------------------------
// bf16 K/V, tensor-core contractions.
// ---------------------------------------------------------------------------
// GQ query rows share each K/V tile: the g query heads of a kv head for each
// of NQ new tokens (NQ > 1: multi-query decode, each token masked causally).
template <int D_, int GQ_, int NW_, int S_, int NQ_ = 1>
struct Bf16Policy {
    static constexpr int D = D_, GQ = GQ_, NW = NW_, S = S_, NQ = NQ_;
    static constexpr int kMinBlocks = 1;
    static constexpr bool kLsuLoad = false;           // tiles arrive by TMA (lane 0 issues)
    static constexpr uint32_t kArrivals = 1;
    static constexpr int BPI = 1;                     // blocks per ring item
    static constexpr int NT = (GQ + 7) / 8;           // 8-head n-tiles
    static constexpr int KS = D / 16;                 // k-steps / m-tiles over D
    static constexpr int HALVES = D / 64;             // 64-column TMA boxes per tile
    static constexpr int TILE = kBlockTokens * D * 2; // bytes of a K (or V) tile
    static constexpr int STAGE = 2 * TILE;
    static constexpr int EXTRA = 0;
    static constexpr int QBYTES = 0;
    static constexpr uint32_t TX = STAGE;
    using Layout = SmemLayout<D, GQ, NW, S, STAGE, EXTRA, QBYTES>;

    struct State {
        uint32_t qf[NT][KS][2]; // Q^T B-fragments
        float m[NT][2], l[NT][2];
        float acc[NT][KS][4];   // O^T accumulators: rows d, cols heads
    };

    __device__ static uint32_t tx_bytes(uint32_t /*mask: 1*/) { return TX; }

    __device__ static void issue(uint32_t dst, uint32_t /*extra*/, const int32_t (&rows)[1],
                                 uint32_t bar, const CUtensorMap *tk, const CUtensorMap *tv,
                                 const DecodeParams & /*p*/, uint64_t pol)
    {
        const int32_t y = rows[0] * kBlockTokens;
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
            tma_load_2d(dst + h * (TILE / HALVES), tk, h * 64, y, bar, pol);
#pragma unroll
        for (int h = 0; h < HALVES; ++h)
            tma_load_2d(dst + TILE + h * (TILE / HALVES), tv, h * 64, y, bar, pol);
    }

    // Issue the loads of a segment's q fragments (they land while the
    // previous segment merges); finish_q completes them at segment start.
    // row_of(v): the q row of query row v, or -1 for a padding row.
    template <class RowFn>
    __device__ static void prefetch_q(State &st, const DecodeParams &p, RowFn row_of)
    {
        const int lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hl = nt * 8 + gid;
            const int64_t qr = hl < GQ ? row_of(hl) : -1;
            const bool ok = qr >= 0;
            const uint32_t *row = reinterpret_cast<const uint32_t *>(p.q + (ok ? qr : 0) * D);
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                st.qf[nt][kk][0] = ok ? __ldg(row + kk * 8 + t4) : 0u;
                st.qf[nt][kk][1] = ok ? __ldg(row + kk * 8 + 4 + t4) : 0u;
            }
        }
    }

    __device__ static void finish_q(State &) {}

    __device__ static void reset(State &st)
    {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                st.m[nt][e] = -INFINITY;
                st.l[nt][e] = 0.f;
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    st.acc[nt][mt][e] = 0.f;
        }
    }

    // One 16-token block: K tile at kt, V tile at kt + TILE (shared addresses).
    // Rows [lo, valid) of the block are attended; the others are masked. rem =
    // ctx - the block's first position (the multi-query causal limit).
    __device__ static void compute(State &st, uint32_t kt, uint32_t /*extra*/, int lo, int valid,
                                   int rem, float scale_log2, uint32_t /*mask: 1*/)
    {
        const int lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
        const int mi = lane >> 3, rr = lane & 7;
        const uint32_t vt = kt + TILE;

        // ---- scores S^T = K Q^T (two accumulator chains for ILP)
        float s0[NT][4], s1[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                s0[nt][e] = s1[nt][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            const int tok = rr + ((mi & 1) << 3);
            const int chunk = 2 * kk + (mi >> 1);
            const uint32_t addr = kt + (chunk >> 3) * (TILE / HALVES) + (uint32_t)(tok * 128) +
                                  (uint32_t)(((chunk & 7) ^ rr) << 4);
            uint32_t a0, a1, a2, a3;
            ldmatrix_x4(addr, a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (kk & 1)
                    mma_bf16_16816(s1[nt], a0, a1, a2, a3, st.qf[nt][kk][0], st.qf[nt][kk][1]);
                else
                    mma_bf16_16816(s0[nt], a0, a1, a2, a3, st.qf[nt][kk][0], st.qf[nt][kk][1]);
            }
        }

        // ---- online softmax (columns = heads; rows = tokens gid, gid+8)
        const bool lo_ok = gid >= lo && gid < valid, hi_ok = gid + 8 >= lo && gid + 8 < valid;
        uint32_t pb0[NT], pb1[NT], pl0[NT], pl1[NT];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            float sc[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sc[e] = (s0[nt][e] + s1[nt][e]) * scale_log2;
            if (!lo_ok) {
                sc[0] = -INFINITY;
                sc[1] = -INFINITY;
            }
            if (!hi_ok) {
                sc[2] = -INFINITY;
                sc[3] = -INFINITY;
            }
            if constexpr (NQ > 1)
                causal_mask<GQ, NQ>(sc, nt, gid, t4, rem);
            // Lazy rescale: the running base m only moves when a tile's max
            // exceeds it by more than 2^kRescaleLog2; otherwise weights up to
            // 2^kRescaleLog2 are accumulated against the old base (exact: acc
            // and l always share one base).
            float alpha[2];
            bool need = false;
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float mx = fmaxf(sc[e], sc[e + 2]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const bool up = mx > st.m[nt][e] + kRescaleLog2;
                const float mnew = up ? mx : st.m[nt][e];
                alpha[e] = up ? fast_exp2(st.m[nt][e] - mnew) : 1.f;
                need |= up;
                st.m[nt][e] = mnew;
                const float base = (mnew == -INFINITY) ? 0.f : mnew;
                sc[e] = fast_exp2(sc[e] - base);
                sc[e + 2] = fast_exp2(sc[e + 2] - base);
            }
            if (__any_sync(0xffffffffu, need)) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    st.l[nt][e] *= alpha[e];
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        st.acc[nt][mt][e] *= alpha[e];
                        st.acc[nt][mt][e + 2] *= alpha[e];
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 2; ++e)
                st.l[nt][e] += sc[e] + sc[e + 2];
            // The weights go to the tensor cores as two bf16 parts, P = hi + lo
            // (hi = bf16(P), lo = bf16(P - hi)): 16 significant bits instead of
            // 8, so the weighted sum stays accurate when V rows differ in
            // magnitude by orders and their terms cancel.
            const uint32_t h0 = pack_bf16x2(sc[0], sc[1]), h1 = pack_bf16x2(sc[2], sc[3]);
            const uint32_t r0 = pack_bf16x2(sc[0] - __uint_as_float(h0 << 16),
                                            sc[1] - __uint_as_float(h0 & 0xffff0000u));
            const uint32_t r1 = pack_bf16x2(sc[2] - __uint_as_float(h1 << 16),
                                            sc[3] - __uint_as_float(h1 & 0xffff0000u));
            pb0[nt] = movmatrix_trans(h0);
            pb1[nt] = movmatrix_trans(h1);
            pl0[nt] = movmatrix_trans(r0);
            pl1[nt] = movmatrix_trans(r1);
        }

        // ---- O^T += V^T P^T. Rows of V outside [lo, valid) may hold anything
        // (even NaN): their operand halves are zeroed, since 0 * NaN is NaN.
        if (lo == 0 && valid == kBlockTokens) {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4_trans(v_addr(vt, mt, mi, rr), a0, a1, a2, a3);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_bf16_16816(st.acc[nt][mt], a0, a1, a2, a3, pb0[nt], pb1[nt]);
                    mma_bf16_16816(st.acc[nt][mt], a0, a1, a2, a3, pl0[nt], pl1[nt]);
                }
            }
        } else {
            const int t0 = 2 * t4;
            auto in = [&](int t) { return t >= lo && t < valid; };
            const uint32_t mlo = (in(t0) ? 0x0000ffffu : 0u) | (in(t0 + 1) ? 0xffff0000u : 0u);
            const uint32_t mhi = (in(t0 + 8) ? 0x0000ffffu : 0u) | (in(t0 + 9) ? 0xffff0000u : 0u);
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                uint32_t a0, a1, a2, a3;
                ldmatrix_x4_trans(v_addr(vt, mt, mi, rr), a0, a1, a2, a3);
                a0 &= mlo;
                a1 &= mlo;
                a2 &= mhi;
                a3 &= mhi;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    mma_bf16_16816(st.acc[nt][mt], a0, a1, a2, a3, pb0[nt], pb1[nt]);
                    mma_bf16_16816(st.acc[nt][mt], a0, a1, a2, a3, pl0[nt], pl1[nt]);
                }
            }
        }
    }

    // ldmatrix.trans row address of V^T m-tile mt: matrices (tokens 0-7 | 8-15)
    // x (d 16mt..+7 | +8..+15) in the order a0..a3 expects.
    __device__ static uint32_t v_addr(uint32_t vt, int mt, int mi, int rr)
    {
        const int tok = rr + ((mi >> 1) << 3);
        const int chunk = 2 * mt + (mi & 1);
        return vt + (chunk >> 3) * (TILE / HALVES) + (uint32_t)(tok * 128) +
               (uint32_t)(((chunk & 7) ^ rr) << 4);
    }

    // This warp's state -> its slice of the merge area: [warp][h] = (m, l, acc[D]).
    __device__ static void to_merge(const State &st, float *merge)
    {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float l = st.l[nt][e];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                const int h = nt * 8 + 2 * t4 + e;
                if (h < GQ) {
                    float *mb = merge + (warp * GQ + h) * (D + 2);
                    if (gid == 0) {
                        mb[0] = st.m[nt][e];
                        mb[1] = l;
                    }
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        mb[2 + 16 * mt + gid] = st.acc[nt][mt][e];
                        mb[2 + 16 * mt + gid + 8] = st.acc[nt][mt][e + 2];
                    }
                }
            }
    }
};

} // namespace pa

#include "pa_decode_quant.cuh"

namespace pa {

// ---------------------------------------------------------------------------
// The kernel: split, ring, segments, merge.
// ---------------------------------------------------------------------------
// PASS 0: decode of each sequence. PASS 2: shared-prefix decode, the groups'
// shared blocks (all query rows of the group at once) and then every
// sequence's remaining blocks, in one launch.
template <class Pol, int PASS = 0>
__global__ void __launch_bounds__(Pol::NW * 32, Pol::kMinBlocks)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeParams p)
{
    constexpr int NW = Pol::NW, S = Pol::S, D = Pol::D, GQ = Pol::GQ;
    using L = typename Pol::Layout;
    static_assert(NW <= 16, "misc scratch holds 16 warp sums");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::kOffBars);
    int32_t *meta = reinterpret_cast<int32_t *>(smem + L::kOffMeta);
    float *merge = reinterpret_cast<float *>(smem + L::kOffMerge);
    float *sink_sc = reinterpret_cast<float *>(smem + L::kOffSinkSc);
    int32_t *misc = reinterpret_cast<int32_t *>(smem + L::kOffMisc);
    int32_t *P = reinterpret_cast<int32_t *>(smem + L::kOffPrefix);

    // The launch may start before the previous kernel on the stream ends (a
    // programmatic dependent launch: the cache append, or the group
    // detection): wait for it to complete before the first read.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n_h = p.n_kv * (GQ / Pol::NQ); // query heads per token

    if (tid == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    constexpr int BPI = Pol::BPI;                // blocks per item
    constexpr int TOK = BPI * kBlockTokens;      // tokens per item
    prefix_blocks<NW * 32, PASS, BPI>(p, P, misc + 8);
    __syncthreads();
    if constexpr (PASS == 0) {
        zero_empty_sequences<D, Pol::NQ>(p, P, n_h);
    } else if constexpr (PASS == 2) {
        // sequences with no blocks (ctx 0 or invalid) sit after the group units
        const int nh = p.n_kv * p.g;
        const int rows16 = nh * D * 2 / 16;
        for (int b = blockIdx.x; b < p.num_real; b += p.num_ctas) {
            if (P[p.num_real + b + 1] != P[p.num_real + b])
                continue;
            uint4 *dst = reinterpret_cast<uint4 *>(p.out + (size_t)b * nh * D);
            for (int i = threadIdx.x; i < rows16; i += blockDim.x)
                dst[i] = make_uint4(0, 0, 0, 0);
        }
    }
    // Cost-weighted split on the virtual line (see virt_first). A CTA whose
    // virtual range holds no block does nothing; the CTAs owning a (sequence,
    // kv head) are exactly the owners of its first through last block, which
    // the split merge counts on.
    const int64_t Wv = virt_total(p, P);
    int64_t G = plan_ctas(p.num_ctas, Wv);
    int64_t lo, hi;
    const int64_t U = PASS == 0 ? whole_unit_grid<NW * 32>(p, P, G, misc + 8) : 0;
    if (U > 0) { // one CTA per unit: every segment is a whole unit
        if ((int64_t)blockIdx.x >= U)
            return;
        unit_items(p, P, blockIdx.x, lo, hi);
        G = U;
    } else {
        if ((int64_t)blockIdx.x >= G)
            return;
        lo = real_at_virtual(p, P, plan_lo(blockIdx.x, Wv, G));
        hi = real_at_virtual(p, P, plan_lo(blockIdx.x + 1, Wv, G));
    }

    if (lane == 0)
        for (int s = 0; s < S; ++s)
            mbar_init(smem_u32(&bars[warp * S + s]), Pol::kArrivals);
    fence_barrier_init();
    __syncthreads();

    // ---- per-warp producer state
    WarpRing<BPI> r;
    r.lo = lo;
    r.warp = warp;
    r.n_items = (hi - lo > warp) ? (hi - lo - warp + NW - 1) / NW : 0;
    r.issued = 0;
    r.batch = 0;
    load_item<NW, PASS>(p, P, r, lane, r.phys_cur, r.kvh_cur);
    load_item<NW, PASS>(p, P, r, 32 + lane, r.phys_next, r.kvh_next);
    const uint64_t pol = PA_KV_EVICT_FIRST ? l2_policy_evict_first() : l2_policy_evict_normal();
    const uint32_t ring_base = smem_u32(smem) + (uint32_t)(warp * S * Pol::STAGE);
    const uint32_t extra_base = smem_u32(smem + L::kOffExtra) + (uint32_t)(warp * S * Pol::EXTRA);
    const uint32_t bar_base = smem_u32(&bars[warp * S]);
    int32_t *wmeta = meta + warp * S;
    float *qsm = reinterpret_cast<float *>(smem + L::kOffQ) + warp * (Pol::QBYTES / 4);
    bool dead = false;    // a wait timed out: stop issuing, skip work
    int64_t fail_k = -1;  // first item whose wait timed out
    int istage = 0;       // ring stage the next issue goes to

    auto issue_next = [&]() {
        const int64_t k = r.issued;
        const int64_t bt = k >> 5;
        if (bt != r.batch) {
#pragma unroll
            for (int j = 0; j < BPI; ++j)
                r.phys_cur[j] = r.phys_next[j];
            r.kvh_cur = r.kvh_next;
            r.batch = bt;
            load_item<NW, PASS>(p, P, r, (bt + 1) * 32 + lane, r.phys_next, r.kvh_next);
        }
        const int32_t kw = __shfl_sync(0xffffffffu, r.kvh_cur, (int)(k & 31));
        const int32_t kvh = kw & 0xffff;
        // rows of the item's blocks in the pool; mask: the blocks to load
        int32_t rows[BPI];
        uint32_t mask = 0;
        bool bad = false;
#pragma unroll
        for (int j = 0; j < BPI; ++j) {
            const int32_t phys = __shfl_sync(0xffffffffu, r.phys_cur[j], (int)(k & 31));
            const bool absent = (kw >> (16 + j)) & 1;
            const bool bad_j = !absent && (phys < 0 || (int64_t)phys >= p.num_blocks);
            bad |= bad_j;
            rows[j] = (absent || bad_j) ? -1 : phys * p.n_kv + kvh;
            mask |= (rows[j] >= 0 ? 1u : 0u) << j;
        }
        const uint32_t bar = bar_base + 8u * istage;
        if (lane == 0) {
            wmeta[istage] = (int32_t)mask;
            if (bad)
                flag_error(p.dev_status, PA_DEV_BAD_BLOCK_BIT);
        }
        if constexpr (Pol::kLsuLoad) {
            // every lane copies its share and arrives when its copies land
            if (mask == 0) {
                mbar_arrive(bar); // the phase completes with no data: the item is skipped
            } else {
                Pol::issue_lanes(ring_base + (uint32_t)(istage * Pol::STAGE),
                                 extra_base + (uint32_t)(istage * Pol::EXTRA), rows, p, p.k_cache,
                                 p.v_cache, pol, lane);
                cp_async_mbar_arrive_noinc(bar);
            }
        } else if (lane == 0) {
            if (mask == 0) {
                mbar_arrive(bar); // completes the phase with no data: the item is skipped
            } else {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bar, Pol::tx_bytes(mask));
                Pol::issue(ring_base + (uint32_t)(istage * Pol::STAGE),
                           extra_base + (uint32_t)(istage * Pol::EXTRA), rows, bar, &tmK, &tmV,
                           p, pol);
            }
        }
        __syncwarp();
        istage = (istage + 1 == S) ? 0 : istage + 1;
        r.issued = k + 1;
    };

    for (int s = 0; s < S; ++s)
        if (r.issued < r.n_items)
            issue_next();

    typename Pol::State st;
    int64_t k = 0;        // items of this warp consumed so far
    int cstage = 0;       // ring stage of item k
    uint32_t cphase = 0;  // barrier phase parity of item k
    int64_t seg_lo = lo;
    int b, kvh, i0, nb;
    auto rows = [&](int s, int kh) {
        return [&p, s, kh](int v) { return unit_row<GQ, Pol::NQ, PASS>(p, s, kh, v); };
    };
    if (seg_lo < hi) {
        locate_item(seg_lo, P, p.num_seqs, p.n_kv, b, kvh, i0, nb);
        Pol::prefetch_q(st, p, rows(b, kvh));
    }
    // the next segment's context length, loaded with its q (pass 0)
    int32_t ctx_next = (PASS == 0 && seg_lo < hi) ? __ldg(p.context_lens + b) : 0;
    while (seg_lo < hi) {
        const int i0_cur = i0;
        const int64_t unit_start = seg_lo - i0;
        const int64_t unit_end = unit_start + nb;
        const int64_t seg_hi = unit_end < hi ? unit_end : hi;
        const bool whole = (i0 == 0) && (unit_end <= hi);
        // Attended positions: [ws, ctx); the pool serves [max(ws, n_sink), ctx)
        // from logical block fb on, the sink rows serve [ws, min(n_sink, ctx)).
        // Pass 2: a group's shared blocks are all full; a sequence's own
        // blocks start after its group's, at block fb = skip[b].
        int32_t ctx, ws, pool_from, fb;
        if constexpr (PASS == 2) {
            ws = pool_from = 0;
            if (b < p.num_real) { // a group's shared blocks, all full
                ctx = __ldg(p.groups + 3 * b + 2) * kBlockTokens;
                fb = 0;
            } else {              // a sequence's blocks after its group's prefix
                ctx = __ldg(p.context_lens + (b - p.num_real));
                fb = __ldg(p.skip + (b - p.num_real));
            }
        } else {
            ctx = ctx_next;
            ws = window_start(p, ctx);
            pool_from = ws > p.n_sink ? ws : p.n_sink;
            fb = seq_first_block(p, ctx);
        }

        Pol::finish_q(st);
        Pol::reset(st);
        int64_t x = lo + warp + k * NW;
        while (k < r.n_items && x < seg_hi) {
            bool ok = !dead;
            // every lane waits (acquire); the warp agrees on the outcome
            if (ok && !__all_sync(0xffffffffu, mbar_wait(bar_base + 8u * cstage, cphase))) {
                ok = false;
                dead = true;
                fail_k = k;
                if (lane == 0)
                    flag_error(p.dev_status, PA_DEV_TIMEOUT_BIT);
            }
            const int32_t mask = ok ? wmeta[cstage] : 0;
            if (mask != 0) {
                const int32_t t0 = (fb + BPI * (int32_t)(x - unit_start)) * kBlockTokens;
                const int lo = pool_from > t0 ? (int)min(pool_from - t0, TOK) : 0;
                const int rem = (int)min(ctx - t0, TOK + kBlockTokens); // >= TOK + NQ - 1
                const int valid = (int)min(rem, TOK);
                // (mask: the item's blocks that were loaded; a bad one is not attended)
                if (lo < valid)
                    Pol::compute(st, ring_base + (uint32_t)(cstage * Pol::STAGE),
                                 extra_base + (uint32_t)(cstage * Pol::EXTRA), lo, valid, rem,
                                 p.scale_log2, (uint32_t)mask);
            }
            __syncwarp();
            if (!dead && r.issued < r.n_items)
                issue_next();
            ++k;
            x += NW;
            if (++cstage == S) {
                cstage = 0;
                cphase ^= 1u;
            }
        }
        // the next segment's q loads overlap this segment's merge
        const int b_cur = b, kvh_cur = kvh;
        const int64_t nb_cur = nb;
        if (seg_hi < hi) {
            locate_item(seg_hi, P, p.num_seqs, p.n_kv, b, kvh, i0, nb);
            Pol::prefetch_q(st, p, rows(b, kvh));
            if constexpr (PASS == 0)
                ctx_next = __ldg(p.context_lens + b);
        }
        Pol::to_merge(st, merge);
        __syncthreads();
        const int32_t s_hi = (PASS == 0 && i0_cur == 0 && p.n_sink > ws) ? min(p.n_sink, ctx) : 0;
        if constexpr (PASS == 2)
            finish_fused<D, GQ, NW>(p, P, merge, misc, b_cur, kvh_cur, Wv, G, whole);
        else
            finish_segment<D, GQ, NW, Pol::NQ>(p, P, merge, misc, sink_sc, b_cur, kvh_cur,
                                               (int)nb_cur, Wv, G, whole, ws,
                                               s_hi > ws ? s_hi : ws);
        seg_lo = seg_hi;
    }

    // After a timeout, give the copies still in flight a bounded chance to
    // land before the CTA's shared memory is released.
    if constexpr (Pol::kLsuLoad) {
        cp_async_wait_all(); // this thread's own copies: ends when they land
    } else if (dead && lane == 0) {
        for (int64_t kk = fail_k; kk < r.issued; ++kk)
            mbar_wait(bar_base + 8u * (uint32_t)(kk % S), (uint32_t)((kk / S) & 1));
    }
}

// Launch of decode_kernel<Pol, PASS> as a programmatic dependent launch: its
// CTAs are scheduled while the previous kernel on the stream (the cache
// append, or the group detection) finishes, and wait for that kernel's
// completion in their first instruction. After anything else on the stream
// it behaves as a plain launch.
template <class Pol, int PASS>
cudaError_t launch_decode(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p,
                          int grid, size_t smem, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Pol::NW * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_kernel<Pol, PASS>, tk, tv, p);
}

} // namespace pa
