// Head-group decode kernel for quantised (INT8 / INT4) pools.
//
// Same result as decode_kernel (pa_decode_kernel.cuh): per sequence b and
// query head h, softmax(scale * q K_b^T) V_b over the b's cached tokens
// ("LLM 推理底层：KV Cache 显存几何、GQA/MLA 压缩与 PagedAttention 调度", eq. for
// o_t), read through the block table (same page, "逻辑块与物理块映射"), with
// codes and per-token scales dequantised as "kv-cache-guide" §4.2 states.
// What differs is how the bytes travel:
//
//  * An item is ONE physical block of HG consecutive kv heads. The pool
//    layout [num_blocks][n_kv][16][d_h] keeps those HG tiles adjacent, and
//    the scale layout [num_blocks][n_kv][16] keeps their scale rows
//    adjacent, so an item is two contiguous runs of codes (K, V) and two of
//    scales: four bulk copies, instead of 2 HG tiles and 2 HG 64-byte scale
//    rows scattered over the pool.
//  * One producer warp streams items into a CTA-wide ring of S stages with
//    TMA (codes: one 2-D box of HG x 16 rows; scales: one 1-D bulk copy),
//    one "full" mbarrier per stage counting the bytes in.
//  * NC = 8 consumer warps; warp w serves head slot w % HG of every item
//    whose index is = w / HG (mod WS = 8 / HG). S is a multiple of WS, so a
//    stage is only ever read by one warp set, fill after fill. The HG warps
//    that consumed a stage release it on its "empty" mbarrier and the
//    producer refills it.
//  * Units of the work line are (sequence, head group); the cost-weighted
//    split, the segment merges, the split-context log-sum-exp reduce and the
//    shared-prefix merge are those of decode_kernel, done over the HG heads
//    of a unit by the consumer warps (named barrier 1; the producer never
//    joins a CTA barrier after the set-up).
// Every wait is bounded (about one second) and reports PA_DEV_TIMEOUT.
#pragma once

#include "pa_decode_kernel.cuh"

namespace pa {

// NC consumer warps (a multiple of 4: a power of two times 1 or 3) plus one
// producer warp.
template <int NC>
__device__ __forceinline__ void consumer_sync()
{
    asm volatile("bar.sync 1, %0;" ::"r"(NC * 32) : "memory");
}

// Runtime carve-up of the head-group kernel's shared memory (offsets from a
// 1024-aligned base). S stages of stage_bytes (a multiple of 1024), then the
// barriers, per-stage masks, the consumers' merge area, sink scores, scratch
// and the per-sequence prefix arrays.
template <int D, int GQ, int NC>
struct HgSmem {
    uint32_t bars, meta, merge, sink, misc, prefix;
    __host__ __device__ HgSmem(int stages, int stage_bytes, int hg)
    {
        bars = (uint32_t)(stages * stage_bytes);
        meta = bars + 16u * stages;
        merge = (meta + 4u * stages + 15u) / 16u * 16u;
        sink = merge + (uint32_t)(NC * GQ * (D + 2) * 4);
        misc = sink + (uint32_t)(hg * GQ * 16 * 4);
        prefix = misc + 128u;
    }
    __host__ __device__ size_t bytes(int num_seqs) const
    {
        return 1024 + prefix + 6 * (size_t)(num_seqs + 1);
    }
};

// End of a segment over HG heads: the consumers' states (merge area [NC][GQ]
// of (m, l, acc[D]); head slot s sits in warps s, s + HG, ...) -> the output,
// or a partial record of the unit when it is split over CTAs; the last CTA
// to publish a record for the unit merges all records. Called by the
// consumer threads.
template <int D, int GQ, int NQ, int NC>
__device__ __forceinline__ void hg_finish_segment(const DecodeParams &p, const int32_t *P,
                                                  const float *merge, int32_t *misc,
                                                  float *sink_sc, int b, int hgi, int nb,
                                                  int64_t Wv, int64_t G, bool whole, int s_lo,
                                                  int s_hi)
{
    constexpr int NT = NC * 32;
    constexpr int REC = D + 2;
    const int HG = p.hg, WS = NC / HG;
    const int u = b * p.ups + hgi;
    const int rows = HG * GQ;
    float *rec = p.partials + ((size_t)blockIdx.x + u) * ((size_t)rows * REC);
    const int ns = s_hi - s_lo;
    if (ns > 0) { // sink-row scores of every head of the group: one warp per (row, sink row)
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int t = warp; t < rows * ns; t += NC) {
            const int r = t / ns, j = s_lo + t % ns;
            const int hs = r / GQ, h = r - hs * GQ, kvh = hgi * HG + hs;
            const __nv_bfloat16 *k = p.sink_k + ((size_t)b * p.n_kv + kvh) * p.n_sink * D;
            const __nv_bfloat16 *q = p.q + qo_row<GQ, NQ>(p, b, kvh, h) * D;
            float a = 0.f;
#pragma unroll
            for (int d = lane; d < D; d += 32)
                a = fmaf(__bfloat162float(q[d]), __bfloat162float(k[j * D + d]), a);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
                a += __shfl_xor_sync(0xffffffffu, a, o);
            if (lane == 0)
                sink_sc[r * 16 + (j - s_lo)] = a * p.scale_log2;
        }
        consumer_sync<NC>();
    }
#pragma unroll 1
    for (int idx = threadIdx.x; idx < rows * D; idx += NT) {
        const int r = idx / D, d = idx - r * D;
        const int hs = r / GQ, h = r - hs * GQ, kvh = hgi * HG + hs;
        float M = -INFINITY;
        for (int j = 0; j < WS; ++j)
            M = fmaxf(M, merge[((hs + j * HG) * GQ + h) * REC]);
        for (int j = 0; j < ns; ++j)
            M = fmaxf(M, sink_sc[r * 16 + j]);
        float O = 0.f, L = 0.f;
        if (M != -INFINITY) {
            for (int j = 0; j < WS; ++j) {
                const float *mb = merge + ((hs + j * HG) * GQ + h) * REC;
                const float sc = (mb[0] == -INFINITY) ? 0.f : fast_exp2(mb[0] - M);
                L = fmaf(sc, mb[1], L);
                O = fmaf(sc, mb[2 + d], O);
            }
            if (ns > 0) {
                const __nv_bfloat16 *sv = p.sink_v + ((size_t)b * p.n_kv + kvh) * p.n_sink * D;
                for (int j = 0; j < ns; ++j) {
                    const float e = fast_exp2(sink_sc[r * 16 + j] - M);
                    L += e;
                    O = fmaf(e, __bfloat162float(sv[(s_lo + j) * D + d]), O);
                }
            }
        }
        if (whole) {
            p.out[qo_row<GQ, NQ>(p, b, kvh, h) * D + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
        } else {
            if (d == 0) {
                rec[r * REC] = M;
                rec[r * REC + 1] = L;
            }
            rec[r * REC + 2 + d] = O;
        }
    }
    consumer_sync<NC>(); // every record store of this CTA is done (CTA scope)
    if (whole)
        return;
    const int64_t v0 = virt_first(p, P, b, hgi, nb);
    const int64_t c_first = plan_owner(v0, Wv, G);
    const int nseg = (int)(plan_owner(v0 + nb - 1, Wv, G) - c_first + 1);
    if (threadIdx.x == 0) {
        const int old = atomic_add_acq_rel_gpu(&p.counters[u], 1);
        const int last = (old == nseg - 1);
        if (last)
            p.counters[u] = 0; // every arrival of this launch is in: reset for the next call
        misc[0] = last;
    }
    consumer_sync<NC>();
    const bool last = misc[0] != 0;
    consumer_sync<NC>(); // misc is reused by the next segment
    if (!last)
        return;
    const float *base = p.partials + ((size_t)c_first + u) * ((size_t)rows * REC);
#pragma unroll 1
    for (int idx = threadIdx.x; idx < rows * D; idx += NT) {
        const int r = idx / D, d = idx - r * D;
        const int hs = r / GQ, h = r - hs * GQ, kvh = hgi * HG + hs;
        float M = -INFINITY;
        for (int s = 0; s < nseg; ++s)
            M = fmaxf(M, __ldcg(base + (size_t)s * rows * REC + r * REC));
        float O = 0.f, L = 0.f;
        if (M != -INFINITY) {
            for (int s = 0; s < nseg; ++s) {
                const float *rr = base + (size_t)s * rows * REC + r * REC;
                const float m = __ldcg(rr);
                const float sc = (m == -INFINITY) ? 0.f : fast_exp2(m - M);
                L = fmaf(sc, __ldcg(rr + 1), L);
                O = fmaf(sc, __ldcg(rr + 2 + d), O);
            }
        }
        p.out[qo_row<GQ, NQ>(p, b, kvh, h) * D + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
    }
}

// ---------------------------------------------------------------------------
// Shared-prefix pass (PASS 2) over head groups. Units s < num_real are
// groups (rows: the g heads of every member), units s >= num_real sequence
// b = s - num_real's blocks after its group's prefix; as finish_fused.
// ---------------------------------------------------------------------------
template <int D, int GQ>
__device__ __forceinline__ void hg_merge_element(const DecodeParams &p, int b, int hgi, int hs,
                                                 int64_t c_first, int nseg, int h, int d)
{
    constexpr int REC = D + 2;
    const int rows = p.hg * GQ;
    const int u = (p.num_real + b) * p.ups + hgi;
    const float *base =
        p.partials + ((size_t)c_first + u) * ((size_t)rows * REC) + (hs * GQ + h) * REC;
    const int kvh = hgi * p.hg + hs;
    const int64_t row = ((int64_t)b * p.n_kv + kvh) * p.g + h;
    float M = -INFINITY, pm = -INFINITY, pl = 0.f, po = 0.f;
    if (__ldg(p.skip + b) > 0) {
        const float *pr = p.pre + row * REC;
        pm = __ldcg(pr);
        pl = __ldcg(pr + 1);
        po = __ldcg(pr + 2 + d);
        M = pm;
    }
    for (int j = 0; j < nseg; ++j)
        M = fmaxf(M, __ldcg(base + (size_t)j * rows * REC));
    float O = 0.f, L = 0.f;
    if (M != -INFINITY) {
        if (pm != -INFINITY) {
            const float sc = fast_exp2(pm - M);
            L = sc * pl;
            O = sc * po;
        }
        for (int j = 0; j < nseg; ++j) {
            const float *r = base + (size_t)j * rows * REC;
            const float m = __ldcg(r);
            const float sc = (m == -INFINITY) ? 0.f : fast_exp2(m - M);
            L = fmaf(sc, __ldcg(r + 1), L);
            O = fmaf(sc, __ldcg(r + 2 + d), O);
        }
    }
    p.out[row * D + d] = __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
}

// One arrival on sequence b's counter for head group hgi (expects its nseg
// record owners, +1 for a group member). True for the last arrival, which
// then merges; the counter is reset for the next launch.
__device__ __forceinline__ bool hg_arrive_one(const DecodeParams &p, const int32_t *P, int b,
                                              int hgi, int64_t Wv, int64_t G, int64_t &c_first,
                                              int &nseg)
{
    const int s = p.num_real + b, u = s * p.ups + hgi;
    unit_owners(p, P, s, hgi, Wv, G, c_first, nseg);
    const int expect = nseg + (__ldg(p.skip + b) > 0 ? 1 : 0);
    const int old = atomic_add_acq_rel_gpu(&p.counters[u], 1);
    const bool last = (old == expect - 1);
    if (last)
        p.counters[u] = 0;
    return last;
}

// Arrivals of sequences b0 .. b0 + n - 1 (n <= 8) for head group hgi, one
// thread each, then the merges of those that came last (all consumers).
template <int D, int GQ, int NC>
__device__ __forceinline__ void hg_arrive_sequences(const DecodeParams &p, const int32_t *P,
                                                    int32_t *misc, int b0, int n, int hgi,
                                                    int64_t Wv, int64_t G)
{
    constexpr int NT = NC * 32;
    int32_t *last = misc, *cf = misc + 8, *ns = misc + 16;
    if (threadIdx.x < n) {
        int64_t c_first;
        int nseg;
        const bool l = hg_arrive_one(p, P, b0 + threadIdx.x, hgi, Wv, G, c_first, nseg);
        last[threadIdx.x] = l;
        cf[threadIdx.x] = (int32_t)c_first;
        ns[threadIdx.x] = nseg;
    }
    consumer_sync<NC>();
    const int per = p.hg * p.g * D; // a sequence's rows of this head group
#pragma unroll 1
    for (int idx = threadIdx.x; idx < n * per; idx += NT) {
        const int j = idx / per, r = idx - j * per;
        const int row = r / D, d = r - row * D;
        const int hs = row / p.g, h = row - hs * p.g;
        if (last[j])
            hg_merge_element<D, GQ>(p, b0 + j, hgi, hs, cf[j], ns[j], h, d);
    }
    consumer_sync<NC>(); // misc is reused by the next segment
}

template <int D, int GQ, int NC>
__device__ __forceinline__ void hg_finish_fused(const DecodeParams &p, const int32_t *P,
                                                const float *merge, int32_t *misc, int s,
                                                int hgi, int64_t Wv, int64_t G, bool whole)
{
    constexpr int NT = NC * 32, REC = D + 2;
    const int HG = p.hg, WS = NC / HG;
    const bool group = s < p.num_real;
    const int b = s - p.num_real;
    const bool member = !group && __ldg(p.skip + b) > 0;
    const int u = s * p.ups + hgi;
    const int rows = HG * GQ;
    float *rec = p.partials + ((size_t)blockIdx.x + u) * ((size_t)rows * REC);
    const bool direct = whole && !group && !member; // a plain sequence in one piece
    // live query rows per head: a group's members' heads, else the sequence's g heads
    const int live = group ? __ldg(p.groups + 3 * s + 1) * p.g : p.g;
#pragma unroll 1
    for (int idx = threadIdx.x; idx < rows * D; idx += NT) {
        const int r = idx / D, d = idx - r * D;
        const int hs = r / GQ, h = r - hs * GQ;
        if (h >= live)
            continue;
        float M = -INFINITY;
        for (int j = 0; j < WS; ++j)
            M = fmaxf(M, merge[((hs + j * HG) * GQ + h) * REC]);
        float O = 0.f, L = 0.f;
        if (M != -INFINITY) {
            for (int j = 0; j < WS; ++j) {
                const float *mb = merge + ((hs + j * HG) * GQ + h) * REC;
                const float sc = (mb[0] == -INFINITY) ? 0.f : fast_exp2(mb[0] - M);
                L = fmaf(sc, mb[1], L);
                O = fmaf(sc, mb[2 + d], O);
            }
        }
        if (direct) {
            const int kvh = hgi * HG + hs;
            p.out[(((int64_t)b * p.n_kv + kvh) * p.g + h) * D + d] =
                __float2bfloat16_rn(L > 0.f ? O / L : 0.f);
        } else {
            if (d == 0) {
                rec[r * REC] = M;
                rec[r * REC + 1] = L;
            }
            rec[r * REC + 2 + d] = O;
        }
    }
    consumer_sync<NC>();
    if (direct)
        return;
    if (!group) { // a piece of sequence b: one arrival
        hg_arrive_sequences<D, GQ, NC>(p, P, misc, b, 1, hgi, Wv, G);
        return;
    }
    // a piece of group s: the last one merges the group's records into the
    // members' prefix states, then arrives once on every member's counter
    if (threadIdx.x == 0) {
        int64_t c_first;
        int nseg;
        unit_owners(p, P, s, hgi, Wv, G, c_first, nseg);
        const int old = atomic_add_acq_rel_gpu(&p.counters[u], 1);
        const int last = (old == nseg - 1);
        if (last)
            p.counters[u] = 0;
        misc[0] = last;
        misc[1] = (int)c_first;
        misc[3] = nseg;
    }
    consumer_sync<NC>();
    const bool last = misc[0] != 0;
    const int64_t c_first = misc[1];
    const int nseg = misc[3];
    consumer_sync<NC>(); // misc is reused below
    if (!last)
        return;
    const int b0 = __ldg(p.groups + 3 * s), n = __ldg(p.groups + 3 * s + 1);
    const float *base = p.partials + ((size_t)c_first + u) * ((size_t)rows * REC);
#pragma unroll 1
    for (int idx = threadIdx.x; idx < rows * D; idx += NT) {
        const int r = idx / D, d = idx - r * D;
        const int hs = r / GQ, h = r - hs * GQ;
        const int j = h / p.g;
        if (j >= n)
            continue;
        float M = -INFINITY;
        for (int k = 0; k < nseg; ++k)
            M = fmaxf(M, __ldcg(base + (size_t)k * rows * REC + r * REC));
        float O = 0.f, L = 0.f;
        if (M != -INFINITY) {
            for (int k = 0; k < nseg; ++k) {
                const float *rr = base + (size_t)k * rows * REC + r * REC;
                const float m = __ldcg(rr);
                const float sc = (m == -INFINITY) ? 0.f : fast_exp2(m - M);
                L = fmaf(sc, __ldcg(rr + 1), L);
                O = fmaf(sc, __ldcg(rr + 2 + d), O);
            }
        }
        const int kvh = hgi * HG + hs;
        float *pr = p.pre + (((int64_t)(b0 + j) * p.n_kv + kvh) * p.g + (h - j * p.g)) * REC;
        if (d == 0) {
            pr[0] = M;
            pr[1] = L;
        }
        pr[2 + d] = O;
    }
    consumer_sync<NC>(); // the pre rows are written (released by the arrivals below)
    hg_arrive_sequences<D, GQ, NC>(p, P, misc, b0, n, hgi, Wv, G);
}

// ---------------------------------------------------------------------------
// The kernel.
// ---------------------------------------------------------------------------
template <class Pol, int PASS, int NC>
__global__ void __launch_bounds__((NC + 1) * 32, 1)
    decode_hg_kernel(const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const DecodeParams p)
{
    constexpr int D = Pol::D, GQ = Pol::GQ, NQ = Pol::NQ, TILE = Pol::TILE;
    static_assert(Pol::BPI == 1, "one block per item");
    using SM = HgSmem<D, GQ, NC>;
    const SM L(p.stages, p.stage_bytes, p.hg);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bars); // full[S], then empty[S]
    int32_t *meta = reinterpret_cast<int32_t *>(smem + L.meta);
    float *merge = reinterpret_cast<float *>(smem + L.merge);
    float *sink_sc = reinterpret_cast<float *>(smem + L.sink);
    int32_t *misc = reinterpret_cast<int32_t *>(smem + L.misc);
    int32_t *P = reinterpret_cast<int32_t *>(smem + L.prefix);

    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.stages, HG = p.hg, WS = NC / HG;
    // Stage s is read by warp set s % WS alone (S is a multiple of WS), so
    // every consumer waits for each fill of its stages in order and never
    // lags a barrier by a whole phase. The host guarantees the shape.
    if (HG < 1 || NC % HG != 0 || S < 2 || S % WS != 0) {
        if (tid == 0)
            flag_error(p.dev_status, PA_DEV_BAD_CONTEXT_BIT);
        return;
    }
    const int n_h = p.n_kv * (GQ / NQ);

    if (tid == 0) {
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    // eight consumer warps scan (on named barrier 2); the other warps wait
    // at the CTA barrier below
    if (warp < 8)
        prefix_blocks<256, PASS, 1, 2>(p, P, misc + 8);
    __syncthreads();
    if constexpr (PASS == 0) {
        zero_empty_sequences<D, NQ>(p, P, n_h);
    } else {
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
    const int64_t Wv = virt_total(p, P);
    const int64_t G = plan_ctas(p.num_ctas, Wv);
    if ((int64_t)blockIdx.x >= G)
        return;
    const int64_t lo = real_at_virtual(p, P, plan_lo(blockIdx.x, Wv, G));
    const int64_t hi = real_at_virtual(p, P, plan_lo(blockIdx.x + 1, Wv, G));
    const int64_t n_items = hi - lo;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(sbase + L.bars + 8u * s, 1);                       // full: producer
            mbar_init(sbase + L.bars + 8u * (S + s), (uint32_t)HG);      // empty: consumers
        }
    }
    fence_barrier_init();
    __syncthreads();

    const uint32_t tx_full = (uint32_t)(2 * HG * TILE + 2 * HG * 64);
    if (warp == NC) {
        // ------------------------------------------------------ producer
        const uint64_t pol =
            PA_KV_EVICT_FIRST ? l2_policy_evict_first() : l2_policy_evict_normal();
        int32_t phys_cur = -1, phys_next = -1, hg_cur = 0, hg_next = 0;
        // lane l holds item 32 * batch + l: its block-table entry and head group
        auto load_entry = [&](int64_t k, int32_t &phys, int32_t &hgo) {
            phys = -1;
            hgo = 0;
            if (k >= n_items)
                return;
            int b, hgi, i, nb;
            locate_item(lo + k, P, p.num_seqs, p.ups, b, hgi, i, nb);
            int first = i;
            if constexpr (PASS == 0) {
                if (p.window > 0)
                    first += seq_first_block(p, __ldg(p.context_lens + b));
            } else {
                if (b >= p.num_real)
                    first += __ldg(p.skip + (b - p.num_real));
            }
            phys = __ldg(p.block_tables + (size_t)seq_table_row<PASS>(p, b) * p.max_blocks + first);
            hgo = hgi;
        };
        load_entry(lane, phys_cur, hg_cur);
        load_entry(32 + lane, phys_next, hg_next);
        int64_t batch = 0, issued = 0;
        int s = 0;            // stage of item k (k mod S, kept incrementally)
        uint32_t fill = 0;    // parity of item k's fill of stage s: (k / S) & 1
        for (int64_t k = 0; k < n_items; ++k) {
            const int64_t bt = k >> 5;
            if (bt != batch) {
                phys_cur = phys_next;
                hg_cur = hg_next;
                batch = bt;
                load_entry((bt + 1) * 32 + lane, phys_next, hg_next);
            }
            const int32_t phys = __shfl_sync(0xffffffffu, phys_cur, (int)(k & 31));
            const int32_t hgi = __shfl_sync(0xffffffffu, hg_cur, (int)(k & 31));
            const uint32_t full = sbase + L.bars + 8u * s;
            const uint32_t empty = sbase + L.bars + 8u * (S + s);
            if (k >= S) { // the consumers of item k - S released this stage
                if (!__all_sync(0xffffffffu, mbar_wait(empty, fill ^ 1u))) {
                    if (lane == 0)
                        flag_error(p.dev_status, PA_DEV_TIMEOUT_BIT);
                    break;
                }
            }
            if (lane == 0) {
                const bool bad = phys < 0 || (int64_t)phys >= p.num_blocks;
                meta[s] = bad ? 0 : 1;
                if (bad) {
                    flag_error(p.dev_status, PA_DEV_BAD_BLOCK_BIT);
                    mbar_arrive(full); // completes the phase with no data: the item is skipped
                } else {
                    const int64_t row = (int64_t)phys * p.n_kv + (int64_t)hgi * HG;
                    const uint32_t dst = sbase + (uint32_t)(s * p.stage_bytes);
                    fence_proxy_async_smem();
                    mbar_arrive_expect_tx(full, tx_full);
                    tma_load_2d(dst, &tmK, 0, (int32_t)(row * kBlockTokens), full, pol);
                    tma_load_2d(dst + HG * TILE, &tmV, 0, (int32_t)(row * kBlockTokens), full, pol);
                    bulk_load_1d(dst + 2 * HG * TILE, p.k_scale + row * kBlockTokens, HG * 64,
                                 full, pol);
                    bulk_load_1d(dst + 2 * HG * TILE + HG * 64, p.v_scale + row * kBlockTokens,
                                 HG * 64, full, pol);
                }
            }
            __syncwarp();
            issued = k + 1;
            if (++s == S) {
                s = 0;
                fill ^= 1u;
            }
        }
        // Before the CTA's shared memory goes away, every copy issued must
        // have landed: wait (bounded) for the last S stages' fills.
        if (lane == 0) {
            const int64_t from = issued > S ? issued - S : 0;
            for (int64_t k = from; k < issued; ++k) {
                const int64_t f = k / S; // a few iterations at the end
                mbar_wait(sbase + L.bars + 8u * (uint32_t)(k - f * S), (uint32_t)(f & 1));
            }
        }
        return;
    }

    // ------------------------------------------------------------ consumers
    const int hs = warp % HG, ws = warp / HG;
    typename Pol::State st;
    int64_t seg_lo = lo;
    int b, hgi, i0, nb;
    bool dead = false;
    auto rows = [&](int s, int kh) {
        return [&p, s, kh](int v) { return unit_row<GQ, NQ, PASS>(p, s, kh, v); };
    };
    if (seg_lo < hi) {
        locate_item(seg_lo, P, p.num_seqs, p.ups, b, hgi, i0, nb);
        Pol::prefetch_q(st, p, rows(b, hgi * HG + hs));
    }
    int cs = 0;          // stage of the CTA's current item (item index mod S)
    uint32_t cfill = 0;  // parity of that item's fill of its stage
    int cset = 0;        // warp set that serves the current item (item index mod WS)
    while (seg_lo < hi) {
        const int i0_cur = i0;
        const int64_t unit_start = seg_lo - i0;
        const int64_t unit_end = unit_start + nb;
        const int64_t seg_hi = unit_end < hi ? unit_end : hi;
        const bool whole = (i0 == 0) && (unit_end <= hi);
        int32_t ctx, ws_pos, pool_from, fb;
        if constexpr (PASS == 2) {
            ws_pos = pool_from = 0;
            if (b < p.num_real) {
                ctx = __ldg(p.groups + 3 * b + 2) * kBlockTokens;
                fb = 0;
            } else {
                ctx = __ldg(p.context_lens + (b - p.num_real));
                fb = __ldg(p.skip + (b - p.num_real));
            }
        } else {
            ctx = __ldg(p.context_lens + b);
            ws_pos = window_start(p, ctx);
            pool_from = ws_pos > p.n_sink ? ws_pos : p.n_sink;
            fb = seq_first_block(p, ctx);
        }
        Pol::finish_q(st);
        Pol::reset(st);
        for (int64_t x = seg_lo; x < seg_hi; ++x) {
            const int s = cs;
            const uint32_t par = cfill;
            const bool mine = cset == ws;
            if (++cs == S) {
                cs = 0;
                cfill ^= 1u;
            }
            if (++cset == WS)
                cset = 0;
            if (!mine)
                continue; // another warp set serves this stage
            const uint32_t full = sbase + L.bars + 8u * s;
            bool ok = !dead;
            if (ok && !__all_sync(0xffffffffu, mbar_wait(full, par))) {
                ok = false;
                dead = true;
                if (lane == 0)
                    flag_error(p.dev_status, PA_DEV_TIMEOUT_BIT);
            }
            if (ok && meta[s] != 0) {
                const int32_t t0 = (fb + (int32_t)(x - unit_start)) * kBlockTokens;
                const int lo_t = pool_from > t0 ? (int)min(pool_from - t0, kBlockTokens) : 0;
                const int rem = (int)min(ctx - t0, 2 * kBlockTokens);
                const int valid = (int)min(rem, kBlockTokens);
                if (lo_t < valid) {
                    const uint32_t st0 = sbase + (uint32_t)(s * p.stage_bytes);
                    const uint32_t sc0 = st0 + 2 * HG * TILE;
                    Pol::compute4(st, st0 + hs * TILE, st0 + (HG + hs) * TILE, sc0 + hs * 64,
                                  sc0 + (HG + hs) * 64, lo_t, valid, rem, p.scale_log2, 1u);
                }
            }
            __syncwarp();
            if (ok && lane == 0)
                mbar_arrive(sbase + L.bars + 8u * (S + s)); // release the stage
        }
        const int b_cur = b, hg_cur = hgi;
        const int64_t nb_cur = nb;
        if (seg_hi < hi) {
            locate_item(seg_hi, P, p.num_seqs, p.ups, b, hgi, i0, nb);
            Pol::prefetch_q(st, p, rows(b, hgi * HG + hs));
        }
        Pol::to_merge(st, merge);
        consumer_sync<NC>();
        if constexpr (PASS == 2) {
            hg_finish_fused<D, GQ, NC>(p, P, merge, misc, b_cur, hg_cur, Wv, G, whole);
        } else {
            const int32_t s_hi = (i0_cur == 0 && p.n_sink > ws_pos) ? min(p.n_sink, ctx) : 0;
            hg_finish_segment<D, GQ, NQ, NC>(p, P, merge, misc, sink_sc, b_cur, hg_cur,
                                         (int)nb_cur, Wv, G, whole, ws_pos,
                                         s_hi > ws_pos ? s_hi : ws_pos);
        }
        seg_lo = seg_hi;
    }
}

// Launch as a programmatic dependent launch (see launch_decode).
template <class Pol, int PASS, int NC>
cudaError_t launch_decode_hg(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p,
                             int grid, size_t smem, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((NC + 1) * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_hg_kernel<Pol, PASS, NC>, tk, tv, p);
}

} // namespace pa
