// Paged decode-attention kernels for sm_103a.
//
// What is computed (per sequence b, query head h; "LLM 推理底层：KV Cache 显存几何、
// GQA/MLA 压缩与 PagedAttention 调度", eq. for o_t):
//     out[b][h] = softmax(scale * q[b][h] K_b^T) V_b
// over the ctx_b cached tokens of sequence b, read through its block table
// (same page, "逻辑块与物理块映射"), with g = n_h / n_kv query heads sharing a
// KV head (same page, GQA row of the "注意力头架构演进" table).
//
// How the work is split.
//   An "item" is BPI consecutive 16-token blocks of one (sequence, kv head)
//   unit (one block for bf16 tiles, two for INT8/INT4). Items are laid out
//   sequence-major, then kv head, then block, so the W items of the whole
//   batch form one line. The split is by cost: each (sequence, kv head) unit
//   with blocks also counts kSegCost items for the merge that ends each of
//   its segments (see virt_first), and CTA c of G takes the items in
//   [c/G, (c+1)/G) of that weighted line. Every CTA gets about the same work whatever the mix of
//   context lengths, and long contexts are split across CTAs
//   ("split-context" decode). A CTA's range is cut at (sequence, kv head)
//   boundaries into segments.
//   The g query heads of one KV head are processed together, so each K/V tile
//   is read from HBM once for all g heads.
// Inside a CTA.
//   Each warp owns every NW-th item of the range and a private ring of S
//   shared-memory stages. bf16: lane 0 issues TMA tile loads
//   (cp.async.bulk.tensor, 128-byte swizzle) S items ahead; INT8/INT4: every
//   lane issues 16-byte cp.async copies of its share. Completion is tracked
//   by one mbarrier per stage. Block-table entries are fetched 32 items
//   ahead, one item per lane.
//   A warp keeps an online-softmax state (running max m, sum l, accumulator)
//   per query head, in the log2 domain.
// Merging.
//   At a segment end the warps' states are merged through shared memory. A
//   segment that is a whole (sequence, kv head) writes the output directly.
//   Otherwise it writes (m, l, acc) to a workspace slot; the last CTA to finish
//   that (sequence, kv head) -- found with one atomic counter, no waiting --
//   merges all slots with the log-sum-exp rule
//       M = max_p m_p,  out = sum_p 2^(m_p-M) acc_p / sum_p 2^(m_p-M) l_p
//   and resets the counter to zero for the next call. With shared prefixes
//   (PASS 2) a sequence's counter also counts its group's arrival, and the
//   group's prefix state joins the same merge (see finish_fused).
#pragma once

#include "pa_internal.h"
#include "pa_plan.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr int kBlockTokens = 16;

struct DecodeParams {
    const __nv_bfloat16 *q;      // [B][n_h][D]
    const float *k_scale;        // INT8: [NB][n_kv][16]
    const float *v_scale;
    const void *k_cache;         // pools (for LSU-loaded tiles; TMA uses the tensor maps)
    const void *v_cache;
    const int32_t *block_tables; // [B][max_blocks]
    const int32_t *context_lens; // [B]
    __nv_bfloat16 *out;          // [B][n_h][D]
    float *partials;             // [(G + B*n_kv)][g][D + 2]
    int32_t *counters;           // [B*n_kv], zero between calls
    int32_t *dev_status;         // optional
    int64_t num_blocks;
    int32_t num_seqs;
    int32_t n_kv;
    int32_t max_blocks;
    int32_t num_ctas;
    float scale_log2;            // softmax scale * log2(e)
    int32_t window;              // > 0: attend the last `window` tokens only
    int32_t n_sink;              // INT8: positions < n_sink read the bf16 sink rows
    const __nv_bfloat16 *sink_k; // [B][n_kv][n_sink][D]
    const __nv_bfloat16 *sink_v;
    int32_t g;                   // query heads per kv head
    int32_t seg_cost;            // virtual items charged per (sequence, kv head) unit
    int32_t seg_cost_lead;       // ... per unit of the first lead_units "sequences"
    int32_t lead_units;          //     (the group units of the shared-prefix launch)
    // Shared prefixes (PASS 2, see pa_share.cu): the line holds num_real
    // group units first, group s = groups[3s..3s+2] = (position of its first
    // member in members, members, shared blocks), member j being sequence
    // members[groups[3s] + j], whose query rows are the g heads of each
    // member; then the num_real sequences' blocks after their first skip[b].
    // A group's softmax state of each member's head h goes to pre[b][h] =
    // (m, l, acc[D]).
    const int32_t *skip;
    float *pre;
    const int32_t *groups;
    const int32_t *members;
    int32_t num_real;
    int32_t grid_fixed;          // 1: the caller chose num_ctas (no whole-unit grid)
};

// Pass 0: decode of each sequence; pass 2: shared-prefix groups, then each
// sequence's remaining blocks. Block-table row of "sequence" s.
template <int PASS>
__device__ __forceinline__ int32_t seq_table_row(const DecodeParams &p, int s)
{
    if constexpr (PASS == 2)
        return s < p.num_real ? __ldg(p.members + __ldg(p.groups + 3 * s)) : s - p.num_real;
    else
        return s;
}

// Row of query row v of (sequence b, kv head kvh) in q and out, laid out
// [B][NQ][n_h][D]: the GQ = G * NQ query rows of a kv head are its G query
// heads for each of the NQ new tokens (v = i * G + h). NQ = 1 is the plain
// single-token decode, [B][n_h][D].
template <int GQ, int NQ>
__device__ __forceinline__ size_t qo_row(const DecodeParams &p, int b, int kvh, int v)
{
    constexpr int G = GQ / NQ;
    const int i = v / G, h = v - i * G;
    return ((size_t)(b * NQ + i) * p.n_kv + kvh) * G + h;
}

// First position a sequence attends: max(0, ctx - window) under a window.
__device__ __forceinline__ int32_t window_start(const DecodeParams &p, int32_t ctx)
{
    return (p.window > 0 && ctx > p.window) ? ctx - p.window : 0;
}

// First block a sequence reads: the window's first block.
__device__ __forceinline__ int32_t seq_first_block(const DecodeParams &p, int32_t ctx)
{
    return window_start(p, ctx) / kBlockTokens;
}

__device__ __forceinline__ void flag_error(int32_t *dev_status, int32_t bit)
{
    if (dev_status)
        atomicOr(dev_status, bit);
}

// ---------------------------------------------------------------------------
// Shared-memory carve-up common to both kernels.
// ---------------------------------------------------------------------------
template <int D, int GQ, int NW, int S, int STAGE_BYTES, int EXTRA_PER_STAGE, int Q_PER_WARP>
struct SmemLayout {
    static constexpr int kRing = NW * S * STAGE_BYTES;                  // 1024-aligned tiles
    static constexpr int kExtra = NW * S * EXTRA_PER_STAGE;             // per-stage side data
    static constexpr int kQ = NW * Q_PER_WARP;                          // per-warp query copy
    static constexpr int kBars = NW * S * 8;
    static constexpr int kMeta = NW * S * 4;
    static constexpr int kMerge = NW * GQ * (D + 2) * 4;                // per-warp (m, l, acc)
    static constexpr int kSinkSc = GQ * 16 * 4;                         // sink-row scores
    static constexpr int kMisc = 256; // 64 int32 of per-CTA scratch (flags, scan sums)
    static constexpr int kOffExtra = kRing;
    static constexpr int kOffQ = kOffExtra + kExtra;
    static constexpr int kOffBars = (kOffQ + kQ + 15) / 16 * 16;
    static constexpr int kOffMeta = kOffBars + kBars;
    static constexpr int kOffMerge = (kOffMeta + kMeta + 15) / 16 * 16;
    static constexpr int kOffSinkSc = kOffMerge + kMerge;
    static constexpr int kOffMisc = kOffSinkSc + kSinkSc;
    static constexpr int kOffPrefix = kOffMisc + kMisc;
    // P[num_seqs + 1] (int32 items) then Z[num_seqs + 1] (uint16: units with items)
    static size_t bytes(int num_seqs) { return 1024 + kOffPrefix + 6 * (size_t)(num_seqs + 1); }
};

// ---------------------------------------------------------------------------
// Prefix over sequences: P[b] = sum_{b' < b} of the blocks sequence b' reads:
// ceil(ctx / 16), less the blocks wholly before a sliding window's start. A
// context length outside [0, max_blocks*16] counts as 0 blocks (and is
// reported).
// ---------------------------------------------------------------------------
// wsum: 32 int32 of scratch (per-warp sums at [w], nonempty counts at
// [16 + w]; up to 16 warps).
template <int NT, int PASS, int BPI>
__device__ __forceinline__ void prefix_blocks(const DecodeParams &p, int32_t *P, int32_t *wsum)
{
    static_assert(NT <= 16 * 32, "the scan's scratch holds 16 warp sums");
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NWARP = NT / 32;
    int32_t carry = 0, zcarry = 0;
    uint16_t *Z = reinterpret_cast<uint16_t *>(P + p.num_seqs + 1); // sequences before b with blocks
    if (tid == 0) {
        P[0] = 0;
        Z[0] = 0;
    }
    for (int base = 0; base < p.num_seqs; base += NT) {
        const int b = base + tid;
        int32_t v = 0;
        if (b < p.num_seqs) {
            if constexpr (PASS == 2) {
                if (b < p.num_real) {
                    v = __ldg(p.groups + 3 * b + 2); // the group's shared blocks (0: unused)
                } else {
                    const int sb = b - p.num_real;
                    const int32_t ctx = p.context_lens[sb];
                    if (ctx < 0 || (int64_t)ctx > (int64_t)p.max_blocks * kBlockTokens) {
                        if (blockIdx.x == 0)
                            flag_error(p.dev_status, PA_DEV_BAD_CONTEXT_BIT);
                    } else {
                        v = (ctx + kBlockTokens - 1) / kBlockTokens - __ldg(p.skip + sb);
                    }
                }
            } else {
                const int32_t ctx = p.context_lens[b];
                if (ctx < 0 || (int64_t)ctx > (int64_t)p.max_blocks * kBlockTokens) {
                    if (blockIdx.x == 0)
                        flag_error(p.dev_status, PA_DEV_BAD_CONTEXT_BIT);
                } else {
                    // blocks from the first one the sequence reads (window / shared prefix)
                    v = (ctx + kBlockTokens - 1) / kBlockTokens - seq_first_block(p, ctx);
                }
            }
        }
        v = (v + BPI - 1) / BPI; // items of BPI blocks
        int32_t x = v, z = v > 0 ? 1 : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            const int32_t yz = __shfl_up_sync(0xffffffffu, z, o);
            if (lane >= o) {
                x += y;
                z += yz;
            }
        }
        if (lane == 31) {
            wsum[warp] = x;
            wsum[16 + warp] = z;
        }
        __syncthreads();
        if (warp == 0) {
            int32_t t = lane < NWARP ? wsum[lane] : 0;
            int32_t tz = lane < NWARP ? wsum[16 + lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, t, o);
                const int32_t yz = __shfl_up_sync(0xffffffffu, tz, o);
                if (lane >= o) {
                    t += y;
                    tz += yz;
                }
            }
            if (lane < NWARP) {
                wsum[lane] = t; // inclusive
                wsum[16 + lane] = tz;
            }
        }
        __syncthreads();
        const int32_t before = warp ? wsum[warp - 1] : 0;
        const int32_t zbefore = warp ? wsum[16 + warp - 1] : 0;
        if (b < p.num_seqs) {
            P[b + 1] = carry + before + x;
            Z[b + 1] = (uint16_t)(zcarry + zbefore + z);
        }
        carry += wsum[NWARP - 1];
        zcarry += wsum[16 + NWARP - 1];
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Cost-weighted split. Besides its blocks, every (sequence, kv head) unit
// costs a fixed merge at the end of each segment that covers it. The split
// runs on a "virtual" line where unit (b, kvh) is kSegCost + nb_b long: the
// first kSegCost positions stand for the merge, the rest for its blocks in
// order. CTA c of G owns virtual [plan_lo(c, Wv, G), plan_lo(c+1, Wv, G)),
// i.e. the contiguous real items whose virtual positions fall there, so a CTA
// covering many short units gets fewer blocks. Every sequence with blocks
// carries n_kv * kSegCost, so the virtual prefix is P[b] + kSegCost * Z[b].
// ---------------------------------------------------------------------------
#ifndef PA_SEG_COST
#define PA_SEG_COST 8
#endif
constexpr int kSegCost = PA_SEG_COST;

// a / b for 0 <= a, 0 < b: in 32-bit arithmetic when a fits (the usual
// case; a 64-bit division is several times longer on the device).
__device__ __forceinline__ int64_t div_small(int64_t a, int64_t b)
{
    if (a <= (int64_t)0xFFFFFFFF && b <= (int64_t)0xFFFFFFFF)
        return (int64_t)((uint32_t)a / (uint32_t)b);
    return a / b;
}

// Virtual position of the first block of unit (b, kvh) (nb = blocks of b).
// Z = P + num_seqs + 1 counts the sequences with blocks: an empty sequence
// has no segment and costs nothing. A unit of one of the first lead_units
// sequences is charged seg_cost_lead, any other seg_cost.
__device__ __forceinline__ int64_t unit_cost(const DecodeParams &p, int b)
{
    return b < p.lead_units ? p.seg_cost_lead : p.seg_cost;
}

__device__ __forceinline__ int64_t virt_start(const DecodeParams &p, const int32_t *P, int b)
{
    const uint16_t *Z = reinterpret_cast<const uint16_t *>(P + p.num_seqs + 1);
    const int64_t zl = Z[b < p.lead_units ? b : p.lead_units];
    return (int64_t)p.n_kv * (P[b] + (int64_t)p.seg_cost * Z[b] +
                              ((int64_t)p.seg_cost_lead - p.seg_cost) * zl);
}

__device__ __forceinline__ int64_t virt_first(const DecodeParams &p, const int32_t *P, int b,
                                              int kvh, int nb)
{
    const int64_t c = unit_cost(p, b);
    return virt_start(p, P, b) + (int64_t)kvh * (nb + c) + c;
}

// Total virtual length.
__device__ __forceinline__ int64_t virt_total(const DecodeParams &p, const int32_t *P)
{
    return virt_start(p, P, p.num_seqs);
}

// First real item whose virtual position is >= y (W for y >= the total).
__device__ __forceinline__ int64_t real_at_virtual(const DecodeParams &p, const int32_t *P,
                                                   int64_t y)
{
    if (y >= virt_total(p, P))
        return (int64_t)p.n_kv * P[p.num_seqs];
    int lo = 0, hi = p.num_seqs;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (virt_start(p, P, mid) <= y)
            lo = mid;
        else
            hi = mid;
    }
    // b has blocks: an empty b has a zero virtual length, so it would not be
    // the largest b with a start <= y
    const int b = lo;
    const int64_t C = unit_cost(p, b);
    const int64_t nb = P[b + 1] - P[b], v = nb + C;
    const int64_t r = y - virt_start(p, P, b);
    const int64_t kvh = div_small(r, v), off = r - kvh * v;
    const int64_t base = (int64_t)p.n_kv * P[b] + kvh * nb;
    return off < C ? base : base + (off - C);
}

// Whole-unit grid. When no more (sequence, kv head) units with blocks than
// CTAs are launched, at least 3/4 as many, and the units are equally long
// within 3%, CTA c takes unit c whole (the rest stay idle): no unit is cut,
// so there are no partial records or merges, and the fewer CTAs still pull
// the HBM stream as fast (measured on the Llama-3-70B layer: 128 units on
// 152 SMs, 87.8 us whole-unit against 91.7 us split). Returns the number of
// units, or 0 to keep the cost-weighted split. Same result in every CTA;
// ends with a CTA barrier.
template <int NT>
__device__ __forceinline__ int64_t whole_unit_grid(const DecodeParams &p, const int32_t *P,
                                                   int64_t G, int32_t *scratch)
{
    if (p.grid_fixed)
        return 0;
    const uint16_t *Z = reinterpret_cast<const uint16_t *>(P + p.num_seqs + 1);
    const int64_t seqs = Z[p.num_seqs], U = (int64_t)p.n_kv * seqs;
    if (U == 0 || U > G || 4 * U < 3 * G)
        return 0;
    int32_t mx = 0;
    for (int b = threadIdx.x; b < p.num_seqs; b += NT)
        mx = max(mx, P[b + 1] - P[b]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if ((threadIdx.x & 31) == 0)
        scratch[threadIdx.x >> 5] = mx;
    __syncthreads();
    mx = 0;
    for (int w = 0; w < NT / 32; ++w)
        mx = max(mx, scratch[w]);
    __syncthreads(); // scratch is reused
    return 100 * (int64_t)mx * seqs <= 103 * (int64_t)P[p.num_seqs] ? U : 0;
}

// Items [lo, hi) of the c-th unit with blocks (sequence-major over the
// sequences with blocks, then kv head).
__device__ __forceinline__ void unit_items(const DecodeParams &p, const int32_t *P, int64_t c,
                                           int64_t &lo, int64_t &hi)
{
    const uint16_t *Z = reinterpret_cast<const uint16_t *>(P + p.num_seqs + 1);
    const int j = (int)(c / p.n_kv), kvh = (int)(c - (int64_t)j * p.n_kv);
    // the sequence b with blocks and Z[b] == j (Z counts the ones before b)
    int l = 0, h = p.num_seqs; // Z[l] <= j < Z[h]
    while (h - l > 1) {
        const int m = (l + h) >> 1;
        if (Z[m] <= j)
            l = m;
        else
            h = m;
    }
    const int64_t nb = P[l + 1] - P[l];
    lo = (int64_t)p.n_kv * P[l] + kvh * nb;
    hi = lo + nb;
}

// Item x -> (sequence b, kv head, block index i within the sequence, blocks
// of the sequence). Largest b with n_kv*P[b] <= x; such a b has blocks.
__device__ __forceinline__ void locate_item(int64_t x, const int32_t *P, int num_seqs, int n_kv,
                                            int &b, int &kvh, int &i, int &nb)
{
    int lo = 0, hi = num_seqs;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)n_kv * P[mid] <= x)
            lo = mid;
        else
            hi = mid;
    }
    b = lo;
    nb = P[b + 1] - P[b];
    const int64_t r = x - (int64_t)n_kv * P[b];
    kvh = (int)div_small(r, nb);
    i = (int)(r - (int64_t)kvh * nb);
}

// Zero the output rows of sequences with no blocks (ctx == 0 or invalid);
// each sequence has NQ * n_h rows.
template <int D, int NQ>
__device__ __forceinline__ void zero_empty_sequences(const DecodeParams &p, const int32_t *P,
                                                     int n_h)
{
    const int rows16 = NQ * n_h * D * 2 / 16; // 16-byte chunks per sequence
    for (int b = blockIdx.x; b < p.num_seqs; b += p.num_ctas) {
        if (P[b + 1] != P[b])
            continue;
        uint4 *dst = reinterpret_cast<uint4 *>(p.out + (size_t)b * NQ * n_h * D);
        for (int i = threadIdx.x; i < rows16; i += blockDim.x)
            dst[i] = make_uint4(0, 0, 0, 0);
    }
}

__device__ __forceinline__ int ld_acquire_gpu(const int32_t *addr)
{
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu(int32_t *addr, int v)
{
    asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

// atom.add with acquire-release semantics at GPU scope: releases this CTA's
// partial record (ordered before it by a CTA barrier) and acquires the
// records of the CTAs that arrived earlier.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int32_t *addr, int v)
{
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(addr), "r"(v)
                 : "memory");
    return old;
}

// ---------------------------------------------------------------------------
// End of a segment: merge the NW warp states (`merge`, [NW][GQ][D+2]: m, l,
// acc[D], each warp against its own running base) and write the output, or
// a partial record when the (sequence, kv head) is split over CTAs; the last
// CTA to publish a record for it merges all records. Called by all threads.
//   M = max_w m_w,  O = sum_w 2^(m_w-M) acc_w,  L = sum_w 2^(m_w-M) l_w
// ---------------------------------------------------------------------------
// Scores (log2 domain) of the bf16 sink rows [s_lo, s_hi) of (b, kvh) for
// the GQ heads: sc[h * 16 + j - s_lo]. One warp per (head, row) pair, lanes
// over d. Called by all threads; ends with a CTA barrier.
template <int D, int GQ, int NW, int NQ>
__device__ __forceinline__ void sink_scores(const DecodeParams &p, int b, int kvh, int s_lo,
                                            int s_hi, float *sc)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ns = s_hi - s_lo;
    const __nv_bfloat16 *k = p.sink_k + ((size_t)b * p.n_kv + kvh) * p.n_sink * D;
    for (int t = warp; t < GQ * ns; t += NW) {
        const int h = t / ns, j = s_lo + t % ns;
        const __nv_bfloat16 *q = p.q + qo_row<GQ, NQ>(p, b, kvh, h) * D;
        float a = 0.f;
#pragma unroll
        for (int d = lane; d < D; d += 32)
            a = fmaf(__bfloat162float(q[d]), __bfloat162float(k[j * D + d]), a);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0)
            sc[h * 16 + (j - s_lo)] = a * p.scale_log2;
    }
    __syncthreads();
}

// Row of query row v of unit (s, kvh) in q, out and pre, or -1 for a padding
// row. Pass 0: qo_row. Pass 2: for a group unit s, member j = v / g of the
// group, query head kvh * g + v % g of that sequence; for a sequence's
// remaining blocks, its g query heads.
template <int GQ, int NQ, int PASS>
__device__ __forceinline__ int64_t unit_row(const DecodeParams &p, int s, int kvh, int v)
{
    if constexpr (PASS == 2) {
        if (s >= p.num_real) { // a sequence's remaining blocks: its g query heads
            if (v >= p.g)
                return -1;
            return ((int64_t)(s - p.num_real) * p.n_kv + kvh) * p.g + v;
        }
    }
    if constexpr (PASS == 2) {
        const int j = v / p.g, h = v - j * p.g;
        if (j >= __ldg(p.groups + 3 * s + 1))
            return -1;
        const int b = __ldg(p.members + __ldg(p.groups + 3 * s) + j);
        return ((int64_t)b * p.n_kv + kvh) * p.g + h;
    } else {
        return (int64_t)qo_row<GQ, NQ>(p, s, kvh, v);
    }
}

// Final output of d and d + 1 (d even) of query row h: one bf16x2 store.
template <int D, int GQ, int NQ>
__device__ __forceinline__ void emit2(const DecodeParams &p, int b, int kvh, int h, int d, float L,
                                      float O0, float O1)
{
    const size_t row = qo_row<GQ, NQ>(p, b, kvh, h);
    *reinterpret_cast<__nv_bfloat162 *>(p.out + row * D + d) =
        __floats2bfloat162_rn(L > 0.f ? O0 / L : 0.f, L > 0.f ? O1 / L : 0.f);
}

// Log-sum-exp state of a run of RUN adjacent d of one row, merged from
// partial states (m, l, o[d]) with a running maximum:
//   M = max m,  L = sum 2^(m - M) l,  O[e] = sum 2^(m - M) o[d0 + e].
template <int RUN>
struct RunState {
    float M, L, O[RUN];
    __device__ __forceinline__ void clear()
    {
        M = -INFINITY;
        L = 0.f;
#pragma unroll
        for (int e = 0; e < RUN; ++e)
            O[e] = 0.f;
    }
};

// Fold the states of nrec rows (row r at base + r * stride, laid out m, l,
// o[D]) for d in [d0, d0 + RUN) into st, RB rows per round of loads.
template <int RUN, int RB>
__device__ __forceinline__ void fold_rows(RunState<RUN> &st, const float *base, size_t stride,
                                          int nrec, int d0)
{
#pragma unroll 1
    for (int s0 = 0; s0 < nrec; s0 += RB) {
        float mr[RB], lr[RB];
        float2 orr[RB][RUN / 2];
#pragma unroll
        for (int j = 0; j < RB; ++j) {
            const bool in = s0 + j < nrec;
            const float *r = base + (size_t)(in ? s0 + j : s0) * stride;
            mr[j] = in ? __ldcg(r) : -INFINITY;
            lr[j] = in ? __ldcg(r + 1) : 0.f;
#pragma unroll
            for (int e = 0; e < RUN / 2; ++e)
                orr[j][e] = in ? __ldcg(reinterpret_cast<const float2 *>(r + 2 + d0) + e)
                               : make_float2(0.f, 0.f);
        }
        float mx = st.M;
#pragma unroll
        for (int j = 0; j < RB; ++j)
            mx = fmaxf(mx, mr[j]);
        if (mx == -INFINITY)
            continue;
        const float a = (st.M == -INFINITY) ? 0.f : fast_exp2(st.M - mx);
        st.L *= a;
#pragma unroll
        for (int e = 0; e < RUN; ++e)
            st.O[e] *= a;
#pragma unroll
        for (int j = 0; j < RB; ++j) {
            const float sc = (mr[j] == -INFINITY) ? 0.f : fast_exp2(mr[j] - mx);
            st.L = fmaf(sc, lr[j], st.L);
#pragma unroll
            for (int e = 0; e < RUN / 2; ++e) {
                st.O[2 * e] = fmaf(sc, orr[j][e].x, st.O[2 * e]);
                st.O[2 * e + 1] = fmaf(sc, orr[j][e].y, st.O[2 * e + 1]);
            }
        }
        st.M = mx;
    }
}

// Run length of the merges: each thread takes RUN adjacent d of one row
// (GQ, D and the CTA's NT threads are powers of two), four rows per round
// of loads (two for the longest runs).
template <int D, int GQ, int NT>
struct MergeRun {
    static constexpr int RUN = GQ * D / NT > 2 ? GQ * D / NT : 2;
    static constexpr int RB = RUN >= 16 ? 2 : 4;
    static_assert(GQ * D / RUN <= NT && D % RUN == 0, "one run per thread");
};

template <int D, int GQ, int NW, int NQ>
__device__ __forceinline__ void finish_segment(const DecodeParams &p, const int32_t *P,
                                               const float *merge, int32_t *misc, float *sink_sc,
                                               int b, int kvh, int nb, int64_t Wv, int64_t G,
                                               bool whole, int s_lo, int s_hi)
{
    constexpr int NT = NW * 32;
    constexpr int REC = D + 2;
    // A thread combines a run of RUN adjacent d of one head, so the head's
    // weights are worked out once per thread.
    constexpr int RUN = MergeRun<D, GQ, NT>::RUN;
    constexpr int RUNS = GQ * D / RUN;
    const int u = b * p.n_kv + kvh;
    float *rec = p.partials + ((size_t)blockIdx.x + u) * (GQ * REC);
    // Sink rows [s_lo, s_hi) join this segment's merge as one more partial
    // state (the segment that holds the sequence's first block has them).
    const int ns = s_hi - s_lo;
    if (ns > 0)
        sink_scores<D, GQ, NW, NQ>(p, b, kvh, s_lo, s_hi, sink_sc);
    const __nv_bfloat16 *sv = p.sink_v + ((size_t)b * p.n_kv + kvh) * p.n_sink * D;

    const bool act = threadIdx.x < RUNS;
    const int h = act ? (int)threadIdx.x * RUN / D : 0;
    const int d0 = act ? (int)threadIdx.x * RUN - h * D : 0;
    if (act) {
        float mw[NW];
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            mw[w] = merge[(w * GQ + h) * REC];
            M = fmaxf(M, mw[w]);
        }
        for (int j = 0; j < ns; ++j)
            M = fmaxf(M, sink_sc[h * 16 + j]);
        float O[RUN], L = 0.f;
#pragma unroll
        for (int e = 0; e < RUN; ++e)
            O[e] = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float *mrow = merge + (w * GQ + h) * REC;
                const float sc = (mw[w] == -INFINITY) ? 0.f : fast_exp2(mw[w] - M);
                L = fmaf(sc, mrow[1], L);
#pragma unroll
                for (int e = 0; e < RUN; e += 2) {
                    const float2 a = *reinterpret_cast<const float2 *>(mrow + 2 + d0 + e);
                    O[e] = fmaf(sc, a.x, O[e]);
                    O[e + 1] = fmaf(sc, a.y, O[e + 1]);
                }
            }
            for (int j = 0; j < ns; ++j) {
                const float ej = fast_exp2(sink_sc[h * 16 + j] - M);
                L += ej;
#pragma unroll
                for (int e = 0; e < RUN; ++e)
                    O[e] = fmaf(ej, __bfloat162float(sv[(s_lo + j) * D + d0 + e]), O[e]);
            }
        }
        if (whole) {
#pragma unroll
            for (int e = 0; e < RUN; e += 2)
                emit2<D, GQ, NQ>(p, b, kvh, h, d0 + e, L, O[e], O[e + 1]);
        } else {
            if (d0 == 0) {
                rec[h * REC] = M;
                rec[h * REC + 1] = L;
            }
#pragma unroll
            for (int e = 0; e < RUN; e += 2)
                *reinterpret_cast<float2 *>(rec + h * REC + 2 + d0 + e) = make_float2(O[e], O[e + 1]);
        }
    }
    __syncthreads(); // also: every record store of this CTA is done (CTA scope)
    if (whole)
        return;
    // the CTAs that own the unit's blocks: owners of its first and last block
    const int64_t v0 = virt_first(p, P, b, kvh, nb);
    const int64_t c_first = plan_owner(v0, Wv, G);
    const int nseg = (int)(plan_owner(v0 + nb - 1, Wv, G) - c_first + 1);
    if (threadIdx.x == 0) {
        const int old = atomic_add_acq_rel_gpu(&p.counters[u], 1);
        const int last = (old == nseg - 1);
        if (last)
            p.counters[u] = 0; // every arrival of this launch is in: reset for the next call
        misc[0] = last;
    }
    __syncthreads();
    if (!misc[0] || !act)
        return;
    // Last arrival: merge the nseg records (each thread's run of d).
    RunState<RUN> st;
    st.clear();
    fold_rows<RUN, MergeRun<D, GQ, NT>::RB>(
        st, p.partials + ((size_t)c_first + u) * (GQ * REC) + h * REC, (size_t)GQ * REC, nseg, d0);
#pragma unroll
    for (int e = 0; e < RUN; e += 2)
        emit2<D, GQ, NQ>(p, b, kvh, h, d0 + e, st.L, st.O[e], st.O[e + 1]);
}

// ---------------------------------------------------------------------------
// Fused shared-prefix pass (PASS 2). Units s < B are groups (their rows are
// the query heads of every member); units s >= B are sequence b = s - B's
// blocks after its group's prefix. Sequence b's output combines its own
// records and, for a group member, the group's state in pre. Counting both
// kinds of arrival on b's counter (nseg + 1 for a member), whichever comes
// last merges: no CTA ever waits for another.
// ---------------------------------------------------------------------------

// CTAs owning the blocks of unit (s, kvh): first and count.
__device__ __forceinline__ void unit_owners(const DecodeParams &p, const int32_t *P, int s,
                                            int kvh, int64_t Wv, int64_t G, int64_t &c_first,
                                            int &nseg)
{
    const int nb = P[s + 1] - P[s];
    const int64_t v0 = virt_first(p, P, s, kvh, nb);
    c_first = plan_owner(v0, Wv, G);
    nseg = (int)(plan_owner(v0 + nb - 1, Wv, G) - c_first + 1);
}

// Output run [d0, d0 + RUN) of head h of sequence b, kv head kvh: its
// records, written by CTAs c_first .. c_first + nseg - 1, and its group's
// prefix state (a pre row has a record's layout).
template <int D, int GQ, int RUN, int RB>
__device__ __forceinline__ void merge_run(const DecodeParams &p, int b, int kvh, int64_t c_first,
                                          int nseg, int h, int d0)
{
    constexpr int REC = D + 2;
    const int u = (p.num_real + b) * p.n_kv + kvh;
    const int64_t row = ((int64_t)b * p.n_kv + kvh) * p.g + h;
    RunState<RUN> st;
    st.clear();
    if (__ldg(p.skip + b) > 0)
        fold_rows<RUN, 1>(st, p.pre + row * REC, 0, 1, d0);
    fold_rows<RUN, RB>(st, p.partials + ((size_t)c_first + u) * (GQ * REC) + h * REC,
                       (size_t)GQ * REC, nseg, d0);
#pragma unroll
    for (int e = 0; e < RUN; e += 2)
        *reinterpret_cast<__nv_bfloat162 *>(p.out + row * D + d0 + e) = __floats2bfloat162_rn(
            st.L > 0.f ? st.O[e] / st.L : 0.f, st.L > 0.f ? st.O[e + 1] / st.L : 0.f);
}

// One arrival on sequence b's counter, which expects nseg arrivals (+1 for
// a group member). Returns whether this was the last; then the caller merges
// and the counter is reset for the next launch.
__device__ __forceinline__ bool arrive_one(const DecodeParams &p, const int32_t *P, int b,
                                           int kvh, int64_t Wv, int64_t G, int64_t &c_first,
                                           int &nseg)
{
    const int s = p.num_real + b, u = s * p.n_kv + kvh;
    unit_owners(p, P, s, kvh, Wv, G, c_first, nseg);
    const int expect = nseg + (__ldg(p.skip + b) > 0 ? 1 : 0);
    const int old = atomic_add_acq_rel_gpu(&p.counters[u], 1);
    const bool last = (old == expect - 1);
    if (last)
        p.counters[u] = 0;
    return last;
}

// Arrivals of sequences map[b0 .. b0 + n - 1] (n <= 8; map NULL: b0 .. b0 +
// n - 1), one thread each, then the merges of those that arrived last, all
// threads together. Called by all threads; the records and pre rows this
// CTA wrote are published by the barrier before the release of each arrival.
template <int D, int GQ, int NW>
__device__ __forceinline__ void arrive_sequences(const DecodeParams &p, const int32_t *P,
                                                 int32_t *misc, const int32_t *map, int b0, int n,
                                                 int kvh, int64_t Wv, int64_t G)
{
    constexpr int NT = NW * 32;
    int32_t *last = misc, *cf = misc + 8, *ns = misc + 16, *seq = misc + 24;
    if (threadIdx.x < n) {
        int64_t c_first;
        int nseg;
        const int b = map ? __ldg(map + b0 + threadIdx.x) : b0 + (int)threadIdx.x;
        const bool l = arrive_one(p, P, b, kvh, Wv, G, c_first, nseg);
        last[threadIdx.x] = l;
        cf[threadIdx.x] = (int32_t)c_first;
        ns[threadIdx.x] = nseg;
        seq[threadIdx.x] = b;
    }
    __syncthreads();
    using MR = MergeRun<D, GQ, NT>;
    const int per = p.g * D / MR::RUN; // runs per sequence
#pragma unroll 1
    for (int idx = threadIdx.x; idx < n * per; idx += NT) {
        const int j = idx / per, k = (idx - j * per) * MR::RUN;
        if (last[j])
            merge_run<D, GQ, MR::RUN, MR::RB>(p, seq[j], kvh, cf[j], ns[j], k / D, k % D);
    }
    // (misc is next written after the two CTA barriers that open the next
    // segment's merge, so no barrier is needed here)
}

template <int D, int GQ, int NW>
__device__ __forceinline__ void finish_fused(const DecodeParams &p, const int32_t *P,
                                             const float *merge, int32_t *misc, int s, int kvh,
                                             int64_t Wv, int64_t G, bool whole)
{
    constexpr int NT = NW * 32, REC = D + 2;
    const bool group = s < p.num_real;
    const int b = s - p.num_real;
    const bool member = !group && __ldg(p.skip + b) > 0;
    const int u = s * p.n_kv + kvh;
    float *rec = p.partials + ((size_t)blockIdx.x + u) * (GQ * REC);
    const bool direct = whole && !group && !member; // a plain sequence in one piece
    // live rows: a group's members' heads, else the sequence's g heads
    const int rows = group ? __ldg(p.groups + 3 * s + 1) * p.g : p.g;
    // warps' states -> this CTA's state of the unit: output or record, a run
    // of RUN adjacent d of one row per thread
    using MR = MergeRun<D, GQ, NT>;
    constexpr int RUN = MR::RUN;
#pragma unroll 1
    for (int idx = threadIdx.x; idx < rows * (D / RUN); idx += NT) {
        const int h = idx * RUN / D, d0 = idx * RUN - h * D;
        float mw[NW];
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            mw[w] = merge[(w * GQ + h) * REC];
            M = fmaxf(M, mw[w]);
        }
        float O[RUN], L = 0.f;
#pragma unroll
        for (int e = 0; e < RUN; ++e)
            O[e] = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float *mrow = merge + (w * GQ + h) * REC;
                const float sc = (mw[w] == -INFINITY) ? 0.f : fast_exp2(mw[w] - M);
                L = fmaf(sc, mrow[1], L);
#pragma unroll
                for (int e = 0; e < RUN; e += 2) {
                    const float2 a = *reinterpret_cast<const float2 *>(mrow + 2 + d0 + e);
                    O[e] = fmaf(sc, a.x, O[e]);
                    O[e + 1] = fmaf(sc, a.y, O[e + 1]);
                }
            }
        }
        if (direct) {
            __nv_bfloat16 *o = p.out + (((int64_t)b * p.n_kv + kvh) * p.g + h) * D + d0;
#pragma unroll
            for (int e = 0; e < RUN; e += 2)
                *reinterpret_cast<__nv_bfloat162 *>(o + e) = __floats2bfloat162_rn(
                    L > 0.f ? O[e] / L : 0.f, L > 0.f ? O[e + 1] / L : 0.f);
        } else {
            if (d0 == 0) {
                rec[h * REC] = M;
                rec[h * REC + 1] = L;
            }
#pragma unroll
            for (int e = 0; e < RUN; e += 2)
                *reinterpret_cast<float2 *>(rec + h * REC + 2 + d0 + e) = make_float2(O[e], O[e + 1]);
        }
    }
    __syncthreads();
    if (direct)
        return;
    if (!group) { // a piece of sequence b: one arrival
        arrive_sequences<D, GQ, NW>(p, P, misc, nullptr, b, 1, kvh, Wv, G);
        return;
    }
    // a piece of group s: the last one merges the group's state into pre and
    // then arrives once on every member's counter
    if (threadIdx.x == 0) {
        int64_t c_first;
        int nseg;
        unit_owners(p, P, s, kvh, Wv, G, c_first, nseg);
        const int old = atomic_add_acq_rel_gpu(&p.counters[u], 1);
        const int last = (old == nseg - 1);
        if (last)
            p.counters[u] = 0;
        misc[0] = last;
        misc[1] = (int)c_first;
        misc[3] = nseg;
    }
    __syncthreads();
    if (!misc[0])
        return; // (misc is next written after the next segment's barriers)
    const int64_t c_first = misc[1];
    const int nseg = misc[3];
    const int b0 = __ldg(p.groups + 3 * s), n = __ldg(p.groups + 3 * s + 1);
    const float *base = p.partials + ((size_t)c_first + u) * (GQ * REC);
#pragma unroll 1
    for (int idx = threadIdx.x; idx < n * p.g * (D / RUN); idx += NT) {
        const int h = idx * RUN / D, d0 = idx * RUN - h * D;
        const int j = h / p.g;
        RunState<RUN> st;
        st.clear();
        fold_rows<RUN, MR::RB>(st, base + h * REC, (size_t)GQ * REC, nseg, d0);
        const int bj = __ldg(p.members + b0 + j);
        float *pr = p.pre + (((int64_t)bj * p.n_kv + kvh) * p.g + (h - j * p.g)) * REC;
        if (d0 == 0) {
            pr[0] = st.M;
            pr[1] = st.L;
        }
#pragma unroll
        for (int e = 0; e < RUN; e += 2)
            *reinterpret_cast<float2 *>(pr + 2 + d0 + e) = make_float2(st.O[e], st.O[e + 1]);
    }
    __syncthreads(); // the pre rows are written (released by the arrivals below)
    arrive_sequences<D, GQ, NW>(p, P, misc, p.members, b0, n, kvh, Wv, G);
}

// Byte offset of 16-byte chunk `c` of row `r` in a TMA-swizzled tile whose
// rows are ROWB bytes (128: SWIZZLE_128B, 64: SWIZZLE_64B).
template <int ROWB>
__device__ __forceinline__ uint32_t swz(int r, int c)
{
    if constexpr (ROWB == 128)
        return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
    else
        return (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

// ---------------------------------------------------------------------------
// Per-warp producer: the TMA ring and the block-table prefetch.
// ---------------------------------------------------------------------------
// An item is BPI consecutive blocks of one (sequence, kv head) unit; the
// last item of a unit may hold fewer.
template <int BPI>
struct WarpRing {
    int64_t lo;             // CTA range start
    int64_t n_items;        // items this warp owns
    int warp;
    int64_t issued;         // items whose loads were issued
    int64_t batch;          // index of the 32-item batch held in the *_cur registers
    int32_t phys_cur[BPI];  // lane l: physical blocks of item 32*batch + l (raw table entries)
    int32_t kvh_cur;        //         its kv head | (mask of absent blocks) << 16
    int32_t phys_next[BPI]; // the same for batch + 1
    int32_t kvh_next;
};

// Block-table entries and kv head of this warp's item k. The loaded values
// are not used here, so the loads' latency overlaps other work; the entries
// are checked when the item is issued.
template <int NW, int PASS, int BPI>
__device__ __forceinline__ void load_item(const DecodeParams &p, const int32_t *P,
                                          const WarpRing<BPI> &r, int64_t k,
                                          int32_t (&phys)[BPI], int32_t &kvh)
{
    if (k >= r.n_items) {
#pragma unroll
        for (int j = 0; j < BPI; ++j)
            phys[j] = -1;
        kvh = 0;
        return;
    }
    const int64_t x = r.lo + r.warp + k * NW;
    int b, i, nb;
    locate_item(x, P, p.num_seqs, p.n_kv, b, kvh, i, nb);
    // first block of the item, and (BPI > 1) the blocks the unit reads
    int first = i * BPI, nblk = 0;
    if constexpr (PASS == 0) {
        if (p.window > 0 || BPI > 1) {
            const int32_t ctx = __ldg(p.context_lens + b);
            const int32_t fb = p.window > 0 ? seq_first_block(p, ctx) : 0;
            first += fb;
            nblk = (ctx + kBlockTokens - 1) / kBlockTokens;
        }
    } else if constexpr (PASS == 2) {
        if (b >= p.num_real) {
            first += __ldg(p.skip + (b - p.num_real));
            if constexpr (BPI > 1)
                nblk = (__ldg(p.context_lens + (b - p.num_real)) + kBlockTokens - 1) / kBlockTokens;
        } else if constexpr (BPI > 1) {
            nblk = __ldg(p.groups + 3 * b + 2);
        }
    }
    const int32_t *row = p.block_tables + (size_t)seq_table_row<PASS>(p, b) * p.max_blocks;
#pragma unroll
    for (int j = 0; j < BPI; ++j) {
        const bool present = j == 0 || first + j < nblk;
        phys[j] = present ? __ldg(row + first + j) : -1;
        if (!present)
            kvh |= 1 << (16 + j);
    }
}

} // namespace pa
