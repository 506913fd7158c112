// Quantised K/V policy for the decode kernel (INT8 or INT4 codes): tensor-core
// contractions on exact fp16 copies of the codes.
//
// The cache holds integer codes and one fp32 scale per (token, kv head)
// ("kv-cache-guide" (guijiagi.com) §4.2: x = code * scale; 8-bit codes in
// [-128, 127], 4-bit codes in [-8, 7] packed two per byte, low nibble first).
// Every code is exact in fp16. A code c becomes fp16 by writing its
// offset-binary form (c + 128, or c + 8) into the mantissa of 1024
// (exponent bits 0x64): that half is B + c with B = 1152 (INT8) or 1032
// (INT4); one fp16x2 subtraction of B (a fused multiply-add for the INT4
// codes that land as 1152 + 16 c) then leaves exactly c. The contractions
// thus see the codes themselves: no bias term is carried through the fp32
// accumulators, whose rounding stays relative to the result. Both
// contractions run as mma.sync m16n8k16 with fp16 inputs and fp32
// accumulation (every product of two fp16 values is exact):
//   S^T[16 tok][8 heads] = Kcode[16 tok][D] . Q'^T[D][8 heads]
//       (tokens on M; the k index is permuted so each thread's A fragments
//        for all k-steps come from one 16-byte (or 8-byte) load of a row)
//   s = S^T * 2^e * k_scale[tok] * scale * log2(e)
//   O^T[D][8 heads] += Vcode^T[D][16 tok] . W^T[16 tok][8 heads]
//       (d on M, so the query group only pads N to 8; the rows of O^T are
//        permuted so each thread's A fragments for all D/16 row tiles come
//        from one load of each of its four token rows)
// INT4 codes take one AND-XOR each (no shifts into place): the nibble at
// bits 0-3 of a 16-bit half becomes 1024 + (c + 8) = 1032 + c, the nibble at
// bits 4-7 becomes 1024 + 16 (c + 8) = 1152 + 16 c; the first loses 1032,
// the second is scaled by 1/16 and loses 72, in one fp16x2 operation each.
// Q' = q * 2^-e with e >= 0 chosen per (sequence, kv head) so that
// max|Q'| < 2^15: the bf16 -> fp16 conversion is then exact for every
// normal value. W = p * v_scale[tok] / s_base, where s_base is a running
// V-scale base that only moves (rescaling O) when a block's largest V scale
// exceeds it 64-fold, so W <= 2^8 * 2^6 stays far below fp16's maximum.
#pragma once

#include <cuda_fp16.h>

#include "pa_decode.cuh"

namespace pa {

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ float lds_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}

// INT4 codes (two's complement nibbles) -> fp16x2. nib_lo: the nibbles at
// bits 0-3 and 16-19 of w as {1032 + c0, 1032 + c1}; nib_hi: those at bits
// 4-7 and 20-23 as {1152 + 16 c0, 1152 + 16 c1}. XOR with 8 (in place) turns
// a code into its offset form c + 8, which lies inside the mantissa of 1024.
__device__ __forceinline__ uint32_t nib_lo(uint32_t w)
{
    return (w & 0x000F000Fu) ^ 0x64086408u;
}

__device__ __forceinline__ uint32_t nib_hi(uint32_t w)
{
    return (w & 0x00F000F0u) ^ 0x64806480u;
}

__device__ __forceinline__ __half2 as_h2(uint32_t x)
{
    __half2 h;
    memcpy(&h, &x, sizeof h);
    return h;
}

__device__ __forceinline__ uint32_t as_u32(__half2 h)
{
    uint32_t x;
    memcpy(&x, &h, sizeof x);
    return x;
}

// fp16x2 {B + c0, B + c1} -> {c0, c1}, exact (every value involved is an
// fp16 integer below 2^11). Written with the half2 intrinsics (not inline
// assembly) so that a constant B can be encoded in the instruction.
__device__ __forceinline__ uint32_t h2_sub(uint32_t x, uint32_t b2)
{
    return as_u32(__hsub2(as_h2(x), as_h2(b2)));
}

// fp16x2 {1152 + 16 c0, 1152 + 16 c1} -> {c0, c1}: x / 16 - 72, exact.
__device__ __forceinline__ uint32_t h2_hi_code(uint32_t x)
{
    return as_u32(__hfma2(as_h2(x), as_h2(0x2C002C00u), as_h2(0xD480D480u)));
}

constexpr uint32_t kH2_1152 = 0x64806480u; // fp16x2 {1152, 1152}
constexpr uint32_t kH2_1032 = 0x64086408u; // fp16x2 {1032, 1032}

// Exact fp16x2 codes: two INT8 codes (bytes of `w` XORed with 0x80, picked
// by SEL, first land as {1152 + c0, 1152 + c1}); two low INT4 nibbles (bits
// 0-3, 16-19); two high ones (4-7, 20-23).
template <uint32_t SEL>
__device__ __forceinline__ uint32_t code8_h2(uint32_t w)
{
    return h2_sub(__byte_perm(w, 0x64646464u, SEL), kH2_1152);
}

__device__ __forceinline__ uint32_t code4_lo_h2(uint32_t w) { return h2_sub(nib_lo(w), kH2_1032); }

__device__ __forceinline__ uint32_t code4_hi_h2(uint32_t w) { return h2_hi_code(nib_hi(w)); }

// fp32 values of the two halves of an fp16x2.
__device__ __forceinline__ void h2_to_f2(uint32_t x, float &lo, float &hi)
{
    asm("{.reg .f16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\tcvt.f32.f16 %1, h;}"
        : "=f"(lo), "=f"(hi)
        : "r"(x));
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// ---------------------------------------------------------------------------
// GQ query rows share each K/V tile: the g query heads of a kv head for each
// of NQ new tokens (NQ > 1: multi-query decode, each token masked causally).
template <int BITS, int D_, int GQ_, int NW_, int S_, int MINB_ = 1, int BPI_ = 2, int NQ_ = 1,
          bool TMA_ = false>
struct QuantMmaPolicy {
    static_assert(BITS == 8 || BITS == 4, "INT8 or INT4 codes");
    static_assert(BPI_ == 1 || BPI_ == 2 || BPI_ == 4, "1, 2 or 4 blocks per ring item");
    static_assert(GQ_ % NQ_ == 0, "GQ = g * NQ");
    static constexpr int D = D_, GQ = GQ_, NW = NW_, S = S_, NQ = NQ_;
    static constexpr int BPI = BPI_;               // blocks per ring item
    static constexpr int kMinBlocks = MINB_;       // resident CTAs per SM the registers allow
    static constexpr int NT = (GQ + 7) / 8;        // 8-head tiles of S^T
    static constexpr int KS = D / 16;              // k-steps of Q.K
    static constexpr int CW = D / 8;               // d values of O^T per thread (see to_merge)
    static constexpr int ROWB = D * BITS / 8;      // bytes per code row: 128/64 (8), 64/32 (4)
    static constexpr int TILE = kBlockTokens * ROWB; // bytes of a K (or V) code tile
    // A stage: the K tiles of the item's blocks, then their V tiles; the
    // extra area: 16 K scales per block, then 16 V scales per block.
    static constexpr int STAGE = 2 * BPI * TILE;
    static constexpr int EXTRA = 128 * BPI;
    static constexpr int QBYTES = 0;
    static constexpr uint32_t TX = STAGE + EXTRA;
    static constexpr float kScaleRatio = 64.f;     // V-scale base moves beyond this
    using Layout = SmemLayout<D, GQ, NW, S, STAGE, EXTRA, QBYTES>;

    struct State {
        uint32_t qf[NT][KS][2]; // Q'^T B-fragments (fp16, k permuted)
        float qexp;             // 2^e: Q' = q * 2^-e
        float m[NT][2], l[NT][2];
        float acc[NT][KS][4];   // O^T accumulators: rows permuted d, cols heads
        float sbase;            // V-scale base of acc (0 until a nonzero scale is seen)
        float sinv;             // 1 / sbase (0 while sbase is 0)
    };

    // Tiles of 1-2 KiB move faster as 16-byte cp.async copies spread over the
    // warp's lanes than as TMA boxes: every lane issues its share of the K
    // and V tiles (and lanes 0-8*BPI-1 the scales), then arrives on the stage
    // barrier once its copies land (the barrier expects 32 arrivals). A block
    // whose row is < 0 (absent or bad) is not loaded.
    // TMA_: lane 0 instead loads each block's K and V tiles as TMA boxes (the
    // pool's tensor maps: 128/64-byte swizzle for INT8 as the readers expect,
    // none for INT4) and its scale rows as 64-byte bulk copies.
    static constexpr bool kLsuLoad = !TMA_;
    static constexpr uint32_t kArrivals = TMA_ ? 1 : 32;
    static constexpr int CHUNKS = TILE / 16;       // 16-byte chunks per tile

    // Shared-memory offset of chunk c of a tile: 16-byte chunk c % (ROWB/16)
    // of row c / (ROWB/16), swizzled as the K/V readers expect.
    __device__ static uint32_t chunk_off(int c)
    {
        constexpr int CPR = ROWB / 16;
        if constexpr (BITS == 8)
            return swz<ROWB>(c / CPR, c % CPR);
        else
            return (uint32_t)(c * 16);
    }

    __device__ static void issue_lanes(uint32_t dst, uint32_t extra, const int32_t (&rows)[BPI],
                                       const DecodeParams &p, const void *kc, const void *vc,
                                       uint64_t pol, int lane)
    {
#pragma unroll
        for (int j = 0; j < BPI; ++j) {
            if (rows[j] < 0)
                continue;
            const uint8_t *ks = static_cast<const uint8_t *>(kc) + (size_t)rows[j] * TILE;
            const uint8_t *vs = static_cast<const uint8_t *>(vc) + (size_t)rows[j] * TILE;
#pragma unroll
            for (int c = lane; c < CHUNKS; c += 32) {
                cp_async_16(dst + j * TILE + chunk_off(c), ks + 16 * c, pol);
                cp_async_16(dst + (BPI + j) * TILE + chunk_off(c), vs + 16 * c, pol);
            }
        }
        if (lane < 8 * BPI) {
            const int t = lane >> 2, kind = t / BPI, j = t - kind * BPI; // t = kind*BPI + j
            int32_t rj = rows[0]; // selects, not an indexed (local-memory) array
#pragma unroll
            for (int i = 1; i < BPI; ++i)
                rj = j == i ? rows[i] : rj;
            if (rj >= 0) {
                const float *sc = (kind ? p.v_scale : p.k_scale) + (size_t)rj * kBlockTokens;
                cp_async_16(extra + 64 * t + 16 * (lane & 3), sc + 4 * (lane & 3), pol);
            }
        }
    }

    __device__ static uint32_t tx_bytes(uint32_t mask)
    {
        return (uint32_t)__popc(mask) * (2u * TILE + 128u);
    }

    __device__ static void issue(uint32_t dst, uint32_t extra, const int32_t (&rows)[BPI],
                                 uint32_t bar, const CUtensorMap *tk, const CUtensorMap *tv,
                                 const DecodeParams &p, uint64_t pol)
    {
#pragma unroll
        for (int j = 0; j < BPI; ++j) {
            if (rows[j] < 0)
                continue;
            const int32_t y = rows[j] * kBlockTokens;
            tma_load_2d(dst + j * TILE, tk, 0, y, bar, pol);
            tma_load_2d(dst + (BPI + j) * TILE, tv, 0, y, bar, pol);
            bulk_load_1d(extra + 64 * j, p.k_scale + (size_t)rows[j] * kBlockTokens, 64, bar, pol);
            bulk_load_1d(extra + 64 * (BPI + j), p.v_scale + (size_t)rows[j] * kBlockTokens, 64,
                         bar, pol);
        }
    }

    // Physical d of the k values thread t holds in k-step kk; the A and B
    // fragments agree on this permutation, so the dot product is unchanged.
    //   INT8: register 0 = (d0, d0+1), register 1 = (d0+2, d0+3), d0 below
    //         (four consecutive bytes of one 16-byte chunk of the row).
    //   INT4: register r = (d, d+4) with d = D/4*t + 8*(kk/2) + (kk%2) + 2*r
    //         (nibbles j, j+4 of one 32-bit word of the thread's slice; odd
    //         k-steps hold the x16 nibbles).
    __device__ static int kperm_d0(int kk, int t) { return 64 * (kk >> 2) + 16 * t + 4 * (kk & 3); }

    // Issue the loads of a segment's raw bf16 q words into st.qf (they land
    // while the previous segment merges); finish_q converts them in place.
    template <class RowFn>
    __device__ static void prefetch_q(State &st, const DecodeParams &p, RowFn row_of)
    {
        const int lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hl = nt * 8 + gid;
            const int64_t qr = hl < GQ ? row_of(hl) : -1;
            const bool ok = qr >= 0;
            const __nv_bfloat16 *row = p.q + (ok ? qr : 0) * D;
            if constexpr (BITS == 8) {
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const uint2 w = ok ? __ldg(reinterpret_cast<const uint2 *>(row + kperm_d0(kk, t4)))
                                       : make_uint2(0u, 0u);
                    st.qf[nt][kk][0] = w.x;
                    st.qf[nt][kk][1] = w.y;
                }
            } else {
#pragma unroll
                for (int wi = 0; wi < KS / 2; ++wi) {
                    const uint4 w = ok ? __ldg(reinterpret_cast<const uint4 *>(
                                             row + (D / 4) * t4 + 8 * wi))
                                       : make_uint4(0u, 0u, 0u, 0u);
                    st.qf[nt][2 * wi][0] = w.x;
                    st.qf[nt][2 * wi][1] = w.y;
                    st.qf[nt][2 * wi + 1][0] = w.z;
                    st.qf[nt][2 * wi + 1][1] = w.w;
                }
            }
        }
    }

    __device__ static void finish_q(State &st)
    {
        float qv[NT][KS][4]; // per k-step: register 0 (lo, hi), register 1 (lo, hi)
        float mx = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            if constexpr (BITS == 8) {
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const uint32_t wx = st.qf[nt][kk][0], wy = st.qf[nt][kk][1];
                    qv[nt][kk][0] = __uint_as_float(wx << 16);
                    qv[nt][kk][1] = __uint_as_float(wx & 0xffff0000u);
                    qv[nt][kk][2] = __uint_as_float(wy << 16);
                    qv[nt][kk][3] = __uint_as_float(wy & 0xffff0000u);
                }
            } else {
#pragma unroll
                for (int wi = 0; wi < KS / 2; ++wi) {
                    // d values D/4*t4 + 8*wi + 0..7
                    float x[8];
                    const uint32_t ww[4] = {st.qf[nt][2 * wi][0], st.qf[nt][2 * wi][1],
                                            st.qf[nt][2 * wi + 1][0], st.qf[nt][2 * wi + 1][1]};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        x[2 * i] = __uint_as_float(ww[i] << 16);
                        x[2 * i + 1] = __uint_as_float(ww[i] & 0xffff0000u);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) { // k-step 2*wi + h: nibbles h, h+2 (+4)
                        qv[nt][2 * wi + h][0] = x[h];
                        qv[nt][2 * wi + h][1] = x[h + 4];
                        qv[nt][2 * wi + h][2] = x[h + 2];
                        qv[nt][2 * wi + h][3] = x[h + 6];
                    }
                }
            }
#pragma unroll
            for (int kk = 0; kk < KS; ++kk)
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    mx = fmaxf(mx, fabsf(qv[nt][kk][i]));
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        // e = max(0, floor(log2 max|q|) - 14): max|q| * 2^-e < 2^15
        const int E = (int)((__float_as_uint(mx) >> 23) & 0xff) - 127;
        const int e = E > 14 ? E - 14 : 0;
        st.qexp = __uint_as_float((uint32_t)(127 + e) << 23);
        const float down = __uint_as_float((uint32_t)(127 - e) << 23);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                st.qf[nt][kk][0] = pack_f16x2(qv[nt][kk][0] * down, qv[nt][kk][1] * down);
                st.qf[nt][kk][1] = pack_f16x2(qv[nt][kk][2] * down, qv[nt][kk][3] * down);
            }
    }

    __device__ static void reset(State &st)
    {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                st.m[nt][e] = -INFINITY;
                st.l[nt][e] = 0.f;
            }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    st.acc[nt][mt][e] = 0.f;
        st.sbase = 0.f;
        st.sinv = 0.f;
    }

    // One item of BPI 16-token blocks: block j's K codes at kt + j*TILE, its V
    // codes at kt + (BPI+j)*TILE, its scales at extra + 64*j (K) and
    // extra + 64*(BPI+j) (V). Tokens [lo, valid) of the item are attended,
    // those of block j only if bit j of mask is set (the block was loaded);
    // rem = ctx - (the item's first position), for the causal mask (NQ > 1).
    __device__ static void compute(State &st, uint32_t kt, uint32_t extra, int lo, int valid,
                                   int rem, float scale_log2, uint32_t mask)
    {
        const int lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;

        // ---- S^T = Kcode . Q'^T per block (INT4: even and odd k-steps in two chains)
        float s0[BPI][NT][4], s1[BPI][NT][4];
#pragma unroll
        for (int j = 0; j < BPI; ++j)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    s0[j][nt][e] = s1[j][nt][e] = 0.f;
        auto kstep = [&](int j, int kk, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (BITS == 4 && (kk & 1)) // INT4: two chains per block; INT8: one
                    mma_f16_16816(s1[j][nt], a0, a1, a2, a3, st.qf[nt][kk][0], st.qf[nt][kk][1]);
                else
                    mma_f16_16816(s0[j][nt], a0, a1, a2, a3, st.qf[nt][kk][0], st.qf[nt][kk][1]);
            }
        };
        if constexpr (BITS == 8) {
            // rows gid, gid+8: 16-byte chunks 4*g4 + t4 (swizzled), 16 codes each
#pragma unroll
            for (int g4 = 0; g4 < D / 64; ++g4)
#pragma unroll
                for (int j = 0; j < BPI; ++j) {
                    const uint32_t kj = kt + j * TILE;
                    const uint4 ka = lds128(kj + swz<ROWB>(gid, 4 * g4 + t4));
                    const uint4 kb = lds128(kj + swz<ROWB>(gid + 8, 4 * g4 + t4));
                    const uint32_t wa[4] = {ka.x ^ 0x80808080u, ka.y ^ 0x80808080u,
                                            ka.z ^ 0x80808080u, ka.w ^ 0x80808080u};
                    const uint32_t wb[4] = {kb.x ^ 0x80808080u, kb.y ^ 0x80808080u,
                                            kb.z ^ 0x80808080u, kb.w ^ 0x80808080u};
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        kstep(j, 4 * g4 + i, code8_h2<0x4140>(wa[i]), code8_h2<0x4140>(wb[i]),
                              code8_h2<0x4342>(wa[i]), code8_h2<0x4342>(wb[i]));
                }
        } else {
            // rows gid, gid+8: the thread's D/8 contiguous bytes (D/4 codes), unswizzled
#pragma unroll
            for (int j = 0; j < BPI; ++j) {
                const uint32_t kj = kt + j * TILE;
                uint32_t wa[KS / 2], wb[KS / 2];
                if constexpr (D == 128) {
                    const uint4 ka = lds128(kj + gid * ROWB + 16 * t4);
                    const uint4 kb = lds128(kj + (gid + 8) * ROWB + 16 * t4);
                    wa[0] = ka.x; wa[1] = ka.y; wa[2] = ka.z; wa[3] = ka.w;
                    wb[0] = kb.x; wb[1] = kb.y; wb[2] = kb.z; wb[3] = kb.w;
                } else {
                    const uint2 ka = lds64(kj + gid * ROWB + 8 * t4);
                    const uint2 kb = lds64(kj + (gid + 8) * ROWB + 8 * t4);
                    wa[0] = ka.x; wa[1] = ka.y;
                    wb[0] = kb.x; wb[1] = kb.y;
                }
#pragma unroll
                for (int wi = 0; wi < KS / 2; ++wi) {
                    // nibbles 0, 4 and (after >> 8) 2, 6: even k-step; 1, 5 and 3, 7: odd
                    const uint32_t xa = wa[wi], xb = wb[wi], ya = xa >> 8, yb = xb >> 8;
                    kstep(j, 2 * wi, code4_lo_h2(xa), code4_lo_h2(xb), code4_lo_h2(ya),
                          code4_lo_h2(yb));
                    kstep(j, 2 * wi + 1, code4_hi_h2(xa), code4_hi_h2(xb), code4_hi_h2(ya),
                          code4_hi_h2(yb));
                }
            }
        }

        // ---- scores in the log2 domain; rows gid, gid+8 of block j are
        // tokens 16j + gid, 16j + gid + 8
        bool lo_ok[BPI], hi_ok[BPI];
        float pr[BPI][NT][4];
        bool need = false; // some lane's score exceeds its column's base by 2^kRescaleLog2
#pragma unroll
        for (int j = 0; j < BPI; ++j) {
            const int tl = 16 * j + gid, th = tl + 8;
            const bool in = (mask >> j) & 1u;
            lo_ok[j] = in && tl >= lo && tl < valid;
            hi_ok[j] = in && th >= lo && th < valid;
            const float f_lo = st.qexp * lds_f32(extra + 64 * j + 4 * gid) * scale_log2;
            const float f_hi = st.qexp * lds_f32(extra + 64 * j + 4 * (gid + 8)) * scale_log2;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // S^T element c: token row gid (c < 2) or gid+8, head column 2t4 + (c & 1)
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float sb = BITS == 8 ? s0[j][nt][c] : s0[j][nt][c] + s1[j][nt][c];
                    const float sc = sb * ((c & 2) ? f_hi : f_lo);
                    pr[j][nt][c] = ((c & 2) ? hi_ok[j] : lo_ok[j]) ? sc : -INFINITY;
                }
                if constexpr (NQ > 1) // block j starts 16j tokens into the item
                    causal_mask<GQ, NQ>(pr[j][nt], nt, gid, t4, rem - 16 * j);
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    need |= fmaxf(pr[j][nt][e], pr[j][nt][e + 2]) > st.m[nt][e] + kRescaleLog2;
            }
        }
        // Lazy rescale (as in the bf16 policy), and the column maxima are only
        // reduced across the lanes when some lane exceeds its base.
        if (__any_sync(0xffffffffu, need)) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float mx = -INFINITY;
#pragma unroll
                    for (int j = 0; j < BPI; ++j)
                        mx = fmaxf(mx, fmaxf(pr[j][nt][e], pr[j][nt][e + 2]));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                    if (mx > st.m[nt][e] + kRescaleLog2) { // same in every lane of the column
                        const float alpha = fast_exp2(st.m[nt][e] - mx);
                        st.m[nt][e] = mx;
                        st.l[nt][e] *= alpha;
#pragma unroll
                        for (int mt = 0; mt < KS; ++mt) {
                            st.acc[nt][mt][e] *= alpha;
                            st.acc[nt][mt][e + 2] *= alpha;
                        }
                    }
                }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const float base = (st.m[nt][e] == -INFINITY) ? 0.f : st.m[nt][e];
#pragma unroll
                for (int j = 0; j < BPI; ++j) {
                    pr[j][nt][e] = fast_exp2(pr[j][nt][e] - base);
                    pr[j][nt][e + 2] = fast_exp2(pr[j][nt][e + 2] - base);
                    st.l[nt][e] += pr[j][nt][e] + pr[j][nt][e + 2];
                }
            }

        // ---- V scales: fold sv / s_base into the weights; the base moves only
        // when some row's scale exceeds it kScaleRatio-fold (then to the max)
        float sv_lo[BPI], sv_hi[BPI], svm = 0.f;
#pragma unroll
        for (int j = 0; j < BPI; ++j) {
            sv_lo[j] = lo_ok[j] ? lds_f32(extra + 64 * (BPI + j) + 4 * gid) : 0.f;
            sv_hi[j] = hi_ok[j] ? lds_f32(extra + 64 * (BPI + j) + 4 * (gid + 8)) : 0.f;
            svm = fmaxf(svm, fmaxf(sv_lo[j], sv_hi[j]));
        }
        if (__any_sync(0xffffffffu, svm > st.sbase * kScaleRatio)) {
            svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, 4));
            svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, 8));
            svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, 16));
            svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, 1));
            svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, 2));
            const float f = st.sbase / svm;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int mt = 0; mt < KS; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        st.acc[nt][mt][e] *= f;
            }
            st.sbase = svm;
            st.sinv = 1.f / svm;
        }
        // W^T as B fragments (tokens x heads): transpose of the score layout.
        uint32_t pb0[BPI][NT], pb1[BPI][NT];
#pragma unroll
        for (int j = 0; j < BPI; ++j) {
            const float r_lo = sv_lo[j] * st.sinv, r_hi = sv_hi[j] * st.sinv;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const uint32_t w0 = pack_f16x2(pr[j][nt][0] * r_lo, pr[j][nt][1] * r_lo);
                const uint32_t w1 = pack_f16x2(pr[j][nt][2] * r_hi, pr[j][nt][3] * r_hi);
                pb0[j][nt] = movmatrix_trans(w0);
                pb1[j][nt] = movmatrix_trans(w1);
            }
        }

        // ---- O^T += Vcode^T . W^T, one k-step per block. Thread rows
        // (tokens) 2t, 2t+1, 2t+8, 2t+9 of the block; its d values are
        // CW*gid + 2*mt + r for row tile mt, r = 0 (A rows gid) or 1 (A rows
        // gid+8): CW contiguous codes of each token row.
#pragma unroll
        for (int j = 0; j < BPI; ++j) {
            const uint32_t vt = kt + (BPI + j) * TILE;
            auto pv = [&](int mt, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_f16_16816(st.acc[nt][mt], a0, a1, a2, a3, pb0[j][nt], pb1[j][nt]);
            };
            if constexpr (BITS == 8) {
                constexpr int WPR = D / 32; // 32-bit words per thread per row
                uint32_t ra[WPR], rb[WPR], rc[WPR], rd[WPR];
                if constexpr (D == 128) {
                    const uint4 x0 = lds128(vt + swz<128>(2 * t4, gid));
                    const uint4 x1 = lds128(vt + swz<128>(2 * t4 + 1, gid));
                    const uint4 x2 = lds128(vt + swz<128>(2 * t4 + 8, gid));
                    const uint4 x3 = lds128(vt + swz<128>(2 * t4 + 9, gid));
                    ra[0] = x0.x; ra[1] = x0.y; ra[2] = x0.z; ra[3] = x0.w;
                    rb[0] = x1.x; rb[1] = x1.y; rb[2] = x1.z; rb[3] = x1.w;
                    rc[0] = x2.x; rc[1] = x2.y; rc[2] = x2.z; rc[3] = x2.w;
                    rd[0] = x3.x; rd[1] = x3.y; rd[2] = x3.z; rd[3] = x3.w;
                } else {
                    const uint32_t off = 8u * (gid & 1);
                    const uint2 x0 = lds64(vt + swz<64>(2 * t4, gid >> 1) + off);
                    const uint2 x1 = lds64(vt + swz<64>(2 * t4 + 1, gid >> 1) + off);
                    const uint2 x2 = lds64(vt + swz<64>(2 * t4 + 8, gid >> 1) + off);
                    const uint2 x3 = lds64(vt + swz<64>(2 * t4 + 9, gid >> 1) + off);
                    ra[0] = x0.x; ra[1] = x0.y;
                    rb[0] = x1.x; rb[1] = x1.y;
                    rc[0] = x2.x; rc[1] = x2.y;
                    rd[0] = x3.x; rd[1] = x3.y;
                }
#pragma unroll
                for (int i = 0; i < WPR; ++i) {
                    // word i holds d values 4i..4i+3: row tiles 2i (bytes 0, 1), 2i+1 (bytes 2, 3)
                    const uint32_t A = ra[i] ^ 0x80808080u, B = rb[i] ^ 0x80808080u;
                    const uint32_t C = rc[i] ^ 0x80808080u, E = rd[i] ^ 0x80808080u;
                    const uint32_t ab_lo = __byte_perm(A, B, 0x5140);
                    const uint32_t ab_hi = __byte_perm(A, B, 0x7362);
                    const uint32_t ce_lo = __byte_perm(C, E, 0x5140);
                    const uint32_t ce_hi = __byte_perm(C, E, 0x7362);
                    pv(2 * i, code8_h2<0x4140>(ab_lo), code8_h2<0x4342>(ab_lo),
                       code8_h2<0x4140>(ce_lo), code8_h2<0x4342>(ce_lo));
                    pv(2 * i + 1, code8_h2<0x4140>(ab_hi), code8_h2<0x4342>(ab_hi),
                       code8_h2<0x4140>(ce_hi), code8_h2<0x4342>(ce_hi));
                }
            } else {
                // CW/2 bytes per row; byte k of word i holds d values 8i+2k (low
                // nibble) and 8i+2k+1 (high nibble): row tile 4i+k
                constexpr int WPR = CW / 8;
                uint32_t ra[WPR], rb[WPR], rc[WPR], rd[WPR];
                if constexpr (D == 128) {
                    const uint2 x0 = lds64(vt + (2 * t4) * ROWB + 8 * gid);
                    const uint2 x1 = lds64(vt + (2 * t4 + 1) * ROWB + 8 * gid);
                    const uint2 x2 = lds64(vt + (2 * t4 + 8) * ROWB + 8 * gid);
                    const uint2 x3 = lds64(vt + (2 * t4 + 9) * ROWB + 8 * gid);
                    ra[0] = x0.x; ra[1] = x0.y;
                    rb[0] = x1.x; rb[1] = x1.y;
                    rc[0] = x2.x; rc[1] = x2.y;
                    rd[0] = x3.x; rd[1] = x3.y;
                } else {
                    ra[0] = lds32(vt + (2 * t4) * ROWB + 4 * gid);
                    rb[0] = lds32(vt + (2 * t4 + 1) * ROWB + 4 * gid);
                    rc[0] = lds32(vt + (2 * t4 + 8) * ROWB + 4 * gid);
                    rd[0] = lds32(vt + (2 * t4 + 9) * ROWB + 4 * gid);
                }
#pragma unroll
                for (int i = 0; i < WPR; ++i) {
                    const uint32_t A = ra[i], B = rb[i], C = rc[i], E = rd[i];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // bytes {A_k, A_k, B_k, B_k}: nibble pairs (row 2t, row 2t+1) of
                        // d (low nibbles) and d + 1 (high nibbles: A rows gid + 8)
                        const uint32_t sel = k | (k << 4) | ((4 + k) << 8) | ((4 + k) << 12);
                        const uint32_t Y = __byte_perm(A, B, sel), Z = __byte_perm(C, E, sel);
                        pv(4 * i + k, code4_lo_h2(Y), code4_hi_h2(Y), code4_lo_h2(Z),
                           code4_hi_h2(Z));
                    }
                }
            }
        }
    }

    // This warp's state -> its slice of the merge area: [warp][h] = (m, l, acc[D]),
    // acc at true scale (times s_base) and in natural d order.
    __device__ static void to_merge(State &st, float *merge)
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
                if (h < GQ && gid == 0) {
                    float *mb = merge + (warp * GQ + h) * (D + 2);
                    mb[0] = st.m[nt][e];
                    mb[1] = l;
                }
            }
        // acc[nt][mt][e]: row gid (e < 2) or gid+8 (e >= 2) of row tile mt is
        // d = CW*gid + 2*mt + (e >> 1); column 2t4 + (e & 1) is the head.
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const int h = nt * 8 + 2 * t4 + c;
                if (h < GQ) {
                    float *mb = merge + (warp * GQ + h) * (D + 2) + 2 + CW * gid;
#pragma unroll
                    for (int mt = 0; mt < KS; ++mt) {
                        mb[2 * mt] = st.acc[nt][mt][c] * st.sbase;
                        mb[2 * mt + 1] = st.acc[nt][mt][c + 2] * st.sbase;
                    }
                }
            }
    }
};

} // namespace pa
