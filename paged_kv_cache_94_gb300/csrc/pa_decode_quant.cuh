// Quantised K/V policy for the decode kernel (INT8 or INT4 codes): tensor-core
// contractions on exact fp16 copies of the codes.
//
// The cache holds integer codes and one fp32 scale per (token, kv head)
// ("kv-cache-guide" (guijiagi.com) §4.2: x = code * scale; 8-bit codes in
// [-128, 127], 4-bit codes in [-8, 7] packed two per byte, low nibble first).
// Every code is exact in fp16. A code c becomes fp16 by writing its
// offset-binary form (c + 128, or c + 8) into the mantissa of 1024
// (exponent bits 0x64): that half is 1024 + offset + c, and one subtraction
// of 1024 + offset leaves c. Both contractions then run as mma.sync
// m16n8k16 with fp16 inputs and fp32 accumulation:
//   S^T[16 tok][8 heads] = Kcode[16 tok][D] . Q'^T[D][8 heads]
//       (tokens on M; the k index is permuted so each thread's A fragments
//        for all k-steps come from one 16-byte (or 8-byte) load of a row)
//   s = S^T * 2^e * k_scale[tok] * scale * log2(e)
//   O[16 heads][D] += W[16 heads][16 tok] . Vcode[16 tok][D]
//       (heads on M; output columns are permuted so each thread's B
//        fragments for all D/8 column tiles come from one load of each of
//        its four token rows)
// Q' = q * 2^-e with e >= 0 chosen per (sequence, kv head) so that
// max|Q'| < 2^15: the bf16 -> fp16 conversion is then exact for every
// normal value. W = p * v_scale[tok] / s_base, where s_base is a running
// V-scale base that only moves (rescaling O) when a block's largest V scale
// exceeds it 64-fold, so W <= 2^8 * 2^6 stays far below fp16's maximum.
#pragma once

#include <cuda_fp16.h>

#include "pa_decode.cuh"

namespace pa {

// Two int8 bytes (b0 low, b1 high, already XORed with 0x80) at byte positions
// selected by SEL of `w` -> fp16x2 {code0, code1}.
template <uint32_t SEL>
__device__ __forceinline__ uint32_t bytes_to_h2(uint32_t w)
{
    uint32_t h = __byte_perm(w, 0x64646464u, SEL);
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64806480u));
    return r;
}

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

// Two 4-bit codes (offset form, nibbles j and j+4 of `w`) -> fp16x2 {code_j, code_j+4}.
template <int J>
__device__ __forceinline__ uint32_t nibs_to_h2(uint32_t w)
{
    const uint32_t h = ((w >> (4 * J)) & 0x000F000Fu) | 0x64006400u;
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(0x64086408u));
    return r;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// ---------------------------------------------------------------------------
template <int BITS, int D_, int GQ_, int NW_, int S_>
struct QuantMmaPolicy {
    static_assert(BITS == 8 || BITS == 4, "INT8 or INT4 codes");
    static constexpr int D = D_, GQ = GQ_, NW = NW_, S = S_;
    static constexpr int NT = (GQ + 7) / 8;        // 8-head tiles of S^T
    static constexpr int KS = D / 16;              // k-steps of Q.K
    static constexpr int VT = D / 8;               // column tiles of O
    static constexpr int CW = D / 8;               // O columns per thread (see to_merge)
    static constexpr int ROWB = D * BITS / 8;      // bytes per code row: 128/64 (8), 64/32 (4)
    static constexpr int TILE = kBlockTokens * ROWB; // bytes of a K (or V) code tile
    static constexpr int STAGE = 2 * TILE;
    static constexpr int EXTRA = 128;              // 16 K scales + 16 V scales
    static constexpr int QBYTES = 0;
    static constexpr uint32_t TX = STAGE + EXTRA;
    static constexpr float kScaleRatio = 64.f;     // V-scale base moves beyond this
    using Layout = SmemLayout<D, GQ, NW, S, STAGE, EXTRA, QBYTES>;

    struct State {
        uint32_t qf[NT][KS][2]; // Q'^T B-fragments (fp16, k permuted)
        float qexp;             // 2^e: Q' = q * 2^-e
        float m[NT][2], l[NT][2];
        float acc[VT][4];       // O accumulators: rows heads gid / gid+8, cols permuted d
        float sbase;            // V-scale base of acc (0 until a nonzero scale is seen)
    };

    __device__ static void issue(uint32_t dst, uint32_t extra, int32_t row, uint32_t bar,
                                 const CUtensorMap *tk, const CUtensorMap *tv,
                                 const DecodeParams &p, uint64_t pol)
    {
        const int32_t y = row * kBlockTokens;
        tma_load_2d(dst, tk, 0, y, bar, pol);
        tma_load_2d(dst + TILE, tv, 0, y, bar, pol);
        bulk_load_1d(extra, p.k_scale + (size_t)row * kBlockTokens, 64, bar, pol);
        bulk_load_1d(extra + 64, p.v_scale + (size_t)row * kBlockTokens, 64, bar, pol);
    }

    // Physical d of the k values thread t holds in k-step kk; the A and B
    // fragments agree on this permutation, so the dot product is unchanged.
    //   INT8: register 0 = (d0, d0+1), register 1 = (d0+2, d0+3), d0 below
    //         (four consecutive bytes of one 16-byte chunk of the row).
    //   INT4: register r = (d, d+4) with d = D/4*t + 8*(kk/2) + 2*(kk%2) + r
    //         (nibbles j, j+4 of one 32-bit word of the thread's slice).
    __device__ static int kperm_d0(int kk, int t) { return 64 * (kk >> 2) + 16 * t + 4 * (kk & 3); }

    __device__ static void load_q(State &st, const DecodeParams &p, int b, int kvh,
                                  float * /*qsm*/)
    {
        const int lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
        const int n_h = p.n_kv * GQ;
        float qv[NT][KS][4]; // per k-step: register 0 (lo, hi), register 1 (lo, hi)
        float mx = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int hl = nt * 8 + gid;
            const bool ok = hl < GQ;
            const __nv_bfloat16 *row =
                p.q + ((size_t)b * n_h + (size_t)kvh * GQ + (ok ? hl : 0)) * D;
            if constexpr (BITS == 8) {
#pragma unroll
                for (int kk = 0; kk < KS; ++kk) {
                    const uint2 w = ok ? __ldg(reinterpret_cast<const uint2 *>(row + kperm_d0(kk, t4)))
                                       : make_uint2(0u, 0u);
                    qv[nt][kk][0] = __uint_as_float(w.x << 16);
                    qv[nt][kk][1] = __uint_as_float(w.x & 0xffff0000u);
                    qv[nt][kk][2] = __uint_as_float(w.y << 16);
                    qv[nt][kk][3] = __uint_as_float(w.y & 0xffff0000u);
                }
            } else {
#pragma unroll
                for (int wi = 0; wi < KS / 2; ++wi) {
                    // d values D/4*t4 + 8*wi + 0..7
                    const uint4 w = ok ? __ldg(reinterpret_cast<const uint4 *>(
                                             row + (D / 4) * t4 + 8 * wi))
                                       : make_uint4(0u, 0u, 0u, 0u);
                    float x[8];
                    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        x[2 * i] = __uint_as_float(ww[i] << 16);
                        x[2 * i + 1] = __uint_as_float(ww[i] & 0xffff0000u);
                    }
#pragma unroll
                    for (int h = 0; h < 2; ++h) { // k-step 2*wi + h: nibbles 2h, 2h+1 (+4)
                        qv[nt][2 * wi + h][0] = x[2 * h];
                        qv[nt][2 * wi + h][1] = x[2 * h + 4];
                        qv[nt][2 * wi + h][2] = x[2 * h + 1];
                        qv[nt][2 * wi + h][3] = x[2 * h + 5];
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
        for (int vt = 0; vt < VT; ++vt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                st.acc[vt][e] = 0.f;
        st.sbase = 0.f;
    }

    // One 16-token block: K codes at kt, V codes at kt + TILE, scales at extra
    // (16 K scales, then 16 V scales). Rows [lo, valid) are attended.
    __device__ static void compute(State &st, uint32_t kt, uint32_t extra, int lo, int valid,
                                   float scale_log2)
    {
        const int lane = threadIdx.x & 31, gid = lane >> 2, t4 = lane & 3;
        const uint32_t vt = kt + TILE;

        // ---- S^T = Kcode . Q'^T (two accumulator chains for ILP)
        float s0[NT][4], s1[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                s0[nt][e] = s1[nt][e] = 0.f;
        auto kstep = [&](int kk, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (kk & 1)
                    mma_f16_16816(s1[nt], a0, a1, a2, a3, st.qf[nt][kk][0], st.qf[nt][kk][1]);
                else
                    mma_f16_16816(s0[nt], a0, a1, a2, a3, st.qf[nt][kk][0], st.qf[nt][kk][1]);
            }
        };
        if constexpr (BITS == 8) {
            // rows gid, gid+8: 16-byte chunks 4*g4 + t4 (swizzled), 16 codes each
#pragma unroll
            for (int g4 = 0; g4 < D / 64; ++g4) {
                const uint4 ka = lds128(kt + swz<ROWB>(gid, 4 * g4 + t4));
                const uint4 kb = lds128(kt + swz<ROWB>(gid + 8, 4 * g4 + t4));
                const uint32_t wa[4] = {ka.x ^ 0x80808080u, ka.y ^ 0x80808080u,
                                        ka.z ^ 0x80808080u, ka.w ^ 0x80808080u};
                const uint32_t wb[4] = {kb.x ^ 0x80808080u, kb.y ^ 0x80808080u,
                                        kb.z ^ 0x80808080u, kb.w ^ 0x80808080u};
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    kstep(4 * g4 + j, bytes_to_h2<0x4140>(wa[j]), bytes_to_h2<0x4140>(wb[j]),
                          bytes_to_h2<0x4342>(wa[j]), bytes_to_h2<0x4342>(wb[j]));
            }
        } else {
            // rows gid, gid+8: the thread's D/8 contiguous bytes (D/4 codes), unswizzled
            uint32_t wa[KS / 2], wb[KS / 2];
            if constexpr (D == 128) {
                const uint4 ka = lds128(kt + gid * ROWB + 16 * t4);
                const uint4 kb = lds128(kt + (gid + 8) * ROWB + 16 * t4);
                wa[0] = ka.x; wa[1] = ka.y; wa[2] = ka.z; wa[3] = ka.w;
                wb[0] = kb.x; wb[1] = kb.y; wb[2] = kb.z; wb[3] = kb.w;
            } else {
                const uint2 ka = lds64(kt + gid * ROWB + 8 * t4);
                const uint2 kb = lds64(kt + (gid + 8) * ROWB + 8 * t4);
                wa[0] = ka.x; wa[1] = ka.y;
                wb[0] = kb.x; wb[1] = kb.y;
            }
#pragma unroll
            for (int wi = 0; wi < KS / 2; ++wi) {
                const uint32_t xa = wa[wi] ^ 0x88888888u, xb = wb[wi] ^ 0x88888888u;
                kstep(2 * wi, nibs_to_h2<0>(xa), nibs_to_h2<0>(xb), nibs_to_h2<1>(xa),
                      nibs_to_h2<1>(xb));
                kstep(2 * wi + 1, nibs_to_h2<2>(xa), nibs_to_h2<2>(xb), nibs_to_h2<3>(xa),
                      nibs_to_h2<3>(xb));
            }
        }

        // ---- scores in the log2 domain; rows gid, gid+8 are tokens
        const bool lo_ok = gid >= lo && gid < valid, hi_ok = gid + 8 >= lo && gid + 8 < valid;
        const float f_lo = st.qexp * lds_f32(extra + 4 * gid) * scale_log2;
        const float f_hi = st.qexp * lds_f32(extra + 4 * (gid + 8)) * scale_log2;
        float pr[NT][4];
        float alpha[NT][2];
        bool need = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            pr[nt][0] = lo_ok ? (s0[nt][0] + s1[nt][0]) * f_lo : -INFINITY;
            pr[nt][1] = lo_ok ? (s0[nt][1] + s1[nt][1]) * f_lo : -INFINITY;
            pr[nt][2] = hi_ok ? (s0[nt][2] + s1[nt][2]) * f_hi : -INFINITY;
            pr[nt][3] = hi_ok ? (s0[nt][3] + s1[nt][3]) * f_hi : -INFINITY;
            // lazy rescale of the softmax base (as in the bf16 policy)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float mx = fmaxf(pr[nt][e], pr[nt][e + 2]);
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                const bool up = mx > st.m[nt][e] + kRescaleLog2;
                const float mnew = up ? mx : st.m[nt][e];
                alpha[nt][e] = up ? fast_exp2(st.m[nt][e] - mnew) : 1.f;
                need |= up;
                st.m[nt][e] = mnew;
                const float base = (mnew == -INFINITY) ? 0.f : mnew;
                pr[nt][e] = fast_exp2(pr[nt][e] - base);
                pr[nt][e + 2] = fast_exp2(pr[nt][e + 2] - base);
            }
        }
        if (__any_sync(0xffffffffu, need)) {
            // O rows are heads gid and gid+8; head h's factor lives in lane
            // (h & 7) >> 1 of S^T tile h >> 3, slot h & 1
            const float a00 = __shfl_sync(0xffffffffu, alpha[0][0], gid >> 1);
            const float a01 = __shfl_sync(0xffffffffu, alpha[0][1], gid >> 1);
            const float al_lo = (gid & 1) ? a01 : a00;
            float al_hi = 1.f;
            if constexpr (NT > 1) {
                const float a10 = __shfl_sync(0xffffffffu, alpha[1][0], gid >> 1);
                const float a11 = __shfl_sync(0xffffffffu, alpha[1][1], gid >> 1);
                al_hi = (gid & 1) ? a11 : a10;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e)
                    st.l[nt][e] *= alpha[nt][e];
#pragma unroll
            for (int v = 0; v < VT; ++v) {
                st.acc[v][0] *= al_lo;
                st.acc[v][1] *= al_lo;
                st.acc[v][2] *= al_hi;
                st.acc[v][3] *= al_hi;
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                st.l[nt][e] += pr[nt][e] + pr[nt][e + 2];

        // ---- V scales: fold sv / s_base into the weights
        const float sv_lo = lo_ok ? lds_f32(extra + 64 + 4 * gid) : 0.f;
        const float sv_hi = hi_ok ? lds_f32(extra + 64 + 4 * (gid + 8)) : 0.f;
        float svm = fmaxf(sv_lo, sv_hi);
        svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, 4));
        svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, 8));
        svm = fmaxf(svm, __shfl_xor_sync(0xffffffffu, svm, 16));
        if (svm > st.sbase * kScaleRatio) { // warp-uniform: svm is the same in all lanes
            const float f = st.sbase / svm;
#pragma unroll
            for (int v = 0; v < VT; ++v)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    st.acc[v][e] *= f;
            st.sbase = svm;
        }
        const float inv = st.sbase > 0.f ? 1.f / st.sbase : 0.f;
        const float r_lo = sv_lo * inv, r_hi = sv_hi * inv;
        uint32_t pa[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            pa[nt][0] = movmatrix_trans(pack_f16x2(pr[nt][0] * r_lo, pr[nt][1] * r_lo));
            pa[nt][1] = movmatrix_trans(pack_f16x2(pr[nt][2] * r_hi, pr[nt][3] * r_hi));
        }
        const uint32_t a0 = pa[0][0], a2 = pa[0][1];
        const uint32_t a1 = NT > 1 ? pa[NT - 1][0] : 0u, a3 = NT > 1 ? pa[NT - 1][1] : 0u;

        // ---- O += W . Vcode; thread rows 2t, 2t+1, 2t+8, 2t+9, columns CW*gid + nt
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
                const uint32_t A = ra[i] ^ 0x80808080u, B = rb[i] ^ 0x80808080u;
                const uint32_t C = rc[i] ^ 0x80808080u, E = rd[i] ^ 0x80808080u;
                const uint32_t ab_lo = __byte_perm(A, B, 0x5140), ab_hi = __byte_perm(A, B, 0x7362);
                const uint32_t ce_lo = __byte_perm(C, E, 0x5140), ce_hi = __byte_perm(C, E, 0x7362);
                mma_f16_16816(st.acc[4 * i + 0], a0, a1, a2, a3, bytes_to_h2<0x4140>(ab_lo),
                              bytes_to_h2<0x4140>(ce_lo));
                mma_f16_16816(st.acc[4 * i + 1], a0, a1, a2, a3, bytes_to_h2<0x4342>(ab_lo),
                              bytes_to_h2<0x4342>(ce_lo));
                mma_f16_16816(st.acc[4 * i + 2], a0, a1, a2, a3, bytes_to_h2<0x4140>(ab_hi),
                              bytes_to_h2<0x4140>(ce_hi));
                mma_f16_16816(st.acc[4 * i + 3], a0, a1, a2, a3, bytes_to_h2<0x4342>(ab_hi),
                              bytes_to_h2<0x4342>(ce_hi));
            }
        } else {
            // CW/2 bytes per row: byte k of word wi holds columns 8wi+2k (low nibble), +1
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
                const uint32_t A = ra[i] ^ 0x88888888u, B = rb[i] ^ 0x88888888u;
                const uint32_t C = rc[i] ^ 0x88888888u, E = rd[i] ^ 0x88888888u;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    // bytes {A_k, A_k, B_k, B_k}: nibble pairs (row 2t, row 2t+1) of one column
                    const uint32_t sel = k | (k << 4) | ((4 + k) << 8) | ((4 + k) << 12);
                    const uint32_t Y = __byte_perm(A, B, sel), Z = __byte_perm(C, E, sel);
                    mma_f16_16816(st.acc[8 * i + 2 * k], a0, a1, a2, a3, nibs_to_h2<0>(Y),
                                  nibs_to_h2<0>(Z));
                    mma_f16_16816(st.acc[8 * i + 2 * k + 1], a0, a1, a2, a3, nibs_to_h2<1>(Y),
                                  nibs_to_h2<1>(Z));
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
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int h = gid + 8 * half;
            if (h < GQ) {
                float *mb = merge + (warp * GQ + h) * (D + 2) + 2;
#pragma unroll
                for (int v = 0; v < VT; ++v) {
                    mb[CW * (2 * t4) + v] = st.acc[v][2 * half] * st.sbase;
                    mb[CW * (2 * t4 + 1) + v] = st.acc[v][2 * half + 1] * st.sbase;
                }
            }
        }
    }
};

} // namespace pa
