// Slot-mapped append of new K/V rows into the paged pool.
//
// "KV Cache 显存管理全景：…" (talentme.airsota.com), 第三章 `write_kv`, and
// "LLM 推理底层：…" (blog.faulkner.fun), "逻辑块与物理块映射": slot s is
// physical block s / 16 at offset s % 16; a row of every KV head goes to
//     cache[s / 16][h][s % 16][:].
// INT8 ("kv-cache-guide" (guijiagi.com) §4.2, quantize_kv_cache with 8 bits):
// per (token, head) row, in IEEE fp32,
//     scale = max|x| / 127,  code = clamp(round_half_even(x / scale), -128, 127).
// The divisions are correctly rounded (__fdiv_rn), rintf rounds half to even,
// and a row of zeros stores scale 0 with zero codes.
// INT4 (same page, num_bits 4): scale = max|x| / 7, code = clamp(round(x /
// scale), -8, 7), two codes per byte: element 2i in the low nibble of byte i.
//
// One warp handles one (token, head) row: lane l owns d = l*E .. l*E+E-1.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_internal.h"

namespace pa {

namespace {

template <int E>
__device__ __forceinline__ void load_row(const __nv_bfloat16 *src, float (&x)[E], uint32_t (&raw)[E / 2])
{
    if constexpr (E == 4) {
        const uint2 w = *reinterpret_cast<const uint2 *>(src);
        raw[0] = w.x;
        raw[1] = w.y;
    } else {
        raw[0] = *reinterpret_cast<const uint32_t *>(src);
    }
#pragma unroll
    for (int i = 0; i < E / 2; ++i) {
        x[2 * i] = __uint_as_float(raw[i] << 16);
        x[2 * i + 1] = __uint_as_float(raw[i] & 0xffff0000u);
    }
}

template <int E>
__device__ __forceinline__ void quantize_store(const float (&x)[E], int8_t *dst_codes, float *dst_scale)
{
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i)
        a = fmaxf(a, fabsf(x[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float scale = __fdiv_rn(a, 127.0f);
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        float c = 0.f;
        if (scale != 0.f) {
            c = rintf(__fdiv_rn(x[i], scale));
            c = fminf(fmaxf(c, -128.0f), 127.0f);
        }
        packed |= (uint32_t)(uint8_t)(int8_t)(int)c << (8 * i);
    }
    const int lane = threadIdx.x & 31;
    if constexpr (E == 4)
        reinterpret_cast<uint32_t *>(dst_codes)[lane] = packed;
    else
        reinterpret_cast<uint16_t *>(dst_codes)[lane] = (uint16_t)packed;
    if (lane == 0)
        *dst_scale = scale;
}

// INT4 codes of a row: lane l packs its E codes into E/2 bytes.
template <int E>
__device__ __forceinline__ void quantize_store4(const float (&x)[E], uint8_t *dst_codes,
                                                float *dst_scale)
{
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < E; ++i)
        a = fmaxf(a, fabsf(x[i]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const float scale = __fdiv_rn(a, 7.0f);
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < E; ++i) {
        float c = 0.f;
        if (scale != 0.f) {
            c = rintf(__fdiv_rn(x[i], scale));
            c = fminf(fmaxf(c, -8.0f), 7.0f);
        }
        packed |= ((uint32_t)(int)c & 0xFu) << (4 * i);
    }
    const int lane = threadIdx.x & 31;
    if constexpr (E == 4)
        reinterpret_cast<uint16_t *>(dst_codes)[lane] = (uint16_t)packed;
    else
        dst_codes[lane] = (uint8_t)packed;
    if (lane == 0)
        *dst_scale = scale;
}

// KIND: 0 bf16, 1 INT8, 2 INT4
template <int D, int KIND>
__global__ void __launch_bounds__(256)
    cache_write_kernel(const __nv_bfloat16 *__restrict__ k, const __nv_bfloat16 *__restrict__ v,
                       const int64_t *__restrict__ slots, int64_t rows, int n_kv, int64_t num_slots,
                       void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                       int32_t *dev_status)
{
    // a decode launched next on the stream may be scheduled now; it waits for
    // this grid to complete before reading the cache
    asm volatile("griddepcontrol.launch_dependents;");
    constexpr int E = D / 32;
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows)
        return;
    const int lane = threadIdx.x & 31;
    const int64_t t = row / n_kv;
    const int h = (int)(row - t * n_kv);
    const int64_t s = slots[t];
    if (s < 0)
        return;
    if (s >= num_slots) {
        if (lane == 0 && h == 0 && dev_status)
            atomicOr(dev_status, PA_DEV_BAD_SLOT_BIT);
        return;
    }
    const int64_t dst_row = ((s >> 4) * n_kv + h) * 16 + (s & 15);
    float xk[E], xv[E];
    uint32_t rk[E / 2], rv[E / 2];
    load_row<E>(k + row * D + lane * E, xk, rk);
    load_row<E>(v + row * D + lane * E, xv, rv);
    if constexpr (KIND == 0) {
        __nv_bfloat16 *kc = static_cast<__nv_bfloat16 *>(k_cache) + dst_row * D + lane * E;
        __nv_bfloat16 *vc = static_cast<__nv_bfloat16 *>(v_cache) + dst_row * D + lane * E;
        if constexpr (E == 4) {
            *reinterpret_cast<uint2 *>(kc) = make_uint2(rk[0], rk[1]);
            *reinterpret_cast<uint2 *>(vc) = make_uint2(rv[0], rv[1]);
        } else {
            *reinterpret_cast<uint32_t *>(kc) = rk[0];
            *reinterpret_cast<uint32_t *>(vc) = rv[0];
        }
    } else if constexpr (KIND == 1) {
        quantize_store<E>(xk, static_cast<int8_t *>(k_cache) + dst_row * D, k_scale + dst_row);
        quantize_store<E>(xv, static_cast<int8_t *>(v_cache) + dst_row * D, v_scale + dst_row);
    } else {
        quantize_store4<E>(xk, static_cast<uint8_t *>(k_cache) + dst_row * (D / 2),
                           k_scale + dst_row);
        quantize_store4<E>(xv, static_cast<uint8_t *>(v_cache) + dst_row * (D / 2),
                           v_scale + dst_row);
    }
}

// Attention-sink rows: row (t, h) with 0 <= positions[t] < n_sink and a valid
// batch row goes to sink[seq_rows[t]][h][positions[t]][:] unchanged (bf16).
// One warp per (token, kv head) row, 16-byte copies.
__global__ void __launch_bounds__(256)
    sink_write_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                      const int32_t *__restrict__ seq_rows, const int32_t *__restrict__ positions,
                      int64_t rows, int n_kv, int chunks, int n_sink, int num_seqs, uint4 *sink_k,
                      uint4 *sink_v)
{
    const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (row >= rows)
        return;
    const int lane = threadIdx.x & 31;
    const int64_t t = row / n_kv;
    const int h = (int)(row - t * n_kv);
    const int32_t pos = positions[t], b = seq_rows[t];
    if (pos < 0 || pos >= n_sink || b < 0 || b >= num_seqs)
        return;
    const int64_t dst = (((int64_t)b * n_kv + h) * n_sink + pos) * chunks;
    for (int c = lane; c < chunks; c += 32) {
        sink_k[dst + c] = k[row * chunks + c];
        sink_v[dst + c] = v[row * chunks + c];
    }
}

} // namespace

cudaError_t launch_sink_write(const void *k, const void *v, const int32_t *seq_rows,
                              const int32_t *positions, int64_t T, int n_kv, int d_h, int n_sink,
                              int num_seqs, void *sink_k, void *sink_v, cudaStream_t stream)
{
    const int64_t rows = T * n_kv;
    const int64_t blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffff)
        return cudaErrorInvalidValue;
    sink_write_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
        static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), seq_rows, positions, rows,
        n_kv, d_h * 2 / 16, n_sink, num_seqs, static_cast<uint4 *>(sink_k),
        static_cast<uint4 *>(sink_v));
    return cudaGetLastError();
}

cudaError_t launch_cache_write(const void *k, const void *v, const int64_t *slots, int64_t T,
                               int n_kv, int d_h, int kind, int64_t num_slots, void *k_cache,
                               void *v_cache, float *k_scale, float *v_scale, int32_t *dev_status,
                               cudaStream_t stream)
{
    const int64_t rows = T * n_kv;
    const int64_t blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffff)
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)blocks), block(256);
    const __nv_bfloat16 *kb = static_cast<const __nv_bfloat16 *>(k);
    const __nv_bfloat16 *vb = static_cast<const __nv_bfloat16 *>(v);
#define PA_CW(D, K)                                                                           \
    cache_write_kernel<D, K><<<grid, block, 0, stream>>>(kb, vb, slots, rows, n_kv, num_slots,    \
                                                         k_cache, v_cache, k_scale, v_scale,     \
                                                         dev_status)
    if (d_h == 128 && kind == 0)
        PA_CW(128, 0);
    else if (d_h == 128 && kind == 1)
        PA_CW(128, 1);
    else if (d_h == 128 && kind == 2)
        PA_CW(128, 2);
    else if (d_h == 64 && kind == 0)
        PA_CW(64, 0);
    else if (d_h == 64 && kind == 1)
        PA_CW(64, 1);
    else if (d_h == 64 && kind == 2)
        PA_CW(64, 2);
    else
        return cudaErrorInvalidValue;
#undef PA_CW
    return cudaGetLastError();
}

} // namespace pa
