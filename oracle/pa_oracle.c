/*
 * CPU oracle for paged decode attention and the slot-mapped cache append.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, obviously correct
 * restatement of what the CUDA library computes. Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it. It shares no
 * code, header, table or helper with the CUDA library.
 *
 * Sources (web pages; cited by title and section):
 *  [F] "LLM 推理底层：KV Cache 显存几何、GQA/MLA 压缩与 PagedAttention 调度"
 *      (blog.faulkner.fun)
 *  [Q] "【infra之路】10-PagedAttention 与 KV Cache 管理" (qwbw.cn)
 *  [G] "kv-cache-guide" (guijiagi.com)
 *  [T] "KV Cache 显存管理全景：内存碎片拟合推导、vLLM PagedAttention 虚拟内存与
 *      Prefix Caching" (talentme.airsota.com)
 *  [H] "LLM 推理引擎设计：KV Cache、PagedAttention 与连续批处理" (hx.sn.cn)
 *
 * Floating point: attention runs in double precision. The INT8 quantiser runs
 * in IEEE single precision (the scales it produces are fp32 numbers, so the
 * codes are defined by fp32 arithmetic); dequantisation forms code*scale in fp32
 * and widens that product to double, as [G] §4.2 `dequantize_kv` does
 * (`k_quant.float() * k_scale`).
 *
 * Layout of the pool (the block layout [num_blocks, H, block_size, D] that
 * [G] §7.1 gives for PagedAttention):
 *   cache[blk][kv_head][offset][d]   (bf16 bit patterns or int8 codes)
 *   scale[blk][kv_head][offset]      (fp32, INT8 only)
 *
 * Status: functions return 0, or OR these bits into *status:
 *   1 = a physical block id outside [0, num_blocks)
 *   2 = a slot outside [0, num_blocks*block_size)
 *   4 = a context length < 0 or larger than the block table can hold
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#include <stdlib.h>

#define ORC_BAD_BLOCK 1
#define ORC_BAD_SLOT 2
#define ORC_BAD_CTX 4

/* bf16 -> float is exact: the bf16 bits are the top half of the fp32 bits. */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------------
 * KV byte formula, [F] "KV Cache 容量公式":
 *   M_KV = 2 * L * n_kv * d_h * S * B * b_dtype
 * (the leading 2 counts K and V). [G] §2.1 and [T] 第二章 state the same
 * product. Returned as double so that b_dtype = 0.5 (INT4) is expressible.
 * ---------------------------------------------------------------------- */
double oracle_kv_bytes(double L, double n_kv, double d_h, double S, double B, double b_dtype)
{
    return 2.0 * L * n_kv * d_h * S * B * b_dtype;
}

/* ------------------------------------------------------------------------
 * Slot-mapped append of new K/V rows ([T] 第三章 `write_kv`; [F]
 * "逻辑块与物理块映射"): a slot s names physical block s / block_size and
 * offset s % block_size. Row t of k (all n_kv heads) goes to
 *   k_cache[s/bs][h][s%bs][:] = k[t][h][:]
 * Slots < 0 are padding and are skipped.
 * ---------------------------------------------------------------------- */
int oracle_cache_write_bf16(const uint16_t *k, const uint16_t *v, const int64_t *slots, int64_t T,
                            int n_kv, int d_h, int block_size, int64_t num_blocks,
                            uint16_t *k_cache, uint16_t *v_cache)
{
    int status = 0;
    for (int64_t t = 0; t < T; ++t) {
        int64_t s = slots[t];
        if (s < 0)
            continue;
        if (s >= num_blocks * block_size) {
            status |= ORC_BAD_SLOT;
            continue;
        }
        int64_t blk = s / block_size, off = s % block_size;
        for (int h = 0; h < n_kv; ++h) {
            const uint16_t *src_k = k + ((t * n_kv + h) * (int64_t)d_h);
            const uint16_t *src_v = v + ((t * n_kv + h) * (int64_t)d_h);
            int64_t dst = ((blk * n_kv + h) * block_size + off) * (int64_t)d_h;
            for (int d = 0; d < d_h; ++d) {
                k_cache[dst + d] = src_k[d];
                v_cache[dst + d] = src_v[d];
            }
        }
    }
    return status;
}

/* ------------------------------------------------------------------------
 * INT8 symmetric quantiser, [G] §4.2 `quantize_kv_cache` (num_bits == 8):
 *   scale = max_d |x_d| / 127         (max over the last dim: per token, per head)
 *   code  = clamp(round(x / scale), -128, 127)
 * in fp32: the amax of bf16 values is exact in fp32, the two divisions are
 * IEEE single-precision divisions, and round() is torch's round-half-to-even
 * (nearbyintf in the default rounding mode). A row of zeros has scale 0; its
 * codes are defined as 0 (the page leaves 0/0 open).
 * ---------------------------------------------------------------------- */
void oracle_quantize_row_int8(const uint16_t *x, int d_h, int8_t *code, float *scale_out)
{
    volatile float amax = 0.0f; /* volatile: keep every step in fp32 */
    for (int d = 0; d < d_h; ++d) {
        float a = fabsf(bf16_bits_to_float(x[d]));
        if (a > amax)
            amax = a;
    }
    volatile float scale = amax / 127.0f;
    *scale_out = scale;
    for (int d = 0; d < d_h; ++d) {
        if (scale == 0.0f) {
            code[d] = 0;
            continue;
        }
        volatile float r = bf16_bits_to_float(x[d]) / scale;
        float n = nearbyintf(r);
        if (n < -128.0f)
            n = -128.0f;
        if (n > 127.0f)
            n = 127.0f;
        code[d] = (int8_t)n;
    }
}

/* Same append as oracle_cache_write_bf16, quantising each (token, head) row. */
int oracle_cache_write_int8(const uint16_t *k, const uint16_t *v, const int64_t *slots, int64_t T,
                            int n_kv, int d_h, int block_size, int64_t num_blocks,
                            int8_t *k_cache, int8_t *v_cache, float *k_scale, float *v_scale)
{
    int status = 0;
    for (int64_t t = 0; t < T; ++t) {
        int64_t s = slots[t];
        if (s < 0)
            continue;
        if (s >= num_blocks * block_size) {
            status |= ORC_BAD_SLOT;
            continue;
        }
        int64_t blk = s / block_size, off = s % block_size;
        for (int h = 0; h < n_kv; ++h) {
            int64_t row = (blk * n_kv + h) * block_size + off;
            oracle_quantize_row_int8(k + (t * n_kv + h) * (int64_t)d_h, d_h,
                                     k_cache + row * d_h, &k_scale[row]);
            oracle_quantize_row_int8(v + (t * n_kv + h) * (int64_t)d_h, d_h,
                                     v_cache + row * d_h, &v_scale[row]);
        }
    }
    return status;
}

/* ------------------------------------------------------------------------
 * INT4 symmetric quantiser, [G] §4.2 `quantize_kv_cache` (num_bits == 4):
 *   scale = max_d |x_d| / 7
 *   code  = clamp(round(x / scale), -8, 7)
 * with the same fp32 steps as the INT8 quantiser. Codes are returned one per
 * int8 here; the cache packs two per byte (see oracle_cache_write_int4).
 * ---------------------------------------------------------------------- */
void oracle_quantize_row_int4(const uint16_t *x, int d_h, int8_t *code, float *scale_out)
{
    volatile float amax = 0.0f;
    for (int d = 0; d < d_h; ++d) {
        float a = fabsf(bf16_bits_to_float(x[d]));
        if (a > amax)
            amax = a;
    }
    volatile float scale = amax / 7.0f;
    *scale_out = scale;
    for (int d = 0; d < d_h; ++d) {
        if (scale == 0.0f) {
            code[d] = 0;
            continue;
        }
        volatile float r = bf16_bits_to_float(x[d]) / scale;
        float n = nearbyintf(r);
        if (n < -8.0f)
            n = -8.0f;
        if (n > 7.0f)
            n = 7.0f;
        code[d] = (int8_t)n;
    }
}

/* INT4 append: each (token, head) row of d_h values becomes d_h/2 bytes, the
 * code of element 2i in the low nibble of byte i and that of 2i+1 in the high
 * nibble, each a 4-bit two's-complement number (the pages say only "packed
 * two per byte"; this order is the plainest reading). */
int oracle_cache_write_int4(const uint16_t *k, const uint16_t *v, const int64_t *slots, int64_t T,
                            int n_kv, int d_h, int block_size, int64_t num_blocks,
                            uint8_t *k_cache, uint8_t *v_cache, float *k_scale, float *v_scale)
{
    int status = 0;
    int8_t *codes = (int8_t *)malloc((size_t)d_h);
    for (int64_t t = 0; t < T; ++t) {
        int64_t s = slots[t];
        if (s < 0)
            continue;
        if (s >= num_blocks * block_size) {
            status |= ORC_BAD_SLOT;
            continue;
        }
        int64_t blk = s / block_size, off = s % block_size;
        for (int h = 0; h < n_kv; ++h) {
            int64_t row = (blk * n_kv + h) * block_size + off;
            for (int which = 0; which < 2; ++which) {
                const uint16_t *x = (which ? v : k) + (t * n_kv + h) * (int64_t)d_h;
                uint8_t *dst = (which ? v_cache : k_cache) + row * (d_h / 2);
                oracle_quantize_row_int4(x, d_h, codes, which ? &v_scale[row] : &k_scale[row]);
                for (int i = 0; i < d_h / 2; ++i)
                    dst[i] = (uint8_t)((codes[2 * i] & 0xF) | ((codes[2 * i + 1] & 0xF) << 4));
            }
        }
    }
    free(codes);
    return status;
}

/* One cached K or V element in double precision. kv_kind: 0 bf16, 1 INT8,
 * 2 INT4. INT8/INT4: the fp32 product code*scale ([G] §4.2
 * `dequantize_kv`), then widened. */
static double cached_elem(const void *cache, const float *scales, int kv_kind, int64_t row, int d,
                          int d_h)
{
    if (kv_kind == 1) {
        const int8_t *c = (const int8_t *)cache;
        float x = (float)c[row * d_h + d] * scales[row];
        return (double)x;
    }
    if (kv_kind == 2) {
        const uint8_t *c = (const uint8_t *)cache;
        int nib = (c[row * (d_h / 2) + d / 2] >> (4 * (d & 1))) & 0xF;
        int code = nib >= 8 ? nib - 16 : nib;
        float x = (float)code * scales[row];
        return (double)x;
    }
    const uint16_t *c = (const uint16_t *)cache;
    return (double)bf16_bits_to_float(c[row * d_h + d]);
}

/* ------------------------------------------------------------------------
 * Decode attention over the paged pool.
 *
 * For each sequence b and query head h ([F] "自回归解码与 KV Cache 的物理来源",
 * eq. for o_t):
 *   o = softmax(q K^T * scale) V  over the ctx_b cached tokens (the new token
 *   included: K_{1:t} holds k_t).
 * GQA ([F] table "注意力头架构演进"): g = n_h / n_kv query heads share one KV
 * head; query head h reads KV head h / g (contiguous groups).
 * Token j of sequence b lives in physical block block_tables[b][j / bs] at
 * offset j % bs ([F] "逻辑块与物理块映射", block_idx / block_offset).
 * The definition is written out directly: every cached token's score, the
 * softmax of all of them (maximum subtracted before exponentiating), then
 * the probability-weighted sum of the V rows; each row is located through
 * the block table as it is needed ([Q] §3.4 describes the same paged
 * computation).
 * ctx_b == 0 gives an all-zero output row.
 * out: double [B][n_h][d_h].
 * ---------------------------------------------------------------------- */
int oracle_decode(const uint16_t *q, const void *k_cache, const void *v_cache, const float *k_scale,
                  const float *v_scale, int kv_kind, const int32_t *block_tables,
                  int max_blocks_per_seq, const int32_t *context_lens, int B, int n_h, int n_kv,
                  int d_h, int block_size, int64_t num_blocks, double scale, double *out)
{
    int status = 0;
    int g = n_h / n_kv;
    double *scores = NULL;
    int64_t cap = 0;
    for (int b = 0; b < B; ++b) {
        int64_t ctx = context_lens[b];
        int bad = 0;
        if (ctx < 0 || ctx > (int64_t)max_blocks_per_seq * block_size) {
            status |= ORC_BAD_CTX;
            bad = 1;
        }
        /* every physical block the sequence uses must exist */
        for (int64_t i = 0; !bad && i * block_size < ctx; ++i) {
            int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + i];
            if (blk < 0 || blk >= num_blocks) {
                status |= ORC_BAD_BLOCK;
                bad = 1;
            }
        }
        if (bad || ctx == 0) {
            for (int h = 0; h < n_h; ++h)
                for (int d = 0; d < d_h; ++d)
                    out[((int64_t)b * n_h + h) * d_h + d] = 0.0;
            continue;
        }
        if (ctx > cap) {
            free(scores);
            cap = ctx;
            scores = (double *)malloc(sizeof(double) * (size_t)cap);
        }
        for (int h = 0; h < n_h; ++h) {
            int kvh = h / g;
            const uint16_t *qh = q + ((int64_t)b * n_h + h) * d_h;
            /* pass 1: scores, block by block */
            double m = -INFINITY;
            for (int64_t j = 0; j < ctx; ++j) {
                int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / block_size];
                int64_t off = j % block_size;
                int64_t row = (blk * n_kv + kvh) * block_size + off;
                double dot = 0.0;
                for (int d = 0; d < d_h; ++d)
                    dot += (double)bf16_bits_to_float(qh[d]) *
                           cached_elem(k_cache, k_scale, kv_kind, row, d, d_h);
                scores[j] = dot * scale;
                if (scores[j] > m)
                    m = scores[j];
            }
            /* softmax */
            double denom = 0.0;
            for (int64_t j = 0; j < ctx; ++j) {
                scores[j] = exp(scores[j] - m);
                denom += scores[j];
            }
            /* pass 2: weighted sum of V, block by block */
            double *o = out + ((int64_t)b * n_h + h) * d_h;
            for (int d = 0; d < d_h; ++d)
                o[d] = 0.0;
            for (int64_t j = 0; j < ctx; ++j) {
                int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / block_size];
                int64_t off = j % block_size;
                int64_t row = (blk * n_kv + kvh) * block_size + off;
                double w = scores[j] / denom;
                for (int d = 0; d < d_h; ++d)
                    o[d] += w * cached_elem(v_cache, v_scale, kv_kind, row, d, d_h);
            }
        }
    }
    free(scores);
    return status;
}

/* ------------------------------------------------------------------------
 * Decode attention with a sliding window and INT8 attention-sink rows.
 *
 * Sliding window ([G] §5.1 `SlidingWindowKVCache`: only the latest w tokens
 * are kept and attended): with window > 0, sequence b attends positions
 * j in [max(0, ctx_b - window), ctx_b); window == 0 attends all ctx_b.
 * Block-table entries of logical blocks wholly before the window are never
 * read (a sliding-window cache may have released them).
 *
 * Attention sink ([G] §4.3: the first k tokens, typically 4, stay
 * unquantised in a quantised cache): for an INT8 or INT4 pool and n_sink > 0, an attended
 * position j < n_sink takes its K and V rows from the bf16 sink rows
 * sink_k/sink_v[b][kv][j][:] ([B][n_kv][n_sink][d_h] bit patterns) instead of
 * dequantising the pool. Every other position reads the pool as in
 * oracle_decode. n_sink must be 0 for a bf16 pool.
 *
 * Validation: a context length outside [0, max_blocks*block_size] and a
 * block id outside the pool among the blocks the window reads (positions
 * >= max(window start, n_sink)) are reported; that sequence's output is 0.
 * The softmax and the two passes are those of oracle_decode.
 * ---------------------------------------------------------------------- */
int oracle_decode_window(const uint16_t *q, const void *k_cache, const void *v_cache,
                         const float *k_scale, const float *v_scale, int kv_kind,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, int B, int n_h, int n_kv, int d_h,
                         int block_size, int64_t num_blocks, double scale, int window, int n_sink,
                         const uint16_t *sink_k, const uint16_t *sink_v, double *out)
{
    int status = 0;
    int g = n_h / n_kv;
    double *scores = NULL;
    int64_t cap = 0;
    for (int b = 0; b < B; ++b) {
        int64_t ctx = context_lens[b];
        int bad = 0;
        if (ctx < 0 || ctx > (int64_t)max_blocks_per_seq * block_size) {
            status |= ORC_BAD_CTX;
            bad = 1;
        }
        int64_t start = (window > 0 && ctx > window) ? ctx - window : 0;
        int64_t pool_from = start > n_sink ? start : n_sink; /* first position read from the pool */
        for (int64_t j = pool_from; !bad && j < ctx; ++j) {
            int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / block_size];
            if (blk < 0 || blk >= num_blocks) {
                status |= ORC_BAD_BLOCK;
                bad = 1;
            }
        }
        if (bad || ctx == 0) {
            for (int h = 0; h < n_h; ++h)
                for (int d = 0; d < d_h; ++d)
                    out[((int64_t)b * n_h + h) * d_h + d] = 0.0;
            continue;
        }
        int64_t n = ctx - start;
        if (n > cap) {
            free(scores);
            cap = n;
            scores = (double *)malloc(sizeof(double) * (size_t)cap);
        }
        for (int h = 0; h < n_h; ++h) {
            int kvh = h / g;
            const uint16_t *qh = q + ((int64_t)b * n_h + h) * d_h;
            double m = -INFINITY;
            for (int64_t j = start; j < ctx; ++j) {
                double dot = 0.0;
                if (j < n_sink) {
                    const uint16_t *kr = sink_k + (((int64_t)b * n_kv + kvh) * n_sink + j) * d_h;
                    for (int d = 0; d < d_h; ++d)
                        dot += (double)bf16_bits_to_float(qh[d]) * (double)bf16_bits_to_float(kr[d]);
                } else {
                    int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / block_size];
                    int64_t row = (blk * n_kv + kvh) * block_size + j % block_size;
                    for (int d = 0; d < d_h; ++d)
                        dot += (double)bf16_bits_to_float(qh[d]) *
                               cached_elem(k_cache, k_scale, kv_kind, row, d, d_h);
                }
                scores[j - start] = dot * scale;
                if (scores[j - start] > m)
                    m = scores[j - start];
            }
            double denom = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                scores[j] = exp(scores[j] - m);
                denom += scores[j];
            }
            double *o = out + ((int64_t)b * n_h + h) * d_h;
            for (int d = 0; d < d_h; ++d)
                o[d] = 0.0;
            for (int64_t j = start; j < ctx; ++j) {
                double w = scores[j - start] / denom;
                if (j < n_sink) {
                    const uint16_t *vr = sink_v + (((int64_t)b * n_kv + kvh) * n_sink + j) * d_h;
                    for (int d = 0; d < d_h; ++d)
                        o[d] += w * (double)bf16_bits_to_float(vr[d]);
                } else {
                    int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / block_size];
                    int64_t row = (blk * n_kv + kvh) * block_size + j % block_size;
                    for (int d = 0; d < d_h; ++d)
                        o[d] += w * cached_elem(v_cache, v_scale, kv_kind, row, d, d_h);
                }
            }
        }
    }
    free(scores);
    return status;
}

/* ------------------------------------------------------------------------
 * Multi-query decode: n_q new tokens per sequence attend at once, as in
 * speculative verification (a draft of k tokens checked in one step, [H]
 * §6 "投机解码") or a chunk of a chunked prefill ([F] "Chunked Prefill"). The
 * n_q new tokens of sequence b are its last n_q positions ctx_b - n_q ..
 * ctx_b - 1 (their K/V already appended); query i (0-based) attends causally
 * to positions [0, ctx_b - n_q + i], i.e. every earlier token and itself.
 * A query whose range is empty (ctx_b < n_q - i) gets a zero output.
 *   q   [B][n_q][n_h][d_h] bf16 bits,  out [B][n_q][n_h][d_h] double.
 * Per query the arithmetic is oracle_decode's: scores, max-subtracted
 * softmax, weighted V sum, in double precision.
 * ---------------------------------------------------------------------- */
int oracle_decode_mq(const uint16_t *q, const void *k_cache, const void *v_cache,
                     const float *k_scale, const float *v_scale, int kv_kind,
                     const int32_t *block_tables, int max_blocks_per_seq,
                     const int32_t *context_lens, int B, int n_q, int n_h, int n_kv, int d_h,
                     int block_size, int64_t num_blocks, double scale, double *out)
{
    int status = 0;
    int g = n_h / n_kv;
    double *scores = NULL;
    int64_t cap = 0;
    for (int b = 0; b < B; ++b) {
        int64_t ctx = context_lens[b];
        int bad = 0;
        if (ctx < 0 || ctx > (int64_t)max_blocks_per_seq * block_size) {
            status |= ORC_BAD_CTX;
            bad = 1;
        }
        for (int64_t i = 0; !bad && i * block_size < ctx; ++i) {
            int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + i];
            if (blk < 0 || blk >= num_blocks) {
                status |= ORC_BAD_BLOCK;
                bad = 1;
            }
        }
        if (ctx > cap) {
            free(scores);
            cap = ctx;
            scores = (double *)malloc(sizeof(double) * (size_t)cap);
        }
        for (int i = 0; i < n_q; ++i) {
            int64_t n = bad ? 0 : ctx - n_q + i + 1; /* attended positions 0 .. n-1 */
            for (int h = 0; h < n_h; ++h) {
                double *o = out + (((int64_t)b * n_q + i) * n_h + h) * d_h;
                for (int d = 0; d < d_h; ++d)
                    o[d] = 0.0;
                if (n <= 0)
                    continue;
                int kvh = h / g;
                const uint16_t *qh = q + (((int64_t)b * n_q + i) * n_h + h) * d_h;
                double m = -INFINITY;
                for (int64_t j = 0; j < n; ++j) {
                    int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / block_size];
                    int64_t row = (blk * n_kv + kvh) * block_size + j % block_size;
                    double dot = 0.0;
                    for (int d = 0; d < d_h; ++d)
                        dot += (double)bf16_bits_to_float(qh[d]) *
                               cached_elem(k_cache, k_scale, kv_kind, row, d, d_h);
                    scores[j] = dot * scale;
                    if (scores[j] > m)
                        m = scores[j];
                }
                double denom = 0.0;
                for (int64_t j = 0; j < n; ++j) {
                    scores[j] = exp(scores[j] - m);
                    denom += scores[j];
                }
                for (int64_t j = 0; j < n; ++j) {
                    int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / block_size];
                    int64_t row = (blk * n_kv + kvh) * block_size + j % block_size;
                    double w = scores[j] / denom;
                    for (int d = 0; d < d_h; ++d)
                        o[d] += w * cached_elem(v_cache, v_scale, kv_kind, row, d, d_h);
                }
            }
        }
    }
    free(scores);
    return status;
}

/* ------------------------------------------------------------------------
 * The raw attention scores s_j = scale * <q_h, K_j> of every query head over
 * its sequence's cached tokens, in double precision: the argument of the
 * softmax in [F] "自回归解码与 KV Cache 的物理来源" (eq. for o_t), with K_j
 * found through the block table as in oracle_decode. Tests use them to check
 * the dynamic range an input reaches (how far the running maximum climbs).
 * out: double [B][n_h][max_ctx]; entries at j >= ctx_b are NaN. Sequences
 * with a bad context length or block id report it and get NaN rows.
 * ---------------------------------------------------------------------- */
int oracle_scores(const uint16_t *q, const void *k_cache, const float *k_scale, int kv_kind,
                  const int32_t *block_tables, int max_blocks_per_seq,
                  const int32_t *context_lens, int B, int n_h, int n_kv, int d_h,
                  int block_size, int64_t num_blocks, double scale, int64_t max_ctx,
                  double *out)
{
    int status = 0;
    int g = n_h / n_kv;
    for (int b = 0; b < B; ++b) {
        int64_t ctx = context_lens[b];
        int bad = ctx < 0 || ctx > max_ctx || ctx > (int64_t)max_blocks_per_seq * block_size;
        if (bad)
            status |= ORC_BAD_CTX;
        for (int64_t j = 0; !bad && j < ctx; j += block_size) {
            int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / block_size];
            if (blk < 0 || blk >= num_blocks) {
                status |= ORC_BAD_BLOCK;
                bad = 1;
            }
        }
        for (int h = 0; h < n_h; ++h) {
            double *row_out = out + ((int64_t)b * n_h + h) * max_ctx;
            for (int64_t j = 0; j < max_ctx; ++j)
                row_out[j] = NAN;
            if (bad)
                continue;
            const uint16_t *qh = q + ((int64_t)b * n_h + h) * d_h;
            for (int64_t j = 0; j < ctx; ++j) {
                int64_t blk = block_tables[(int64_t)b * max_blocks_per_seq + j / block_size];
                int64_t row = (blk * n_kv + h / g) * block_size + j % block_size;
                double dot = 0.0;
                for (int d = 0; d < d_h; ++d)
                    dot += (double)bf16_bits_to_float(qh[d]) *
                           cached_elem(k_cache, k_scale, kv_kind, row, d, d_h);
                row_out[j] = dot * scale;
            }
        }
    }
    return status;
}
