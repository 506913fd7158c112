// Device half of copy-on-write: copy whole physical blocks of the pool.
//
// "LLM 推理底层：KV Cache 显存几何、GQA/MLA 压缩与 PagedAttention 调度", section
// "Prefix Caching 与 Copy-on-Write": a branch that appends to a shared, partly
// filled last block gets a fresh block holding the filled slots; "KV Cache
// 显存管理全景", 考点 4: only that 16-token block is copied.
//
// One block of one tensor is n_kv * 16 * d_h elements, contiguous in the
// [num_blocks][n_kv][16][d_h] pool (32 KiB for 8 bf16 heads of 128), plus
// n_kv * 16 fp32 scales for INT8 and INT4. CTA (x, z) copies chunk x % chunks of pair
// x / chunks of tensor z (0 = K, 1 = V): 256 threads, four 16-byte loads in
// flight each, then four stores. The copy is HBM-bound: read + write of the
// block bytes, nothing else.
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr int64_t kChunkBytes = (int64_t)kThreads * 16 * kUnroll; // 16 KiB

__global__ void __launch_bounds__(kThreads)
block_copy_kernel(uint8_t *k_cache, uint8_t *v_cache, float *k_scale, float *v_scale,
                  const int32_t *__restrict__ pairs, int64_t num_blocks, int64_t tile_bytes,
                  int chunks, int scales_per_block, int32_t *dev_status)
{
    const int64_t pair = blockIdx.x / chunks;
    const int chunk = (int)(blockIdx.x - pair * chunks);
    const int32_t src = __ldg(pairs + 2 * pair), dst = __ldg(pairs + 2 * pair + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (chunk == 0 && blockIdx.z == 0 && threadIdx.x == 0 && dev_status)
            atomicOr(dev_status, PA_DEV_BAD_BLOCK_BIT);
        return;
    }
    uint8_t *pool = blockIdx.z ? v_cache : k_cache;
    const uint4 *from = reinterpret_cast<const uint4 *>(pool + (int64_t)src * tile_bytes);
    uint4 *to = reinterpret_cast<uint4 *>(pool + (int64_t)dst * tile_bytes);
    const int64_t n16 = tile_bytes / 16;
    const int64_t base = (int64_t)chunk * (kChunkBytes / 16) + threadIdx.x;
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = base + (int64_t)u * kThreads;
        if (i < n16)
            r[u] = __ldcs(from + i);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = base + (int64_t)u * kThreads;
        if (i < n16)
            to[i] = r[u];
    }
    if (scales_per_block && chunk == 0) {
        float *sc = blockIdx.z ? v_scale : k_scale;
        const float4 *sf = reinterpret_cast<const float4 *>(sc + (int64_t)src * scales_per_block);
        float4 *sd = reinterpret_cast<float4 *>(sc + (int64_t)dst * scales_per_block);
        for (int i = threadIdx.x; i < scales_per_block / 4; i += kThreads)
            sd[i] = __ldcs(sf + i);
    }
}

} // namespace

cudaError_t launch_block_copy(void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                              const int32_t *pairs, int32_t num_pairs, int64_t num_blocks,
                              int n_kv, int d_h, int kind, int32_t *dev_status,
                              cudaStream_t stream)
{
    // bytes of one block of one tensor: bf16 2, INT8 1, INT4 1/2 per element
    const int64_t tile_bytes = (int64_t)n_kv * 16 * d_h * (kind == 0 ? 4 : kind == 1 ? 2 : 1) / 2;
    const int chunks = (int)((tile_bytes + kChunkBytes - 1) / kChunkBytes);
    const int64_t gx = (int64_t)num_pairs * chunks;
    if (gx > INT32_MAX)
        return cudaErrorInvalidValue;
    block_copy_kernel<<<dim3((unsigned)gx, 1, 2), kThreads, 0, stream>>>(
        static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), k_scale, v_scale, pairs,
        num_blocks, tile_bytes, chunks, kind ? n_kv * 16 : 0, dev_status);
    return cudaGetLastError();
}

} // namespace pa
