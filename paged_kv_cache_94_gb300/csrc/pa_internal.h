// Declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#define PA_DEV_BAD_BLOCK_BIT 0x1
#define PA_DEV_BAD_SLOT_BIT 0x2
#define PA_DEV_BAD_CONTEXT_BIT 0x4
#define PA_DEV_TIMEOUT_BIT 0x8

namespace pa {

struct DecodeParams;

// One compiled decode kernel (a dtype, head dim and group size).
struct DecodeKernel {
    const void *fn;                    // __global__ entry (attributes, occupancy)
    int threads;                       // block size
    size_t (*smem_bytes)(int num_seqs); // dynamic shared memory for a batch size
    cudaError_t (*launch)(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p,
                          int grid, size_t smem, cudaStream_t stream);
};

// NULL when the combination is not compiled.
const DecodeKernel *find_decode_kernel_bf16(int d_h, int group);
const DecodeKernel *find_decode_kernel_int8(int d_h, int group);
const DecodeKernel *find_decode_kernel_int4(int d_h, int group);
// Shared-prefix decode: members per group for group size g (g * members <=
// 16 query rows per kv head), its kernels, and the group detection kernel
// (pa_share.cu).
constexpr int kShareMembers(int g) { return g <= 2 ? 8 : 16 / g; }
constexpr int kShareMinBlocks = 8;
// Split charge per unit in the shared-prefix launch (items; see kSegCost):
// sequence units, and group units.
#ifndef PA_SHARE_SEG_COST
#define PA_SHARE_SEG_COST 8
#endif
constexpr int kShareSegCost = PA_SHARE_SEG_COST;
#ifndef PA_SHARE_GROUP_SEG_COST
#define PA_SHARE_GROUP_SEG_COST PA_SHARE_SEG_COST
#endif
constexpr int kShareGroupSegCost = PA_SHARE_GROUP_SEG_COST;
const DecodeKernel *find_prefix_kernel(int kv_dtype, int d_h, int group);
// Bounded-wait self-test (pa_selftest.cu).
cudaError_t launch_wait_selftest(int32_t *dev_status, uint64_t limit_ns, cudaStream_t stream);
cudaError_t launch_share_detect(const int32_t *block_tables, int max_blocks,
                                const int32_t *context_lens, int B, int gm, int min_blocks,
                                int32_t *skip, int32_t *groups, int32_t *order, bool sort,
                                cudaStream_t stream);

// Multi-query (nq new tokens per sequence) bf16 kernels; NULL when not compiled.
const DecodeKernel *find_decode_kernel_bf16_mq(int d_h, int group, int nq);
const DecodeKernel *find_decode_kernel_int8_mq(int d_h, int group, int nq);
const DecodeKernel *find_decode_kernel_int4_mq(int d_h, int group, int nq);

cudaError_t launch_cache_write(const void *k, const void *v, const int64_t *slots, int64_t T,
                               int n_kv, int d_h, int kind, int64_t num_slots, void *k_cache,
                               void *v_cache, float *k_scale, float *v_scale, int32_t *dev_status,
                               cudaStream_t stream);

cudaError_t launch_sink_write(const void *k, const void *v, const int32_t *seq_rows,
                              const int32_t *positions, int64_t T, int n_kv, int d_h, int n_sink,
                              int num_seqs, void *sink_k, void *sink_v, cudaStream_t stream);

cudaError_t launch_block_copy(void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                              const int32_t *pairs, int32_t num_pairs, int64_t num_blocks,
                              int n_kv, int d_h, int kind, int32_t *dev_status,
                              cudaStream_t stream);

} // namespace pa
