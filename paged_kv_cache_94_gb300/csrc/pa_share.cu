// Shared-prefix groups of a decode step.
//
// With prefix caching ("LLM 推理底层：KV Cache 显存几何、GQA/MLA 压缩与
// PagedAttention 调度", section "Prefix Caching 与 Copy-on-Write"), sequences
// that share a prompt prefix point at the same physical blocks. Attending a
// shared block once for all of its readers gives the same result as each
// reader attending it (softmax states merge exactly by log-sum-exp), with the
// readers' query rows filling the tensor cores' N side.
//
// This kernel finds the sharing from the block tables alone. With `sort`,
// the sequences are first ordered by a hash of their first min_blocks table
// entries (a sequence with fewer full blocks sorts last), ties by index, so
// that sequences sharing a prefix become neighbours wherever they sit in the
// batch; without it the order is the batch's own (sharers must then be
// adjacent). order[i] is the i-th sequence of that order. For each position
// i > 0, lcp[i] = the number of leading block-table entries of order[i]
// equal to those of order[i - 1], among blocks both sequences fill
// completely and excluding each sequence's last block (so every sequence
// keeps at least one block for the decode pass). Runs of neighbours with
// lcp >= min_blocks are cut into groups of at most gm members; a group
// shares S = the minimum lcp over its members after the first. Output:
//   skip[b]        S of b's group (0 if b is in no group of >= 2 members)
//   groups[3 s..]  (position of the first member in order, members, S) for
//                  groups s = 0 .. NG-1, then (0, 0, 0) up to s = B-1
//   order[i]       the sequences in that order: member j of group s is
//                  order[groups[3 s] + j]
// One CTA of 1024 threads; B <= 8192.
#include <atomic>

#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kThreads = 1024;
constexpr int kMaxPer = 8; // sequences per thread at most (B <= 8192)
constexpr int kMaxSeqs = kThreads * kMaxPer;
// dynamic shared memory: the sort keys (one 64-bit key per power-of-two slot)
constexpr size_t kSortBytes = (size_t)kMaxSeqs * 8;

__device__ __forceinline__ int32_t blocks_of(int32_t ctx, int32_t max_blocks)
{
    if (ctx <= 0 || (int64_t)ctx > (int64_t)max_blocks * 16)
        return 0;
    return (ctx + 15) / 16;
}

// Inclusive block-wide scan of kPer values per thread (op: add or max).
template <bool MAX, int kPer>
__device__ __forceinline__ void block_scan(int32_t (&v)[kPer], int32_t *wsum)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int i = 1; i < kPer; ++i)
        v[i] = MAX ? max(v[i], v[i - 1]) : v[i] + v[i - 1];
    int32_t x = v[kPer - 1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o)
            x = MAX ? max(x, y) : x + y;
    }
    if (lane == 31)
        wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t t = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o)
                t = MAX ? max(t, y) : t + y;
        }
        wsum[lane] = t;
    }
    __syncthreads();
    // exclusive carry into this thread: warps before, lanes before in the warp
    int32_t carry = warp ? wsum[warp - 1] : (MAX ? INT32_MIN : 0);
    const int32_t within = __shfl_up_sync(0xffffffffu, x, 1);
    if (lane > 0)
        carry = MAX ? max(carry, within) : carry + within;
    if (warp > 0 || lane > 0) {
#pragma unroll
        for (int i = 0; i < kPer; ++i)
            v[i] = MAX ? max(v[i], carry) : v[i] + carry;
    }
    __syncthreads();
}

// kPer sequences per thread: 1 up to 1024 sequences, else 8.
// Hash of the first N table entries of a row (FNV-1a over the entries; the
// N loads are issued together).
template <int N>
__device__ __forceinline__ uint32_t prefix_hash(const int32_t *row)
{
    int32_t e[N];
#pragma unroll
    for (int i = 0; i < N; ++i)
        e[i] = __ldg(row + i);
    uint32_t h = 2166136261u;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        h ^= (uint32_t)e[i];
        h *= 16777619u;
    }
    return h;
}

template <int kPer>
__global__ void __launch_bounds__(kThreads)
    share_detect_kernel(const int32_t *__restrict__ block_tables, int max_blocks,
                        const int32_t *__restrict__ context_lens, int B, int gm, int min_blocks,
                        int32_t *skip, int32_t *groups, int32_t *order_out, bool sort)
{
    extern __shared__ uint64_t key[]; // [N]: (hash << 32 | index), then lcp
    __shared__ int32_t ord[kThreads * kPer];
    __shared__ int32_t wsum[32];
    int32_t *lcp = reinterpret_cast<int32_t *>(key); // reuses the keys once sorted
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // the decode launch that reads these results may be scheduled now; it
    // waits for this grid to complete before its first read
    asm volatile("griddepcontrol.launch_dependents;");

    // ---- order: bitonic sort of N = 2^k >= B keys (padding sorts last), or
    // the batch's order
    int N = 1;
    while (N < B)
        N <<= 1;
    if (!sort)
        N = 0;
    for (int i = tid; i < N; i += kThreads) {
        uint64_t k = ~0ull;
        if (i < B) {
            const int32_t nb = blocks_of(__ldg(context_lens + i), max_blocks);
            const uint32_t h = nb > min_blocks
                                   ? prefix_hash<kShareMinBlocks>(block_tables +
                                                                  (size_t)i * max_blocks)
                                   : 0xFFFFFFFFu;
            k = ((uint64_t)h << 32) | (uint32_t)i;
        }
        key[i] = k;
    }
    __syncthreads();
    for (int size = 2; size <= N; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = tid; t < N / 2; t += kThreads) {
                const int i = 2 * t - (t & (stride - 1)); // lower index of the pair
                const int j = i + stride;
                const bool up = (i & size) == 0;
                const uint64_t a = key[i], c = key[j];
                if ((a > c) == up) {
                    key[i] = c;
                    key[j] = a;
                }
            }
            __syncthreads();
        }
    for (int i = tid; i < B; i += kThreads) {
        const int32_t b = sort ? (int32_t)(uint32_t)key[i] : i;
        ord[i] = b;
        order_out[i] = b;
    }
    __syncthreads();

    // ---- lcp with the previous sequence in that order: one warp per
    // position; each round compares 256 entries with all loads in flight
    constexpr int kRound = 8; // entries per lane per round
    for (int b = warp; b < B; b += kThreads / 32) {
        int32_t l = 0;
        if (b > 0) {
            const int32_t s0 = ord[b - 1], s1 = ord[b];
            const int32_t nb0 = blocks_of(__ldg(context_lens + s0), max_blocks);
            const int32_t nb1 = blocks_of(__ldg(context_lens + s1), max_blocks);
            const int32_t lim = max(0, min(nb0, nb1) - 1);
            const int32_t *r0 = block_tables + (size_t)s0 * max_blocks;
            const int32_t *r1 = block_tables + (size_t)s1 * max_blocks;
            for (int i0 = 0; i0 < lim; i0 += 32 * kRound) {
                int32_t a[kRound], c[kRound];
#pragma unroll
                for (int j = 0; j < kRound; ++j) {
                    const int i = i0 + 32 * j + lane;
                    a[j] = i < lim ? __ldg(r0 + i) : 0;
                    c[j] = i < lim ? __ldg(r1 + i) : 1;
                }
                uint32_t diff = 0;
                int j = 0;
                for (; j < kRound; ++j) {
                    diff = __ballot_sync(0xffffffffu, a[j] != c[j]);
                    if (diff)
                        break;
                }
                if (diff) {
                    l = i0 + 32 * j + __ffs(diff) - 1;
                    break;
                }
                l = min(i0 + 32 * kRound, lim);
            }
        }
        if (lane == 0)
            lcp[b] = l;
    }
    __syncthreads();

    // ---- run starts: b == 0 or lcp[b] < min_blocks; start[b] = last run start <= b
    int32_t st[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int b = tid * kPer + i;
        st[i] = (b < B && (b == 0 || lcp[b] < min_blocks)) ? b : INT32_MIN;
    }
    block_scan<true, kPer>(st, wsum);

    // ---- chunks of gm members per run: leaders own groups
    int32_t lead[kPer], cnt[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int b = tid * kPer + i;
        lead[i] = 0;
        cnt[i] = 0;
        if (b < B && (b - st[i]) % gm == 0) {
            int n = 1;
            int32_t S = INT32_MAX;
            while (n < gm && b + n < B && lcp[b + n] >= min_blocks) {
                S = min(S, lcp[b + n]);
                ++n;
            }
            lead[i] = n >= 2 ? S : 0;
            cnt[i] = n;
            for (int j = 0; j < n; ++j)
                skip[ord[b + j]] = n >= 2 ? S : 0;
        }
    }
    // ---- compact the groups of >= 2 members
    int32_t idx[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i)
        idx[i] = lead[i] > 0 ? 1 : 0;
    block_scan<false, kPer>(idx, wsum);
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int b = tid * kPer + i;
        if (b < B && lead[i] > 0) {
            const int s = idx[i] - 1;
            groups[3 * s] = b;
            groups[3 * s + 1] = cnt[i];
            groups[3 * s + 2] = lead[i];
        }
    }
    if (tid == kThreads - 1)
        wsum[0] = idx[kPer - 1]; // inclusive count at the last sequence slot
    __syncthreads();
    for (int s = wsum[0] + tid; s < B; s += kThreads) {
        groups[3 * s] = 0;
        groups[3 * s + 1] = 0;
        groups[3 * s + 2] = 0;
    }
}

} // namespace

cudaError_t launch_share_detect(const int32_t *block_tables, int max_blocks,
                                const int32_t *context_lens, int B, int gm, int min_blocks,
                                int32_t *skip, int32_t *groups, int32_t *order, bool sort,
                                cudaStream_t stream)
{
    if (B < 1 || B > kMaxSeqs || gm < 2 || min_blocks != kShareMinBlocks) // the hash's width
        return cudaErrorInvalidValue;
    size_t N = 1;
    while (N < (size_t)B)
        N <<= 1;
    const size_t smem = sort ? N * 8 : (size_t)B * 4; // keys, then lcp
    // the opt-in above 48 KiB of shared memory, once per device
    static std::atomic<bool> raised[kMaxDevices];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    if (!raised[dev].load()) {
        if (cudaFuncSetAttribute(share_detect_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSortBytes) != cudaSuccess ||
            cudaFuncSetAttribute(share_detect_kernel<kMaxPer>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kSortBytes) != cudaSuccess)
            return cudaErrorInvalidValue;
        raised[dev].store(true);
    }
    if (B <= kThreads)
        share_detect_kernel<1><<<1, kThreads, smem, stream>>>(
            block_tables, max_blocks, context_lens, B, gm, min_blocks, skip, groups, order,
            sort);
    else
        share_detect_kernel<kMaxPer><<<1, kThreads, smem, stream>>>(
            block_tables, max_blocks, context_lens, B, gm, min_blocks, skip, groups, order,
            sort);
    return cudaGetLastError();
}

} // namespace pa
