// Read-only probe of a decode's K/V access pattern.
//
// pa_kv_read_probe reads every K/V byte (and fp32 scale) that a decode of the
// same batch reads, through the same block tables, with plain 16-byte loads
// and no arithmetic besides an XOR that keeps the loads alive. Its time is
// the ceiling that the scattered pattern allows on this GPU, which a decode
// kernel's time can be compared with. A "read" is one physical block of one
// group of `hg` consecutive kv heads: hg = 1 reads the (block, head) tiles
// one at a time, hg = n_kv reads all heads of a block as one contiguous run
// (the pool layout [num_blocks][n_kv][16][d_h] keeps them adjacent).
//
// Work split: the reads of the batch lie on one line (sequence, then block,
// then head group); CTA c of G takes reads [c W / G, (c + 1) W / G), and its
// warps take every 8th read of that range, two at a time, each lane loading
// its share of the two reads' chunks before combining any of them.
#include <cuda_runtime.h>

#include "pa.h"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxSeqs = 8192;

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

struct ProbeArgs {
    const uint8_t *k_cache, *v_cache;
    const uint8_t *k_scale, *v_scale; // NULL for bf16 pools
    const int32_t *block_tables;
    const int32_t *context_lens;
    uint32_t *sink;
    int64_t num_blocks;
    int32_t max_blocks, num_seqs, n_kv, hg, tile_bytes;
};

// Address of 16-byte chunk c of a read whose first (block, head) row is
// `row` (= block * n_kv + first head): K tiles, V tiles, then the K and V
// scale rows.
__device__ __forceinline__ const uint8_t *chunk_addr(const ProbeArgs &a, int64_t row, int c,
                                                     int kc, int sc)
{
    if (c < kc)
        return a.k_cache + row * a.tile_bytes + 16 * (int64_t)c;
    c -= kc;
    if (c < kc)
        return a.v_cache + row * a.tile_bytes + 16 * (int64_t)c;
    c -= kc;
    if (c < sc)
        return a.k_scale + row * 64 + 16 * (int64_t)c;
    return a.v_scale + row * 64 + 16 * (int64_t)(c - sc);
}

__global__ void __launch_bounds__(kThreads) kv_read_probe_kernel(const ProbeArgs a)
{
    __shared__ int32_t P[kMaxSeqs + 1]; // reads before sequence b
    __shared__ int32_t part[kThreads];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int groups = a.n_kv / a.hg;
    // prefix of the reads per sequence: each thread sums a run of sequences
    const int per = (a.num_seqs + kThreads - 1) / kThreads;
    int32_t own = 0;
    for (int j = 0; j < per; ++j) {
        const int b = tid * per + j;
        if (b < a.num_seqs) {
            const int32_t ctx = a.context_lens[b];
            const int32_t nb = (ctx > 0 && ctx <= a.max_blocks * 16) ? (ctx + 15) / 16 : 0;
            own += nb * groups;
        }
    }
    part[tid] = own;
    __syncthreads();
    if (tid == 0) {
        int32_t run = 0;
        for (int t = 0; t < kThreads; ++t) {
            const int32_t x = part[t];
            part[t] = run;
            run += x;
        }
    }
    __syncthreads();
    int32_t run = part[tid];
    for (int j = 0; j < per; ++j) {
        const int b = tid * per + j;
        if (b < a.num_seqs) {
            P[b] = run;
            const int32_t ctx = a.context_lens[b];
            const int32_t nb = (ctx > 0 && ctx <= a.max_blocks * 16) ? (ctx + 15) / 16 : 0;
            run += nb * groups;
        }
    }
    if (tid == kThreads - 1)
        P[a.num_seqs] = part[kThreads - 1] + own;
    __syncthreads();
    const int64_t W = P[a.num_seqs];
    const int64_t lo = W * blockIdx.x / gridDim.x, hi = W * (blockIdx.x + 1) / gridDim.x;
    const int kc = a.hg * a.tile_bytes / 16;              // chunks of the K (or V) tiles
    const int sc = a.k_scale ? a.hg * 64 / 16 : 0;        // chunks of the K (or V) scales
    const int cpr = 2 * kc + 2 * sc;
    // read r -> first (block, head) row, or -1 for a bad block
    auto row_of = [&](int64_t r) -> int64_t {
        int l = 0, h = a.num_seqs;
        while (h - l > 1) {
            const int m = (l + h) >> 1;
            if (P[m] <= r)
                l = m;
            else
                h = m;
        }
        const int32_t off = (int32_t)(r - P[l]);
        const int32_t blk = off / groups, g = off - blk * groups;
        const int32_t phys = __ldg(a.block_tables + (int64_t)l * a.max_blocks + blk);
        if (phys < 0 || phys >= a.num_blocks)
            return -1;
        return (int64_t)phys * a.n_kv + (int64_t)g * a.hg;
    };
    uint32_t acc = 0;
    constexpr int kMaxPerLane = 8; // chunks per lane per read held in flight
    for (int64_t r = lo + warp; r < hi; r += 2 * kWarps) {
        const int64_t r2 = r + kWarps;
        const int64_t row0 = row_of(r), row1 = r2 < hi ? row_of(r2) : -1;
        for (int c0 = 0; c0 < cpr; c0 += 32 * kMaxPerLane) {
            uint4 v0[kMaxPerLane], v1[kMaxPerLane];
#pragma unroll
            for (int u = 0; u < kMaxPerLane; ++u) {
                const int c = c0 + lane + 32 * u;
                v0[u] = (row0 >= 0 && c < cpr) ? ld_stream(chunk_addr(a, row0, c, kc, sc))
                                               : make_uint4(0, 0, 0, 0);
                v1[u] = (row1 >= 0 && c < cpr) ? ld_stream(chunk_addr(a, row1, c, kc, sc))
                                               : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < kMaxPerLane; ++u)
                acc ^= v0[u].x ^ v0[u].y ^ v0[u].z ^ v0[u].w ^ v1[u].x ^ v1[u].y ^ v1[u].z ^
                       v1[u].w;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    __shared__ uint32_t wacc[kWarps];
    if (lane == 0)
        wacc[warp] = acc;
    __syncthreads();
    if (tid == 0) {
        uint32_t x = 0;
        for (int w = 0; w < kWarps; ++w)
            x ^= wacc[w];
        a.sink[blockIdx.x] = x;
    }
}

} // namespace
} // namespace pa

extern "C" pa_status pa_kv_read_probe(const void *k_cache, const void *v_cache,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *block_tables, int32_t max_blocks_per_seq,
                                      const int32_t *context_lens, int32_t num_seqs,
                                      int32_t heads_per_read, int32_t num_ctas, uint32_t *sink,
                                      pa_geom geom, void *stream)
{
    if (geom.reserved != 0 || geom.n_kv <= 0 || geom.num_blocks <= 0 || geom.block_size != 16 ||
        (geom.d_h != 64 && geom.d_h != 128))
        return PA_ERR_SHAPE;
    if (geom.kv_dtype != PA_KV_BF16 && geom.kv_dtype != PA_KV_INT8 && geom.kv_dtype != PA_KV_INT4)
        return PA_ERR_DTYPE;
    if (num_seqs < 0 || num_seqs > pa::kMaxSeqs || max_blocks_per_seq <= 0 || num_ctas <= 0 ||
        heads_per_read <= 0 || geom.n_kv % heads_per_read != 0)
        return PA_ERR_SHAPE;
    if (num_seqs == 0)
        return PA_OK;
    if (!k_cache || !v_cache || !block_tables || !context_lens || !sink)
        return PA_ERR_NULL;
    const bool quant = geom.kv_dtype != PA_KV_BF16;
    if (quant != (k_scale != nullptr) || quant != (v_scale != nullptr))
        return PA_ERR_SHAPE;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache) |
                          reinterpret_cast<uintptr_t>(k_scale) | reinterpret_cast<uintptr_t>(v_scale);
    if (mis & 15)
        return PA_ERR_ALIGNMENT;
    pa::ProbeArgs a;
    a.k_cache = static_cast<const uint8_t *>(k_cache);
    a.v_cache = static_cast<const uint8_t *>(v_cache);
    a.k_scale = reinterpret_cast<const uint8_t *>(k_scale);
    a.v_scale = reinterpret_cast<const uint8_t *>(v_scale);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.sink = sink;
    a.num_blocks = geom.num_blocks;
    a.max_blocks = max_blocks_per_seq;
    a.num_seqs = num_seqs;
    a.n_kv = geom.n_kv;
    a.hg = heads_per_read;
    a.tile_bytes = 16 * geom.d_h * (geom.kv_dtype == PA_KV_BF16 ? 2 : 1) /
                   (geom.kv_dtype == PA_KV_INT4 ? 2 : 1);
    pa::kv_read_probe_kernel<<<num_ctas, pa::kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
