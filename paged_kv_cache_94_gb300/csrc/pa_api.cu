// C ABI of libpa.so: argument checks, tensor maps, grid sizing and launches.
// Every function here runs on the host and only enqueues work.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "pa.h"
#include "pa_decode.cuh"
#include "pa_internal.h"

namespace {

// An NVTX range around each entry point (named after it), so that a
// profiler's timeline shows the library's calls; free when no tool listens.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};


using pa::DecodeKernel;
using pa::DecodeParams;

constexpr int kMaxSeqs = 8192;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int group_of(const pa_geom &g) { return g.n_h / g.n_kv; }

pa_status check_geom(const pa_geom &g)
{
    if (g.reserved != 0)
        return PA_ERR_SHAPE;
    if (g.kv_dtype != PA_KV_BF16 && g.kv_dtype != PA_KV_INT8 && g.kv_dtype != PA_KV_INT4)
        return PA_ERR_DTYPE;
    if (g.n_h <= 0 || g.n_kv <= 0 || g.n_h % g.n_kv != 0 || g.num_blocks <= 0)
        return PA_ERR_SHAPE;
    if (g.block_size != 16 || (g.d_h != 64 && g.d_h != 128))
        return PA_ERR_UNSUPPORTED;
    const int gq = group_of(g);
    if (gq != 1 && gq != 2 && gq != 4 && gq != 8 && gq != 16)
        return PA_ERR_UNSUPPORTED;
    // TMA row coordinates (block * n_kv + head) * 16 must fit in int32
    if (g.num_blocks * (int64_t)g.n_kv * 16 >= (int64_t(1) << 31))
        return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

const DecodeKernel *kernel_for(const pa_geom &g, int nq = 1)
{
    const int gq = group_of(g);
    if (nq != 1)
        return g.kv_dtype == PA_KV_INT8   ? pa::find_decode_kernel_int8_mq(g.d_h, gq, nq)
               : g.kv_dtype == PA_KV_INT4 ? pa::find_decode_kernel_int4_mq(g.d_h, gq, nq)
                                          : pa::find_decode_kernel_bf16_mq(g.d_h, gq, nq);
    return g.kv_dtype == PA_KV_INT8   ? pa::find_decode_kernel_int8(g.d_h, gq)
           : g.kv_dtype == PA_KV_INT4 ? pa::find_decode_kernel_int4(g.d_h, gq)
                                      : pa::find_decode_kernel_bf16(g.d_h, gq);
}

// --------------------------------------------------------------- device info
struct DeviceInfo {
    int sms = 0;
};

DeviceInfo g_dev[64];
std::mutex g_mu;

pa_status current_device(int &dev, int &sms)
{
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_dev[dev].sms == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return PA_ERR_CUDA;
        g_dev[dev].sms = n;
    }
    sms = g_dev[dev].sms;
    return PA_OK;
}

// Resident CTAs per SM of a kernel at a given shared-memory size on the
// current device. The kernel's dynamic shared-memory limit is raised once per
// (kernel, device) to the device maximum; results are cached per (kernel,
// device, size), so steady-state calls make no CUDA runtime queries.
struct OccEntry {
    const void *fn;
    int dev;
    size_t smem;
    int per_sm;
};
constexpr int kOccCache = 64;
OccEntry g_occ[kOccCache];
int g_occ_n = 0;
struct AttrEntry {
    const void *fn;
    int dev;
};
AttrEntry g_attr[kOccCache];
int g_attr_n = 0;

pa_status ctas_per_sm(const DecodeKernel *kd, size_t smem, int &n)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    for (int i = 0; i < g_occ_n; ++i)
        if (g_occ[i].fn == kd->fn && g_occ[i].dev == dev && g_occ[i].smem == smem) {
            n = g_occ[i].per_sm;
            return n > 0 ? PA_OK : PA_ERR_UNSUPPORTED;
        }
    bool attr_set = false;
    for (int i = 0; i < g_attr_n; ++i)
        attr_set |= (g_attr[i].fn == kd->fn && g_attr[i].dev == dev);
    if (!attr_set) {
        int max_optin = 0;
        if (cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess ||
            cudaFuncSetAttribute(kd->fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_optin) !=
                cudaSuccess)
            return PA_ERR_CUDA;
        if (g_attr_n < kOccCache)
            g_attr[g_attr_n++] = {kd->fn, dev};
    }
    n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kd->fn, kd->threads, smem) != cudaSuccess)
        return PA_ERR_CUDA;
    g_occ[g_occ_n < kOccCache ? g_occ_n++ : (int)(smem % kOccCache)] = {kd->fn, dev, smem, n};
    if (n <= 0)
        return PA_ERR_UNSUPPORTED; // does not fit on an SM
    return PA_OK;
}

pa_status default_ctas(const pa_geom &g, int num_seqs, int &grid, int nq = 1)
{
    const DecodeKernel *kd = kernel_for(g, nq);
    if (!kd)
        return PA_ERR_UNSUPPORTED;
    int dev, sms, per;
    pa_status st = current_device(dev, sms);
    if (st != PA_OK)
        return st;
    st = ctas_per_sm(kd, kd->smem_bytes(num_seqs), per);
    if (st != PA_OK)
        return st;
    grid = sms * per;
    return PA_OK;
}

size_t counters_bytes(int64_t units) { return (size_t)((units * 4 + 255) / 256 * 256); }

size_t workspace_bytes_for(const pa_geom &g, int num_seqs, int grid, int nq = 1)
{
    const int64_t units = (int64_t)num_seqs * g.n_kv;
    const int64_t rec = (int64_t)group_of(g) * nq * (g.d_h + 2) * 4;
    return counters_bytes(units) + (size_t)((grid + units) * rec);
}

// Shared-prefix decode (one launch over 2B "sequences": B group units, then
// B sequences' remaining blocks). Workspace:
//   counters  [2B * n_kv] int32 (zero on entry and on exit)
//   records   (grid + 2B * n_kv) x (g * members) x (d_h + 2) fp32
//   skip[B], groups[3B], order[B] int32, pre[B][n_h][d_h + 2] fp32
struct ShareLayout {
    size_t zero_end, records, skip, groups, order, pre, end;
};

size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// Shared memory and resident CTAs per SM of the shared-prefix kernel for a
// batch (its 2 * num_seqs units' prefix arrays grow with the batch);
// PA_ERR_UNSUPPORTED when not even one CTA fits on an SM.
pa_status share_fits(const DecodeKernel *kp, int num_seqs, size_t &smem, int &per)
{
    smem = kp->smem_bytes(2 * num_seqs);
    int dev = -1, max_optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
            cudaSuccess)
        return PA_ERR_CUDA;
    if (smem > (size_t)max_optin)
        return PA_ERR_UNSUPPORTED;
    return ctas_per_sm(kp, smem, per);
}

ShareLayout share_layout(const pa_geom &g, int num_seqs, int grid)
{
    ShareLayout L;
    const size_t units2 = 2 * (size_t)num_seqs * g.n_kv;
    L.zero_end = round256(4 * units2);
    L.records = L.zero_end;
    const size_t rec = (size_t)group_of(g) * pa::kShareMembers(group_of(g)) * (g.d_h + 2) * 4;
    L.skip = round256(L.records + (grid + units2) * rec);
    L.groups = L.skip + round256(4 * (size_t)num_seqs);
    L.order = L.groups + round256(12 * (size_t)num_seqs);
    L.pre = L.order + round256(4 * (size_t)num_seqs);
    L.end = L.pre + (size_t)num_seqs * g.n_h * (g.d_h + 2) * 4;
    return L;
}

// ---------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D view of a pool: one row per (block, head, offset); a box is one 16-row
// tile of at most 128 bytes per row. bf16 and INT8 tiles are swizzled so that
// ldmatrix/ld.shared of 8 consecutive rows hit distinct banks; INT4 rows (64
// or 32 bytes) are read as whole contiguous runs and stay unswizzled.
pa_status encode_pool_uncached(CUtensorMap &m, const void *base, const pa_geom &g)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return PA_ERR_CUDA;
    const bool bf16 = g.kv_dtype == PA_KV_BF16, i4 = g.kv_dtype == PA_KV_INT4;
    const int row_elems = i4 ? g.d_h / 2 : g.d_h; // bytes for INT8/INT4, elements for bf16
    const int esz = bf16 ? 2 : 1;
    const cuuint64_t dims[2] = {(cuuint64_t)row_elems, (cuuint64_t)(g.num_blocks * g.n_kv * 16)};
    const cuuint64_t strides[1] = {(cuuint64_t)row_elems * esz};
    const cuuint32_t box_x = (cuuint32_t)((row_elems * esz > 128) ? 128 / esz : row_elems);
    const cuuint32_t box[2] = {box_x, 16};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = i4                     ? CU_TENSOR_MAP_SWIZZLE_NONE
                                  : (box_x * esz == 128) ? CU_TENSOR_MAP_SWIZZLE_128B
                                                         : CU_TENSOR_MAP_SWIZZLE_64B;
    const CUresult r =
        fn(&m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
           const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// Encoded maps are cached by (pool address, geometry): a decode step reuses
// the same pools call after call. A map only describes the pool's address and
// shape, so a hit is exact.
struct MapEntry {
    const void *base;
    int64_t num_blocks;
    int32_t n_kv, d_h, kv_dtype;
    CUtensorMap map;
};
constexpr int kMapCache = 64;
MapEntry g_maps[kMapCache];
int g_maps_n = 0, g_maps_next = 0;

pa_status encode_pool(CUtensorMap &m, const void *base, const pa_geom &g)
{
    {
        std::lock_guard<std::mutex> lk(g_mu);
        for (int i = 0; i < g_maps_n; ++i) {
            const MapEntry &e = g_maps[i];
            if (e.base == base && e.num_blocks == g.num_blocks && e.n_kv == g.n_kv &&
                e.d_h == g.d_h && e.kv_dtype == g.kv_dtype) {
                m = e.map;
                return PA_OK;
            }
        }
    }
    const pa_status st = encode_pool_uncached(m, base, g);
    if (st != PA_OK)
        return st;
    std::lock_guard<std::mutex> lk(g_mu);
    MapEntry &e = g_maps[g_maps_next];
    e = {base, g.num_blocks, g.n_kv, g.d_h, g.kv_dtype, m};
    g_maps_next = (g_maps_next + 1) % kMapCache;
    if (g_maps_n < kMapCache)
        ++g_maps_n;
    return PA_OK;
}

pa_status decode_impl(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                      const float *v_scale, const int32_t *block_tables, int32_t max_blocks,
                      const int32_t *context_lens, int32_t num_seqs, float scale, void *out,
                      void *workspace, size_t workspace_bytes, pa_geom g, int32_t *dev_status,
                      void *stream, int32_t num_ctas, const pa_decode_opts *opts = nullptr,
                      int nq = 1)
{
    pa_status st = check_geom(g);
    if (st != PA_OK)
        return st;
    const pa_decode_opts none = {0, 0, nullptr, nullptr, 0, 0, 0};
    const pa_decode_opts &o = opts ? *opts : none;
    if (o.window < 0 || o.n_sink < 0 || o.n_sink > 16 || o.reserved != 0 ||
        (o.share_prefix < 0 || o.share_prefix > 2))
        return PA_ERR_SHAPE;
    bool share = o.share_prefix != 0;
    if (share && (nq != 1 || o.window != 0 || o.n_sink != 0 || group_of(g) > 8))
        return PA_ERR_UNSUPPORTED;
    if (o.n_sink > 0) {
        if (g.kv_dtype == PA_KV_BF16)
            return PA_ERR_SHAPE;
        if (!o.sink_k || !o.sink_v)
            return PA_ERR_NULL;
        if (!aligned(o.sink_k, 2) || !aligned(o.sink_v, 2))
            return PA_ERR_ALIGNMENT;
    }
    if (num_seqs < 0 || num_seqs > kMaxSeqs || max_blocks <= 0 || num_ctas < 0)
        return PA_ERR_SHAPE;
    if ((int64_t)num_seqs * max_blocks >= (int64_t(1) << 31))
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0)
        return PA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace)
        return !workspace ? PA_ERR_WORKSPACE : PA_ERR_NULL;
    const bool i8 = g.kv_dtype != PA_KV_BF16; // INT8 or INT4: fp32 scales
    if (i8 && (!k_scale || !v_scale))
        return PA_ERR_NULL;
    if (!i8 && (k_scale || v_scale))
        return PA_ERR_SHAPE;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(workspace, 256) || (i8 && (!aligned(k_scale, 16) || !aligned(v_scale, 16))))
        return PA_ERR_ALIGNMENT;

    const DecodeKernel *kd = kernel_for(g, nq);
    if (!kd)
        return PA_ERR_UNSUPPORTED;
    int dev, sms, per;
    if ((st = current_device(dev, sms)) != PA_OK)
        return st;
    const size_t smem = kd->smem_bytes(num_seqs);
    if ((st = ctas_per_sm(kd, smem, per)) != PA_OK)
        return st;
    int grid = num_ctas > 0 ? num_ctas : sms * per;
    const DecodeKernel *kp = share ? pa::find_prefix_kernel(g.kv_dtype, g.d_h, group_of(g)) : nullptr;
    if (share && !kp)
        return PA_ERR_UNSUPPORTED;
    size_t smem_sh = 0;
    int per_sh = 0;
    if (share && (st = share_fits(kp, num_seqs, smem_sh, per_sh)) != PA_OK) {
        if (st != PA_ERR_UNSUPPORTED)
            return st;
        share = false; // the batch's prefix arrays do not fit: decode without sharing
    }
    if (share) // default: one wave of resident CTAs
        grid = num_ctas > 0 ? num_ctas : sms * per_sh;
    const ShareLayout SL = share ? share_layout(g, num_seqs, grid) : ShareLayout{};
    if (workspace_bytes < (share ? SL.end : workspace_bytes_for(g, num_seqs, grid, nq)))
        return PA_ERR_WORKSPACE;

    CUtensorMap tk, tv;
    if ((st = encode_pool(tk, k_cache, g)) != PA_OK || (st = encode_pool(tv, v_cache, g)) != PA_OK)
        return st;

    DecodeParams p;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = static_cast<__nv_bfloat16 *>(out);
    const int64_t units = (int64_t)num_seqs * g.n_kv;
    p.counters = static_cast<int32_t *>(workspace);
    p.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + counters_bytes(units));
    p.dev_status = dev_status;
    p.num_blocks = g.num_blocks;
    p.num_seqs = num_seqs;
    p.n_kv = g.n_kv;
    p.max_blocks = max_blocks;
    p.num_ctas = grid;
    p.scale_log2 = (float)((double)scale * 1.4426950408889634);
    p.window = o.window;
    p.n_sink = o.n_sink;
    p.sink_k = static_cast<const __nv_bfloat16 *>(o.n_sink > 0 ? o.sink_k : nullptr);
    p.sink_v = static_cast<const __nv_bfloat16 *>(o.n_sink > 0 ? o.sink_v : nullptr);
    p.g = group_of(g);
    p.seg_cost = pa::kSegCost;
    p.seg_cost_lead = pa::kSegCost;
    p.lead_units = 0;
    p.skip = nullptr;
    p.pre = nullptr;
    p.groups = nullptr;
    p.members = nullptr;
    const cudaStream_t cs = static_cast<cudaStream_t>(stream);
    p.num_real = num_seqs;
    p.grid_fixed = num_ctas > 0 ? 1 : 0;
    if (share) {
        // 1) groups of sequences sharing leading blocks; 2) one
        //    launch over the group units, then every sequence's remaining
        //    blocks; the last arrival on each sequence merges its records and
        //    its group's prefix state
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        int32_t *skip = reinterpret_cast<int32_t *>(ws + SL.skip);
        int32_t *groups = reinterpret_cast<int32_t *>(ws + SL.groups);
        int32_t *order = reinterpret_cast<int32_t *>(ws + SL.order);
        cudaError_t e = pa::launch_share_detect(block_tables, max_blocks, context_lens, num_seqs,
                                                pa::kShareMembers(p.g), pa::kShareMinBlocks, skip,
                                                groups, order, o.share_prefix == 2, cs);
        if (e != cudaSuccess)
            return PA_ERR_CUDA;
        p.num_seqs = 2 * num_seqs;
        p.seg_cost = pa::kShareSegCost; // every unit ends in records and a merge
        p.seg_cost_lead = pa::kShareGroupSegCost;
        p.lead_units = num_seqs;
        p.counters = reinterpret_cast<int32_t *>(ws);
        p.partials = reinterpret_cast<float *>(ws + SL.records);
        p.skip = skip;
        p.groups = groups;
        p.members = order;
        p.pre = reinterpret_cast<float *>(ws + SL.pre);
        p.num_ctas = grid;
        return kp->launch(tk, tv, p, grid, smem_sh, cs) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    const cudaError_t e = kd->launch(tk, tv, p, grid, smem, cs);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

} // namespace

namespace pa {
const DecodeKernel *find_decode_kernel_bf16_d64(int group);
const DecodeKernel *find_decode_kernel_bf16_d128(int group);
const DecodeKernel *find_decode_kernel_int8_d64(int group);
const DecodeKernel *find_decode_kernel_int8_d128(int group);

const DecodeKernel *find_decode_kernel_bf16(int d_h, int group)
{
    return d_h == 128 ? find_decode_kernel_bf16_d128(group)
                      : d_h == 64 ? find_decode_kernel_bf16_d64(group) : nullptr;
}

const DecodeKernel *find_decode_kernel_int4_d64(int group);
const DecodeKernel *find_decode_kernel_int4_d128(int group);
const DecodeKernel *find_prefix_kernel_bf16_d128(int group);
const DecodeKernel *find_prefix_kernel_bf16_d64(int group);
const DecodeKernel *find_prefix_kernel_int8_d128(int group);
const DecodeKernel *find_prefix_kernel_int8_d64(int group);
const DecodeKernel *find_prefix_kernel_int4_d128(int group);
const DecodeKernel *find_prefix_kernel_int4_d64(int group);

const DecodeKernel *find_prefix_kernel(int kv_dtype, int d_h, int group)
{
    if (d_h != 128 && d_h != 64)
        return nullptr;
    const bool big = d_h == 128;
    switch (kv_dtype) {
    case PA_KV_BF16: return big ? find_prefix_kernel_bf16_d128(group) : find_prefix_kernel_bf16_d64(group);
    case PA_KV_INT8: return big ? find_prefix_kernel_int8_d128(group) : find_prefix_kernel_int8_d64(group);
    case PA_KV_INT4: return big ? find_prefix_kernel_int4_d128(group) : find_prefix_kernel_int4_d64(group);
    default: return nullptr;
    }
}

const DecodeKernel *find_decode_kernel_int4(int d_h, int group)
{
    return d_h == 128 ? find_decode_kernel_int4_d128(group)
                      : d_h == 64 ? find_decode_kernel_int4_d64(group) : nullptr;
}

const DecodeKernel *find_decode_kernel_int8_mq_d128(int group, int nq);
const DecodeKernel *find_decode_kernel_int8_mq_d64(int group, int nq);
const DecodeKernel *find_decode_kernel_int4_mq_d128(int group, int nq);
const DecodeKernel *find_decode_kernel_int4_mq_d64(int group, int nq);

const DecodeKernel *find_decode_kernel_int8_mq(int d_h, int group, int nq)
{
    return d_h == 128 ? find_decode_kernel_int8_mq_d128(group, nq)
                      : d_h == 64 ? find_decode_kernel_int8_mq_d64(group, nq) : nullptr;
}

const DecodeKernel *find_decode_kernel_int4_mq(int d_h, int group, int nq)
{
    return d_h == 128 ? find_decode_kernel_int4_mq_d128(group, nq)
                      : d_h == 64 ? find_decode_kernel_int4_mq_d64(group, nq) : nullptr;
}

const DecodeKernel *find_decode_kernel_int8(int d_h, int group)
{
    return d_h == 128 ? find_decode_kernel_int8_d128(group)
                      : d_h == 64 ? find_decode_kernel_int8_d64(group) : nullptr;
}
} // namespace pa

extern "C" {

pa_status pa_cache_write(const void *k, const void *v, const int64_t *slot_mapping,
                         int64_t num_tokens, void *k_cache, void *v_cache, float *k_scale,
                         float *v_scale, pa_geom geom, int32_t *dev_status, void *stream)
{
    const NvtxRange range("pa_cache_write");
    pa_status st = check_geom(geom);
    if (st != PA_OK)
        return st;
    if (num_tokens < 0)
        return PA_ERR_SHAPE;
    if (num_tokens == 0)
        return PA_OK;
    if (num_tokens * geom.n_kv > (int64_t(1) << 33))
        return PA_ERR_UNSUPPORTED;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache)
        return PA_ERR_NULL;
    const bool i8 = geom.kv_dtype != PA_KV_BF16; // INT8 or INT4: fp32 scales
    if (i8 && (!k_scale || !v_scale))
        return PA_ERR_NULL;
    if (!i8 && (k_scale || v_scale))
        return PA_ERR_SHAPE;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8) || (i8 && (!aligned(k_scale, 4) || !aligned(v_scale, 4))))
        return PA_ERR_ALIGNMENT;
    const cudaError_t e = pa::launch_cache_write(
        k, v, slot_mapping, num_tokens, geom.n_kv, geom.d_h, geom.kv_dtype, geom.num_blocks * 16,
        k_cache,
        v_cache, k_scale, v_scale, dev_status, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_block_copy(void *k_cache, void *v_cache, float *k_scale, float *v_scale,
                        const int32_t *pairs, int32_t num_pairs, pa_geom geom,
                        int32_t *dev_status, void *stream)
{
    const NvtxRange range("pa_block_copy");
    pa_status st = check_geom(geom);
    if (st != PA_OK)
        return st;
    if (num_pairs < 0)
        return PA_ERR_SHAPE;
    if (num_pairs == 0)
        return PA_OK;
    if (!k_cache || !v_cache || !pairs)
        return PA_ERR_NULL;
    const bool i8 = geom.kv_dtype != PA_KV_BF16; // INT8 or INT4: fp32 scales
    if (i8 && (!k_scale || !v_scale))
        return PA_ERR_NULL;
    if (!i8 && (k_scale || v_scale))
        return PA_ERR_SHAPE;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(pairs, 4) ||
        (i8 && (!aligned(k_scale, 16) || !aligned(v_scale, 16))))
        return PA_ERR_ALIGNMENT;
    const cudaError_t e = pa::launch_block_copy(k_cache, v_cache, k_scale, v_scale, pairs,
                                                num_pairs, geom.num_blocks, geom.n_kv, geom.d_h,
                                                geom.kv_dtype, dev_status,
                                                static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_decode_workspace_size(pa_geom geom, int32_t num_seqs, int32_t num_ctas)
{
    if (check_geom(geom) != PA_OK || num_seqs < 0 || num_seqs > kMaxSeqs || num_ctas < 0)
        return 0;
    int grid = num_ctas;
    if (grid == 0 && default_ctas(geom, num_seqs, grid) != PA_OK)
        return 0;
    return workspace_bytes_for(geom, num_seqs, grid);
}

pa_status pa_decode_workspace_init(void *workspace, size_t workspace_bytes, void *stream)
{
    if (!workspace)
        return PA_ERR_WORKSPACE;
    return cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

pa_status pa_decode(const void *q, const void *k_cache, const void *v_cache, const float *k_scale,
                    const float *v_scale, const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *context_lens, int32_t num_seqs, float scale, void *out,
                    void *workspace, size_t workspace_bytes, pa_geom geom, int32_t *dev_status,
                    void *stream)
{
    const NvtxRange range("pa_decode");
    return decode_impl(q, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, scale, out, workspace, workspace_bytes, geom,
                       dev_status, stream, 0);
}

pa_status pa_decode_ex(const void *q, const void *k_cache, const void *v_cache,
                       const float *k_scale, const float *v_scale, const int32_t *block_tables,
                       int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                       float scale, void *out, void *workspace, size_t workspace_bytes,
                       pa_geom geom, int32_t *dev_status, void *stream, int32_t num_ctas)
{
    const NvtxRange range("pa_decode_ex");
    if (num_ctas <= 0)
        return PA_ERR_SHAPE;
    return decode_impl(q, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, scale, out, workspace, workspace_bytes, geom,
                       dev_status, stream, num_ctas);
}

size_t pa_decode_opt_workspace_size(pa_geom geom, int32_t num_seqs, const pa_decode_opts *opts)
{
    if (check_geom(geom) != PA_OK || num_seqs < 0 || num_seqs > kMaxSeqs)
        return 0;
    const int num_ctas = opts ? opts->num_ctas : 0;
    if (num_ctas < 0)
        return 0;
    int grid = num_ctas;
    if (grid == 0 && default_ctas(geom, num_seqs, grid) != PA_OK)
        return 0;
    if (!opts || opts->share_prefix == 0)
        return workspace_bytes_for(geom, num_seqs, grid);
    const DecodeKernel *kp = pa::find_prefix_kernel(geom.kv_dtype, geom.d_h, group_of(geom));
    int dev, sms, per;
    size_t smem;
    if (!kp || current_device(dev, sms) != PA_OK)
        return 0;
    const pa_status st = share_fits(kp, num_seqs, smem, per);
    if (st == PA_ERR_UNSUPPORTED) // decoded without sharing
        return workspace_bytes_for(geom, num_seqs, grid);
    if (st != PA_OK)
        return 0;
    return share_layout(geom, num_seqs, num_ctas > 0 ? num_ctas : sms * per).end;
}

pa_status pa_decode_opt(const void *q, const void *k_cache, const void *v_cache,
                        const float *k_scale, const float *v_scale, const int32_t *block_tables,
                        int32_t max_blocks_per_seq, const int32_t *context_lens,
                        int32_t num_seqs, float scale, void *out, void *workspace,
                        size_t workspace_bytes, pa_geom geom, const pa_decode_opts *opts,
                        int32_t *dev_status, void *stream)
{
    const NvtxRange range("pa_decode_opt");
    return decode_impl(q, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, scale, out, workspace, workspace_bytes, geom,
                       dev_status, stream, opts ? opts->num_ctas : 0, opts);
}

size_t pa_decode_mq_workspace_size(pa_geom geom, int32_t num_seqs, int32_t n_q,
                                   int32_t num_ctas)
{
    if (check_geom(geom) != PA_OK || num_seqs < 0 || num_seqs > kMaxSeqs || num_ctas < 0 ||
        n_q < 1 || !kernel_for(geom, n_q))
        return 0;
    int grid = num_ctas;
    if (grid == 0 && default_ctas(geom, num_seqs, grid, n_q) != PA_OK)
        return 0;
    return workspace_bytes_for(geom, num_seqs, grid, n_q);
}

pa_status pa_decode_mq(const void *q, const void *k_cache, const void *v_cache,
                       const float *k_scale, const float *v_scale, const int32_t *block_tables,
                       int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                       int32_t n_q, float scale, void *out, void *workspace,
                       size_t workspace_bytes, pa_geom geom, int32_t *dev_status, void *stream)
{
    const NvtxRange range("pa_decode_mq");
    if (n_q < 1)
        return PA_ERR_SHAPE;
    return decode_impl(q, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, scale, out, workspace, workspace_bytes, geom,
                       dev_status, stream, 0, nullptr, n_q);
}

pa_status pa_decode_mq_ex(const void *q, const void *k_cache, const void *v_cache,
                          const float *k_scale, const float *v_scale,
                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *context_lens, int32_t num_seqs, int32_t n_q,
                          float scale, void *out, void *workspace, size_t workspace_bytes,
                          pa_geom geom, int32_t *dev_status, void *stream, int32_t num_ctas)
{
    const NvtxRange range("pa_decode_mq_ex");
    if (n_q < 1 || num_ctas <= 0)
        return PA_ERR_SHAPE;
    return decode_impl(q, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, scale, out, workspace, workspace_bytes, geom,
                       dev_status, stream, num_ctas, nullptr, n_q);
}

pa_status pa_sink_write(const void *k, const void *v, const int32_t *seq_rows,
                        const int32_t *positions, int64_t num_tokens, void *sink_k, void *sink_v,
                        int32_t n_sink, int32_t num_seqs, pa_geom geom, void *stream)
{
    const NvtxRange range("pa_sink_write");
    pa_status st = check_geom(geom);
    if (st != PA_OK)
        return st;
    if (num_tokens < 0 || n_sink < 1 || n_sink > 16 || num_seqs < 1)
        return PA_ERR_SHAPE;
    if (num_tokens == 0)
        return PA_OK;
    if (num_tokens * geom.n_kv > (int64_t(1) << 33))
        return PA_ERR_UNSUPPORTED;
    if (!k || !v || !seq_rows || !positions || !sink_k || !sink_v)
        return PA_ERR_NULL;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(sink_k, 16) || !aligned(sink_v, 16) ||
        !aligned(seq_rows, 4) || !aligned(positions, 4))
        return PA_ERR_ALIGNMENT;
    const cudaError_t e = pa::launch_sink_write(
        k, v, seq_rows, positions, num_tokens, geom.n_kv, geom.d_h, n_sink, num_seqs, sink_k,
        sink_v, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_share_groups(const int32_t *block_tables, int32_t max_blocks_per_seq,
                          const int32_t *context_lens, int32_t num_seqs, int32_t g,
                          int32_t mode, int32_t *skip, int32_t *groups, int32_t *order,
                          void *stream)
{
    const NvtxRange range("pa_share_groups");
    if (num_seqs < 0 || num_seqs > kMaxSeqs || max_blocks_per_seq <= 0 || mode < 1 || mode > 2)
        return PA_ERR_SHAPE;
    if (g != 1 && g != 2 && g != 4 && g != 8)
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0)
        return PA_OK;
    if (!block_tables || !context_lens || !skip || !groups || !order)
        return PA_ERR_NULL;
    return pa::launch_share_detect(block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                   pa::kShareMembers(g), pa::kShareMinBlocks, skip, groups,
                                   order, mode == 2, static_cast<cudaStream_t>(stream)) ==
                       cudaSuccess
               ? PA_OK
               : PA_ERR_CUDA;
}

int32_t pa_decode_default_ctas(pa_geom geom, int32_t num_seqs)
{
    pa_status st = check_geom(geom);
    if (st != PA_OK)
        return st;
    if (num_seqs < 0 || num_seqs > kMaxSeqs)
        return PA_ERR_SHAPE;
    int grid = 0;
    st = default_ctas(geom, num_seqs, grid);
    return st != PA_OK ? st : grid;
}

int32_t pa_plan_owner(int64_t item, int64_t total_items, int32_t num_ctas)
{
    if (total_items <= 0 || num_ctas <= 0 || item < 0 || item >= total_items)
        return -1;
    return (int32_t)pa::plan_owner(item, total_items, pa::plan_ctas(num_ctas, total_items));
}

const char *pa_status_string(pa_status s)
{
    switch (s) {
    case PA_OK: return "PA_OK";
    case PA_ERR_NULL: return "PA_ERR_NULL: a required pointer is NULL";
    case PA_ERR_SHAPE: return "PA_ERR_SHAPE: a size or argument combination is invalid";
    case PA_ERR_DTYPE: return "PA_ERR_DTYPE: unknown kv_dtype";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: geometry not supported";
    case PA_ERR_BAD_BLOCK: return "PA_ERR_BAD_BLOCK: block table entry outside the pool";
    case PA_ERR_BAD_SLOT: return "PA_ERR_BAD_SLOT: slot outside the pool";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: a CUDA call failed";
    case PA_ERR_BAD_CONTEXT: return "PA_ERR_BAD_CONTEXT: context length outside the block table";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT: a pipeline wait gave up";
    case PA_ERR_ALIGNMENT: return "PA_ERR_ALIGNMENT: a pointer is not aligned as required";
    case PA_ERR_OUT_OF_BLOCKS: return "PA_ERR_OUT_OF_BLOCKS: not enough free KV cache blocks";
    case PA_ERR_STATE: return "PA_ERR_STATE: a block table names a block that is not held";
    }
    return "unknown pa_status";
}

pa_status pa_status_from_device(int32_t w)
{
    if (w & PA_DEV_BAD_BLOCK)
        return PA_ERR_BAD_BLOCK;
    if (w & PA_DEV_BAD_SLOT)
        return PA_ERR_BAD_SLOT;
    if (w & PA_DEV_BAD_CONTEXT)
        return PA_ERR_BAD_CONTEXT;
    if (w & PA_DEV_TIMEOUT)
        return PA_ERR_TIMEOUT;
    return PA_OK;
}

int32_t pa_version(void) { return 100; }

pa_status pa_wait_selftest(int32_t *dev_status, int32_t limit_us, void *stream)
{
    if (!dev_status)
        return PA_ERR_NULL;
    if (limit_us < 1 || limit_us > 1000000)
        return PA_ERR_SHAPE;
    const cudaError_t e = pa::launch_wait_selftest(dev_status, (uint64_t)limit_us * 1000u,
                                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

} // extern "C"

namespace pa {
// pa_decode_ex's body with a caller-chosen workspace, for entry points in
// other translation units (num_ctas = 0: the default grid).
pa_status decode_with_workspace(const void *q, const void *k_cache, const void *v_cache,
                                const float *k_scale, const float *v_scale,
                                const int32_t *block_tables, int32_t max_blocks,
                                const int32_t *context_lens, int32_t num_seqs, float scale,
                                void *out, void *workspace, size_t workspace_bytes, pa_geom g,
                                int32_t *dev_status, void *stream)
{
    return decode_impl(q, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks,
                       context_lens, num_seqs, scale, out, workspace, workspace_bytes, g,
                       dev_status, stream, 0);
}
} // namespace pa
