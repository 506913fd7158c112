// pa_decode_noalloc: pa_decode for callers that cannot allocate device memory.
//
// Some callers are not allowed to allocate GPU memory at the point where they
// run decode attention: for example a plugin whose host framework owns every
// byte of device memory and forbids allocations inside its execute callback,
// or a latency-critical serving loop that must not risk an allocation's stall
// or failure mid-step. pa_decode needs a caller-provided workspace; this entry
// point instead uses one fixed scratch array that the library itself places in
// device memory when it is loaded.
//
// The scratch is a file-scope __device__ array. Host code cannot use its name
// as a device address (on the host the name is only a stand-in), so the first
// call on each device looks its address up with cudaGetSymbolAddress while
// that device is current and remembers it. Every later call on the device
// reuses that address. The lookup can load the library's device code, so the
// first call on a device should happen before any stream capture begins.
// The address belongs to the device's primary context: cudaDeviceReset
// destroys it, and a process that resets a device must reload the library
// before it calls this entry point on that device again.
#include <cuda_runtime.h>

#include <mutex>

#include "pa.h"

namespace pa {
pa_status decode_with_workspace(const void *q, const void *k_cache, const void *v_cache,
                                const float *k_scale, const float *v_scale,
                                const int32_t *block_tables, int32_t max_blocks,
                                const int32_t *context_lens, int32_t num_seqs, float scale,
                                void *out, void *workspace, size_t workspace_bytes, pa_geom g,
                                int32_t *dev_status, void *stream);
}

namespace {

// One copy per device that loads the library, kept until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once).
pa_status scratch_address(void **ptr)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return PA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return PA_OK;
}

} // namespace

extern "C" pa_status pa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                       const float *k_scale, const float *v_scale,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       const int32_t *context_lens, int32_t num_seqs, float scale,
                                       void *out, pa_geom geom, int32_t *dev_status, void *stream)
{
    if (num_seqs == 0)
        return PA_OK;
    const size_t need = pa_decode_workspace_size(geom, num_seqs, 0);
    if (need == 0)
        return PA_ERR_SHAPE;
    if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES)
        return PA_ERR_WORKSPACE; // this batch needs more scratch than the fixed array holds
    void *scratch = nullptr;
    pa_status st = scratch_address(&scratch);
    if (st != PA_OK)
        return st;
    // The array keeps whatever the previous call left. Only the leading
    // per-(sequence, kv head) counters must start at zero; a call with more
    // sequences than the last one would find old partial results there.
    const size_t counters = ((size_t)num_seqs * geom.n_kv * 4 + 255) / 256 * 256;
    if (cudaMemsetAsync(scratch, 0, counters, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PA_ERR_CUDA;
    return pa::decode_with_workspace(q, k_cache, v_cache, k_scale, v_scale, block_tables,
                                     max_blocks_per_seq, context_lens, num_seqs, scale, out,
                                     scratch, PA_NOALLOC_SCRATCH_BYTES, geom, dev_status, stream);
}
