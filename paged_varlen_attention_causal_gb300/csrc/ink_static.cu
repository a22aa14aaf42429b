// ink_static.cu -- the entry point for callers that cannot allocate device memory.
//
// Some programs that call this attention own every byte of device memory
// themselves: a serving engine that reserves nearly all of HBM up front for its
// paged KV-cache pool and its own arenas, or a plugin interface that hands an
// operator its input and output tensors but no scratch buffer and no allocator.
// Inside such a host a cudaMalloc issued by the operator either fails for lack
// of free memory or breaks the host's contract, so these callers cannot provide
// the workspace that ink_rel_attn_varlen takes.  ink_rel_attn_varlen_static
// runs the same computation on a fixed scratch area compiled into this library.
#include <mutex>

#include "ink_common.cuh"

namespace {

// The library's own scratch area.  Every GPU that loads the library holds it
// until the process exits.
static __device__ __align__(256) uint8_t g_ink_static_scratch[INK_STATIC_SCRATCH_BYTES];

constexpr int kMaxStaticDevices = 64;
void *g_scratch_addr[kMaxStaticDevices] = {};
std::mutex g_scratch_mutex;

// In host code, g_ink_static_scratch names a host-side stand-in for the device
// symbol, not a device address.  Its device address is looked up once per
// device, with that device current, and cached.
ink_status scratch_address(void **addr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxStaticDevices) return INK_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ink_static_scratch) != cudaSuccess || !p) return INK_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return INK_OK;
}

}  // namespace

extern "C" INK_API ink_status ink_rel_attn_varlen_static(
    const ink_attn_dims *dims, const void *q, const void *key_cache, const void *value_cache,
    const int32_t *block_table, const int32_t *cache_seqlens, const int32_t *cu_seqlens_q, int32_t max_seqlen_q,
    float softmax_scale, int causal, int32_t window_left, int32_t window_right, int32_t rel_extent,
    const float *rel_logits, int32_t num_splits, void *out, float *lse, ink_stream_t stream)
{
    // Work that needs more scratch than the fixed area is refused before anything runs: the call
    // below checks its actual plan (window and causality included) against the area and returns
    // INK_ERR_WORKSPACE; room left over stages K/V for the prefill as with any workspace.
    void *scratch = nullptr;
    const ink_status st = scratch_address(&scratch);
    if (st != INK_OK) return st;
    // The call's first kernel clears the header of the scratch area (error word and
    // work counters); everything else in it is written before it is read.
    return ink_rel_attn_varlen(dims, q, key_cache, value_cache, block_table, cache_seqlens, cu_seqlens_q,
                               max_seqlen_q, softmax_scale, causal, window_left, window_right, rel_extent,
                               rel_logits, num_splits, out, lse, scratch, (size_t)INK_STATIC_SCRATCH_BYTES, stream);
}
