// ink_append.cu -- KV append ("reshape_and_cache"): this step's keys and values
// into the paged cache at their slots, just before attention.
//
// A token's Hkv x 128 values are one contiguous block in the input and one
// contiguous block in the cache (a cache slot holds every KV head), so the copy
// is a gather of whole 16-byte chunks: consecutive threads take consecutive
// chunks of the same token, reading and writing coalesced, and a grid-stride
// loop covers K and V of every token.  The bound is HBM: 2 x (read + write) x
// T x Hkv x 256 bytes.
#include "ink_common.cuh"

namespace ink {

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads)
    ink_append_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value, uint4 *key_cache,
                      uint4 *value_cache, const int64_t *__restrict__ slot_mapping, long long num_tokens,
                      int chunks_per_token, long long num_slots, uint32_t *flags)
{
    const long long total = num_tokens * chunks_per_token;  // 16-byte chunks per tensor
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long c = (long long)blockIdx.x * blockDim.x + threadIdx.x; c < total; c += stride) {
        const long long t = c / chunks_per_token;
        const int r = (int)(c - t * chunks_per_token);
        const long long s = __ldg(slot_mapping + t);
        if (s < 0) continue;  // padding
        if (s >= num_slots) {
            if (r == 0 && flags) atomicOr(flags, INK_DEVERR_PAGE_ID);
            continue;
        }
        const long long dst = s * chunks_per_token + r;
        const uint4 k = __ldcs(key + c);  // read once: streaming loads
        const uint4 v = __ldcs(value + c);
        key_cache[dst] = k;
        value_cache[dst] = v;
    }
}

cudaError_t launch_append(const ink_attn_dims *d, const void *key, const void *value, void *key_cache,
                          void *value_cache, const int64_t *slot_mapping, uint32_t *flags, int sms,
                          cudaStream_t stream)
{
    const int chunks = d->num_kv_heads * kHeadDim * 2 / 16;
    const long long total = (long long)d->num_tokens * chunks;
    // enough CTAs to fill every SM a few times over; each thread loops over its chunks
    const long long want = (total + kAppendThreads - 1) / kAppendThreads;
    const int grid = (int)(want < 8ll * sms ? (want > 0 ? want : 1) : 8ll * sms);
    ink_append_kernel<<<grid, kAppendThreads, 0, stream>>>(
        static_cast<const uint4 *>(key), static_cast<const uint4 *>(value), static_cast<uint4 *>(key_cache),
        static_cast<uint4 *>(value_cache), slot_mapping, d->num_tokens, chunks,
        (long long)d->num_blocks * d->block_size, flags);
    return cudaGetLastError();
}

}  // namespace ink
