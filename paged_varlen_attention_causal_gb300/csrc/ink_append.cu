// ink_append.cu -- KV append ("reshape_and_cache"): this step's keys and values
// into the paged cache at their slots, just before attention.
//
// A token's Hkv x 128 values are one contiguous block in the input and one
// contiguous block in the cache (a cache slot holds every KV head), so the copy
// is a gather of whole 16-byte chunks: consecutive threads take consecutive
// chunks of the same token, reading and writing coalesced, and a grid-stride
// loop covers K and V of every token.  The bound is HBM: 2 x (read + write) x
// T x Hkv x 256 bytes.
//
// FP8 cache (ink_append_fp8_kernel): each 16-byte chunk of 8 bf16 values is
// stored as 8 E4M3 bytes, code = E4M3(fp32(x) / scale), the correctly rounded
// fp32 quotient followed by the hardware's round-to-nearest-even, saturating
// conversion; HBM bytes 2 x (256 read + 128 written) x T x Hkv.
#include "ink_common.cuh"

namespace ink {

constexpr int kAppendThreads = 256;

__global__ void __launch_bounds__(kAppendThreads)
    ink_append_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value, uint4 *key_cache,
                      uint4 *value_cache, const int64_t *__restrict__ slot_mapping, long long num_tokens,
                      int chunks_per_token, long long num_slots, uint32_t *flags)
{
    pdl_wait();  // the previous kernel of the stream may still be finishing
    pdl_launch_dependents();
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

// Two fp32 values (lo first) to two E4M3 bytes (lo in the low byte): nearest even, saturating at 448.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// x / scale correctly rounded (fp32), with rcp = RN(1 / scale) computed once on the host: Markstein's
// correction step (q = RN(x rcp), remainder x - q scale exact by FMA, RN(q + remainder rcp)) gives the
// correctly rounded quotient when the quotient and its intermediates are finite normal numbers.  An exact
// quotient (zero remainder, which keeps -0) and infinite inputs return q itself; quotients that underflow
// quantize to an E4M3 zero of the right sign either way.
__device__ __forceinline__ float div_by_scale(float x, float scale, float rcp)
{
    const float q = x * rcp;
    const float r = fmaf(-q, scale, x);
    return (r == 0.f || !isfinite(q)) ? q : fmaf(r, rcp, q);
}

// Eight bf16 values / scale -> eight E4M3 bytes.
__device__ __forceinline__ uint2 quantize8(uint4 x, float scale, float rcp)
{
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        b[i] = f32x2_to_e4m3x2(div_by_scale(__uint_as_float(w[i] << 16), scale, rcp),
                               div_by_scale(__uint_as_float(w[i] & 0xffff0000u), scale, rcp));
    return make_uint2(b[0] | (b[1] << 16), b[2] | (b[3] << 16));
}

__global__ void __launch_bounds__(kAppendThreads)
    ink_append_fp8_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value, uint2 *key_cache,
                          uint2 *value_cache, const int64_t *__restrict__ slot_mapping, long long num_tokens,
                          int chunks_per_token, long long num_slots, float k_scale, float v_scale, float k_rcp,
                          float v_rcp, uint32_t *flags)
{
    pdl_wait();  // the previous kernel of the stream may still be finishing
    pdl_launch_dependents();
    const long long total = num_tokens * chunks_per_token;  // 16-byte bf16 chunks per tensor
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
        const long long dst = s * chunks_per_token + r;  // 8-byte E4M3 chunk of the slot
        key_cache[dst] = quantize8(__ldcs(key + c), k_scale, k_rcp);
        value_cache[dst] = quantize8(__ldcs(value + c), v_scale, v_rcp);
    }
}

cudaError_t launch_append_fp8(const ink_attn_dims *d, const void *key, const void *value, void *key_cache,
                              void *value_cache, const int64_t *slot_mapping, float k_scale, float v_scale,
                              uint32_t *flags, int sms, cudaStream_t stream)
{
    const int chunks = d->num_kv_heads * d->head_dim * 2 / 16;
    const long long total = (long long)d->num_tokens * chunks;
    const long long want = (total + kAppendThreads - 1) / kAppendThreads;
    const int grid = (int)(want < 8ll * sms ? (want > 0 ? want : 1) : 8ll * sms);
    return launch_pdl(ink_append_fp8_kernel, (unsigned)grid, kAppendThreads, 0, stream,
                      static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
                      static_cast<uint2 *>(key_cache), static_cast<uint2 *>(value_cache), slot_mapping,
                      (long long)d->num_tokens, chunks, (long long)d->num_blocks * d->block_size, k_scale, v_scale,
                      1.0f / k_scale, 1.0f / v_scale, flags);
}

cudaError_t launch_append(const ink_attn_dims *d, const void *key, const void *value, void *key_cache,
                          void *value_cache, const int64_t *slot_mapping, uint32_t *flags, int sms,
                          cudaStream_t stream)
{
    const int chunks = d->num_kv_heads * d->head_dim * 2 / 16;
    const long long total = (long long)d->num_tokens * chunks;
    // enough CTAs to fill every SM a few times over; each thread loops over its chunks
    const long long want = (total + kAppendThreads - 1) / kAppendThreads;
    const int grid = (int)(want < 8ll * sms ? (want > 0 ? want : 1) : 8ll * sms);
    return launch_pdl(ink_append_kernel, (unsigned)grid, kAppendThreads, 0, stream,
                      static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
                      static_cast<uint4 *>(key_cache), static_cast<uint4 *>(value_cache), slot_mapping,
                      (long long)d->num_tokens, chunks, (long long)d->num_blocks * d->block_size, flags);
}

}  // namespace ink
