// ink_stage.cu -- K/V staging for the prefill kernel: a page gather that copies
// the K and V pages of every staged prefill-shaped request (the prepass chooses
// them) out of the paged cache into a contiguous area of the workspace, one
// plane per KV head: ks[g][off + j][:] = key_cache[block_table[b][j / bs]][j % bs][g][:]
// for keys j < Lk (whole 16-key pages), and the same for V.  An E4M3 cache is
// converted to bf16 on the way (exactly: every E4M3 value is a bf16 value).
//
// Why: the prefill reads each K and V tile of a request once per q tile and KV
// head.  From the paged layout a tile of one KV head is 128 rows of 256 bytes,
// 2 KB apart (every KV head of a key sits side by side); from the staging area it
// is 32 KB of consecutive bytes, one TMA box, which the L2 delivers at a much
// higher rate.  The copy reads every page once, in whole 16-key pages (all KV
// heads contiguous), and writes it once.
//
// One CTA per page (grid-stride over the prepass's page list): 256 threads move
// 16 bytes each per step, reading the page in order and writing 256-byte rows.
#include <cuda_fp16.h>

#include "ink_common.cuh"

namespace ink {

constexpr int kStageThreads = 256;

// Two E4M3 bytes (low byte first) to a bf16 pair: through fp16, which holds every E4M3 value exactly,
// then to bf16, which does too (at most 4 significant bits, exponents 2^-9 .. 2^8).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint32_t two)
{
    uint32_t h;
    const uint16_t in = (uint16_t)(two & 0xffffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(in));
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&h));
    return pack_bf16x2(f.x, f.y);
}

// Eight E4M3 bytes (two words, low byte first) to eight bf16 values.
__device__ __forceinline__ uint4 e4m3x8_to_bf16x8(uint32_t lo, uint32_t hi)
{
    return make_uint4(e4m3x2_to_bf16x2(lo), e4m3x2_to_bf16x2(lo >> 16), e4m3x2_to_bf16x2(hi),
                      e4m3x2_to_bf16x2(hi >> 16));
}

__global__ void __launch_bounds__(kStageThreads) ink_stage_kernel(const Params p)
{
    pdl_wait();
    pdl_launch_dependents();
    const int total = (int)*(volatile uint32_t *)&p.hdr->stage_pages;
    const int chunks = kKeyGroup * p.Hkv * (kHeadDim * 2 / 16);  // 16-byte chunks of one tensor's page
    for (int pg = blockIdx.x; pg < total; pg += gridDim.x) {
        int lo = 0, hi = p.B - 1;  // request owning page pg: last b with stg_pg_off[b] <= pg
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(p.stg_pg_off + mid) <= pg) lo = mid; else hi = mid - 1;
        }
        const int b = lo;
        const int j = pg - __ldg(p.stg_pg_off + b);  // 16-key group of the request
        const int key = j * kKeyGroup;
        const int pid = __ldg(p.bt + (size_t)b * p.MAXBLK + key / p.BS);
        const bool page_ok = pid >= 0 && pid < p.NB;
        if (!page_ok && threadIdx.x == 0) report(p, INK_DEVERR_PAGE_ID);
        const size_t src_row = ((size_t)pid * p.BS + key % p.BS) * p.Hkv;  // first (key, head) row of the group
        const size_t dst_key = (size_t)__ldg(p.stg_off + b) + key;
        if (p.kv_fp8) {
            // E4M3 bytes: a 16-byte chunk holds 16 values of one (key, head) row, written as 32 bytes of bf16
            // (every E4M3 value is exact in fp16 and in bf16); the scales are applied by the prefill
            const uint8_t *k8 = reinterpret_cast<const uint8_t *>(p.kc), *v8 = reinterpret_cast<const uint8_t *>(p.vc);
            for (int c = threadIdx.x; c < chunks / 2; c += kStageThreads) {
                const int kr = c / (p.Hkv * 8), g = (c / 8) % p.Hkv, ch = c % 8;
                const size_t src = (src_row + (size_t)kr * p.Hkv + g) * kHeadDim + ch * 16;
                const size_t dst = ((size_t)g * p.stage_cap + dst_key + kr) * kHeadDim + ch * 16;
                uint4 kb = make_uint4(0, 0, 0, 0), vb = make_uint4(0, 0, 0, 0);
                if (page_ok) {
                    kb = __ldg(reinterpret_cast<const uint4 *>(k8 + src));
                    vb = __ldg(reinterpret_cast<const uint4 *>(v8 + src));
                }
                uint4 *kd = reinterpret_cast<uint4 *>(p.ks + dst), *vd = reinterpret_cast<uint4 *>(p.vs + dst);
                kd[0] = e4m3x8_to_bf16x8(kb.x, kb.y);
                kd[1] = e4m3x8_to_bf16x8(kb.z, kb.w);
                vd[0] = e4m3x8_to_bf16x8(vb.x, vb.y);
                vd[1] = e4m3x8_to_bf16x8(vb.z, vb.w);
            }
            continue;
        }
        for (int c = threadIdx.x; c < chunks; c += kStageThreads) {
            const int kr = c / (p.Hkv * 16), g = (c / 16) % p.Hkv, ch = c % 16;
            const size_t src = (src_row + (size_t)kr * p.Hkv + g) * kHeadDim + ch * 8;
            const size_t dst = ((size_t)g * p.stage_cap + dst_key + kr) * kHeadDim + ch * 8;
            uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
            if (page_ok) {
                kv = __ldg(reinterpret_cast<const uint4 *>(p.kc + src));
                vv = __ldg(reinterpret_cast<const uint4 *>(p.vc + src));
            }
            *reinterpret_cast<uint4 *>(p.ks + dst) = kv;
            *reinterpret_cast<uint4 *>(p.vs + dst) = vv;
        }
    }
}

// The grid covers every SM a few times; CTAs past the page list return at once.
cudaError_t launch_stage(const Params &p, int sms, cudaStream_t stream)
{
    return launch_pdl(ink_stage_kernel, 8 * sms, kStageThreads, 0, stream, p);
}

}  // namespace ink
