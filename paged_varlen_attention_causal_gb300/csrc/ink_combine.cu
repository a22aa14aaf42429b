// ink_combine.cu -- split-KV merge (a11): for every (token, head) row whose
// work unit was cut into more than one split, merge the per-split normalised
// outputs O_s and log-sum-exps lse_s:
//     lse = log sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * O_s.
// This is the log-sum-exp Phase 2 of the "paged_attention_v2_pytorch.py"
// page (global max, per-partition weights exp(m_s - gmax) * l_s, weighted sum
// divided by the weight total) written with lse_s = m_s + ln l_s.  Splits
// with no visible key carry lse_s = -inf and weigh nothing.
// One warp per row; lane l owns d values 4l..4l+3.
#include "ink_common.cuh"

namespace ink {

constexpr int kCombineWarps = 8;

__global__ void __launch_bounds__(kCombineWarps * 32) ink_combine_kernel(const Params p)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * kCombineWarps + warp;
    if (row >= (long long)p.T * p.H) return;
    const int t = (int)(row / p.H), h = (int)(row % p.H);
    // request owning token t: last b with cu[b] <= t and cu[b+1] > t
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(p.cu + mid + 1) > t) hi = mid; else lo = mid + 1;
    }
    const int b = lo;
    const Req r = load_req(p, b);
    if (!r.ok || t < r.t0 || t >= r.t0 + r.Lq) return;
    const int i = t - r.t0;

    const float *po;
    const float *pl;
    size_t stride_blk, first;  // partial row of split s = first + s * stride_blk
    int nact;
    if (is_decode_req(p, r)) {
        const UnitSplit u = unit_split(r.Lk - r.Lq, r.Lk - 1, r.Lk, p.causal, p.wl, p.wr, p.chunk_dec, 0);
        nact = u.nact;
        if (nact <= 1) return;
        first = (size_t)__ldg(p.dec_off + b) * p.dec_rows + (size_t)i * p.H + h;
        stride_blk = (size_t)p.dec_rows;
        po = p.part_dec_o;
        pl = p.part_dec_lse;
    } else {
        const int qt = i / p.tpt, k = i % p.tpt;
        const int i0 = qt * p.tpt, i1 = min(r.Lq, i0 + p.tpt) - 1;
        const UnitSplit u = unit_split(i0 + r.Lk - r.Lq, i1 + r.Lk - r.Lq, r.Lk, p.causal, p.wl, p.wr, p.chunk_pf, 0);
        nact = u.nact;
        if (nact <= 1) return;
        const int g = h / p.G, j = h % p.G;
        const size_t rows = (size_t)p.Hkv * kTileRows;
        first = (size_t)(__ldg(p.unit_off + b) + qt) * p.S_pf * rows + (size_t)g * kTileRows +
                pf_row_of(p.fast_pack, p.G, k, j);
        stride_blk = rows;
        po = p.part_pf_o;
        pl = p.part_pf_lse;
    }
    // global maximum of the split log-sum-exps
    float m = -INFINITY;
    for (int s = lane; s < nact; s += 32) m = fmaxf(m, pl[first + (size_t)s * stride_blk]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (m != -INFINITY) {
        for (int s0 = 0; s0 < nact; s0 += 32) {
            const int s = s0 + lane;
            const float w_l = (s < nact) ? __expf(pl[first + (size_t)s * stride_blk] - m) : 0.f;
            const int n = min(32, nact - s0);
            for (int q = 0; q < n; ++q) {
                const float w = __shfl_sync(0xffffffffu, w_l, q);
                wsum += w;
                if (w != 0.f) {
                    const float4 v = *reinterpret_cast<const float4 *>(po + (first + (size_t)(s0 + q) * stride_blk) * kHeadDim + 4 * lane);
                    acc.x = fmaf(w, v.x, acc.x);
                    acc.y = fmaf(w, v.y, acc.y);
                    acc.z = fmaf(w, v.z, acc.z);
                    acc.w = fmaf(w, v.w, acc.w);
                }
            }
        }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    uint2 outv;
    outv.x = pack_bf16x2(acc.x * inv, acc.y * inv);
    outv.y = pack_bf16x2(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2 *>(p.out + (size_t)row * kHeadDim + 4 * lane) = outv;
    if (p.lse && lane == 0) p.lse[row] = wsum > 0.f ? m + __logf(wsum) : -INFINITY;
}

cudaError_t launch_combine(const Params &p, int grid, cudaStream_t stream)
{
    ink_combine_kernel<<<grid, kCombineWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace ink
