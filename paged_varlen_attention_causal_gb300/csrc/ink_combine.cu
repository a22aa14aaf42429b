// ink_combine.cu -- split-KV merge: for every (token, head) row whose
// work unit was cut into more than one split, merge the per-split normalised
// outputs O_s and log-sum-exps lse_s:
//     lse = log sum_s exp(lse_s),   out = sum_s exp(lse_s - lse) * O_s.
// This is the log-sum-exp Phase 2 of the "paged_attention_v2_pytorch.py"
// page (global max, per-partition weights exp(m_s - gmax) * l_s, weighted sum
// divided by the weight total) written with lse_s = m_s + ln l_s, streamed:
// each warp keeps a running maximum and rescales its sums when it grows.
// Splits with no visible key carry lse_s = -inf and weigh nothing.
//
// kWarpsPerRow warps share one row (warp w takes splits w, w + kWarpsPerRow, ...)
// and merge their states through shared memory; lane l owns D / 32 consecutive
// d values.  Loads are issued kBatch splits at a time.  The merge is bound by the
// latency of those loads, not by their bytes, so the host gives a row as many
// warps as keep each warp's share of its splits to about one batch.
#include <algorithm>

#include "ink_common.cuh"

namespace ink {

struct RowPartials {
    const float *po, *pl;
    size_t first, stride;  // partial row of split s = first + s * stride
    int nact;
};

// The per-request arrays a merge row is located by: shared-memory copies when the batch is small
// (each lookup below would otherwise be a dependent global load), else the global arrays.
constexpr int kCombSmemReqs = 512;

struct CombMeta {
    const int *cu, *seqk, *comb_off, *dec_off, *unit_off;
};

// Row r of the merge list: token c = r / H of the list (request b, token t) and head h.
// The prepass lists, per request, every token of a request that was split.
__device__ __forceinline__ void list_row(const Params &p, const CombMeta &mt, long long r, int &b, int &t, int &h)
{
    const int c = (int)(r / p.H);
    h = (int)(r % p.H);
    int lo = 0, hi = p.B - 1;  // request owning list token c: last b with comb_off[b] <= c
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (mt.comb_off[mid] <= c) lo = mid; else hi = mid - 1;
    }
    b = lo;
    t = mt.cu[b] + (c - mt.comb_off[b]);
}

// Locate the partials of row (t, h) of request b; false when the row needs no merge.
__device__ __forceinline__ bool row_partials(const Params &p, const CombMeta &mt, int b, int t, int h,
                                             RowPartials &rp)
{
    const Req r = make_req(p, mt.cu[b], mt.cu[b + 1], mt.seqk[b]);
    if (!r.ok || t < r.t0 || t >= r.t0 + r.Lq) return false;
    const int i = t - r.t0;
    if (is_decode_req(p, r)) {
        const UnitSplit u = unit_split(r.Lk - r.Lq, r.Lk - 1, r.Lk, p.causal, p.wl, p.wr, p.chunk_dec, 0);
        rp.nact = u.nact;
        if (rp.nact <= 1) return false;
        rp.first = (size_t)mt.dec_off[b] * p.dec_rows + (size_t)i * p.H + h;
        rp.stride = (size_t)p.dec_rows;
        rp.po = p.part_dec_o;
        rp.pl = p.part_dec_lse;
    } else {
        const int qt = i / p.tpt, k = i % p.tpt;
        const int i0 = qt * p.tpt, i1 = min(r.Lq, i0 + p.tpt) - 1;
        const UnitSplit u = unit_split(i0 + r.Lk - r.Lq, i1 + r.Lk - r.Lq, r.Lk, p.causal, p.wl, p.wr, p.chunk_pf, 0);
        rp.nact = u.nact;
        if (rp.nact <= 1) return false;
        const int g = h / p.G, j = h % p.G;
        const size_t rows = (size_t)p.Hkv * kTileRows;
        rp.first = (size_t)(mt.unit_off[b] + qt) * p.S_pf * rows + (size_t)g * kTileRows +
                   pf_row_of(p.fast_pack, p.G, k, j);
        rp.stride = rows;
        rp.po = p.part_pf_o;
        rp.pl = p.part_pf_lse;
    }
    return true;
}

// V consecutive floats of one lane (V = D / 32): loads and the bf16 store.
template <int V>
__device__ __forceinline__ void ld_vec(const float *src, float (&x)[V])
{
    if constexpr (V == 2) {
        const float2 a = __ldg(reinterpret_cast<const float2 *>(src));
        x[0] = a.x; x[1] = a.y;
    } else {
#pragma unroll
        for (int q = 0; q < V / 4; ++q) {
            const float4 a = __ldg(reinterpret_cast<const float4 *>(src) + q);
            x[4 * q] = a.x; x[4 * q + 1] = a.y; x[4 * q + 2] = a.z; x[4 * q + 3] = a.w;
        }
    }
}

template <int V>
__device__ __forceinline__ void st_bf16(__nv_bfloat16 *dst, const float (&x)[V], float scale)
{
    uint32_t w[V / 2];
#pragma unroll
    for (int q = 0; q < V / 2; ++q) w[q] = pack_bf16x2(x[2 * q] * scale, x[2 * q + 1] * scale);
    if constexpr (V == 2) {
        *reinterpret_cast<uint32_t *>(dst) = w[0];
    } else if constexpr (V == 4) {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
    } else {
        *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Threads of a combine CTA: 8 warps, or one row's warps when a row takes more.
template <int kWarpsPerRow>
__host__ __device__ constexpr int combine_threads() { return kWarpsPerRow > 8 ? 32 * kWarpsPerRow : 256; }

template <int kWarpsPerRow, int D>
__global__ void __launch_bounds__(combine_threads<kWarpsPerRow>()) ink_combine_kernel(const Params p)
{
    constexpr int kCombineThreads = combine_threads<kWarpsPerRow>();
    constexpr int kRowsPerCta = kCombineThreads / 32 / kWarpsPerRow;
    constexpr int V = D / 32;  // head-dim values per lane: lane l owns V l .. V l + V - 1
    // splits whose loads are in flight at once (fewer in a 1024-thread CTA: 64 registers a thread)
    constexpr int kBatch = kWarpsPerRow > 8 ? (V <= 2 ? 8 : 16 / V) : (V <= 4 ? 8 : 4);
    __shared__ float s_m[kCombineThreads / 32], s_l[kCombineThreads / 32];
    __shared__ float s_acc[kWarpsPerRow > 1 ? kCombineThreads / 32 : 1][32][V];
    __shared__ int s_cu[kCombSmemReqs + 1], s_seqk[kCombSmemReqs], s_comb[kCombSmemReqs + 1];
    __shared__ int s_doff[kCombSmemReqs + 1], s_uoff[kCombSmemReqs + 1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = warp % kWarpsPerRow;  // this warp's share of the row's splits
    // The prepass's outputs (merge-list size, per-request offsets) and the call's inputs are complete before
    // this grid can start: it launches early only once every CTA of the kernel before it has passed its own
    // wait, and so on back to the prepass.  Only the split partials, written by that kernel, need the wait.
    const long long nrows = (long long)*(volatile uint32_t *)&p.hdr->comb_tokens * p.H;
    CombMeta mt{p.cu, p.seqk, p.comb_off, p.dec_off, p.unit_off};
    if (p.B <= kCombSmemReqs) {  // one round of loads for all of them (read-only here)
        for (int i = threadIdx.x; i <= p.B; i += kCombineThreads) {
            s_cu[i] = __ldg(p.cu + i);
            s_comb[i] = __ldg(p.comb_off + i);
            s_doff[i] = __ldg(p.dec_off + i);
            s_uoff[i] = __ldg(p.unit_off + i);
            if (i < p.B) s_seqk[i] = __ldg(p.seqk + i);
        }
        mt = CombMeta{s_cu, s_seqk, s_comb, s_doff, s_uoff};
        __syncthreads();
    }
    pdl_wait();
    pdl_launch_dependents();
    // Grid-stride over the merge list; the trip count is the same for all warps of a CTA.
    for (long long row0 = (long long)blockIdx.x * kRowsPerCta; row0 < nrows; row0 += (long long)gridDim.x * kRowsPerCta) {
        const long long row = row0 + warp / kWarpsPerRow;
        RowPartials rp;
        int b = 0, t = 0, h = 0;
        bool active = row < nrows;
        if (active) {
            list_row(p, mt, row, b, t, h);
            active = row_partials(p, mt, b, t, h, rp);
        }
        float m = -INFINITY, l = 0.f;
        float acc[V];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = 0.f;
        if (active) {
            for (int s0 = sub; s0 < rp.nact; s0 += kWarpsPerRow * kBatch) {
                float ls[kBatch];
                float os[kBatch][V];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {  // issue the batch's loads before using any of them
                    const int s = s0 + u * kWarpsPerRow;
                    ls[u] = -INFINITY;
#pragma unroll
                    for (int e = 0; e < V; ++e) os[u][e] = 0.f;
                    if (s < rp.nact) {
                        const size_t pr = rp.first + (size_t)s * rp.stride;
                        ls[u] = __ldg(rp.pl + pr);
                        ld_vec<V>(rp.po + pr * D + V * lane, os[u]);
                    }
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    if (ls[u] == -INFINITY) continue;
                    if (ls[u] > m) {
                        const float a = __expf(m - ls[u]);  // m = -inf gives 0
#pragma unroll
                        for (int e = 0; e < V; ++e) acc[e] *= a;
                        l *= a;
                        m = ls[u];
                    }
                    const float w = __expf(ls[u] - m);
                    l += w;
#pragma unroll
                    for (int e = 0; e < V; ++e) acc[e] = fmaf(w, os[u][e], acc[e]);
                }
            }
        }
        if (kWarpsPerRow > 1) {
            if (lane == 0) {
                s_m[warp] = m;
                s_l[warp] = l;
            }
#pragma unroll
            for (int e = 0; e < V; ++e) s_acc[warp][lane][e] = acc[e];
            __syncthreads();
            if (active && sub == 0) {
                float gm = -INFINITY;
#pragma unroll
                for (int w = 0; w < kWarpsPerRow; ++w) gm = fmaxf(gm, s_m[warp + w]);
                l = 0.f;
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] = 0.f;
                if (gm != -INFINITY) {
#pragma unroll
                    for (int w = 0; w < kWarpsPerRow; ++w) {
                        if (s_m[warp + w] == -INFINITY) continue;
                        const float a = __expf(s_m[warp + w] - gm);
                        l = fmaf(a, s_l[warp + w], l);
#pragma unroll
                        for (int e = 0; e < V; ++e) acc[e] = fmaf(a, s_acc[warp + w][lane][e], acc[e]);
                    }
                }
                m = gm;
            }
            __syncthreads();  // s_* are rewritten by the next row
            if (sub != 0) continue;
        }
        if (!active) continue;
        const size_t orow = (size_t)t * p.H + h;
        st_bf16<V>(p.out + orow * D + V * lane, acc, l > 0.f ? 1.f / l : 0.f);
        if (p.lse && lane == 0) p.lse[orow] = l > 0.f ? m + __logf(l) : -INFINITY;
    }
}

template <int W, int D>
cudaError_t launch_combine_w(const Params &p, int sms, cudaStream_t stream)
{
    constexpr long long per = combine_threads<W>() / 32 / W;  // rows a CTA takes at a time
    const long long rows = (long long)p.T * p.H;
    const long long grid = std::min<long long>((rows + per - 1) / per, 16ll * sms);
    return launch_pdl(ink_combine_kernel<W, D>, (unsigned)grid, combine_threads<W>(), 0, stream, p);
}

// Warps per row: enough that a warp takes about one batch of loads (8 splits at D <= 128) of the row
// with the most splits, from 1 to 32, but no more than keep every row's warps resident at once (64
// warps an SM): past that, extra warps only add CTAs and their shared-memory merges.  The grid is
// sized for every row of the call; CTAs past the merge list the prepass wrote return at once.
template <int D>
cudaError_t launch_combine_d(const Params &p, int sms, int max_splits, cudaStream_t stream)
{
    const long long rows = (long long)p.T * p.H, resident = 64ll * sms;
    const int by_splits = max_splits <= 8 ? 1 : max_splits <= 32 ? 4 : max_splits <= 64 ? 8 : 32;
    const int by_rows = rows * 32 <= resident ? 32 : rows * 8 <= resident ? 8 : rows * 4 <= resident ? 4 : 1;
    switch (std::min(by_splits, by_rows)) {
        case 1: return launch_combine_w<1, D>(p, sms, stream);
        case 4: return launch_combine_w<4, D>(p, sms, stream);
        case 8: return launch_combine_w<8, D>(p, sms, stream);
        default: return launch_combine_w<32, D>(p, sms, stream);
    }
}

cudaError_t launch_combine(const Params &p, int sms, int max_splits, cudaStream_t stream)
{
    switch (p.D) {
        case 64: return launch_combine_d<64>(p, sms, max_splits, stream);
        case 128: return launch_combine_d<128>(p, sms, max_splits, stream);
        case 256: return launch_combine_d<256>(p, sms, max_splits, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ink
