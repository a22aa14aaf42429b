// ink_prepass.cu -- device-side plan of one call (validation and work
// decomposition), so that the host never has to read cu_seqlens_q or
// cache_seqlens and the whole call stays free of host synchronisation.
//
// One CTA of 1024 threads:
//   1. clears the workspace header (error word, counters);
//   2. validates every request and classifies it as decode-shaped (one unit)
//      or prefill-shaped (q tiles of `tpt` tokens);
//   3. writes the decode work items (request, split) in request order;
//   4. writes the prefill work items (request, q tile, split, KV head) sorted
//      by decreasing number of 128-key tiles (a counting sort), so that the
//      persistent prefill kernel hands out the longest items first.
#include "ink_common.cuh"

namespace ink {

constexpr int kPrepassThreads = 1024;
constexpr int kCostBuckets = 1024;
constexpr int kSmemReqs = 2048;  // batches up to this size keep their per-request offsets in shared memory too

// Exclusive block-wide scan of one int per thread; returns the block total.
__device__ int block_exclusive_scan(int v, int *out, int *warp_sums)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const int total = warp_sums[31];
    *out = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
    __syncthreads();
    return total;
}

// Four such scans at once (one set of barriers for the four counts of pass 1).
__device__ int4 block_exclusive_scan4(int4 v, int4 *out, int4 *warp_sums)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int4 x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y0 = __shfl_up_sync(0xffffffffu, x.x, o), y1 = __shfl_up_sync(0xffffffffu, x.y, o);
        const int y2 = __shfl_up_sync(0xffffffffu, x.z, o), y3 = __shfl_up_sync(0xffffffffu, x.w, o);
        if (lane >= o) {
            x.x += y0;
            x.y += y1;
            x.z += y2;
            x.w += y3;
        }
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int4 w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y0 = __shfl_up_sync(0xffffffffu, w.x, o), y1 = __shfl_up_sync(0xffffffffu, w.y, o);
            const int y2 = __shfl_up_sync(0xffffffffu, w.z, o), y3 = __shfl_up_sync(0xffffffffu, w.w, o);
            if (lane >= o) {
                w.x += y0;
                w.y += y1;
                w.z += y2;
                w.w += y3;
            }
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const int4 total = warp_sums[31];
    const int4 before = warp > 0 ? warp_sums[warp - 1] : make_int4(0, 0, 0, 0);
    *out = make_int4(x.x - v.x + before.x, x.y - v.y + before.y, x.z - v.z + before.z, x.w - v.w + before.w);
    __syncthreads();
    return total;
}

// The same scan in 64 bits (sums that may exceed the int range).
__device__ long long block_exclusive_scan_ll(long long v, long long *out, long long *warp_sums)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        long long w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const long long total = warp_sums[31];
    *out = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
    __syncthreads();
    return total;
}

__device__ __forceinline__ void pf_unit_of(const Params &p, const Req &r, int qt, int &qa0, int &qa1)
{
    const int ut = p.pair ? 2 * p.tpt : p.tpt;  // tokens per unit: one q tile, or a pair for the 2-SM prefill
    const int i0 = qt * ut, i1 = min(r.Lq, i0 + ut) - 1;
    qa0 = i0 + r.Lk - r.Lq;
    qa1 = i1 + r.Lk - r.Lq;
}

// Cost of a prefill split in 128-key tiles, clamped to the bucket range.
__device__ __forceinline__ int pf_cost_bucket(const UnitSplit &u)
{
    const int groups = u.ge - u.gb;
    const int tiles = (groups + 7) / 8;
    return min(tiles, kCostBuckets - 1);
}

__global__ void __launch_bounds__(kPrepassThreads, 1) ink_prepass_kernel(Params p)
{
    __shared__ int warp_sums[32];
    __shared__ int4 warp_sums4[32];
    __shared__ int s_dec_off[kSmemReqs + 1], s_unit_off[kSmemReqs + 1];  // copies for the searches below
    __shared__ int bucket_count[kCostBuckets];
    __shared__ int bucket_base[kCostBuckets];
    __shared__ int s_carry[4];
    __shared__ long long warp_sums_ll[32];
    __shared__ long long s_stg_carry;
    __shared__ int s_pg_carry;
    __shared__ uint32_t s_err;
    __shared__ int s_overflow;
    __shared__ int4 s_req[kPrepassThreads];  // (t0, Lq, Lk) of the first kPrepassThreads requests

    int *dec_off = p.dec_off;
    int *unit_off = p.unit_off;
    int *comb_off = p.comb_off;
    const int tid = threadIdx.x;
    pdl_wait();  // the previous kernel of the stream (e.g. the last call's merge, which reads this workspace)
    pdl_launch_dependents();
    // this thread's request among the first kPrepassThreads (the whole batch, mostly), loaded here so that
    // the loads overlap the header checks below
    const Req pre = tid < p.B ? load_req(p, tid) : Req{};

    if (tid == 0) {
        p.hdr->errors = 0;
        p.hdr->dec_count = 0;
        p.hdr->pf_count = 0;
        p.hdr->dec_next = 0;
        p.hdr->pf_next = 0;
        p.hdr->comb_tokens = 0;
        s_carry[0] = s_carry[1] = s_carry[2] = s_carry[3] = 0;
        s_stg_carry = 0;
        s_pg_carry = 0;
        p.hdr->stage_pages = 0;
        uint32_t e = 0;
        if (__ldg(p.cu) != 0 || __ldg(p.cu + p.B) != p.T) e |= INK_DEVERR_CU_SEQLENS;
        s_err = e;
    }
    for (int i = tid; i < kCostBuckets; i += blockDim.x) bucket_count[i] = 0;
    __syncthreads();

    // K/V staging: prefill-shaped requests, in request order, take whole 128-key tiles of the
    // staging area while it has room; the rest read the paged cache.  Then the page work list
    // of the copy (one entry per staged 16-key page).
    if (p.stage_cap > 0) {
        for (int base = 0; base < p.B; base += blockDim.x) {
            const int b = base + tid;
            long long need = 0;
            int pages = 0;
            if (b < p.B) {
                const Req r = base == 0 ? pre : load_req(p, b);
                if (r.ok && r.Lq > 0 && !is_decode_req(p, r) && r.Lk > 0) need = stage_keys_of(r.Lk);
            }
            long long x;
            const long long tot = block_exclusive_scan_ll(need, &x, warp_sums_ll);
            bool staged = false;
            if (b < p.B) {
                const long long at = s_stg_carry + x;
                staged = need > 0 && at + need <= p.stage_cap;
                p.stg_off[b] = staged ? (int)at : -1;
                if (staged) pages = (__ldg(p.seqk + b) + kKeyGroup - 1) / kKeyGroup;
            }
            int xp;
            const int totp = block_exclusive_scan(pages, &xp, warp_sums);
            if (b < p.B) p.stg_pg_off[b] = s_pg_carry + xp;
            __syncthreads();
            if (tid == 0) {
                s_stg_carry += tot;
                s_pg_carry += totp;
            }
            __syncthreads();
        }
        if (tid == 0) {
            p.stg_pg_off[p.B] = s_pg_carry;
            p.hdr->stage_pages = (uint32_t)s_pg_carry;
        }
    } else {
        for (int b = tid; b < p.B; b += blockDim.x) p.stg_off[b] = -1;
    }
    __syncthreads();

    // pass 1: per request, decode split count, prefill q-tile count and the tokens whose
    // rows the split-KV merge must visit (all of a request's tokens once it is split); scans.
    uint32_t my_err = 0;
    for (int base = 0; base < p.B; base += blockDim.x) {
        const int b = base + tid;
        int ndec = 0, nq = 0, nc = 0, ntile = 0;  // ntile: q tiles of tpt tokens, for the budget check
        if (b < p.B) {
            Req r = base == 0 ? pre : load_req(p, b);
            if (base == 0) s_req[b] = make_int4(r.t0, r.Lq, r.Lk, 0);
            my_err |= r.err;
            if (r.ok && r.Lq > 0) {
                if (is_decode_req(p, r)) {
                    UnitSplit u = unit_split(r.Lk - r.Lq, r.Lk - 1, r.Lk, p.causal, p.wl, p.wr, p.chunk_dec, 0);
                    ndec = u.nact;
                    nc = ndec > 1 ? r.Lq : 0;
                } else if (p.kv_fp8 && p.stg_off[b] < 0) {
                    // an FP8 cache is read by the prefill only through the staging copy
                    my_err |= INK_DEVERR_STAGE;
                } else {
                    const int ut = p.pair ? 2 * p.tpt : p.tpt;
                    nq = (r.Lq + ut - 1) / ut;
                    ntile = (r.Lq + p.tpt - 1) / p.tpt;
                    nc = p.S_pf > 1 ? r.Lq : 0;
                }
                if (p.causal && r.Lk < r.Lq) my_err |= INK_DEVERR_EMPTY_ROWS;
            }
        }
        int4 x;
        const int4 tot = block_exclusive_scan4(make_int4(ndec, nq, nc, ntile), &x, warp_sums4);
        if (b < p.B) {
            dec_off[b] = s_carry[0] + x.x;
            unit_off[b] = s_carry[1] + x.y;
            comb_off[b] = s_carry[2] + x.z;
            if (p.B <= kSmemReqs) {
                s_dec_off[b] = s_carry[0] + x.x;
                s_unit_off[b] = s_carry[1] + x.y;
            }
        }
        __syncthreads();
        if (tid == 0) {
            s_carry[0] += tot.x;
            s_carry[1] += tot.y;
            s_carry[2] += tot.z;
            s_carry[3] += tot.w;
        }
        __syncthreads();
    }
    if (tid == 0) {
        dec_off[p.B] = s_carry[0];
        unit_off[p.B] = s_carry[1];
        comb_off[p.B] = s_carry[2];
        // Requests whose token ranges overlap (a cu_seqlens_q entry that steps back between valid
        // neighbours) can need more q tiles than T tokens allow, and the prefill partials are sized
        // for T: such a batch is flagged and runs nothing.
        s_overflow = s_carry[3] > p.units_cap;  // counted in single q tiles, whichever kernel runs them
        if (s_overflow) s_err |= INK_DEVERR_CU_SEQLENS;
        p.hdr->comb_tokens = s_overflow ? 0u : (uint32_t)s_carry[2];
    }
    __syncthreads();
    if (my_err) atomicOr(&s_err, my_err);
    __syncthreads();
    __threadfence_block();

    const int n_dec = s_overflow ? 0 : min(s_carry[0], p.dec_items_cap);
    const int n_units = s_overflow ? 0 : s_carry[1];

    const int *doff = p.B <= kSmemReqs ? s_dec_off : dec_off;
    const int *uoff = p.B <= kSmemReqs ? s_unit_off : unit_off;

    // pass 2: decode items (request, split), request order; one item per thread, so that a
    // single long request's splits are written in parallel.
    for (int i = tid; i < n_dec; i += blockDim.x) {
        int lo = 0, hi = p.B - 1;  // request owning item i: last b with dec_off[b] <= i
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (doff[mid] <= i) lo = mid; else hi = mid - 1;
        }
        int4 rq;  // a decode item's request is valid (t0, Lq <= 16, Lk), and its split index < 2^27
        if (lo < kPrepassThreads) {
            rq = s_req[lo];
        } else {
            const Req r = load_req(p, lo);
            rq = make_int4(r.t0, r.Lq, r.Lk, 0);
        }
        p.dec_items[i] = make_int4(lo, (int)((unsigned)(i - doff[lo]) | ((unsigned)rq.y << 27)), rq.x, rq.z);
    }
    if (n_units == 0) {  // no prefill unit: nothing to sort
        if (tid == 0) {
            p.hdr->pf_count = 0u;
            p.hdr->dec_count = (uint32_t)n_dec;
            atomicOr(&p.hdr->errors, s_err);
        }
        return;
    }

    // pass 3: prefill units -> cost histogram of their splits.
    for (int u = tid; u < n_units; u += blockDim.x) {
        int lo = 0, hi = p.B - 1;  // request owning unit u: last b with unit_off[b] <= u
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (uoff[mid] <= u) lo = mid; else hi = mid - 1;
        }
        const int b = lo, qt = u - uoff[b];
        Req r = load_req(p, b);
        int qa0, qa1;
        pf_unit_of(p, r, qt, qa0, qa1);
        UnitSplit u0 = unit_split(qa0, qa1, r.Lk, p.causal, p.wl, p.wr, p.chunk_pf, 0);
        for (int s = 0; s < u0.nact; ++s) {
            UnitSplit us = unit_split(qa0, qa1, r.Lk, p.causal, p.wl, p.wr, p.chunk_pf, s);
            atomicAdd(&bucket_count[pf_cost_bucket(us)], p.Hkv);
        }
    }
    __syncthreads();
    // descending-cost bucket bases: bucket k starts after every bucket > k
    {
        int x = 0;
        const int k = kCostBuckets - 1 - tid;  // tid 0 -> highest cost
        const int c = (k >= 0) ? bucket_count[k] : 0;
        const int total = block_exclusive_scan(c, &x, warp_sums);
        if (k >= 0) bucket_base[k] = x;
        if (tid == 0) {
            p.hdr->pf_count = (uint32_t)min(total, p.pf_items_cap);
            p.hdr->dec_count = (uint32_t)n_dec;
        }
    }
    for (int i = tid; i < kCostBuckets; i += blockDim.x) bucket_count[i] = 0;  // reused as cursors
    __syncthreads();
    // pass 4: scatter the prefill items, KV heads of one split side by side
    const int cap = p.pf_items_cap;
    for (int u = tid; u < n_units; u += blockDim.x) {
        int lo = 0, hi = p.B - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (uoff[mid] <= u) lo = mid; else hi = mid - 1;
        }
        const int b = lo, qt = u - uoff[b];
        Req r = load_req(p, b);
        int qa0, qa1;
        pf_unit_of(p, r, qt, qa0, qa1);
        UnitSplit u0 = unit_split(qa0, qa1, r.Lk, p.causal, p.wl, p.wr, p.chunk_pf, 0);
        for (int s = 0; s < u0.nact; ++s) {
            UnitSplit us = unit_split(qa0, qa1, r.Lk, p.causal, p.wl, p.wr, p.chunk_pf, s);
            const int c = pf_cost_bucket(us);
            const int pos = bucket_base[c] + atomicAdd(&bucket_count[c], p.Hkv);
            for (int g = 0; g < p.Hkv; ++g)
                if (pos + g < cap) p.pf_items[pos + g] = make_int4(b, qt, s, g);
        }
    }
    __syncthreads();
    if (tid == 0) atomicOr(&p.hdr->errors, s_err);
}

// The same plan for a call of at most 32 requests that can hold only decode-shaped ones (the host's bound
// max_seqlen_q * G <= 16): one warp, a lane per request, warp scans instead of block-wide barriers.  It writes
// what the block version writes for such a call: the header, the per-request offsets (no unit, no staging),
// the merge list and the decode items.
constexpr int kSmallBatch = 32;

__global__ void __launch_bounds__(32, 1) ink_prepass_small_kernel(Params p)
{
    __shared__ int s_off[kSmallBatch + 1];
    __shared__ int4 s_rq[kSmallBatch];
    const int lane = threadIdx.x;
    pdl_wait();  // the previous kernel of the stream (e.g. the last call's merge, which reads this workspace)
    pdl_launch_dependents();
    const bool have = lane < p.B;
    const Req r = have ? load_req(p, lane) : Req{};
    uint32_t err = 0;
    int ndec = 0, nc = 0;
    if (have) {
        err = r.err;
        if (r.ok && r.Lq > 0) {  // decode-shaped: the host's bound on max_seqlen_q leaves no other kind
            const UnitSplit u = unit_split(r.Lk - r.Lq, r.Lk - 1, r.Lk, p.causal, p.wl, p.wr, p.chunk_dec, 0);
            ndec = u.nact;
            nc = ndec > 1 ? r.Lq : 0;
            if (p.causal && r.Lk < r.Lq) err |= INK_DEVERR_EMPTY_ROWS;
        }
    }
    if (lane == 0 && (__ldg(p.cu) != 0 || __ldg(p.cu + p.B) != p.T)) err |= INK_DEVERR_CU_SEQLENS;
    int xd = ndec, xc = nc;  // inclusive scans of the decode items and merge tokens
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yd = __shfl_up_sync(0xffffffffu, xd, o), yc = __shfl_up_sync(0xffffffffu, xc, o);
        if (lane >= o) {
            xd += yd;
            xc += yc;
        }
    }
    const int dec_total = __shfl_sync(0xffffffffu, xd, 31), comb_total = __shfl_sync(0xffffffffu, xc, 31);
    err = __reduce_or_sync(0xffffffffu, err);
    if (have) {
        p.dec_off[lane] = xd - ndec;
        p.unit_off[lane] = 0;
        p.comb_off[lane] = xc - nc;
        p.stg_off[lane] = -1;
        s_off[lane] = xd - ndec;
        s_rq[lane] = make_int4(r.t0, r.Lq, r.Lk, 0);
    }
    if (lane == 0) {
        p.dec_off[p.B] = dec_total;
        p.unit_off[p.B] = 0;
        p.comb_off[p.B] = comb_total;
    }
    __syncwarp();
    const int n_dec = min(dec_total, p.dec_items_cap);
    for (int i = lane; i < n_dec; i += 32) {
        int lo = 0, hi = p.B - 1;  // request owning item i: last b with dec_off[b] <= i
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_off[mid] <= i) lo = mid; else hi = mid - 1;
        }
        const int4 rq = s_rq[lo];
        p.dec_items[i] = make_int4(lo, (int)((unsigned)(i - s_off[lo]) | ((unsigned)rq.y << 27)), rq.x, rq.z);
    }
    if (lane == 0) {
        p.hdr->errors = err;  // this kernel ran every check the block version would
        p.hdr->dec_count = (uint32_t)n_dec;
        p.hdr->pf_count = 0u;
        p.hdr->dec_next = 0u;
        p.hdr->pf_next = 0u;
        p.hdr->comb_tokens = (uint32_t)comb_total;
        p.hdr->stage_pages = 0u;
    }
}

cudaError_t launch_prepass(const Params &p, bool decode_only, cudaStream_t stream)
{
    const cudaError_t e = decode_only && p.B <= kSmallBatch
                              ? launch_pdl(ink_prepass_small_kernel, 1, 32, 0, stream, p)
                              : launch_pdl(ink_prepass_kernel, 1, kPrepassThreads, 0, stream, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace ink
