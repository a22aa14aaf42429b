// ink_decode.cu -- decode / streaming kernel: page gather, bias, masks, online
// softmax, PV and epilogue specialised for requests whose Lq * G packed rows fit
// one 16-row mma block.
//
// Design (GB300):
//  * persistent CTAs, one per SM, take (request, split) items from a
//    device-built list through an atomic counter;
//  * warp 8 is the page-gather producer: for every 16-key group of the item it
//    reads the block_table entry and issues TMA boxes (per KV head and d-half,
//    128-byte swizzle) for K and V, plus one fp32 box of rel_logits per query
//    token when the group lies in the bias band, into a multi-stage ring
//    guarded by mbarriers (paged direct addressing: no gather copy);
//  * warps 0-7 compute.  Warp w serves KV head w % Hkv (GQA packing: the G
//    query heads of every token of the request share one row block, so each
//    K/V byte is read from HBM once) and, when Hkv < 8, one d-slice of the
//    PV product, so no cross-warp merge is needed;
//  * QK^T and PV are bf16 mma.sync m16n8k16 with fp32 accumulation: decode
//    moves ~G flop per byte, far below any tensor-core ridge, so the kernel is
//    bound by HBM and the legacy tensor path is ample;
//  * online softmax in the log2 domain with the bias added after the scale
//    (score = scale * q.k + bias); the result is written directly when the
//    unit has one split, else as an fp32 partial plus its log-sum-exp.
#include "ink_common.cuh"

namespace ink {

constexpr int kDecComputeWarps = 8;
constexpr int kDecThreads = (kDecComputeWarps + 1) * 32;

struct DecItem {
    int b, t0, Lq, Lk;
    int gb, ge;     // 16-key groups of this split
    int split, nact;
    int valid;      // 0: sentinel, no more work
    int index;      // item index (selects the partial block when split)
    int pad[2];
};

struct DecShared {
    uint64_t full[8];
    uint64_t empty[8];
    uint64_t item_full[2];
    uint64_t item_empty[2];
    DecItem item[2];
    int abort;
};

__device__ __forceinline__ int floor4(int x) { return x >= 0 ? (x & ~3) : -(((-x) + 3) & ~3); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Rows of the bias band touched by group gi for query positions [qa0, qa1].
__device__ __forceinline__ bool group_in_band(int qa0, int qa1, int gi, int E)
{
    const int rd_min = qa0 - (gi * kKeyGroup + kKeyGroup - 1);
    const int rd_max = qa1 - gi * kKeyGroup;
    return E > 0 && rd_max >= 0 && rd_min < E;
}

template <int kDSlices>  // d-slices per KV head = 8 / Hkv
__global__ void __launch_bounds__(kDecThreads, 1)
    ink_decode_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_bias,
                      int nstages, int stage_bytes, int kv_bytes, int bias_slot_bytes)
{
    extern __shared__ __align__(1024) uint8_t dsmem[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    DecShared &sh = *reinterpret_cast<DecShared *>(ring + (size_t)nstages * stage_bytes);
    volatile int *abort = &sh.abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int Hkv = p.Hkv, G = p.G, H = p.H;
    const int lq_max = kDecodeRows / G;

    if (threadIdx.x == 0) {
        for (int s = 0; s < nstages; ++s) {
            mbar_init(&sh.full[s], 1);
            mbar_init(&sh.empty[s], kDecComputeWarps);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&sh.item_full[s], 1);
            mbar_init(&sh.item_empty[s], kDecComputeWarps);
        }
        sh.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kDecComputeWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            if (p.bias_tma) prefetch_tmap(&tm_bias);
        }
        const uint64_t pol_kv = policy_evict_first();
        const int total = (int)*(volatile uint32_t *)&p.hdr->dec_count;
        int next = 0;
        if (lane == 0) next = (int)atomicAdd(&p.hdr->dec_next, 1u);
        next = __shfl_sync(0xffffffffu, next, 0);
        uint32_t n = 0;  // stage sequence number
        for (uint32_t iseq = 0;; ++iseq) {
            const int cur = next;
            if (cur < total) {
                if (lane == 0) next = (int)atomicAdd(&p.hdr->dec_next, 1u);
                next = __shfl_sync(0xffffffffu, next, 0);
            }
            const int slot = iseq & 1;
            if (!mbar_wait_warp(&sh.item_empty[slot], ((iseq >> 1) & 1) ^ 1, abort, p)) break;
            DecItem it;
            it.valid = 0;
            if (cur < total) {
                const int2 di = p.dec_items[cur];
                const Req r = load_req(p, di.x);
                const UnitSplit u = unit_split(r.Lk - r.Lq, r.Lk - 1, r.Lk, p.causal, p.wl, p.wr, p.chunk_dec, di.y);
                it.b = di.x; it.t0 = r.t0; it.Lq = r.Lq; it.Lk = r.Lk;
                it.gb = u.gb; it.ge = u.ge; it.split = di.y; it.nact = u.nact; it.valid = 1;
                it.index = cur;
            }
            if (lane == 0) {
                sh.item[slot] = it;
                mbar_arrive(&sh.item_full[slot]);
            }
            if (!it.valid) break;
            const int qa0 = it.Lk - it.Lq, qa1 = it.Lk - 1;
            const int32_t *bt_row = p.bt + (size_t)it.b * p.MAXBLK;
            int pages = -1;
            for (int gi = it.gb; gi < it.ge; ++gi) {
                const int rel = (gi - it.gb) & 31;
                if (rel == 0) {  // 32 groups' page ids at a time, one per lane
                    const int gl = gi + lane;
                    pages = -1;
                    if (gl < it.ge) {
                        const int pid = __ldg(bt_row + (gl * kKeyGroup) / p.BS);
                        pages = (pid >= 0 && pid < p.NB) ? pid : -1;
                        if (pages < 0) report(p, INK_DEVERR_PAGE_ID);
                    }
                }
                const int page = __shfl_sync(0xffffffffu, pages, rel);
                const int stage = n % nstages;
                if (!mbar_wait_warp(&sh.empty[stage], ((n / nstages) & 1) ^ 1, abort, p)) break;
                const bool band = p.bias_tma && group_in_band(qa0, qa1, gi, p.E);
                uint8_t *st = ring + (size_t)stage * stage_bytes;
                if (lane == 0) {
                    const uint32_t bytes = 2u * kv_bytes + (band ? (uint32_t)it.Lq * H * 20 * 4 : 0u);
                    mbar_arrive_expect_tx(&sh.full[stage], bytes);
                }
                __syncwarp();
                // invalid page: an out-of-range key coordinate makes TMA fill zeros
                const int key0 = page >= 0 ? page * p.BS + (gi * kKeyGroup) % p.BS : -kKeyGroup;
                if (lane < 2) {  // one 4-D box per tensor: every KV head and d half of the page
                    tma_load_4d_hint(st + lane * kv_bytes, lane ? &tm_v : &tm_k, 0, key0, 0, 0, &sh.full[stage], pol_kv);
                }
                if (band) {
                    for (int i = lane; i < it.Lq; i += 32) {
                        const int qa = qa0 + i;
                        const int x0 = floor4(qa - (gi * kKeyGroup + kKeyGroup - 1));
                        tma_load_3d(st + 2 * kv_bytes + i * bias_slot_bytes, &tm_bias, x0, 0, it.t0 + i,
                                    &sh.full[stage]);
                    }
                }
                __syncwarp();
                ++n;
            }
            if (*abort) break;
        }
        // let copies still in flight land before the CTA can exit
        for (uint32_t k = (n > (uint32_t)nstages ? n - nstages : 0); k < n; ++k)
            mbar_wait(&sh.full[k % nstages], (k / nstages) & 1, abort, p);
        return;
    }

    // ---------------------------------------------------------------- compute
    const int g = warp % Hkv;
    const int dsl = warp / Hkv;                 // d-slice of this warp
    constexpr int kDW = kHeadDim / kDSlices;    // d width per warp
    constexpr int kNT = kDW / 8;                // n-tiles of 8 in the PV product
    const int d0 = dsl * kDW;
    const float log2e = 1.4426950408889634f;
    const int rA = lane >> 2, rB = rA + 8;      // the two rows this thread holds
    const int cq = (lane & 3) * 2;              // column pair within an 8-wide tile

    uint32_t n = 0;
    for (uint32_t iseq = 0;; ++iseq) {
        const int slot = iseq & 1;
        if (!mbar_wait_warp(&sh.item_full[slot], (iseq >> 1) & 1, abort, p)) break;
        const DecItem it = sh.item[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.item_empty[slot]);
        if (!it.valid) break;

        const int rows = it.Lq * G;
        const int qa0 = it.Lk - it.Lq, qa1 = it.Lk - 1;
        // per-row geometry
        int tokA = rA / G, tokB = rB / G;
        const bool vA = rA < rows, vB = rB < rows;
        const int hA = g * G + rA % G, hB = g * G + rB % G;
        const int qaA = qa0 + tokA, qaB = qa0 + tokB;
        int loA, hiA, loB, hiB;
        visible_range(qaA, qaA, it.Lk, p.causal, p.wl, p.wr, loA, hiA);
        visible_range(qaB, qaB, it.Lk, p.causal, p.wl, p.wr, loB, hiB);
        if (!vA) { loA = 1; hiA = 0; }
        if (!vB) { loB = 1; hiB = 0; }
        int int_lo, int_hi, tmp;
        visible_range(qa1, qa1, it.Lk, p.causal, p.wl, p.wr, int_lo, tmp);
        visible_range(qa0, qa0, it.Lk, p.causal, p.wl, p.wr, tmp, int_hi);

        // Q fragments (A operand): rows rA / rB, 8 k-steps over d
        uint32_t qf[8][4];
        {
            const uint32_t *qa_row = reinterpret_cast<const uint32_t *>(p.q + ((size_t)(it.t0 + tokA) * H + hA) * kHeadDim);
            const uint32_t *qb_row = reinterpret_cast<const uint32_t *>(p.q + ((size_t)(it.t0 + tokB) * H + hB) * kHeadDim);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const int c = (kk * 16 + cq) >> 1;
                qf[kk][0] = vA ? __ldg(qa_row + c) : 0u;
                qf[kk][1] = vB ? __ldg(qb_row + c) : 0u;
                qf[kk][2] = vA ? __ldg(qa_row + c + 4) : 0u;
                qf[kk][3] = vB ? __ldg(qb_row + c + 4) : 0u;
            }
        }
        float o[kNT][4];
#pragma unroll
        for (int j = 0; j < kNT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
        float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
        const float *relA = p.rel ? p.rel + ((size_t)(it.t0 + tokA) * H + hA) * p.E : nullptr;
        const float *relB = p.rel ? p.rel + ((size_t)(it.t0 + tokB) * H + hB) * p.E : nullptr;

        for (int gi = it.gb; gi < it.ge; ++gi, ++n) {
            const int stage = n % nstages;
            if (!mbar_wait_warp(&sh.full[stage], (n / nstages) & 1, abort, p)) break;
            const uint8_t *st = ring + (size_t)stage * stage_bytes;
            const uint32_t kbase = smem_u32(st) + g * 4096;
            const uint32_t vbase = kbase + kv_bytes;

            // S = Q K^T for 16 keys (2 n-tiles)
            float s[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
            {
                const int mi = lane >> 3, rr = lane & 7;
                const int key = rr + 8 * (mi >> 1);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int dh = kk >> 2;
                    const int chunk = ((kk & 3) << 1) + (mi & 1);
                    const uint32_t addr = kbase + dh * 2048 + key * 128 + ((chunk ^ (key & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(addr, b0, b1, b2, b3);
                    mma_bf16(s[0], qf[kk], b0, b1);
                    mma_bf16(s[1], qf[kk], b2, b3);
                }
            }
            // scale into the log2 domain, bias, mask
            const int kbase_key = gi * kKeyGroup;
            const bool band = group_in_band(qa0, qa1, gi, p.E);
            const bool need_mask = (kbase_key < int_lo) || (kbase_key + kKeyGroup - 1 > int_hi);
            const float *bsm = reinterpret_cast<const float *>(st + 2 * kv_bytes);
            float x[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int key = kbase_key + j * 8 + cq + (e & 1);
                    const bool rowB = e >= 2;
                    float v = s[j][e] * p.scale_log2;
                    if (band) {
                        const int qa = rowB ? qaB : qaA;
                        const int rd = qa - key;
                        float bias = 0.f;
                        if (p.bias_tma) {
                            const int tok = rowB ? tokB : tokA;
                            const int h = rowB ? hB : hA;
                            const int x0 = floor4(qa - (kbase_key + kKeyGroup - 1));
                            if ((rowB ? vB : vA))
                                bias = bsm[(tok * bias_slot_bytes) / 4 + h * 20 + (rd - x0)];
                        } else if (rd >= 0 && rd < p.E && (rowB ? vB : vA)) {
                            bias = __ldg((rowB ? relB : relA) + rd);
                        }
                        v = fmaf(bias, log2e, v);
                    }
                    if (need_mask) {
                        const int lo = rowB ? loB : loA, hi = rowB ? hiB : hiA;
                        if (key < lo || key > hi) v = -INFINITY;
                    }
                    x[j][e] = v;
                }
            }
            // online softmax (running max per row; rescale when it grows)
            float tA = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
            float tB = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
            tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, 1));
            tA = fmaxf(tA, __shfl_xor_sync(0xffffffffu, tA, 2));
            tB = fmaxf(tB, __shfl_xor_sync(0xffffffffu, tB, 1));
            tB = fmaxf(tB, __shfl_xor_sync(0xffffffffu, tB, 2));
            if (tA > mA) {
                const float alpha = (mA == -INFINITY) ? 0.f : fast_exp2(mA - tA);
                mA = tA;
                lA *= alpha;
#pragma unroll
                for (int j = 0; j < kNT; ++j) { o[j][0] *= alpha; o[j][1] *= alpha; }
            }
            if (tB > mB) {
                const float alpha = (mB == -INFINITY) ? 0.f : fast_exp2(mB - tB);
                mB = tB;
                lB *= alpha;
#pragma unroll
                for (int j = 0; j < kNT; ++j) { o[j][2] *= alpha; o[j][3] *= alpha; }
            }
            const float subA = (mA == -INFINITY) ? 0.f : mA;
            const float subB = (mB == -INFINITY) ? 0.f : mB;
            float pr[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                pr[j][0] = fast_exp2(x[j][0] - subA);
                pr[j][1] = fast_exp2(x[j][1] - subA);
                pr[j][2] = fast_exp2(x[j][2] - subB);
                pr[j][3] = fast_exp2(x[j][3] - subB);
                lA += pr[j][0] + pr[j][1];
                lB += pr[j][2] + pr[j][3];
            }
            uint32_t pa[4];
            pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
            pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
            pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
            pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);

            // O += P V over this warp's d-slice
            {
                const int tail = it.Lk - kbase_key;  // keys >= tail are beyond the cache length
                const int mi = lane >> 3, rr = lane & 7;
                const int key = rr + 8 * (mi & 1);
#pragma unroll
                for (int jj = 0; jj < kNT / 2; ++jj) {
                    const int dcol = d0 + jj * 16;          // 16 d values = 2 chunks
                    const int dh = dcol >> 6;
                    const int chunk = ((dcol & 63) >> 3) + (mi >> 1);
                    const uint32_t addr = vbase + dh * 2048 + key * 128 + ((chunk ^ (key & 7)) << 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(addr, b0, b1, b2, b3);
                    if (tail < kKeyGroup) {  // zero V entries of keys past the cache length
                        const int k0 = cq, k1 = cq + 8;
                        if (k0 >= tail) { b0 &= 0xffff0000u; b2 &= 0xffff0000u; }
                        if (k0 + 1 >= tail) { b0 &= 0x0000ffffu; b2 &= 0x0000ffffu; }
                        if (k1 >= tail) { b1 &= 0xffff0000u; b3 &= 0xffff0000u; }
                        if (k1 + 1 >= tail) { b1 &= 0x0000ffffu; b3 &= 0x0000ffffu; }
                    }
                    mma_bf16(o[2 * jj], pa, b0, b1);
                    mma_bf16(o[2 * jj + 1], pa, b2, b3);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.empty[stage]);
        }
        if (*abort) break;

        // epilogue
        lA += __shfl_xor_sync(0xffffffffu, lA, 1);
        lA += __shfl_xor_sync(0xffffffffu, lA, 2);
        lB += __shfl_xor_sync(0xffffffffu, lB, 1);
        lB += __shfl_xor_sync(0xffffffffu, lB, 2);
        const float ln2 = 0.6931471805599453f;
        const float invA = lA > 0.f ? 1.f / lA : 0.f;
        const float invB = lB > 0.f ? 1.f / lB : 0.f;
        const float lseA = lA > 0.f ? (mA + __log2f(lA)) * ln2 : -INFINITY;
        const float lseB = lB > 0.f ? (mB + __log2f(lB)) * ln2 : -INFINITY;
        const size_t rowA = (size_t)(it.t0 + tokA) * H + hA;
        const size_t rowB = (size_t)(it.t0 + tokB) * H + hB;
        if (it.nact == 1) {
#pragma unroll
            for (int j = 0; j < kNT; ++j) {
                const int d = d0 + j * 8 + cq;
                if (vA) *reinterpret_cast<uint32_t *>(p.out + rowA * kHeadDim + d) = pack_bf16x2(o[j][0] * invA, o[j][1] * invA);
                if (vB) *reinterpret_cast<uint32_t *>(p.out + rowB * kHeadDim + d) = pack_bf16x2(o[j][2] * invB, o[j][3] * invB);
            }
            if (p.lse && dsl == 0 && (lane & 3) == 0) {
                if (vA) p.lse[rowA] = lseA;
                if (vB) p.lse[rowB] = lseB;
            }
        } else {
            // partial block of this item: rows (token i, head h) -> i * H + h
            const size_t blk = (size_t)it.index * p.dec_rows;
            const size_t pA = blk + (size_t)tokA * H + hA, pB = blk + (size_t)tokB * H + hB;
#pragma unroll
            for (int j = 0; j < kNT; ++j) {
                const int d = d0 + j * 8 + cq;
                if (vA) *reinterpret_cast<float2 *>(p.part_dec_o + pA * kHeadDim + d) = make_float2(o[j][0] * invA, o[j][1] * invA);
                if (vB) *reinterpret_cast<float2 *>(p.part_dec_o + pB * kHeadDim + d) = make_float2(o[j][2] * invB, o[j][3] * invB);
            }
            if (dsl == 0 && (lane & 3) == 0) {
                if (vA) p.part_dec_lse[pA] = lseA;
                if (vB) p.part_dec_lse[pB] = lseB;
            }
        }
    }
}

cudaError_t launch_decode(const Params &p, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                          const CUtensorMap &tm_bias, int nstages, int stage_bytes, int kv_bytes,
                          int bias_slot_bytes, int grid, size_t smem, cudaStream_t stream)
{
    auto go = [&](auto kernel) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kernel<<<grid, kDecThreads, smem, stream>>>(p, tm_k, tm_v, tm_bias, nstages, stage_bytes, kv_bytes,
                                                    bias_slot_bytes);
        return cudaGetLastError();
    };
    switch (8 / p.Hkv) {
        case 1: return go(ink_decode_kernel<1>);
        case 2: return go(ink_decode_kernel<2>);
        case 4: return go(ink_decode_kernel<4>);
        default: return go(ink_decode_kernel<8>);
    }
}

}  // namespace ink
