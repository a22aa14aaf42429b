// ink_decode.cu -- decode / streaming kernel: page gather, bias, masks, online
// softmax, PV and epilogue specialised for requests whose Lq * G packed rows fit
// one 16-row mma block.
//
// Design (GB300):
//  * persistent CTAs, one per SM, take (request, split) items from a
//    device-built list through an atomic counter;
//  * warp 8 is the page-gather producer: for every 16-key group of the item it
//    reads the block_table entry and issues one 4-D TMA box per tensor (every
//    KV head and d half of the page, 128-byte swizzle) for K and V, plus one
//    fp32 box of rel_logits per query token when the group lies in the bias
//    band, into a multi-stage ring guarded by mbarriers (paged direct
//    addressing: no gather copy);
//  * warps 0-7 compute.  Warp w serves KV head w % Hkv (GQA packing: the G
//    query heads of every token of the request share one row block, so each
//    K/V byte is read from HBM once) and, when Hkv < 8, one d-slice of the
//    PV product, so no cross-warp merge is needed;
//  * QK^T and PV are mma.sync m16n8k16 with fp32 accumulation: decode moves
//    ~G flop per byte, far below any tensor-core ridge, so the kernel is bound
//    by HBM and the legacy tensor path is ample.  Items with at most 8 packed
//    rows compute the transposes (S^T = K Q^T, O^T += V^T P^T) so that the 16
//    keys of a page fill the mma's M and the rows its N = 8, half the work of
//    the 16-row block; with a ring of at least 4 stages they take two pages
//    per step;
//  * online softmax in the log2 domain with the bias added after the scale
//    (score = scale * q.k + bias); the result is written directly when the
//    unit has one split, else as an fp32 partial plus its log-sum-exp.
//
// FP8 KV cache (kFp8): pages hold E4M3 bytes, one 2 KB [16 keys][128 B] block
// per KV head and tensor, and K = k_scale * E4M3, V = v_scale * E4M3.  Every
// E4M3 value is exact in fp16, so the products run as f16 mma.sync with fp32
// accumulation (q converted from bf16 to fp16 once per item, p in fp16):
//  * QK^T: ldmatrix reads the E4M3 key rows as they landed; a thread's
//    register holds 4 consecutive bytes (d = 16 kk + 4 c .. + 3 of k-step kk),
//    converted in registers to two f16 pairs of its K fragment.  q's fragment
//    uses the same order of d within each k-step, so the dot product is
//    unchanged;
//  * PV: a transposed ldmatrix over the E4M3 V rows read as byte pairs gives a
//    thread two keys at two adjacent d; the even bytes are the operand of the
//    tile holding even d, the odd bytes that of the tile holding odd d, so no
//    conversion pass through shared memory is needed;
//  * k_scale joins the softmax scale and v_scale the final normalisation.
#include <type_traits>

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

__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 matrix of 16-bit pairs held in the mma fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t r;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

// Two E4M3 bytes (low byte first) to an f16 pair (low half first); exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two)
{
    uint32_t r;
    const uint16_t h = (uint16_t)(two & 0xffffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
    return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// A bf16 pair to an f16 pair (exact for magnitudes in [2^-14, 65504]).
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t u)
{
    return pack_f16x2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// E4M3 bytes 0 and 2 (even) or 1 and 3 (odd) of a word as an f16 pair.  ldmatrix.trans over E4M3 rows read as
// 16-bit pairs gives a thread keys k, k + 1 at two adjacent d (bytes: [k][d], [k][d+1], [k+1][d], [k+1][d+1]);
// the even bytes are the (k, k + 1) pair at d, the odd bytes the pair at d + 1.
__device__ __forceinline__ uint32_t e4m3_even_f16x2(uint32_t w) { return e4m3x2_to_f16x2(__byte_perm(w, 0u, 0x0020)); }
__device__ __forceinline__ uint32_t e4m3_odd_f16x2(uint32_t w) { return e4m3x2_to_f16x2(__byte_perm(w, 0u, 0x0031)); }

// Zero the halves of a key-pair register (keys k, k + 1) whose keys are at or past `tail`.
__device__ __forceinline__ void mask_key_pair(uint32_t &x, int k, int tail)
{
    if (k >= tail) x &= 0xffff0000u;
    if (k + 1 >= tail) x &= 0x0000ffffu;
}

// Rows of the bias band touched by group gi for query positions [qa0, qa1].
__device__ __forceinline__ bool group_in_band(int qa0, int qa1, int gi, int E)
{
    const int rd_min = qa0 - (gi * kKeyGroup + kKeyGroup - 1);
    const int rd_max = qa1 - gi * kKeyGroup;
    return E > 0 && rd_max >= 0 && rd_min < E;
}

// kD: head size (64, 128 or 256; E4M3 pages at 128 only); kDSlices: d-slices per KV head = 8 / Hkv; kFp8:
// E4M3 K/V pages; kPerSm: CTAs an SM (2: half the shared memory and registers each, twice the warps to hide
// the per-page dependency chain); kSmall: every item of the call has at most 8 packed rows, so the 16-row
// path is left out (fewer registers); kOneTok: every decode-shaped request has one query token (max_seqlen_q
// 1), so a thread's rows share their token, position and visible range
template <int kD, int kDSlices, bool kFp8, int kPerSm, bool kSmall, bool kOneTok>
__global__ void __launch_bounds__(kDecThreads, kPerSm)
    ink_decode_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_bias,
                      int nstages, int stage_bytes, int kv_bytes, int bias_slot_bytes, float k_scale,
                      float v_scale)
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
    // The work list and (for a staged call) the staging copy are complete after the wait.  In a decode-only
    // call of at most 32 requests the producer waits only after its first item, whose pages stream while the
    // prepass runs; the compute warps read nothing the prepass writes.  Dependents launch only after a wait,
    // so a kernel that follows can rely on the prepass's outputs.
    if (!p.dec_local) {
        pdl_wait();
        pdl_launch_dependents();
    }

    if (warp == kDecComputeWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            if (p.bias_tma) prefetch_tmap(&tm_bias);
        }
        const uint64_t pol_kv = policy_evict_first();
        // CTA c takes item c first and then items gridDim.x + k in the order of the shared counter, so
        // the first item needs no atomic; its entry is read speculatively beside the item count.
        int total = 0, next = blockIdx.x;
        int4 di_next = make_int4(0, 0, 0, 0);
        bool waited = !p.dec_local;
        uint32_t held_err = 0;  // page-id errors found before the wait (the prepass rewrites the error word)
        if (p.dec_local) {
            // item c from the inputs, by the prepass's own rule: requests in order, each cut by unit_split,
            // item c owned by the last request whose first item is at or before c
            const Req r = lane < p.B ? load_req(p, lane) : Req{};
            const int na = (lane < p.B && r.ok && r.Lq > 0)
                               ? unit_split(r.Lk - r.Lq, r.Lk - 1, r.Lk, p.causal, p.wl, p.wr, p.chunk_dec, 0).nact
                               : 0;
            int x = na;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            const int off = x - na;
            total = min(__shfl_sync(0xffffffffu, x, 31), p.dec_items_cap);
            const unsigned own = __ballot_sync(0xffffffffu, lane < p.B && off <= next);
            const int b = own ? 31 - __clz(own) : 0;
            const int split = next - __shfl_sync(0xffffffffu, off, b);
            const int t0 = __shfl_sync(0xffffffffu, r.t0, b), lq = __shfl_sync(0xffffffffu, r.Lq, b);
            const int lk = __shfl_sync(0xffffffffu, r.Lk, b);
            if (next < total) di_next = make_int4(b, (int)((unsigned)split | ((unsigned)lq << 27)), t0, lk);
        } else {
            total = (int)*(volatile uint32_t *)&p.hdr->dec_count;
            if (next < p.dec_items_cap) di_next = p.dec_items[next];
        }
        // the plan's queue: the next item after a wait on the prepass
        auto claim_next = [&](int cur) {
            if (cur < total) {
                if (lane == 0) next = (int)gridDim.x + (int)atomicAdd(&p.hdr->dec_next, 1u);
                next = __shfl_sync(0xffffffffu, next, 0);
                if (next < total) di_next = p.dec_items[next];
            }
        };
        uint32_t n = 0;  // stage sequence number
        for (uint32_t iseq = 0;; ++iseq) {
            const int cur = next;
            const int4 di = di_next;
            if (waited) claim_next(cur);
            const int slot = iseq & 1;
            if (!mbar_wait_warp(&sh.item_empty[slot], ((iseq >> 1) & 1) ^ 1, abort, p)) break;
            DecItem it;
            it.valid = 0;
            if (cur < total) {
                const int split = di.y & ((1 << 27) - 1), Lq = (int)((unsigned)di.y >> 27);
                const UnitSplit u = unit_split(di.w - Lq, di.w - 1, di.w, p.causal, p.wl, p.wr, p.chunk_dec, split);
                it.b = di.x; it.t0 = di.z; it.Lq = Lq; it.Lk = di.w;
                it.gb = u.gb; it.ge = u.ge; it.split = split; it.nact = u.nact; it.valid = 1;
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
                        if (pages < 0) {
                            if (waited) report(p, INK_DEVERR_PAGE_ID);
                            else held_err |= INK_DEVERR_PAGE_ID;
                        }
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
            if (!waited) {  // first item issued: from here on the prepass's plan is needed
                pdl_wait();
                pdl_launch_dependents();
                waited = true;
                if (held_err) report(p, held_err);
                claim_next(cur);
            }
        }
        if (!waited) pdl_wait();  // this CTA ends only after the prepass, so that kernels after it can rely on it
        // let copies still in flight land before the CTA can exit
        for (uint32_t k = (n > (uint32_t)nstages ? n - nstages : 0); k < n; ++k)
            mbar_wait(&sh.full[k % nstages], (k / nstages) & 1, abort, p);
        return;
    }

    // ---------------------------------------------------------------- compute
    const int g = warp % Hkv;
    const int dsl = warp / Hkv;                 // d-slice of this warp
    static_assert(!kFp8 || kD == 128, "E4M3 pages are read at head size 128 only");
    constexpr int kDW = kD / kDSlices;          // d width per warp
    static_assert(kDW >= 16, "a warp's d-slice is at least one 16-wide mma tile");
    constexpr int kKSteps = kD / 16;            // k-steps of 16 d in QK^T
    // a stage holds, per tensor and KV head, kD / 64 blocks of [16 keys][64 d] (128-byte swizzled rows);
    // E4M3: one [16 keys][128 B] block
    constexpr int kHeadBytes = kFp8 ? 2048 : kD * 32;
    constexpr int kNT = kDW / 8;                // n-tiles of 8 in the PV product
    const int d0 = dsl * kDW;
    const float log2e = 1.4426950408889634f;
    const int rA = lane >> 2, rB = rA + 8;      // the two rows this thread holds
    const int cq = (lane & 3) * 2;              // column pair within an 8-wide tile
    const int c4 = (lane & 3) * 4;              // FP8: first of the 4 d values of a k-step a thread holds
    const float scale_log2 = kFp8 ? p.scale_log2 * k_scale : p.scale_log2;
    // FP8 V: 32-d blocks of this warp's d-slice read per ldmatrix.trans, and the offset of a block's second
    // 16 d (0 when the slice is only 16 d wide: the second half then repeats the first and is not used)
    constexpr int kVB = kDW >= 32 ? kDW / 32 : 1;
    constexpr int kDSec = kDW >= 32 ? 16 : 0;
    uint32_t n = 0;
    for (uint32_t iseq = 0;; ++iseq) {
        const int slot = iseq & 1;
        if (!mbar_wait_warp(&sh.item_full[slot], (iseq >> 1) & 1, abort, p)) break;
        const DecItem it = sh.item[slot];
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh.item_empty[slot]);
        if (!it.valid) break;

        const int rows = kOneTok ? G : it.Lq * G;
        const int qa0 = it.Lk - (kOneTok ? 1 : it.Lq), qa1 = it.Lk - 1;

        if (kSmall || rows <= 8) {
            // ---- at most 8 packed rows: S^T = K Q^T and O^T += V^T P^T, so the 16 keys of a page fill
            // the mma's M and the rows its N = 8 (half the mma and softmax work of the 16-row block).
            // Fragments: this thread's S^T / O^T accumulators hold rows 2t and 2t + 1 at keys (or d)
            // gq and gq + 8; its Q^T and P^T fragments hold row gq.
            const int gq = lane >> 2, t = lane & 3;
            const int r0 = 2 * t, r1 = 2 * t + 1;
            const bool v0 = r0 < rows, v1 = r1 < rows, vq = gq < rows;
            const int tok0 = kOneTok ? 0 : r0 / G, tok1 = kOneTok ? 0 : r1 / G, tokq = kOneTok ? 0 : gq / G;
            const int h0 = g * G + (kOneTok ? r0 : r0 % G), h1 = g * G + (kOneTok ? r1 : r1 % G);
            const int hq = g * G + (kOneTok ? gq : gq % G);
            const int qa_0 = qa0 + tok0, qa_1 = qa0 + tok1;
            int lo0, hi0, lo1, hi1, nlo, nhi, tmp;
            visible_range(qa_0, qa_0, it.Lk, p.causal, p.wl, p.wr, lo0, hi0);
            visible_range(qa_1, qa_1, it.Lk, p.causal, p.wl, p.wr, lo1, hi1);
            if (!v0) { lo0 = 1; hi0 = 0; }
            if (!v1) { lo1 = 1; hi1 = 0; }
            visible_range(qa1, qa1, it.Lk, p.causal, p.wl, p.wr, nlo, tmp);
            visible_range(qa0, qa0, it.Lk, p.causal, p.wl, p.wr, tmp, nhi);

            // Q^T fragments (B operand) of row gq, 8 k-steps over d
            uint32_t qb[kKSteps][2];
            {
                const uint32_t *q_row =
                    reinterpret_cast<const uint32_t *>(p.q + ((size_t)(it.t0 + tokq) * H + hq) * kD);
#pragma unroll
                for (int kk = 0; kk < kKSteps; ++kk) {
                    if constexpr (kFp8) {  // d = 16 kk + 4t + {0,1} and + {2,3}: the E4M3 rows' order
                        const uint2 u = vq ? __ldg(reinterpret_cast<const uint2 *>(q_row + 8 * kk + 2 * t))
                                           : make_uint2(0u, 0u);
                        qb[kk][0] = bf16x2_to_f16x2(u.x);
                        qb[kk][1] = bf16x2_to_f16x2(u.y);
                    } else {
                        qb[kk][0] = vq ? __ldg(q_row + 8 * kk + t) : 0u;
                        qb[kk][1] = vq ? __ldg(q_row + 8 * kk + t + 4) : 0u;
                    }
                }
            }
            // m-tiles (16 rows of O^T) of this warp's slice in the PV product; E4M3: tile 2vb holds d = D + 2gq
            // (+ 16) of 32-d block vb at D, tile 2vb + 1 the odd d next to them
            constexpr int kMT = kFp8 ? 2 * kVB : kDW / 16;
            float o[kMT][4];
#pragma unroll
            for (int mt = 0; mt < kMT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
            float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
            const float *rel0 = p.rel ? p.rel + ((size_t)(it.t0 + tok0) * H + h0) * p.E : nullptr;
            const float *rel1 = p.rel ? p.rel + ((size_t)(it.t0 + tok1) * H + h1) * p.E : nullptr;
            const int lkey = (lane & 7) + 8 * ((lane >> 3) & 1);  // ldmatrix row of this lane (K)

            // S^T of one page (16 keys x 8 rows); even and odd k-steps in two accumulators (shorter chains)
            auto qk_page = [&](uint32_t kbase, float (&sc)[4]) {
                float sd[4] = {0.f, 0.f, 0.f, 0.f};
                sc[0] = sc[1] = sc[2] = sc[3] = 0.f;
                if constexpr (kFp8) {
#pragma unroll
                    for (int kp = 0; kp < 4; ++kp) {  // k-steps 2kp, 2kp + 1: E4M3 chunks 2kp + (lane >> 4)
                        const int chunk = 2 * kp + (lane >> 4);
                        uint32_t r[4];
                        ldsm_x4(kbase + lkey * 128 + ((chunk ^ (lkey & 7)) << 4), r[0], r[1], r[2], r[3]);
                        const uint32_t a0[4] = {e4m3x2_to_f16x2(r[0]), e4m3x2_to_f16x2(r[1]),
                                                e4m3x2_to_f16x2(r[0] >> 16), e4m3x2_to_f16x2(r[1] >> 16)};
                        mma_f16(sc, a0, qb[2 * kp][0], qb[2 * kp][1]);
                        const uint32_t a1[4] = {e4m3x2_to_f16x2(r[2]), e4m3x2_to_f16x2(r[3]),
                                                e4m3x2_to_f16x2(r[2] >> 16), e4m3x2_to_f16x2(r[3] >> 16)};
                        mma_f16(sd, a1, qb[2 * kp + 1][0], qb[2 * kp + 1][1]);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < kKSteps; ++kk) {
                        const int chunk = ((kk & 3) << 1) + (lane >> 4);
                        uint32_t a[4];
                        ldsm_x4(kbase + (kk >> 2) * 2048 + lkey * 128 + ((chunk ^ (lkey & 7)) << 4), a[0], a[1],
                                a[2], a[3]);
                        mma_bf16((kk & 1) ? sd : sc, a, qb[kk][0], qb[kk][1]);
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[e] += sd[e];
            };
            // scale into the log2 domain, bias, masks: x[e] is row (e & 1 ? r1 : r0) at key gq + 8 (e >> 1)
            auto score_page = [&](int gi, const uint8_t *st, const float (&sc)[4], float (&x)[4]) {
                const int kbase_key = gi * kKeyGroup;
                const bool band = group_in_band(qa0, qa1, gi, p.E);
                const bool need_mask = (kbase_key < nlo) || (kbase_key + kKeyGroup - 1 > nhi);
                const float *bsm = reinterpret_cast<const float *>(st + 2 * kv_bytes);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const bool second = e & 1;
                    const int key = kbase_key + gq + 8 * (e >> 1);
                    float v = sc[e] * scale_log2;
                    if (band) {
                        const int qa = second ? qa_1 : qa_0;
                        const int rd = qa - key;
                        float bias = 0.f;
                        if (kPerSm == 2 || p.bias_tma) {  // two an SM: launched only with the bias by TMA
                            const int x0 = floor4(qa - (kbase_key + kKeyGroup - 1));
                            if (second ? v1 : v0)
                                bias = bsm[((second ? tok1 : tok0) * bias_slot_bytes) / 4 + (second ? h1 : h0) * 20 +
                                           (rd - x0)];
                        } else if (rd >= 0 && rd < p.E && (second ? v1 : v0)) {
                            bias = __ldg((second ? rel1 : rel0) + rd);
                        }
                        v = fmaf(bias, log2e, v);
                    }
                    if (need_mask) {
                        const int lo = second ? lo1 : lo0, hi = second ? hi1 : hi0;
                        if (key < lo || key > hi) v = -INFINITY;
                    }
                    x[e] = v;
                }
            };
            // O^T += V^T P^T of one page over this warp's d-slice; keys >= tail are beyond the cache length
            auto pv_page = [&](uint32_t vbase, uint32_t pb0, uint32_t pb1, int tail) {
                if constexpr (kFp8) {
                    // E4M3 V^T operands straight from the landed rows: matrices (keys 0-7 | 8-15) x (d D | D + 16)
                    const int vkey = (lane & 7) + 8 * (lane >> 4);
#pragma unroll
                    for (int vb = 0; vb < kVB; ++vb) {
                        const int chunk = (d0 + 32 * vb + ((lane >> 3) & 1) * kDSec) >> 4;
                        uint32_t r[4];
                        ldsm_x4_t(vbase + vkey * 128 + ((chunk ^ (vkey & 7)) << 4), r[0], r[1], r[2], r[3]);
                        if (tail < kKeyGroup) {
                            mask_key_pair(r[0], 2 * t, tail);
                            mask_key_pair(r[1], 2 * t, tail);
                            mask_key_pair(r[2], 2 * t + 8, tail);
                            mask_key_pair(r[3], 2 * t + 8, tail);
                        }
                        const uint32_t ae[4] = {e4m3_even_f16x2(r[0]), e4m3_even_f16x2(r[1]), e4m3_even_f16x2(r[2]),
                                                e4m3_even_f16x2(r[3])};
                        const uint32_t ao[4] = {e4m3_odd_f16x2(r[0]), e4m3_odd_f16x2(r[1]), e4m3_odd_f16x2(r[2]),
                                                e4m3_odd_f16x2(r[3])};
                        mma_f16(o[2 * vb], ae, pb0, pb1);
                        mma_f16(o[2 * vb + 1], ao, pb0, pb1);
                    }
                } else {  // one m-tile of 16 d at a time
                    const int vkey = (lane & 7) + 8 * (lane >> 4);
#pragma unroll
                    for (int mt = 0; mt < kMT; ++mt) {
                        const int d = d0 + 16 * mt;
                        const int chunk = ((d & 63) >> 3) + ((lane >> 3) & 1);
                        uint32_t a[4];
                        ldsm_x4_t(vbase + (d >> 6) * 2048 + vkey * 128 + ((chunk ^ (vkey & 7)) << 4), a[0], a[1],
                                  a[2], a[3]);
                        if (tail < kKeyGroup) {
                            mask_key_pair(a[0], 2 * t, tail);
                            mask_key_pair(a[1], 2 * t, tail);
                            mask_key_pair(a[2], 2 * t + 8, tail);
                            mask_key_pair(a[3], 2 * t + 8, tail);
                        }
                        mma_bf16(o[mt], a, pb0, pb1);
                    }
                }
            };

            // two pages per step when the ring is deep enough to hold two and still prefetch (at least 4
            // stages): two independent QK chains, and one max exchange and rescale decision per 32 keys
            const bool pair_pages = kPerSm == 1 && nstages >= 4;
            for (int gi = it.gb; gi < it.ge;) {
                const bool two = pair_pages && gi + 1 < it.ge;
                const int sa = n % nstages, sb = (n + 1) % nstages;
                if (!mbar_wait_warp(&sh.full[sa], (n / nstages) & 1, abort, p)) break;
                if (two && !mbar_wait_warp(&sh.full[sb], ((n + 1) / nstages) & 1, abort, p)) break;
                const uint8_t *stA = ring + (size_t)sa * stage_bytes, *stB = ring + (size_t)sb * stage_bytes;
                const uint32_t kA = smem_u32(stA) + g * kHeadBytes;
                const uint32_t kB = smem_u32(stB) + g * kHeadBytes;
                float scA[4], scB[4], xA[4], xB[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                qk_page(kA, scA);
                if (two) qk_page(kB, scB);
                score_page(gi, stA, scA, xA);
                if (two) score_page(gi + 1, stB, scB, xB);

                // row maxima over the step: this thread's keys, then the 8 lanes with the same t
                float t0 = fmaxf(fmaxf(xA[0], xA[2]), fmaxf(xB[0], xB[2]));
                float t1 = fmaxf(fmaxf(xA[1], xA[3]), fmaxf(xB[1], xB[3]));
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    t0 = fmaxf(t0, __shfl_xor_sync(0xffffffffu, t0, off));
                    t1 = fmaxf(t1, __shfl_xor_sync(0xffffffffu, t1, off));
                }
                if (t0 > m0) {
                    const float alpha = (m0 == -INFINITY) ? 0.f : fast_exp2(m0 - t0);
                    m0 = t0;
                    l0 *= alpha;
#pragma unroll
                    for (int mt = 0; mt < kMT; ++mt) { o[mt][0] *= alpha; o[mt][2] *= alpha; }
                }
                if (t1 > m1) {
                    const float alpha = (m1 == -INFINITY) ? 0.f : fast_exp2(m1 - t1);
                    m1 = t1;
                    l1 *= alpha;
#pragma unroll
                    for (int mt = 0; mt < kMT; ++mt) { o[mt][1] *= alpha; o[mt][3] *= alpha; }
                }
                const float sub0 = (m0 == -INFINITY) ? 0.f : m0;
                const float sub1 = (m1 == -INFINITY) ? 0.f : m1;
                float pA[4], pB[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    pA[e] = fast_exp2(xA[e] - ((e & 1) ? sub1 : sub0));
                    pB[e] = fast_exp2(xB[e] - ((e & 1) ? sub1 : sub0));
                }
                l0 += (pA[0] + pA[2]) + (pB[0] + pB[2]);
                l1 += (pA[1] + pA[3]) + (pB[1] + pB[3]);
                // P^T fragments (B operand of PV): each page's two 8-key blocks of P, transposed in registers
                const uint32_t pa0 = movmatrix_trans(kFp8 ? pack_f16x2(pA[0], pA[1]) : pack_bf16x2(pA[0], pA[1]));
                const uint32_t pa1 = movmatrix_trans(kFp8 ? pack_f16x2(pA[2], pA[3]) : pack_bf16x2(pA[2], pA[3]));
                pv_page(kA + kv_bytes, pa0, pa1, it.Lk - gi * kKeyGroup);
                if (two) {
                    const uint32_t pc0 = movmatrix_trans(kFp8 ? pack_f16x2(pB[0], pB[1]) : pack_bf16x2(pB[0], pB[1]));
                    const uint32_t pc1 = movmatrix_trans(kFp8 ? pack_f16x2(pB[2], pB[3]) : pack_bf16x2(pB[2], pB[3]));
                    pv_page(kB + kv_bytes, pc0, pc1, it.Lk - (gi + 1) * kKeyGroup);
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&sh.empty[sa]);
                    if (two) mbar_arrive(&sh.empty[sb]);
                }
                n += two ? 2 : 1;
                gi += two ? 2 : 1;
            }
            if (*abort) break;

            // epilogue: row sums over the 8 lanes that share t, then rows r0 / r1 at d = d0 + 16 mt + gq (+ 8)
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                l0 += __shfl_xor_sync(0xffffffffu, l0, off);
                l1 += __shfl_xor_sync(0xffffffffu, l1, off);
            }
            const float ln2 = 0.6931471805599453f;
            float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
            if constexpr (kFp8) {
                inv0 *= v_scale;
                inv1 *= v_scale;
            }
            const float lse0 = l0 > 0.f ? (m0 + __log2f(l0)) * ln2 : -INFINITY;
            const float lse1 = l1 > 0.f ? (m1 + __log2f(l1)) * ln2 : -INFINITY;
            const size_t row0 = (size_t)(it.t0 + tok0) * H + h0, row1 = (size_t)(it.t0 + tok1) * H + h1;
            if constexpr (kFp8) {  // tiles 2vb / 2vb + 1: the even / odd d of pair gq, at D and D + 16
                const size_t blk = (size_t)it.index * p.dec_rows;
                const size_t pr0 = blk + (size_t)tok0 * H + h0, pr1 = blk + (size_t)tok1 * H + h1;
#pragma unroll
                for (int vb = 0; vb < kVB; ++vb) {
#pragma unroll
                    for (int sec = 0; sec < (kDSec ? 2 : 1); ++sec) {
                        const int d = d0 + 32 * vb + 16 * sec + 2 * gq;
                        const float e0 = o[2 * vb][2 * sec] * inv0, f0 = o[2 * vb + 1][2 * sec] * inv0;
                        const float e1 = o[2 * vb][2 * sec + 1] * inv1, f1 = o[2 * vb + 1][2 * sec + 1] * inv1;
                        if (it.nact == 1) {
                            if (v0) *reinterpret_cast<uint32_t *>(p.out + row0 * kD + d) = pack_bf16x2(e0, f0);
                            if (v1) *reinterpret_cast<uint32_t *>(p.out + row1 * kD + d) = pack_bf16x2(e1, f1);
                        } else {
                            if (v0) *reinterpret_cast<float2 *>(p.part_dec_o + pr0 * kD + d) = make_float2(e0, f0);
                            if (v1) *reinterpret_cast<float2 *>(p.part_dec_o + pr1 * kD + d) = make_float2(e1, f1);
                        }
                    }
                }
                if (dsl == 0 && gq == 0) {
                    if (it.nact == 1) {
                        if (p.lse && v0) p.lse[row0] = lse0;
                        if (p.lse && v1) p.lse[row1] = lse1;
                    } else {
                        if (v0) p.part_dec_lse[pr0] = lse0;
                        if (v1) p.part_dec_lse[pr1] = lse1;
                    }
                }
            } else if (it.nact == 1) {
#pragma unroll
                for (int mt = 0; mt < kMT; ++mt) {
                    const int d = d0 + 16 * mt + gq;
                    if (v0) {
                        p.out[row0 * kD + d] = __float2bfloat16_rn(o[mt][0] * inv0);
                        p.out[row0 * kD + d + 8] = __float2bfloat16_rn(o[mt][2] * inv0);
                    }
                    if (v1) {
                        p.out[row1 * kD + d] = __float2bfloat16_rn(o[mt][1] * inv1);
                        p.out[row1 * kD + d + 8] = __float2bfloat16_rn(o[mt][3] * inv1);
                    }
                }
                if (p.lse && dsl == 0 && gq == 0) {
                    if (v0) p.lse[row0] = lse0;
                    if (v1) p.lse[row1] = lse1;
                }
            } else {
                const size_t blk = (size_t)it.index * p.dec_rows;
                const size_t pr0 = blk + (size_t)tok0 * H + h0, pr1 = blk + (size_t)tok1 * H + h1;
#pragma unroll
                for (int mt = 0; mt < kMT; ++mt) {
                    const int d = d0 + 16 * mt + gq;
                    if (v0) {
                        p.part_dec_o[pr0 * kD + d] = o[mt][0] * inv0;
                        p.part_dec_o[pr0 * kD + d + 8] = o[mt][2] * inv0;
                    }
                    if (v1) {
                        p.part_dec_o[pr1 * kD + d] = o[mt][1] * inv1;
                        p.part_dec_o[pr1 * kD + d + 8] = o[mt][3] * inv1;
                    }
                }
                if (dsl == 0 && gq == 0) {
                    if (v0) p.part_dec_lse[pr0] = lse0;
                    if (v1) p.part_dec_lse[pr1] = lse1;
                }
            }
            continue;
        }

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
        uint32_t qf[kKSteps][4];
        {
            const uint32_t *qa_row = reinterpret_cast<const uint32_t *>(p.q + ((size_t)(it.t0 + tokA) * H + hA) * kD);
            const uint32_t *qb_row = reinterpret_cast<const uint32_t *>(p.q + ((size_t)(it.t0 + tokB) * H + hB) * kD);
            if constexpr (kFp8) {
                // fp16, d = 16 kk + c4 + {0,1} in a0 / a1 and + {2,3} in a2 / a3 (the key rows' order)
#pragma unroll
                for (int kk = 0; kk < kKSteps; ++kk) {
                    const int c = (kk * 16 + c4) >> 1;
                    const uint2 ua = vA ? __ldg(reinterpret_cast<const uint2 *>(qa_row + c)) : make_uint2(0u, 0u);
                    const uint2 ub = vB ? __ldg(reinterpret_cast<const uint2 *>(qb_row + c)) : make_uint2(0u, 0u);
                    qf[kk][0] = bf16x2_to_f16x2(ua.x);
                    qf[kk][1] = bf16x2_to_f16x2(ub.x);
                    qf[kk][2] = bf16x2_to_f16x2(ua.y);
                    qf[kk][3] = bf16x2_to_f16x2(ub.y);
                }
            } else {
#pragma unroll
                for (int kk = 0; kk < kKSteps; ++kk) {
                    const int c = (kk * 16 + cq) >> 1;
                    qf[kk][0] = vA ? __ldg(qa_row + c) : 0u;
                    qf[kk][1] = vB ? __ldg(qb_row + c) : 0u;
                    qf[kk][2] = vA ? __ldg(qa_row + c + 4) : 0u;
                    qf[kk][3] = vB ? __ldg(qb_row + c + 4) : 0u;
                }
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
            const uint32_t kbase = smem_u32(st) + g * kHeadBytes;
            const uint32_t vbase = kbase + kv_bytes;

            // S = Q K^T for 16 keys (2 n-tiles)
            float s[2][4];
#pragma unroll
            for (int j = 0; j < 2; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
            if constexpr (kFp8) {
                const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int key = rr + 8 * j;
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int chunk = 4 * h + mi;  // matrix mi = 16-d chunk 4h + mi = k-step
                        uint32_t r[4];
                        ldsm_x4(kbase + key * 128 + ((chunk ^ (key & 7)) << 4), r[0], r[1], r[2], r[3]);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            mma_f16(s[j], qf[4 * h + i], e4m3x2_to_f16x2(r[i]), e4m3x2_to_f16x2(r[i] >> 16));
                    }
                }
            } else {
                const int mi = lane >> 3, rr = lane & 7;
                const int key = rr + 8 * (mi >> 1);
#pragma unroll
                for (int kk = 0; kk < kKSteps; ++kk) {
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
                    float v = s[j][e] * scale_log2;
                    if (band) {
                        const int qa = rowB ? qaB : qaA;
                        const int rd = qa - key;
                        float bias = 0.f;
                        if (kPerSm == 2 || p.bias_tma) {
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
            if constexpr (kFp8) {
                pa[0] = pack_f16x2(pr[0][0], pr[0][1]);
                pa[1] = pack_f16x2(pr[0][2], pr[0][3]);
                pa[2] = pack_f16x2(pr[1][0], pr[1][1]);
                pa[3] = pack_f16x2(pr[1][2], pr[1][3]);
            } else {
                pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
                pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
                pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
                pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
            }

            // O += P V over this warp's d-slice
            if constexpr (kFp8) {
                // E4M3 V operands straight from the landed rows: matrices (keys 0-7 | 8-15) x (d D | D + 16);
                // n-tile 4vb (+2 for D + 16) holds d = D + 2n, n-tile 4vb + 1 (+2) holds d = D + 2n + 1
                const int tail = it.Lk - kbase_key;
                const int vkey = (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
                for (int vb = 0; vb < kVB; ++vb) {
                    const int chunk = (d0 + 32 * vb + (lane >> 4) * kDSec) >> 4;
                    uint32_t r[4];
                    ldsm_x4_t(vbase + vkey * 128 + ((chunk ^ (vkey & 7)) << 4), r[0], r[1], r[2], r[3]);
                    if (tail < kKeyGroup) {
                        mask_key_pair(r[0], cq, tail);
                        mask_key_pair(r[1], cq + 8, tail);
                        mask_key_pair(r[2], cq, tail);
                        mask_key_pair(r[3], cq + 8, tail);
                    }
                    mma_f16(o[4 * vb], pa, e4m3_even_f16x2(r[0]), e4m3_even_f16x2(r[1]));
                    mma_f16(o[4 * vb + 1], pa, e4m3_odd_f16x2(r[0]), e4m3_odd_f16x2(r[1]));
                    if constexpr (kDSec != 0) {
                        mma_f16(o[4 * vb + 2], pa, e4m3_even_f16x2(r[2]), e4m3_even_f16x2(r[3]));
                        mma_f16(o[4 * vb + 3], pa, e4m3_odd_f16x2(r[2]), e4m3_odd_f16x2(r[3]));
                    }
                }
            } else {
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
        float invA = lA > 0.f ? 1.f / lA : 0.f;
        float invB = lB > 0.f ? 1.f / lB : 0.f;
        if constexpr (kFp8) {
            invA *= v_scale;
            invB *= v_scale;
        }
        const float lseA = lA > 0.f ? (mA + __log2f(lA)) * ln2 : -INFINITY;
        const float lseB = lB > 0.f ? (mB + __log2f(lB)) * ln2 : -INFINITY;
        const size_t rowA = (size_t)(it.t0 + tokA) * H + hA;
        const size_t rowB = (size_t)(it.t0 + tokB) * H + hB;
        if constexpr (kFp8) {
            // n-tiles 4vb + 2sec (even d) and 4vb + 2sec + 1 (odd d): a row's four values of a 16-d half are
            // d .. d + 3 with d = d0 + 32vb + 16sec + 4t, in the order (even0, odd0, even1, odd1)
            const size_t blk = (size_t)it.index * p.dec_rows;
            const size_t pA = blk + (size_t)tokA * H + hA, pB = blk + (size_t)tokB * H + hB;
#pragma unroll
            for (int vb = 0; vb < kVB; ++vb) {
#pragma unroll
                for (int sec = 0; sec < (kDSec ? 2 : 1); ++sec) {
                    const int je = 4 * vb + 2 * sec, jo = je + 1;
                    const int d = d0 + 32 * vb + 16 * sec + 4 * (lane & 3);
                    if (it.nact == 1) {
                        if (vA) {
                            *reinterpret_cast<uint32_t *>(p.out + rowA * kD + d) = pack_bf16x2(o[je][0] * invA, o[jo][0] * invA);
                            *reinterpret_cast<uint32_t *>(p.out + rowA * kD + d + 2) = pack_bf16x2(o[je][1] * invA, o[jo][1] * invA);
                        }
                        if (vB) {
                            *reinterpret_cast<uint32_t *>(p.out + rowB * kD + d) = pack_bf16x2(o[je][2] * invB, o[jo][2] * invB);
                            *reinterpret_cast<uint32_t *>(p.out + rowB * kD + d + 2) = pack_bf16x2(o[je][3] * invB, o[jo][3] * invB);
                        }
                    } else {
                        if (vA)
                            *reinterpret_cast<float4 *>(p.part_dec_o + pA * kD + d) =
                                make_float4(o[je][0] * invA, o[jo][0] * invA, o[je][1] * invA, o[jo][1] * invA);
                        if (vB)
                            *reinterpret_cast<float4 *>(p.part_dec_o + pB * kD + d) =
                                make_float4(o[je][2] * invB, o[jo][2] * invB, o[je][3] * invB, o[jo][3] * invB);
                    }
                }
            }
            if (dsl == 0 && (lane & 3) == 0) {
                if (it.nact == 1) {
                    if (p.lse && vA) p.lse[rowA] = lseA;
                    if (p.lse && vB) p.lse[rowB] = lseB;
                } else {
                    if (vA) p.part_dec_lse[pA] = lseA;
                    if (vB) p.part_dec_lse[pB] = lseB;
                }
            }
        } else if (it.nact == 1) {
#pragma unroll
            for (int j = 0; j < kNT; ++j) {
                const int d = d0 + j * 8 + cq;
                if (vA) *reinterpret_cast<uint32_t *>(p.out + rowA * kD + d) = pack_bf16x2(o[j][0] * invA, o[j][1] * invA);
                if (vB) *reinterpret_cast<uint32_t *>(p.out + rowB * kD + d) = pack_bf16x2(o[j][2] * invB, o[j][3] * invB);
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
                if (vA) *reinterpret_cast<float2 *>(p.part_dec_o + pA * kD + d) = make_float2(o[j][0] * invA, o[j][1] * invA);
                if (vB) *reinterpret_cast<float2 *>(p.part_dec_o + pB * kD + d) = make_float2(o[j][2] * invB, o[j][3] * invB);
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
                          int bias_slot_bytes, int kv_fp8, float k_scale, float v_scale, int per_sm, int small,
                          int one_tok, int grid, size_t smem, cudaStream_t stream)
{
    auto go = [&](auto kernel) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        return launch_pdl(kernel, (unsigned)grid, kDecThreads, smem, stream, p, tm_k, tm_v, tm_bias, nstages,
                          stage_bytes, kv_bytes, bias_slot_bytes, k_scale, v_scale);
    };
    // the d-slices of a KV head (8 / Hkv), for one head size and build
    auto slices = [&](auto d, auto fp8, auto two, auto sm, auto one) -> cudaError_t {
        constexpr int D = decltype(d)::value;
        constexpr bool F = decltype(fp8)::value, M = decltype(sm)::value, O = decltype(one)::value;
        constexpr int S = decltype(two)::value ? 2 : 1;
        switch (8 / p.Hkv) {
            case 1: return go(ink_decode_kernel<D, 1, F, S, M, O>);
            case 2: return go(ink_decode_kernel<D, 2, F, S, M, O>);
            case 4: return go(ink_decode_kernel<D, 4, F, S, M, O>);
            default:
                if constexpr (D / 8 >= 16) return go(ink_decode_kernel<D, 8, F, S, M, O>);
                else return cudaErrorInvalidValue;  // D = 64 with one KV head: d-slices narrower than a tile
        }
    };
    // the small-rows builds where the registers are capped (two CTAs an SM), and at one CTA an SM for calls of
    // one query token a request (no spills there either)
    auto builds = [&](auto d, auto fp8) -> cudaError_t {
        using T = std::true_type;
        using N = std::false_type;
        if (per_sm != 2) return small && one_tok ? slices(d, fp8, N{}, T{}, T{}) : slices(d, fp8, N{}, N{}, N{});
        if (!small) return slices(d, fp8, T{}, N{}, N{});
        return one_tok ? slices(d, fp8, T{}, T{}, T{}) : slices(d, fp8, T{}, T{}, N{});
    };
    if (kv_fp8) {
        if (p.D != 128) return cudaErrorInvalidValue;
        return builds(std::integral_constant<int, 128>{}, std::true_type{});
    }
    switch (p.D) {
        case 64: return builds(std::integral_constant<int, 64>{}, std::false_type{});
        case 128: return builds(std::integral_constant<int, 128>{}, std::false_type{});
        case 256: return builds(std::integral_constant<int, 256>{}, std::false_type{});
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ink
