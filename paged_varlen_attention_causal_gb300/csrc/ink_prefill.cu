// ink_prefill.cu -- prefill kernels: paged varlen causal GQA attention on the
// 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
// Two kernels share the code below: the one-CTA kernel (ink_prefill_kernel),
// which runs prefill units that are split over the key range, and the 2-SM
// pair kernel (ink_prefill_pair_kernel, at the end of the file), which runs
// unsplit units two q tiles at a time on a CTA pair with cta_group::2 MMAs.
// The one-CTA kernel:
//
// One work item = (request, q tile, split, KV head): 128 packed rows, i.e.
// 128/G tokens x the G query heads that share KV head g (GQA packing).
// Persistent CTAs (one per SM) walk the device-built item list, longest
// items first.  Tensor memory: a 2-slot ring of S tiles (128 x 128 fp32),
// the O accumulator (128 x 128 fp32) and the Q tile (128 x 128 bf16).
// Warp roles:
//   warp 0      page-gather producer: block_table entries are prefetched 32
//               groups ahead; per 16-key page two TMA boxes of K (d halves,
//               128-byte swizzle) and one 4-D box of V (both d halves) into
//               a 3-slot K/V ring (a staged request: one 32 KB box per tile);
//   warp 1      tensor-memory allocator and single-thread MMA issuer:
//               S = Q K^T with Q read from tensor memory (M128 N128 K16 x 8),
//               O += P V with P read from tensor memory (M128 N128 K16 x 8);
//   warp 2      bias producer: per bias tile and key half one fp32 TMA box of
//               rel_logits per 8 tokens (fewer when shared memory is short;
//               out-of-range distances read as 0) into a 3-stage ring of half
//               tiles, each stage read by one softmax warpgroup;
//   warps 4-11  online softmax in two warpgroups: warps 4-7 take keys 0-63 of
//               every S tile, warps 8-11 keys 64-127 (thread = TMEM lane = row);
//               each adds its half of the relative bias from the staged boxes
//               and applies the masks, and the two halves of a row agree on
//               the row maximum through shared memory; they also run the
//               epilogue and write the next item's Q rows into tensor memory.
// Row packing is token-strided per warp so that every row of a warp has the
// same q_abs mod 4, which makes the misalignment of its bias span (relative
// to a 16-byte TMA box start) a warp-uniform constant.
#include <algorithm>

#include "ink_common.cuh"

namespace ink {

constexpr int kPfThreads = 12 * 32;
constexpr int kPfLaunchRegs = 168;          // registers per thread at launch (65536 / 384, rounded down to 8)
constexpr int kPfProducerRegs = 80;         // warpgroup 0 (warps 0-3) after setmaxnreg.dec
constexpr int kPfSoftmaxRegs = 208;        // warpgroups 1 and 2 (softmax) after setmaxnreg.inc
static_assert(128 * kPfProducerRegs + 256 * kPfSoftmaxRegs <= kPfThreads * kPfLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kKvSlots = kPfKvSlots;
constexpr int kSSlots = 2;
constexpr int kBiasSlots = kPfBiasSlots;      // half-tile bias stages
constexpr int kSlotBytes = 32768;           // one K or V tile: 2 d halves x 128 rows x 128 B
constexpr int kRescaleThreshold = 8;        // log2 units (factor 256)
constexpr uint32_t kTmemCols = 512;         // S ring 2 x 128 | O 128 | Q 64 (bf16 pairs)
constexpr int kSoftmaxWarps = 8;            // two warpgroups, one half of the keys each

// Instruction descriptor, kind::f16: D f32, A bf16, B bf16, M 128, N 128.
constexpr uint32_t kIdescQK = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
// Same with B (V) in MN-major layout.
constexpr uint32_t kIdescPV = kIdescQK | (1u << 16);

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= 1ull << 46;   // descriptor version for sm_100-class tensor cores
    d |= 2ull << 61;   // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

#define INK_TMEM_LD32(taddr, r)                                                                                  \
    asm volatile(                                                                                                \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17," \
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                                       \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),         \
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),   \
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), \
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])  \
        : "r"(taddr))

#define INK_TMEM_ST32(taddr, r)                                                                                  \
    asm volatile(                                                                                                \
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"  \
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),                       \
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),       \
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),          \
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),         \
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])                      \
        : "memory")

struct PfShared {
    uint64_t kv_full[kKvSlots], kv_empty[kKvSlots];
    uint64_t bias_full[kBiasSlots], bias_empty[kBiasSlots];
    uint64_t q_full;
    uint64_t s_full[kSSlots], p_full[kSSlots], pv_done[kSSlots];
    uint64_t o_full;
    uint64_t xbar[4][2];      // row-half exchange between warps w and w + 4 (per lane quarter, 2 buffers)
    int32_t tile_keys[4][8];  // producer's record of recent tiles' key coordinates (reused by V)
    uint32_t tmem_base;
    int abort;
    uint32_t mma_tiles;  // tiles whose MMAs were issued for this CTA (set by warp 1 at its end)
    float xchg[2][2][kTileRows];  // [buffer][key half][row]: partial row maxima, then row sums
};
static_assert(sizeof(PfShared) <= kPfSharedBytes, "prefill bookkeeping exceeds its shared-memory budget");

// Everything a role needs to know about one work item; every role computes
// it from the item with the same code.
struct PfItem {
    int b, qt, s, g;
    int t0, Lq, Lk;
    int i0, ntok;        // first token of the tile, valid tokens in it
    int qa_min, qa_max;  // q_abs of the first / last valid token
    int gb, ge, nact;    // 16-key groups of the split, splits of the unit
    int ntiles;          // 128-key tiles (8 groups each) of the split
    int lo_max, hi_min;  // keys visible to every valid row (inside the split)
    int rot;             // processing order: tile n of the loop is tile (n + rot) mod ntiles of the split
};

__device__ __forceinline__ PfItem pf_item(const Params &p, int4 v)
{
    PfItem it;
    it.b = v.x; it.qt = v.y; it.s = v.z; it.g = v.w;
    const Req r = load_req(p, it.b);
    it.t0 = r.t0; it.Lq = r.Lq; it.Lk = r.Lk;
    it.i0 = it.qt * p.tpt;
    it.ntok = min(p.tpt, it.Lq - it.i0);
    it.qa_min = it.i0 + it.Lk - it.Lq;
    it.qa_max = it.qa_min + it.ntok - 1;
    const UnitSplit u = unit_split(it.qa_min, it.qa_max, it.Lk, p.causal, p.wl, p.wr, p.chunk_pf, it.s);
    it.gb = u.gb; it.ge = u.ge; it.nact = u.nact;
    it.ntiles = (it.ge - it.gb + 7) / 8;
    int lo, hi, t;
    visible_range(it.qa_max, it.qa_max, it.Lk, p.causal, p.wl, p.wr, lo, t);
    visible_range(it.qa_min, it.qa_min, it.Lk, p.causal, p.wl, p.wr, t, hi);
    it.lo_max = max(lo, it.gb * kKeyGroup);
    it.hi_min = min(hi, it.ge * kKeyGroup - 1);
    it.rot = 0;
    return it;
}

// First key of the tile the loop handles at step n (the online softmax is the same in any tile order).
__device__ __forceinline__ int pf_tile_key0(const PfItem &it, int n)
{
    const int m = n + it.rot;
    return (it.gb + 8 * (m < it.ntiles ? m : m - it.ntiles)) * kKeyGroup;
}

__device__ __forceinline__ bool pf_tile_bias(const Params &p, const PfItem &it, int n)
{
    const int j0 = pf_tile_key0(it, n);
    const int rd_min = it.qa_min - (j0 + kTileKeys - 1), rd_max = it.qa_max - j0;
    return p.E > 0 && it.ntok > 0 && rd_max >= 0 && rd_min < p.E;
}

__device__ __forceinline__ bool pf_tile_mask(const PfItem &it, int n)
{
    const int j0 = pf_tile_key0(it, n);
    return j0 < it.lo_max || j0 + kTileKeys - 1 > it.hi_min;
}

// Row L of the tile -> (token offset k, head j); false when the row is padding.
__device__ __forceinline__ bool pf_row(const Params &p, int L, int &k, int &j)
{
    if (p.fast_pack) {
        const int q = L >> 5, l = L & 31;
        k = 4 * (l / p.G) + q;
        j = l % p.G;
        return true;
    }
    k = L / p.G;
    j = L % p.G;
    return k < p.tpt;
}

// Item of round r for this CTA: snake order over the cost-sorted list.
__device__ __forceinline__ int pf_item_index(int r)
{
    return r * gridDim.x + ((r & 1) ? (gridDim.x - 1 - blockIdx.x) : blockIdx.x);
}

// Every PV commit arrives on a pv_done barrier, which the softmax waits on only
// when it rescales O; the final phase of each slot (the CTA's last two tiles) is
// awaited here before teardown, so that no arrival is still pending when the
// CTA exits.  Called once every softmax warp has passed its last o_full wait: by
// then no slot is more than one phase short of its final one, which is what the
// parity waits need.
template <typename Wait>
__device__ __forceinline__ void drain_pv_done(uint64_t *pv_done, uint32_t ntiles, Wait wait)
{
    static_assert(kSSlots == 2, "one final phase per slot: tiles ntiles - 1 and ntiles - 2");
    if (ntiles >= 1 && wait(&pv_done[(ntiles - 1) & 1], ((ntiles - 1) >> 1) & 1) && ntiles >= 2)
        wait(&pv_done[ntiles & 1], ((ntiles - 2) >> 1) & 1);
}

// One key half (64 columns) of a row's relative bias, added to its raw scores:
// s[c] += inv_scale * box[O + 63 - c], where box starts at the half's first
// 16-byte chunk and O = (q_abs - j0 - 127) mod 4 is a compile-time constant
// here.  17 aligned 16-byte loads cover the 68 floats the half needs.
template <int O>
__device__ __forceinline__ void bias_add(uint32_t box, float inv_scale, uint32_t (&s)[64])
{
#pragma unroll
    for (int m = 0; m < 17; ++m) {
        float e[4];
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(e[0]), "=f"(e[1]), "=f"(e[2]), "=f"(e[3])
                     : "r"(box + 16 * m));
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = O + 63 - (4 * m + u);
            if (c >= 0 && c < 64) s[c] = __float_as_uint(fmaf(e[u], inv_scale, __uint_as_float(s[c])));
        }
    }
}

__global__ void __launch_bounds__(kPfThreads, 1)
    ink_prefill_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_bias,
                       const __grid_constant__ CUtensorMap tm_ks, const __grid_constant__ CUtensorMap tm_vs)
{
    extern __shared__ __align__(1024) uint8_t dsmem[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    uint8_t *kv_smem = base;                                  // kKvSlots x 32 KB
    uint8_t *bias_smem = kv_smem + kKvSlots * kSlotBytes;     // kBiasSlots x (tpt x G rows of a key half)
    const int bias_nb = 1 << p.bias_tok_log2;  // tokens per bias box
    const int bias_w = p.bias_w;                 // floats per box row
    const int bias_box = pf_bias_box_stride(p.G, bias_nb, bias_w);
    const int bias_stage = pf_bias_stage_bytes(p.G, p.tpt, bias_nb, bias_w);
    PfShared &sh = *reinterpret_cast<PfShared *>(bias_smem + kBiasSlots * bias_stage);
    volatile int *abort = &sh.abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The host requests at most the per-CTA limit, which leaves less than 1 KB for aligning
    // the base when G = 1; if the window is too small after alignment, do nothing (CTA-uniform).
    if ((uintptr_t)(reinterpret_cast<uint8_t *>(&sh + 1) - dsmem) > dynamic_smem_bytes()) {
        pdl_wait();
        if (threadIdx.x == 0) report(p, INK_DEVERR_SMEM);
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kKvSlots; ++s) {
            mbar_init(&sh.kv_full[s], 1);
            mbar_init(&sh.kv_empty[s], 1);
        }
        for (int s = 0; s < kBiasSlots; ++s) {
            mbar_init(&sh.bias_full[s], 1);
            mbar_init(&sh.bias_empty[s], kSoftmaxWarps / 2);
        }
        mbar_init(&sh.q_full, kSoftmaxWarps);
        for (int s = 0; s < kSSlots; ++s) {
            mbar_init(&sh.s_full[s], 1);
            mbar_init(&sh.p_full[s], kSoftmaxWarps);
            mbar_init(&sh.pv_done[s], 1);
        }
        mbar_init(&sh.o_full, 1);
        for (int q = 0; q < 4; ++q) {
            mbar_init(&sh.xbar[q][0], 2);
            mbar_init(&sh.xbar[q][1], 2);
        }
        sh.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();  // barriers and tensor memory are set up; now the work list, staging copy and inputs
    pdl_launch_dependents();
    const int total = (int)*(volatile uint32_t *)&p.hdr->pf_count;
    const uint32_t tmem = sh.tmem_base;
    const uint32_t tmem_o = tmem + kSSlots * 128;
    const uint32_t tmem_q = tmem_o + 128;

    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPfProducerRegs));
    if (warp == 0) {
        // ---------------------------------------------------------------- K/V producer
        if (lane == 0) {
            if (!p.kv_fp8) {  // an FP8 call has no paged maps: it reads staged tiles only
                prefetch_tmap(&tm_k);
                prefetch_tmap(&tm_v);
            }
            if (p.stage_cap > 0) {
                prefetch_tmap(&tm_ks);
                prefetch_tmap(&tm_vs);
            }
        }
        const uint64_t pol_kv = policy_evict_last();
        uint32_t seq = 0;
        for (int r = 0;; ++r) {
            const int idx = pf_item_index(r);
            if (idx >= total || *abort) break;
            const PfItem it = pf_item(p, p.pf_items[idx]);
            if (it.ntiles == 0) continue;
            // staged request: its keys sit at staged key so + j of each KV head's plane
            const int so = p.stage_cap > 0 ? __ldg(p.stg_off + it.b) : -1;
            const int32_t *bt_row = p.bt + (size_t)it.b * p.MAXBLK;
            // key coordinate of group gb + 32 * chunk + lane (-16, i.e. zero fill, past the split or on a bad page)
            auto load_keys = [&](int chunk) {
                const int gi = it.gb + 32 * chunk + lane;
                int key = -kKeyGroup;
                if (gi < it.ge) {
                    const int pid = __ldg(bt_row + (gi * kKeyGroup) / p.BS);
                    if (pid >= 0 && pid < p.NB) key = pid * p.BS + (gi * kKeyGroup) % p.BS;
                    else report(p, INK_DEVERR_PAGE_ID);
                }
                return key;
            };
            int keys_cur = so >= 0 ? 0 : load_keys(0), keys_nxt = so >= 0 ? 0 : load_keys(1), chunk = 0;
            // load order: K0, then K_n, V_{n-1} for n >= 1, then V_{last}
            for (int step = 0; step <= it.ntiles; ++step) {
                for (int which = 0; which < 2; ++which) {
                    int n, isV;
                    if (step == 0) { if (which) break; n = 0; isV = 0; }
                    else if (step == it.ntiles) { if (which) break; n = it.ntiles - 1; isV = 1; }
                    else { n = which ? step - 1 : step; isV = which; }
                    int key0;
                    if (so >= 0) {
                        key0 = so + pf_tile_key0(it, n);
                    } else if (!isV) {
                        while (chunk < n / 4) {  // advance the prefetch window by 32 groups
                            keys_cur = keys_nxt;
                            ++chunk;
                            keys_nxt = load_keys(chunk + 1);
                        }
                        key0 = __shfl_sync(0xffffffffu, keys_cur, (n % 4) * 8 + (lane & 7));
                        if (lane < 8) sh.tile_keys[n % 4][lane] = key0;
                    } else {
                        key0 = sh.tile_keys[n % 4][lane & 7];
                    }
                    __syncwarp();
                    const int slot = seq % kKvSlots;
                    if (!mbar_wait_warp(&sh.kv_empty[slot], ((seq / kKvSlots) & 1) ^ 1, abort, p)) break;
                    if (lane == 0) mbar_arrive_expect_tx(&sh.kv_full[slot], kSlotBytes);
                    __syncwarp();
                    if (so >= 0) {
                        // staged: the tile is 128 consecutive keys of the KV head's plane, one box that
                        // lands as [d half][128 keys][128 B] for K and for V
                        if (lane == 0)
                            tma_load_4d_hint(kv_smem + slot * kSlotBytes, isV ? &tm_vs : &tm_ks, 0, key0, 0, it.g,
                                             &sh.kv_full[slot], pol_kv);
                    } else if (!isV && lane < 16) {
                        // K tile: [d half][128 keys][128 B]; one box per page and d half
                        const int grp = lane & 7, dh = lane >> 3;
                        uint8_t *dst = kv_smem + slot * kSlotBytes + dh * 16384 + grp * 2048;
                        tma_load_3d_hint(dst, &tm_k, dh * 64, it.g, key0, &sh.kv_full[slot], pol_kv);
                    } else if (isV && lane < 8) {
                        // V tile: [page][d half][16 keys][128 B]; one box per page covers both halves
                        uint8_t *dst = kv_smem + slot * kSlotBytes + lane * 4096;
                        tma_load_4d_hint(dst, &tm_v, 0, key0, 0, it.g, &sh.kv_full[slot], pol_kv);
                    }
                    __syncwarp();
                    ++seq;
                }
                if (*abort) break;
            }
        }
        // let copies still in flight land before the CTA can exit
        if (lane == 0)
            for (uint32_t k = (seq > kKvSlots ? seq - kKvSlots : 0); k < seq; ++k)
                mbar_wait(&sh.kv_full[k % kKvSlots], (k / kKvSlots) & 1, abort, p);
    } else if (warp == 2) {
        // ---------------------------------------------------------------- bias producer
        if (p.bias_tma) {
            if (lane == 0) prefetch_tmap(&tm_bias);
            const uint64_t pol_bias = policy_evict_first();
            uint32_t bseq = 0;
            for (int r = 0;; ++r) {
                const int idx = pf_item_index(r);
                if (idx >= total || *abort) break;
                const PfItem it = pf_item(p, p.pf_items[idx]);
                bool stop = false;
                for (int n = 0; n < it.ntiles && !stop; ++n) {
                    if (!pf_tile_bias(p, it, n)) continue;
                    const int nbox = (it.ntok + bias_nb - 1) >> p.bias_tok_log2;
                    // keys 64h .. 64h + 63 of the tile, read by softmax warpgroup h
                    for (int h = 0; h < 2; ++h) {
                        const int bs = bseq % kBiasSlots;
                        if (!mbar_wait_warp(&sh.bias_empty[bs], ((bseq / kBiasSlots) & 1) ^ 1, abort, p)) {
                            stop = true;
                            break;
                        }
                        const int j0 = pf_tile_key0(it, n) + 64 * h;
                        if (lane == 0)
                            mbar_arrive_expect_tx(&sh.bias_full[bs], (uint32_t)(nbox * pf_bias_box_bytes(p.G, bias_nb, bias_w)));
                        __syncwarp();
                        for (int b = lane; b < nbox; b += 32) {
                            const int k0 = b << p.bias_tok_log2;
                            // distance span of token k0: from q_abs - (j0 + 63) up; rounded down to 16 bytes
                            const int x0 = (it.qa_min + k0 - j0 - 63) & ~3;
                            tma_load_3d_hint(bias_smem + bs * bias_stage + b * bias_box, &tm_bias, x0, it.g * p.G,
                                             it.t0 + it.i0 + k0, &sh.bias_full[bs], pol_bias);
                        }
                        __syncwarp();
                        ++bseq;
                    }
                }
                if (*abort) break;
            }
            if (lane == 0)
                for (uint32_t k = (bseq > kBiasSlots ? bseq - kBiasSlots : 0); k < bseq; ++k)
                    mbar_wait(&sh.bias_full[k % kBiasSlots], (k / kBiasSlots) & 1, abort, p);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        uint32_t seq = 0, tc = 0, qseq = 0;
        for (int r = 0;; ++r) {
            const int idx = pf_item_index(r);
            if (idx >= total || *abort) break;
            const PfItem it = pf_item(p, p.pf_items[idx]);
            if (it.ntiles == 0) continue;
            if (!mbar_wait_warp(&sh.q_full, qseq & 1, abort, p)) break;
            const uint32_t tc0 = tc;
            const bool staged = p.stage_cap > 0 && __ldg(p.stg_off + it.b) >= 0;
            auto zero_tail = [&](int slot, int n, bool v_layout) {
                // keys at or beyond Lk inside loaded groups may hold stale data: zero them.  A
                // staged tile holds 128 keys whatever the split: zero every key past the split
                // too (the staging area beyond a request's last page is never written).
                const int j0 = pf_tile_key0(it, n);
                int loaded = min(8, it.ge - (it.gb + 8 * n)) * kKeyGroup;
                int z0 = max(0, it.Lk - j0);
                if (staged) {
                    z0 = min(z0, loaded);
                    loaded = kTileKeys;
                    v_layout = false;  // staged V lands as [d half][128 keys][128 B], like K
                }
                if (z0 < loaded) {
                    uint8_t *t = kv_smem + slot * kSlotBytes;
                    for (int c = lane; c < (loaded - z0) * 16; c += 32) {  // 16 chunks of 16 B per row
                        const int row = z0 + c / 16, ch = c % 16;
                        const int off = v_layout ? (row >> 4) * 4096 + (ch >> 3) * 2048 + (row & 15) * 128
                                                 : (ch >> 3) * 16384 + row * 128;
                        *reinterpret_cast<uint4 *>(t + off + (ch & 7) * 16) = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
            };
            // Ring positions of the item's K and V tiles in the producer's order (K0, then K_n, V_{n-1}
            // for n >= 1, then V_last).
            auto seq_k = [&](int n) { return seq + (n == 0 ? 0u : (uint32_t)(2 * n - 1)); };
            auto seq_v = [&](int m) { return seq + (m == it.ntiles - 1 ? (uint32_t)(2 * it.ntiles - 1) : (uint32_t)(2 * m + 2)); };
            auto issue_qk = [&](int n) {
                const uint32_t t = tc0 + n, sq = seq_k(n);
                const int ss = t % kSSlots, slot = sq % kKvSlots;
                zero_tail(slot, n, false);
                tc_fence_after();
                if (lane == 0) {
                    // S slot ss was last read by PV(t - 2), issued earlier by this thread: the
                    // tensor core runs them in order
                    const uint32_t kaddr = smem_u32(kv_smem + slot * kSlotBytes);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
                        const uint64_t bdesc = smem_desc(kaddr + off, 16, 1024);
                        mma_ts(tmem + ss * 128, tmem_q + kk * 8, bdesc, kIdescQK, kk > 0 ? 1u : 0u);
                    }
                    mma_commit(&sh.s_full[ss]);
                    mma_commit(&sh.kv_empty[slot]);
                }
                __syncwarp();
            };
            auto issue_pv = [&](int m) {
                const uint32_t t = tc0 + m, sq = seq_v(m);
                const int ss = t % kSSlots, slot = sq % kKvSlots;
                zero_tail(slot, m, true);
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t vaddr = smem_u32(kv_smem + slot * kSlotBytes);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        // keys 16kk .. 16kk + 15: paged, page kk, d halves 2 KB apart; staged, rows
                        // 16kk.. of [d half][128 keys], d halves 16 KB apart; 8-key groups 1 KB apart
                        const uint64_t bdesc = staged ? smem_desc(vaddr + kk * 2048, 16384, 1024)
                                                      : smem_desc(vaddr + kk * 4096, 2048, 1024);
                        mma_ts(tmem_o, tmem + ss * 128 + kk * 8, bdesc, kIdescPV, (m > 0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&sh.kv_empty[slot]);
                    mma_commit(&sh.pv_done[ss]);
                }
                __syncwarp();
            };
            // Step n issues QK(n) and PV(n - 1), whichever can go first: QK(n) needs K(n), PV(n - 1)
            // needs P(n - 1) and V(n - 1).  They touch different S slots, and QK(n)'s slot was last
            // read by PV(n - 2), issued in the previous step, so either order is safe.  Polling both
            // keeps a late K(n) from holding back PV(n - 1) and the reverse.
            bool ok = true;
            for (int n = 0; n <= it.ntiles && ok; ++n) {
                bool qk_todo = n < it.ntiles, pv_todo = n >= 1;
                const uint64_t t0 = global_timer_ns();
                while (qk_todo || pv_todo) {
                    if (qk_todo) {
                        const uint32_t sq = seq_k(n);
                        if (warp_poll(&sh.kv_full[sq % kKvSlots], (sq / kKvSlots) & 1)) {
                            issue_qk(n);
                            qk_todo = false;
                            continue;
                        }
                    }
                    if (pv_todo) {
                        const uint32_t t = tc0 + n - 1, sq = seq_v(n - 1);
                        if (warp_poll(&sh.p_full[t % kSSlots], (t / kSSlots) & 1) &&
                            warp_poll(&sh.kv_full[sq % kKvSlots], (sq / kKvSlots) & 1)) {
                            issue_pv(n - 1);
                            pv_todo = false;
                            continue;
                        }
                    }
                    if (*abort) { ok = false; break; }
                    __nanosleep(20);
                    if (global_timer_ns() - t0 > kWaitLimitNs) {
                        report(p, INK_DEVERR_TIMEOUT);
                        *abort = 1;
                        ok = false;
                        break;
                    }
                }
            }
            seq += 2 * it.ntiles;
            if (ok && lane == 0) mma_commit(&sh.o_full);
            __syncwarp();
            tc += it.ntiles;
            ++qseq;
            if (!ok) break;
        }
        if (lane == 0) sh.mma_tiles = tc;
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPfSoftmaxRegs));
        // ---------------------------------------------------------------- softmax + epilogue + Q
        const int h = (warp >= 8) ? 1 : 0;   // key half: columns 64h .. 64h + 63 of every S tile
        const int quarter = warp & 3;        // TMEM lanes 32 * quarter .. + 31
        const int L = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const float sl2 = p.scale_log2;
        const float inv_scale = p.inv_scale;
        const float ln2 = 0.6931471805599453f;
        // Q rows of an item into tensor memory (this half's 64 dims as bf16 pairs), then signal the MMA warp.
        auto write_q = [&](const PfItem &it) {
            int k, j;
            const bool row_ok = pf_row(p, L, k, j) && k < it.ntok;
            uint32_t qv[32];
            if (row_ok) {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    p.q + ((size_t)(it.t0 + it.i0 + k) * p.H + it.g * p.G + j) * kHeadDim + 64 * h);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = __ldg(src + c);
                    qv[4 * c] = v.x; qv[4 * c + 1] = v.y; qv[4 * c + 2] = v.z; qv[4 * c + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) qv[c] = 0u;
            }
            INK_TMEM_ST32(tmem_q + lane_addr + 32 * h, qv);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.q_full);
        };
        // next item (round > r) that has tiles, or -1
        auto next_with_tiles = [&](int r, PfItem &nx) {
            for (int r2 = r + 1;; ++r2) {
                const int idx = pf_item_index(r2);
                if (idx >= total) return false;
                nx = pf_item(p, p.pf_items[idx]);
                if (nx.ntiles > 0) return true;
            }
        };
        // The two warps that share this lane quarter (w and w + 4) swap one float per row.
        // Buffer b is reused two exchanges later, after the partner has read it.
        uint32_t xseq = 0;
        auto exchange = [&](float mine, float &theirs) {
            const int b = xseq & 1;
            sh.xchg[b][h][L] = mine;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.xbar[quarter][b]);
            const bool ok = mbar_wait_warp(&sh.xbar[quarter][b], (xseq >> 1) & 1, abort, p);
            tc_fence_after();
            theirs = sh.xchg[b][h ^ 1][L];
            ++xseq;
            return ok;
        };
        {
            PfItem first;
            if (next_with_tiles(-1, first)) write_q(first);
        }
        uint32_t tc = 0, oseq = 0, bseq = 0;
        for (int r = 0;; ++r) {
            const int idx = pf_item_index(r);
            if (idx >= total || *abort) break;
            const PfItem it = pf_item(p, p.pf_items[idx]);
            int k, j;
            const bool row_ok = pf_row(p, L, k, j) && k < it.ntok;
            const int qa = it.qa_min + k;
            int lo = 1, hi = 0;  // visible keys of this row inside the split (empty for padding rows)
            if (row_ok) {
                visible_range(qa, qa, it.Lk, p.causal, p.wl, p.wr, lo, hi);
                lo = max(lo, it.gb * kKeyGroup);
                hi = min(hi, it.ge * kKeyGroup - 1);
            }
            // This row's bias span inside its box: it starts ko floats after the box start
            // (tiles start at multiples of 16 keys, so ko is the same for every tile); the
            // 16-byte chunk that holds it is read whole and the remainder bo is a compile-time
            // shift below.  With warp-strided packing bo is the same for every row of a warp.
            const int kb = k >> p.bias_tok_log2, ki = k & (bias_nb - 1);
            const int ko = (qa - (kTileKeys - 1)) - ((it.qa_min + (kb << p.bias_tok_log2) - (kTileKeys - 1)) & ~3);
            const int bo = ko & 3;
            const uint32_t box_row = smem_u32(bias_smem) + kb * bias_box + ((ki * p.G + j) * bias_w + 4 * (ko >> 2)) * 4;
            const float *rel_row = p.rel ? p.rel + ((size_t)(it.t0 + it.i0 + k) * p.H + it.g * p.G + j) * p.E : nullptr;
            float m_used = -INFINITY;  // raw-score units
            float l = 0.f;             // this half's share of the row sum
            bool ok = true;
            for (int n = 0; n < it.ntiles; ++n) {
                const uint32_t t = tc + n;
                const int ss = t % kSSlots;
                const int j0 = pf_tile_key0(it, n) + 64 * h;  // first key of this half
                if (!mbar_wait_warp(&sh.s_full[ss], (t / kSSlots) & 1, abort, p)) { ok = false; break; }
                tc_fence_after();
                uint32_t sv[64];
                const uint32_t sa = tmem + lane_addr + ss * 128 + 64 * h;
                INK_TMEM_LD32(sa + 0, (sv + 0));
                INK_TMEM_LD32(sa + 32, (sv + 32));
                tc_wait_ld();
                if (pf_tile_bias(p, it, n)) {
                    if (p.bias_tma) {
                        // the tile's two half stages are bias sequence numbers 2 bseq (keys 0-63) and 2 bseq + 1
                        const uint32_t hseq = 2 * bseq + h;
                        const int bs = hseq % kBiasSlots;
                        if (!mbar_wait_warp(&sh.bias_full[bs], (hseq / kBiasSlots) & 1, abort, p)) { ok = false; break; }
                        if (row_ok) {
                            const uint32_t box = box_row + bs * bias_stage;
                            switch (bo) {
                                case 0: bias_add<0>(box, inv_scale, sv); break;
                                case 1: bias_add<1>(box, inv_scale, sv); break;
                                case 2: bias_add<2>(box, inv_scale, sv); break;
                                default: bias_add<3>(box, inv_scale, sv); break;
                            }
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sh.bias_empty[bs]);
                        ++bseq;
                    } else if (row_ok) {  // rows without 16-byte alignment: direct loads
#pragma unroll
                        for (int c = 0; c < 64; ++c) {
                            const int rd = qa - (j0 + c);
                            if (rd >= 0 && rd < p.E)
                                sv[c] = __float_as_uint(fmaf(__ldg(rel_row + rd), inv_scale, __uint_as_float(sv[c])));
                        }
                    }
                }
                if (pf_tile_mask(it, n)) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const int key = j0 + c;
                        if (key < lo || key > hi) sv[c] = __float_as_uint(-INFINITY);
                    }
                }
                // this half's maximum: a tree of three-input maxima (max is exact in any order)
                float m21[22];
#pragma unroll
                for (int i = 0; i < 21; ++i)
                    m21[i] = fmax3(__uint_as_float(sv[3 * i]), __uint_as_float(sv[3 * i + 1]), __uint_as_float(sv[3 * i + 2]));
                m21[21] = __uint_as_float(sv[63]);
                float m7[8];
#pragma unroll
                for (int i = 0; i < 7; ++i) m7[i] = fmax3(m21[3 * i], m21[3 * i + 1], m21[3 * i + 2]);
                m7[7] = m21[21];
                float mx = fmax3(fmax3(m7[0], m7[1], m7[2]), fmax3(m7[3], m7[4], m7[5]), fmaxf(m7[6], m7[7]));
                // Both halves now hold their S values in registers, so either may overwrite the slot.
                float mx_other;
                if (!exchange(mx, mx_other)) { ok = false; break; }
                mx = fmaxf(mx, mx_other);  // the row maximum, identical in both halves
                // The running maximum moves only when it grows past the threshold (or was -inf).
                float alpha = 1.f;
                bool scale_o = false;
                if (mx > m_used && (m_used == -INFINITY || (mx - m_used) * sl2 > (float)kRescaleThreshold)) {
                    alpha = (m_used == -INFINITY) ? 0.f : fast_exp2((m_used - mx) * sl2);
                    l *= alpha;
                    scale_o = n > 0 && m_used != -INFINITY;
                    m_used = mx;
                }
                // The decision is per row, but tcgen05.ld/st are warp-collective: the warp
                // rescales its 32 rows together (its 64 O columns), by 1 where the maximum stayed.
                if (__any_sync(0xffffffffu, scale_o)) {
                    // O holds tiles 0..n-1 once PV(t - 1) is done.  S(t) being complete means every
                    // MMA issued before QK(t) is, so PV(t - 1) is the only one that may be pending
                    // and its phase is the only one of this barrier that can be outstanding.
                    const uint32_t tp = t - 1;
                    if (!mbar_wait_warp(&sh.pv_done[tp % kSSlots], (tp / kSSlots) & 1, abort, p)) { ok = false; break; }
                    tc_fence_after();
                    const float a = scale_o ? alpha : 1.f;
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint32_t ov[32];
                        INK_TMEM_LD32(tmem_o + lane_addr + 64 * h + cc * 32, ov);
                        tc_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * a);
                        INK_TMEM_ST32(tmem_o + lane_addr + 64 * h + cc * 32, ov);
                    }
                }
                const float moff = (m_used == -INFINITY) ? 0.f : m_used * sl2;
                const uint64_t sl2x2 = f32x2(sl2, sl2), nmoff2 = f32x2(-moff, -moff);
                uint32_t pk[32];
                uint64_t ls2[2] = {0ull, 0ull};  // four independent partial sums, as two pairs
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    float x0 = __uint_as_float(sv[2 * c]), x1 = __uint_as_float(sv[2 * c + 1]);
                    fma_x2(x0, x1, sl2x2, nmoff2);
                    const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                    add_x2(ls2[c & 1], p0, p1);
                    pk[c] = pack_bf16x2(p0, p1);
                }
                l += sum_x2(ls2[0]) + sum_x2(ls2[1]);
                // P of keys 64h .. 64h + 63 as bf16 pairs: columns 32h .. 32h + 31 of the slot
                INK_TMEM_ST32(tmem + lane_addr + ss * 128 + 32 * h, pk);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sh.p_full[ss]);
            }
            if (!ok) break;
            if (it.ntiles > 0) {
                // every QK of this item is complete: the next item's Q may replace this one
                PfItem nx;
                if (next_with_tiles(r, nx)) write_q(nx);
            }
            // epilogue: the row sum is the sum of the two halves' shares
            if (it.ntiles > 0) {
                if (!mbar_wait_warp(&sh.o_full, oseq & 1, abort, p)) break;
                ++oseq;
                tc_fence_after();
            }
            float l_other;
            if (!exchange(l, l_other)) break;
            l += l_other;
            const float inv = l > 0.f ? p.out_scale / l : 0.f;
            const float lse = l > 0.f ? (m_used * sl2 + __log2f(l)) * ln2 : -INFINITY;
            const size_t row = (size_t)(it.t0 + it.i0 + k) * p.H + it.g * p.G + j;
            const bool final_out = it.nact == 1;
            // partial block of (unit, split): rows g * 128 + L
            size_t prow = 0;
            if (!final_out)
                prow = ((size_t)(__ldg(p.unit_off + it.b) + it.qt) * p.S_pf + it.s) * ((size_t)p.Hkv * kTileRows) +
                       (size_t)it.g * kTileRows + L;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int d0 = 64 * h + 32 * cc;  // first of the 32 dims handled here
                uint32_t ov[32];
                if (it.ntiles > 0) {
                    INK_TMEM_LD32(tmem_o + lane_addr + d0, ov);
                    tc_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = 0u;
                }
                if (row_ok) {
                    if (final_out) {
                        uint4 *dst = reinterpret_cast<uint4 *>(p.out + row * kHeadDim + d0);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(ov[8 * q4 + 0]) * inv, __uint_as_float(ov[8 * q4 + 1]) * inv);
                            w.y = pack_bf16x2(__uint_as_float(ov[8 * q4 + 2]) * inv, __uint_as_float(ov[8 * q4 + 3]) * inv);
                            w.z = pack_bf16x2(__uint_as_float(ov[8 * q4 + 4]) * inv, __uint_as_float(ov[8 * q4 + 5]) * inv);
                            w.w = pack_bf16x2(__uint_as_float(ov[8 * q4 + 6]) * inv, __uint_as_float(ov[8 * q4 + 7]) * inv);
                            dst[q4] = w;
                        }
                    } else {
                        float4 *dst = reinterpret_cast<float4 *>(p.part_pf_o + prow * kHeadDim + d0);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            dst[q4] = make_float4(__uint_as_float(ov[4 * q4]) * inv, __uint_as_float(ov[4 * q4 + 1]) * inv,
                                                  __uint_as_float(ov[4 * q4 + 2]) * inv, __uint_as_float(ov[4 * q4 + 3]) * inv);
                    }
                }
            }
            if (row_ok && h == 0) {
                if (final_out) {
                    if (p.lse) p.lse[row] = lse;
                } else {
                    p.part_pf_lse[prow] = lse;
                }
            }
            tc_fence_before();
            tc += it.ntiles;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1 && !*abort)
        drain_pv_done(sh.pv_done, sh.mma_tiles, [&](uint64_t *b, uint32_t par) { return mbar_wait_warp(b, par, abort, p); });
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ===========================================================================
// 2-SM variant (ink_prefill_pair_kernel).  A cluster of two CTAs on two SMs
// takes pair items: two consecutive q tiles of one (request, KV head), CTA rank
// r holding tile 2 qp + r in its own tensor memory.  One thread of rank 0
// issues M256 N128 K16 MMAs with cta_group::2: every K and V tile is split
// between the pair (rank r holds keys 64r .. 64r + 63 of a K tile and d half r
// of a V tile, 16 KB each), so each SM loads and feeds the tensor core half of
// the operand bytes per flop of the one-CTA kernel.  What stays per CTA: its
// K/V half ring (filled by its own TMA, landing on its own barriers), its bias
// ring and softmax warpgroups, its rows' S, P, O and Q in tensor memory.
// Cross-CTA hand-offs: a relay warp in each CTA waits for its half to land,
// zeroes keys past the request, and arrives on rank 0's kv_ready barrier;
// both CTAs' softmax warps arrive on rank 0's p_full / q_full; rank 0's MMA
// completions are committed to both CTAs' barriers at once (multicast).
// ===========================================================================

constexpr int kPrProducerRegs = 72;    // register split of the pair kernel: fewer spills than 80 / 208
constexpr int kPrSoftmaxRegs = 216;
static_assert(128 * kPrProducerRegs + 256 * kPrSoftmaxRegs <= kPfThreads * kPfLaunchRegs,
              "register split exceeds the launch allocation");
constexpr int kPrSlotBytes = 16384;    // K: [d half][64 keys][128 B]; V: [128 keys][128 B] (one d half)
// Instruction descriptors, kind::f16, M 256 (the pair), N 128: D f32, A and B bf16; PV with B MN-major.
constexpr uint32_t kIdescQK2 = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((256u >> 4) << 24);
constexpr uint32_t kIdescPV2 = kIdescQK2 | (1u << 16);

struct PrShared {
    uint64_t kv_full[kPrKvSlots], kv_empty[kPrKvSlots], kv_ready[kPrKvSlots];
    uint64_t bias_full[kBiasSlots], bias_empty[kBiasSlots];
    uint64_t q_full;
    uint64_t s_full[kSSlots], p_full[kSSlots], pv_done[kSSlots];
    uint64_t o_full;
    uint64_t xbar[4][2];
    int32_t tile_keys[4][8];
    uint32_t tmem_base;
    int abort;
    uint32_t mma_tiles;  // tiles of this CTA's items (set by warp 1 at its end)
    float xchg[2][2][kTileRows];
};
static_assert(sizeof(PrShared) <= kPfSharedBytes, "pair bookkeeping exceeds its shared-memory budget");

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of both CTAs: release this CTA's prior writes and wait for the peer's.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of the same variable in CTA rank 0.
__device__ __forceinline__ uint32_t rank0_addr(const void *ptr)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(smem_u32(ptr)));
    return r;
}

// Arrive on the barrier at this offset in CTA rank 0: a local arrive on rank 0 itself, an arrive through the
// cluster window from rank 1 (default semantics, as for the local one: what it hands over -- tensor-memory
// stores waited for and fenced, rows fenced to the async proxy -- is ordered before it by those fences).
__device__ __forceinline__ void arrive_rank0(const uint64_t *bar, int rank)
{
    if (rank == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
    else
        asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(rank0_addr(bar)) : "memory");
}

// Polls a barrier that the peer CTA (or rank 0's multicast commit) arrives on.  The remote arrivals are
// releases at cluster scope of work the peer ordered before them (its tensor-memory stores waited for and
// fenced, its zeroed rows fenced to the async proxy); the waiter observes the phase flip with a CTA-scope
// acquire, and what it issues next (tcgen05 operations, after the thread-sync fence) is ordered after it.
__device__ __forceinline__ bool warp_poll_cl(uint64_t *bar, uint32_t parity)
{
    return __all_sync(0xffffffffu, mbar_test_wait(bar, parity));
}

// Bounded warp-uniform wait at cluster scope (polling, 2 s limit, then the abort path).
__device__ __forceinline__ bool mbar_wait_warp_cl(uint64_t *bar, uint32_t parity, volatile int *abort,
                                                  const Params &p)
{
    if (warp_poll_cl(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        __nanosleep(32);
        if (warp_poll_cl(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            if ((threadIdx.x & 31) == 0) report(p, INK_DEVERR_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
}

__device__ __forceinline__ void mma2_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// The same with the B descriptor's address field advanced by OFF (bytes / 16) inside the instruction's own
// block, so that the compiler keeps one descriptor per tile rather than eight.
template <uint32_t OFF>
__device__ __forceinline__ void mma2_ts_off(uint32_t d_tmem, uint32_t a_tmem, uint64_t b0, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 bd;\n\t"
        "add.s64 bd, %2, %5;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], bd, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b0), "r"(idesc), "r"(acc), "n"((unsigned long long)OFF)
        : "memory");
}

// Arrive on the barrier at this offset in both CTAs once the MMAs issued so far are complete.
__device__ __forceinline__ void mma2_commit_both(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((uint16_t)3)
        : "memory");
}

// Pair item of round r for this cluster (snake order over the cost-sorted list).
__device__ __forceinline__ int pr_item_index(int r)
{
    const int nc = gridDim.x >> 1, c = blockIdx.x >> 1;
    return r * nc + ((r & 1) ? (nc - 1 - c) : c);
}

// A pair item as seen by CTA `rank`: the key range (split) is the pair's, the rows are the CTA's own tile.
__device__ __forceinline__ PfItem pr_item(const Params &p, int4 v, int rank)
{
    PfItem it;
    it.b = v.x; it.s = v.z; it.g = v.w;
    it.qt = 2 * v.y + rank;
    const Req r = load_req(p, it.b);
    it.t0 = r.t0; it.Lq = r.Lq; it.Lk = r.Lk;
    const int p0 = 2 * v.y * p.tpt, p1 = min(r.Lq, p0 + 2 * p.tpt) - 1;  // the pair's tokens
    const UnitSplit u = unit_split(p0 + r.Lk - r.Lq, p1 + r.Lk - r.Lq, r.Lk, p.causal, p.wl, p.wr, p.chunk_pf, it.s);
    it.gb = u.gb; it.ge = u.ge; it.nact = u.nact;
    it.ntiles = (it.ge - it.gb + 7) / 8;
    it.i0 = it.qt * p.tpt;
    it.ntok = max(0, min(p.tpt, it.Lq - it.i0));
    it.qa_min = it.i0 + it.Lk - it.Lq;
    it.qa_max = it.qa_min + it.ntok - 1;
    if (it.ntok > 0) {
        int lo, hi, t;
        visible_range(it.qa_max, it.qa_max, it.Lk, p.causal, p.wl, p.wr, lo, t);
        visible_range(it.qa_min, it.qa_min, it.Lk, p.causal, p.wl, p.wr, t, hi);
        it.lo_max = max(lo, it.gb * kKeyGroup);
        it.hi_min = min(hi, it.ge * kKeyGroup - 1);
    } else {  // no rows here (the request's last, odd q tile): every tile takes the masked path
        it.lo_max = 0x7fffffff;
        it.hi_min = -1;
    }
    // Items start their tiles at different offsets, so that the clusters running at any moment do not all
    // stream their bias band (the last tiles before the diagonal) from HBM at the same time.  The offset is
    // a function of the item alone (which cluster takes an item varies between calls; the result must
    // not, and it is the same whether the item reads the staging copy or the pages).  Only long items (48
    // tiles or more: the band is then a distinct tail; on the window-limited items of a continuous batch
    // rotating costs time).
    const unsigned h = ((unsigned)it.b * 131u + (unsigned)v.y * 17u + (unsigned)it.g * 7u + (unsigned)it.s) * 37u;
    it.rot = it.ntiles >= 48 ? (int)(h % (unsigned)it.ntiles) : 0;
    return it;
}

__global__ void __launch_bounds__(kPfThreads, 1)
    ink_prefill_pair_kernel(const __grid_constant__ Params p, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_bias,
                            const __grid_constant__ CUtensorMap tm_kh, const __grid_constant__ CUtensorMap tm_vh)
{
    extern __shared__ __align__(1024) uint8_t dsmem[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(dsmem) + 1023) & ~uintptr_t(1023));
    uint8_t *kv_smem = base;                                    // kPrKvSlots x 16 KB (this CTA's halves)
    uint8_t *bias_smem = kv_smem + kPrKvSlots * kPrSlotBytes;   // kBiasSlots x (tpt x G rows of a key half)
    const int bias_nb = 1 << p.bias_tok_log2;
    const int bias_w = p.bias_w;
    const int bias_box = pf_bias_box_stride(p.G, bias_nb, bias_w);
    const int bias_stage = pf_bias_stage_bytes(p.G, p.tpt, bias_nb, bias_w);
    PrShared &sh = *reinterpret_cast<PrShared *>(bias_smem + kBiasSlots * bias_stage);
    volatile int *abort = &sh.abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)cluster_rank();
    // The host launches this kernel only when the layout fits after aligning the base; if it did not,
    // both CTAs (same layout, same base) return here before touching shared memory or tensor memory.
    if ((uintptr_t)(reinterpret_cast<uint8_t *>(&sh + 1) - dsmem) > dynamic_smem_bytes()) {
        pdl_wait();
        if (threadIdx.x == 0) report(p, INK_DEVERR_SMEM);
        return;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPrKvSlots; ++s) {
            mbar_init(&sh.kv_full[s], 1);
            mbar_init(&sh.kv_empty[s], 1);
            mbar_init(&sh.kv_ready[s], 2);  // rank 0's: one relay arrival per CTA
        }
        for (int s = 0; s < kBiasSlots; ++s) {
            mbar_init(&sh.bias_full[s], 1);
            mbar_init(&sh.bias_empty[s], kSoftmaxWarps / 2);
        }
        mbar_init(&sh.q_full, 2 * kSoftmaxWarps);  // rank 0's: both CTAs' softmax warps
        for (int s = 0; s < kSSlots; ++s) {
            mbar_init(&sh.s_full[s], 1);
            mbar_init(&sh.p_full[s], 2 * kSoftmaxWarps);
            mbar_init(&sh.pv_done[s], 1);
        }
        mbar_init(&sh.o_full, 1);
        for (int q = 0; q < 4; ++q) {
            mbar_init(&sh.xbar[q][0], 2);
            mbar_init(&sh.xbar[q][1], 2);
        }
        sh.abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {  // one warp in each CTA of the pair allocates, collectively, the same columns in both
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sh.tmem_base)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers are initialised before any remote arrival
    tc_fence_after();
    pdl_wait();
    pdl_launch_dependents();
    const int total = (int)*(volatile uint32_t *)&p.hdr->pf_count;
    const uint32_t tmem = sh.tmem_base;
    const uint32_t tmem_o = tmem + kSSlots * 128;
    const uint32_t tmem_q = tmem_o + 128;

    if (warp < 4) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPrProducerRegs));
    if (warp == 0) {
        // ---------------------------------------------------------------- K/V half producer
        // Load order per item: K0, then K_n, V_{n-1} for n >= 1, then V_last; this CTA's half of each.
        if (lane == 0) {
            if (!p.kv_fp8) {
                prefetch_tmap(&tm_k);
                prefetch_tmap(&tm_v);
            }
            if (p.stage_cap > 0) {
                prefetch_tmap(&tm_kh);
                prefetch_tmap(&tm_vh);
            }
        }
        const uint64_t pol_kv = policy_evict_last();
        uint32_t seq = 0;
        for (int r = 0;; ++r) {
            const int idx = pr_item_index(r);
            if (idx >= total || *abort) break;
            const PfItem it = pr_item(p, p.pf_items[idx], rank);
            if (it.ntiles == 0) continue;
            const int so = p.stage_cap > 0 ? __ldg(p.stg_off + it.b) : -1;
            const int32_t *bt_row = p.bt + (size_t)it.b * p.MAXBLK;
            // key coordinate of page (lane & 7) of the tile whose first key is j0 (-16, i.e. zero fill, past the
            // split or on a bad page)
            auto page_key_of = [&](int j0) {
                const int gi = j0 / kKeyGroup + (lane & 7);
                int key = -kKeyGroup;
                if (gi < it.ge) {
                    const int pid = __ldg(bt_row + (gi * kKeyGroup) / p.BS);
                    if (pid >= 0 && pid < p.NB) key = pid * p.BS + (gi * kKeyGroup) % p.BS;
                    else if (lane < 8) report(p, INK_DEVERR_PAGE_ID);
                }
                return key;
            };
            for (int step = 0; step <= it.ntiles; ++step) {
                for (int which = 0; which < 2; ++which) {
                    int n, isV;
                    if (step == 0) { if (which) break; n = 0; isV = 0; }
                    else if (step == it.ntiles) { if (which) break; n = it.ntiles - 1; isV = 1; }
                    else { n = which ? step - 1 : step; isV = which; }
                    int page_key = 0;  // paged: key coordinate of page (lane & 7) of tile n
                    if (so < 0) {
                        if (!isV) {
                            page_key = page_key_of(pf_tile_key0(it, n));
                            if (lane < 8) sh.tile_keys[n % 4][lane] = page_key;
                        } else {
                            page_key = sh.tile_keys[n % 4][lane & 7];
                        }
                    }
                    // K: pages 4 rank .. 4 rank + 3 of the tile (its keys 64 rank ..), lane -> (d half, page)
                    const int k_key = __shfl_sync(0xffffffffu, page_key, 4 * rank + (lane & 3));
                    __syncwarp();
                    const int slot = seq % kPrKvSlots;
                    if (!mbar_wait_warp(&sh.kv_empty[slot], ((seq / kPrKvSlots) & 1) ^ 1, abort, p)) break;
                    if (lane == 0) mbar_arrive_expect_tx(&sh.kv_full[slot], kPrSlotBytes);
                    __syncwarp();
                    uint8_t *dst = kv_smem + slot * kPrSlotBytes;
                    if (so >= 0) {
                        const int key0 = so + pf_tile_key0(it, n);
                        if (lane == 0) {
                            if (!isV)  // keys 64 rank .. + 63, both d halves: [d half][64 keys][128 B]
                                tma_load_4d_hint(dst, &tm_kh, 0, key0 + 64 * rank, 0, it.g, &sh.kv_full[slot], pol_kv);
                            else       // d half `rank` of all 128 keys: [128 keys][128 B]
                                tma_load_4d_hint(dst, &tm_vh, 0, key0, rank, it.g, &sh.kv_full[slot], pol_kv);
                        }
                    } else if (lane < 8) {
                        if (!isV) {
                            const int grp = lane & 3, dh = lane >> 2;
                            tma_load_3d_hint(dst + dh * 8192 + grp * 2048, &tm_k, dh * 64, it.g, k_key,
                                             &sh.kv_full[slot], pol_kv);
                        } else {
                            tma_load_3d_hint(dst + lane * 2048, &tm_v, 64 * rank, it.g, page_key, &sh.kv_full[slot],
                                             pol_kv);
                        }
                    }
                    __syncwarp();
                    ++seq;
                }
                if (*abort) break;
            }
        }
        // let copies in flight land, and the MMAs that read this CTA's last halves finish, before exit
        if (lane == 0) {
            for (uint32_t k = (seq > kPrKvSlots ? seq - kPrKvSlots : 0); k < seq; ++k)
                mbar_wait(&sh.kv_full[k % kPrKvSlots], (k / kPrKvSlots) & 1, abort, p);
            for (uint32_t k = (seq > kPrKvSlots ? seq - kPrKvSlots : 0); k < seq; ++k)
                mbar_wait(&sh.kv_empty[k % kPrKvSlots], (k / kPrKvSlots) & 1, abort, p);
        }
    } else if (warp == 2) {
        // ---------------------------------------------------------------- bias producer
        if (p.bias_tma) {
            if (lane == 0) prefetch_tmap(&tm_bias);
            const uint64_t pol_bias = policy_evict_first();
            uint32_t bseq = 0;
            for (int r = 0;; ++r) {
                const int idx = pr_item_index(r);
                if (idx >= total || *abort) break;
                const PfItem it = pr_item(p, p.pf_items[idx], rank);
                bool stop = false;
                for (int n = 0; n < it.ntiles && !stop; ++n) {
                    if (!pf_tile_bias(p, it, n)) continue;
                    const int nbox = (it.ntok + bias_nb - 1) >> p.bias_tok_log2;
                    // keys 64h .. 64h + 63 of the tile, read by softmax warpgroup h
                    for (int h = 0; h < 2; ++h) {
                        const int bs = bseq % kBiasSlots;
                        if (!mbar_wait_warp(&sh.bias_empty[bs], ((bseq / kBiasSlots) & 1) ^ 1, abort, p)) {
                            stop = true;
                            break;
                        }
                        const int j0 = pf_tile_key0(it, n) + 64 * h;
                        if (lane == 0)
                            mbar_arrive_expect_tx(&sh.bias_full[bs], (uint32_t)(nbox * pf_bias_box_bytes(p.G, bias_nb, bias_w)));
                        __syncwarp();
                        for (int b = lane; b < nbox; b += 32) {
                            const int k0 = b << p.bias_tok_log2;
                            // distance span of token k0: from q_abs - (j0 + 63) up; rounded down to 16 bytes
                            const int x0 = (it.qa_min + k0 - j0 - 63) & ~3;
                            tma_load_3d_hint(bias_smem + bs * bias_stage + b * bias_box, &tm_bias, x0, it.g * p.G,
                                             it.t0 + it.i0 + k0, &sh.bias_full[bs], pol_bias);
                        }
                        __syncwarp();
                        ++bseq;
                    }
                }
                if (*abort) break;
            }
            if (lane == 0)
                for (uint32_t k = (bseq > kBiasSlots ? bseq - kBiasSlots : 0); k < bseq; ++k)
                    mbar_wait(&sh.bias_full[k % kBiasSlots], (k / kBiasSlots) & 1, abort, p);
        }
    } else if (warp == 3) {
        // ---------------------------------------------------------------- relay
        // For each K/V half in load order: wait until it has landed here, zero its keys at or past the end
        // of the request (or split), then tell rank 0's MMA warp it is ready.
        uint32_t seq = 0;
        for (int r = 0;; ++r) {
            const int idx = pr_item_index(r);
            if (idx >= total || *abort) break;
            const PfItem it = pr_item(p, p.pf_items[idx], rank);
            if (it.ntiles == 0) continue;
            const int kend = min(it.Lk, it.ge * kKeyGroup);  // first key that must read as zero
            bool ok = true;
            for (int step = 0; step <= it.ntiles && ok; ++step) {
                for (int which = 0; which < 2; ++which) {
                    int n, isV;
                    if (step == 0) { if (which) break; n = 0; isV = 0; }
                    else if (step == it.ntiles) { if (which) break; n = it.ntiles - 1; isV = 1; }
                    else { n = which ? step - 1 : step; isV = which; }
                    const int slot = seq % kPrKvSlots;
                    if (!mbar_wait_warp(&sh.kv_full[slot], (seq / kPrKvSlots) & 1, abort, p)) { ok = false; break; }
                    uint8_t *t = kv_smem + slot * kPrSlotBytes;
                    const int j0 = pf_tile_key0(it, n) + (isV ? 0 : 64 * rank);  // key of the half's first row
                    const int nrows = isV ? 128 : 64;
                    const int z0 = max(0, min(nrows, kend - j0));                // rows z0 .. nrows - 1 are zeroed
                    if (z0 < nrows) {
                        for (int c = lane; c < (nrows - z0) * 8; c += 32) {  // 8 chunks of 16 B per 128-byte row
                            const int row = z0 + c / 8, ch = c % 8;
                            if (isV) {
                                *reinterpret_cast<uint4 *>(t + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                            } else {
                                *reinterpret_cast<uint4 *>(t + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                                *reinterpret_cast<uint4 *>(t + 8192 + row * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
                            }
                        }
                        fence_proxy_async_smem();  // the tensor core reads these rows through the async proxy
                    }
                    __syncwarp();
                    if (lane == 0) arrive_rank0(&sh.kv_ready[slot], rank);
                    ++seq;
                }
            }
            if (!ok) break;
        }
    } else if (warp == 1 && rank == 0) {
        // ---------------------------------------------------------------- MMA issuer (rank 0 only)
        uint32_t seq = 0, tc = 0, qseq = 0;
        for (int r = 0;; ++r) {
            const int idx = pr_item_index(r);
            if (idx >= total || *abort) break;
            const PfItem it = pr_item(p, p.pf_items[idx], rank);
            if (it.ntiles == 0) continue;
            if (!mbar_wait_warp_cl(&sh.q_full, qseq & 1, abort, p)) break;
            tc_fence_after();
            const uint32_t tc0 = tc;
            auto seq_k = [&](int n) { return seq + (n == 0 ? 0u : (uint32_t)(2 * n - 1)); };
            auto seq_v = [&](int m) { return seq + (m == it.ntiles - 1 ? (uint32_t)(2 * it.ntiles - 1) : (uint32_t)(2 * m + 2)); };
            auto issue_qk = [&](int n) {
                const uint32_t t = tc0 + n, sq = seq_k(n);
                const int ss = t % kSSlots, slot = sq % kPrKvSlots;
                tc_fence_after();
                if (lane == 0) {
                    // one descriptor for the slot; the k steps add their byte offset / 16 to its address field
                    const uint64_t bdesc0 = smem_desc(smem_u32(kv_smem + slot * kPrSlotBytes), 16, 1024);
                    const uint32_t sd = tmem + ss * 128;  // d 16 kk ..: d half kk / 4, 32-byte step kk % 4
                    mma2_ts_off<0>(sd, tmem_q + 0, bdesc0, kIdescQK2, 0u);
                    mma2_ts_off<2>(sd, tmem_q + 8, bdesc0, kIdescQK2, 1u);
                    mma2_ts_off<4>(sd, tmem_q + 16, bdesc0, kIdescQK2, 1u);
                    mma2_ts_off<6>(sd, tmem_q + 24, bdesc0, kIdescQK2, 1u);
                    mma2_ts_off<512>(sd, tmem_q + 32, bdesc0, kIdescQK2, 1u);
                    mma2_ts_off<514>(sd, tmem_q + 40, bdesc0, kIdescQK2, 1u);
                    mma2_ts_off<516>(sd, tmem_q + 48, bdesc0, kIdescQK2, 1u);
                    mma2_ts_off<518>(sd, tmem_q + 56, bdesc0, kIdescQK2, 1u);
                    mma2_commit_both(&sh.s_full[ss]);
                    mma2_commit_both(&sh.kv_empty[slot]);
                }
                __syncwarp();
            };
            auto issue_pv = [&](int m) {
                const uint32_t t = tc0 + m, sq = seq_v(m);
                const int ss = t % kSSlots, slot = sq % kPrKvSlots;
                tc_fence_after();
                if (lane == 0) {
                    const uint64_t bdesc0 = smem_desc(smem_u32(kv_smem + slot * kPrSlotBytes), 16384, 1024);
                    const uint32_t pa = tmem + ss * 128;  // keys 16 kk ..: 8-key groups 1 KB apart
                    mma2_ts_off<0>(tmem_o, pa + 0, bdesc0, kIdescPV2, m > 0 ? 1u : 0u);
                    mma2_ts_off<128>(tmem_o, pa + 8, bdesc0, kIdescPV2, 1u);
                    mma2_ts_off<256>(tmem_o, pa + 16, bdesc0, kIdescPV2, 1u);
                    mma2_ts_off<384>(tmem_o, pa + 24, bdesc0, kIdescPV2, 1u);
                    mma2_ts_off<512>(tmem_o, pa + 32, bdesc0, kIdescPV2, 1u);
                    mma2_ts_off<640>(tmem_o, pa + 40, bdesc0, kIdescPV2, 1u);
                    mma2_ts_off<768>(tmem_o, pa + 48, bdesc0, kIdescPV2, 1u);
                    mma2_ts_off<896>(tmem_o, pa + 56, bdesc0, kIdescPV2, 1u);
                    mma2_commit_both(&sh.kv_empty[slot]);
                    mma2_commit_both(&sh.pv_done[ss]);
                }
                __syncwarp();
            };
            bool ok = true;
            for (int n = 0; n <= it.ntiles && ok; ++n) {
                bool qk_todo = n < it.ntiles, pv_todo = n >= 1;
                uint64_t t0 = 0;  // read on the first round that finds nothing to issue
                while (qk_todo || pv_todo) {
                    if (qk_todo) {
                        const uint32_t sq = seq_k(n);
                        if (warp_poll_cl(&sh.kv_ready[sq % kPrKvSlots], (sq / kPrKvSlots) & 1)) {
                            issue_qk(n);
                            qk_todo = false;
                            continue;
                        }
                    }
                    if (pv_todo) {
                        const uint32_t t = tc0 + n - 1, sq = seq_v(n - 1);
                        if (warp_poll_cl(&sh.p_full[t % kSSlots], (t / kSSlots) & 1) &&
                            warp_poll_cl(&sh.kv_ready[sq % kPrKvSlots], (sq / kPrKvSlots) & 1)) {
                            issue_pv(n - 1);
                            pv_todo = false;
                            continue;
                        }
                    }
                    if (*abort) { ok = false; break; }
                    __nanosleep(20);
                    if (t0 == 0) t0 = global_timer_ns();
                    else if (global_timer_ns() - t0 > kWaitLimitNs) {
                        if (lane == 0) report(p, INK_DEVERR_TIMEOUT);
                        *abort = 1;
                        ok = false;
                        break;
                    }
                }
            }
            seq += 2 * it.ntiles;
            if (ok && lane == 0) mma2_commit_both(&sh.o_full);
            __syncwarp();
            tc += it.ntiles;
            ++qseq;
            if (!ok) break;
        }
        if (lane == 0) sh.mma_tiles = tc;
    } else if (warp == 1) {
        // rank 1: the commits of rank 0's MMAs also arrive here; count the pair's tiles for the drain
        uint32_t n = 0;
        for (int r = 0;; ++r) {
            const int idx = pr_item_index(r);
            if (idx >= total) break;
            n += (uint32_t)pr_item(p, p.pf_items[idx], rank).ntiles;
        }
        if (lane == 0) sh.mma_tiles = n;
    }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPrSoftmaxRegs));
        // ---------------------------------------------------------------- softmax + epilogue + Q
        const int h = (warp >= 8) ? 1 : 0;   // key half: columns 64h .. 64h + 63 of every S tile
        const int quarter = warp & 3;        // TMEM lanes 32 * quarter .. + 31
        const int L = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const float sl2 = p.scale_log2;
        const float inv_scale = p.inv_scale;
        const float ln2 = 0.6931471805599453f;
        // Q rows of an item into tensor memory (this half's 64 dims as bf16 pairs), then signal the MMA warp.
        auto write_q = [&](const PfItem &it) {
            int k, j;
            const bool row_ok = pf_row(p, L, k, j) && k < it.ntok;
            uint32_t qv[32];
            if (row_ok) {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    p.q + ((size_t)(it.t0 + it.i0 + k) * p.H + it.g * p.G + j) * kHeadDim + 64 * h);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 v = __ldg(src + c);
                    qv[4 * c] = v.x; qv[4 * c + 1] = v.y; qv[4 * c + 2] = v.z; qv[4 * c + 3] = v.w;
                }
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) qv[c] = 0u;
            }
            INK_TMEM_ST32(tmem_q + lane_addr + 32 * h, qv);
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_rank0(&sh.q_full, rank);
        };
        // next item (round > r) that has tiles, or -1
        auto next_with_tiles = [&](int r, PfItem &nx) {
            for (int r2 = r + 1;; ++r2) {
                const int idx = pr_item_index(r2);
                if (idx >= total) return false;
                nx = pr_item(p, p.pf_items[idx], rank);
                if (nx.ntiles > 0) return true;
            }
        };
        // The two warps that share this lane quarter (w and w + 4) swap one float per row.
        // Buffer b is reused two exchanges later, after the partner has read it.
        uint32_t xseq = 0;
        auto exchange = [&](float mine, float &theirs) {
            const int b = xseq & 1;
            sh.xchg[b][h][L] = mine;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sh.xbar[quarter][b]);
            const bool ok = mbar_wait_warp(&sh.xbar[quarter][b], (xseq >> 1) & 1, abort, p);
            tc_fence_after();
            theirs = sh.xchg[b][h ^ 1][L];
            ++xseq;
            return ok;
        };
        {
            PfItem first;
            if (next_with_tiles(-1, first)) write_q(first);
        }
        uint32_t tc = 0, oseq = 0, bseq = 0;
        for (int r = 0;; ++r) {
            const int idx = pr_item_index(r);
            if (idx >= total || *abort) break;
            const PfItem it = pr_item(p, p.pf_items[idx], rank);
            int k, j;
            const bool row_ok = pf_row(p, L, k, j) && k < it.ntok;
            const int qa = it.qa_min + k;
            int lo = 1, hi = 0;  // visible keys of this row inside the split (empty for padding rows)
            if (row_ok) {
                visible_range(qa, qa, it.Lk, p.causal, p.wl, p.wr, lo, hi);
                lo = max(lo, it.gb * kKeyGroup);
                hi = min(hi, it.ge * kKeyGroup - 1);
            }
            // This row's bias span inside its box: it starts ko floats after the box start
            // (tiles start at multiples of 16 keys, so ko is the same for every tile); the
            // 16-byte chunk that holds it is read whole and the remainder bo is a compile-time
            // shift below.  With warp-strided packing bo is the same for every row of a warp.
            const int kb = k >> p.bias_tok_log2, ki = k & (bias_nb - 1);
            const int ko = (qa - (kTileKeys - 1)) - ((it.qa_min + (kb << p.bias_tok_log2) - (kTileKeys - 1)) & ~3);
            const int bo = ko & 3;
            const uint32_t box_row = smem_u32(bias_smem) + kb * bias_box + ((ki * p.G + j) * bias_w + 4 * (ko >> 2)) * 4;
            const float *rel_row = p.rel ? p.rel + ((size_t)(it.t0 + it.i0 + k) * p.H + it.g * p.G + j) * p.E : nullptr;
            float m_used = -INFINITY;  // raw-score units
            float l = 0.f;             // this half's share of the row sum
            bool ok = true;
            for (int n = 0; n < it.ntiles; ++n) {
                const uint32_t t = tc + n;
                const int ss = t % kSSlots;
                const int j0 = pf_tile_key0(it, n) + 64 * h;  // first key of this half
                if (!mbar_wait_warp_cl(&sh.s_full[ss], (t / kSSlots) & 1, abort, p)) { ok = false; break; }
                tc_fence_after();
                uint32_t sv[64];
                const uint32_t sa = tmem + lane_addr + ss * 128 + 64 * h;
                INK_TMEM_LD32(sa + 0, (sv + 0));
                INK_TMEM_LD32(sa + 32, (sv + 32));
                tc_wait_ld();
                if (pf_tile_bias(p, it, n)) {
                    if (p.bias_tma) {
                        // the tile's two half stages are bias sequence numbers 2 bseq (keys 0-63) and 2 bseq + 1
                        const uint32_t hseq = 2 * bseq + h;
                        const int bs = hseq % kBiasSlots;
                        if (!mbar_wait_warp(&sh.bias_full[bs], (hseq / kBiasSlots) & 1, abort, p)) { ok = false; break; }
                        if (row_ok) {
                            const uint32_t box = box_row + bs * bias_stage;
                            switch (bo) {
                                case 0: bias_add<0>(box, inv_scale, sv); break;
                                case 1: bias_add<1>(box, inv_scale, sv); break;
                                case 2: bias_add<2>(box, inv_scale, sv); break;
                                default: bias_add<3>(box, inv_scale, sv); break;
                            }
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sh.bias_empty[bs]);
                        ++bseq;
                    } else if (row_ok) {  // rows without 16-byte alignment: direct loads
#pragma unroll
                        for (int c = 0; c < 64; ++c) {
                            const int rd = qa - (j0 + c);
                            if (rd >= 0 && rd < p.E)
                                sv[c] = __float_as_uint(fmaf(__ldg(rel_row + rd), inv_scale, __uint_as_float(sv[c])));
                        }
                    }
                }
                if (pf_tile_mask(it, n)) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const int key = j0 + c;
                        if (key < lo || key > hi) sv[c] = __float_as_uint(-INFINITY);
                    }
                }
                // this half's maximum: a tree of three-input maxima (max is exact in any order)
                float m21[22];
#pragma unroll
                for (int i = 0; i < 21; ++i)
                    m21[i] = fmax3(__uint_as_float(sv[3 * i]), __uint_as_float(sv[3 * i + 1]), __uint_as_float(sv[3 * i + 2]));
                m21[21] = __uint_as_float(sv[63]);
                float m7[8];
#pragma unroll
                for (int i = 0; i < 7; ++i) m7[i] = fmax3(m21[3 * i], m21[3 * i + 1], m21[3 * i + 2]);
                m7[7] = m21[21];
                float mx = fmax3(fmax3(m7[0], m7[1], m7[2]), fmax3(m7[3], m7[4], m7[5]), fmaxf(m7[6], m7[7]));
                // Both halves now hold their S values in registers, so either may overwrite the slot.
                float mx_other;
                if (!exchange(mx, mx_other)) { ok = false; break; }
                mx = fmaxf(mx, mx_other);  // the row maximum, identical in both halves
                // The running maximum moves only when it grows past the threshold (or was -inf).
                float alpha = 1.f;
                bool scale_o = false;
                if (mx > m_used && (m_used == -INFINITY || (mx - m_used) * sl2 > (float)kRescaleThreshold)) {
                    alpha = (m_used == -INFINITY) ? 0.f : fast_exp2((m_used - mx) * sl2);
                    l *= alpha;
                    scale_o = n > 0 && m_used != -INFINITY;
                    m_used = mx;
                }
                // The decision is per row, but tcgen05.ld/st are warp-collective: the warp
                // rescales its 32 rows together (its 64 O columns), by 1 where the maximum stayed.
                if (__any_sync(0xffffffffu, scale_o)) {
                    // O holds tiles 0..n-1 once PV(t - 1) is done.  S(t) being complete means every
                    // MMA issued before QK(t) is, so PV(t - 1) is the only one that may be pending
                    // and its phase is the only one of this barrier that can be outstanding.
                    const uint32_t tp = t - 1;
                    if (!mbar_wait_warp_cl(&sh.pv_done[tp % kSSlots], (tp / kSSlots) & 1, abort, p)) { ok = false; break; }
                    tc_fence_after();
                    const float a = scale_o ? alpha : 1.f;
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        uint32_t ov[32];
                        INK_TMEM_LD32(tmem_o + lane_addr + 64 * h + cc * 32, ov);
                        tc_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * a);
                        INK_TMEM_ST32(tmem_o + lane_addr + 64 * h + cc * 32, ov);
                    }
                }
                const float moff = (m_used == -INFINITY) ? 0.f : m_used * sl2;
                const uint64_t sl2x2 = f32x2(sl2, sl2), nmoff2 = f32x2(-moff, -moff);
                uint32_t pk[32];
                uint64_t ls2[2] = {0ull, 0ull};  // four independent partial sums, as two pairs
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    float x0 = __uint_as_float(sv[2 * c]), x1 = __uint_as_float(sv[2 * c + 1]);
                    fma_x2(x0, x1, sl2x2, nmoff2);
                    const float p0 = fast_exp2(x0), p1 = fast_exp2(x1);
                    add_x2(ls2[c & 1], p0, p1);
                    pk[c] = pack_bf16x2(p0, p1);
                }
                l += sum_x2(ls2[0]) + sum_x2(ls2[1]);
                // P of keys 64h .. 64h + 63 as bf16 pairs: columns 32h .. 32h + 31 of the slot
                INK_TMEM_ST32(tmem + lane_addr + ss * 128 + 32 * h, pk);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) arrive_rank0(&sh.p_full[ss], rank);
            }
            if (!ok) break;
            if (it.ntiles > 0) {
                // every QK of this item is complete: the next item's Q may replace this one
                PfItem nx;
                if (next_with_tiles(r, nx)) write_q(nx);
            }
            // epilogue: the row sum is the sum of the two halves' shares
            if (it.ntiles > 0) {
                if (!mbar_wait_warp_cl(&sh.o_full, oseq & 1, abort, p)) break;
                ++oseq;
                tc_fence_after();
            }
            float l_other;
            if (!exchange(l, l_other)) break;
            l += l_other;
            const float inv = l > 0.f ? p.out_scale / l : 0.f;
            const float lse = l > 0.f ? (m_used * sl2 + __log2f(l)) * ln2 : -INFINITY;
            const size_t row = (size_t)(it.t0 + it.i0 + k) * p.H + it.g * p.G + j;
            const bool final_out = it.nact == 1;
            // partial block of (unit, split): rows g * 128 + L
            size_t prow = 0;
            if (!final_out)
                prow = ((size_t)(__ldg(p.unit_off + it.b) + it.qt) * p.S_pf + it.s) * ((size_t)p.Hkv * kTileRows) +
                       (size_t)it.g * kTileRows + L;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int d0 = 64 * h + 32 * cc;  // first of the 32 dims handled here
                uint32_t ov[32];
                if (it.ntiles > 0) {
                    INK_TMEM_LD32(tmem_o + lane_addr + d0, ov);
                    tc_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = 0u;
                }
                if (row_ok) {
                    if (final_out) {
                        uint4 *dst = reinterpret_cast<uint4 *>(p.out + row * kHeadDim + d0);
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint4 w;
                            w.x = pack_bf16x2(__uint_as_float(ov[8 * q4 + 0]) * inv, __uint_as_float(ov[8 * q4 + 1]) * inv);
                            w.y = pack_bf16x2(__uint_as_float(ov[8 * q4 + 2]) * inv, __uint_as_float(ov[8 * q4 + 3]) * inv);
                            w.z = pack_bf16x2(__uint_as_float(ov[8 * q4 + 4]) * inv, __uint_as_float(ov[8 * q4 + 5]) * inv);
                            w.w = pack_bf16x2(__uint_as_float(ov[8 * q4 + 6]) * inv, __uint_as_float(ov[8 * q4 + 7]) * inv);
                            dst[q4] = w;
                        }
                    } else {
                        float4 *dst = reinterpret_cast<float4 *>(p.part_pf_o + prow * kHeadDim + d0);
#pragma unroll
                        for (int q4 = 0; q4 < 8; ++q4)
                            dst[q4] = make_float4(__uint_as_float(ov[4 * q4]) * inv, __uint_as_float(ov[4 * q4 + 1]) * inv,
                                                  __uint_as_float(ov[4 * q4 + 2]) * inv, __uint_as_float(ov[4 * q4 + 3]) * inv);
                    }
                }
            }
            if (row_ok && h == 0) {
                if (final_out) {
                    if (p.lse) p.lse[row] = lse;
                } else {
                    p.part_pf_lse[prow] = lse;
                }
            }
            tc_fence_before();
            tc += it.ntiles;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1 && !*abort)
        drain_pv_done(sh.pv_done, sh.mma_tiles,
                      [&](uint64_t *b, uint32_t par) { return mbar_wait_warp_cl(b, par, abort, p); });
    cluster_sync();  // neither CTA frees tensor memory or exits while its peer may still use the pair's
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

cudaError_t launch_prefill(const Params &p, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                           const CUtensorMap &tm_bias, const CUtensorMap &tm_ks, const CUtensorMap &tm_vs, int grid,
                           size_t smem, cudaStream_t stream)
{
    // setmaxnreg redistributes the registers the CTA was launched with: the split above
    // assumes exactly kPfLaunchRegs per thread, so refuse to launch on any other count.
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, ink_prefill_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kPfLaunchRegs) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(ink_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(ink_prefill_kernel, (unsigned)grid, kPfThreads, smem, stream, p, tm_k, tm_v, tm_bias, tm_ks, tm_vs);
}

}  // namespace ink

namespace ink {

// The 2-SM prefill: clusters of two CTAs, as many as fit at once (one CTA per SM) and no more than the
// pair items need.  `max_pairs` bounds the items; the kernel reads the actual count from the work list.
cudaError_t launch_prefill_pair(const Params &p, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                const CUtensorMap &tm_bias, const CUtensorMap &tm_kh, const CUtensorMap &tm_vh,
                                long long max_pairs, size_t smem, cudaStream_t stream)
{
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, ink_prefill_pair_kernel);
    if (e != cudaSuccess) return e;
    if (fa.numRegs != kPfLaunchRegs) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(ink_prefill_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kPfThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    cfg.gridDim = dim3(2);
    e = cudaOccupancyMaxActiveClusters(&clusters, ink_prefill_pair_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (clusters < 1) return cudaErrorInvalidConfiguration;
    const long long pairs = std::max(1ll, std::min<long long>(clusters, max_pairs));
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, ink_prefill_pair_kernel, p, tm_k, tm_v, tm_bias, tm_kh, tm_vh);
}

}  // namespace ink
