// ink_common.cuh -- shared device-side definitions of the GB300 attention path:
// launch parameters, workspace layout, the work-unit arithmetic every kernel
// must agree on, and thin inline-PTX wrappers (mbarrier, TMA, tcgen05).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ink_attn.h"

namespace ink {

constexpr int kHeadDim = 128;     // D
constexpr int kKeyGroup = 16;     // keys per TMA box / per decode stage
constexpr int kTileKeys = 128;    // keys per prefill KV tile (8 groups)
constexpr int kTileRows = 128;    // packed (token, head) rows per prefill tile
constexpr int kDecodeRows = 16;   // packed rows per KV head in the decode kernel
constexpr int kPfSharedBytes = 2560;  // prefill barriers and bookkeeping (upper bound)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bounded waits give up after ~2 s
constexpr uint32_t kWaitHintNs = 100000;           // longest single suspension of a wait (100 us)

// ---------------------------------------------------------------------------
// Workspace layout (all offsets 256-byte aligned).
//   header | dec_items[int4] | pf_items[int4] | part_lse[f32] | part_o[f32]
// ---------------------------------------------------------------------------
struct WsHeader {
    uint32_t errors;       // INK_DEVERR_* bits
    uint32_t dec_count;    // decode work items written by the prepass
    uint32_t pf_count;     // prefill work items written by the prepass
    uint32_t dec_next;     // dynamic scheduler counter of the decode kernel
    uint32_t pf_next;      // dynamic scheduler counter of the prefill kernel
    uint32_t comb_tokens;  // tokens whose rows the split-KV merge visits (prepass)
    uint32_t stage_pages;  // 16-key pages the K/V staging copies (prepass)
    uint32_t pad[57];
};
static_assert(sizeof(WsHeader) == 256, "header is one 256-byte block");

struct Params {
    // shapes
    int T, B, H, Hkv, G, NB, BS, MAXBLK, max_seqlen_q;
    int D;  // head size: 128 on the tcgen05 prefill / decode path, 64 or 256 on the head-size-generic path
    // scalars
    float softmax_scale, scale_log2, inv_scale;
    int causal, wl, wr, E;
    // tensors
    const __nv_bfloat16 *q, *kc, *vc;
    const int32_t *bt, *seqk, *cu;
    const float *rel;
    __nv_bfloat16 *out;
    float *lse;
    // workspace
    WsHeader *hdr;
    int4 *dec_items;  // (b, split | Lq << 27, t0, Lk): the request's fields ride with the item
    int dec_items_cap;
    int4 *pf_items;
    int pf_items_cap;
    int *dec_off;      // (B+1) first decode item of each request (prepass)
    int *unit_off;     // (B+1) first prefill unit (q tile) of each request (prepass)
    int *comb_off;     // (B+1) first merge-list token of each request (prepass)
    // K/V staging: prefill-shaped requests whose keys fit get a contiguous copy of their K and V
    // pages, per KV head, in the workspace (see ink_stage.cu)
    int *stg_off;      // (B) first staged key of each request, -1 when it reads the paged cache (prepass)
    int *stg_pg_off;   // (B+1) first staged page of each request in the copy's work list (prepass)
    int stage_cap;     // keys per KV head the staging area holds (0: no staging)
    __nv_bfloat16 *ks, *vs;  // staging area: (Hkv, stage_cap, D) each
    int kv_fp8;        // the caches hold E4M3 bytes (the staging copy converts them to bf16)
    float out_scale;   // prefill: multiplies every output row (v_scale of an FP8 cache, else 1)
    // split partials: one block per decode item, and per (prefill unit, split)
    float *part_dec_o, *part_dec_lse;  // (dec_items_cap, dec_rows, D), (dec_items_cap, dec_rows)
    int dec_rows;                      // rows per decode block: (16 / G) * H
    float *part_pf_o, *part_pf_lse;    // (units_cap * S_pf, Hkv * 128, D), (..., Hkv * 128)
    int units_cap;
    int S_pf;                          // splits per prefill unit (1: no partials)
    // scheduling
    int decode_kernel;   // 1: decode-shaped requests go to the decode kernel
    int dec_local;       // 1: a decode-only call of at most 32 requests (each decode CTA finds its first item)
    int chunk_dec;       // 16-key groups per split for decode units
    int chunk_pf;        // 16-key groups per split for prefill units
    int tpt;             // prefill tokens per 128-row tile (128 / G)
    int pair;            // prefill units are pairs of q tiles (2 tpt tokens) for the 2-SM prefill kernel
    int fast_pack;       // prefill: warp-strided token packing (G divides 32)
    int bias_tma;        // prefill: bias staged by TMA (E % 4 == 0)
    int bias_tok_log2;   // prefill: tokens per bias TMA box = 1 << bias_tok_log2
    int bias_w;          // prefill: floats per bias box row (at least pf_bias_width of the box's tokens)
};

// ---------------------------------------------------------------------------
// Requests and work units.  A request is decode-shaped when its Lq*G rows fit
// one mma row block (<= 16) and the decode kernel is enabled; such a request
// is one unit.  Other requests are cut into q tiles of `tpt` tokens.  Each
// unit's visible key range is cut into splits of `chunk` 16-key groups.
// ---------------------------------------------------------------------------
struct Req {
    int t0, Lq, Lk;
    bool ok;
    uint32_t err;
};

// Request b from its cu_seqlens_q pair (c0, c1) and cache_seqlens entry lk, validated.
__device__ __forceinline__ Req make_req(const Params &p, int c0, int c1, int lk)
{
    Req r;
    r.t0 = c0;
    r.Lq = c1 - c0;
    r.Lk = lk;
    r.err = 0;
    if (!(c0 >= 0 && c0 <= c1 && c1 <= p.T)) r.err |= INK_DEVERR_CU_SEQLENS;
    if (r.Lq > p.max_seqlen_q) r.err |= INK_DEVERR_SEQLEN_Q;
    if (lk < 0 || (long long)lk > (long long)p.MAXBLK * p.BS) r.err |= INK_DEVERR_SEQLEN_K;
    r.ok = (r.err == 0);
    return r;
}

__device__ __forceinline__ Req load_req(const Params &p, int b)
{
    return make_req(p, __ldg(p.cu + b), __ldg(p.cu + b + 1), __ldg(p.seqk + b));
}

__device__ __forceinline__ bool is_decode_req(const Params &p, const Req &r)
{
    return p.decode_kernel && r.Lq * p.G <= kDecodeRows;
}

// Inclusive visible key range of the rows whose q_abs lies in [qa0, qa1].
// Both ends are non-decreasing in q_abs, so the union is [lo(qa0), hi(qa1)].
__host__ __device__ __forceinline__ void visible_range(int qa0, int qa1, int Lk, int causal, int wl,
                                                       int wr, int &lo, int &hi)
{
    lo = 0;
    if (wl >= 0) lo = max(0, qa0 - wl);
    hi = Lk - 1;
    if (causal) hi = min(hi, qa1);
    if (wr >= 0) hi = min(hi, qa1 + wr);
}

struct UnitSplit {
    int gb, ge;    // 16-key groups [gb, ge) of this split (may be empty)
    int nact;      // number of splits of the unit (>= 1)
    int klo, khi;  // unit visible key range (inclusive; khi < klo when empty)
};

__host__ __device__ __forceinline__ UnitSplit unit_split(int qa0, int qa1, int Lk, int causal, int wl,
                                                         int wr, int chunk, int s)
{
    UnitSplit u;
    visible_range(qa0, qa1, Lk, causal, wl, wr, u.klo, u.khi);
    if (u.khi < u.klo) {
        u.nact = 1;
        u.gb = u.ge = 0;
        return u;
    }
    const int g0 = u.klo / kKeyGroup, g1 = u.khi / kKeyGroup + 1;
    u.nact = (g1 - g0 + chunk - 1) / chunk;
    u.gb = g0 + s * chunk;
    u.ge = min(g1, u.gb + chunk);
    if (u.ge < u.gb) u.ge = u.gb;
    return u;
}

// Keys a staged request occupies in the staging area: its cache length rounded up to whole
// 128-key tiles, so that every tile box of the request stays inside its own keys.
__host__ __device__ __forceinline__ int stage_keys_of(int Lk) { return (Lk + kTileKeys - 1) / kTileKeys * kTileKeys; }

// Prefill bias staging, by half tiles: one TMA box holds, for one 64-key half of a 128-key
// tile, the rel_logits rows of nb consecutive tokens (all G heads).  The distance span of
// token k + 1 starts one key later than token k's, so a common start rounded down to 16
// bytes and a width of 64 + 3 + (nb - 1) floats, rounded up to 16 bytes, cover every token
// of the box (the softmax reads 17 whole 16-byte chunks from the one holding a row's start).
constexpr int kPfKvSlots = 3;     // prefill K/V ring (32 KB slots; 4 to 6 slots measured no faster)
constexpr int kPfBiasSlots = 3;   // prefill bias ring (half-tile stages)
__host__ __device__ __forceinline__ int pf_bias_width(int nb) { return (70 + nb) & ~3; }
// Bytes a box of w-float rows transfers, and its shared-memory footprint (a TMA destination is
// 128-byte aligned).  A wider row than the minimum changes where the rows fall among the shared-memory
// banks (the host picks the width).
__host__ __device__ __forceinline__ int pf_bias_box_bytes(int G, int nb, int w) { return nb * G * w * 4; }
__host__ __device__ __forceinline__ int pf_bias_box_stride(int G, int nb, int w)
{
    return (pf_bias_box_bytes(G, nb, w) + 127) & ~127;
}
// One stage: the boxes of a q tile of tpt tokens, for one key half.
__host__ __device__ __forceinline__ int pf_bias_stage_bytes(int G, int tpt, int nb, int w)
{
    return (tpt + nb - 1) / nb * pf_bias_box_stride(G, nb, w);
}
// The prefill kernel's shared-memory layout: K/V ring, bias ring, bookkeeping.
__host__ __device__ __forceinline__ size_t pf_layout_bytes(int G, int tpt, int nb, int w)
{
    return (size_t)kPfKvSlots * 32768 + (size_t)kPfBiasSlots * pf_bias_stage_bytes(G, tpt, nb, w) + kPfSharedBytes;
}
// The 2-SM prefill kernel's: a ring of 16 KB K/V halves, then the same bias ring and bookkeeping.
constexpr int kPrKvSlots = 4;
__host__ __device__ __forceinline__ size_t pr_layout_bytes(int G, int tpt, int nb, int w)
{
    return (size_t)kPrKvSlots * 16384 + (size_t)kPfBiasSlots * pf_bias_stage_bytes(G, tpt, nb, w) + kPfSharedBytes;
}

// Packed row of (token offset k, head j) inside a prefill tile, and back.
__host__ __device__ __forceinline__ int pf_row_of(int fast_pack, int G, int k, int j)
{
    return fast_pack ? 32 * (k & 3) + (k >> 2) * G + j : k * G + j;
}

__device__ __forceinline__ void report(const Params &p, uint32_t bits)
{
    if (bits) atomicOr(&p.hdr->errors, bits);
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *ptr)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

// Bytes of dynamic shared memory this CTA was launched with.
__device__ __forceinline__ uint32_t dynamic_smem_bytes()
{
    uint32_t n;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(n));
    return n;
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of a phase parity (acquire when it has completed).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same test for a whole warp: true only when every lane has seen the phase complete
// (each lane acquires for itself), so the lanes agree and stay converged.
__device__ __forceinline__ bool warp_poll(uint64_t *bar, uint32_t parity)
{
    return __all_sync(0xffffffffu, mbar_test_wait(bar, parity));
}

// try_wait whose suspension is bounded by a hint (ns), so that a caller can
// look at the clock between attempts.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(kWaitHintNs)
        : "memory");
    return ok != 0;
}

// Bounded wait on a phase parity.  Returns false (and raises the timeout
// bit, and sets *abort) when the phase did not complete within the limit or
// another role already gave up.  The clock is checked after every bounded
// suspension, so a stuck pipeline ends within about kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort,
                                          const Params &p)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_hint(bar, parity)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            report(p, INK_DEVERR_TIMEOUT);
            *abort = 1;
            return false;
        }
    }
}

// The same wait for a whole warp: every lane waits and the lanes agree on the
// outcome, so that a warp stays converged for the warp-collective instructions
// (tcgen05.ld/st, mma.sync, shuffles) that follow even when a wait gives up.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t *bar, uint32_t parity, volatile int *abort,
                                               const Params &p)
{
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, p));
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// TMA tiled loads into shared memory, completing on an mbarrier.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_hint(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                                 uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d_hint(void *dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                                 uint64_t *bar, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 128-byte swizzle of a byte offset inside a 1024-byte aligned atom: the
// 16-byte chunk index (bits 4-6) is XOR-ed with the row within the atom
// (bits 7-9).  This is the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B
// and the tensor core reads with layout type "128B swizzle".
__device__ __forceinline__ uint32_t swz128(uint32_t off)
{
    return off ^ (((off >> 7) & 7u) << 4);
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float fast_exp2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Blackwell's three-input maximum and paired fp32 arithmetic (each lane of a pair rounds as the scalar op).
__device__ __forceinline__ float fmax3(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ uint64_t f32x2(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

// (a.lo * b.lo + c.lo, a.hi * b.hi + c.hi) for a = (lo, hi)
__device__ __forceinline__ void fma_x2(float &lo, float &hi, uint64_t b, uint64_t c)
{
    asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%0, %1};\n\tfma.rn.f32x2 t, t, %2, %3;\n\tmov.b64 {%0, %1}, t;\n\t}"
        : "+f"(lo), "+f"(hi)
        : "l"(b), "l"(c));
}

// acc += (lo, hi), lane by lane
__device__ __forceinline__ void add_x2(uint64_t &acc, float lo, float hi)
{
    asm("{\n\t.reg .b64 t;\n\tmov.b64 t, {%1, %2};\n\tadd.rn.f32x2 %0, %0, t;\n\t}" : "+l"(acc) : "f"(lo), "f"(hi));
}

__device__ __forceinline__ float sum_x2(uint64_t v)
{
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}

// Programmatic dependent launch.  Every kernel of a call (and the KV append) is launched so that it
// may begin while the kernel before it in the stream is finishing: its CTAs set up shared memory,
// barriers and tensor memory, then pdl_wait() blocks until the previous kernel has completed and its
// writes are visible -- before any global memory is read or written -- and pdl_launch_dependents()
// lets the next kernel start its own set-up.  A kernel triggers only after its wait returns, so at
// most two consecutive kernels of a stream overlap, and only in those set-up phases.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                              cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Host-side launchers, one per translation unit (ink_api.cu calls these).
// decode_only: the call can hold only decode-shaped requests (max_seqlen_q * G <= 16 with the decode kernel)
cudaError_t launch_prepass(const Params &p, bool decode_only, cudaStream_t stream);
// kv_fp8: K/V pages are E4M3 bytes dequantized with k_scale / v_scale (decode kernel only); per_sm: CTAs an SM
// the kernel is compiled and sized for (1 or 2); small: no item of the call has more than 8 packed rows;
// one_tok: every decode-shaped request has one query token (max_seqlen_q 1).
cudaError_t launch_decode(const Params &p, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                          const CUtensorMap &tm_bias, int nstages, int stage_bytes, int kv_bytes,
                          int bias_slot_bytes, int kv_fp8, float k_scale, float v_scale, int per_sm, int small,
                          int one_tok, int grid, size_t smem, cudaStream_t stream);
cudaError_t launch_prefill(const Params &p, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                           const CUtensorMap &tm_bias, const CUtensorMap &tm_ks, const CUtensorMap &tm_vs, int grid,
                           size_t smem, cudaStream_t stream);
cudaError_t launch_prefill_pair(const Params &p, const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                const CUtensorMap &tm_bias, const CUtensorMap &tm_kh, const CUtensorMap &tm_vh,
                                long long max_pairs, size_t smem, cudaStream_t stream);
// max_splits: the most splits any row of the call was cut into (sizes the warps a row gets)
cudaError_t launch_combine(const Params &p, int sms, int max_splits, cudaStream_t stream);
cudaError_t launch_stage(const Params &p, int sms, cudaStream_t stream);
cudaError_t launch_generic(const Params &p, int sms, cudaStream_t stream);
cudaError_t launch_append(const ink_attn_dims *d, const void *key, const void *value, void *key_cache,
                          void *value_cache, const int64_t *slot_mapping, uint32_t *flags, int sms,
                          cudaStream_t stream);
cudaError_t launch_append_fp8(const ink_attn_dims *d, const void *key, const void *value, void *key_cache,
                              void *value_cache, const int64_t *slot_mapping, float k_scale, float v_scale,
                              uint32_t *flags, int sms, cudaStream_t stream);

}  // namespace ink
