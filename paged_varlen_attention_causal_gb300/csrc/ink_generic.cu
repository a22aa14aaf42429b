// ink_generic.cu -- paged varlen GQA attention with the relative bias for head
// sizes other than 128 (64 and 256, the other sizes a paged backend serves).
//
// It consumes the prefill work list the prepass builds (one item = request, q
// tile of 128 / G tokens, split, KV head: 128 packed rows, row L = token L / G,
// head L % G of the KV head's group) and writes the same outputs: the bf16 rows
// and lse, or per-split partials that the split-KV merge combines.  Decode-shaped
// requests go to the decode kernel (templated on the head size) unless a warp's
// d-slice there would be narrower than 16 (D 64 with one KV head): those, too,
// become items here.
//
// Eight warps, 16 rows each; persistent CTAs take items from a shared counter.
// Per item: the q tile goes to shared memory once; 64-key tiles of K and V are
// gathered page by page (block_table) with 16-byte cp.async copies into a ring
// (4 tiles deep at D = 64, two CTAs per SM; 2 deep at D = 256), later tiles
// loading while the current one is used.  Per tile and warp:
//   S = Q K^T        mma.sync m16n8k16 (bf16 in, fp32 accumulate), Q and K
//                    fragments by ldmatrix from padded rows (no bank conflicts)
//   S += bias        rel_logits[token, head, q_abs - key] for 0 <= rd < E
//   masks            causal, window, split and tail bounds -> -inf
//   online softmax   running max and sum per row in registers (log2 domain),
//                    the output rescaled when the maximum grows
//   O += P V         P from the S accumulators as bf16, V by ldmatrix.trans
// The output accumulator is D / 2 fp32 registers per thread (128 at D = 256).
#include <algorithm>

#include "ink_common.cuh"

namespace ink {
namespace {

constexpr int kGenThreads = 256;
constexpr int kGenKeys = 64;  // keys per K/V tile

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid)
{
    // src-size 0 fills the 16 bytes with zeros
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int D>
struct GenLayout {
    static constexpr int kRowBytes = D * 2 + 16;  // padded shared-memory row: ldmatrix rows hit distinct banks
    static constexpr int kQBytes = kTileRows * kRowBytes;
    static constexpr int kKvBytes = kGenKeys * kRowBytes;  // one K or V tile
    static constexpr int kStages = D <= 64 ? 4 : 2;        // K/V ring depth (shared memory bounds it at D = 256)
    static constexpr int kCtasPerSm = D <= 64 ? 2 : 1;
    static constexpr int kBytes = kQBytes + 2 * kStages * kKvBytes;  // Q, then K0 V0 K1 V1 ...
    static constexpr int kChunks = D * 2 / 16;                        // 16-byte chunks per row
};

template <int D>
__global__ void __launch_bounds__(kGenThreads, GenLayout<D>::kCtasPerSm) ink_generic_kernel(const Params p)
{
    using L = GenLayout<D>;
    extern __shared__ __align__(128) uint8_t gsmem[];
    const uint32_t sbase = smem_u32(gsmem);
    const uint32_t s_q = sbase;
    auto s_k = [&](int buf) { return sbase + L::kQBytes + (2 * buf) * L::kKvBytes; };
    auto s_v = [&](int buf) { return sbase + L::kQBytes + (2 * buf + 1) * L::kKvBytes; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_wait();
    pdl_launch_dependents();
    const int total = (int)*(volatile uint32_t *)&p.hdr->pf_count;
    const float sl2 = p.scale_log2;
    const float log2e = 1.4426950408889634f;

    // CTA c takes item c first, then the next free item of the shared counter (items come longest first, so
    // a CTA that lands late or shares its SM with a long item does not hold back the launch)
    __shared__ int s_next;
    for (int idx = blockIdx.x; idx < total;) {
        const int4 w = p.pf_items[idx];
        const int b = w.x, qt = w.y, s = w.z, g = w.w;
        const Req r = load_req(p, b);
        const int i0 = qt * p.tpt;
        const int ntok = min(p.tpt, r.Lq - i0);
        const int qa_min = i0 + r.Lk - r.Lq;
        const UnitSplit u = unit_split(qa_min, qa_min + ntok - 1, r.Lk, p.causal, p.wl, p.wr, p.chunk_pf, s);
        const int key_lo = u.gb * kKeyGroup, key_hi = min(u.ge * kKeyGroup, r.Lk);  // split keys [key_lo, key_hi)
        const int ntiles = key_hi > key_lo ? (key_hi - key_lo + kGenKeys - 1) / kGenKeys : 0;
        const int32_t *bt_row = p.bt + (size_t)b * p.MAXBLK;

        // q tile: packed row R = token R / G, head R % G (rows past the tile's tokens are zero)
        for (int c = tid; c < kTileRows * L::kChunks; c += kGenThreads) {
            const int row = c / L::kChunks, ch = c % L::kChunks;
            const int k = row / p.G, j = row % p.G;
            const bool ok = k < ntok;
            const __nv_bfloat16 *src =
                p.q + ((size_t)(r.t0 + i0 + (ok ? k : 0)) * p.H + g * p.G + j) * D + ch * 8;
            cp_async16(s_q + row * L::kRowBytes + ch * 16, ok ? (const void *)src : (const void *)p.q, ok);
        }
        // K and V tile n into ring buffer n % kStages: keys past the split or Lk, and keys on a bad page,
        // read as zeros
        auto load_kv = [&](int n) {
            const int buf = n % L::kStages;
            const int j0 = key_lo + n * kGenKeys;
            for (int c = tid; c < kGenKeys * L::kChunks; c += kGenThreads) {
                const int kr = c / L::kChunks, ch = c % L::kChunks;
                const int key = j0 + kr;
                bool ok = key < key_hi;
                size_t row = 0;
                if (ok) {
                    const int pid = __ldg(bt_row + key / p.BS);
                    if (pid >= 0 && pid < p.NB) {
                        row = ((size_t)pid * p.BS + key % p.BS) * p.Hkv + g;
                    } else {
                        ok = false;
                        if (ch == 0) report(p, INK_DEVERR_PAGE_ID);
                    }
                }
                const uint32_t off = kr * L::kRowBytes + ch * 16;
                cp_async16(s_k(buf) + off, ok ? (const void *)(p.kc + row * D + ch * 8) : (const void *)p.kc, ok);
                cp_async16(s_v(buf) + off, ok ? (const void *)(p.vc + row * D + ch * 8) : (const void *)p.vc, ok);
            }
        };
        // prologue: the q tile and the first kStages - 1 K/V tiles, one commit group each
#pragma unroll
        for (int st = 0; st < L::kStages - 1; ++st) {
            if (st < ntiles) load_kv(st);
            cp_async_commit();
        }

        // this thread's two rows of the warp's 16: R0 = 16 warp + lane / 4, R1 = R0 + 8
        const int R0 = 16 * warp + (lane >> 2), R1 = R0 + 8;
        const int k0 = R0 / p.G, j0r = R0 % p.G, k1 = R1 / p.G, j1r = R1 % p.G;
        const bool ok0 = k0 < ntok, ok1 = k1 < ntok;
        const bool warp_live = (16 * warp) / p.G < ntok;  // warp-uniform: some row of the warp is a real row
        const int qa0 = qa_min + k0, qa1 = qa_min + k1;
        int lo0 = 1, hi0 = 0, lo1 = 1, hi1 = 0;  // visible keys inside the split (empty for padding rows)
        if (ok0) {
            visible_range(qa0, qa0, r.Lk, p.causal, p.wl, p.wr, lo0, hi0);
            lo0 = max(lo0, key_lo);
            hi0 = min(hi0, key_hi - 1);
        }
        if (ok1) {
            visible_range(qa1, qa1, r.Lk, p.causal, p.wl, p.wr, lo1, hi1);
            lo1 = max(lo1, key_lo);
            hi1 = min(hi1, key_hi - 1);
        }
        const float *rel0 = (p.E > 0 && ok0) ? p.rel + ((size_t)(r.t0 + i0 + k0) * p.H + g * p.G + j0r) * p.E : nullptr;
        const float *rel1 = (p.E > 0 && ok1) ? p.rel + ((size_t)(r.t0 + i0 + k1) * p.H + g * p.G + j1r) * p.E : nullptr;

        float o[D / 8][4];
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // log2-domain running max, partial sums

        for (int n = 0; n < ntiles; ++n) {
            const int buf = n % L::kStages;
            cp_async_wait<L::kStages - 2>();  // tile n (and the q tile) landed: groups complete in order
            __syncthreads();                  // ... for every thread; and tile n - 1's buffer is free again
            if (n + L::kStages - 1 < ntiles) load_kv(n + L::kStages - 1);
            cp_async_commit();
            if (warp_live) {
                // this tile's bias terms first, so that their loads are in flight during S = Q K^T
                const int jt = key_lo + n * kGenKeys;
                float bz[8][4];
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int key = jt + 8 * nt + 2 * (lane & 3) + e;
                        const int rd0 = qa0 - key, rd1 = qa1 - key;
                        bz[nt][e] = (rel0 && rd0 >= 0 && rd0 < p.E) ? __ldg(rel0 + rd0) : 0.f;
                        bz[nt][2 + e] = (rel1 && rd1 >= 0 && rd1 < p.E) ? __ldg(rel1 + rd1) : 0.f;
                    }
                }
                // S = Q K^T for the warp's 16 rows and the tile's 64 keys
                float sc[8][4];
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
                const int mi = lane >> 3, mr = lane & 7;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(s_q + (16 * warp + mr + 8 * (mi & 1)) * L::kRowBytes + (16 * kk + 8 * (mi >> 1)) * 2, a0, a1,
                            a2, a3);
#pragma unroll
                    for (int np = 0; np < 4; ++np) {  // key tiles 2np, 2np + 1
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4(s_k(buf) + (16 * np + mr + 8 * (mi >> 1)) * L::kRowBytes + (16 * kk + 8 * (mi & 1)) * 2,
                                b0, b1, b2, b3);
                        mma_bf16(sc[2 * np], a0, a1, a2, a3, b0, b1);
                        mma_bf16(sc[2 * np + 1], a0, a1, a2, a3, b2, b3);
                    }
                }
                // scale (log2 domain), bias, masks; this tile's row maxima
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int key = jt + 8 * nt + 2 * (lane & 3) + e;
                        float v0 = fmaf(bz[nt][e], log2e, sc[nt][e] * sl2);
                        float v1 = fmaf(bz[nt][2 + e], log2e, sc[nt][2 + e] * sl2);
                        if (key < lo0 || key > hi0) v0 = -INFINITY;
                        if (key < lo1 || key > hi1) v1 = -INFINITY;
                        sc[nt][e] = v0;
                        sc[nt][2 + e] = v1;
                        mx0 = fmaxf(mx0, v0);
                        mx1 = fmaxf(mx1, v1);
                    }
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
                // rescale what was accumulated (alpha = 0 when nothing was; rows that saw no key stay empty)
                const float al0 = (m0 == -INFINITY) ? 0.f : fast_exp2(m0 - mn0);
                const float al1 = (m1 == -INFINITY) ? 0.f : fast_exp2(m1 - mn1);
                m0 = mn0;
                m1 = mn1;
                const float off0 = (mn0 == -INFINITY) ? 0.f : mn0, off1 = (mn1 == -INFINITY) ? 0.f : mn1;
                l0 *= al0;
                l1 *= al1;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt) {
                    o[nt][0] *= al0; o[nt][1] *= al0;
                    o[nt][2] *= al1; o[nt][3] *= al1;
                }
                // P = exp2(S - m) as bf16 A fragments (keys 16 kk .. 16 kk + 15), then O += P V
                uint32_t pa[4][4];
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    const float p00 = fast_exp2(sc[nt][0] - off0), p01 = fast_exp2(sc[nt][1] - off0);
                    const float p10 = fast_exp2(sc[nt][2] - off1), p11 = fast_exp2(sc[nt][3] - off1);
                    l0 += p00 + p01;
                    l1 += p10 + p11;
                    pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(p00, p01);
                    pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(p10, p11);
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
                    for (int dp = 0; dp < D / 16; ++dp) {  // d tiles 2dp, 2dp + 1
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(s_v(buf) + (16 * kk + mr + 8 * (mi & 1)) * L::kRowBytes + (16 * dp + 8 * (mi >> 1)) * 2,
                                  b0, b1, b2, b3);
                        mma_bf16(o[2 * dp], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b0, b1);
                        mma_bf16(o[2 * dp + 1], pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3], b2, b3);
                    }
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();  // the q tile and the ring are rewritten by the next item

        // epilogue: the row sums over the quad, then out = O / l and lse, or the split's partials
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        const bool final_out = u.nact == 1;
        const float ln2 = 0.6931471805599453f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const bool ok = half ? ok1 : ok0;
            if (!ok) continue;
            const int k = half ? k1 : k0, j = half ? j1r : j0r, R = half ? R1 : R0;
            const float l = half ? l1 : l0, m = half ? m1 : m0;
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const float lse = l > 0.f ? (m + __log2f(l)) * ln2 : -INFINITY;
            if (final_out) {
                const size_t row = (size_t)(r.t0 + i0 + k) * p.H + g * p.G + j;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt) {
                    const int d = 8 * nt + 2 * (lane & 3);
                    *reinterpret_cast<uint32_t *>(p.out + row * D + d) =
                        pack_bf16x2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
                }
                if (p.lse && (lane & 3) == 0) p.lse[row] = lse;
            } else {
                const size_t prow = ((size_t)(__ldg(p.unit_off + b) + qt) * p.S_pf + s) * ((size_t)p.Hkv * kTileRows) +
                                    (size_t)g * kTileRows + R;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt) {
                    const int d = 8 * nt + 2 * (lane & 3);
                    *reinterpret_cast<float2 *>(p.part_pf_o + prow * D + d) =
                        make_float2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
                }
                if ((lane & 3) == 0) p.part_pf_lse[prow] = lse;
            }
        }
        // every thread reads s_next before the next item's barriers, which thread 0 passes before rewriting it
        if (tid == 0) s_next = (int)gridDim.x + (int)atomicAdd(&p.hdr->pf_next, 1u);
        __syncthreads();
        idx = s_next;
    }
}

template <int D>
cudaError_t launch_generic_d(const Params &p, int sms, cudaStream_t stream)
{
    const int smem = GenLayout<D>::kBytes;
    cudaError_t e = cudaFuncSetAttribute(ink_generic_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ink_generic_kernel<D>, kGenThreads, smem);
    if (e != cudaSuccess) return e;
    const long long grid = std::min<long long>((long long)sms * std::max(1, per_sm), std::max(1, p.pf_items_cap));
    return launch_pdl(ink_generic_kernel<D>, (unsigned)grid, kGenThreads, (size_t)smem, stream, p);
}

}  // namespace

// Every request of the call as 128-row items over the paged cache; head sizes 64 and 256.
cudaError_t launch_generic(const Params &p, int sms, cudaStream_t stream)
{
    switch (p.D) {
        case 64: return launch_generic_d<64>(p, sms, stream);
        case 256: return launch_generic_d<256>(p, sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace ink
