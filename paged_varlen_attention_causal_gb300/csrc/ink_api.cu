// ink_api.cu -- host plan and C ABI: argument validation, the split
// heuristic re-derived for the GB300 SM count, workspace layout, TMA tensor
// maps, and the stream-ordered launches (prepass, decode, prefill, combine).
// Nothing here synchronises the host; nothing here allocates.
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cudaTypedefs.h>

#include "ink_common.cuh"

namespace ink {

namespace {

constexpr int kMaxDevices = 64;
constexpr size_t kSmemLimit = 232448;  // 227 KB of dynamic shared memory per CTA on sm_100-class SMs
constexpr size_t kSmemPerSm = 233472;  // 228 KB of shared memory per SM
constexpr size_t kSmemReserved = 1024;  // shared memory the system reserves per CTA
constexpr int kDecSharedBytes = 512;   // mbarriers + item ring of the decode kernel (upper bound)
constexpr int kDecMaxStages = 8;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct TimingHook {
    cudaEvent_t start = nullptr, stop = nullptr;
};
TimingHook g_hooks[7];
std::mutex g_hook_mutex;
std::atomic<unsigned long long> g_launches{0};

// Launch `fn` (returning cudaError_t) between the optional timing events of `kernel`.
template <typename F>
cudaError_t timed_launch(int kernel, cudaStream_t stream, F &&fn)
{
    TimingHook h;
    {
        std::lock_guard<std::mutex> lk(g_hook_mutex);
        h = g_hooks[kernel];
    }
    if (h.start && cudaEventRecord(h.start, stream) != cudaSuccess) return cudaErrorInvalidValue;
    cudaError_t e = fn();
    if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
    if (e == cudaSuccess && h.stop) e = cudaEventRecord(h.stop, stream);
    return e;
}

int sm_count_of_current_device()
{
    static int cache[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < kMaxDevices && cache[dev] > 0) return cache[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < kMaxDevices) cache[dev] = n;
    return n;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

struct Plan {
    int G = 0, tpt = 0, fast_pack = 0, decode_kernel = 0, bias_tok_log2 = 0, bias_w = 0;
    bool pair = false;  // prefill units are pairs of q tiles for the 2-SM prefill kernel
    int S_dec = 1, S_pf = 1, chunk_dec = 1, chunk_pf = 1;
    int dec_rows = 0, lq_dec = 0;
    long long dec_cap = 0, pf_cap = 0, units_cap = 0;
    bool any_prefill = false, any_decode = false;
    // workspace offsets
    size_t off_dec_items = 0, off_pf_items = 0, off_dec_off = 0, off_unit_off = 0, off_comb_off = 0;
    size_t off_stg_off = 0, off_stg_pg_off = 0;
    size_t off_pdo = 0, off_pdl = 0, off_ppo = 0, off_ppl = 0, total = 0;
};

bool dims_ok(const ink_attn_dims *d)
{
    return d && d->num_tokens >= 0 && d->batch >= 1 && d->num_heads >= 1 && d->num_kv_heads >= 1 &&
           d->num_heads % d->num_kv_heads == 0 && d->head_dim >= 1 && d->num_blocks >= 1 && d->block_size >= 1 &&
           d->max_blocks_per_seq >= 1;
}

// Head sizes: 128 runs the tcgen05 prefill and the decode kernel; 64 and 256 run the
// head-size-generic kernel.
bool head_dim_supported(int D) { return D == 64 || D == kHeadDim || D == 256; }

bool dims_supported(const ink_attn_dims *d)
{
    const int G = d->num_heads / d->num_kv_heads;
    return head_dim_supported(d->head_dim) && d->block_size % kKeyGroup == 0 && G <= kTileRows &&
           (long long)d->num_blocks * d->block_size < (1ll << 31);
}

long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// Upper bound on the visible 16-key groups of a unit whose q rows span
// `span` consecutive positions.
long long max_groups(const ink_attn_dims *d, int span, int causal, int wl, int wr)
{
    const long long keys = (long long)d->max_blocks_per_seq * d->block_size;
    long long g = ceil_div(keys, kKeyGroup);
    if (wl >= 0 && (causal || wr >= 0)) {
        const long long right = causal ? (wr >= 0 ? std::min(wr, 0) : 0) : wr;
        const long long w = (long long)wl + span + right;
        g = std::min(g, ceil_div(w, kKeyGroup) + 1);
    }
    return std::max(1ll, g);
}

// Split counts re-derived for this GPU from the page heuristic's intent:
// fill every SM several times over, never split below 16 keys, and keep the
// partial traffic a small fraction of the KV bytes.
int heuristic_splits_decode(long long batch, long long groups, int sms)
{
    const long long target_chunk = 32;  // 512 keys per split
    const long long s_wave = ceil_div(4ll * sms, batch);  // units that fill every SM four times
    long long s = ceil_div(groups, target_chunk);
    if (batch * s < 4ll * sms) s = s_wave;
    s = std::min<long long>(s, std::max<long long>(64, s_wave));  // long rows: whole waves, fewer partials
    s = std::min<long long>(s, ceil_div(groups, 16));  // at least 256 keys a split: shorter items cost more
                                                        // in per-item setup than they gain in balance
    // ... unless that leaves SMs idle: then one full wave, with at least 128 keys a split
    if (batch * s < sms && groups >= 8 * ceil_div(sms, batch)) s = ceil_div(sms, batch);
    s = std::min<long long>(s, groups);
    s = std::min<long long>(s, 1024);
    return (int)std::max(1ll, s);
}

int heuristic_splits_prefill(long long units, long long groups, int sms)
{
    if (units >= 2ll * sms) return 1;
    long long s = ceil_div(2ll * sms, std::max(1ll, units));
    s = std::min<long long>(s, ceil_div(groups, 8));  // at least one 128-key tile per split
    s = std::min<long long>(s, 256);
    return (int)std::max(1ll, s);
}

// Shared-memory wavefronts of the softmax's 16-byte bias loads (one load instruction of each of the four
// lane quarters), for the worst start phase of a box: each 8-lane phase of a 128-bit load takes as many
// wavefronts as the most 16-byte chunks it has in one bank group (address / 16 mod 8).  Rows follow the
// kernels' packing (pf_row) and box layout: the row of token k, head j starts ((k mod nb) G + j) w floats
// into box k / nb, plus whole chunks for the token's shift inside the box.
int bias_load_waves(int G, int tpt, int fast_pack, int nb, int w)
{
    const int wc = w / 4, box_chunks = pf_bias_box_stride(G, nb, w) / 16;
    int worst = 0;
    for (int c0 = 0; c0 < 4; ++c0) {
        int tot = 0;
        for (int q = 0; q < 4; ++q)
            for (int ph = 0; ph < 4; ++ph) {
                int cnt[8] = {0, 0, 0, 0, 0, 0, 0, 0}, mx = 0;
                for (int l = 8 * ph; l < 8 * ph + 8; ++l) {
                    int k, j;
                    if (fast_pack) {
                        k = 4 * (l / G) + q;
                        j = l % G;
                    } else {
                        k = (32 * q + l) / G;
                        j = (32 * q + l) % G;
                    }
                    if (k >= tpt) continue;
                    const int kb = k / nb, ki = k % nb, ckb = (c0 + kb * nb) & 3;
                    const int off = kb * box_chunks + (ki * G + j) * wc + ((ki + ckb) >> 2);
                    mx = std::max(mx, ++cnt[off & 7]);
                }
                tot += mx;
            }
        worst = std::max(worst, tot);
    }
    return worst;
}

bool make_plan(const ink_attn_dims *d, int max_seqlen_q, int num_splits, int causal, int wl, int wr, int sms,
               Plan &pl)
{
    const int T = d->num_tokens, B = d->batch, H = d->num_heads, Hkv = d->num_kv_heads;
    pl.G = H / Hkv;
    pl.tpt = kTileRows / pl.G;
    // prefill bias boxes: as many tokens per box (up to 8) as the shared-memory budget allows
    for (int lg = 3; lg >= 0; --lg) {
        if ((1 << lg) > pl.tpt) continue;
        const size_t need = 1024 + pf_layout_bytes(pl.G, pl.tpt, 1 << lg, pf_bias_width(1 << lg));
        if (need <= kSmemLimit || lg == 0) {
            pl.bias_tok_log2 = lg;
            break;
        }
    }
    pl.bias_w = pf_bias_width(1 << pl.bias_tok_log2);
    const bool generic = d->head_dim != kHeadDim;  // head-size-generic kernel for the prefill-shaped requests
    pl.fast_pack = (!generic && 32 % pl.G == 0) ? 1 : 0;
    const long long msq = std::min<long long>(max_seqlen_q, std::max(T, 1));
    // the decode kernel serves every head size where a warp's d-slice (D * Hkv / 8) is at least 16 wide and
    // its ring holds two stages of a bf16 page (K and V of every KV head, 16 keys) plus the bias room
    const long long dec_stage =
        (2ll * Hkv * 32 * d->head_dim + std::min<long long>(kDecodeRows / std::max(1, pl.G), msq) *
                                            (((long long)H * 80 + 127) & ~127ll) + 1023) & ~1023ll;
    pl.decode_kernel = (Hkv == 1 || Hkv == 2 || Hkv == 4 || Hkv == 8) && pl.G <= kDecodeRows &&
                               d->head_dim * Hkv / 8 >= 16 && 1024 + 2 * dec_stage + kDecSharedBytes <= (long long)kSmemLimit
                           ? 1
                           : 0;
    pl.any_decode = pl.decode_kernel != 0;
    pl.any_prefill = !pl.decode_kernel || msq * pl.G > kDecodeRows;
    if (!pl.decode_kernel) pl.any_decode = false;
    pl.lq_dec = pl.decode_kernel ? (int)std::min<long long>(kDecodeRows / pl.G, msq) : 0;
    pl.dec_rows = pl.lq_dec * H;

    const long long g_dec = max_groups(d, kDecodeRows / std::max(1, pl.G), causal, wl, wr);
    const long long g_pf = max_groups(d, pl.tpt, causal, wl, wr);
    if (num_splits > 0) {
        pl.S_dec = pl.S_pf = num_splits;
    } else {
        pl.S_dec = heuristic_splits_decode(B, g_dec, sms);
        const long long units = (long long)B * Hkv * ceil_div(msq * pl.G, kTileRows);
        pl.S_pf = heuristic_splits_prefill(units, g_pf, sms);
    }
    pl.chunk_dec = (int)std::max(1ll, ceil_div(g_dec, pl.S_dec));
    pl.chunk_pf = (int)std::max(1ll, ceil_div(g_pf, pl.S_pf));
    if (pl.S_pf > 1) pl.chunk_pf = (int)(ceil_div(pl.chunk_pf, 8) * 8);  // whole 128-key tiles
    const long long sdec_eff = ceil_div(g_dec, pl.chunk_dec);
    const long long spf_eff = ceil_div(g_pf, pl.chunk_pf);
    pl.S_pf = (int)std::max(1ll, spf_eff);
    // 2-SM prefill: unsplit prefill units become pairs of q tiles (the one-CTA prefill kernel keeps split
    // units); a pair spans 2 tpt query positions, so its one chunk must cover the visible groups of that span
    // Its bias boxes: the shape (tokens per box, row width) with the fewest shared-memory wavefronts for
    // the softmax's loads, then the smallest stage, then the most tokens per box, among those that fit.
    int pr_lg = -1, pr_w = 0, pr_waves = 0, pr_stage = 0;
    if (!generic && pl.any_prefill && pl.S_pf == 1) {
        for (int lg = 3; lg >= 0; --lg) {
            const int nb = 1 << lg;
            if (nb > pl.tpt) continue;
            for (int w = pf_bias_width(nb); w <= pf_bias_width(nb) + 32; w += 4) {
                if (pr_layout_bytes(pl.G, pl.tpt, nb, w) + 1024 > kSmemLimit) break;
                const int wv = bias_load_waves(pl.G, pl.tpt, pl.fast_pack, nb, w);
                const int st = pf_bias_stage_bytes(pl.G, pl.tpt, nb, w);
                if (pr_lg < 0 || wv < pr_waves || (wv == pr_waves && st < pr_stage)) {
                    pr_lg = lg, pr_w = w, pr_waves = wv, pr_stage = st;
                }
            }
        }
    }
    pl.pair = pr_lg >= 0;
    if (pl.pair) {
        pl.bias_tok_log2 = pr_lg;
        pl.bias_w = pr_w;
        pl.chunk_pf = (int)std::max(1ll, max_groups(d, 2 * pl.tpt, causal, wl, wr));
    }

    pl.dec_cap = pl.any_decode ? (long long)B * sdec_eff : 0;
    pl.units_cap = pl.any_prefill ? ceil_div(T, pl.tpt) + B : 0;
    pl.pf_cap = pl.any_prefill ? pl.units_cap * pl.S_pf * Hkv : 0;
    if (pl.dec_cap > (1ll << 30) || pl.pf_cap > (1ll << 30)) return false;

    size_t off = sizeof(WsHeader);
    pl.off_dec_items = off; off = align256(off + sizeof(int4) * (size_t)pl.dec_cap);
    pl.off_pf_items = off; off = align256(off + sizeof(int4) * (size_t)pl.pf_cap);
    pl.off_dec_off = off; off = align256(off + sizeof(int) * (size_t)(B + 1));
    pl.off_unit_off = off; off = align256(off + sizeof(int) * (size_t)(B + 1));
    pl.off_comb_off = off; off = align256(off + sizeof(int) * (size_t)(B + 1));
    pl.off_stg_off = off; off = align256(off + sizeof(int) * (size_t)B);
    pl.off_stg_pg_off = off; off = align256(off + sizeof(int) * (size_t)(B + 1));
    const bool dec_parts = pl.any_decode && sdec_eff > 1;
    const bool pf_parts = pl.any_prefill && pl.S_pf > 1;
    const size_t dec_rows_total = dec_parts ? (size_t)pl.dec_cap * pl.dec_rows : 0;
    const size_t pf_rows_total = pf_parts ? (size_t)pl.units_cap * pl.S_pf * Hkv * kTileRows : 0;
    pl.off_pdl = off; off = align256(off + sizeof(float) * dec_rows_total);
    pl.off_pdo = off; off = align256(off + sizeof(float) * dec_rows_total * d->head_dim);
    pl.off_ppl = off; off = align256(off + sizeof(float) * pf_rows_total);
    pl.off_ppo = off; off = align256(off + sizeof(float) * pf_rows_total * d->head_dim);
    pl.total = off;
    return true;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// FP8 cache scales: normal fp32 numbers whose reciprocal is normal too, so that the append's
// quotient x * (1 / scale), corrected by one remainder step, is the correctly rounded x / scale
// (and a zero input stays zero), and the attention's scale products stay finite.
bool fp8_scale_ok(float s) { return std::isfinite(s) && s >= 0x1p-126f && s <= 0x1p126f; }

bool encode(CUtensorMap *map, CUtensorMapDataType dt, int rank, const void *base, const cuuint64_t *dims,
            const cuuint64_t *strides, const cuuint32_t *box, CUtensorMapSwizzle swz)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(map, dt, (cuuint32_t)rank, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Element format of the K/V caches.
struct KvFormat {
    int fp8;          // 0: bf16; 1: E4M3 bytes (decode-shaped calls only)
    float k_scale, v_scale;
};

ink_status attn_impl(const ink_attn_dims *dims, const void *q, const void *key_cache, const void *value_cache,
                     const KvFormat &kv, const int32_t *block_table, const int32_t *cache_seqlens,
                     const int32_t *cu_seqlens_q, int32_t max_seqlen_q, float softmax_scale, int causal,
                     int32_t window_left, int32_t window_right, int32_t rel_extent, const float *rel_logits,
                     int32_t num_splits, void *out, float *lse, void *workspace, size_t workspace_bytes,
                     ink_stream_t stream_handle);

}  // namespace
}  // namespace ink

using namespace ink;

extern "C" {

int32_t ink_attn_version(void) { return 100; }

void ink_set_timing_events(ink_kernel_id kernel, void *start_event, void *stop_event)
{
    if ((int)kernel < 1 || (int)kernel > 6) return;
    std::lock_guard<std::mutex> lk(g_hook_mutex);
    g_hooks[kernel].start = static_cast<cudaEvent_t>(start_event);
    g_hooks[kernel].stop = static_cast<cudaEvent_t>(stop_event);
}

uint64_t ink_launch_count(void) { return (uint64_t)g_launches.load(); }

const char *ink_status_string(ink_status s)
{
    switch (s) {
        case INK_OK: return "ok";
        case INK_ERR_INVALID_ARG: return "invalid argument";
        case INK_ERR_UNSUPPORTED: return "unsupported configuration";
        case INK_ERR_WORKSPACE: return "workspace too small";
        case INK_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

size_t ink_rel_attn_workspace_size(const ink_attn_dims *dims, int32_t max_seqlen_q, int32_t num_splits)
{
    if (!dims_ok(dims) || max_seqlen_q < 1 || num_splits < 0 || !dims_supported(dims)) return 0;
    const int sms = sm_count_of_current_device();
    Plan pl;
    // no window: the largest split count the heuristic can choose for these dims
    if (!make_plan(dims, max_seqlen_q, num_splits, 1, -1, -1, sms > 0 ? sms : 152, pl)) return 0;
    Plan pl2;  // non-causal needs no more than causal; take the max of both to be safe
    if (make_plan(dims, max_seqlen_q, num_splits, 0, -1, -1, sms > 0 ? sms : 152, pl2))
        return std::max(pl.total, pl2.total);
    return pl.total;
}

size_t ink_rel_attn_stage_bytes(const ink_attn_dims *dims, int64_t prefill_kv_tokens)
{
    if (!dims_ok(dims) || prefill_kv_tokens < 0) return 0;
    if (dims->head_dim != kHeadDim) return 0;  // the head-size-generic kernel reads the paged cache directly
    // every staged request occupies whole 128-key tiles: at most 127 keys of rounding per request
    const long long keys = prefill_kv_tokens + (long long)dims->batch * (kTileKeys - 1);
    const long long tiles = (keys + kTileKeys - 1) / kTileKeys;
    return (size_t)tiles * kTileKeys * dims->num_kv_heads * kHeadDim * 2 * 2;
}

int32_t ink_rel_attn_num_splits(const ink_attn_dims *dims, int32_t max_seqlen_q, int32_t max_kv_len,
                                int32_t window_left, int32_t window_right)
{
    if (!dims_ok(dims) || max_seqlen_q < 1 || max_kv_len < 0 || !dims_supported(dims)) return 0;
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return 0;
    ink_attn_dims d = *dims;
    const long long blocks = ceil_div(std::max(1, max_kv_len), d.block_size);
    d.max_blocks_per_seq = (int)std::min<long long>(d.max_blocks_per_seq, blocks);
    Plan pl;
    if (!make_plan(&d, max_seqlen_q, 0, 1, window_left, window_right, sms, pl)) return 0;
    const long long msq = std::min<long long>(max_seqlen_q, std::max(d.num_tokens, 1));
    const bool decode_shaped = pl.decode_kernel && msq * pl.G <= kDecodeRows;
    return decode_shaped ? pl.S_dec : pl.S_pf;
}

ink_status ink_rel_attn_varlen(const ink_attn_dims *dims, const void *q, const void *key_cache,
                               const void *value_cache, const int32_t *block_table, const int32_t *cache_seqlens,
                               const int32_t *cu_seqlens_q, int32_t max_seqlen_q, float softmax_scale, int causal,
                               int32_t window_left, int32_t window_right, int32_t rel_extent,
                               const float *rel_logits, int32_t num_splits, void *out, float *lse, void *workspace,
                               size_t workspace_bytes, ink_stream_t stream_handle)
{
    return attn_impl(dims, q, key_cache, value_cache, KvFormat{0, 1.f, 1.f}, block_table, cache_seqlens,
                     cu_seqlens_q, max_seqlen_q, softmax_scale, causal, window_left, window_right, rel_extent,
                     rel_logits, num_splits, out, lse, workspace, workspace_bytes, stream_handle);
}

ink_status ink_rel_attn_varlen_fp8kv(const ink_attn_dims *dims, const void *q, const void *key_cache,
                                     const void *value_cache, float k_scale, float v_scale,
                                     const int32_t *block_table, const int32_t *cache_seqlens,
                                     const int32_t *cu_seqlens_q, int32_t max_seqlen_q, float softmax_scale,
                                     int causal, int32_t window_left, int32_t window_right, int32_t rel_extent,
                                     const float *rel_logits, int32_t num_splits, void *out, float *lse,
                                     void *workspace, size_t workspace_bytes, ink_stream_t stream_handle)
{
    if (!fp8_scale_ok(k_scale) || !fp8_scale_ok(v_scale)) return INK_ERR_INVALID_ARG;
    return attn_impl(dims, q, key_cache, value_cache, KvFormat{1, k_scale, v_scale}, block_table, cache_seqlens,
                     cu_seqlens_q, max_seqlen_q, softmax_scale, causal, window_left, window_right, rel_extent,
                     rel_logits, num_splits, out, lse, workspace, workspace_bytes, stream_handle);
}

}  // extern "C"

namespace ink {
namespace {

ink_status attn_impl(const ink_attn_dims *dims, const void *q, const void *key_cache, const void *value_cache,
                     const KvFormat &kv, const int32_t *block_table, const int32_t *cache_seqlens,
                     const int32_t *cu_seqlens_q, int32_t max_seqlen_q, float softmax_scale, int causal,
                     int32_t window_left, int32_t window_right, int32_t rel_extent, const float *rel_logits,
                     int32_t num_splits, void *out, float *lse, void *workspace, size_t workspace_bytes,
                     ink_stream_t stream_handle)
{
    if (!dims_ok(dims)) return INK_ERR_INVALID_ARG;
    if (!q || !key_cache || !value_cache || !block_table || !cache_seqlens || !cu_seqlens_q || !out || !workspace)
        return INK_ERR_INVALID_ARG;
    if (max_seqlen_q < 1 || window_left < -1 || window_right < -1 || rel_extent < 0 || num_splits < 0)
        return INK_ERR_INVALID_ARG;
    if (!(std::isfinite(softmax_scale) && softmax_scale > 0.f)) return INK_ERR_INVALID_ARG;
    if (rel_extent > 0 && !rel_logits) return INK_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) || !aligned(out, 16) ||
        !aligned(block_table, 4) || !aligned(cache_seqlens, 4) || !aligned(cu_seqlens_q, 4) ||
        (lse && !aligned(lse, 4)) || (rel_logits && !aligned(rel_logits, 4)) || !aligned(workspace, 256))
        return INK_ERR_INVALID_ARG;
    if (!dims_supported(dims)) return INK_ERR_UNSUPPORTED;
    if (kv.fp8 && dims->head_dim != kHeadDim) return INK_ERR_UNSUPPORTED;  // an E4M3 cache is read at D = 128 only
    if (dims->num_tokens == 0) return INK_OK;

    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return INK_ERR_CUDA;
    Plan pl;
    if (!make_plan(dims, max_seqlen_q, num_splits, causal ? 1 : 0, window_left, window_right, sms, pl))
        return INK_ERR_UNSUPPORTED;
    if (workspace_bytes < pl.total) return INK_ERR_WORKSPACE;

    const int T = dims->num_tokens, H = dims->num_heads, Hkv = dims->num_kv_heads, E = rel_extent;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    Params p;
    memset(&p, 0, sizeof p);
    const bool generic = dims->head_dim != kHeadDim;  // head size 64 or 256: prefill by the head-size-generic kernel
    p.T = T; p.B = dims->batch; p.H = H; p.Hkv = Hkv; p.G = pl.G; p.NB = dims->num_blocks;
    p.D = dims->head_dim;
    p.BS = dims->block_size; p.MAXBLK = dims->max_blocks_per_seq; p.max_seqlen_q = max_seqlen_q;
    p.softmax_scale = softmax_scale;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.inv_scale = 1.0f / softmax_scale;
    p.causal = causal ? 1 : 0; p.wl = window_left; p.wr = window_right; p.E = E;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.kc = static_cast<const __nv_bfloat16 *>(key_cache);
    p.vc = static_cast<const __nv_bfloat16 *>(value_cache);
    p.bt = block_table; p.seqk = cache_seqlens; p.cu = cu_seqlens_q;
    p.rel = E > 0 ? rel_logits : nullptr;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.lse = lse;
    p.hdr = reinterpret_cast<WsHeader *>(ws);
    p.dec_items = reinterpret_cast<int4 *>(ws + pl.off_dec_items);
    p.dec_items_cap = (int)pl.dec_cap;
    p.pf_items = reinterpret_cast<int4 *>(ws + pl.off_pf_items);
    p.pf_items_cap = (int)pl.pf_cap;
    p.dec_off = reinterpret_cast<int *>(ws + pl.off_dec_off);
    p.unit_off = reinterpret_cast<int *>(ws + pl.off_unit_off);
    p.comb_off = reinterpret_cast<int *>(ws + pl.off_comb_off);
    p.part_dec_lse = reinterpret_cast<float *>(ws + pl.off_pdl);
    p.part_dec_o = reinterpret_cast<float *>(ws + pl.off_pdo);
    p.dec_rows = pl.dec_rows;
    p.stg_off = reinterpret_cast<int *>(ws + pl.off_stg_off);
    p.stg_pg_off = reinterpret_cast<int *>(ws + pl.off_stg_pg_off);
    // K/V staging: workspace beyond the minimum holds whole 128-key tiles of K and V planes for
    // prefill-shaped requests (an FP8 cache and decode-only calls stage nothing)
    {
        const size_t per_key = (size_t)Hkv * kHeadDim * 2 * 2;  // K and V, every KV head
        const size_t extra = workspace_bytes - pl.total;
        long long cap = (long long)(extra / per_key) / kTileKeys * kTileKeys;
        cap = std::min<long long>(cap, 1ll << 24);
        p.stage_cap = (!generic && pl.any_prefill && cap >= kTileKeys) ? (int)cap : 0;
        // an FP8 cache reaches the prefill only through the staging copy (converted to bf16)
        if (kv.fp8 && pl.any_prefill && p.stage_cap == 0) return INK_ERR_WORKSPACE;
        p.ks = reinterpret_cast<__nv_bfloat16 *>(ws + pl.total);
        p.vs = p.ks + (size_t)Hkv * p.stage_cap * kHeadDim;
    }
    p.part_pf_lse = reinterpret_cast<float *>(ws + pl.off_ppl);
    p.part_pf_o = reinterpret_cast<float *>(ws + pl.off_ppo);
    p.units_cap = (int)pl.units_cap;
    p.S_pf = pl.S_pf;
    p.decode_kernel = pl.decode_kernel;
    p.chunk_dec = pl.chunk_dec;
    p.chunk_pf = pl.chunk_pf;
    p.tpt = pl.tpt;
    // 2-SM prefill: pairs of q tiles per cluster when the prefill units are not split
    p.pair = pl.pair ? 1 : 0;
    p.fast_pack = pl.fast_pack;
    p.bias_tok_log2 = pl.bias_tok_log2;
    p.bias_w = pl.bias_w;
    p.kv_fp8 = kv.fp8;
    p.out_scale = 1.f;

    // tensor maps: K/V as (d, Hkv, keys) bf16 with 64 x 1 x 16 boxes, 128-byte swizzle
    alignas(64) CUtensorMap tm_k, tm_v, tm_vp, tm_kd, tm_vd, tm_bdec, tm_bpf;
    memset(&tm_k, 0, sizeof tm_k); memset(&tm_v, 0, sizeof tm_v); memset(&tm_vp, 0, sizeof tm_vp);
    memset(&tm_kd, 0, sizeof tm_kd); memset(&tm_vd, 0, sizeof tm_vd);
    memset(&tm_bdec, 0, sizeof tm_bdec); memset(&tm_bpf, 0, sizeof tm_bpf);
    if (kv.fp8) {
        // E4M3 K and V as (128 d bytes, keys, 1, Hkv): one 128 x 16 x 1 x Hkv box per page lands as
        // [KV head][16 keys][128 B], 128-byte swizzle
        const cuuint64_t gd8[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)dims->num_blocks * dims->block_size, 1,
                                   (cuuint64_t)Hkv};
        const cuuint64_t gs8[3] = {(cuuint64_t)Hkv * kHeadDim, (cuuint64_t)kHeadDim, (cuuint64_t)kHeadDim};
        const cuuint32_t box8[4] = {(cuuint32_t)kHeadDim, (cuuint32_t)kKeyGroup, 1, (cuuint32_t)Hkv};
        if (!encode(&tm_kd, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, key_cache, gd8, gs8, box8, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode(&tm_vd, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, value_cache, gd8, gs8, box8, CU_TENSOR_MAP_SWIZZLE_128B))
            return INK_ERR_CUDA;
    } else if (!generic) {
        const cuuint64_t gd[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)Hkv,
                                  (cuuint64_t)dims->num_blocks * dims->block_size};
        const cuuint64_t gs[2] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)Hkv * kHeadDim * 2};
        const cuuint32_t box[3] = {64, 1, (cuuint32_t)kKeyGroup};
        if (!encode(&tm_k, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, key_cache, gd, gs, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode(&tm_v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, value_cache, gd, gs, box, CU_TENSOR_MAP_SWIZZLE_128B))
            return INK_ERR_CUDA;
        // prefill V as (64 d, keys, d half, Hkv) with one 64 x 16 x 2 box per page: the box lands as
        // [d half][16 keys][128 B], so a page needs one copy instead of two
        const cuuint64_t gd4[4] = {64, (cuuint64_t)dims->num_blocks * dims->block_size, 2, (cuuint64_t)Hkv};
        const cuuint64_t gs4[3] = {(cuuint64_t)Hkv * kHeadDim * 2, 128, (cuuint64_t)kHeadDim * 2};
        const cuuint32_t box4[4] = {64, (cuuint32_t)kKeyGroup, 2, 1};
        if (!encode(&tm_vp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, value_cache, gd4, gs4, box4, CU_TENSOR_MAP_SWIZZLE_128B))
            return INK_ERR_CUDA;
    }
    if (!kv.fp8 && pl.decode_kernel && Hkv <= 8) {
        // decode K and V as (64 d, keys, D / 64 d-blocks, Hkv) with a box over every KV head, which lands as
        // [KV head][d-block][16 keys][128 B]: a whole page per copy
        const int D = dims->head_dim, nb = D / 64;
        const cuuint64_t gdd[4] = {64, (cuuint64_t)dims->num_blocks * dims->block_size, (cuuint64_t)nb,
                                   (cuuint64_t)Hkv};
        const cuuint64_t gsd[3] = {(cuuint64_t)Hkv * D * 2, 128, (cuuint64_t)D * 2};
        const cuuint32_t boxd[4] = {64, (cuuint32_t)kKeyGroup, (cuuint32_t)nb, (cuuint32_t)Hkv};
        if (!encode(&tm_kd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, key_cache, gdd, gsd, boxd, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode(&tm_vd, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, value_cache, gdd, gsd, boxd, CU_TENSOR_MAP_SWIZZLE_128B))
            return INK_ERR_CUDA;
    }
    // bias maps: rel_logits as (E, H, T) fp32, no swizzle; needs 16-byte rows
    bool bias_dec_tma = false, bias_pf_tma = false;
    if (E > 0 && E % 4 == 0 && aligned(rel_logits, 16)) {
        const cuuint64_t gd[3] = {(cuuint64_t)E, (cuuint64_t)H, (cuuint64_t)T};
        const cuuint64_t gs[2] = {(cuuint64_t)E * 4, (cuuint64_t)E * H * 4};
        if (H <= 256) {
            const cuuint32_t box[3] = {20, (cuuint32_t)H, 1};
            bias_dec_tma = encode(&tm_bdec, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, rel_logits, gd, gs, box,
                                  CU_TENSOR_MAP_SWIZZLE_NONE);
        }
        const cuuint32_t box2[3] = {(cuuint32_t)pl.bias_w, (cuuint32_t)pl.G,
                                    (cuuint32_t)(1 << pl.bias_tok_log2)};
        if (!generic)
            bias_pf_tma = encode(&tm_bpf, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, rel_logits, gd, gs, box2,
                                 CU_TENSOR_MAP_SWIZZLE_NONE);
    }

    // staging planes as (64 d, keys, d half, Hkv): one (64, 128, 2, 1) box is a 128-key tile of one
    // KV head, 32 KB of consecutive bytes, landing as [d half][128 keys][128 B] (128-byte swizzle)
    alignas(64) CUtensorMap tm_ks, tm_vs, tm_kh, tm_vh;
    memset(&tm_ks, 0, sizeof tm_ks); memset(&tm_vs, 0, sizeof tm_vs);
    memset(&tm_kh, 0, sizeof tm_kh); memset(&tm_vh, 0, sizeof tm_vh);
    if (p.stage_cap > 0) {
        const cuuint64_t gds[4] = {64, (cuuint64_t)p.stage_cap, 2, (cuuint64_t)Hkv};
        const cuuint64_t gss[3] = {(cuuint64_t)kHeadDim * 2, 128, (cuuint64_t)p.stage_cap * kHeadDim * 2};
        const cuuint32_t boxs[4] = {64, (cuuint32_t)kTileKeys, 2, 1};
        if (!encode(&tm_ks, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.ks, gds, gss, boxs, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode(&tm_vs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.vs, gds, gss, boxs, CU_TENSOR_MAP_SWIZZLE_128B))
            return INK_ERR_CUDA;
        if (p.pair) {
            // the 2-SM prefill's halves: 64 keys with both d halves (K), or one d half of 128 keys (V)
            const cuuint32_t boxk[4] = {64, 64, 2, 1}, boxv[4] = {64, (cuuint32_t)kTileKeys, 1, 1};
            if (!encode(&tm_kh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.ks, gds, gss, boxk, CU_TENSOR_MAP_SWIZZLE_128B) ||
                !encode(&tm_vh, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, p.vs, gds, gss, boxv, CU_TENSOR_MAP_SWIZZLE_128B))
                return INK_ERR_CUDA;
        }
    }

    // 1. device-side plan
    if (timed_launch(INK_KERNEL_PREPASS, stream, [&] { return launch_prepass(p, !pl.any_prefill, stream); }) !=
        cudaSuccess)
        return INK_ERR_CUDA;

    // 1b. K/V staging copy for the prefill
    if (p.stage_cap > 0) {
        if (timed_launch(INK_KERNEL_STAGE, stream, [&] { return launch_stage(p, sms, stream); }) != cudaSuccess)
            return INK_ERR_CUDA;
    }

    // 2. decode kernel
    if (pl.any_decode && pl.dec_cap > 0) {
        Params pd = p;
        pd.bias_tma = bias_dec_tma ? 1 : 0;
        const int kv_bytes = Hkv * (kv.fp8 ? 2048 : 32 * dims->head_dim);  // one 16-key page of K (or V), all KV heads
        const int bias_slot = (H * 80 + 127) & ~127;
        // bias room for the most query tokens a decode-shaped request of this call can have (Lq <=
        // max_seqlen_q, and Lq * G <= 16): with one token per request the stages are smaller and the ring
        // holds more pages (an E4M3 decode batch: 6 stages instead of 5)
        const int bias_bytes = pl.lq_dec * bias_slot;
        const int stage_bytes = (2 * kv_bytes + bias_bytes + 1023) & ~1023;
        // Two CTAs an SM when half of its shared memory still holds a ring of three stages (E4M3 pages, or
        // bf16 pages of at most 4 KV heads): twice the warps in flight for the per-page chain of dependent
        // steps, at 96 registers a thread.
        const int nst2 = (int)((kSmemPerSm / 2 - kSmemReserved - 1024 - kDecSharedBytes) / stage_bytes);
        // (the two-an-SM build reads the bias band only from its stages: a call whose bias cannot go by TMA
        // keeps one CTA an SM)
        const int per_sm = nst2 >= 3 && (E == 0 || bias_dec_tma) ? 2 : 1;
        // every decode item has at most lq_dec tokens (longer ones are rejected against max_seqlen_q)
        const int small = pl.lq_dec * pl.G <= 8 ? 1 : 0;
        const int one_tok = pl.lq_dec == 1 ? 1 : 0;  // max_seqlen_q 1: one query token a request
        int nst = per_sm == 2 ? nst2 : (int)((kSmemLimit - 1024 - kDecSharedBytes) / stage_bytes);
        nst = std::min(nst, kDecMaxStages);
        if (nst < 2) return INK_ERR_UNSUPPORTED;
        const size_t smem = 1024 + (size_t)nst * stage_bytes + kDecSharedBytes;
        const int grid = (int)std::min<long long>((long long)per_sm * sms, pl.dec_cap);
        // A decode-only call of at most 32 requests (the one-warp prepass) whose items all fit one wave of CTAs:
        // each decode CTA finds its one item itself and streams it while the prepass runs.  With more items
        // than CTAs the early start measured slower (the next item is claimed only after the wait).
        pd.dec_local = (!pl.any_prefill && dims->batch <= 32 && pl.dec_cap <= (long long)per_sm * sms) ? 1 : 0;
        if (timed_launch(INK_KERNEL_DECODE, stream, [&] {
                return launch_decode(pd, tm_kd, tm_vd, tm_bdec, nst, stage_bytes, kv_bytes, bias_slot, kv.fp8,
                                     kv.k_scale, kv.v_scale, per_sm, small, one_tok, grid, smem, stream);
            }) != cudaSuccess)
            return INK_ERR_CUDA;
    }

    // 3. prefill kernel: head sizes 64 and 256 run the head-size-generic kernel over the 128-row items
    if (generic && pl.any_prefill && pl.pf_cap > 0) {
        if (timed_launch(INK_KERNEL_PREFILL, stream, [&] { return launch_generic(p, sms, stream); }) != cudaSuccess)
            return INK_ERR_CUDA;
    } else if (pl.any_prefill && pl.pf_cap > 0) {
        Params pp = p;
        pp.bias_tma = bias_pf_tma ? 1 : 0;
        if (kv.fp8) {
            // staged K and V hold the E4M3 values themselves: k_scale joins the softmax scale, v_scale the output
            const float eff = softmax_scale * kv.k_scale;
            pp.scale_log2 = eff * 1.4426950408889634f;
            pp.inv_scale = 1.0f / eff;
            pp.out_scale = kv.v_scale;
        }
        // layout plus up to 1 KB for aligning the base (the kernel checks what it was given)
        const size_t layout = p.pair ? pr_layout_bytes(pl.G, pl.tpt, 1 << pl.bias_tok_log2, pl.bias_w)
                                     : pf_layout_bytes(pl.G, pl.tpt, 1 << pl.bias_tok_log2, pl.bias_w);
        if (layout > kSmemLimit) return INK_ERR_UNSUPPORTED;
        const size_t smem = std::min(layout + 1024, kSmemLimit);
        const int grid = (int)std::min<long long>(sms, pl.pf_cap);
        if (timed_launch(INK_KERNEL_PREFILL, stream, [&] {
                return p.pair ? launch_prefill_pair(pp, tm_k, tm_v, tm_bpf, tm_kh, tm_vh, pl.pf_cap, smem, stream)
                              : launch_prefill(pp, tm_k, tm_vp, tm_bpf, tm_ks, tm_vs, grid, smem, stream);
            }) != cudaSuccess)
            return INK_ERR_CUDA;
    }

    // 4. split-KV merge
    const long long sdec_eff = ceil_div(max_groups(dims, kDecodeRows / std::max(1, pl.G), causal, window_left,
                                                   window_right),
                                        pl.chunk_dec);
    if ((pl.any_decode && sdec_eff > 1) || (pl.any_prefill && pl.S_pf > 1)) {
        const int max_splits = (int)std::max<long long>(pl.any_decode ? sdec_eff : 1, pl.any_prefill ? pl.S_pf : 1);
        if (timed_launch(INK_KERNEL_COMBINE, stream, [&] { return launch_combine(p, sms, max_splits, stream); }) !=
            cudaSuccess)
            return INK_ERR_CUDA;
    }
    return INK_OK;
}

}  // namespace
}  // namespace ink

extern "C" {

ink_status ink_reshape_and_cache(const ink_attn_dims *dims, const void *key, const void *value, void *key_cache,
                                 void *value_cache, const int64_t *slot_mapping, uint32_t *flags,
                                 ink_stream_t stream_handle)
{
    if (!dims || dims->num_tokens < 0 || dims->num_kv_heads < 1 || dims->head_dim < 1 || dims->num_blocks < 1 ||
        dims->block_size < 1)
        return INK_ERR_INVALID_ARG;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return INK_ERR_INVALID_ARG;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
        !aligned(slot_mapping, 8) || (flags && !aligned(flags, 4)))
        return INK_ERR_INVALID_ARG;
    if (!head_dim_supported(dims->head_dim)) return INK_ERR_UNSUPPORTED;
    if (dims->num_tokens == 0) return INK_OK;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return INK_ERR_CUDA;
    if (timed_launch(INK_KERNEL_APPEND, stream, [&] {
            return launch_append(dims, key, value, key_cache, value_cache, slot_mapping, flags, sms, stream);
        }) != cudaSuccess)
        return INK_ERR_CUDA;
    return INK_OK;
}

ink_status ink_reshape_and_cache_fp8(const ink_attn_dims *dims, const void *key, const void *value, void *key_cache,
                                     void *value_cache, const int64_t *slot_mapping, float k_scale, float v_scale,
                                     uint32_t *flags, ink_stream_t stream_handle)
{
    if (!dims || dims->num_tokens < 0 || dims->num_kv_heads < 1 || dims->head_dim < 1 || dims->num_blocks < 1 ||
        dims->block_size < 1)
        return INK_ERR_INVALID_ARG;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return INK_ERR_INVALID_ARG;
    if (!fp8_scale_ok(k_scale) || !fp8_scale_ok(v_scale)) return INK_ERR_INVALID_ARG;
    if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
        !aligned(slot_mapping, 8) || (flags && !aligned(flags, 4)))
        return INK_ERR_INVALID_ARG;
    if (dims->head_dim != kHeadDim) return INK_ERR_UNSUPPORTED;
    if (dims->num_tokens == 0) return INK_OK;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    const int sms = sm_count_of_current_device();
    if (sms <= 0) return INK_ERR_CUDA;
    if (timed_launch(INK_KERNEL_APPEND, stream, [&] {
            return launch_append_fp8(dims, key, value, key_cache, value_cache, slot_mapping, k_scale, v_scale, flags,
                                     sms, stream);
        }) != cudaSuccess)
        return INK_ERR_CUDA;
    return INK_OK;
}

ink_status ink_rel_attn_read_device_errors(const void *workspace, ink_stream_t stream_handle, uint32_t *flags)
{
    if (!workspace || !flags) return INK_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, stream) != cudaSuccess) return INK_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return INK_ERR_CUDA;
    *flags = v;
    return INK_OK;
}

}  // extern "C"
