/*
 * ink_attn.h -- C ABI of the GB300 (sm_103a) paged varlen causal GQA
 * attention with the Inkling additive relative bias.
 *
 * The operation is the one `inkling_fa4_rel_attention` performs in vLLM's
 * fa4_rel_attention.py, as quoted and explained by the article
 * "vllm中提取Inkling FA4 Relative Attention算子基础的base优化版本"
 * (nxmr.cn/news/19446): its wrapper signature (the article's layer 3
 * "参数签名"), the score modification that adds the bias (score_mod_rel_bias)
 * and the split-KV count (inkling_fa4_num_splits).  The split-KV merge
 * follows the log-sum-exp Phase 2 of the "paged_attention_v2_pytorch.py"
 * page (dev.modelhub.org.cn), and the paged/varlen conventions follow the
 * mini-vllm tutorial "Step 15: FlashAttention 封装" (block_table and
 * cu_seqlens sections).
 *
 * Definition.  For request b with Lq = cu_seqlens_q[b+1] - cu_seqlens_q[b]
 * and Lk = cache_seqlens[b], token i < Lq (global row t = cu_seqlens_q[b] + i)
 * and query head h (KV head g = h / (num_heads / num_kv_heads)):
 *     q_abs = i + Lk - Lq                      (bottom-right causal alignment)
 *     key j < Lk is visible iff (!causal || j <= q_abs)
 *                             && (window_left  < 0 || j >= q_abs - window_left)
 *                             && (window_right < 0 || j <= q_abs + window_right)
 *     s_j = softmax_scale * <q[t][h], K_j[g]> + bias,  rd = q_abs - j,
 *     bias = rel_logits[t][h][rd] if 0 <= rd < rel_extent, else 0
 *     K_j = key_cache[block_table[b][j / block_size]][j % block_size]
 *     out[t][h] = sum_j softmax(s)_j V_j[g]   (bf16, round to nearest even)
 *     lse[t][h] = ln sum_j exp(s_j)           (natural log, fp32)
 * A row with no visible key gets out = 0 and lse = -inf.
 *
 * Besides the attention over a bf16 cache (ink_rel_attn_varlen and its
 * allocation-free twin ink_rel_attn_varlen_static) the library has the same
 * attention over an FP8 (E4M3) cache with per-tensor scales
 * (ink_rel_attn_varlen_fp8kv) and the KV append that
 * precedes attention on every step (ink_reshape_and_cache, and
 * ink_reshape_and_cache_fp8 which quantizes into an E4M3 cache).
 *
 * The attention and append calls are asynchronous on `stream`, allocate
 * nothing and perform no host synchronisation; ink_rel_attn_read_device_errors
 * is the one call that waits for its stream.  The only state kept between
 * calls is a per-device SM count, the measurement hooks below and the static
 * scratch area of ink_rel_attn_varlen_static.
 */
#ifndef INK_ATTN_H
#define INK_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define INK_API __attribute__((visibility("default")))
#else
#define INK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle (the same type as cudaStream_t / CUstream). */
typedef struct CUstream_st *ink_stream_t;

/* Shapes a C interface cannot read from tensors. */
typedef struct {
    int32_t num_tokens;          /* T: rows of q, out, lse, rel_logits      */
    int32_t batch;               /* B: requests                               */
    int32_t num_heads;           /* H: query heads                            */
    int32_t num_kv_heads;        /* Hkv: KV heads, H % Hkv == 0               */
    int32_t head_dim;            /* D: 64, 128 or 256 (FP8 cache: 128 only)   */
    int32_t num_blocks;          /* physical pages in each cache              */
    int32_t block_size;          /* keys per page: a multiple of 16           */
    int32_t max_blocks_per_seq;  /* width of block_table                      */
} ink_attn_dims;

typedef enum {
    INK_OK = 0,
    INK_ERR_INVALID_ARG = 1,  /* bad pointer, shape, scalar or alignment     */
    INK_ERR_UNSUPPORTED = 2,  /* valid but not built: head_dim not in {64, 128, 256}, ... */
    INK_ERR_WORKSPACE = 3,    /* workspace smaller than the size query says  */
    INK_ERR_CUDA = 4          /* a CUDA runtime / driver call failed         */
} ink_status;

/* Device-side data errors, OR-ed into the workspace's error word by the
 * kernels (they never trap); read with ink_rel_attn_read_device_errors.
 * A request that raises CU_SEQLENS, SEQLEN_Q or SEQLEN_K is skipped: its
 * rows of out and lse are left as they were.  When the valid requests' token
 * ranges overlap (an inner cu_seqlens_q entry that steps back) so far that
 * they need more query tiles than T tokens can, CU_SEQLENS is raised and the
 * whole call is skipped.  With PAGE_ID the keys of the bad page read as zeros. */
#define INK_DEVERR_PAGE_ID    0x01u /* block_table entry needed for a visible key is outside [0, num_blocks) */
#define INK_DEVERR_CU_SEQLENS 0x02u /* cu_seqlens_q not non-decreasing within [0, T], or cu[0] != 0, cu[B] != T */
#define INK_DEVERR_SEQLEN_Q   0x04u /* a request has more query tokens than max_seqlen_q */
#define INK_DEVERR_SEQLEN_K   0x08u /* cache_seqlens[b] < 0 or > max_blocks_per_seq * block_size */
#define INK_DEVERR_EMPTY_ROWS 0x10u /* informational: some rows saw no key (out 0, lse -inf), e.g. causal with Lk < Lq */
#define INK_DEVERR_TIMEOUT    0x100u /* a bounded pipeline wait gave up; outputs of the call are undefined */
#define INK_DEVERR_SMEM       0x200u /* a kernel found less shared memory than its layout needs and did nothing */
#define INK_DEVERR_STAGE      0x400u /* an FP8-cache prefill-shaped request found no room in the K/V staging area: it was skipped */

/*
 * Bytes of device workspace one call needs.  `num_splits` as in
 * ink_rel_attn_varlen (0 = the library's choice; the size then covers every
 * choice the library can make for these dims).  The workspace holds the
 * error word, the device-built work lists and, when splits are used, the
 * per-split partial outputs (fp32) and log-sum-exps.  Returns 0 for
 * invalid dims.
 */
INK_API size_t ink_rel_attn_workspace_size(const ink_attn_dims *dims, int32_t max_seqlen_q,
                                   int32_t num_splits);

/*
 * Extra workspace bytes that let the prefill read the K and V of prefill-shaped
 * requests (max_seqlen_q * H / Hkv > 16 rows) holding `prefill_kv_tokens` cache
 * keys in total from a contiguous staging copy instead of the paged cache.
 * The pages print no counterpart: this is a GB300 layout choice.  One K or V
 * tile of one KV head is then 32 KB of consecutive bytes (one TMA box) instead
 * of 128 rows of 256 bytes spread over 16-key pages, which the L2 delivers at a
 * much higher rate.
 * Workspace beyond ink_rel_attn_workspace_size is always used this way: each
 * call copies, in request order, the pages of every prefill-shaped request
 * whose keys (rounded up to whole 128-key tiles) still fit, and the rest read
 * the paged cache.  Results do not depend on it.  Returns 0 for invalid dims
 * and for head sizes other than 128 (the head-size-generic kernel, their
 * prefill path, reads the paged cache directly).
 */
INK_API size_t ink_rel_attn_stage_bytes(const ink_attn_dims *dims, int64_t prefill_kv_tokens);

/*
 * The split-KV count the library picks when called with num_splits = 0:
 * the cap on splits per work unit for decode-shaped calls
 * (max_seqlen_q * H / Hkv <= 16) and for prefill-shaped calls otherwise.
 * It is re-derived for the GB300 SM count from the page's heuristic
 * (inkling_fa4_num_splits): enough units to fill every
 * SM several times, with at least 16 keys per split.  `max_kv_len` bounds
 * cache_seqlens.  Returns 0 for invalid dims.  Needs a current CUDA device.
 */
INK_API int32_t ink_rel_attn_num_splits(const ink_attn_dims *dims, int32_t max_seqlen_q,
                                int32_t max_kv_len, int32_t window_left, int32_t window_right);

/*
 * The attention itself.
 *   q             bf16 (T, H, D), contiguous, 16-byte aligned.
 *   key_cache     bf16 (num_blocks, block_size, Hkv, D), contiguous, 16-byte aligned.
 *   value_cache   same shape and alignment as key_cache (two pointers into a
 *                 stacked (2, ...) cache are fine).
 *   block_table   int32 (B, max_blocks_per_seq): logical page -> physical page.
 *                 Entries at or beyond ceil(Lk / block_size) are never read
 *                 (padding with -1 is fine); pages may be shared.
 *   cache_seqlens int32 (B): KV length of each request, including this
 *                 step's query tokens (the KV write happens first).
 *   cu_seqlens_q  int32 (B+1): cu[0] = 0, non-decreasing, cu[B] = T.
 *   max_seqlen_q  host bound on every Lq (a scheduling bound only: results
 *                 do not depend on it as long as it is >= every Lq).
 *   softmax_scale multiplies q.k before the bias is added; finite and > 0.
 *   causal        nonzero: bottom-right causal mask.
 *   window_left/right  -1 = unbounded on that side; (-1, -1) = no window.
 *   rel_extent    E >= 0; rel_logits fp32 (T, H, E) contiguous, may be NULL
 *                 when E == 0.  Entries at rd >= Lk or beyond a window are
 *                 never read.
 *   num_splits    0 = library choice, 1 = no split (no combine pass),
 *                 S > 1: each work unit's visible KV range is cut into
 *                 chunks of ceil(max visible keys / S) keys (rounded to 16).
 *   out           bf16 (T, H, D), contiguous, 16-byte aligned.
 *   lse           fp32 (T, H) or NULL.
 *   workspace     device memory of at least
 *                 ink_rel_attn_workspace_size(dims, max_seqlen_q, num_splits)
 *                 bytes, 256-byte aligned; it must not be used by another
 *                 call that overlaps this one on the GPU.  Bytes beyond that
 *                 size stage K/V for the prefill (ink_rel_attn_stage_bytes).
 *   stream        CUDA stream the kernels are launched on.
 * Head sizes: D = 128 runs the tcgen05 prefill and the decode kernel; D = 64
 * and 256 (the other head sizes the vLLM V1 attention page lists for a paged
 * backend; the PagedAttention V2 page's GQA example uses 256) run the decode
 * kernel for decode-shaped requests (where a warp's share of the head, D * Hkv
 * / 8, is at least 16 and two bf16 pages fit its ring) and a head-size-generic
 * kernel (mma.sync, the same work list) for the rest.
 * Host-side checks return INK_ERR_INVALID_ARG / UNSUPPORTED / WORKSPACE
 * before anything is launched; a launch failure returns INK_ERR_CUDA.
 * Data errors found on the device are reported through the error word.
 */
INK_API ink_status ink_rel_attn_varlen(const ink_attn_dims *dims,
                               const void *q, const void *key_cache, const void *value_cache,
                               const int32_t *block_table, const int32_t *cache_seqlens,
                               const int32_t *cu_seqlens_q, int32_t max_seqlen_q,
                               float softmax_scale, int causal,
                               int32_t window_left, int32_t window_right,
                               int32_t rel_extent, const float *rel_logits,
                               int32_t num_splits,
                               void *out, float *lse,
                               void *workspace, size_t workspace_bytes,
                               ink_stream_t stream);

/*
 * The same attention over an FP8 KV cache.  The FP8 cache is
 * the TurboQuant backend's (vLLM V1 attention page, section 12.1: an FP8
 * cache dequantized when decoding), with per-tensor k_scale / v_scale applied
 * to the gathered K and V rows as paged_attention_v2_pytorch does on the
 * PagedAttention V2 page.
 *   key_cache, value_cache  OCP FP8 E4M3 bytes, (num_blocks, block_size,
 *                 Hkv, D) with D = 128 (other head sizes return
 *                 INK_ERR_UNSUPPORTED), contiguous, 16-byte aligned; the values attended
 *                 over are k_scale * E4M3(byte) and v_scale * E4M3(byte).
 *   k_scale, v_scale  in [2^-126, 2^126] (normal, with a normal reciprocal),
 *                 else INK_ERR_INVALID_ARG.
 * Decode-shaped requests (max_seqlen_q * (H / Hkv) <= 16 with Hkv in
 * {1, 2, 4, 8}) run in the decode kernel: the products run in fp16 with fp32
 * accumulation (every E4M3 value is exact in fp16; q is converted from bf16 to
 * fp16, exact for magnitudes in [2^-14, 65504]).  Prefill-shaped requests are
 * read from the K/V staging area (ink_rel_attn_stage_bytes), into which each
 * call copies their pages converted to bf16 (exact for every E4M3 value); the
 * prefill then multiplies bf16 q with them, k_scale joining the softmax scale
 * and v_scale the output.  A call with prefill-shaped requests needs staging
 * room: none at all returns INK_ERR_WORKSPACE, and a request that does not fit
 * raises INK_DEVERR_STAGE and is skipped.  All other arguments, results and
 * errors are those of ink_rel_attn_varlen.
 */
INK_API ink_status ink_rel_attn_varlen_fp8kv(const ink_attn_dims *dims,
                                             const void *q, const void *key_cache, const void *value_cache,
                                             float k_scale, float v_scale,
                                             const int32_t *block_table, const int32_t *cache_seqlens,
                                             const int32_t *cu_seqlens_q, int32_t max_seqlen_q,
                                             float softmax_scale, int causal,
                                             int32_t window_left, int32_t window_right,
                                             int32_t rel_extent, const float *rel_logits,
                                             int32_t num_splits, void *out, float *lse,
                                             void *workspace, size_t workspace_bytes,
                                             ink_stream_t stream);

/*
 * Allocation-free variant (this entry point has no counterpart on the source
 * pages).  For callers that cannot allocate device memory: programs embedded in
 * a host that owns all device memory itself, such as a serving engine that has
 * reserved nearly all of HBM for its paged KV-cache pool, or a plugin interface
 * that passes an operator its tensors but no scratch buffer and no allocator.
 * Same arguments and results as ink_rel_attn_varlen, without the workspace: the
 * call runs on a scratch area of INK_STATIC_SCRATCH_BYTES compiled into the
 * library, which every GPU that loads the library holds until the process exits.
 *   - Work that needs more scratch than that (see ink_rel_attn_workspace_size)
 *     returns INK_ERR_WORKSPACE before anything is launched; scratch left over
 *     stages K/V for the prefill, as with any workspace.
 *   - The first call on a device looks up the scratch area's device address for
 *     that device (with it current) and caches it; make that first call before
 *     any stream capture.  The cached address is not valid after a reset of the
 *     device (cudaDeviceReset): do not call this entry point after one.
 *   - Every call, on every stream, shares the one scratch area of its device, and
 *     the area keeps the last call's contents (each call clears what must start
 *     at zero).  Calls that overlap on the GPU race on it: order them, for
 *     example on one stream.
 *   - It allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 */
#define INK_STATIC_SCRATCH_BYTES (32u << 20)
INK_API ink_status ink_rel_attn_varlen_static(const ink_attn_dims *dims,
                                              const void *q, const void *key_cache, const void *value_cache,
                                              const int32_t *block_table, const int32_t *cache_seqlens,
                                              const int32_t *cu_seqlens_q, int32_t max_seqlen_q,
                                              float softmax_scale, int causal,
                                              int32_t window_left, int32_t window_right,
                                              int32_t rel_extent, const float *rel_logits,
                                              int32_t num_splits, void *out, float *lse,
                                              ink_stream_t stream);

/*
 * KV append: writes this step's keys and values into the paged cache before
 * attention reads it ("reshape_and_cache" with the slot mapping of the vLLM V1
 * attention page, metadata builder step 2 and appendix O).  For every token t
 * with s = slot_mapping[t] >= 0:
 *     key_cache[s / block_size][s % block_size][h][:]   = key[t][h][:]
 *     value_cache[s / block_size][s % block_size][h][:] = value[t][h][:]
 * for every KV head h; negative slots are padding and are skipped.
 *
 *   dims        num_tokens, num_kv_heads, head_dim (64, 128 or 256), num_blocks
 *               and block_size are read; the other fields are ignored.
 *   key, value  device, bf16 (num_tokens, num_kv_heads, head_dim), 16-byte
 *               aligned; read only.
 *   key_cache, value_cache
 *               device, bf16 (num_blocks, block_size, num_kv_heads,
 *               head_dim), 16-byte aligned; written at the mapped slots only.
 *   slot_mapping device int64 (num_tokens).  Slots must be distinct.
 *   flags       device uint32 or NULL: INK_DEVERR_PAGE_ID is OR-ed in when a
 *               slot is >= num_blocks * block_size (that token is skipped).
 *   stream      the call is stream-ordered; it allocates nothing.
 * Returns INK_ERR_INVALID_ARG for null pointers, bad shapes or misalignment,
 * INK_ERR_UNSUPPORTED for a head_dim outside {64, 128, 256}, INK_ERR_CUDA on a
 * launch error.
 */
INK_API ink_status ink_reshape_and_cache(const ink_attn_dims *dims, const void *key, const void *value,
                                         void *key_cache, void *value_cache, const int64_t *slot_mapping,
                                         uint32_t *flags, ink_stream_t stream);

/*
 * KV append into an FP8 cache: the quantize-on-store of the TurboQuant
 * backend (vLLM V1 attention page, section 12.1), inverse to the
 * k_scale / v_scale read of ink_rel_attn_varlen_fp8kv.  Slots, padding and
 * flags as ink_reshape_and_cache; each stored element is the OCP FP8 E4M3
 * byte of fp32(x) / k_scale (keys) or fp32(x) / v_scale (values): one IEEE
 * fp32 division, then round to nearest with ties to the even code, magnitudes
 * above 448 saturated to 448, NaN stays NaN.
 *   key, value  device, bf16 (num_tokens, num_kv_heads, 128), 16-byte aligned.
 *   key_cache, value_cache  device, E4M3 bytes (num_blocks, block_size,
 *               num_kv_heads, 128), 16-byte aligned.
 *   k_scale, v_scale  in [2^-126, 2^126] (normal, with a normal reciprocal),
 *                 else INK_ERR_INVALID_ARG.
 * Other errors as ink_reshape_and_cache, except that head_dim must be 128
 * (the size the FP8 attention reads), else INK_ERR_UNSUPPORTED.
 */
INK_API ink_status ink_reshape_and_cache_fp8(const ink_attn_dims *dims, const void *key, const void *value,
                                             void *key_cache, void *value_cache, const int64_t *slot_mapping,
                                             float k_scale, float v_scale, uint32_t *flags, ink_stream_t stream);

/* Human-readable name of a status code (static storage). */
INK_API const char *ink_status_string(ink_status status);

/*
 * Debug helper: copies the error word of the last call that used
 * `workspace` into *flags (INK_DEVERR_* bits).  Synchronises `stream`.
 */
INK_API ink_status ink_rel_attn_read_device_errors(const void *workspace, ink_stream_t stream,
                                           uint32_t *flags);

/* Library version, e.g. 100 for 0.1.0. */
INK_API int32_t ink_attn_version(void);

/*
 * Measurement hooks (no effect on results).
 * ink_set_timing_events: while set, every call records `start_event` on its
 * stream just before launching the named kernel and `stop_event` just after
 * it (both cudaEvent_t, owned by the caller; NULL clears the hook).  The hooks
 * are process-wide, one per kernel id, and are the only state the library keeps
 * between calls besides the launch counter: they are for single-threaded
 * measurement -- set them, make calls from one host thread on one stream, clear
 * them -- because a call from any other thread or stream made meanwhile records
 * into the same events.  Setting or clearing a hook while another thread is
 * inside a call is a data race.
 * ink_launch_count: number of kernels this library has launched in the
 * process so far.
 */
typedef enum {
    INK_KERNEL_PREPASS = 1,
    INK_KERNEL_DECODE = 2,
    INK_KERNEL_PREFILL = 3,
    INK_KERNEL_COMBINE = 4,
    INK_KERNEL_APPEND = 5,
    INK_KERNEL_STAGE = 6
} ink_kernel_id;

INK_API void ink_set_timing_events(ink_kernel_id kernel, void *start_event, void *stop_event);
INK_API uint64_t ink_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* INK_ATTN_H */
