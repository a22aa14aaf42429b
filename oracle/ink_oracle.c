/*
 * ink_oracle.c -- plain, slow, fp64 CPU oracle for paged varlen causal GQA
 * attention with the Inkling additive relative bias.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code, header or table
 * with the CUDA path.
 *
 * What it computes (definition written out, no blocking or reordering):
 *
 *   For request b:  Lq = cu[b+1]-cu[b],  Lk = cache_seqlens[b].
 *   For token i < Lq and head h:  t = cu[b]+i,  g = h / (H/Hkv),
 *     q_abs = i + Lk - Lq                 (bottom-right causal alignment:
 *        "seqlen_local_offset = seqlen_k - seqlen_q" in score_mod_rel_bias,
 *        fa4_rel_attention.py, nxmr.cn article)
 *   For key j < Lk:
 *     visible(j) = (!causal || j <= q_abs)
 *                  && (wl < 0 || j >= q_abs - wl) && (wr < 0 || j <= q_abs + wr)
 *     page  = block_table[b][j / bs],   row = j % bs          (paged direct
 *        addressing: mini-vllm tutorial step 15, "block_table" section)
 *     s_j = softmax_scale * sum_d q[t][h][d] * K[page][row][g][d]
 *           + bias(rd),  rd = q_abs - j,
 *     bias(rd) = rel_logits[t][h][rd] if 0 <= rd < rel_extent else 0
 *        (score_mod_rel_bias steps 1-4: clamp to [0, rel_extent-1], look
 *         up, and drop the bias when the clamp changed the distance)
 *   Softmax over the visible keys, two passes in fp64:
 *     m = max s_j,  l = sum exp(s_j - m),  o = sum exp(s_j - m) v_j / l,
 *     lse = m + ln l;   no visible key  ->  o = 0, lse = -inf
 *        (PagedAttention V2 page: zero output for an empty sequence,
 *         -inf for unused partition maxima).
 *
 * The split variant cuts each row's key range [0, Lk) into contiguous chunks
 * of `chunk_keys` keys, computes (m_c, l_c, o_c = acc_c / l_c) per chunk and
 * merges them with the PagedAttention V2 page's Phase-2 rule:
 *     gmax = max_c m_c,  w_c = exp(m_c - gmax) * l_c,
 *     o = sum_c w_c o_c / sum_c w_c,   lse = gmax + ln(sum_c w_c).
 * (That rule is exact only when o_c is normalised by its own l_c; see the
 * reading recorded for it in the design notes.)
 *
 * FP8 KV cache (ink_oracle_attn_fp8kv): the caches hold one byte per element
 * in the OCP 8-bit floating-point format E4M3, and an element's value is its
 * decoded E4M3 value times the tensor's scale (k_scale for K, v_scale for V),
 * as the PagedAttention V2 page's paged_attention_v2_pytorch multiplies the
 * gathered K and V rows by k_scale and v_scale, and as the vLLM V1 attention
 * page's TurboQuant backend dequantizes an FP8 cache when it decodes
 * (section 12.1).  Everything else is the definition above.
 *
 * bf16 inputs are passed as their 16-bit patterns and widened exactly.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_PAGE 2
#define ORACLE_ERR_CU 3
#define ORACLE_ERR_ALLOC 4

typedef struct {
    int32_t T, B, H, Hkv, D, NB, BS, MAXBLK;
    const uint16_t *q, *kc, *vc;
    const uint8_t *kc8, *vc8;       /* E4M3 caches when kv_fp8, else unused */
    int kv_fp8;
    double k_scale, v_scale;
    const int32_t *bt, *seqk, *cu;
    double scale;
    int causal;
    int32_t wl, wr, E;
    const float *rel;
} oracle_args;

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3: sign bit, 4 exponent bits (bias 7), 3
 * mantissa bits.  Exponent field 0 holds zero and the subnormals m/8 * 2^-6;
 * exponent 15 with mantissa 7 is NaN; there are no infinities (the largest
 * finite value is 1.75 * 2^8 = 448). */
static double e4m3_bits_to_double(uint8_t bits)
{
    const int sign = bits >> 7, e = (bits >> 3) & 15, m = bits & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Element idx of the K (value == 0) or V (value == 1) cache as a real number. */
static double cache_elem(const oracle_args *a, int value, int64_t idx)
{
    if (a->kv_fp8)
        return (value ? a->v_scale : a->k_scale) * e4m3_bits_to_double((value ? a->vc8 : a->kc8)[idx]);
    return bf16_bits_to_double((value ? a->vc : a->kc)[idx]);
}

/* Request owning token t (cu is non-decreasing, checked by the caller). */
static int32_t owner_of(const oracle_args *a, int64_t t)
{
    int32_t lo = 0, hi = a->B - 1;
    while (lo < hi) {               /* first b with cu[b+1] > t */
        int32_t mid = (lo + hi) / 2;
        if ((int64_t)a->cu[mid + 1] > t) hi = mid; else lo = mid + 1;
    }
    return lo;
}

static int key_visible(const oracle_args *a, int64_t q_abs, int64_t j)
{
    if (a->causal && j > q_abs) return 0;
    if (a->wl >= 0 && j < q_abs - a->wl) return 0;
    if (a->wr >= 0 && j > q_abs + a->wr) return 0;
    return 1;
}

/*
 * Softmax statistics of row (t, h) over the visible keys j in
 * [j_begin, j_end).  Writes m, l and acc[d] = sum exp(s_j - m) v_j[d].
 * Returns the number of visible keys, or -1 on a bad page id.
 * `s` is scratch of at least (j_end - j_begin) doubles.
 */
static int64_t row_stats(const oracle_args *a, int64_t t, int32_t h,
                         int64_t j_begin, int64_t j_end,
                         double *m_out, double *l_out, double *acc, double *s)
{
    const int32_t b = owner_of(a, t);
    const int64_t Lq = (int64_t)a->cu[b + 1] - a->cu[b];
    const int64_t Lk = a->seqk[b];
    const int64_t i = t - a->cu[b];
    const int64_t q_abs = i + Lk - Lq;
    const int32_t G = a->H / a->Hkv;
    const int32_t g = h / G;
    const uint16_t *qrow = a->q + ((int64_t)t * a->H + h) * a->D;
    int64_t n = 0;
    double m = -INFINITY;

    if (j_end > Lk) j_end = Lk;
    for (int32_t d = 0; d < a->D; ++d) acc[d] = 0.0;

    /* pass 1: scores of visible keys and their maximum */
    for (int64_t j = j_begin; j < j_end; ++j) {
        double sj = -INFINITY;
        if (key_visible(a, q_abs, j)) {
            const int32_t page = a->bt[(int64_t)b * a->MAXBLK + j / a->BS];
            if (page < 0 || page >= a->NB) return -1;
            const int64_t krow =
                (((int64_t)page * a->BS + j % a->BS) * a->Hkv + g) * a->D;
            double dot = 0.0;
            for (int32_t d = 0; d < a->D; ++d)
                dot += bf16_bits_to_double(qrow[d]) * cache_elem(a, 0, krow + d);
            sj = a->scale * dot;
            const int64_t rd = q_abs - j;
            if (rd >= 0 && rd < a->E)
                sj += (double)a->rel[((int64_t)t * a->H + h) * a->E + rd];
            if (sj > m) m = sj;
            ++n;
        }
        s[j - j_begin] = sj;
    }
    /* pass 2: exponentials against the maximum, weighted sum of V rows */
    double l = 0.0;
    if (n > 0) {
        for (int64_t j = j_begin; j < j_end; ++j) {
            const double sj = s[j - j_begin];
            if (sj == -INFINITY) continue;
            const double p = exp(sj - m);
            const int32_t page = a->bt[(int64_t)b * a->MAXBLK + j / a->BS];
            const int64_t vrow =
                (((int64_t)page * a->BS + j % a->BS) * a->Hkv + g) * a->D;
            l += p;
            for (int32_t d = 0; d < a->D; ++d) acc[d] += p * cache_elem(a, 1, vrow + d);
        }
    }
    *m_out = m;
    *l_out = l;
    return n;
}

static int check_args(const oracle_args *a)
{
    if (a->T < 0 || a->B < 1 || a->H < 1 || a->Hkv < 1 || a->D < 1 || a->BS < 1 ||
        a->MAXBLK < 0 || a->NB < 0 || a->H % a->Hkv != 0 || a->E < 0)
        return ORACLE_ERR_ARG;
    if (a->E > 0 && a->rel == NULL) return ORACLE_ERR_ARG;
    if (a->cu[0] != 0 || a->cu[a->B] != a->T) return ORACLE_ERR_CU;
    for (int32_t b = 0; b < a->B; ++b) {
        if (a->cu[b + 1] < a->cu[b]) return ORACLE_ERR_CU;
        if (a->seqk[b] < 0 || (int64_t)a->seqk[b] > (int64_t)a->MAXBLK * a->BS) return ORACLE_ERR_ARG;
    }
    return ORACLE_OK;
}

/* Row list: NULL means every (t, h) in order t*H + h. */
static int64_t row_at(const int64_t *rows, int64_t r) { return rows ? rows[r] : r; }

static int64_t max_seqk(const oracle_args *a)
{
    int64_t mx = 1;
    for (int32_t b = 0; b < a->B; ++b) if (a->seqk[b] > mx) mx = a->seqk[b];
    return mx;
}

static int run_rows(const oracle_args *a, const int64_t *rows, int64_t n_rows,
                    int64_t chunk_keys, double *out, double *lse)
{
    int status = check_args(a);
    if (status != ORACLE_OK) return status;
    const int64_t smax = max_seqk(a);
    if (n_rows < 0) return ORACLE_ERR_ARG;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t row = row_at(rows, r);
        if (row < 0 || row >= (int64_t)a->T * a->H) return ORACLE_ERR_ARG;
    }
    int bad_page = 0, bad_alloc = 0;

#pragma omp parallel reduction(|| : bad_page, bad_alloc)
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)smax);
        double *acc = (double *)malloc(sizeof(double) * (size_t)a->D);
        double *tot = (double *)malloc(sizeof(double) * (size_t)a->D);
        if (!s || !acc || !tot) bad_alloc = 1;
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; ++r) {
            if (!s || !acc || !tot) continue;
            const int64_t row = row_at(rows, r);
            const int64_t t = row / a->H;
            const int32_t h = (int32_t)(row % a->H);
            const int32_t b = owner_of(a, t);
            const int64_t Lk = a->seqk[b];
            double *o = out + r * a->D;
            if (chunk_keys <= 0) {
                double m, l;
                int64_t n = row_stats(a, t, h, 0, Lk, &m, &l, acc, s);
                if (n < 0) { bad_page = 1; continue; }
                if (n == 0) {
                    for (int32_t d = 0; d < a->D; ++d) o[d] = 0.0;
                    lse[r] = -INFINITY;
                } else {
                    for (int32_t d = 0; d < a->D; ++d) o[d] = acc[d] / l;
                    lse[r] = m + log(l);
                }
            } else {
                /* split variant: per-chunk statistics, then the Phase-2 merge */
                int64_t nchunks = (Lk + chunk_keys - 1) / chunk_keys;
                double gmax = -INFINITY;
                for (int64_t c = 0; c < nchunks; ++c) {
                    double m, l;
                    int64_t n = row_stats(a, t, h, c * chunk_keys, (c + 1) * chunk_keys,
                                          &m, &l, acc, s);
                    if (n < 0) { bad_page = 1; break; }
                    if (n > 0 && m > gmax) gmax = m;
                }
                if (bad_page) continue;
                double wsum = 0.0;
                for (int32_t d = 0; d < a->D; ++d) tot[d] = 0.0;
                if (gmax != -INFINITY) {
                    for (int64_t c = 0; c < nchunks; ++c) {
                        double m, l;
                        int64_t n = row_stats(a, t, h, c * chunk_keys, (c + 1) * chunk_keys,
                                              &m, &l, acc, s);
                        if (n <= 0) continue;
                        const double w = exp(m - gmax) * l;   /* Phase-2 weight */
                        wsum += w;
                        for (int32_t d = 0; d < a->D; ++d) tot[d] += w * (acc[d] / l);
                    }
                }
                if (wsum == 0.0) {
                    for (int32_t d = 0; d < a->D; ++d) o[d] = 0.0;
                    lse[r] = -INFINITY;
                } else {
                    for (int32_t d = 0; d < a->D; ++d) o[d] = tot[d] / wsum;
                    lse[r] = gmax + log(wsum);
                }
            }
        }
        free(s);
        free(acc);
        free(tot);
    }
    if (bad_alloc) return ORACLE_ERR_ALLOC;
    if (bad_page) return ORACLE_ERR_PAGE;
    return ORACLE_OK;
}

/*
 * Paged varlen attention, fp64.  Argument order follows the wrapper
 * signature of inkling_fa4_rel_attention (nxmr.cn article, layer 3
 * "参数签名"), with the shape integers a C interface needs.
 *
 *   q           bf16 bits, (T, H, D)
 *   key_cache   bf16 bits, (NB, BS, Hkv, D); value_cache likewise
 *   block_table (B, MAXBLK) int32; cache_seqlens (B); cu_seqlens_q (B+1)
 *   rel_logits  fp32 (T, H, E); may be NULL when E == 0
 *   rows        optional list of flattened rows t*H + h (NULL: all T*H rows)
 *   chunk_keys  <= 0: unsplit definition; > 0: split variant
 *   out         (n_rows, D) fp64;  lse (n_rows) fp64
 * Returns 0, or 1 bad argument, 2 page id out of range, 3 bad cu_seqlens_q,
 * 4 out of memory.
 */
int ink_oracle_attn(int32_t T, int32_t B, int32_t H, int32_t Hkv, int32_t D,
                    int32_t NB, int32_t BS, int32_t MAXBLK,
                    const uint16_t *q, const uint16_t *key_cache, const uint16_t *value_cache,
                    const int32_t *block_table, const int32_t *cache_seqlens,
                    const int32_t *cu_seqlens_q,
                    double softmax_scale, int causal, int32_t window_left, int32_t window_right,
                    int32_t rel_extent, const float *rel_logits,
                    const int64_t *rows, int64_t n_rows, int64_t chunk_keys,
                    double *out, double *lse)
{
    oracle_args a;
    a.T = T; a.B = B; a.H = H; a.Hkv = Hkv; a.D = D; a.NB = NB; a.BS = BS; a.MAXBLK = MAXBLK;
    a.q = q; a.kc = key_cache; a.vc = value_cache;
    a.kc8 = NULL; a.vc8 = NULL; a.kv_fp8 = 0; a.k_scale = 1.0; a.v_scale = 1.0;
    a.bt = block_table; a.seqk = cache_seqlens; a.cu = cu_seqlens_q;
    a.scale = softmax_scale; a.causal = causal; a.wl = window_left; a.wr = window_right;
    a.E = rel_extent; a.rel = rel_logits;
    if (!q || !key_cache || !value_cache || !block_table || !cache_seqlens || !cu_seqlens_q ||
        !out || !lse || window_left < -1 || window_right < -1)
        return ORACLE_ERR_ARG;
    if (rows == NULL && n_rows != (int64_t)T * H) return ORACLE_ERR_ARG;
    return run_rows(&a, rows, n_rows, chunk_keys, out, lse);
}

/*
 * The same attention over an FP8 (E4M3) KV cache: key_cache / value_cache
 * hold one byte per element, (NB, BS, Hkv, D), and K = k_scale * E4M3(byte),
 * V = v_scale * E4M3(byte).  Other arguments and results as ink_oracle_attn.
 */
int ink_oracle_attn_fp8kv(int32_t T, int32_t B, int32_t H, int32_t Hkv, int32_t D,
                          int32_t NB, int32_t BS, int32_t MAXBLK,
                          const uint16_t *q, const uint8_t *key_cache, const uint8_t *value_cache,
                          double k_scale, double v_scale,
                          const int32_t *block_table, const int32_t *cache_seqlens,
                          const int32_t *cu_seqlens_q,
                          double softmax_scale, int causal, int32_t window_left, int32_t window_right,
                          int32_t rel_extent, const float *rel_logits,
                          const int64_t *rows, int64_t n_rows, int64_t chunk_keys,
                          double *out, double *lse)
{
    oracle_args a;
    a.T = T; a.B = B; a.H = H; a.Hkv = Hkv; a.D = D; a.NB = NB; a.BS = BS; a.MAXBLK = MAXBLK;
    a.q = q; a.kc = NULL; a.vc = NULL;
    a.kc8 = key_cache; a.vc8 = value_cache; a.kv_fp8 = 1; a.k_scale = k_scale; a.v_scale = v_scale;
    a.bt = block_table; a.seqk = cache_seqlens; a.cu = cu_seqlens_q;
    a.scale = softmax_scale; a.causal = causal; a.wl = window_left; a.wr = window_right;
    a.E = rel_extent; a.rel = rel_logits;
    if (!q || !key_cache || !value_cache || !block_table || !cache_seqlens || !cu_seqlens_q ||
        !out || !lse || window_left < -1 || window_right < -1)
        return ORACLE_ERR_ARG;
    if (rows == NULL && n_rows != (int64_t)T * H) return ORACLE_ERR_ARG;
    return run_rows(&a, rows, n_rows, chunk_keys, out, lse);
}

/* E4M3 bytes to their values (for the decoder's own pins). */
void ink_oracle_e4m3_decode(const uint8_t *bits, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_bits_to_double(bits[i]);
}

/* Number of threads the OpenMP runtime will use (for reporting). */
int ink_oracle_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        {
#ifdef _OPENMP
            extern int omp_get_num_threads(void);
            n = omp_get_num_threads();
#endif
        }
    }
    return n;
}
