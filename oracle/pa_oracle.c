/*
 * pa_oracle.c -- plain, slow, fp64 CPU oracle for paged-KV GQA attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or helper with the CUDA path, and nothing here imports or
 * links that path.
 *
 * Every function computes the plain definition of the operation, in double
 * precision, with bf16 inputs widened exactly (a bf16 value is the top 16 bits
 * of an IEEE binary32).  No tiling, no online softmax, no fusion: scores are
 * materialised per (sequence or query row, query head), the maximum is
 * subtracted, exponentials are summed, and the weighted sum of value rows is
 * divided by that sum.
 *
 * Sources (pages of the reference material, cited by title and section):
 *  - "paged_attn.py" (vLLM PagedAttention backend for Iluvatar BI-V100):
 *      PagedAttention.write_to_paged_cache  -> oracle_write_cache
 *      PagedAttention._forward_decode_pytorch -> oracle_decode
 *      PagedAttention.forward_decode, V2 branch (512-token partitions with
 *        exp_sums / max_logits / tmp_output)  -> oracle_decode_partitions,
 *        oracle_merge_partitions
 *      PagedAttention._forward_prefix_pytorch (cached context, then the new
 *        chunk under the mask k_rel > q_rel)   -> oracle_prefill, paged mode
 *      PagedAttention.swap_blocks / copy_blocks -> oracle_swap_blocks,
 *        oracle_copy_blocks
 *  - "spark_runtime/flashinfer.rs" (Atlas): ragged_prefill_bf16_hd256 and its
 *      CPU reference test (per request, per head, kh = h / group, causal)
 *                                            -> oracle_prefill, contiguous mode
 *
 * Readings taken where the pages are silent (each is stated where it is used):
 *  R1 slot = page * block_size + row; slot < 0 means "skip this token".
 *  R2 causal alignment is bottom-right: query row i of a request with qo rows
 *     and kv keys sits at absolute position kv - qo + i and sees keys j <= that.
 *  R3 a query row (or a sequence) with no visible key yields an all-zero row.
 *  R4 partition p covers tokens [P*p, min(P*(p+1), L)); o_p is normalised by
 *     l_p, m_p is the max of the scaled scores (natural-log units).
 *  R13 a page-copy pair with a negative entry is padding and is skipped.
 *  R15 an "fp8" KV cache ("paged_attn.py": kv_cache_dtype, k_scale, v_scale on
 *     write_to_paged_cache and forward_decode) holds OCP FP8 E4M3 codes.  The
 *     write stores the code nearest to the fp32 quotient x / scale (x the bf16
 *     input widened to fp32; round to nearest, ties to the even code;
 *     saturating at +-448); a read gives code value * scale.
 *  R14 a sliding window of W > 0 keys ("paged_attn.py", forward_prefix's
 *     sliding_window; "libmir-cuda attention/mod.rs", active_partitions(token
 *     count, window)): a query at position pos sees only keys j > pos - W, the
 *     W most recent keys including its own position (and, if causal, j <= pos).
 *     W <= 0 means no window.  In decode pos = L - 1.  Split partitions keep
 *     their absolute 512-token ranges; partitions wholly before the window are
 *     neither computed nor merged.
 *
 * Parity status: every function here is pinned by the CPU test-suite
 * (brute-force dense attention written separately, closed forms and
 * invariants); none is "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- bf16 widening (exact) ------------------------------------------------ */

static double widen_bf16(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---- FP8 E4M3 (R15) --------------------------------------------------------- */

/*
 * Value of an E4M3 code, from the format's definition (OCP 8-bit floating point,
 * E4M3): bit 7 sign, bits 6..3 exponent e with bias 7, bits 2..0 mantissa m.
 * e = 0 is subnormal, 2^-6 * m / 8; otherwise 2^(e - 7) * (1 + m / 8).  There are
 * no infinities; e = 15 with m = 7 is NaN, so the largest finite value is 448.
 */
double oracle_e4m3_value(uint8_t code) {
    int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    double v = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/*
 * The E4M3 code of the finite value nearest to x: the non-negative codes are
 * searched for the one nearest to |x|, a tie going to the even code (the even
 * mantissa), and x's sign is kept.  Beyond 448 the nearest finite value is 448
 * (saturation; infinities too); NaN gives 0x7F.
 */
uint8_t oracle_e4m3_encode(float x) {
    if (x != x) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (isinf(a)) return sign | 0x7E;
    int best = 0;
    double best_err = a;  /* code 0 is the value 0 */
    for (int c = 1; c <= 0x7E; ++c) {
        double err = fabs(oracle_e4m3_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

void oracle_e4m3_encode_array(const float *x, uint8_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

/* A K or V pool: bf16 elements, or E4M3 codes read as code value * scale (R15). */
typedef struct {
    const void *base;
    int fp8;
    double scale;
} kv_pool;

static double pool_elem(const kv_pool *p, int64_t idx) {
    if (p->fp8) return oracle_e4m3_value(((const uint8_t *)p->base)[idx]) * p->scale;
    return widen_bf16(((const uint16_t *)p->base)[idx]);
}

/* ---- a tiny work-item thread pool ----------------------------------------- */

typedef void (*item_fn)(void *ctx, int64_t item);

typedef struct {
    item_fn fn;
    void *ctx;
    int64_t n_items;
    int64_t next;
    pthread_mutex_t lock;
} pool_t;

static void *pool_worker(void *arg) {
    pool_t *p = (pool_t *)arg;
    for (;;) {
        int64_t it;
        pthread_mutex_lock(&p->lock);
        it = p->next++;
        pthread_mutex_unlock(&p->lock);
        if (it >= p->n_items) break;
        p->fn(p->ctx, it);
    }
    return NULL;
}

/* Runs fn(ctx, i) for i in [0, n_items) on nthreads threads (<= 1: inline). */
static void run_items(item_fn fn, void *ctx, int64_t n_items, int nthreads) {
    if (nthreads <= 1 || n_items <= 1) {
        for (int64_t i = 0; i < n_items; ++i) fn(ctx, i);
        return;
    }
    if (nthreads > 256) nthreads = 256;
    pool_t p;
    p.fn = fn;
    p.ctx = ctx;
    p.n_items = n_items;
    p.next = 0;
    pthread_mutex_init(&p.lock, NULL);
    pthread_t th[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, pool_worker, &p) != 0) break;
        ++started;
    }
    if (started == 0) pool_worker(&p);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
    pthread_mutex_destroy(&p.lock);
}

/* ---- the softmax-weighted sum of one query row over a key list ------------ */

/*
 * out[d] = sum_j exp(s_j - max s) * V_j[d] / sum_j exp(s_j - max s),
 * s_j = scale * sum_d q[d] * K_j[d], over the n keys whose rows are given as
 * element offsets koff[j] / voff[j].  n == 0 gives an all-zero row (R3).
 * scores is caller scratch of length >= n.
 */
static void attend_row(double *out, const uint16_t *q, const kv_pool *kp,
                       const kv_pool *vp, const int64_t *koff,
                       const int64_t *voff, int64_t n, int hd, double scale,
                       double *scores) {
    for (int d = 0; d < hd; ++d) out[d] = 0.0;
    if (n <= 0) return;
    double mx = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        double s = 0.0;
        for (int d = 0; d < hd; ++d) s += widen_bf16(q[d]) * pool_elem(kp, koff[j] + d);
        s *= scale;
        scores[j] = s;
        if (s > mx) mx = s;
    }
    double den = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double p = exp(scores[j] - mx);
        scores[j] = p;
        den += p;
    }
    for (int64_t j = 0; j < n; ++j) {
        double w = scores[j];
        for (int d = 0; d < hd; ++d) out[d] += w * pool_elem(vp, voff[j] + d);
    }
    for (int d = 0; d < hd; ++d) out[d] /= den;
}

/* First key a query at position pos sees under a sliding window of w keys (R14). */
static int64_t window_first(int64_t pos, int64_t w) {
    if (w <= 0 || pos - w + 1 <= 0) return 0;
    return pos - w + 1;
}

/* ---- cache write ------------------------------------------------------------ */

/*
 * reshape_and_cache ("paged_attn.py", PagedAttention.write_to_paged_cache):
 * for every token t with slot = slot_mapping[t] >= 0 (R1), copy the bits of
 * k[t][h][:] to k_cache at (page = slot / bs, head h, row = slot % bs), and
 * the same for v.  Caches are addressed by element strides (s_block, s_head,
 * s_token); head_dim is contiguous.  k, v are [num_tokens][nkv][hd].
 * With kv_fp8 (kv_cache_dtype "fp8", R15) the caches hold bytes and each
 * element is stored as the E4M3 code of (float)x / k_scale (v_scale for v),
 * the quotient formed in fp32.
 * Returns the number of tokens whose slot was >= num_blocks * bs (those are
 * not written).
 */
int64_t oracle_write_cache(const uint16_t *k, const uint16_t *v, void *k_cache,
                           void *v_cache, const int64_t *slot_mapping,
                           int64_t num_tokens, int nkv, int hd, int bs,
                           int64_t num_blocks, int64_t s_block, int64_t s_head,
                           int64_t s_token, int kv_fp8, float k_scale, float v_scale) {
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * (int64_t)bs) {
            ++bad;
            continue;
        }
        int64_t page = slot / bs, row = slot % bs;
        for (int h = 0; h < nkv; ++h) {
            int64_t dst = page * s_block + h * s_head + row * s_token;
            int64_t src = (t * nkv + h) * (int64_t)hd;
            for (int d = 0; d < hd; ++d) {
                if (kv_fp8) {
                    float kx = (float)widen_bf16(k[src + d]), vx = (float)widen_bf16(v[src + d]);
                    ((uint8_t *)k_cache)[dst + d] = oracle_e4m3_encode(kx / k_scale);
                    ((uint8_t *)v_cache)[dst + d] = oracle_e4m3_encode(vx / v_scale);
                } else {
                    ((uint16_t *)k_cache)[dst + d] = k[src + d];
                    ((uint16_t *)v_cache)[dst + d] = v[src + d];
                }
            }
        }
    }
    return bad;
}

/* ---- decode ------------------------------------------------------------------ */

typedef struct {
    double *out;               /* [B][nq][hd] */
    const uint16_t *q;         /* [B][nq][hd] */
    kv_pool kc, vc;            /* paged pools */
    int64_t s_block, s_head, s_token;
    const int32_t *bt;         /* [B][max_blocks] */
    const int32_t *seq_lens;   /* [B] */
    int nq, nkv, hd, bs, max_blocks;
    double scale;
    const int32_t *items;      /* optional list of b*nq+h items */
    int window;                /* sliding window in keys (R14); <= 0: none */
} decode_ctx;

/* Element offset of token j of sequence b, kv head kh, in the paged pool. */
static int64_t paged_offset(const decode_ctx *c, int b, int kh, int64_t j) {
    int64_t page = c->bt[(int64_t)b * c->max_blocks + j / c->bs];
    return page * c->s_block + (int64_t)kh * c->s_head + (j % c->bs) * c->s_token;
}

static void decode_item(void *vctx, int64_t it) {
    const decode_ctx *c = (const decode_ctx *)vctx;
    int64_t bh = c->items ? c->items[it] : it;
    int b = (int)(bh / c->nq), h = (int)(bh % c->nq);
    int g = c->nq / c->nkv;
    int kh = h / g; /* contiguous GQA groups */
    int64_t L = c->seq_lens[b];
    if (L < 0) L = 0;
    /* keys j0 .. L-1: all of them, or the window's (R14) */
    int64_t j0 = L > 0 ? window_first(L - 1, c->window) : 0;
    int64_t n = L - j0;
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    double *sc = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int64_t j = j0; j < L; ++j) off[j - j0] = paged_offset(c, b, kh, j);
    attend_row(c->out + bh * c->hd, c->q + bh * c->hd, &c->kc, &c->vc, off, off, n,
               c->hd, c->scale, sc);
    free(off);
    free(sc);
}

/*
 * Decode ("paged_attn.py", PagedAttention._forward_decode_pytorch, stated as
 * the exact softmax it computes tile by tile): for sequence b and query head h,
 * kh = h / (nq / nkv); the L = seq_lens[b] keys are token j at page
 * bt[b][j / bs], row j % bs.  out[b][h] = softmax(scale * q K^T) V; L == 0
 * gives zeros (the "seq_len == 0" branch of the same function).  With a
 * window > 0 only the last `window` keys are attended (R14).  With kv_fp8 the
 * pools hold E4M3 codes read as code value * k_scale / v_scale (R15).
 * items (optional, n_items entries of b * nq + h) restricts the work to those
 * output rows; the others are left untouched.
 */
int oracle_decode(double *out, const uint16_t *q, const void *k_cache,
                  const void *v_cache, int64_t s_block, int64_t s_head,
                  int64_t s_token, const int32_t *block_tables,
                  const int32_t *seq_lens, int num_seqs, int nq, int nkv, int hd,
                  int bs, int max_blocks, double scale, const int32_t *items,
                  int64_t n_items, int nthreads, int window, int kv_fp8,
                  double k_scale, double v_scale) {
    if (nkv <= 0 || nq % nkv != 0) return -1;
    decode_ctx c = {out, q, {k_cache, kv_fp8, k_scale}, {v_cache, kv_fp8, v_scale},
                    s_block, s_head, s_token, block_tables, seq_lens, nq, nkv, hd, bs,
                    max_blocks, scale, items, window};
    int64_t n = items ? n_items : (int64_t)num_seqs * nq;
    run_items(decode_item, &c, n, nthreads);
    return 0;
}

/* ---- split-KV partitions and their merge ----------------------------------- */

typedef struct {
    decode_ctx d;
    double *m, *l, *o; /* [B][nq][P], [B][nq][P], [B][nq][P][hd] */
    int part, max_parts;
} part_ctx;

static void part_item(void *vctx, int64_t it) {
    const part_ctx *c = (const part_ctx *)vctx;
    const decode_ctx *d = &c->d;
    int64_t bh = it;
    int b = (int)(bh / d->nq), h = (int)(bh % d->nq);
    int kh = h / (d->nq / d->nkv);
    int64_t L = d->seq_lens[b];
    if (L < 0) L = 0;
    int64_t np = (L + c->part - 1) / c->part;
    /* the window's first key and the partition holding it (R14) */
    int64_t jw = L > 0 ? window_first(L - 1, d->window) : 0;
    double *sc = (double *)malloc(sizeof(double) * (size_t)c->part);
    const uint16_t *qr = d->q + bh * d->hd;
    for (int64_t p = jw / c->part; p < np && p < c->max_parts; ++p) {
        int64_t j0 = p * c->part, j1 = j0 + c->part;
        if (j1 > L) j1 = L;
        if (j0 < jw) j0 = jw;
        /* m_p: max of the scaled scores in the partition (R4) */
        double mx = -INFINITY;
        for (int64_t j = j0; j < j1; ++j) {
            int64_t kr = paged_offset(d, b, kh, j);
            double s = 0.0;
            for (int e = 0; e < d->hd; ++e) s += widen_bf16(qr[e]) * pool_elem(&d->kc, kr + e);
            s *= d->scale;
            sc[j - j0] = s;
            if (s > mx) mx = s;
        }
        /* l_p = sum exp(s - m_p); o_p = sum exp(s - m_p) V / l_p */
        double lsum = 0.0;
        double *op = c->o + ((bh * c->max_parts) + p) * d->hd;
        for (int e = 0; e < d->hd; ++e) op[e] = 0.0;
        for (int64_t j = j0; j < j1; ++j) {
            double w = exp(sc[j - j0] - mx);
            lsum += w;
            int64_t vr = paged_offset(d, b, kh, j);
            for (int e = 0; e < d->hd; ++e) op[e] += w * pool_elem(&d->vc, vr + e);
        }
        for (int e = 0; e < d->hd; ++e) op[e] /= lsum;
        c->m[bh * c->max_parts + p] = mx;
        c->l[bh * c->max_parts + p] = lsum;
    }
    free(sc);
}

/*
 * Split-KV partition pass ("paged_attn.py", PagedAttention.forward_decode, V2
 * branch: _PARTITION_SIZE-token partitions, per-partition max_logits, exp_sums
 * and tmp_output).  For p < ceil(L / part): m_p, l_p, o_p as in R4.  Entries
 * for p >= ceil(L / part) are left untouched.  With a window > 0 (R14) the
 * partitions run from the one holding key L - window on, that first one over
 * its keys inside the window only; the earlier entries are left untouched.
 * kv_fp8, k_scale, v_scale as in oracle_decode (R15).
 */
int oracle_decode_partitions(double *m, double *l, double *o, const uint16_t *q,
                             const void *k_cache, const void *v_cache,
                             int64_t s_block, int64_t s_head, int64_t s_token,
                             const int32_t *block_tables, const int32_t *seq_lens,
                             int num_seqs, int nq, int nkv, int hd, int bs,
                             int max_blocks, double scale, int part, int max_parts,
                             int nthreads, int window, int kv_fp8, double k_scale,
                             double v_scale) {
    if (nkv <= 0 || nq % nkv != 0 || part <= 0) return -1;
    part_ctx c;
    decode_ctx d = {NULL, q, {k_cache, kv_fp8, k_scale}, {v_cache, kv_fp8, v_scale},
                    s_block, s_head, s_token, block_tables, seq_lens, nq, nkv, hd, bs,
                    max_blocks, scale, NULL, window};
    c.d = d;
    c.m = m;
    c.l = l;
    c.o = o;
    c.part = part;
    c.max_parts = max_parts;
    run_items(part_item, &c, (int64_t)num_seqs * nq, nthreads);
    return 0;
}

/*
 * Log-sum-exp merge of the partitions of one (b, h): M = max_p m_p,
 * w_p = l_p * exp(m_p - M), out = sum_p w_p o_p / sum_p w_p over
 * p < ceil(L / part); L == 0 gives zeros.  This is the rescale-and-add rule
 * that "paged_attn.py" (_forward_decode_pytorch) applies between tiles,
 * applied once over all partitions -- with a window > 0, over the partitions
 * from the one holding key L - window on (R14).
 */
int oracle_merge_partitions(double *out, const double *m, const double *l,
                            const double *o, const int32_t *seq_lens, int num_seqs,
                            int nq, int hd, int part, int max_parts, int window) {
    if (part <= 0) return -1;
    for (int b = 0; b < num_seqs; ++b) {
        int64_t L = seq_lens[b] > 0 ? seq_lens[b] : 0;
        int64_t np = (L + part - 1) / part;
        if (np > max_parts) np = max_parts;
        int64_t p0 = (L > 0 ? window_first(L - 1, window) : 0) / part;
        for (int h = 0; h < nq; ++h) {
            int64_t bh = (int64_t)b * nq + h;
            double *dst = out + bh * hd;
            for (int e = 0; e < hd; ++e) dst[e] = 0.0;
            if (np == 0) continue;
            double M = -INFINITY;
            for (int64_t p = p0; p < np; ++p)
                if (m[bh * max_parts + p] > M) M = m[bh * max_parts + p];
            double W = 0.0;
            for (int64_t p = p0; p < np; ++p) {
                double w = l[bh * max_parts + p] * exp(m[bh * max_parts + p] - M);
                W += w;
                const double *op = o + (bh * max_parts + p) * hd;
                for (int e = 0; e < hd; ++e) dst[e] += w * op[e];
            }
            for (int e = 0; e < hd; ++e) dst[e] /= W;
        }
    }
    return 0;
}

/* ---- ragged prefill ------------------------------------------------------------ */

typedef struct {
    double *out;                  /* [total_qo][nq][hd] */
    const uint16_t *q;            /* [total_qo][nq][hd] */
    kv_pool k, v;                 /* bf16: contiguous [total_kv][nkv][hd], or paged pools */
    const int32_t *qo_indptr, *kv_indptr; /* [batch + 1] */
    const int32_t *bt;            /* NULL: contiguous; else [batch][max_blocks] */
    int max_blocks, bs;
    int64_t s_block, s_head, s_token;
    int batch, nq, nkv, hd, causal;
    double scale;
    const int64_t *rows;          /* optional list of query rows */
    int window;                   /* sliding window in keys (R14); <= 0: none */
} prefill_ctx;

static void prefill_item(void *vctx, int64_t it) {
    const prefill_ctx *c = (const prefill_ctx *)vctx;
    int64_t row = c->rows ? c->rows[it / c->nq] : it / c->nq;
    int h = (int)(it % c->nq);
    /* request r owning this row: qo_indptr[r] <= row < qo_indptr[r + 1] */
    int r = 0;
    while (r + 1 < c->batch && c->qo_indptr[r + 1] <= row) ++r;
    int64_t qo = c->qo_indptr[r + 1] - c->qo_indptr[r];
    int64_t kv = c->kv_indptr[r + 1] - c->kv_indptr[r];
    int64_t i = row - c->qo_indptr[r];
    int kh = h / (c->nq / c->nkv);
    /* visible keys: j < kv and, if causal, j <= i + (kv - qo)  (R2) */
    int64_t n = kv;
    if (c->causal) {
        int64_t lim = i + (kv - qo) + 1;
        if (lim < n) n = lim;
    }
    if (n < 0) n = 0;
    /* and j > pos - window for the row's position pos = i + (kv - qo) (R14) */
    int64_t lo = window_first(i + (kv - qo), c->window);
    int64_t cnt = n > lo ? n - lo : 0;
    int64_t *off = (int64_t *)malloc(sizeof(int64_t) * (size_t)(cnt > 0 ? cnt : 1));
    double *sc = (double *)malloc(sizeof(double) * (size_t)(cnt > 0 ? cnt : 1));
    for (int64_t j = lo; j < n; ++j) {
        if (c->bt) {
            int64_t page = c->bt[(int64_t)r * c->max_blocks + j / c->bs];
            off[j - lo] = page * c->s_block + (int64_t)kh * c->s_head + (j % c->bs) * c->s_token;
        } else {
            off[j - lo] = ((c->kv_indptr[r] + j) * c->nkv + kh) * (int64_t)c->hd;
        }
    }
    int64_t oidx = (row * c->nq + h) * (int64_t)c->hd;
    attend_row(c->out + oidx, c->q + oidx, &c->k, &c->v, off, off, cnt, c->hd, c->scale, sc);
    free(off);
    free(sc);
}

/*
 * Ragged (varlen) prefill.  Request r owns query rows
 * [qo_indptr[r], qo_indptr[r+1]) and kv_len = kv_indptr[r+1] - kv_indptr[r]
 * keys.  Contiguous mode (block_tables == NULL; "spark_runtime/flashinfer.rs",
 * ragged_prefill_bf16_hd256 and its CPU reference): key j is row
 * kv_indptr[r] + j of k / v.  Paged mode ("paged_attn.py",
 * _forward_prefix_pytorch, with the new chunk's K/V already written to the
 * cache): key j is token j of the request's block table row, addressed as in
 * decode.  Query head h reads kv head h / (nq / nkv); causal masking per R2;
 * rows with no visible key are zero (R3).
 * A window > 0 further limits row i to keys j > i + (kv - qo) - window (R14).
 * rows (optional, n_rows entries) restricts the work to those query rows (all
 * heads of each); other output rows are left untouched.
 */
int oracle_prefill(double *out, const uint16_t *q, const uint16_t *k, const uint16_t *v,
                   const int32_t *qo_indptr, const int32_t *kv_indptr,
                   const int32_t *block_tables, int max_blocks, int bs, int64_t s_block,
                   int64_t s_head, int64_t s_token, int batch, int nq, int nkv, int hd,
                   double scale, int causal, const int64_t *rows, int64_t n_rows,
                   int nthreads, int window) {
    if (nkv <= 0 || nq % nkv != 0 || batch <= 0) return -1;
    prefill_ctx c = {out, q, {k, 0, 1.0}, {v, 0, 1.0}, qo_indptr, kv_indptr, block_tables,
                     max_blocks, bs,
                     s_block, s_head, s_token, batch, nq, nkv, hd, causal, scale, rows,
                     window};
    int64_t nr = rows ? n_rows : (int64_t)qo_indptr[batch];
    run_items(prefill_item, &c, nr * nq, nthreads);
    return 0;
}

/* ---- whole-page copies ------------------------------------------------------ */

/*
 * swap_blocks ("paged_attn.py", PagedAttention.swap_blocks, which applies the
 * op to the key pool and then to the value pool): the pairs are taken in order;
 * pair i is (s, d) = (mapping[2i], mapping[2i + 1]) and copies page s of src --
 * the block_bytes bytes from byte s * block_bytes on -- to page d of dst.
 * R13: a pair with a negative entry is padding and is skipped, as a negative
 * slot is in the cache write; a pair with s >= src_blocks or d >= dst_blocks is
 * skipped and counted.  Returns that count.
 */
int64_t oracle_swap_blocks(const uint8_t *src, uint8_t *dst, const int64_t *mapping,
                           int64_t num_pairs, int64_t src_blocks, int64_t dst_blocks,
                           int64_t block_bytes) {
    int64_t bad = 0;
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t s = mapping[2 * i], d = mapping[2 * i + 1];
        if (s < 0 || d < 0) continue;
        if (s >= src_blocks || d >= dst_blocks) {
            ++bad;
            continue;
        }
        const uint8_t *from = src + s * block_bytes;
        uint8_t *to = dst + d * block_bytes;
        for (int64_t b = 0; b < block_bytes; ++b) to[b] = from[b];
    }
    return bad;
}

/*
 * copy_blocks ("paged_attn.py", PagedAttention.copy_blocks: the same pairs
 * applied to every layer's key pool and value pool): the page copy above with
 * source and destination the same pool, for each of the num_pools pools.
 * Returns the number of out-of-range pairs (counted once per pool).
 */
int64_t oracle_copy_blocks(uint8_t *const *pools, int num_pools, const int64_t *mapping,
                           int64_t num_pairs, int64_t num_blocks, int64_t block_bytes) {
    int64_t bad = 0;
    for (int t = 0; t < num_pools; ++t)
        bad += oracle_swap_blocks(pools[t], pools[t], mapping, num_pairs, num_blocks,
                                  num_blocks, block_bytes);
    return bad;
}
