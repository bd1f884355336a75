/*
 * Oracle: exact scaled-dot-product attention forward, computed in fp64 on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call this
 * file. Its users are the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark. It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes (the plain definition, no tiling, no online softmax):
 *
 *   For every batch b, query head hq and query row i:
 *     kv     = hq / (Hq / Hkv)                     grouped-query head map
 *     L      = key_len ? key_len[b] : N            valid (unpadded) length of batch b
 *     J(i)   = { j in [0,N) : i < L && j < L
 *                             && (!causal || j <= i)
 *                             && (window == 0 || i - j < window)
 *                             && (window == 0 || causal || j - i < window) }
 *     s_ij   = scale * sum_c q[b,hq,i,c] * k[b,kv,j,c]        for j in J(i)
 *     m_i    = max_j s_ij
 *     lse_i  = m_i + ln( sum_j exp(s_ij - m_i) )             natural-log log-sum-exp
 *     o[b,hq,i,c] = sum_j exp(s_ij - lse_i) * v[b,kv,j,c]
 *
 * Sources, by page and section:
 *   - score = QK^T / sqrt(D) and Attention = Softmax(score) V: the SpAtten review
 *     (coolstone2000.github.io), "Background - Attention Mechanism" formulas.
 *   - probability p_i = exp(s_i) / sum_j exp(s_j): same page, "Progressive
 *     Quantization" (attention probability equation).
 *   - scaling by sqrt(d_k), softmax, weighted sum of V; multi-head as independent
 *     heads; the look-ahead mask lets a token attend to itself and earlier tokens:
 *     palettepath-it.com self-attention guide, sections "어텐션 스코어 계산과 스케일링
 *     닷 프로덕트", "소프트맥스 정규화와 가중치 합산", "병렬 어텐션 헤드의 동작 원리",
 *     "룩어헤드 마스킹 (Look-Ahead Masking)".
 *   - grouped-query attention and sliding-window attention are named as compared
 *     variants on the "Attentions Under the Microscope" summary (gist.science),
 *     section "방법론". The head map kv = hq / G (consecutive groups) and the window
 *     rule i - j < window are the plainest readings; the pages fix neither. Without
 *     the look-ahead mask the window is read symmetrically, |i - j| < window (the
 *     local window of Longformer-style sparse attention, devhandbook.co.kr table
 *     "2. Attention 메커니즘 최적화 기법 비교").
 *   - padding: padding tokens neither give nor receive attention, their scores being
 *     set to -inf (palettepath-it.com guide, "패딩 마스킹 (Padding Masking)"); with
 *     per-token validity as in the blog's variable-length example (devhandbook.co.kr,
 *     "Example 7"), read as right padding: batch b's first key_len[b] tokens are
 *     valid. A padded query row therefore has no visible key.
 *
 * Decode shape (attn_ref_decode_rows_f64): Nq query rows against Nk >= Nq keys, the
 * queries being the last Nq positions of the sequence: query row i stands at position
 * i + Nk - Nq, and the mask above applies to that position (a key-value cache read by
 * the newest tokens, the generation stage of the SpAtten review's "Background"
 * section). With Nq = Nk this is the plain forward.
 *
 * Inputs are bf16 bit patterns (uint16); each is widened exactly to fp64.
 * A row whose visible set is empty (impossible for valid arguments, since j = i is
 * always visible) yields o = 0 and lse = -inf.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_bits_to_double(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int key_visible(int64_t i, int64_t j, int causal, int64_t window, int64_t L) {
    if (i >= L || j >= L) return 0;
    if (causal && j > i) return 0;
    if (window > 0 && i - j >= window) return 0;
    if (window > 0 && !causal && j - i >= window) return 0;
    return 1;
}

typedef struct {
    const uint16_t *q, *k, *v;
    const double *qd64, *kd64, *vd64;   /* fp64 inputs instead of bf16 bits, when set */
    int64_t B, Hq, Hkv, N, d;   /* N: query rows per head */
    int64_t Nk;                 /* keys per head; query row i stands at i + Nk - N */
    int causal;
    int64_t window;
    double scale;
    const int32_t *key_len; /* valid length per batch, or NULL (all N valid) */
    const int64_t *rows; /* flat row ids ((b*Hq)+hq)*N + i, or NULL for all rows */
    int64_t row_begin, row_end;
    double *o, *lse;     /* o: one d-vector per requested row; lse: one per row */
} job_t;

/* One query row, straight from the definition above. */
static void one_row(const job_t *jb, int64_t flat, double *o_row, double *lse_out,
                    double *qd, double *s) {
    const int64_t N = jb->N, d = jb->d, Nk = jb->Nk;
    const int64_t i = flat % N;
    const int64_t bh = flat / N;
    const int64_t hq = bh % jb->Hq;
    const int64_t b = bh / jb->Hq;
    const int64_t group = jb->Hq / jb->Hkv;
    const int64_t kv = hq / group;
    int64_t L = jb->key_len ? (int64_t)jb->key_len[b] : Nk;
    if (L < 0) L = 0;
    if (L > Nk) L = Nk;
    const int64_t pos = i + (Nk - N);   /* position of query row i in the sequence */

    const int64_t qoff = ((b * jb->Hq + hq) * N + i) * d;
    const int64_t kvoff = (b * jb->Hkv + kv) * Nk * d;
    const uint16_t *qrow = jb->q ? jb->q + qoff : NULL;
    const uint16_t *kbase = jb->k ? jb->k + kvoff : NULL;
    const uint16_t *vbase = jb->v ? jb->v + kvoff : NULL;
    const double *qrow64 = jb->qd64 ? jb->qd64 + qoff : NULL;
    const double *kbase64 = jb->kd64 ? jb->kd64 + kvoff : NULL;
    const double *vbase64 = jb->vd64 ? jb->vd64 + kvoff : NULL;
#define KVAL(j, c) (kbase64 ? kbase64[(j) * d + (c)] : bf16_bits_to_double(kbase[(j) * d + (c)]))
#define VVAL(j, c) (vbase64 ? vbase64[(j) * d + (c)] : bf16_bits_to_double(vbase[(j) * d + (c)]))

    for (int64_t c = 0; c < d; ++c) qd[c] = qrow64 ? qrow64[c] : bf16_bits_to_double(qrow[c]);

    /* scores over the visible keys */
    double m = -INFINITY;
    int64_t nvis = 0;
    for (int64_t j = 0; j < Nk; ++j) {
        if (!key_visible(pos, j, jb->causal, jb->window, L)) continue;
        double dot = 0.0;
        for (int64_t c = 0; c < d; ++c) dot += qd[c] * KVAL(j, c);
        s[j] = jb->scale * dot;
        if (s[j] > m) m = s[j];
        ++nvis;
    }
    for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
    if (nvis == 0) {
        *lse_out = -INFINITY;
        return;
    }

    /* log-sum-exp */
    double l = 0.0;
    for (int64_t j = 0; j < Nk; ++j) {
        if (!key_visible(pos, j, jb->causal, jb->window, L)) continue;
        l += exp(s[j] - m);
    }
    const double lse = m + log(l);
    *lse_out = lse;

    /* probability-weighted sum of value rows */
    for (int64_t j = 0; j < Nk; ++j) {
        if (!key_visible(pos, j, jb->causal, jb->window, L)) continue;
        const double p = exp(s[j] - lse);
        for (int64_t c = 0; c < d; ++c) o_row[c] += p * VVAL(j, c);
    }
#undef KVAL
#undef VVAL
}

static void *worker(void *arg) {
    const job_t *jb = (const job_t *)arg;
    double *qd = (double *)malloc(sizeof(double) * (size_t)jb->d);
    double *s = (double *)malloc(sizeof(double) * (size_t)jb->Nk);
    if (qd && s) {
        for (int64_t r = jb->row_begin; r < jb->row_end; ++r) {
            const int64_t flat = jb->rows ? jb->rows[r] : r;
            one_row(jb, flat, jb->o + r * jb->d, jb->lse + r, qd, s);
        }
    }
    free(qd);
    free(s);
    return NULL;
}

static int check_args(int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d,
                      int causal, int64_t window, double scale) {
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || N <= 0 || d <= 0) return -3;
    if (Hq % Hkv != 0) return -3;
    if (window < 0) return -3;
    if (!(scale > 0.0) || !isfinite(scale)) return -3;
    return 0;
}

/*
 * Compute the rows listed in `rows` (flat ids ((b*Hq)+hq)*N + i); when rows is NULL,
 * compute all B*Hq*N rows in order (nrows must then equal B*Hq*N).
 * o: nrows * d doubles, lse: nrows doubles. Returns 0, or a negative code for bad
 * arguments (-1 null pointer, -3 shape, -4 unsupported combination).
 */
static int rows_core(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const double *q64, const double *k64, const double *v64,
                     int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t Nk, int64_t d,
                     int causal, int64_t window, double scale, const int32_t *key_len,
                     const int64_t *rows, int64_t nrows, double *o, double *lse, int nthreads) {
    if (!(q || q64) || !(k || k64) || !(v || v64) || !o || !lse) return -1;
    int rc = check_args(B, Hq, Hkv, N, d, causal, window, scale);
    if (rc) return rc;
    if (Nk < N) return -3;
    if (nrows < 0) return -3;
    if (!rows && nrows != B * Hq * N) return -3;
    if (rows) {
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= B * Hq * N) return -3;
    }
    if (nrows == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = (int)nrows;

    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return -5;
    }
    for (int t = 0; t < nthreads; ++t) {
        job_t *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v;
        jb->qd64 = q64; jb->kd64 = k64; jb->vd64 = v64;
        jb->B = B; jb->Hq = Hq; jb->Hkv = Hkv; jb->N = N; jb->d = d; jb->Nk = Nk;
        jb->causal = causal; jb->window = window; jb->scale = scale;
        jb->key_len = key_len;
        jb->rows = rows;
        jb->row_begin = nrows * t / nthreads;
        jb->row_end = nrows * (t + 1) / nthreads;
        jb->o = o; jb->lse = lse;
    }
    int spawned = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, worker, &jobs[t]) != 0) break;
        spawned = t;
    }
    worker(&jobs[0]);
    for (int t = 1; t <= spawned; ++t) pthread_join(tids[t], NULL);
    /* rows of threads that failed to spawn are done here, serially */
    for (int t = spawned + 1; t < nthreads; ++t) worker(&jobs[t]);
    free(jobs);
    free(tids);
    return 0;
}

/* Plain forward (Nq = Nk = N): the rows listed in `rows` (flat ids ((b*Hq)+hq)*N + i),
 * or all rows in order when rows is NULL. key_len may be NULL. */
int attn_ref_fwd_rows_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d,
                          int causal, int64_t window, double scale, const int32_t *key_len,
                          const int64_t *rows, int64_t nrows, double *o, double *lse,
                          int nthreads) {
    return rows_core(q, k, v, NULL, NULL, NULL, B, Hq, Hkv, N, N, d, causal, window, scale, key_len,
                     rows, nrows, o, lse, nthreads);
}

/* Decode shape: q [B,Hq,Nq,d], k and v [B,Hkv,Nk,d], Nk >= Nq; rows are flat ids
 * ((b*Hq)+hq)*Nq + i, or all rows when NULL; o [nrows,d], lse [nrows]. */
int attn_ref_decode_rows_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                             int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nk, int64_t d,
                             int causal, int64_t window, double scale,
                             const int64_t *rows, int64_t nrows, double *o, double *lse,
                             int nthreads) {
    return rows_core(q, k, v, NULL, NULL, NULL, B, Hq, Hkv, Nq, Nk, d, causal, window, scale, NULL,
                     rows, nrows, o, lse, nthreads);
}

/* All rows: o is [B,Hq,N,d], lse is [B,Hq,N], both fp64. key_len may be NULL. */
int attn_ref_fwd_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d,
                     int causal, int64_t window, double scale, const int32_t *key_len,
                     double *o, double *lse, int nthreads) {
    return attn_ref_fwd_rows_f64(q, k, v, B, Hq, Hkv, N, d, causal, window, scale, key_len,
                                 NULL, B * Hq * N, o, lse, nthreads);
}

/* Plain forward on fp64 inputs (q [B,Hq,N,d], k and v [B,Hkv,N,d]): the same definition,
 * for inputs that are not bf16 values (for instance dequantised FP8 blocks). */
int attn_ref_fwd_rows_f64in(const double *q, const double *k, const double *v,
                            int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d,
                            int causal, int64_t window, double scale,
                            const int64_t *rows, int64_t nrows, double *o, double *lse,
                            int nthreads) {
    return rows_core(NULL, NULL, NULL, q, k, v, B, Hq, Hkv, N, N, d, causal, window, scale, NULL,
                     rows, nrows, o, lse, nthreads);
}

/*
 * FP8 (e4m3) block quantisation, after the FlashAttention-3 review's "Block
 * Quantization" and FP8 answers (deepmi.me): e4m3 has a sign bit, a 4-bit exponent and
 * a 3-bit mantissa; Q, K and V are split into blocks of B_r rows x d, each block gets
 * its own scale from its largest magnitude, and the scaled values are rounded to FP8.
 *
 * The e4m3 encoding used here (the OCP "E4M3FN" variant): exponent bias 7, no infinity,
 * the all-ones pattern S.1111.111 is NaN, so the largest finite magnitude is
 * 1.75 x 2^8 = 448; exponent field 0 holds subnormals m/8 x 2^-6. Rounding is to
 * nearest, ties to even, and magnitudes beyond 448 saturate to 448.
 */
static double e4m3_value(uint8_t code) {
    const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
    double mag;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        mag = ldexp((double)m / 8.0, -6);
    else
        mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* Round x (finite) to the nearest e4m3 value, ties to the even code; saturate at 448. */
static uint8_t e4m3_round(double x) {
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);  /* 448 = 1.75 x 2^8 */
    /* candidates: the two representable magnitudes around a, by exhaustive search over
     * the 127 non-negative finite codes (simple and obviously correct) */
    uint8_t best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double err = fabs(e4m3_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = (uint8_t)c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

void attn_ref_e4m3_decode(const uint8_t *codes, int64_t n, double *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
}

void attn_ref_e4m3_encode(const double *x, int64_t n, uint8_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_round(x[i]);
}

/*
 * Block quantisation of a bf16 tensor [BH, N, d] in blocks of `rows` x d: for block k of
 * head h, amax = max |x| (as fp32), inv = 448 / amax computed in fp32 (1 when amax is
 * 0), code = e4m3(x * inv) with the product rounded to fp32 first, and the block's
 * scale = amax / 448 in fp32 (the dequantised value is code x scale). Writes codes
 * [BH, N, d] and scales [BH, ceil(N / rows)].
 */
int attn_ref_quantize_e4m3_blocks(const uint16_t *x, int64_t BH, int64_t N, int64_t d, int64_t rows,
                                  uint8_t *codes, float *scales) {
    if (!x || !codes || !scales || BH < 1 || N < 1 || d < 1 || rows < 1) return -1;
    const int64_t nblk = (N + rows - 1) / rows;
    for (int64_t h = 0; h < BH; ++h) {
        for (int64_t k = 0; k < nblk; ++k) {
            const int64_t r0 = k * rows, r1 = (r0 + rows < N) ? r0 + rows : N;
            float amax = 0.0f;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t c = 0; c < d; ++c) {
                    const float a = fabsf((float)bf16_bits_to_double(x[(h * N + r) * d + c]));
                    if (a > amax) amax = a;
                }
            const float inv = (amax > 0.0f) ? 448.0f / amax : 1.0f;
            scales[h * nblk + k] = (amax > 0.0f) ? amax / 448.0f : 1.0f;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t c = 0; c < d; ++c) {
                    const volatile float prod = (float)bf16_bits_to_double(x[(h * N + r) * d + c]) * inv;
                    codes[(h * N + r) * d + c] = e4m3_round((double)prod);
                }
        }
    }
    return 0;
}

/*
 * Block quantisation of real-valued inputs [BH, N, d] (fp64), for the incoherent-processing
 * path, whose rotated values are not bf16: for block k of head h, amax = max |x|,
 * code = e4m3(x * 448 / amax) and scale = amax / 448, all in fp64 (the exact definition);
 * an all-zero block gets scale 1 and zero codes. Writes codes [BH, N, d] and scales
 * [BH, ceil(N / rows)].
 */
int attn_ref_quantize_e4m3_blocks_f64(const double *x, int64_t BH, int64_t N, int64_t d, int64_t rows,
                                      uint8_t *codes, double *scales) {
    if (!x || !codes || !scales || BH < 1 || N < 1 || d < 1 || rows < 1) return -1;
    const int64_t nblk = (N + rows - 1) / rows;
    for (int64_t h = 0; h < BH; ++h) {
        for (int64_t k = 0; k < nblk; ++k) {
            const int64_t r0 = k * rows, r1 = (r0 + rows < N) ? r0 + rows : N;
            double amax = 0.0;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t c = 0; c < d; ++c) {
                    const double a = fabs(x[(h * N + r) * d + c]);
                    if (a > amax) amax = a;
                }
            scales[h * nblk + k] = amax > 0.0 ? amax / 448.0 : 1.0;
            for (int64_t r = r0; r < r1; ++r)
                for (int64_t c = 0; c < d; ++c)
                    codes[(h * N + r) * d + c] =
                        amax > 0.0 ? e4m3_round(x[(h * N + r) * d + c] * (448.0 / amax)) : (uint8_t)0;
        }
    }
    return 0;
}

/*
 * Backward pass: gradients of the attention forward (o above) with respect to q, k, v
 * for an upstream gradient do_ = dL/do, restated from the chain rule through the
 * definition (the pages only say that the backward pass exists and costs about 2.5x the
 * forward, FlashAttention-3 review, FLOPs answer):
 *
 *   p_ij  = exp(s_ij - lse_i) for j in J(i), 0 otherwise       (the softmax weights)
 *   dp_ij = do_i . v_j                                          (dL/dp)
 *   ds_ij = p_ij (dp_ij - sum_l p_il dp_il)                     (through the softmax)
 *   dq_i  = scale sum_j ds_ij k_j
 *   dk_j  = scale sum over (query head of the group, i) of ds_ij q_i
 *   dv_j  = sum over (query head of the group, i) of p_ij do_i
 *
 * Inputs bf16 bits (q, k, v, do_ as for the forward); outputs fp64, dq [B,Hq,N,d], dk and
 * dv [B,Hkv,N,d].
 *
 * Threads: the flat query rows (b * Hq + hq) * N + i are split into contiguous slices,
 * one per thread. dq rows are disjoint between slices. Each slice adds its dk and dv
 * terms into private buffers that cover the key-value heads its rows read, and the
 * buffers are then added into dk and dv in slice order, so a given thread count always
 * gives the same bits. With one thread the sums are formed in exactly the order of a
 * plain loop over b, hq, i.
 *
 * o_in: NULL, or a given forward output [B,Hq,N,d] (fp64). A backward pass that takes
 * the forward's output as an input forms the row sum sum_l p_il dp_il as do_i . o_i,
 * which equals it exactly when o_i is the exact output (o_i = sum_l p_il v_l); with a
 * given o_in the row sum is do_i . o_in_i, so the gradients are those a backward pass
 * computes from that o.
 */
typedef struct {
    const uint16_t *q, *k, *v, *do_;
    const double *o_in;
    int64_t B, Hq, Hkv, N, d, window, group;
    int causal;
    double scale;
    const int32_t *key_len;
    int64_t row_begin, row_end; /* flat query rows of this slice */
    int64_t kv_first;           /* first flat key-value head (b * Hkv + kv) the slice reads */
    double *dq;                 /* shared; the slice writes only its own rows */
    double *dk, *dv;            /* private, from head kv_first on */
    int rc;
} bwd_job_t;

static void *bwd_worker(void *arg) {
    bwd_job_t *jb = (bwd_job_t *)arg;
    const int64_t N = jb->N, d = jb->d, Hq = jb->Hq, Hkv = jb->Hkv;
    double *p = (double *)malloc(sizeof(double) * (size_t)N);
    double *dp = (double *)malloc(sizeof(double) * (size_t)N);
    if (!p || !dp) {
        free(p);
        free(dp);
        jb->rc = -5;
        return NULL;
    }
    for (int64_t r = jb->row_begin; r < jb->row_end; ++r) {
        const int64_t bh = r / N, i = r % N, b = bh / Hq, hq = bh % Hq, kv = hq / jb->group;
        int64_t L = jb->key_len ? (int64_t)jb->key_len[b] : N;
        if (L < 0) L = 0;
        if (L > N) L = N;
        const uint16_t *qh = jb->q + bh * N * d, *doh = jb->do_ + bh * N * d;
        const uint16_t *kh = jb->k + (b * Hkv + kv) * N * d, *vh = jb->v + (b * Hkv + kv) * N * d;
        double *dqh = jb->dq + bh * N * d;
        double *dkh = jb->dk + (b * Hkv + kv - jb->kv_first) * N * d;
        double *dvh = jb->dv + (b * Hkv + kv - jb->kv_first) * N * d;
        /* scores, their maximum and the log-sum-exp over the visible keys */
        double m = -INFINITY;
        int64_t nvis = 0;
        for (int64_t j = 0; j < N; ++j) {
            p[j] = 0.0;
            if (!key_visible(i, j, jb->causal, jb->window, L)) continue;
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += bf16_bits_to_double(qh[i * d + c]) * bf16_bits_to_double(kh[j * d + c]);
            p[j] = jb->scale * dot; /* the score, for now */
            if (p[j] > m) m = p[j];
            ++nvis;
        }
        if (nvis == 0) continue; /* a row with no visible key contributes nothing */
        double l = 0.0;
        for (int64_t j = 0; j < N; ++j)
            if (key_visible(i, j, jb->causal, jb->window, L)) l += exp(p[j] - m);
        const double lse = m + log(l);
        double pdp = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            if (!key_visible(i, j, jb->causal, jb->window, L)) {
                p[j] = 0.0;
                dp[j] = 0.0;
                continue;
            }
            p[j] = exp(p[j] - lse);
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += bf16_bits_to_double(doh[i * d + c]) * bf16_bits_to_double(vh[j * d + c]);
            dp[j] = dot;
            pdp += p[j] * dp[j];
        }
        if (jb->o_in) {
            const double *oi = jb->o_in + (bh * N + i) * d;
            pdp = 0.0;
            for (int64_t c = 0; c < d; ++c) pdp += bf16_bits_to_double(doh[i * d + c]) * oi[c];
        }
        for (int64_t j = 0; j < N; ++j) {
            if (p[j] == 0.0 && dp[j] == 0.0) continue;
            const double ds = p[j] * (dp[j] - pdp);
            for (int64_t c = 0; c < d; ++c) {
                dqh[i * d + c] += jb->scale * ds * bf16_bits_to_double(kh[j * d + c]);
                dkh[j * d + c] += jb->scale * ds * bf16_bits_to_double(qh[i * d + c]);
                dvh[j * d + c] += p[j] * bf16_bits_to_double(doh[i * d + c]);
            }
        }
    }
    free(p);
    free(dp);
    return NULL;
}

static int bwd_core(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *do_,
                    const double *o_in, int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d,
                    int causal, int64_t window, double scale, const int32_t *key_len,
                    double *dq, double *dk, double *dv, int nthreads) {
    if (!q || !k || !v || !do_ || !dq || !dk || !dv) return -1;
    int rc = check_args(B, Hq, Hkv, N, d, causal, window, scale);
    if (rc) return rc;
    const int64_t group = Hq / Hkv, nrows = B * Hq * N;
    for (int64_t i = 0; i < B * Hq * N * d; ++i) dq[i] = 0.0;
    for (int64_t i = 0; i < B * Hkv * N * d; ++i) dk[i] = dv[i] = 0.0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = (int)nrows;
    bwd_job_t *jobs = (bwd_job_t *)calloc((size_t)nthreads, sizeof(bwd_job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    int ok = jobs && tids;
    for (int t = 0; ok && t < nthreads; ++t) {
        bwd_job_t *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->do_ = do_; jb->o_in = o_in;
        jb->B = B; jb->Hq = Hq; jb->Hkv = Hkv; jb->N = N; jb->d = d;
        jb->window = window; jb->group = group; jb->causal = causal; jb->scale = scale;
        jb->key_len = key_len;
        jb->row_begin = nrows * t / nthreads;
        jb->row_end = nrows * (t + 1) / nthreads;
        jb->dq = dq;
        /* rows of head bh read key-value head bh / group (b * Hkv + hq / group) */
        jb->kv_first = (jb->row_begin / N) / group;
        const int64_t kv_last = ((jb->row_end - 1) / N) / group;
        const size_t n = (size_t)(kv_last - jb->kv_first + 1) * (size_t)(N * d);
        jb->dk = (double *)calloc(n, sizeof(double));
        jb->dv = (double *)calloc(n, sizeof(double));
        if (!jb->dk || !jb->dv) ok = 0;
    }
    if (ok) {
        int spawned = 0;
        for (int t = 1; t < nthreads; ++t) {
            if (pthread_create(&tids[t], NULL, bwd_worker, &jobs[t]) != 0) break;
            spawned = t;
        }
        bwd_worker(&jobs[0]);
        for (int t = 1; t <= spawned; ++t) pthread_join(tids[t], NULL);
        /* slices whose thread failed to start run here, serially */
        for (int t = spawned + 1; t < nthreads; ++t) bwd_worker(&jobs[t]);
        /* the private dk, dv partials, added in slice order */
        for (int t = 0; t < nthreads; ++t) {
            const bwd_job_t *jb = &jobs[t];
            if (jb->rc) ok = 0;
            const int64_t kv_last = ((jb->row_end - 1) / N) / group;
            const int64_t off = jb->kv_first * N * d, n = (kv_last - jb->kv_first + 1) * N * d;
            for (int64_t e = 0; e < n; ++e) {
                dk[off + e] += jb->dk[e];
                dv[off + e] += jb->dv[e];
            }
        }
    }
    if (jobs)
        for (int t = 0; t < nthreads; ++t) {
            free(jobs[t].dk);
            free(jobs[t].dv);
        }
    free(jobs);
    free(tids);
    return ok ? 0 : -5;
}

int attn_ref_bwd_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *do_,
                     int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d, int causal,
                     int64_t window, double scale, const int32_t *key_len,
                     double *dq, double *dk, double *dv, int nthreads) {
    return bwd_core(q, k, v, do_, NULL, B, Hq, Hkv, N, d, causal, window, scale, key_len, dq, dk, dv,
                    nthreads);
}

/*
 * The query gradient of selected rows, each from its own row of the definition (the
 * backward above restricted to dq): for flat query row r = (b * Hq + hq) * N + i,
 * p_ij and dp_ij over the keys row i sees, D_i = sum_j p_ij dp_ij, and
 * dq_i = scale sum_j p_ij (dp_ij - D_i) k_j. Writes dq [nrows, d] (fp64). Cost O(N d)
 * per row, so rows of full-size problems can be checked one by one.
 */
int attn_ref_bwd_dq_rows_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *do_,
                             int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d, int causal,
                             int64_t window, double scale, const int32_t *key_len, const int64_t *rows,
                             int64_t nrows, double *dq) {
    if (!q || !k || !v || !do_ || !rows || !dq || nrows < 0) return -1;
    int rc = check_args(B, Hq, Hkv, N, d, causal, window, scale);
    if (rc) return rc;
    const int64_t group = Hq / Hkv;
    double *p = (double *)malloc(sizeof(double) * (size_t)N);
    double *dp = (double *)malloc(sizeof(double) * (size_t)N);
    if (!p || !dp) {
        free(p);
        free(dp);
        return -5;
    }
    for (int64_t n = 0; n < nrows; ++n) {
        const int64_t r = rows[n];
        double *out = dq + n * d;
        for (int64_t c = 0; c < d; ++c) out[c] = 0.0;
        if (r < 0 || r >= B * Hq * N) {
            free(p);
            free(dp);
            return -2;
        }
        const int64_t bh = r / N, i = r % N, b = bh / Hq, hq = bh % Hq, kv = hq / group;
        int64_t L = key_len ? (int64_t)key_len[b] : N;
        if (L < 0) L = 0;
        if (L > N) L = N;
        const uint16_t *qi = q + r * d, *doi = do_ + r * d;
        const uint16_t *kh = k + (b * Hkv + kv) * N * d, *vh = v + (b * Hkv + kv) * N * d;
        double m = -INFINITY;
        for (int64_t j = 0; j < N; ++j) {
            p[j] = 0.0;
            if (!key_visible(i, j, causal, window, L)) continue;
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c) dot += bf16_bits_to_double(qi[c]) * bf16_bits_to_double(kh[j * d + c]);
            p[j] = scale * dot;
            if (p[j] > m) m = p[j];
        }
        if (m == -INFINITY) continue; /* no visible key: dq = 0 */
        double l = 0.0;
        for (int64_t j = 0; j < N; ++j)
            if (key_visible(i, j, causal, window, L)) l += exp(p[j] - m);
        const double lse = m + log(l);
        double dsum = 0.0;
        for (int64_t j = 0; j < N; ++j) {
            dp[j] = 0.0;
            if (!key_visible(i, j, causal, window, L)) {
                p[j] = 0.0;
                continue;
            }
            p[j] = exp(p[j] - lse);
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c) dot += bf16_bits_to_double(doi[c]) * bf16_bits_to_double(vh[j * d + c]);
            dp[j] = dot;
            dsum += p[j] * dp[j];
        }
        for (int64_t j = 0; j < N; ++j) {
            if (p[j] == 0.0) continue;
            const double ds = p[j] * (dp[j] - dsum);
            for (int64_t c = 0; c < d; ++c) out[c] += scale * ds * bf16_bits_to_double(kh[j * d + c]);
        }
    }
    free(p);
    free(dp);
    return 0;
}

int attn_ref_bwd_given_o_f64(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *do_,
                             const double *o_in, int64_t B, int64_t Hq, int64_t Hkv, int64_t N, int64_t d,
                             int causal, int64_t window, double scale, const int32_t *key_len,
                             double *dq, double *dk, double *dv, int nthreads) {
    if (!o_in) return -1;
    return bwd_core(q, k, v, do_, o_in, B, Hq, Hkv, N, d, causal, window, scale, key_len, dq, dk, dv,
                    nthreads);
}
