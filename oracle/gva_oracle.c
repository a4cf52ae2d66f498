/*
 * gva_oracle.c -- plain fp64 CPU oracle for Grouped Value Attention (GVA) decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU
 * baseline leg load this file's library.  It shares no code, header, table or
 * constant generator with the CUDA library; the two meet only through the seeded
 * inputs that both are handed.
 *
 * Sources (web pages, cited by title and section):
 *   [A]  "GVA：KV 缓存里的 Key 其实可以不存——从 Value 里"现算"出来就行"
 *        (shibing624.github.io analysis of arXiv 2609.13285)
 *   [S]  "Grouped Value Attention: Efficient KV Caching via On-Demand Key
 *        Reconstruction" (agihunt.info summary)
 *   [K]  "KV Cache 优化（一）：从 MHA 到 MQA 与 GQA" (liumengxuan04.github.io)
 *   [C]  KV-cache compression survey MHA -> MQA -> GQA -> MLA (ttsmallhot.github.io)
 *
 * Everything here is the definition written out, in the order the pages state it:
 * no blocking, no fusion, no online softmax.  All floating point is double except
 * the append path, whose stored bf16/fp32 code is decided in fp32 (see od_append).
 *
 * Readings taken where the pages are silent:
 *   - RoPE pairs are interleaved (x[2i], x[2i+1]), theta_i = base^(-2i/d_r),
 *     angle = p * theta_i with 0-based position p; Rot(p): y0 = x0 c - x1 s,
 *     y1 = x0 s + x1 c.  ([A] "关键技巧二" names only the relative rotation R_{j-t}.)
 *   - The query of a decode step sits at position t = L_b - 1: the newest token is
 *     appended first and attended to ([K] §1: append, then read all history 1..t).
 *   - The head-to-group map is contiguous blocks of r = H/G heads ([C] §2.2, [K] §4).
 *   - L_b = 0 gives out = 0 and lse = -inf.
 *   - The softmax scale is a caller argument (the workloads use 1/sqrt(d_n + d_r)).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* threads                                                                    */
/* ------------------------------------------------------------------------- */
void od_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int od_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------- */
/* storage rows: where logical token (b, j) lives                              */
/* ------------------------------------------------------------------------- */
/* kind 0: contiguous, row = b*T_cap + j
 * kind 1: ragged,     row = offsets[b] + j
 * kind 2: paged,      row = block_table[b*max_pages + j/page_size]*page_size + j%page_size
 * (paging changes only where bytes sit, not the attention maths: [K] §7) */
typedef struct {
    int kind;
    long long T_cap;
    const long long *offsets;
    const long long *block_table;
    int max_pages;
    int page_size;
} od_rows;

long long od_row(const od_rows *R, int b, long long j)
{
    if (R->kind == 0) return (long long)b * R->T_cap + j;
    if (R->kind == 1) return R->offsets[b] + j;
    {
        long long page = R->block_table[(long long)b * R->max_pages + j / R->page_size];
        return page * R->page_size + j % R->page_size;
    }
}

/* ------------------------------------------------------------------------- */
/* RoPE                                                                       */
/* ------------------------------------------------------------------------- */
/* theta_i = base^(-2i/d_r) */
double od_rope_theta(int i, int d_r, double base)
{
    return pow(base, -(2.0 * (double)i) / (double)d_r);
}

/* y = Rot(p) x on interleaved pairs, fp64. */
void od_rotate(const double *x, double *y, int d_r, long long p, double base)
{
    int i;
    for (i = 0; i < d_r / 2; ++i) {
        double ang = (double)p * od_rope_theta(i, d_r, base);
        double c = cos(ang), s = sin(ang);
        double x0 = x[2 * i], x1 = x[2 * i + 1];
        y[2 * i] = x0 * c - x1 * s;
        y[2 * i + 1] = x0 * s + x1 * c;
    }
}

/* fp32 cos/sin table [max_pos][d_r/2][2]: each value is the fp64 libm result
 * rounded once to fp32. */
void od_rope_table_f32(float *tab, int max_pos, int d_r, double base)
{
    long long p;
    int i;
    for (p = 0; p < max_pos; ++p)
        for (i = 0; i < d_r / 2; ++i) {
            double ang = (double)p * od_rope_theta(i, d_r, base);
            tab[(p * (d_r / 2) + i) * 2 + 0] = (float)cos(ang);
            tab[(p * (d_r / 2) + i) * 2 + 1] = (float)sin(ang);
        }
}

/* ------------------------------------------------------------------------- */
/* bf16 round-to-nearest-even from fp32 bits                                   */
/* ------------------------------------------------------------------------- */
uint16_t od_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
        return (uint16_t)((u >> 16) | 0x0040u);          /* NaN stays NaN (quiet) */
    u += 0x7fffu + ((u >> 16) & 1u);                      /* ties go to even */
    return (uint16_t)(u >> 16);
}

void od_bf16_rne_array(const float *x, uint16_t *y, long long n)
{
    long long i;
    for (i = 0; i < n; ++i) y[i] = od_bf16_rne(x[i]);
}

/* ------------------------------------------------------------------------- */
/* Query absorption  ([A] "关键技巧一", [S])                                    */
/* ------------------------------------------------------------------------- */
/* q_tilde[b,h,i] = scale * sum_k q_nope[b,h,k] * M[h,i,k]     (q~_h = q_h^nope M_h^T,
 *                                                              M_h in R^{d_h x d_n})
 * q_hat[b,h]     = scale * Rot(t) q_rope[b,h],  t = L_b - 1 (0 when L_b = 0)  */
void od_absorb(int B, int H, int d_h, int d_n, int d_r,
               const double *q_nope, const double *q_rope, const double *M,
               const long long *seq_len, double scale, double base,
               double *q_tilde, double *q_hat)
{
    int b, h, i, k;
    for (b = 0; b < B; ++b)
        for (h = 0; h < H; ++h) {
            const double *qn = q_nope + ((long long)b * H + h) * d_n;
            const double *Mh = M + (long long)h * d_h * d_n;
            double *qt = q_tilde + ((long long)b * H + h) * d_h;
            long long t = seq_len[b] > 0 ? seq_len[b] - 1 : 0;
            for (i = 0; i < d_h; ++i) {
                double acc = 0.0;
                for (k = 0; k < d_n; ++k) acc += qn[k] * Mh[(long long)i * d_n + k];
                qt[i] = scale * acc;
            }
            if (d_r > 0) {
                double *qh = q_hat + ((long long)b * H + h) * d_r;
                od_rotate(q_rope + ((long long)b * H + h) * d_r, qh, d_r, t, base);
                for (i = 0; i < d_r; ++i) qh[i] *= scale;
            }
        }
}

/* ------------------------------------------------------------------------- */
/* Query RMSNorm  ([A] 实验: "GVA scale-matched + query RMSNorm"; [S] results   */
/* table "GVA, scale-matched + query RMSNorm")                                  */
/* ------------------------------------------------------------------------- */
/* The pages name the variant without its formula.  The reading taken here, the
 * ordinary RMSNorm: each head's content query is divided by its root mean square over
 * its d_n values, then multiplied by a per-dimension gain (ones when gain is NULL):
 *   y[b,h,k] = gain[k] * x[b,h,k] / sqrt( (1/d_n) sum_k' x[b,h,k']^2 + eps )
 * The positional query is not normalised. */
void od_query_rmsnorm(int B, int H, int d_n, const double *x, const double *gain, double eps,
                      double *y)
{
    long long bh;
    int k;
    for (bh = 0; bh < (long long)B * H; ++bh) {
        const double *xr = x + bh * d_n;
        double ss = 0.0, inv;
        for (k = 0; k < d_n; ++k) ss += xr[k] * xr[k];
        inv = 1.0 / sqrt(ss / (double)d_n + eps);
        for (k = 0; k < d_n; ++k) y[bh * d_n + k] = (gain ? gain[k] : 1.0) * xr[k] * inv;
    }
}

/* ------------------------------------------------------------------------- */
/* exact widening of one stored cache element to double                        */
/* ------------------------------------------------------------------------- */
/* bf16 storage: the 16 bits are the top half of an fp32; fp32 storage as is.
 * Both widen to double exactly. */
static double od_load(const void *base_ptr, long long idx, int is_bf16)
{
    if (is_bf16) {
        uint32_t u = (uint32_t)((const uint16_t *)base_ptr)[idx] << 16;
        float f;
        memcpy(&f, &u, 4);
        return (double)f;
    }
    return (double)((const float *)base_ptr)[idx];
}

/* ------------------------------------------------------------------------- */
/* softmax-weighted sum over one sequence's scores (two-pass, max subtracted)  */
/* ------------------------------------------------------------------------- */
/* out[i] = sum_j softmax(z)_j * val_j[i],  lse = max z + ln sum exp(z - max z)
 * ([K] §1 eq. for o_t; [C] §1.1 single-head attention) */
static void softmax_sum(const double *z, long long L, const od_rows *R, int b,
                        const void *vals, int vals_bf16, long long row_stride,
                        long long col0, int width, double *out, double *lse)
{
    long long j;
    int i;
    double zmax = -INFINITY, den = 0.0;
    for (i = 0; i < width; ++i) out[i] = 0.0;
    if (L == 0) {
        *lse = -INFINITY;
        return;
    }
    for (j = 0; j < L; ++j)
        if (z[j] > zmax) zmax = z[j];
    for (j = 0; j < L; ++j) den += exp(z[j] - zmax);
    for (j = 0; j < L; ++j) {
        double p = exp(z[j] - zmax) / den;
        long long v0 = od_row(R, b, j) * row_stride + col0;
        for (i = 0; i < width; ++i) out[i] += p * od_load(vals, v0 + i, vals_bf16);
    }
    *lse = zmax + log(den);
}

/* ------------------------------------------------------------------------- */
/* GVA decode, absorbed path  ([A] "关键技巧一/二", [S])                         */
/* ------------------------------------------------------------------------- */
/* For each (b, h), g = h / (H/G), t = L_b - 1:
 *   z_j = scale * ( (q_nope M_h^T) . v_{j,g} + (Rot(t) q_rope) . k_rope_j ),  j < L_b
 *   out[b,h] = sum_j softmax(z)_j v_{j,g};  lse[b,h] = logsumexp(z)
 * V rows hold [G][d_h]; K_rope rows hold [d_r] (already rotated to their own
 * position, [S]). */
void od_gva_decode(int B, int H, int G, int d_h, int d_n, int d_r,
                   const double *q_nope, const double *q_rope, const double *M,
                   const long long *seq_len, const od_rows *R,
                   const void *V, const void *Kr, int cache_bf16, double scale,
                   double base, double *out, double *lse)
{
    int r = H / G;
    long long bh;
#pragma omp parallel for schedule(dynamic, 1)
    for (bh = 0; bh < (long long)B * H; ++bh) {
        int b = (int)(bh / H), h = (int)(bh % H), g = h / r, i, k, c;
        long long L = seq_len[b], t = L > 0 ? L - 1 : 0, j;
        const double *qn = q_nope + bh * d_n;
        const double *Mh = M + (long long)h * d_h * d_n;
        double *qt = (double *)malloc(sizeof(double) * (size_t)d_h);
        double *qh = (double *)malloc(sizeof(double) * (size_t)(d_r > 0 ? d_r : 1));
        double *z = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        for (i = 0; i < d_h; ++i) {
            double acc = 0.0;
            for (k = 0; k < d_n; ++k) acc += qn[k] * Mh[(long long)i * d_n + k];
            qt[i] = acc;
        }
        if (d_r > 0) od_rotate(q_rope + bh * d_r, qh, d_r, t, base);
        for (j = 0; j < L; ++j) {
            long long row = od_row(R, b, j);
            long long v0 = (row * G + g) * d_h;
            double s = 0.0;
            for (i = 0; i < d_h; ++i) s += qt[i] * od_load(V, v0 + i, cache_bf16);
            for (c = 0; c < d_r; ++c) s += qh[c] * od_load(Kr, row * d_r + c, cache_bf16);
            z[j] = scale * s;
        }
        softmax_sum(z, L, R, b, V, cache_bf16, (long long)G * d_h, (long long)g * d_h, d_h,
                    out + bh * d_h, lse + bh);
        free(qt);
        free(qh);
        free(z);
    }
}

/* ------------------------------------------------------------------------- */
/* GVA decode, explicit path: the content key is materialised                  */
/* ------------------------------------------------------------------------- */
/* K_h[j] = v_{j,g} M_h (width d_n, [A] eq. K_h = V_{g(h)} M_h); the key of token
 * j is [K_h[j] ; k_rope_j], the query is [q_nope ; Rot(t) q_rope], and the score
 * is the ordinary scaled dot product ([A] "关键技巧二": q k^T = q^nope k^nope +
 * q^rope k^rope).  Used to check the absorption identity; costs d_h*d_n per
 * token and head. */
void od_gva_decode_explicit(int B, int H, int G, int d_h, int d_n, int d_r,
                            const double *q_nope, const double *q_rope, const double *M,
                            const long long *seq_len, const od_rows *R,
                            const void *V, const void *Kr, int cache_bf16, double scale,
                            double base, double *out, double *lse)
{
    int r = H / G;
    long long bh;
#pragma omp parallel for schedule(dynamic, 1)
    for (bh = 0; bh < (long long)B * H; ++bh) {
        int b = (int)(bh / H), h = (int)(bh % H), g = h / r, i, k, c;
        long long L = seq_len[b], t = L > 0 ? L - 1 : 0, j;
        const double *qn = q_nope + bh * d_n;
        const double *Mh = M + (long long)h * d_h * d_n;
        double *key = (double *)malloc(sizeof(double) * (size_t)(d_n + d_r));
        double *qfull = (double *)malloc(sizeof(double) * (size_t)(d_n + d_r));
        double *z = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        for (k = 0; k < d_n; ++k) qfull[k] = qn[k];
        if (d_r > 0) od_rotate(q_rope + bh * d_r, qfull + d_n, d_r, t, base);
        for (j = 0; j < L; ++j) {
            long long row = od_row(R, b, j);
            long long v0 = (row * G + g) * d_h;
            double s = 0.0;
            for (k = 0; k < d_n; ++k) {          /* (v M_h)[k] = sum_i v[i] M_h[i,k] */
                double acc = 0.0;
                for (i = 0; i < d_h; ++i) acc += od_load(V, v0 + i, cache_bf16) * Mh[(long long)i * d_n + k];
                key[k] = acc;
            }
            for (c = 0; c < d_r; ++c) key[d_n + c] = od_load(Kr, row * d_r + c, cache_bf16);
            for (k = 0; k < d_n + d_r; ++k) s += qfull[k] * key[k];
            z[j] = scale * s;
        }
        softmax_sum(z, L, R, b, V, cache_bf16, (long long)G * d_h, (long long)g * d_h, d_h,
                    out + bh * d_h, lse + bh);
        free(key);
        free(qfull);
        free(z);
    }
}

/* ------------------------------------------------------------------------- */
/* GVA with ordinary RoPE on the reconstructed key (the non-absorbable variant) */
/* ------------------------------------------------------------------------- */
/* [S] (results discussion): the scale-matched row rotates the rebuilt key itself with
 * plain RoPE, so M cannot be folded into the query there; [A] 关键技巧二: the relative rotation
 * R_{j-t} sits between q and M^T, so no single transformed query serves every cached
 * position.  The pages give no formula; the reading taken: the key of token j for head h is
 * K_h[j] = v_{j,g(h)} M_h (width d_n), rotated by its own position j; the query q_h
 * (width d_n, the whole query) is rotated by t = L_b - 1 with the same pairing;
 *   z_j = scale * (Rot(t) q_h) . (Rot(j) K_h[j]),   out = softmax(z) V_g (unrotated);
 * there is no separate positional key.  pos_offset adds a constant to every position
 * (t and all j), for the relative-position check. */
void od_gva_decode_rope_keys(int B, int H, int G, int d_h, int d_n, const double *q,
                             const double *M, const long long *seq_len, const od_rows *R,
                             const void *V, int cache_bf16, double scale, double base,
                             long long pos_offset, double *out, double *lse)
{
    int r = H / G;
    long long bh;
#pragma omp parallel for schedule(dynamic, 1)
    for (bh = 0; bh < (long long)B * H; ++bh) {
        int b = (int)(bh / H), h = (int)(bh % H), g = h / r, i, k;
        long long L = seq_len[b], t = L > 0 ? L - 1 : 0, j;
        const double *Mh = M + (long long)h * d_h * d_n;
        double *key = (double *)malloc(sizeof(double) * (size_t)d_n);
        double *keyr = (double *)malloc(sizeof(double) * (size_t)d_n);
        double *qr = (double *)malloc(sizeof(double) * (size_t)d_n);
        double *z = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        od_rotate(q + bh * d_n, qr, d_n, t + pos_offset, base);
        for (j = 0; j < L; ++j) {
            long long v0 = (od_row(R, b, j) * G + g) * d_h;
            double s = 0.0;
            for (k = 0; k < d_n; ++k) {          /* (v M_h)[k] = sum_i v[i] M_h[i,k] */
                double acc = 0.0;
                for (i = 0; i < d_h; ++i) acc += od_load(V, v0 + i, cache_bf16) * Mh[(long long)i * d_n + k];
                key[k] = acc;
            }
            od_rotate(key, keyr, d_n, j + pos_offset, base);
            for (k = 0; k < d_n; ++k) s += qr[k] * keyr[k];
            z[j] = scale * s;
        }
        softmax_sum(z, L, R, b, V, cache_bf16, (long long)G * d_h, (long long)g * d_h, d_h,
                    out + bh * d_h, lse + bh);
        free(key);
        free(keyr);
        free(qr);
        free(z);
    }
}

/* ------------------------------------------------------------------------- */
/* MLA-shaped decode (a second comparator; [A] 问题 and 对 MLA 的优势: a joint latent   */
/* of width d_c plus one shared RoPE channel, T(d_c + d_r) cached scalars; [C]    */
/* 3.1.2-3.1.3: per-head up-projections of the latent to K and V, decoupled RoPE)  */
/* ------------------------------------------------------------------------- */
/* Explicit path.  Cache rows: latent c_j [d_c], shared positional key k_rope_j [d_r]
 * (already rotated, as for GVA).  For head h, with row-vector products as for GVA's
 * K_h = V M_h:
 *   K_h[j] = c_j Wuk_h  (Wuk_h in R^{d_c x d_n}),   V_h[j] = c_j Wuv_h  (Wuv_h in R^{d_c x d_h})
 *   key_j = [K_h[j] ; k_rope_j],  query = [q_nope ; Rot(t) q_rope],  t = L_b - 1
 *   z_j = scale * query . key_j,  out[b,h] = sum_j softmax(z)_j V_h[j],  lse = logsumexp(z)
 * The reading taken where the pages differ: the positional key is one shared stream
 * ([A]; [C] describes per-head positional keys, which is DeepSeek's MLA, not the
 * T(d_c + d_r) count the GVA pages compare with). */
void od_mla_decode(int B, int H, int d_c, int d_n, int d_h, int d_r, const double *q_nope,
                   const double *q_rope, const double *Wuk, const double *Wuv,
                   const long long *seq_len, const od_rows *R, const void *C, const void *Kr,
                   int cache_bf16, double scale, double base, double *out, double *lse)
{
    long long bh;
#pragma omp parallel for schedule(dynamic, 1)
    for (bh = 0; bh < (long long)B * H; ++bh) {
        int b = (int)(bh / H), h = (int)(bh % H), i, k, c;
        long long L = seq_len[b], t = L > 0 ? L - 1 : 0, j;
        const double *Wk = Wuk + (long long)h * d_c * d_n;
        const double *Wv = Wuv + (long long)h * d_c * d_h;
        double *qh = (double *)malloc(sizeof(double) * (size_t)(d_r > 0 ? d_r : 1));
        double *z = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        double zmax = -INFINITY, den = 0.0;
        if (d_r > 0) od_rotate(q_rope + bh * d_r, qh, d_r, t, base);
        for (j = 0; j < L; ++j) {
            long long row = od_row(R, b, j);
            double s = 0.0;
            for (k = 0; k < d_n; ++k) {          /* (c_j Wuk_h)[k] */
                double acc = 0.0;
                for (c = 0; c < d_c; ++c) acc += od_load(C, row * d_c + c, cache_bf16) * Wk[(long long)c * d_n + k];
                s += q_nope[bh * d_n + k] * acc;
            }
            for (c = 0; c < d_r; ++c) s += qh[c] * od_load(Kr, row * d_r + c, cache_bf16);
            z[j] = scale * s;
            if (z[j] > zmax) zmax = z[j];
        }
        for (i = 0; i < d_h; ++i) out[bh * d_h + i] = 0.0;
        if (L == 0) {
            lse[bh] = -INFINITY;
        } else {
            for (j = 0; j < L; ++j) den += exp(z[j] - zmax);
            for (j = 0; j < L; ++j) {
                long long row = od_row(R, b, j);
                double p = exp(z[j] - zmax) / den;
                for (i = 0; i < d_h; ++i) {      /* (c_j Wuv_h)[i] */
                    double acc = 0.0;
                    for (c = 0; c < d_c; ++c) acc += od_load(C, row * d_c + c, cache_bf16) * Wv[(long long)c * d_h + i];
                    out[bh * d_h + i] += p * acc;
                }
            }
            lse[bh] = zmax + log(den);
        }
        free(qh);
        free(z);
    }
}

/* ------------------------------------------------------------------------- */
/* GQA decode (the matched comparator)  ([K] §4, [C] §2.2)                     */
/* ------------------------------------------------------------------------- */
/* head_h = softmax(scale * q_h K_g^T) V_g with explicit K and V rows [G][d_h]. */
void od_gqa_decode(int B, int H, int G, int d_h, const double *q,
                   const long long *seq_len, const od_rows *R,
                   const void *K, const void *V, int cache_bf16, double scale,
                   double *out, double *lse)
{
    int r = H / G;
    long long bh;
#pragma omp parallel for schedule(dynamic, 1)
    for (bh = 0; bh < (long long)B * H; ++bh) {
        int b = (int)(bh / H), h = (int)(bh % H), g = h / r, i;
        long long L = seq_len[b], j;
        const double *qh = q + bh * d_h;
        double *z = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
        for (j = 0; j < L; ++j) {
            long long k0 = (od_row(R, b, j) * G + g) * d_h;
            double s = 0.0;
            for (i = 0; i < d_h; ++i) s += qh[i] * od_load(K, k0 + i, cache_bf16);
            z[j] = scale * s;
        }
        softmax_sum(z, L, R, b, V, cache_bf16, (long long)G * d_h, (long long)g * d_h, d_h,
                    out + bh * d_h, lse + bh);
        free(z);
    }
}

/* ------------------------------------------------------------------------- */
/* Cache append  ([S]: the positional key is cached already rotated;           */
/*                [K] §1: the current token is appended, then attended)        */
/* ------------------------------------------------------------------------- */
/* Writes token b at logical position pos[b]:
 *   V[row]      = v_new[b]                    (one rounding to the cache dtype)
 *   K_rope[row] = Rot(pos[b]) k_new[b]
 * The stored code of the rotated key is decided in fp32, in this fixed order,
 * with no fused multiply-add (the file is built with -ffp-contract=off):
 *   y0 = (x0*c) - (x1*s),  y1 = (x0*s) + (x1*c),  c/s from od_rope_table_f32,
 * then one RNE rounding to bf16 (cache_bf16 != 0) or kept as fp32.
 * V and K_rope are uint16 arrays (bf16 bits) when cache_bf16, else float. */
void od_append(int B, int G, int d_h, int d_r, const float *v_new, const float *k_new,
               const long long *pos, const od_rows *R, int cache_bf16,
               void *V, void *Kr, const float *rope_tab)
{
    int b, e, i;
    for (b = 0; b < B; ++b) {
        long long p = pos[b];
        long long row = od_row(R, b, p);
        for (e = 0; e < G * d_h; ++e) {
            float x = v_new[(long long)b * G * d_h + e];
            if (cache_bf16) ((uint16_t *)V)[row * G * d_h + e] = od_bf16_rne(x);
            else ((float *)V)[row * G * d_h + e] = x;
        }
        for (i = 0; i < d_r / 2; ++i) {
            float x0 = k_new[(long long)b * d_r + 2 * i];
            float x1 = k_new[(long long)b * d_r + 2 * i + 1];
            float c = rope_tab[(p * (d_r / 2) + i) * 2 + 0];
            float s = rope_tab[(p * (d_r / 2) + i) * 2 + 1];
            float a = x0 * c, bb = x1 * s, cc = x0 * s, d = x1 * c;
            float y0 = a - bb, y1 = cc + d;
            if (cache_bf16) {
                ((uint16_t *)Kr)[row * d_r + 2 * i] = od_bf16_rne(y0);
                ((uint16_t *)Kr)[row * d_r + 2 * i + 1] = od_bf16_rne(y1);
            } else {
                ((float *)Kr)[row * d_r + 2 * i] = y0;
                ((float *)Kr)[row * d_r + 2 * i + 1] = y1;
            }
        }
    }
}

/* The same rotation in fp64 (no intermediate fp32 rounding): out[b][d_r]. */
void od_rotate_keys_f64(int B, int d_r, const double *k_new, const long long *pos,
                        double base, double *out)
{
    int b;
    for (b = 0; b < B; ++b) od_rotate(k_new + (long long)b * d_r, out + (long long)b * d_r, d_r, pos[b], base);
}
