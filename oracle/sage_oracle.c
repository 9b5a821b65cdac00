/*
 * sage_oracle.c -- plain, slow CPU oracle for INT8-QK quantized attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * Every function follows one passage of the source pages (cited by page
 * title and section):
 *   [P1] "INT8 QK MMAC on gfx936 DCU: paged access, fragment mapping and
 *        GQA" (forum.sourcefind.cn), sections 1-7.
 *   [P3] "SageAttention -- MetaX MXMACA port" README (gitlink.org.cn),
 *        sections "feature matrix", "quant kernel", "advanced config".
 *
 * Precision: the quantisation decision is taken in IEEE fp32 (each op
 * correctly rounded, no FMA contraction: build with -ffp-contract=off);
 * integer dot products in int64; scores, softmax, P.V and LSE in fp64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Symmetric dynamic INT8 quantisation.                                */
/* [P1] section 4: sQ = max(abs(Q)) / 127, Qq = round(Q / sQ).          */
/* [P3] quant kernel table: groups are one token row (per token) or a   */
/* block of consecutive tokens (per block, 128 for Q and 64 for K).     */
/* Readings: the quotient is fp32 x / fp32 s (correctly rounded), then  */
/* rounded to the nearest integer with ties to even; a group whose      */
/* amax is 0 gets s = 0 and all codes 0; codes are clamped to           */
/* [-127, 127] (the clamp never binds except for rounding noise).       */
/* ------------------------------------------------------------------ */

static int8_t quant_one(float x, float s)
{
    if (s == 0.0f)
        return 0;
    float r = x / s;          /* fp32, correctly rounded */
    float n = nearbyintf(r);  /* default rounding mode: nearest, ties to even */
    if (n > 127.0f) n = 127.0f;
    if (n < -127.0f) n = -127.0f;
    return (int8_t)n;
}

/*
 * x      : fp32 [BH][S][D] (token rows of BH independent sequences)
 * gtok   : tokens per quantisation group (1 = per token)
 * mu     : optional fp32 [BH][D]; when given, x is first replaced by
 *          fl32(x - mu[c]) (smooth_k, [P3] feature matrix "K smoothing")
 * q      : int8 [BH][S][D]
 * scale  : fp32 [BH][ceil(S/gtok)]
 */
void oracle_quant_int8(const float *x, int64_t BH, int64_t S, int D, int gtok,
                       const float *mu, int8_t *q, float *scale)
{
    int64_t ngroups = (S + gtok - 1) / gtok;
    for (int64_t bh = 0; bh < BH; ++bh) {
        for (int64_t g = 0; g < ngroups; ++g) {
            int64_t t0 = g * gtok;
            int64_t t1 = t0 + gtok < S ? t0 + gtok : S;
            float amax = 0.0f;
            for (int64_t t = t0; t < t1; ++t) {
                for (int c = 0; c < D; ++c) {
                    float v = x[(bh * S + t) * D + c];
                    if (mu) v = v - mu[bh * D + c];
                    float a = fabsf(v);
                    if (a > amax) amax = a;
                }
            }
            float s = amax / 127.0f;
            scale[bh * ngroups + g] = s;
            for (int64_t t = t0; t < t1; ++t) {
                for (int c = 0; c < D; ++c) {
                    float v = x[(bh * S + t) * D + c];
                    if (mu) v = v - mu[bh * D + c];
                    q[(bh * S + t) * D + c] = quant_one(v, s);
                }
            }
        }
    }
}

/*
 * smooth_k mean ([P3] feature matrix "K smoothing (with LSE correction)";
 * [P3] advanced config: smooth_k removes the per-channel K mean).
 * mu[bh][c] = fl32( (sum over t of x[bh][t][c], fp64, token order) / S ).
 */
void oracle_token_mean(const float *x, int64_t BH, int64_t S, int D, float *mu)
{
    for (int64_t bh = 0; bh < BH; ++bh) {
        for (int c = 0; c < D; ++c) {
            double acc = 0.0;
            for (int64_t t = 0; t < S; ++t)
                acc += (double)x[(bh * S + t) * D + c];
            mu[bh * D + c] = (float)(acc / (double)S);
        }
    }
}

/*
 * Row bias b_i = sum_c x_ic * mu_c (fp64): the amount the smoothed
 * scores Q.(K - mu)^T fall short of Q.K^T; adding it back restores the
 * un-smoothed score (the "LSE correction" of [P3]).
 * x: fp32 [B][H][S][D]; mu: fp32 [B][Hmu][D]; head h uses mu head
 * h / (H / Hmu).  bias: fp64 [B][H][S].
 */
void oracle_row_bias(const float *x, int64_t B, int64_t H, int64_t S, int D,
                     const float *mu, int64_t Hmu, double *bias)
{
    int64_t group = H / Hmu;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t t = 0; t < S; ++t) {
                const float *row = x + ((b * H + h) * S + t) * D;
                const float *m = mu + (b * Hmu + h / group) * D;
                double acc = 0.0;
                for (int c = 0; c < D; ++c)
                    acc += (double)row[c] * (double)m[c];
                bias[(b * H + h) * S + t] = acc;
            }
}

/*
 * Raw INT8 scores ([P1] sections 1 and 2.1): acc_ij = sum_c q_ic k_jc,
 * accumulated exactly (int64 here), stored as int32.  Returns the
 * number of entries whose magnitude exceeds D * 127 * 127 (the bound
 * stated in [P1] 2.1); 0 for valid int8 codes in [-127, 127].
 */
int64_t oracle_qk_int32(const int8_t *q, int64_t Sq, const int8_t *k, int64_t Sk,
                        int D, int32_t *acc)
{
    int64_t bound = (int64_t)D * 127 * 127, bad = 0;
    for (int64_t i = 0; i < Sq; ++i)
        for (int64_t j = 0; j < Sk; ++j) {
            int64_t a = 0;
            for (int c = 0; c < D; ++c)
                a += (int64_t)q[i * D + c] * (int64_t)k[j * D + c];
            if (a > bound || a < -bound) ++bad;
            acc[i * Sk + j] = (int32_t)a;
        }
    return bad;
}

/*
 * Attention of nq query rows against one key set ([P1] section 1;
 * [P3] pipeline steps 3-8).
 *
 *   acc_ij = sum_c q_ic k_jc                              (exact integer)
 *   z_ij   = sm_scale * (acc_ij * sq_i * sk_j + [smoothed_j] * qbias_i)
 *   key j is visible to row i unless causal and j > qpos_i + causal_offset
 *   P_ij   = exp(z_ij) / sum_visible exp(z_ij)            (fp64)
 *   o_i    = sum_j P_ij v_j ;  lse_i = ln sum_visible exp(z_ij)
 *
 * The pages apply sm_scale*log2(e) and use base-2 exponentials; in exact
 * arithmetic that is the same softmax, so the oracle uses base e.
 * A row with no visible key gets o = 0 and lse = -inf.
 *
 * q: int8 [nq][D], sq: fp32 [nq], qbias: fp64 [nq] or NULL,
 * qpos: int64 [nq] or NULL (only read when causal),
 * k: int8 [nk][D], sk: fp32 [nk], smoothed: uint8 [nk] or NULL,
 * v: fp64 [nk][D] (values as the PV step sees them, already dequantised),
 * o: fp64 [nq][D], lse: fp64 [nq].
 * Returns the number of raw scores outside the INT32 bound of [P1] 2.1.
 */
int64_t oracle_attend(int64_t nq, int D, const int8_t *q, const float *sq,
                      const double *qbias, const int64_t *qpos, int64_t nk,
                      const int8_t *k, const float *sk, const uint8_t *smoothed,
                      const double *v, int causal, int64_t causal_offset,
                      double sm_scale, double *o, double *lse)
{
    int64_t bound = (int64_t)D * 127 * 127, bad = 0;
    double *z = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    for (int64_t i = 0; i < nq; ++i) {
        int64_t last = nk - 1;
        if (causal) {
            int64_t lim = qpos[i] + causal_offset;
            if (lim < last) last = lim;
        }
        double *oi = o + i * D;
        for (int c = 0; c < D; ++c) oi[c] = 0.0;
        if (last < 0) {
            lse[i] = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j <= last; ++j) {
            int64_t a = 0;
            for (int c = 0; c < D; ++c)
                a += (int64_t)q[i * D + c] * (int64_t)k[j * D + c];
            if (a > bound || a < -bound) ++bad;
            double s = (double)a * (double)sq[i] * (double)sk[j];
            if (smoothed && smoothed[j] && qbias) s += qbias[i];
            z[j] = sm_scale * s;
            if (z[j] > m) m = z[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j <= last; ++j) {
            double p = exp(z[j] - m);
            l += p;
            const double *vj = v + j * D;
            for (int c = 0; c < D; ++c) oi[c] += p * vj[c];
        }
        for (int c = 0; c < D; ++c) oi[c] /= l;
        lse[i] = m + log(l);
    }
    free(z);
    return bad;
}

/*
 * Attention with INT8 P.V (decode over INT8 values; [P1] sections 6 and 8
 * name INT8 P.V with "V scale fusion" and "probability quantization").
 * The V scale is folded into the probabilities, the product is quantised
 * symmetrically per group of `block` consecutive keys (one 16-token cache
 * page; the last group may be short), and the INT8 codes multiply the INT8
 * values exactly:
 *   z_j  = sm_scale * acc_j * sq_i * sk_j,  M = max_j z_j
 *   p_j  = exp(z_j - M),  l = sum_j p_j   (unquantised: the denominator)
 *   w_j  = p_j * sv_j
 *   s_g  = max_{j in g} w_j / 127,  code_j = rne(w_j / s_g)  (0 if s_g = 0)
 *   o    = (sum_g s_g * sum_{j in g} code_j * v_j) / l,  lse = M + ln l
 * Readings (the algorithm's own text is not on the pages): one scale per
 * (query row, key group) -- a common factor of a group's w cancels in its
 * codes, so the codes do not depend on which row maximum the softmax uses --
 * codes in [0, 127] (w >= 0), ties to even as for Q and K.  The code
 * decision is taken here in fp64 from the exact probabilities.
 * v: int8 [nk][D] codes, sv: fp32 [nk] per-token scales.
 */
int64_t oracle_attend_pv_int8(int64_t nq, int D, const int8_t *q, const float *sq, int64_t nk,
                              const int8_t *k, const float *sk, const int8_t *v, const float *sv,
                              int block, double sm_scale, double *o, double *lse)
{
    int64_t bound = (int64_t)D * 127 * 127, bad = 0;
    double *z = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    double *w = (double *)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    for (int64_t i = 0; i < nq; ++i) {
        double *oi = o + i * D;
        for (int c = 0; c < D; ++c) oi[c] = 0.0;
        if (nk == 0) {
            lse[i] = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < nk; ++j) {
            int64_t a = 0;
            for (int c = 0; c < D; ++c)
                a += (int64_t)q[i * D + c] * (int64_t)k[j * D + c];
            if (a > bound || a < -bound) ++bad;
            z[j] = sm_scale * ((double)a * (double)sq[i] * (double)sk[j]);
            if (z[j] > m) m = z[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
            double p = exp(z[j] - m);
            l += p;
            w[j] = p * (double)sv[j];
        }
        for (int64_t g0 = 0; g0 < nk; g0 += block) {
            int64_t g1 = g0 + block < nk ? g0 + block : nk;
            double wmax = 0.0;
            for (int64_t j = g0; j < g1; ++j)
                if (w[j] > wmax) wmax = w[j];
            if (wmax == 0.0) continue;
            double s = wmax / 127.0;
            for (int64_t j = g0; j < g1; ++j) {
                double code = nearbyint(w[j] / s);   /* ties to even */
                if (code > 127.0) code = 127.0;
                const int8_t *vj = v + j * D;
                for (int c = 0; c < D; ++c) oi[c] += s * code * (double)vj[c];
            }
        }
        for (int c = 0; c < D; ++c) oi[c] /= l;
        lse[i] = m + log(l);
    }
    free(z);
    free(w);
    return bad;
}

/*
 * Split-K combine of segment partials (segments are the split-K pieces
 * of [P1] section 4; the pages return the LSE "for concatenation" in
 * [P3] advanced config).  For each row r with S segments:
 *   L = M + ln sum_s exp(lse_s - M),  M = max_s lse_s
 *   o = sum_s exp(lse_s - L) * o_s
 * Segments with lse = -inf carry no keys and are skipped; a row whose
 * segments are all empty gets o = 0, L = -inf.
 * opart: fp64 [R][S][D], lpart: fp64 [R][S], o: fp64 [R][D], lse: [R].
 */
void oracle_splitk_combine(const double *opart, const double *lpart, int64_t R,
                           int64_t S, int D, double *o, double *lse)
{
    for (int64_t r = 0; r < R; ++r) {
        double M = -INFINITY;
        for (int64_t s = 0; s < S; ++s)
            if (lpart[r * S + s] > M) M = lpart[r * S + s];
        double *orow = o + r * D;
        for (int c = 0; c < D; ++c) orow[c] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int64_t s = 0; s < S; ++s)
            if (lpart[r * S + s] != -INFINITY) sum += exp(lpart[r * S + s] - M);
        double L = M + log(sum);
        for (int64_t s = 0; s < S; ++s) {
            double ls = lpart[r * S + s];
            if (ls == -INFINITY) continue;
            double w = exp(ls - L);
            const double *os = opart + (r * S + s) * D;
            for (int c = 0; c < D; ++c) orow[c] += w * os[c];
        }
        lse[r] = L;
    }
}

/* ------------------------------------------------------------------ */
/* KV producer: quantise new key/value rows and write them into the   */
/* paged INT8 cache.                                                   */
/* [P1] section 4: K and V are quantised per token and per KV head     */
/* (s = max|x| / 127 over the row's D channels, codes round(x / s));   */
/* [P1] section 3: token t of sequence b lives in page                 */
/* block_table[b][t / 16], slot t % 16, channel c at                   */
/* [page][kv_head][c / 16][slot][c % 16]; its scale at                  */
/* [page][kv_head][slot].                                              */
/* x: [B][H][n][D] fp32 (the new rows); pos[b]: position of row 0 of   */
/* sequence b.  Returns the number of rows skipped because their page  */
/* index was outside [0, num_blocks).                                  */
/* ------------------------------------------------------------------ */

int64_t oracle_kv_append(const float *x, int64_t B, int64_t H, int64_t n, int D,
                         const int32_t *block_table, int64_t max_blocks, const int32_t *pos,
                         int64_t num_blocks, int8_t *cache, float *scale)
{
    int64_t skipped = 0;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t t = 0; t < n; ++t) {
                const float *row = x + ((b * H + h) * n + t) * D;
                const int64_t p = (int64_t)pos[b] + t;
                const int64_t blk = block_table[b * max_blocks + p / 16];
                const int64_t slot = p % 16;
                if (blk < 0 || blk >= num_blocks) {
                    ++skipped;
                    continue;
                }
                float amax = 0.0f;
                for (int c = 0; c < D; ++c) {
                    const float a = fabsf(row[c]);
                    if (a > amax)
                        amax = a;
                }
                const float s = amax / 127.0f;
                int8_t *page = cache + (blk * H + h) * (int64_t)D * 16;
                for (int c = 0; c < D; ++c)
                    page[(c / 16) * 256 + slot * 16 + (c % 16)] = quant_one(row[c], s);
                scale[(blk * H + h) * 16 + slot] = s;
            }
    return skipped;
}
