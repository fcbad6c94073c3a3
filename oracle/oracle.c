/*
 * Oracle for the DeepSeek sparse-attention (DSA) hot path: a plain, slow,
 * obviously correct CPU restatement of what the path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check of
 * __graft_entry__ and the cpu_baseline leg of bench.py may load this
 * library.  It shares no code, header, table or constant with the CUDA
 * library under sparse_latent_attention_indexer_gb300/csrc, and the product
 * path never calls it.
 *
 * Conventions
 *   - Inputs arrive as float32 arrays.  Every bf16, fp32 and dequantised
 *     e4m3 value of the workloads is exactly representable in float32, so
 *     the oracle sees the exact input values.  All arithmetic is done in
 *     double precision; nothing is rounded on the way.
 *   - One call handles rows of ONE sequence.  A "row" is a query token; its
 *     absolute position p (start_pos + t) is passed per row in `pos`.
 *     Keys are numbered 0..S-1 within the sequence.
 *   - Loops are plain: no blocking, no reassociation beyond the order the
 *     definitions give.  OpenMP only distributes independent rows.
 *
 * Sources (page title, section / equation):
 *   [P3] "DeepSeek-V3.2-Exp" atlas page, MoE transformer block, "All 43
 *        steps": the sparse latent attention equations (q^C, k^C = c^KV W_UK,
 *        K_i = [K^C_i; k^R], v = c^KV W_UV, the indexer score S^I_{t,s},
 *        S~^I = S^I + M, and the selection mask M^sel with top_2048).
 *   [P1] "nnterp encyclopedia: deepseek_v32", The Notes: "Up to 2048 tokens
 *        the sparse attention is plain causal attention" (unselected keys
 *        take the dtype minimum before the softmax; probabilities are zero
 *        outside the selection and sum to one over it; the selection is
 *        int32 key indices [batch, query, min(index_topk, seq)]), and
 *        "Latent attention: every head's key comes from one latent".
 *   [P4] "DeepSeek-V3.2-Exp - Block input", config_671B_v3.2.json excerpt:
 *        dtype fp8, scale_fmt ue8m0, index_n_heads 64, index_head_dim 128,
 *        index_topk 2048.
 *   [P5] "DeepSeek-V3.2-Exp - Attention input", mla-init excerpt: the
 *        softmax scale qk_head_dim^-0.5 (times mscale^2 under YaRN).
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ------------------------------------------------------------------------
 * 1. Lightning-indexer score with the causal mask  [P3, equations S^I and
 *    S~^I = S^I + M].
 *
 *    S^I_{t,s} = 1/(sqrt(H_I) sqrt(D_I)) * sum_h w_{t,h} ReLU(q^I_{h,t} . k^I_s)
 *
 *    The page prints the constant for H_I = 64, D_I = 128 as
 *    1/(sqrt(64) sqrt(128)); other head shapes use sqrt(H_I) sqrt(D_I).
 *    M_{t,s} = 0 for s <= p and -inf for s > p (causal).
 *
 *    qI   [nrows, H_I, D_I]   indexer queries of the rows
 *    w    [nrows, H_I]        per-head weights of the rows
 *    kI   [S, D_I]            indexer keys of the sequence
 *    pos  [nrows]             absolute position p of each row
 *    scores  [nrows, S]       out: S~^I (finite for s <= p, -inf after)
 *    absterm [nrows, S]       out (may be NULL): the same sum with |w|, i.e.
 *                             1/(sqrt(H_I) sqrt(D_I)) sum_h |w| ReLU(q.k),
 *                             used by the tests to size rounding bands.
 * ---------------------------------------------------------------------- */
ORACLE_API void oracle_indexer_scores(const float *qI, const float *w, const float *kI,
                                      const int64_t *pos, int64_t nrows, int64_t S,
                                      int H_I, int D_I, double *scores, double *absterm)
{
    const double c = 1.0 / (sqrt((double)H_I) * sqrt((double)D_I));
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        for (int64_t s = 0; s < S; ++s) {
            double *out = &scores[r * S + s];
            if (s > pos[r]) {
                *out = -INFINITY;
                if (absterm) absterm[r * S + s] = 0.0;
                continue;
            }
            double sum = 0.0, abssum = 0.0;
            for (int h = 0; h < H_I; ++h) {
                double dot = 0.0;
                for (int d = 0; d < D_I; ++d)
                    dot += (double)qI[(r * H_I + h) * D_I + d] * (double)kI[s * D_I + d];
                double relu = dot > 0.0 ? dot : 0.0;
                double wh = (double)w[r * H_I + h];
                sum += wh * relu;
                abssum += fabs(wh) * relu;
            }
            *out = c * sum;
            if (absterm) absterm[r * S + s] = c * abssum;
        }
    }
}

/* ------------------------------------------------------------------------
 * 2. Top-k selection  [P3, M^sel_{t,s} = M_{t,s} if s in top_k(S~^I_t)].
 *
 *    Only causal keys (s <= p) can be selected with a finite mask, so the
 *    row keeps n = min(k, p + 1) keys: the n causal keys with the largest
 *    score.  Equal scores are ordered by the lower key index first (the
 *    pages fix no tie rule; any consistent rule gives a valid selection).
 *    The row is padded with -1 up to k entries.  The selection lists keys
 *    in decreasing score order.
 * ---------------------------------------------------------------------- */
typedef struct {
    double score;
    int64_t key;
} scored_key;

static int cmp_scored_key_desc(const void *a, const void *b)
{
    const scored_key *x = (const scored_key *)a, *y = (const scored_key *)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->key > y->key) - (x->key < y->key);
}

ORACLE_API void oracle_topk(const double *scores, const int64_t *pos, int64_t nrows,
                            int64_t S, int k, int32_t *idx)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t last = pos[r] < S - 1 ? pos[r] : S - 1; /* last causal key */
        int64_t ncausal = last + 1;
        scored_key *buf = (scored_key *)malloc((size_t)(ncausal > 0 ? ncausal : 1) * sizeof(scored_key));
        for (int64_t s = 0; s < ncausal; ++s) {
            buf[s].score = scores[r * S + s];
            buf[s].key = s;
        }
        qsort(buf, (size_t)ncausal, sizeof(scored_key), cmp_scored_key_desc);
        int64_t n = ncausal < k ? ncausal : k;
        for (int64_t j = 0; j < k; ++j)
            idx[r * k + j] = j < n ? (int32_t)buf[j].key : -1;
        free(buf);
    }
}

/* ------------------------------------------------------------------------
 * 3. Key/value up-projection of the latent  [P3, k^C = c^KV W_UK,
 *    v = c^KV W_UV; P1, "every head's key comes from one latent"].
 *
 *    Weight layouts (the halves of wkv_b, per head):
 *      W_UK [H, d_n, d_c]:  K^C[s,h,d] = sum_c W_UK[h,d,c] * c[s,c]
 *      W_UV [H, d_c, d_v]:  V[s,h,e]   = sum_c c[s,c] * W_UV[h,c,e]
 *    ckv rows have stride ld_ckv (a packed [S, d_c + d_r] cache is allowed).
 * ---------------------------------------------------------------------- */
ORACLE_API void oracle_kv_up(const float *ckv, int64_t S, int64_t ld_ckv,
                             const float *W_UK, const float *W_UV,
                             int H, int d_n, int d_c, int d_v, double *KC, double *V)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t s = 0; s < S; ++s) {
        const float *c = ckv + s * ld_ckv;
        for (int h = 0; h < H; ++h) {
            for (int d = 0; d < d_n; ++d) {
                double acc = 0.0;
                for (int j = 0; j < d_c; ++j)
                    acc += (double)W_UK[((int64_t)h * d_n + d) * d_c + j] * (double)c[j];
                KC[(s * H + h) * d_n + d] = acc;
            }
            for (int e = 0; e < d_v; ++e) {
                double acc = 0.0;
                for (int j = 0; j < d_c; ++j)
                    acc += (double)c[j] * (double)W_UV[((int64_t)h * d_c + j) * d_v + e];
                V[(s * H + h) * d_v + e] = acc;
            }
        }
    }
}

/* A selected index takes part in the attention when it names a key of the
 * sequence that is causal for the row (0 <= s <= p, s < S).  Entries -1 and
 * out-of-window entries behave as masked (M^sel = -inf). */
static int selected_key_is_live(int32_t s, int64_t p, int64_t S)
{
    return s >= 0 && (int64_t)s < S && (int64_t)s <= p;
}

/* ------------------------------------------------------------------------
 * 4. Sparse latent attention, unabsorbed form  [P3: Q = [Q^C; Q^R],
 *    K_i = [K^C_i; k^R], V; M^sel; P1: softmax over the selection].
 *
 *    For row t and head h, over the live selected keys s:
 *      z[h,s]   = scale * (q_nope[t,h] . K^C[s,h] + q_pe[t,h] . k_pe[s])
 *      P[h,s]   = exp(z - max) / sum exp(z - max)        (two passes)
 *      out[t,h] = sum_s P[h,s] V[s,h]
 *      lse[t,h] = max + log(sum exp(z - max))
 *    A row with no live key gives out = 0 and lse = -inf.
 *
 *    q_nope [nrows,H,d_n], q_pe [nrows,H,d_r], KC [S,H,d_n] and V [S,H,d_v]
 *    from oracle_kv_up, k_pe rows with stride ld_kpe, idx [nrows,k].
 * ---------------------------------------------------------------------- */
ORACLE_API void oracle_sparse_mla_unabsorbed(const float *q_nope, const float *q_pe,
                                             const double *KC, const float *kpe, int64_t ld_kpe,
                                             const double *V, const int32_t *idx,
                                             const int64_t *pos, int64_t nrows, int k, int64_t S,
                                             int H, int d_n, int d_r, int d_v, double scale,
                                             double *out, double *lse)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        double *z = (double *)malloc((size_t)k * sizeof(double));
        for (int h = 0; h < H; ++h) {
            const float *qn = q_nope + (r * H + h) * d_n;
            const float *qr = q_pe + (r * H + h) * d_r;
            double zmax = -INFINITY;
            for (int j = 0; j < k; ++j) {
                int32_t s = idx[r * k + j];
                if (!selected_key_is_live(s, pos[r], S)) {
                    z[j] = -INFINITY;
                    continue;
                }
                double dot = 0.0;
                for (int d = 0; d < d_n; ++d)
                    dot += (double)qn[d] * KC[((int64_t)s * H + h) * d_n + d];
                for (int d = 0; d < d_r; ++d)
                    dot += (double)qr[d] * (double)kpe[(int64_t)s * ld_kpe + d];
                z[j] = scale * dot;
                if (z[j] > zmax) zmax = z[j];
            }
            double *o = out + (r * H + h) * d_v;
            for (int e = 0; e < d_v; ++e) o[e] = 0.0;
            if (zmax == -INFINITY) {
                if (lse) lse[r * H + h] = -INFINITY;
                continue;
            }
            double sum = 0.0;
            for (int j = 0; j < k; ++j)
                if (z[j] != -INFINITY) sum += exp(z[j] - zmax);
            for (int j = 0; j < k; ++j) {
                if (z[j] == -INFINITY) continue;
                double p = exp(z[j] - zmax) / sum;
                int32_t s = idx[r * k + j];
                for (int e = 0; e < d_v; ++e) o[e] += p * V[((int64_t)s * H + h) * d_v + e];
            }
            if (lse) lse[r * H + h] = zmax + log(sum);
        }
        free(z);
    }
}

/* ------------------------------------------------------------------------
 * 5. Sparse latent attention, absorbed form.  The same quantity as (4),
 *    regrouped by associativity of the products in [P3]:
 *      q~[t,h,c]  = sum_d q_nope[t,h,d] W_UK[h,d,c]      (so q~ . c[s] = q^C . K^C[s])
 *      z[h,s]     = scale * (q~[t,h] . c[s] + q_pe[t,h] . k_pe[s])
 *      o_lat[t,h] = sum_s P[h,s] c[s]                    (latent context)
 *      out[t,h,e] = sum_c o_lat[t,h,c] W_UV[h,c,e]
 *    Optional outputs: qt [nrows,H,d_c] (q~) and olat [nrows,H,d_c].
 * ---------------------------------------------------------------------- */
ORACLE_API void oracle_sparse_mla_absorbed(const float *q_nope, const float *q_pe,
                                           const float *ckv, int64_t ld_ckv,
                                           const float *kpe, int64_t ld_kpe,
                                           const float *W_UK, const float *W_UV,
                                           const int32_t *idx, const int64_t *pos,
                                           int64_t nrows, int k, int64_t S,
                                           int H, int d_n, int d_r, int d_c, int d_v,
                                           double scale, double *out, double *lse,
                                           double *qt_out, double *olat_out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        double *z = (double *)malloc((size_t)k * sizeof(double));
        double *qt = (double *)malloc((size_t)d_c * sizeof(double));
        double *ol = (double *)malloc((size_t)d_c * sizeof(double));
        for (int h = 0; h < H; ++h) {
            const float *qn = q_nope + (r * H + h) * d_n;
            const float *qr = q_pe + (r * H + h) * d_r;
            for (int j = 0; j < d_c; ++j) {
                double acc = 0.0;
                for (int d = 0; d < d_n; ++d)
                    acc += (double)qn[d] * (double)W_UK[((int64_t)h * d_n + d) * d_c + j];
                qt[j] = acc;
            }
            if (qt_out)
                for (int j = 0; j < d_c; ++j) qt_out[(r * H + h) * d_c + j] = qt[j];
            double zmax = -INFINITY;
            for (int j = 0; j < k; ++j) {
                int32_t s = idx[r * k + j];
                if (!selected_key_is_live(s, pos[r], S)) {
                    z[j] = -INFINITY;
                    continue;
                }
                double dot = 0.0;
                for (int c = 0; c < d_c; ++c) dot += qt[c] * (double)ckv[(int64_t)s * ld_ckv + c];
                for (int d = 0; d < d_r; ++d) dot += (double)qr[d] * (double)kpe[(int64_t)s * ld_kpe + d];
                z[j] = scale * dot;
                if (z[j] > zmax) zmax = z[j];
            }
            for (int c = 0; c < d_c; ++c) ol[c] = 0.0;
            double sum = 0.0;
            if (zmax != -INFINITY) {
                for (int j = 0; j < k; ++j)
                    if (z[j] != -INFINITY) sum += exp(z[j] - zmax);
                for (int j = 0; j < k; ++j) {
                    if (z[j] == -INFINITY) continue;
                    double p = exp(z[j] - zmax) / sum;
                    int32_t s = idx[r * k + j];
                    for (int c = 0; c < d_c; ++c) ol[c] += p * (double)ckv[(int64_t)s * ld_ckv + c];
                }
            }
            if (olat_out)
                for (int c = 0; c < d_c; ++c) olat_out[(r * H + h) * d_c + c] = ol[c];
            double *o = out + (r * H + h) * d_v;
            for (int e = 0; e < d_v; ++e) {
                double acc = 0.0;
                for (int c = 0; c < d_c; ++c) acc += ol[c] * (double)W_UV[((int64_t)h * d_c + c) * d_v + e];
                o[e] = acc;
            }
            if (lse) lse[r * H + h] = zmax == -INFINITY ? -INFINITY : zmax + log(sum);
        }
        free(z);
        free(qt);
        free(ol);
    }
}

/* ------------------------------------------------------------------------
 * 6. Dense masked latent attention, written literally from [P3] and [P1]:
 *    the scores of EVERY key s in [0, S) are formed, the mask
 *      M_{t,s}      = 0 if s <= p else -inf                 (causal)
 *      M^sel_{t,s}  = M_{t,s} if sel[t,s] else -inf         (selection)
 *    is added, and a softmax over all S keys is taken (exp(-inf) = 0).
 *    With sel == NULL the selection holds every key, which is the plain
 *    causal attention that the pages state the sparse attention equals
 *    while the sequence is no longer than index_topk.
 *    sel [nrows, S] bytes (1 = selected), may be NULL.
 * ---------------------------------------------------------------------- */
ORACLE_API void oracle_dense_masked_mla(const float *q_nope, const float *q_pe,
                                        const double *KC, const float *kpe, int64_t ld_kpe,
                                        const double *V, const uint8_t *sel,
                                        const int64_t *pos, int64_t nrows, int64_t S,
                                        int H, int d_n, int d_r, int d_v, double scale,
                                        double *out, double *lse)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nrows; ++r) {
        double *z = (double *)malloc((size_t)(S > 0 ? S : 1) * sizeof(double));
        for (int h = 0; h < H; ++h) {
            const float *qn = q_nope + (r * H + h) * d_n;
            const float *qr = q_pe + (r * H + h) * d_r;
            double zmax = -INFINITY;
            for (int64_t s = 0; s < S; ++s) {
                double dot = 0.0;
                for (int d = 0; d < d_n; ++d) dot += (double)qn[d] * KC[(s * H + h) * d_n + d];
                for (int d = 0; d < d_r; ++d) dot += (double)qr[d] * (double)kpe[s * ld_kpe + d];
                double m = s <= pos[r] ? 0.0 : -INFINITY;
                double msel = (sel == NULL || sel[r * S + s]) ? m : -INFINITY;
                z[s] = scale * dot + msel;
                if (z[s] > zmax) zmax = z[s];
            }
            double *o = out + (r * H + h) * d_v;
            for (int e = 0; e < d_v; ++e) o[e] = 0.0;
            if (zmax == -INFINITY) {
                if (lse) lse[r * H + h] = -INFINITY;
                continue;
            }
            double sum = 0.0;
            for (int64_t s = 0; s < S; ++s) sum += exp(z[s] - zmax);
            for (int64_t s = 0; s < S; ++s) {
                double p = exp(z[s] - zmax) / sum;
                if (p == 0.0) continue;
                for (int e = 0; e < d_v; ++e) o[e] += p * V[(s * H + h) * d_v + e];
            }
            if (lse) lse[r * H + h] = zmax + log(sum);
        }
        free(z);
    }
}

/* ------------------------------------------------------------------------
 * 7. FP8 e4m3 with power-of-two (ue8m0) block scales  [P4: dtype fp8,
 *    scale_fmt ue8m0].
 *
 *    e4m3 (the OCP "E4M3FN" format): 1 sign, 4 exponent bits with bias 7,
 *    3 mantissa bits, no infinities, S.1111.111 is NaN.  Normal codes
 *    (exponent field E = 1..15) are (1 + m/8) 2^(E-7); subnormal codes
 *    (E = 0) are (m/8) 2^-6.  The largest finite value is 448.
 *
 *    Block recipe (the pages give only "ue8m0"; this is the reading used):
 *    a block is 128 consecutive values.  Its scale is 2^e with e the
 *    smallest integer such that amax <= 448 * 2^e, clamped to the ue8m0
 *    exponent range [-127, 127]; amax = 0 gives e = 0.  Each value is
 *    divided by 2^e (exact) and rounded to the nearest e4m3 value, ties to
 *    the code with an even mantissa, saturating to +-448.
 * ---------------------------------------------------------------------- */
ORACLE_API double oracle_e4m3_value(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int E = (code >> 3) & 15;
    int m = code & 7;
    if (E == 15 && m == 7) return NAN;
    double mag = E == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, E - 7);
    return sign ? -mag : mag;
}

/* Nearest e4m3 code by exhaustive search over the 127 finite magnitudes. */
static uint8_t e4m3_encode_rne_satfinite(double v)
{
    int neg = v < 0.0 || (v == 0.0 && signbit(v));
    double a = fabs(v);
    uint8_t best = 0;
    double best_err = INFINITY;
    for (int code = 0; code <= 0x7E; ++code) {
        double err = fabs(oracle_e4m3_value((uint8_t)code) - a);
        if (err < best_err || (err == best_err && (code & 1) == 0)) {
            best = (uint8_t)code;
            best_err = err;
        }
    }
    /* above the top the nearest finite code is 448: that is the saturation */
    return (uint8_t)(best | (neg ? 0x80 : 0));
}

ORACLE_API void oracle_quant_e4m3_ue8m0(const float *x, int64_t n_blocks, uint8_t *codes,
                                        int32_t *exps)
{
#pragma omp parallel for schedule(static)
    for (int64_t b = 0; b < n_blocks; ++b) {
        const float *blk = x + b * 128;
        double amax = 0.0;
        for (int i = 0; i < 128; ++i)
            if (fabs((double)blk[i]) > amax) amax = fabs((double)blk[i]);
        int e = 0;
        if (amax > 0.0) {
            e = -127;
            while (e < 127 && amax > 448.0 * ldexp(1.0, e)) ++e;
        }
        exps[b] = e;
        for (int i = 0; i < 128; ++i)
            codes[b * 128 + i] = e4m3_encode_rne_satfinite(ldexp((double)blk[i], -e));
    }
}

/* ------------------------------------------------------------------------
 * 8. The projections on either side of the path.
 *
 *    Before it [P5 mla-init and mla-kv excerpts; P4 RMSNorm excerpt; P1
 *    printout of DeepseekV32Attention and its indexer]:
 *        kv      = wkv_a(x)                      (dim -> kv_lora_rank + rope)
 *        kv, k_pe = split(kv, [kv_lora_rank, qk_rope_head_dim])
 *        kv      = kv_norm(kv)                   (RMSNorm, gain, eps 1e-6, float32 compute)
 *        k_pe    = rotary(k_pe, freqs_cis)       (served de-interleaved)
 *        k^I     = k_norm(wk(x))                 (LayerNorm(128), gain and bias, eps 1e-6)
 *        w       = weights_proj(x)               (dim -> 64 per-head weights)
 *    After it [P5 mla-init excerpt: wo maps n_heads * v_head_dim -> dim]:
 *        y       = wo(out)                       (out [T, H * d_v] of the attention)
 *
 *    Every Linear here has no bias: y = x W^T with W stored [out, in].
 *    The linear outputs go into the norms and the rotary step unrounded.
 * ---------------------------------------------------------------------- */

/* y[n, N] = x[n, D] . W[N, D]^T */
ORACLE_API void oracle_linear(const float *x, const float *W, int64_t n, int64_t D, int64_t N, double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < n; ++r)
        for (int64_t o = 0; o < N; ++o) {
            double sum = 0.0;
            for (int64_t i = 0; i < D; ++i) sum += (double)x[r * D + i] * (double)W[o * D + i];
            y[r * N + o] = sum;
        }
}

/* RMSNorm of rows of d values [P4 RMSNorm excerpt]: y = gain * x / sqrt(mean(x^2) + eps). */
ORACLE_API void oracle_rmsnorm(const double *x, int64_t n, int64_t d, const float *gain, double eps, double *y)
{
    for (int64_t r = 0; r < n; ++r) {
        double ms = 0.0;
        for (int64_t i = 0; i < d; ++i) ms += x[r * d + i] * x[r * d + i];
        ms /= (double)d;
        const double inv = 1.0 / sqrt(ms + eps);
        for (int64_t i = 0; i < d; ++i) y[r * d + i] = (double)gain[i] * (x[r * d + i] * inv);
    }
}

/* LayerNorm of rows of d values with gain and bias [P1 printout: k_norm
 * LayerNorm((128,), eps=1e-06, elementwise_affine=True, bias=True)]:
 * y = (x - mean) / sqrt(var + eps) * gain + bias, var = mean of (x - mean)^2. */
ORACLE_API void oracle_layernorm(const double *x, int64_t n, int64_t d, const float *gain, const float *bias,
                                 double eps, double *y)
{
    for (int64_t r = 0; r < n; ++r) {
        double mean = 0.0;
        for (int64_t i = 0; i < d; ++i) mean += x[r * d + i];
        mean /= (double)d;
        double var = 0.0;
        for (int64_t i = 0; i < d; ++i) var += (x[r * d + i] - mean) * (x[r * d + i] - mean);
        var /= (double)d;
        const double inv = 1.0 / sqrt(var + eps);
        for (int64_t i = 0; i < d; ++i)
            y[r * d + i] = (x[r * d + i] - mean) * inv * (double)gain[i] + (double)bias[i];
    }
}

/* Rotary embedding of rows of 2*half values [P5 mla-kv excerpt,
 * apply_rotary_emb with freqs_cis; P1 "The rotary part is served
 * de-interleaved": pair (2i, 2i+1) is turned by the angle of frequency i and
 * lands in dimensions i and half + i]:
 *     y[i]        = x[2i] cos_i - x[2i+1] sin_i
 *     y[half + i] = x[2i] sin_i + x[2i+1] cos_i
 * cos_t, sin_t: [n, half], the row's position already applied. */
ORACLE_API void oracle_rope_deinterleave(const double *x, int64_t n, int64_t half, const float *cos_t,
                                         const float *sin_t, double *y)
{
    for (int64_t r = 0; r < n; ++r)
        for (int64_t i = 0; i < half; ++i) {
            const double a = x[r * 2 * half + 2 * i], b = x[r * 2 * half + 2 * i + 1];
            const double c = (double)cos_t[r * half + i], s = (double)sin_t[r * half + i];
            y[r * 2 * half + i] = a * c - b * s;
            y[r * 2 * half + half + i] = a * s + b * c;
        }
}

/* Number of OpenMP threads this library runs with (reported by the bench). */
ORACLE_API int oracle_num_threads(void)
{
    int n = 1;
#pragma omp parallel
    {
#pragma omp single
        n = omp_get_num_threads();
    }
    return n;
}
