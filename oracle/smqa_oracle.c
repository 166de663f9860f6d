/*
 * smqa_oracle.c -- plain fp64 CPU oracle for top-k sparse multi-query
 * attention with a per-head attention sink, forward and backward, and for
 * the lightning-indexer backward (at the end of this file).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA library; both sides only read the same seeded input tensors.
 *
 * What it follows (DeepSeek-V4 kernel API pages of NeMo AutoModel):
 *   - tilelang_sparse_mla_fwd, `sparse_mqa_fwd_interface`: q [B,S,H,D] bf16,
 *     one shared keys/values tensor kv [B,S_kv,D] bf16, attn_sink [H] fp32
 *     ("denominator biases"), topk_idxs [B,S,topk] whose entries outside
 *     [0,S_kv) are masked, sm_scale defaulting to D^-1/2; returns O bf16 and
 *     an fp32 log2 LSE that the backward consumes.
 *   - tilelang_sparse_mla_bwd, `sparse_mqa_bwd_interface` and its
 *     preprocess / bwd / postprocess kernels: gradients of O with respect to
 *     q and kv, given dO and the forward's LSE.
 *
 * The method is exact attention over the listed rows, so the oracle is that
 * definition written out in double precision, one (token, head) at a time,
 * with no blocking, no online rescaling and no fusion:
 *
 *   z_j   = c * <q[b,s,h,:], kv[b,idx_j,:]>            for valid slots j
 *   M     = max(max_j z_j, sink_h)
 *   Z     = sum_j exp(z_j - M) + exp(sink_h - M)
 *   p_j   = exp(z_j - M) / Z
 *   O     = sum_j p_j kv[b,idx_j,:]
 *   LSE2  = (M + ln Z) / ln 2                           (log base 2)
 *
 *   Delta = <dO, O>,  dP_j = <dO, kv[b,idx_j,:]>,  g_j = p_j (dP_j - Delta)
 *   dQ    = c sum_j g_j kv[b,idx_j,:]
 *   dKV[b,r] += c g_j q + p_j dO            for every slot j with idx_j = r
 *   dsink_h  += -(exp(sink_h - M)/Z) Delta  (not returned by the pages)
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes): the sink enters as exp(sink_h), unscaled by c; no causal
 * mask beyond what the indices encode; indices address rows of the same batch
 * element; a duplicated index counts once per slot; an all-masked row gives
 * O = 0 and LSE2 = sink_h / ln 2.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bits -> exact double (bf16 is the top half of an IEEE binary32). */
static double bf16_to_f64(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* An input tensor is either raw bf16 bits or fp64 (the fp64 form exists so
 * that finite-difference checks can perturb inputs below bf16 resolution). */
typedef struct { const void* p; int is_f64; } tref;

static void load_row(tref t, size_t off, int n, double* dst)
{
    if (t.is_f64) {
        const double* s = (const double*)t.p + off;
        for (int i = 0; i < n; ++i) dst[i] = s[i];
    } else {
        const uint16_t* s = (const uint16_t*)t.p + off;
        for (int i = 0; i < n; ++i) dst[i] = bf16_to_f64(s[i]);
    }
}

/* A slot is used iff its index names a row of this batch element. */
static int slot_is_valid(int32_t r, int S_kv) { return r >= 0 && r < S_kv; }

int smqa_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Per-(token, head) softmax over the valid slots plus the sink.
 * Fills p[j] with p_j (0 for masked slots) and returns M and Z through the
 * pointers.  kvrows holds the token's gathered key rows as doubles.
 */
static void head_probs(const double* qh, const double* kvrows, const unsigned char* valid,
                       int topk, int D, double c, double sink_h,
                       double* p, double* M_out, double* Z_out)
{
    double M = sink_h;
    for (int j = 0; j < topk; ++j) {
        if (!valid[j]) { p[j] = 0.0; continue; }
        const double* k = kvrows + (size_t)j * D;
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += qh[d] * k[d];
        p[j] = c * acc;               /* temporarily z_j */
        if (p[j] > M) M = p[j];
    }
    double Z = exp(sink_h - M);
    for (int j = 0; j < topk; ++j) {
        if (!valid[j]) continue;
        p[j] = exp(p[j] - M);
        Z += p[j];
    }
    for (int j = 0; j < topk; ++j) p[j] /= Z;
    *M_out = M;
    *Z_out = Z;
}

/* Gather one token's topk kv rows (masked slots left as zeros). */
static void gather_rows(tref kv, const int32_t* idx_row, int b, int S_kv, int D,
                        int topk, double* rows, unsigned char* valid)
{
    for (int j = 0; j < topk; ++j) {
        int32_t r = idx_row[j];
        valid[j] = (unsigned char)slot_is_valid(r, S_kv);
        double* dst = rows + (size_t)j * D;
        if (!valid[j]) { memset(dst, 0, sizeof(double) * (size_t)D); continue; }
        load_row(kv, ((size_t)b * S_kv + (size_t)r) * D, D, dst);
    }
}

/*
 * Forward.  tokens == NULL means every token t = b*S + s in order
 * (n_tok must then equal B*S); otherwise tokens[i] names the flat token whose
 * results go to row i of o / lse2.
 *   o    : double [n_tok, H, D]
 *   lse2 : double [n_tok, H]
 * Returns 0, or -1 on a bad argument / allocation failure.
 */
static int fwd_impl(tref q, tref kv, const double* sink, const int32_t* idx,
                    int B, int S, int S_kv, int H, int D, int topk, double sm_scale,
                    const int64_t* tokens, int64_t n_tok, double* o, double* lse2)
{
    if (B <= 0 || S <= 0 || S_kv <= 0 || H <= 0 || D <= 0 || topk <= 0 || n_tok < 0) return -1;
    if (!tokens && n_tok != (int64_t)B * S) return -1;
    int err = 0;
#pragma omp parallel
    {
        double* rows = (double*)malloc(sizeof(double) * (size_t)topk * D);
        unsigned char* valid = (unsigned char*)malloc((size_t)topk);
        double* qh = (double*)malloc(sizeof(double) * (size_t)D);
        double* p = (double*)malloc(sizeof(double) * (size_t)topk);
        if (!rows || !valid || !qh || !p) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < n_tok; ++i) {
                int64_t t = tokens ? tokens[i] : i;
                if (t < 0 || t >= (int64_t)B * S) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                int b = (int)(t / S);
                gather_rows(kv, idx + (size_t)t * topk, b, S_kv, D, topk, rows, valid);
                for (int h = 0; h < H; ++h) {
                    load_row(q, ((size_t)t * H + h) * D, D, qh);
                    double M, Z;
                    head_probs(qh, rows, valid, topk, D, sm_scale, sink[h], p, &M, &Z);
                    double* orow = o + ((size_t)i * H + h) * D;
                    for (int d = 0; d < D; ++d) orow[d] = 0.0;
                    for (int j = 0; j < topk; ++j) {
                        if (!valid[j]) continue;
                        const double* v = rows + (size_t)j * D;
                        for (int d = 0; d < D; ++d) orow[d] += p[j] * v[d];
                    }
                    lse2[(size_t)i * H + h] = (M + log(Z)) / log(2.0);
                }
            }
        }
        free(rows); free(valid); free(qh); free(p);
    }
    return err ? -1 : 0;
}

/*
 * Backward.  Same token selection as the forward.  O, p and Delta are taken
 * from this oracle's own fp64 forward, not from any stored output.
 *   dq    : double [n_tok, H, D]            (overwritten)
 *   dkv   : double [B, S_kv, D]             (ACCUMULATED into; caller zeroes)
 *   dsink : double [H] or NULL               (ACCUMULATED into)
 *   delta : double [n_tok, H] or NULL        (overwritten)
 */
static int bwd_impl(tref q, tref kv, const double* sink, const int32_t* idx,
                    tref dout, int B, int S, int S_kv, int H, int D, int topk,
                    double sm_scale, const int64_t* tokens, int64_t n_tok,
                    double* dq, double* dkv, double* dsink, double* delta)
{
    if (B <= 0 || S <= 0 || S_kv <= 0 || H <= 0 || D <= 0 || topk <= 0 || n_tok < 0) return -1;
    if (!tokens && n_tok != (int64_t)B * S) return -1;
    int err = 0;
#pragma omp parallel
    {
        double* rows = (double*)malloc(sizeof(double) * (size_t)topk * D);
        unsigned char* valid = (unsigned char*)malloc((size_t)topk);
        double* qh = (double*)malloc(sizeof(double) * (size_t)D);
        double* doh = (double*)malloc(sizeof(double) * (size_t)D);
        double* oh = (double*)malloc(sizeof(double) * (size_t)D);
        double* p = (double*)malloc(sizeof(double) * (size_t)topk);
        double* g = (double*)malloc(sizeof(double) * (size_t)topk);
        if (!rows || !valid || !qh || !doh || !oh || !p || !g) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < n_tok; ++i) {
                int64_t t = tokens ? tokens[i] : i;
                if (t < 0 || t >= (int64_t)B * S) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                int b = (int)(t / S);
                const int32_t* idx_row = idx + (size_t)t * topk;
                gather_rows(kv, idx_row, b, S_kv, D, topk, rows, valid);
                for (int h = 0; h < H; ++h) {
                    load_row(q, ((size_t)t * H + h) * D, D, qh);
                    load_row(dout, ((size_t)t * H + h) * D, D, doh);
                    double M, Z;
                    head_probs(qh, rows, valid, topk, D, sm_scale, sink[h], p, &M, &Z);
                    /* O from the fp64 forward, then Delta = <dO, O>. */
                    for (int d = 0; d < D; ++d) oh[d] = 0.0;
                    for (int j = 0; j < topk; ++j) {
                        if (!valid[j]) continue;
                        const double* v = rows + (size_t)j * D;
                        for (int d = 0; d < D; ++d) oh[d] += p[j] * v[d];
                    }
                    double Delta = 0.0;
                    for (int d = 0; d < D; ++d) Delta += doh[d] * oh[d];
                    if (delta) delta[(size_t)i * H + h] = Delta;
                    /* g_j = p_j (dP_j - Delta), dP_j = <dO, v_j>. */
                    for (int j = 0; j < topk; ++j) {
                        if (!valid[j]) { g[j] = 0.0; continue; }
                        const double* v = rows + (size_t)j * D;
                        double dP = 0.0;
                        for (int d = 0; d < D; ++d) dP += doh[d] * v[d];
                        g[j] = p[j] * (dP - Delta);
                    }
                    double* dqrow = dq + ((size_t)i * H + h) * D;
                    for (int d = 0; d < D; ++d) dqrow[d] = 0.0;
                    for (int j = 0; j < topk; ++j) {
                        if (!valid[j]) continue;
                        const double* k = rows + (size_t)j * D;
                        for (int d = 0; d < D; ++d) dqrow[d] += sm_scale * g[j] * k[d];
                        double* dst = dkv + ((size_t)b * S_kv + (size_t)idx_row[j]) * D;
                        for (int d = 0; d < D; ++d) {
                            double contrib = sm_scale * g[j] * qh[d] + p[j] * doh[d];
#pragma omp atomic
                            dst[d] += contrib;
                        }
                    }
                    if (dsink) {
                        double psink = exp(sink[h] - M) / Z;
#pragma omp atomic
                        dsink[h] += -psink * Delta;
                    }
                }
            }
        }
        free(rows); free(valid); free(qh); free(doh); free(oh); free(p); free(g);
    }
    return err ? -1 : 0;
}

/* ---- exported entry points ------------------------------------------------
 * *_bf16: q, kv, dout are raw bf16 bits (uint16), attn_sink is fp32, exactly
 *         as the CUDA library receives them.
 * *_f64 : the same computation on fp64 inputs (sink fp64), for
 *         finite-difference and library-reference checks.
 */
static double* sink_to_f64(const float* s, int H)
{
    double* out = (double*)malloc(sizeof(double) * (size_t)(H > 0 ? H : 1));
    if (out)
        for (int h = 0; h < H; ++h) out[h] = (double)s[h];
    return out;
}

int smqa_oracle_fwd(const uint16_t* q, const uint16_t* kv, const float* sink, const int32_t* idx,
                    int B, int S, int S_kv, int H, int D, int topk, double sm_scale,
                    const int64_t* tokens, int64_t n_tok, double* o, double* lse2)
{
    double* s64 = sink_to_f64(sink, H);
    if (!s64) return -1;
    tref tq = {q, 0}, tkv = {kv, 0};
    int rc = fwd_impl(tq, tkv, s64, idx, B, S, S_kv, H, D, topk, sm_scale, tokens, n_tok, o, lse2);
    free(s64);
    return rc;
}

int smqa_oracle_bwd(const uint16_t* q, const uint16_t* kv, const float* sink, const int32_t* idx,
                    const uint16_t* dout, int B, int S, int S_kv, int H, int D, int topk,
                    double sm_scale, const int64_t* tokens, int64_t n_tok,
                    double* dq, double* dkv, double* dsink, double* delta)
{
    double* s64 = sink_to_f64(sink, H);
    if (!s64) return -1;
    tref tq = {q, 0}, tkv = {kv, 0}, tdo = {dout, 0};
    int rc = bwd_impl(tq, tkv, s64, idx, tdo, B, S, S_kv, H, D, topk, sm_scale, tokens, n_tok,
                      dq, dkv, dsink, delta);
    free(s64);
    return rc;
}

int smqa_oracle_fwd_f64(const double* q, const double* kv, const double* sink, const int32_t* idx,
                        int B, int S, int S_kv, int H, int D, int topk, double sm_scale,
                        const int64_t* tokens, int64_t n_tok, double* o, double* lse2)
{
    tref tq = {q, 1}, tkv = {kv, 1};
    return fwd_impl(tq, tkv, sink, idx, B, S, S_kv, H, D, topk, sm_scale, tokens, n_tok, o, lse2);
}

int smqa_oracle_bwd_f64(const double* q, const double* kv, const double* sink, const int32_t* idx,
                        const double* dout, int B, int S, int S_kv, int H, int D, int topk,
                        double sm_scale, const int64_t* tokens, int64_t n_tok,
                        double* dq, double* dkv, double* dsink, double* delta)
{
    tref tq = {q, 1}, tkv = {kv, 1}, tdo = {dout, 1};
    return bwd_impl(tq, tkv, sink, idx, tdo, B, S, S_kv, H, D, topk, sm_scale, tokens, n_tok,
                    dq, dkv, dsink, delta);
}

/* ==========================================================================
 * Lightning-indexer backward (DeepSeek-V4 kernel API pages of NeMo
 * AutoModel, tilelang_indexer_bwd: `indexer_bwd_interface` for one batch
 * element and `batched_indexer_bwd`).  The pages give the tensors only:
 * index_q [S,H,D] bf16, weights [S,H] fp32, index_k [S_kv,D] bf16,
 * topk_indices [S,topk] int32, grad_scores [S,topk] fp32, and one returned
 * tensor [S,H,D] bf16, the gradient with respect to index_q.  They print no
 * scoring formula.  Reading (reading-dependent: not pinned by the pages):
 * the lightning indexer's score of slot j of token t is
 *
 *   score[t,j] = sum_h w[t,h] * ReLU(<q[t,h,:], k[idx[t,j],:]>)
 *
 * with masked slots (index outside [0,S_kv)) scoring 0, so
 *
 *   dq[t,h,:] = w[t,h] * sum_{valid j} g[t,j] * [<q[t,h,:], k_j> > 0] * k_j
 *
 * (the ReLU's derivative taken as 0 at 0).  A slot listed twice counts twice.
 *
 * The gate [<q,k_j> > 0] is a decision taken in floating point: a GPU that
 * forms <q,k_j> in fp32 can decide differently where the exact value lies
 * within its rounding of 0.  With amb > 0 every (token, head, slot) whose
 * fp64 logit has |<q,k_j>| <= amb * sum_d |q_d k_jd| is left out of dq and
 * the magnitude of its term |w g k_j| is added to slack[t,h,:], so a result
 * that takes either decision there lies within slack of dq.  amb = 0 gives
 * the plain definition (slack stays 0).
 * ========================================================================== */

/* score[i,j] for the selected tokens (scores: double [n_tok, topk]). */
static int indexer_scores_impl(tref q, const double* w, tref k, const int32_t* idx, int S,
                               int S_kv, int H, int D, int topk, const int64_t* tokens,
                               int64_t n_tok, double* scores)
{
    if (S <= 0 || S_kv <= 0 || H <= 0 || D <= 0 || topk <= 0 || n_tok < 0) return -1;
    if (!tokens && n_tok != (int64_t)S) return -1;
    int err = 0;
#pragma omp parallel
    {
        double* qh = (double*)malloc(sizeof(double) * (size_t)D);
        double* kj = (double*)malloc(sizeof(double) * (size_t)D);
        if (!qh || !kj) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t i = 0; i < n_tok; ++i) {
                int64_t t = tokens ? tokens[i] : i;
                if (t < 0 || t >= (int64_t)S) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                const int32_t* idx_row = idx + (size_t)t * topk;
                for (int j = 0; j < topk; ++j) {
                    double sc = 0.0;
                    if (slot_is_valid(idx_row[j], S_kv)) {
                        load_row(k, (size_t)idx_row[j] * D, D, kj);
                        for (int h = 0; h < H; ++h) {
                            load_row(q, ((size_t)t * H + h) * D, D, qh);
                            double l = 0.0;
                            for (int d = 0; d < D; ++d) l += qh[d] * kj[d];
                            if (l > 0.0) sc += w[(size_t)t * H + h] * l;
                        }
                    }
                    scores[(size_t)i * topk + j] = sc;
                }
            }
        }
        free(qh); free(kj);
    }
    return err ? -1 : 0;
}

/* dq (and slack) for the selected tokens: double [n_tok, H, D] each. */
static int indexer_bwd_impl(tref q, const double* w, tref k, const int32_t* idx,
                            const double* g, int S, int S_kv, int H, int D, int topk,
                            const int64_t* tokens, int64_t n_tok, double amb, double* dq,
                            double* slack)
{
    if (S <= 0 || S_kv <= 0 || H <= 0 || D <= 0 || topk <= 0 || n_tok < 0 || amb < 0.0) return -1;
    if (!tokens && n_tok != (int64_t)S) return -1;
    int err = 0;
#pragma omp parallel
    {
        double* qh = (double*)malloc(sizeof(double) * (size_t)D);
        double* rows = (double*)malloc(sizeof(double) * (size_t)topk * D);
        unsigned char* valid = (unsigned char*)malloc((size_t)topk);
        if (!qh || !rows || !valid) {
#pragma omp atomic write
            err = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t i = 0; i < n_tok; ++i) {
                int64_t t = tokens ? tokens[i] : i;
                if (t < 0 || t >= (int64_t)S) {
#pragma omp atomic write
                    err = 1;
                    continue;
                }
                const int32_t* idx_row = idx + (size_t)t * topk;
                for (int j = 0; j < topk; ++j) {
                    valid[j] = (unsigned char)slot_is_valid(idx_row[j], S_kv);
                    if (valid[j]) load_row(k, (size_t)idx_row[j] * D, D, rows + (size_t)j * D);
                }
                for (int h = 0; h < H; ++h) {
                    load_row(q, ((size_t)t * H + h) * D, D, qh);
                    const double wh = w[(size_t)t * H + h];
                    double* dqrow = dq + ((size_t)i * H + h) * D;
                    double* slrow = slack ? slack + ((size_t)i * H + h) * D : NULL;
                    for (int d = 0; d < D; ++d) dqrow[d] = 0.0;
                    if (slrow)
                        for (int d = 0; d < D; ++d) slrow[d] = 0.0;
                    for (int j = 0; j < topk; ++j) {
                        if (!valid[j]) continue;
                        const double* kj = rows + (size_t)j * D;
                        double l = 0.0, mag = 0.0;
                        for (int d = 0; d < D; ++d) {
                            l += qh[d] * kj[d];
                            mag += fabs(qh[d] * kj[d]);
                        }
                        const double gj = g[(size_t)t * topk + j];
                        if (amb > 0.0 && fabs(l) <= amb * mag) {
                            if (slrow)
                                for (int d = 0; d < D; ++d) slrow[d] += fabs(wh * gj * kj[d]);
                            continue;
                        }
                        if (l > 0.0)
                            for (int d = 0; d < D; ++d) dqrow[d] += wh * gj * kj[d];
                    }
                }
            }
        }
        free(qh); free(rows); free(valid);
    }
    return err ? -1 : 0;
}

static double* f32_to_f64(const float* s, size_t n)
{
    double* out = (double*)malloc(sizeof(double) * (n > 0 ? n : 1));
    if (out)
        for (size_t i = 0; i < n; ++i) out[i] = (double)s[i];
    return out;
}

int smqa_oracle_indexer_bwd(const uint16_t* q, const float* w, const uint16_t* k,
                            const int32_t* idx, const float* g, int S, int S_kv, int H, int D,
                            int topk, const int64_t* tokens, int64_t n_tok, double amb,
                            double* dq, double* slack)
{
    double* w64 = f32_to_f64(w, (size_t)S * (size_t)H);
    double* g64 = f32_to_f64(g, (size_t)S * (size_t)topk);
    int rc = -1;
    if (w64 && g64) {
        tref tq = {q, 0}, tk = {k, 0};
        rc = indexer_bwd_impl(tq, w64, tk, idx, g64, S, S_kv, H, D, topk, tokens, n_tok, amb, dq,
                              slack);
    }
    free(w64); free(g64);
    return rc;
}

int smqa_oracle_indexer_bwd_f64(const double* q, const double* w, const double* k,
                                const int32_t* idx, const double* g, int S, int S_kv, int H,
                                int D, int topk, const int64_t* tokens, int64_t n_tok,
                                double amb, double* dq, double* slack)
{
    tref tq = {q, 1}, tk = {k, 1};
    return indexer_bwd_impl(tq, w, tk, idx, g, S, S_kv, H, D, topk, tokens, n_tok, amb, dq,
                            slack);
}

int smqa_oracle_indexer_scores_f64(const double* q, const double* w, const double* k,
                                   const int32_t* idx, int S, int S_kv, int H, int D, int topk,
                                   const int64_t* tokens, int64_t n_tok, double* scores)
{
    tref tq = {q, 1}, tk = {k, 1};
    return indexer_scores_impl(tq, w, tk, idx, S, S_kv, H, D, topk, tokens, n_tok, scores);
}
