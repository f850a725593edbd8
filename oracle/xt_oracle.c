/*
 * xt_oracle.c -- plain, slow, double-precision CPU oracle of the causal
 * grouped-query attention core: per-head QK-RMSNorm, then rotate_half RoPE,
 * then causal grouped-query scaled-dot-product attention, forward and a
 * hand-derived backward.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference leg load this library. The CUDA path never links,
 * loads or calls it, and the two share no code.
 *
 * Sources (web pages, cited by title and section):
 *   [T9]   xtrain "Phase T9: Export to xserv" (docs/08-export-xserv.md):
 *          architecture-diff table (RMSNorm formula, rotate_half RoPE with
 *          freq = theta^(-2i/hd) and pos = row, scale 1/sqrt(hd), additive
 *          -1e9 causal mask) and Decision 1 (per-head QK-norm with one
 *          [head_dim] gamma, applied after the reshape and before RoPE).
 *   [MINT] Mint project report (morn.ink docs): 5.3.1 single-head attention
 *          formula chain, 5.4.1-5.4.4 RoPE rotation, angle, relative-position
 *          property and backward, 5.5.1-5.5.2 RMSNorm forward and backward.
 *   [T5]   xtrain "Phase T5: Tiny Transformer" (docs/04-tiny-transformer.md):
 *          Key Design Decisions (additive [seq,seq] mask, 0 on and below the
 *          diagonal, -1e9 above; RoPE position = token row) and the
 *          multi-head layout pipeline (per-head 2D SDPA on [nh, seq, hd]).
 *   [T15]  xtrain "Phase T15: Grouped-Query Attention" (docs/14-gqa.md):
 *          "What is GQA" (q head qh reads kv head qh/group) and Decision 2
 *          (repeat_kv forward copy; backward = in-order group-row sum).
 *   [MINT 8.2] Mint project report, 8.2 (forward pass of a flattened chat
 *          batch): samples are packed into [total] rows, RoPE numbers the
 *          positions inside each sample, and a block-causal mask hides other
 *          samples' rows entirely and, inside a sample, the later rows.
 *
 * Arithmetic is double throughout. Matrix products are written as the plain
 * triple loop; every output element is accumulated over its summation index
 * in ascending order (the loop nest is ordered so that the innermost loop
 * runs over independent outputs, which changes no sum).
 *
 * Layouts (row-major, contiguous):
 *   q [B,S,H,D]; k, v [B,S,G,D]; out, dout, dq [B,S,H,D]; dk, dv [B,S,G,D];
 *   lse [B,H,S]; qhat [B,H,S,D]; khat [B,G,S,D]; rstd_q [B,S,H];
 *   rstd_k [B,S,G]; gamma_q, gamma_k, dgamma_q, dgamma_k [D].
 * Packed batches use the same layouts with B = 1 and S = total rows.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* [T5] Key Design Decisions, [T9] diff table: additive mask above the diagonal. */
#define ORC_MASK_VALUE (-1e9)

/* ------------------------------------------------------------------------ */
/* RMSNorm over rows of length D.                                             */
/* [MINT 5.5.1]: rms^2 = (1/d) sum_j x_j^2 + eps ; y_j = x_j * g_j / rms.     */
/* [T9 Decision 1]: applied to every [head_dim] vector of Q and of K, with    */
/* one [head_dim] gamma shared by all heads.                                  */
/* ------------------------------------------------------------------------ */
void orc_rmsnorm_rows(long rows, int D, const double *x, const double *gamma,
                      double eps, double *y, double *rstd)
{
    for (long r = 0; r < rows; ++r) {
        const double *xr = x + r * D;
        double *yr = y + r * D;
        double ss = 0.0;
        for (int j = 0; j < D; ++j) ss += xr[j] * xr[j];
        double rms = sqrt(ss / D + eps);
        for (int j = 0; j < D; ++j) yr[j] = xr[j] * gamma[j] / rms;
        if (rstd) rstd[r] = 1.0 / rms;
    }
}

/* [MINT 5.5.2]: dot = sum_j g_j dy_j x_j ;
 *               dx_j = g_j dy_j / rms - x_j dot / (d rms^3) ;
 *               dg_j += dy_j x_j / rms  (accumulated over rows, in row order). */
void orc_rmsnorm_rows_bwd(long rows, int D, const double *x, const double *gamma,
                          double eps, const double *dy, double *dx, double *dgamma)
{
    for (long r = 0; r < rows; ++r) {
        const double *xr = x + r * D, *dyr = dy + r * D;
        double *dxr = dx + r * D;
        double ss = 0.0;
        for (int j = 0; j < D; ++j) ss += xr[j] * xr[j];
        double rms = sqrt(ss / D + eps);
        double dot = 0.0;
        for (int j = 0; j < D; ++j) dot += gamma[j] * dyr[j] * xr[j];
        for (int j = 0; j < D; ++j)
            dxr[j] = gamma[j] * dyr[j] / rms - xr[j] * dot / (D * rms * rms * rms);
        if (dgamma)
            for (int j = 0; j < D; ++j) dgamma[j] += dyr[j] * (xr[j] / rms);
    }
}

/* ------------------------------------------------------------------------ */
/* rotate_half RoPE on rows of length D, row r at position pos[r].            */
/* [MINT 5.4.1]: pair (i, i + D/2); x' = x cos - y sin ; y' = x sin + y cos.  */
/* [MINT 5.4.2], [T9 diff table]: angle = pos * theta^(-2i/D), i < D/2.       */
/* [MINT 5.4.4]: the backward rotates by the negative angle (inverse != 0).   */
/* ------------------------------------------------------------------------ */
void orc_rope_rows(long rows, int D, double theta, const long *pos,
                   const double *x, double *y, int inverse)
{
    int half = D / 2;
    for (long r = 0; r < rows; ++r) {
        const double *xr = x + r * D;
        double *yr = y + r * D;
        for (int i = 0; i < half; ++i) {
            double angle = (double)pos[r] * pow(theta, -2.0 * i / D);
            double c = cos(angle), s = sin(angle);
            if (inverse) s = -s;
            double a = xr[i], b = xr[i + half];
            yr[i] = a * c - b * s;
            yr[i + half] = a * s + b * c;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* repeat_kv, [T15 Decision 2]: out[b*H + qh] = in[b*G + qh/group] as whole   */
/* [S*D] blocks; the backward is the group-row sum                            */
/* din[b*G + kvh] = sum_{r=0}^{group-1} dout[b*H + kvh*group + r], in r order.*/
/* ------------------------------------------------------------------------ */
void orc_repeat_kv(int B, int H, int G, long SD, const double *in, double *out)
{
    int group = H / G;
    for (int b = 0; b < B; ++b)
        for (int qh = 0; qh < H; ++qh)
            memcpy(out + ((long)b * H + qh) * SD, in + ((long)b * G + qh / group) * SD,
                   sizeof(double) * SD);
}

void orc_repeat_kv_bwd(int B, int H, int G, long SD, const double *dout, double *din)
{
    int group = H / G;
    for (int b = 0; b < B; ++b)
        for (int kvh = 0; kvh < G; ++kvh) {
            double *d = din + ((long)b * G + kvh) * SD;
            const double *s0 = dout + ((long)b * H + (long)kvh * group) * SD;
            for (long e = 0; e < SD; ++e) d[e] = s0[e];
            for (int r = 1; r < group; ++r) {
                const double *sr = dout + ((long)b * H + (long)kvh * group + r) * SD;
                for (long e = 0; e < SD; ++e) d[e] += sr[e];
            }
        }
}

/* ------------------------------------------------------------------------ */
/* Causal SDPA of one head on [S, D] rows ([T5] multi-head pipeline,         */
/* [MINT 5.3.1]).                                                             */
/*   scores = (q k^T) * (1/sqrt(D)) + mask   (mask 0 for j <= t, -1e9 above)  */
/*   p      = row softmax with the row max subtracted                          */
/*   o      = p v ;  lse_t = max_t + ln sum_j exp(scores_tj - max_t)           */
/* p is the caller's [S, S] buffer and holds the probabilities on return.     */
/* ------------------------------------------------------------------------ */
/* blk (may be NULL): sample id of every row, for the block-causal mask of
 * [MINT 8.2]: key j is visible to row t iff j <= t and blk[j] == blk[t];
 * every other key gets the additive -1e9. NULL is the plain causal mask.   */
void orc_sdpa_head_fwd_blk(int S, int D, const int *blk, const double *q, const double *k,
                           const double *v, double *p, double *o, double *lse)
{
    double scale = 1.0 / sqrt((double)D);
    double *kt = (double *)malloc(sizeof(double) * (size_t)D * S);
    for (int j = 0; j < S; ++j)
        for (int d = 0; d < D; ++d) kt[(long)d * S + j] = k[(long)j * D + d];

    for (int t = 0; t < S; ++t) {
        double *pr = p + (long)t * S;
        for (int j = 0; j < S; ++j) pr[j] = 0.0;
        for (int d = 0; d < D; ++d) {
            double qd = q[(long)t * D + d];
            const double *ktd = kt + (long)d * S;
            for (int j = 0; j < S; ++j) pr[j] += qd * ktd[j];
        }
        for (int j = 0; j < S; ++j) {
            int visible = j <= t && (blk == NULL || blk[j] == blk[t]);
            pr[j] = pr[j] * scale + (visible ? 0.0 : ORC_MASK_VALUE);
        }
        double m = pr[0];
        for (int j = 1; j < S; ++j) if (pr[j] > m) m = pr[j];
        double sum = 0.0;
        for (int j = 0; j < S; ++j) { pr[j] = exp(pr[j] - m); sum += pr[j]; }
        for (int j = 0; j < S; ++j) pr[j] /= sum;
        lse[t] = m + log(sum);
        double *orow = o + (long)t * D;
        for (int d = 0; d < D; ++d) orow[d] = 0.0;
        for (int j = 0; j < S; ++j) {
            double pj = pr[j];
            const double *vj = v + (long)j * D;
            for (int d = 0; d < D; ++d) orow[d] += pj * vj[d];
        }
    }
    free(kt);
}

void orc_sdpa_head_fwd(int S, int D, const double *q, const double *k, const double *v,
                       double *p, double *o, double *lse)
{
    orc_sdpa_head_fwd_blk(S, D, NULL, q, k, v, p, o, lse);
}

/* Backward of one head, by hand from the forward above (the softmax Jacobian):
 *   dv = p^T do ; dp = do v^T ; ds = p o (dp - rowsum(dp o p)) ;
 *   dq = (ds k) / sqrt(D) ; dk = (ds^T q) / sqrt(D).
 * p holds the forward probabilities; dq, dk, dv are overwritten.            */
void orc_sdpa_head_bwd(int S, int D, const double *q, const double *k, const double *v,
                       const double *p, const double *dout, double *dq, double *dk, double *dv)
{
    double scale = 1.0 / sqrt((double)D);
    double *vt = (double *)malloc(sizeof(double) * (size_t)D * S);
    double *ds = (double *)malloc(sizeof(double) * (size_t)S * S);
    for (int j = 0; j < S; ++j)
        for (int d = 0; d < D; ++d) vt[(long)d * S + j] = v[(long)j * D + d];

    memset(dv, 0, sizeof(double) * (size_t)S * D);
    memset(dk, 0, sizeof(double) * (size_t)S * D);
    for (int t = 0; t < S; ++t) {
        const double *pr = p + (long)t * S;
        const double *dot_ = dout + (long)t * D;
        /* dv[j] += p[t, j] * do[t]   (ascending t for every dv[j][d]) */
        for (int j = 0; j < S; ++j) {
            double pj = pr[j];
            double *dvj = dv + (long)j * D;
            for (int d = 0; d < D; ++d) dvj[d] += pj * dot_[d];
        }
        /* dp[t, j] = sum_d do[t, d] v[j, d] */
        double *dsr = ds + (long)t * S;
        for (int j = 0; j < S; ++j) dsr[j] = 0.0;
        for (int d = 0; d < D; ++d) {
            double g = dot_[d];
            const double *vtd = vt + (long)d * S;
            for (int j = 0; j < S; ++j) dsr[j] += g * vtd[j];
        }
        /* ds = p o (dp - sum_j dp p) */
        double rowdot = 0.0;
        for (int j = 0; j < S; ++j) rowdot += dsr[j] * pr[j];
        for (int j = 0; j < S; ++j) dsr[j] = pr[j] * (dsr[j] - rowdot);
    }
    for (int t = 0; t < S; ++t) {
        const double *dsr = ds + (long)t * S;
        double *dqt = dq + (long)t * D;
        for (int d = 0; d < D; ++d) dqt[d] = 0.0;
        for (int j = 0; j < S; ++j) {
            double g = dsr[j];
            const double *kj = k + (long)j * D;
            for (int d = 0; d < D; ++d) dqt[d] += g * kj[d];
        }
        for (int d = 0; d < D; ++d) dqt[d] *= scale;
        /* dk[j] += ds[t, j] * q[t]   (ascending t) */
        const double *qt = q + (long)t * D;
        for (int j = 0; j < S; ++j) {
            double g = dsr[j];
            double *dkj = dk + (long)j * D;
            for (int d = 0; d < D; ++d) dkj[d] += g * qt[d];
        }
    }
    for (long e = 0; e < (long)S * D; ++e) dk[e] *= scale;
    free(vt);
    free(ds);
}

/* ------------------------------------------------------------------------ */
/* Thread pool over independent (b, h) heads: each head is computed by one   */
/* thread into its own output slice, so results do not depend on the thread  */
/* count.                                                                     */
/* ------------------------------------------------------------------------ */
typedef struct {
    pthread_mutex_t lock;
    long next, count;
    void (*fn)(void *ctx, long unit);
    void *ctx;
} orc_pool;

static void *orc_pool_worker(void *arg)
{
    orc_pool *pl = (orc_pool *)arg;
    for (;;) {
        pthread_mutex_lock(&pl->lock);
        long u = pl->next++;
        pthread_mutex_unlock(&pl->lock);
        if (u >= pl->count) break;
        pl->fn(pl->ctx, u);
    }
    return NULL;
}

static void orc_parallel(long count, int nthreads, void (*fn)(void *, long), void *ctx)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > count) nthreads = (int)(count > 0 ? count : 1);
    orc_pool pl;
    pthread_mutex_init(&pl.lock, NULL);
    pl.next = 0; pl.count = count; pl.fn = fn; pl.ctx = ctx;
    if (nthreads == 1) {
        orc_pool_worker(&pl);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, orc_pool_worker, &pl);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&pl.lock);
}

/* ------------------------------------------------------------------------ */
/* Whole forward pipeline, in the pages' op order ([T9 Decision 1], [T5]     */
/* layout pipeline, [T15]):                                                   */
/*   reshape to [B*S*heads, D] rows -> RMSNorm -> RoPE (pos = s) ->           */
/*   transpose to [B, heads, S, D] -> repeat_kv of K and V ->                  */
/*   per-head 2D causal SDPA -> merge back to [B, S, H, D].                   */
/* ------------------------------------------------------------------------ */

/* Norm + RoPE of x [B,S,NH,D] into xhat [B,NH,S,D]; rstd [B,S,NH]. tokpos
 * (may be NULL) gives the RoPE position of every token row b*S+s (packed
 * batches, [MINT 8.2]); NULL means position s. */
static void orc_qk_prologue(int B, int S, int NH, int D, double eps, double theta,
                            const long *tokpos, const double *x, const double *gamma,
                            double *xhat, double *rstd)
{
    long rows = (long)B * S * NH;
    double *y = (double *)malloc(sizeof(double) * rows * D);
    double *yr = (double *)malloc(sizeof(double) * rows * D);
    long *pos = (long *)malloc(sizeof(long) * rows);
    orc_rmsnorm_rows(rows, D, x, gamma, eps, y, rstd);
    for (long r = 0; r < rows; ++r)   /* row (b, s, h) sits at s (or at its packed position) */
        pos[r] = tokpos ? tokpos[r / NH] : (r / NH) % S;
    orc_rope_rows(rows, D, theta, pos, y, yr, 0);
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < S; ++s)
            for (int h = 0; h < NH; ++h)
                memcpy(xhat + (((long)b * NH + h) * S + s) * D,
                       yr + (((long)b * S + s) * NH + h) * D, sizeof(double) * D);
    free(y); free(yr); free(pos);
}

/* [B,S,NH,D] <-> [B,NH,S,D] */
static void orc_to_head_major(int B, int S, int NH, int D, const double *x, double *y)
{
    for (int b = 0; b < B; ++b)
        for (int s = 0; s < S; ++s)
            for (int h = 0; h < NH; ++h)
                memcpy(y + (((long)b * NH + h) * S + s) * D,
                       x + (((long)b * S + s) * NH + h) * D, sizeof(double) * D);
}

static void orc_to_token_major(int B, int S, int NH, int D, const double *x, double *y)
{
    for (int b = 0; b < B; ++b)
        for (int h = 0; h < NH; ++h)
            for (int s = 0; s < S; ++s)
                memcpy(y + (((long)b * S + s) * NH + h) * D,
                       x + (((long)b * NH + h) * S + s) * D, sizeof(double) * D);
}

typedef struct {
    int S, D;
    const int *blk;                        /* [S] sample ids (packed) or NULL */
    const double *qh, *krep, *vrep, *dor;  /* [B*H, S, D] */
    double *o, *lse;                       /* [B*H, S, D], [B*H, S] */
    double *dq, *dk, *dv;                  /* [B*H, S, D] (backward only) */
} orc_heads_ctx;

static void orc_head_fwd_unit(void *vctx, long u)
{
    orc_heads_ctx *c = (orc_heads_ctx *)vctx;
    long SD = (long)c->S * c->D;
    double *p = (double *)malloc(sizeof(double) * (size_t)c->S * c->S);
    orc_sdpa_head_fwd_blk(c->S, c->D, c->blk, c->qh + u * SD, c->krep + u * SD,
                          c->vrep + u * SD, p, c->o + u * SD, c->lse + u * c->S);
    free(p);
}

static void orc_head_bwd_unit(void *vctx, long u)
{
    orc_heads_ctx *c = (orc_heads_ctx *)vctx;
    long SD = (long)c->S * c->D;
    double *p = (double *)malloc(sizeof(double) * (size_t)c->S * c->S);
    double *o = (double *)malloc(sizeof(double) * SD);
    double *lse = (double *)malloc(sizeof(double) * c->S);
    orc_sdpa_head_fwd_blk(c->S, c->D, c->blk, c->qh + u * SD, c->krep + u * SD,
                          c->vrep + u * SD, p, o, lse);
    orc_sdpa_head_bwd(c->S, c->D, c->qh + u * SD, c->krep + u * SD, c->vrep + u * SD, p,
                      c->dor + u * SD, c->dq + u * SD, c->dk + u * SD, c->dv + u * SD);
    free(p); free(o); free(lse);
}

static int orc_check_shape(int B, int S, int H, int G, int D)
{
    if (B <= 0 || S <= 0 || H <= 0 || G <= 0 || D <= 0) return 1;
    if (H % G != 0 || D % 2 != 0) return 1;
    return 0;
}

/* Forward. out [B,S,H,D], lse [B,H,S]; qhat/khat/rstd_q/rstd_k may be NULL.
 * blk / tokpos: sample ids and positions of the rows of a packed batch (B = 1),
 * or NULL. */
static int orc_attn_fwd_impl(int B, int S, int H, int G, int D, double eps, double theta,
                             const int *blk, const long *tokpos,
                             const double *q, const double *k, const double *v,
                             const double *gamma_q, const double *gamma_k,
                             double *out, double *lse, double *qhat_out, double *khat_out,
                             double *rstd_q_out, double *rstd_k_out, int nthreads)
{
    if (orc_check_shape(B, S, H, G, D)) return 1;
    long SD = (long)S * D;
    double *qh = (double *)malloc(sizeof(double) * B * H * SD);
    double *kh = (double *)malloc(sizeof(double) * B * G * SD);
    double *vh = (double *)malloc(sizeof(double) * B * G * SD);
    double *krep = (double *)malloc(sizeof(double) * B * H * SD);
    double *vrep = (double *)malloc(sizeof(double) * B * H * SD);
    double *oh = (double *)malloc(sizeof(double) * B * H * SD);
    double *rq = (double *)malloc(sizeof(double) * B * S * H);
    double *rk = (double *)malloc(sizeof(double) * B * S * G);

    orc_qk_prologue(B, S, H, D, eps, theta, tokpos, q, gamma_q, qh, rq);
    orc_qk_prologue(B, S, G, D, eps, theta, tokpos, k, gamma_k, kh, rk);
    orc_to_head_major(B, S, G, D, v, vh);
    orc_repeat_kv(B, H, G, SD, kh, krep);
    orc_repeat_kv(B, H, G, SD, vh, vrep);

    orc_heads_ctx c = {S, D, blk, qh, krep, vrep, NULL, oh, lse, NULL, NULL, NULL};
    orc_parallel((long)B * H, nthreads, orc_head_fwd_unit, &c);
    orc_to_token_major(B, S, H, D, oh, out);

    if (qhat_out) memcpy(qhat_out, qh, sizeof(double) * B * H * SD);
    if (khat_out) memcpy(khat_out, kh, sizeof(double) * B * G * SD);
    if (rstd_q_out) memcpy(rstd_q_out, rq, sizeof(double) * B * S * H);
    if (rstd_k_out) memcpy(rstd_k_out, rk, sizeof(double) * B * S * G);
    free(qh); free(kh); free(vh); free(krep); free(vrep); free(oh); free(rq); free(rk);
    return 0;
}

int orc_attn_fwd(int B, int S, int H, int G, int D, double eps, double theta,
                 const double *q, const double *k, const double *v,
                 const double *gamma_q, const double *gamma_k,
                 double *out, double *lse, double *qhat_out, double *khat_out,
                 double *rstd_q_out, double *rstd_k_out, int nthreads)
{
    return orc_attn_fwd_impl(B, S, H, G, D, eps, theta, NULL, NULL, q, k, v, gamma_q, gamma_k,
                             out, lse, qhat_out, khat_out, rstd_q_out, rstd_k_out, nthreads);
}

/* Backward by the chain rule, in reverse op order: per-head SDPA backward ->
 * repeat_kv backward (group-row sum) -> RoPE backward (negative angle) ->
 * RMSNorm backward. dgamma_q / dgamma_k are overwritten with the sum over all
 * (b, s, head) rows in that row order. */
static int orc_attn_bwd_impl(int B, int S, int H, int G, int D, double eps, double theta,
                             const int *blk, const long *tokpos,
                             const double *q, const double *k, const double *v,
                             const double *gamma_q, const double *gamma_k, const double *dout,
                             double *dq, double *dk, double *dv, double *dgamma_q,
                             double *dgamma_k, int nthreads)
{
    if (orc_check_shape(B, S, H, G, D)) return 1;
    long SD = (long)S * D;
    double *qh = (double *)malloc(sizeof(double) * B * H * SD);
    double *kh = (double *)malloc(sizeof(double) * B * G * SD);
    double *vh = (double *)malloc(sizeof(double) * B * G * SD);
    double *krep = (double *)malloc(sizeof(double) * B * H * SD);
    double *vrep = (double *)malloc(sizeof(double) * B * H * SD);
    double *doh = (double *)malloc(sizeof(double) * B * H * SD);
    double *dqh = (double *)malloc(sizeof(double) * B * H * SD);
    double *dkrep = (double *)malloc(sizeof(double) * B * H * SD);
    double *dvrep = (double *)malloc(sizeof(double) * B * H * SD);
    double *dkh = (double *)malloc(sizeof(double) * B * G * SD);
    double *dvh = (double *)malloc(sizeof(double) * B * G * SD);
    double *lse = (double *)malloc(sizeof(double) * B * H * S);
    double *rq = (double *)malloc(sizeof(double) * B * S * H);
    double *rk = (double *)malloc(sizeof(double) * B * S * G);

    orc_qk_prologue(B, S, H, D, eps, theta, tokpos, q, gamma_q, qh, rq);
    orc_qk_prologue(B, S, G, D, eps, theta, tokpos, k, gamma_k, kh, rk);
    orc_to_head_major(B, S, G, D, v, vh);
    orc_repeat_kv(B, H, G, SD, kh, krep);
    orc_repeat_kv(B, H, G, SD, vh, vrep);
    orc_to_head_major(B, S, H, D, dout, doh);

    orc_heads_ctx c = {S, D, blk, qh, krep, vrep, doh, NULL, lse, dqh, dkrep, dvrep};
    orc_parallel((long)B * H, nthreads, orc_head_bwd_unit, &c);

    orc_repeat_kv_bwd(B, H, G, SD, dkrep, dkh);
    orc_repeat_kv_bwd(B, H, G, SD, dvrep, dvh);
    orc_to_token_major(B, S, G, D, dvh, dv);

    /* RoPE backward then RMSNorm backward on token-major rows. */
    long rq_rows = (long)B * S * H, rk_rows = (long)B * S * G;
    double *dyq = (double *)malloc(sizeof(double) * rq_rows * D);
    double *dyk = (double *)malloc(sizeof(double) * rk_rows * D);
    double *tmpq = (double *)malloc(sizeof(double) * rq_rows * D);
    double *tmpk = (double *)malloc(sizeof(double) * rk_rows * D);
    long *posq = (long *)malloc(sizeof(long) * rq_rows);
    long *posk = (long *)malloc(sizeof(long) * rk_rows);
    orc_to_token_major(B, S, H, D, dqh, tmpq);
    orc_to_token_major(B, S, G, D, dkh, tmpk);
    for (long r = 0; r < rq_rows; ++r) posq[r] = tokpos ? tokpos[r / H] : (r / H) % S;
    for (long r = 0; r < rk_rows; ++r) posk[r] = tokpos ? tokpos[r / G] : (r / G) % S;
    orc_rope_rows(rq_rows, D, theta, posq, tmpq, dyq, 1);
    orc_rope_rows(rk_rows, D, theta, posk, tmpk, dyk, 1);
    memset(dgamma_q, 0, sizeof(double) * D);
    memset(dgamma_k, 0, sizeof(double) * D);
    orc_rmsnorm_rows_bwd(rq_rows, D, q, gamma_q, eps, dyq, dq, dgamma_q);
    orc_rmsnorm_rows_bwd(rk_rows, D, k, gamma_k, eps, dyk, dk, dgamma_k);

    free(qh); free(kh); free(vh); free(krep); free(vrep); free(doh); free(dqh);
    free(dkrep); free(dvrep); free(dkh); free(dvh); free(lse); free(rq); free(rk);
    free(dyq); free(dyk); free(tmpq); free(tmpk); free(posq); free(posk);
    return 0;
}

int orc_attn_bwd(int B, int S, int H, int G, int D, double eps, double theta,
                 const double *q, const double *k, const double *v,
                 const double *gamma_q, const double *gamma_k, const double *dout,
                 double *dq, double *dk, double *dv, double *dgamma_q, double *dgamma_k,
                 int nthreads)
{
    return orc_attn_bwd_impl(B, S, H, G, D, eps, theta, NULL, NULL, q, k, v, gamma_q, gamma_k,
                             dout, dq, dk, dv, dgamma_q, dgamma_k, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Packed batches ([MINT 8.2]): nseq samples, sample s on rows cu[s] ..      */
/* cu[s+1]-1 of [T = cu[nseq]] rows; positions restart at 0 in every sample; */
/* the block-causal mask keeps samples apart. Layouts as above with B = 1,   */
/* S = T: q [T,H,D], k/v [T,G,D], out [T,H,D], lse [H,T], qhat [H,T,D],      */
/* khat [G,T,D], rstd_q [T,H], rstd_k [T,G]. Empty samples are allowed.      */
/* ------------------------------------------------------------------------ */
static int orc_packed_rows(int nseq, const long *cu, int **blk, long **tokpos)
{
    if (nseq <= 0 || cu[0] != 0) return 1;
    for (int s = 0; s < nseq; ++s)
        if (cu[s + 1] < cu[s]) return 1;
    long T = cu[nseq];
    if (T <= 0 || T > 2147483647L) return 1;
    *blk = (int *)malloc(sizeof(int) * T);
    *tokpos = (long *)malloc(sizeof(long) * T);
    for (int s = 0; s < nseq; ++s)
        for (long t = cu[s]; t < cu[s + 1]; ++t) {
            (*blk)[t] = s;
            (*tokpos)[t] = t - cu[s];
        }
    return 0;
}

int orc_attn_fwd_packed(int nseq, const long *cu, int H, int G, int D, double eps, double theta,
                        const double *q, const double *k, const double *v,
                        const double *gamma_q, const double *gamma_k,
                        double *out, double *lse, double *qhat_out, double *khat_out,
                        double *rstd_q_out, double *rstd_k_out, int nthreads)
{
    int *blk = NULL;
    long *tokpos = NULL;
    if (orc_packed_rows(nseq, cu, &blk, &tokpos)) return 1;
    int rc = orc_attn_fwd_impl(1, (int)cu[nseq], H, G, D, eps, theta, blk, tokpos, q, k, v,
                               gamma_q, gamma_k, out, lse, qhat_out, khat_out, rstd_q_out,
                               rstd_k_out, nthreads);
    free(blk); free(tokpos);
    return rc;
}

int orc_attn_bwd_packed(int nseq, const long *cu, int H, int G, int D, double eps, double theta,
                        const double *q, const double *k, const double *v,
                        const double *gamma_q, const double *gamma_k, const double *dout,
                        double *dq, double *dk, double *dv, double *dgamma_q, double *dgamma_k,
                        int nthreads)
{
    int *blk = NULL;
    long *tokpos = NULL;
    if (orc_packed_rows(nseq, cu, &blk, &tokpos)) return 1;
    int rc = orc_attn_bwd_impl(1, (int)cu[nseq], H, G, D, eps, theta, blk, tokpos, q, k, v,
                               gamma_q, gamma_k, dout, dq, dk, dv, dgamma_q, dgamma_k, nthreads);
    free(blk); free(tokpos);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Row-restricted forms of the same definitions, for shapes whose [S, S]     */
/* per-head matrices are too large to materialise. For a query row t, the    */
/* masked keys j > t get scores near -1e9, whose exponentials underflow to   */
/* exactly 0 in double, so summing over j <= t only gives the same numbers.  */
/* ------------------------------------------------------------------------ */

typedef struct {
    int B, S, H, G, D;
    double eps, theta;
    const double *q, *k, *v, *gq, *gk, *dout;
} orc_problem;

/* normalised + rotated row of x [B,S,NH,D] at (b, s, h) */
static void orc_hat_row(const orc_problem *P, const double *x, const double *gamma, int NH,
                        int b, int s, int h, double *out)
{
    int D = P->D;
    double *y = (double *)malloc(sizeof(double) * D);
    long pos = s;
    orc_rmsnorm_rows(1, D, x + (((long)b * P->S + s) * NH + h) * D, gamma, P->eps, y, NULL);
    orc_rope_rows(1, D, P->theta, &pos, y, out, 0);
    free(y);
}

/* khat [S, D] of kv head g of batch b */
static double *orc_khat_all(const orc_problem *P, int b, int g)
{
    double *kh = (double *)malloc(sizeof(double) * (size_t)P->S * P->D);
    for (int s = 0; s < P->S; ++s) orc_hat_row(P, P->k, P->gk, P->G, b, s, g, kh + (long)s * P->D);
    return kh;
}

/* Row t of head h: scores (j <= t), probabilities p[0..t], lse, o.  */
static void orc_row_fwd(const orc_problem *P, int b, int h, int t, const double *khat,
                        const double *qhat_t, double *p, double *lse, double *o)
{
    int D = P->D, group = P->H / P->G, g = h / group;
    double scale = 1.0 / sqrt((double)D);
    for (int j = 0; j <= t; ++j) {
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += qhat_t[d] * khat[(long)j * D + d];
        p[j] = s * scale;
    }
    double m = p[0];
    for (int j = 1; j <= t; ++j) if (p[j] > m) m = p[j];
    double sum = 0.0;
    for (int j = 0; j <= t; ++j) { p[j] = exp(p[j] - m); sum += p[j]; }
    for (int j = 0; j <= t; ++j) p[j] /= sum;
    *lse = m + log(sum);
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    for (int j = 0; j <= t; ++j) {
        const double *vj = P->v + (((long)b * P->S + j) * P->G + g) * D;
        for (int d = 0; d < D; ++d) o[d] += p[j] * vj[d];
    }
}

typedef struct {
    const orc_problem *P;
    const long *idx;      /* n x 3 */
    double *o1, *o2, *o3; /* outputs, per request */
} orc_rows_ctx;

static void orc_fwd_row_unit(void *vctx, long u)
{
    orc_rows_ctx *c = (orc_rows_ctx *)vctx;
    const orc_problem *P = c->P;
    int b = (int)c->idx[3 * u], h = (int)c->idx[3 * u + 1], t = (int)c->idx[3 * u + 2];
    int group = P->H / P->G;
    double *khat = orc_khat_all(P, b, h / group);
    double *qt = (double *)malloc(sizeof(double) * P->D);
    double *p = (double *)malloc(sizeof(double) * (size_t)(t + 1));
    orc_hat_row(P, P->q, P->gq, P->H, b, t, h, qt);
    orc_row_fwd(P, b, h, t, khat, qt, p, c->o2 + u, c->o1 + u * P->D);
    free(khat); free(qt); free(p);
}

/* dq row (b, h, t): ds_tj = p_tj (dp_tj - sum_j dp p), dqhat = sum_j ds k_j / sqrt(D),
 * then RoPE backward and RMSNorm backward of that row. */
static void orc_dq_row_unit(void *vctx, long u)
{
    orc_rows_ctx *c = (orc_rows_ctx *)vctx;
    const orc_problem *P = c->P;
    int D = P->D, group = P->H / P->G;
    int b = (int)c->idx[3 * u], h = (int)c->idx[3 * u + 1], t = (int)c->idx[3 * u + 2];
    int g = h / group;
    double scale = 1.0 / sqrt((double)D);
    double *khat = orc_khat_all(P, b, g);
    double *qt = (double *)malloc(sizeof(double) * D);
    double *o = (double *)malloc(sizeof(double) * D);
    double *p = (double *)malloc(sizeof(double) * (size_t)(t + 1));
    double *ds = (double *)malloc(sizeof(double) * (size_t)(t + 1));
    double *dqh = (double *)malloc(sizeof(double) * D);
    double *dy = (double *)malloc(sizeof(double) * D);
    double lse;
    orc_hat_row(P, P->q, P->gq, P->H, b, t, h, qt);
    orc_row_fwd(P, b, h, t, khat, qt, p, &lse, o);
    const double *dot_ = P->dout + (((long)b * P->S + t) * P->H + h) * D;
    for (int j = 0; j <= t; ++j) {
        const double *vj = P->v + (((long)b * P->S + j) * P->G + g) * D;
        double dp = 0.0;
        for (int d = 0; d < D; ++d) dp += dot_[d] * vj[d];
        ds[j] = dp;
    }
    double rowdot = 0.0;
    for (int j = 0; j <= t; ++j) rowdot += ds[j] * p[j];
    for (int j = 0; j <= t; ++j) ds[j] = p[j] * (ds[j] - rowdot);
    for (int d = 0; d < D; ++d) dqh[d] = 0.0;
    for (int j = 0; j <= t; ++j)
        for (int d = 0; d < D; ++d) dqh[d] += ds[j] * khat[(long)j * D + d];
    for (int d = 0; d < D; ++d) dqh[d] *= scale;
    long pos = t;
    orc_rope_rows(1, D, P->theta, &pos, dqh, dy, 1);
    orc_rmsnorm_rows_bwd(1, D, P->q + (((long)b * P->S + t) * P->H + h) * D, P->gq, P->eps,
                         dy, c->o1 + u * D, NULL);
    free(khat); free(qt); free(o); free(p); free(ds); free(dqh); free(dy);
}

/* dk, dv rows (b, g, j): summed over the group's query heads r = 0..group-1
 * (outer, in order) of the per-head sums over query rows t >= j (ascending). */
static void orc_dkdv_row_unit(void *vctx, long u)
{
    orc_rows_ctx *c = (orc_rows_ctx *)vctx;
    const orc_problem *P = c->P;
    int D = P->D, S = P->S, group = P->H / P->G;
    int b = (int)c->idx[3 * u], g = (int)c->idx[3 * u + 1], j = (int)c->idx[3 * u + 2];
    double scale = 1.0 / sqrt((double)D);
    double *khat = orc_khat_all(P, b, g);
    double *qt = (double *)malloc(sizeof(double) * D);
    double *o = (double *)malloc(sizeof(double) * D);
    double *p = (double *)malloc(sizeof(double) * (size_t)S);
    double *dkh = (double *)calloc((size_t)D, sizeof(double));
    double *dvj = (double *)calloc((size_t)D, sizeof(double));
    double *hk = (double *)malloc(sizeof(double) * D);
    double *hv = (double *)malloc(sizeof(double) * D);
    double *dy = (double *)malloc(sizeof(double) * D);
    const double *vj = P->v + (((long)b * S + j) * P->G + g) * D;
    for (int r = 0; r < group; ++r) {
        int h = g * group + r;
        for (int d = 0; d < D; ++d) { hk[d] = 0.0; hv[d] = 0.0; }
        for (int t = j; t < S; ++t) {
            double lse;
            orc_hat_row(P, P->q, P->gq, P->H, b, t, h, qt);
            orc_row_fwd(P, b, h, t, khat, qt, p, &lse, o);
            const double *dot_ = P->dout + (((long)b * S + t) * P->H + h) * D;
            /* rowsum(dp o p) for row t equals do_t . o_t */
            double rowdot = 0.0;
            for (int jj = 0; jj <= t; ++jj) {
                const double *vjj = P->v + (((long)b * S + jj) * P->G + g) * D;
                double dp = 0.0;
                for (int d = 0; d < D; ++d) dp += dot_[d] * vjj[d];
                rowdot += dp * p[jj];
            }
            double dpj = 0.0;
            for (int d = 0; d < D; ++d) dpj += dot_[d] * vj[d];
            double dsj = p[j] * (dpj - rowdot);
            for (int d = 0; d < D; ++d) hv[d] += p[j] * dot_[d];
            for (int d = 0; d < D; ++d) hk[d] += dsj * qt[d];
        }
        for (int d = 0; d < D; ++d) { dkh[d] += hk[d] * scale; dvj[d] += hv[d]; }
    }
    long pos = j;
    orc_rope_rows(1, D, P->theta, &pos, dkh, dy, 1);
    orc_rmsnorm_rows_bwd(1, D, P->k + (((long)b * S + j) * P->G + g) * D, P->gk, P->eps,
                         dy, c->o1 + u * D, NULL);
    memcpy(c->o2 + u * D, dvj, sizeof(double) * D);
    free(khat); free(qt); free(o); free(p); free(dkh); free(dvj); free(hk); free(hv); free(dy);
}

/* O and LSE for n query rows idx[i] = (b, h, t). o [n, D], lse [n]. */
int orc_attn_fwd_rows(int B, int S, int H, int G, int D, double eps, double theta,
                      const double *q, const double *k, const double *v,
                      const double *gamma_q, const double *gamma_k,
                      long n, const long *idx, double *o, double *lse, int nthreads)
{
    if (orc_check_shape(B, S, H, G, D)) return 1;
    orc_problem P = {B, S, H, G, D, eps, theta, q, k, v, gamma_q, gamma_k, NULL};
    orc_rows_ctx c = {&P, idx, o, lse, NULL};
    orc_parallel(n, nthreads, orc_fwd_row_unit, &c);
    return 0;
}

/* dq for n query rows idx[i] = (b, h, t). dq [n, D] */
int orc_attn_dq_rows(int B, int S, int H, int G, int D, double eps, double theta,
                     const double *q, const double *k, const double *v,
                     const double *gamma_q, const double *gamma_k, const double *dout,
                     long n, const long *idx, double *dq, int nthreads)
{
    if (orc_check_shape(B, S, H, G, D)) return 1;
    orc_problem P = {B, S, H, G, D, eps, theta, q, k, v, gamma_q, gamma_k, dout};
    orc_rows_ctx c = {&P, idx, dq, NULL, NULL};
    orc_parallel(n, nthreads, orc_dq_row_unit, &c);
    return 0;
}

/* dk, dv for n key rows idx[i] = (b, g, j). dk, dv [n, D] */
int orc_attn_dkdv_rows(int B, int S, int H, int G, int D, double eps, double theta,
                       const double *q, const double *k, const double *v,
                       const double *gamma_q, const double *gamma_k, const double *dout,
                       long n, const long *idx, double *dk, double *dv, int nthreads)
{
    if (orc_check_shape(B, S, H, G, D)) return 1;
    orc_problem P = {B, S, H, G, D, eps, theta, q, k, v, gamma_q, gamma_k, dout};
    orc_rows_ctx c = {&P, idx, dk, dv, NULL};
    orc_parallel(n, nthreads, orc_dkdv_row_unit, &c);
    return 0;
}
