/*
 * gdn_oracle.c -- FP64 CPU oracle of the Gated DeltaNet (GDN) training path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the package's smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code with the CUDA library.
 *
 * What it computes (plain per-token recurrence, one document and one q/k head
 * group at a time; the state is reset to zero at the document start):
 *
 *   q^_t = l(q_t),  k^_t = l(k_t)       l = x / sqrt(x.x + eps) if l2norm else x
 *   a_t  = exp(g_t)
 *   p_t  = S_{t-1}^T k^_t                                   (dv)
 *   u_t  = beta_t (v_t - a_t p_t)
 *   S_t  = a_t S_{t-1} + k^_t u_t^T                          (dk x dv)
 *   o_t  = scale S_t^T q^_t
 *
 * i.e. S_t = a_t S_{t-1} + beta_t k_t (v_t - a_t S_{t-1}^T k_t)^T, the gated
 * delta rule with a 128x128 state per value head that the flashinfer Cake GDN
 * pages train ("feat(cake_gdn_kcp) ... #8172" page: per-v-head state of
 * 64 KiB FP32 in the save-set description; "#8542" page, Correctness: optional
 * in-kernel q/k L2 norm).  One q/k head serves G = HV/H consecutive value heads
 * (v-head h reads q/k head h / G).
 *
 * Optionally the document starts from a given state S_0 = S_in instead of
 * zero and its last state S_L is returned (S_out); the backward then starts
 * from a given dS_L = dS_out (the gradient of the loss with respect to S_out,
 * zero if absent) and returns dS_0, the gradient with respect to S_in.  These
 * are the per-document boundary states that a document split across calls
 * (or across devices) passes on.
 *
 * The backward is reverse-mode differentiation of the loop above written out
 * by hand, one token at a time, from the last token of the document to the
 * first.  dS is the gradient with respect to S_t; it starts at dS_out (zero
 * without one) after the last token:
 *
 *   dS   += scale q^_t do_t^T            dq^_t += scale S_t do_t
 *   dk^_t += dS u_t        du = dS^T k^_t       da = <dS, S_{t-1}>
 *   dbeta_t = <du, v_t - a_t p_t>   dv_t = beta_t du   dp = -a_t beta_t du
 *   da  -= beta_t <du, p_t>
 *   dk^_t += S_{t-1} dp    dS_{t-1} = a_t dS + k^_t dp^T    dg_t = a_t da
 *   L2 norm:  dx = dx^/n - x (x.dx^)/n^3,  n = sqrt(x.x + eps)
 *
 * dq, dk are summed over the G value heads of the group before the norm
 * backward.  To keep memory at O(L/64 * dk * dv) the forward stores S every
 * CK tokens and the backward recomputes the states inside each block.
 *
 * All arithmetic is in double precision; inputs are the exact BF16/FP32
 * values the GPU sees, widened to double by the caller.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define CK 64 /* checkpoint interval of the forward states */

static double l2_normalise(const double *x, double *y, int d, int on, double eps)
{
    if (!on) {
        memcpy(y, x, sizeof(double) * (size_t)d);
        return 1.0;
    }
    double ss = 0.0;
    for (int i = 0; i < d; ++i) ss += x[i] * x[i];
    double n = sqrt(ss + eps);
    for (int i = 0; i < d; ++i) y[i] = x[i] / n;
    return n;
}

/* One token of the forward: S <- a S + k (beta (v - a S^T k))^T.
 * Writes p = S_{t-1}^T k and u if they are non-NULL. */
static void token_step(double *S, int dk, int dv, const double *kh, const double *vt,
                       double a, double b, double *p, double *u)
{
    for (int j = 0; j < dv; ++j) p[j] = 0.0;
    for (int i = 0; i < dk; ++i) {
        const double ki = kh[i];
        const double *Si = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) p[j] += Si[j] * ki;
    }
    for (int j = 0; j < dv; ++j) u[j] = b * (vt[j] - a * p[j]);
    for (int i = 0; i < dk; ++i) {
        const double ki = kh[i];
        double *Si = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) Si[j] = a * Si[j] + ki * u[j];
    }
}

static void token_out(const double *S, int dk, int dv, const double *qh, double scale,
                      double *o)
{
    for (int j = 0; j < dv; ++j) o[j] = 0.0;
    for (int i = 0; i < dk; ++i) {
        const double qi = qh[i];
        const double *Si = S + (size_t)i * dv;
        for (int j = 0; j < dv; ++j) o[j] += Si[j] * qi;
    }
    for (int j = 0; j < dv; ++j) o[j] *= scale;
}

/*
 * gdn_oracle_group_states: forward (and, if dout != NULL, backward) of one
 * document segment for one q/k head and its G value heads.
 *
 *   q, k    [L][dk]        v, dout, o, dv_out  [G][L][dv]
 *   g, beta [G][L]         dg, dbeta          [G][L]
 *   dq, dk_out [L][dk]     (sums over the group, after the norm backward)
 *   s_chunk  optional [ceil(L/chunk)][G][dk][dv]: the state entering each
 *            chunk of `chunk` tokens (chunk 0 enters with S_in)
 *   s_in, ds_out  optional [G][dk][dv]: the state entering the segment and
 *            the gradient with respect to the state leaving it (zero if NULL)
 *   s_out, ds_in  optional [G][dk][dv]: the state leaving the segment and
 *            the gradient with respect to s_in (ds_in needs dout)
 *
 * Returns 0 on success, -1 if memory could not be allocated, -2 on bad sizes.
 */
int gdn_oracle_group_states(int L, int dk, int dv, int G,
                            const double *q, const double *k, const double *v,
                            const double *g, const double *beta, const double *dout,
                            int l2norm, double eps, double scale,
                            double *o, double *dq, double *dk_out, double *dv_out,
                            double *dg, double *dbeta, double *s_chunk, int chunk,
                            const double *s_in, double *s_out, const double *ds_out,
                            double *ds_in)
{
    if (L < 0 || dk <= 0 || dv <= 0 || G <= 0 || (s_chunk && chunk <= 0) || (ds_in && !dout)) return -2;
    const size_t SD = (size_t)dk * dv;
    if (L == 0) {   /* nothing happens: the state passes through, and so does its gradient */
        for (int h = 0; h < G; ++h) {
            if (s_out) {
                if (s_in) memcpy(s_out + h * SD, s_in + h * SD, sizeof(double) * SD);
                else memset(s_out + h * SD, 0, sizeof(double) * SD);
            }
            if (ds_in) {
                if (ds_out) memcpy(ds_in + h * SD, ds_out + h * SD, sizeof(double) * SD);
                else memset(ds_in + h * SD, 0, sizeof(double) * SD);
            }
        }
        return 0;
    }
    const int nblk = (L + CK - 1) / CK;
    double *qh = malloc(sizeof(double) * (size_t)L * dk);
    double *kh = malloc(sizeof(double) * (size_t)L * dk);
    double *nq = malloc(sizeof(double) * (size_t)L);
    double *nk = malloc(sizeof(double) * (size_t)L);
    double *S = malloc(sizeof(double) * SD);
    double *ckpt = dout ? malloc(sizeof(double) * SD * (size_t)nblk) : NULL;
    double *blk = dout ? malloc(sizeof(double) * SD * (size_t)(CK + 1)) : NULL;
    double *dS = dout ? malloc(sizeof(double) * SD) : NULL;
    double *dqh = dout ? calloc((size_t)L * dk, sizeof(double)) : NULL;
    double *dkh = dout ? calloc((size_t)L * dk, sizeof(double)) : NULL;
    double *p = malloc(sizeof(double) * (size_t)dv);
    double *u = malloc(sizeof(double) * (size_t)dv);
    double *du = malloc(sizeof(double) * (size_t)dv);
    double *dp = malloc(sizeof(double) * (size_t)dv);
    int rc = 0;
    if (!qh || !kh || !nq || !nk || !S || !p || !u || !du || !dp ||
        (dout && (!ckpt || !blk || !dS || !dqh || !dkh))) {
        rc = -1;
        goto done;
    }
    for (int t = 0; t < L; ++t) {
        nq[t] = l2_normalise(q + (size_t)t * dk, qh + (size_t)t * dk, dk, l2norm, eps);
        nk[t] = l2_normalise(k + (size_t)t * dk, kh + (size_t)t * dk, dk, l2norm, eps);
    }

    for (int h = 0; h < G; ++h) {
        const double *vh = v + (size_t)h * L * dv;
        const double *gh = g + (size_t)h * L;
        const double *bh = beta + (size_t)h * L;
        double *oh = o + (size_t)h * L * dv;

        /* ---- forward ---- */
        if (s_in) memcpy(S, s_in + (size_t)h * SD, sizeof(double) * SD);
        else memset(S, 0, sizeof(double) * SD);
        for (int t = 0; t < L; ++t) {
            if (ckpt && t % CK == 0) memcpy(ckpt + (size_t)(t / CK) * SD, S, sizeof(double) * SD);
            if (s_chunk && t % chunk == 0)
                memcpy(s_chunk + ((size_t)(t / chunk) * G + h) * SD, S, sizeof(double) * SD);
            token_step(S, dk, dv, kh + (size_t)t * dk, vh + (size_t)t * dv, exp(gh[t]), bh[t], p, u);
            token_out(S, dk, dv, qh + (size_t)t * dk, scale, oh + (size_t)t * dv);
        }
        if (s_out) memcpy(s_out + (size_t)h * SD, S, sizeof(double) * SD);
        if (!dout) continue;

        /* ---- backward, block by block from the end ---- */
        const double *doh = dout + (size_t)h * L * dv;
        double *dvh = dv_out + (size_t)h * L * dv;
        double *dgh = dg + (size_t)h * L;
        double *dbh = dbeta + (size_t)h * L;
        if (ds_out) memcpy(dS, ds_out + (size_t)h * SD, sizeof(double) * SD);
        else memset(dS, 0, sizeof(double) * SD);
        for (int bi = nblk - 1; bi >= 0; --bi) {
            const int t0 = bi * CK;
            const int t1 = (t0 + CK < L) ? t0 + CK : L;
            /* blk[r] = S_{t0-1+r}, r = 0..t1-t0 (r = 0 is the state before t0) */
            memcpy(blk, ckpt + (size_t)bi * SD, sizeof(double) * SD);
            for (int t = t0; t < t1; ++t) {
                double *nxt = blk + (size_t)(t - t0 + 1) * SD;
                memcpy(nxt, blk + (size_t)(t - t0) * SD, sizeof(double) * SD);
                token_step(nxt, dk, dv, kh + (size_t)t * dk, vh + (size_t)t * dv, exp(gh[t]), bh[t], p, u);
            }
            for (int t = t1 - 1; t >= t0; --t) {
                const double *Sp = blk + (size_t)(t - t0) * SD;     /* S_{t-1} */
                const double *St = blk + (size_t)(t - t0 + 1) * SD; /* S_t */
                const double *qt = qh + (size_t)t * dk;
                const double *kt = kh + (size_t)t * dk;
                const double *vt = vh + (size_t)t * dv;
                const double *dot = doh + (size_t)t * dv;
                double *dqt = dqh + (size_t)t * dk;
                double *dkt = dkh + (size_t)t * dk;
                const double a = exp(gh[t]), b = bh[t];
                /* recompute p_t = S_{t-1}^T k^_t and u_t */
                for (int j = 0; j < dv; ++j) p[j] = 0.0;
                for (int i = 0; i < dk; ++i)
                    for (int j = 0; j < dv; ++j) p[j] += Sp[(size_t)i * dv + j] * kt[i];
                for (int j = 0; j < dv; ++j) u[j] = b * (vt[j] - a * p[j]);
                /* o_t = scale S_t^T q^_t */
                for (int i = 0; i < dk; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; ++j) {
                        dS[(size_t)i * dv + j] += scale * qt[i] * dot[j];
                        acc += St[(size_t)i * dv + j] * dot[j];
                    }
                    dqt[i] += scale * acc;
                }
                /* S_t = a S_{t-1} + k^ u^T */
                double da = 0.0;
                for (int j = 0; j < dv; ++j) du[j] = 0.0;
                for (int i = 0; i < dk; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; ++j) {
                        const double d = dS[(size_t)i * dv + j];
                        acc += d * u[j];
                        du[j] += d * kt[i];
                        da += d * Sp[(size_t)i * dv + j];
                    }
                    dkt[i] += acc;
                }
                /* u = b (v - a p) */
                double db = 0.0, dup = 0.0;
                for (int j = 0; j < dv; ++j) {
                    db += du[j] * (vt[j] - a * p[j]);
                    dup += du[j] * p[j];
                    dvh[(size_t)t * dv + j] = b * du[j];
                    dp[j] = -a * b * du[j];
                }
                da -= b * dup;
                /* p = S_{t-1}^T k^ ; dS_{t-1} = a dS + k^ dp^T */
                for (int i = 0; i < dk; ++i) {
                    double acc = 0.0;
                    for (int j = 0; j < dv; ++j) {
                        acc += Sp[(size_t)i * dv + j] * dp[j];
                        dS[(size_t)i * dv + j] = a * dS[(size_t)i * dv + j] + kt[i] * dp[j];
                    }
                    dkt[i] += acc;
                }
                dbh[t] = db;
                dgh[t] = a * da;
            }
        }
        if (ds_in) memcpy(ds_in + (size_t)h * SD, dS, sizeof(double) * SD);   /* dS_0 */
    }

    if (dout) {
        /* norm backward on the group sums */
        for (int t = 0; t < L; ++t) {
            const double *x[2] = {q + (size_t)t * dk, k + (size_t)t * dk};
            const double *dxh[2] = {dqh + (size_t)t * dk, dkh + (size_t)t * dk};
            double *dx[2] = {dq + (size_t)t * dk, dk_out + (size_t)t * dk};
            const double n[2] = {nq[t], nk[t]};
            for (int m = 0; m < 2; ++m) {
                if (!l2norm) {
                    memcpy(dx[m], dxh[m], sizeof(double) * (size_t)dk);
                    continue;
                }
                double xd = 0.0;
                for (int i = 0; i < dk; ++i) xd += x[m][i] * dxh[m][i];
                const double n3 = n[m] * n[m] * n[m];
                for (int i = 0; i < dk; ++i) dx[m][i] = dxh[m][i] / n[m] - x[m][i] * xd / n3;
            }
        }
    }
done:
    free(qh); free(kh); free(nq); free(nk); free(S); free(ckpt); free(blk); free(dS);
    free(dqh); free(dkh); free(p); free(u); free(du); free(dp);
    return rc;
}

/* The same with zero boundary states and none returned. */
int gdn_oracle_group(int L, int dk, int dv, int G,
                     const double *q, const double *k, const double *v,
                     const double *g, const double *beta, const double *dout,
                     int l2norm, double eps, double scale,
                     double *o, double *dq, double *dk_out, double *dv_out,
                     double *dg, double *dbeta, double *s_chunk, int chunk)
{
    return gdn_oracle_group_states(L, dk, dv, G, q, k, v, g, beta, dout, l2norm, eps, scale, o, dq,
                                   dk_out, dv_out, dg, dbeta, s_chunk, chunk, NULL, NULL, NULL, NULL);
}
