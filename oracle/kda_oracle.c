/*
 * kda_oracle.c -- plain fp64 CPU reference for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * arm use it. It shares no code, header or constant with the CUDA library.
 *
 * What it computes. KDA ("Kimi K3 on Fireworks: Fast RL at frontier scale",
 * training section, KDA paragraph; also the section "KDA：从循环记忆到高效 GPU
 * 执行" of "Fireworks 发布 Kimi K3 大规模强化学习技术报告") is linear attention
 * whose per-head recurrent state S (dk x dv, stored [k][v]) is updated with
 * channel-wise gating. Written out token by token (the gated delta rule):
 *
 *     q^ = scale * q / sqrt(sum q^2 + eps),   k^ = k / sqrt(sum k^2 + eps)
 *     S' = Diag(exp(g_t)) S                    (decay rows c by exp(g_t[c]))
 *     u  = beta_t (v_t - S'^T k^)
 *     S  = S' + k^ u^T        (== (I - beta k^ k^T) Diag(exp g) S + beta k^ v^T)
 *     o_t = S^T q^
 *
 * The benchmark caption of the first page says the measured KDA core includes
 * the Q/K normalisation; it is therefore part of the op here.
 *
 * Inputs are read in their stored precision (bf16 bit patterns or fp32) and
 * widened exactly to double; every sum is carried in double. No chunking,
 * blocking, fusion or reordering is used: one token after another.
 *
 * The backward is hand-written backpropagation through time over the same
 * loop, in double, recomputing the forward from state checkpoints taken every
 * CKPT tokens.
 *
 * Decode / draft-verify ("ReplaySSM ... advances KDA state only through the
 * accepted prefix", rollout section of the second page): the same loop over L
 * tokens returning all L outputs, with the state committed after `accept`
 * tokens (accept = 0: the state is left as it was).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int64_t T;           /* tokens in this (sequence, head) task                   */
    int32_t dk, dv;      /* key and value widths                                   */
    int32_t io_bf16;     /* q, k, v, dO hold bf16 bit patterns (1) or fp32 (0)     */
    double scale, eps;   /* q scale; epsilon inside the L2-norm square root         */
    const void *q, *k, *v, *dO;   /* element (t, c) at base[t * stride + c]         */
    int64_t sq, sk, sv, sdo;      /* token strides, in elements                     */
    const float *beta;  int64_t sbeta;   /* beta_t at beta[t * sbeta]               */
    const float *g;     int64_t sg;      /* g_t[c] at g[t * sg + c]                 */
    const float *h0;     /* [dk][dv] initial state, or NULL for zero               */
    const float *dhT;    /* [dk][dv] gradient of the final state, or NULL (bwd)    */
    int64_t accept;      /* decode: commit the state after this many tokens        */
    /* outputs (double); token t of a [T][d] output lives at base[t * so + c]      */
    int64_t so, sb;      /* token strides of o/dq/dk/dv/dg and of dbeta            */
    double *o;           /* [T][dv]                                                */
    double *hT;          /* [dk][dv] final (or committed) state                    */
    double *dq, *dk_, *dv_, *dg;   /* [T][dk|dv]                                   */
    double *dbeta;       /* [T]                                                    */
    double *dh0;         /* [dk][dv]                                               */
} kda_oracle_task;

#define CKPT 64

static double load_io(const void *base, int64_t idx, int bf16)
{
    if (bf16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[idx];
}

/* x^ = s * x / sqrt(sum x^2 + eps); returns 1/sqrt(sum x^2 + eps). */
static double l2norm_row(const void *base, int64_t off, int n, int bf16, double s,
                         double eps, double *raw, double *out)
{
    double ss = 0.0;
    for (int c = 0; c < n; ++c) {
        raw[c] = load_io(base, off + c, bf16);
        ss += raw[c] * raw[c];
    }
    double r = 1.0 / sqrt(ss + eps);
    for (int c = 0; c < n; ++c) out[c] = s * raw[c] * r;
    return r;
}

/* One token of the recurrence, in place on S. Returns nothing; fills u, resid
 * (v - S'^T k^) and o. S' (the decayed state) is written to Sp when non-NULL. */
static void token_step(const kda_oracle_task *t, int64_t i, double *S, const double *qn,
                       const double *kn, double *u, double *resid, double *o, double *Sp)
{
    const int dk = t->dk, dv = t->dv;
    const double beta = (double)t->beta[i * t->sbeta];
    const float *gi = t->g + i * t->sg;
    /* S' = Diag(exp(g)) S */
    for (int c = 0; c < dk; ++c) {
        double dec = exp((double)gi[c]);
        for (int j = 0; j < dv; ++j) S[c * dv + j] *= dec;
    }
    if (Sp) memcpy(Sp, S, sizeof(double) * dk * dv);
    /* w = S'^T k^ ; u = beta (v - w) */
    for (int j = 0; j < dv; ++j) resid[j] = 0.0;
    for (int c = 0; c < dk; ++c)
        for (int j = 0; j < dv; ++j) resid[j] += S[c * dv + j] * kn[c];
    for (int j = 0; j < dv; ++j) {
        resid[j] = load_io(t->v, i * t->sv + j, t->io_bf16) - resid[j];
        u[j] = beta * resid[j];
    }
    /* S = S' + k^ u^T */
    for (int c = 0; c < dk; ++c)
        for (int j = 0; j < dv; ++j) S[c * dv + j] += kn[c] * u[j];
    /* o = S^T q^ */
    for (int j = 0; j < dv; ++j) o[j] = 0.0;
    for (int c = 0; c < dk; ++c)
        for (int j = 0; j < dv; ++j) o[j] += S[c * dv + j] * qn[c];
}

static void init_state(const kda_oracle_task *t, double *S)
{
    const int64_t n = (int64_t)t->dk * t->dv;
    for (int64_t e = 0; e < n; ++e) S[e] = t->h0 ? (double)t->h0[e] : 0.0;
}

/* Forward (and decode when commit_at >= 0): o for every token; hT = final state,
 * or the state after commit_at tokens. */
static void run_forward(const kda_oracle_task *t, int64_t commit_at)
{
    const int dk = t->dk, dv = t->dv;
    double *S = malloc(sizeof(double) * dk * dv);
    double *raw = malloc(sizeof(double) * (dk > dv ? dk : dv));
    double *qn = malloc(sizeof(double) * dk), *kn = malloc(sizeof(double) * dk);
    double *u = malloc(sizeof(double) * dv), *res = malloc(sizeof(double) * dv);
    double *o = malloc(sizeof(double) * dv);
    init_state(t, S);
    if (commit_at == 0 && t->hT) memcpy(t->hT, S, sizeof(double) * dk * dv);
    for (int64_t i = 0; i < t->T; ++i) {
        l2norm_row(t->q, i * t->sq, dk, t->io_bf16, t->scale, t->eps, raw, qn);
        l2norm_row(t->k, i * t->sk, dk, t->io_bf16, 1.0, t->eps, raw, kn);
        token_step(t, i, S, qn, kn, u, res, o, NULL);
        if (t->o)
            for (int j = 0; j < dv; ++j) t->o[i * t->so + j] = o[j];
        if (commit_at == i + 1 && t->hT) memcpy(t->hT, S, sizeof(double) * dk * dv);
    }
    if (commit_at < 0 && t->hT) memcpy(t->hT, S, sizeof(double) * dk * dv);
    free(S); free(raw); free(qn); free(kn); free(u); free(res); free(o);
}

/* Backward: gradients of <dO, o> + <dhT, hT> with respect to q, k, v, beta, g, h0. */
static void run_backward(const kda_oracle_task *t)
{
    const int dk = t->dk, dv = t->dv;
    const int64_t T = t->T, nst = (int64_t)dk * dv;
    const int64_t nseg = (T + CKPT - 1) / CKPT;
    double *ck = malloc(sizeof(double) * nst * (nseg > 0 ? nseg : 1)); /* S before each segment */
    double *S = malloc(sizeof(double) * nst);
    double *Sp = malloc(sizeof(double) * nst * CKPT);    /* S' per token of a segment  */
    double *Sn = malloc(sizeof(double) * nst * CKPT);    /* S after each token         */
    double *U = malloc(sizeof(double) * dv * CKPT), *R = malloc(sizeof(double) * dv * CKPT);
    double *QN = malloc(sizeof(double) * dk * CKPT), *KN = malloc(sizeof(double) * dk * CKPT);
    double *RQ = malloc(sizeof(double) * CKPT), *RK = malloc(sizeof(double) * CKPT);
    double *QR = malloc(sizeof(double) * dk * CKPT), *KR = malloc(sizeof(double) * dk * CKPT);
    double *o = malloc(sizeof(double) * dv);
    double *dS = malloc(sizeof(double) * nst), *dSp = malloc(sizeof(double) * nst);
    double *dqn = malloc(sizeof(double) * dk), *dkn = malloc(sizeof(double) * dk);
    double *du = malloc(sizeof(double) * dv), *dov = malloc(sizeof(double) * dv);

    /* forward pass, keeping the state at the start of every segment */
    init_state(t, S);
    for (int64_t i = 0; i < T; ++i) {
        if (i % CKPT == 0) memcpy(ck + (i / CKPT) * nst, S, sizeof(double) * nst);
        l2norm_row(t->q, i * t->sq, dk, t->io_bf16, t->scale, t->eps, QR, QN);
        l2norm_row(t->k, i * t->sk, dk, t->io_bf16, 1.0, t->eps, KR, KN);
        token_step(t, i, S, QN, KN, U, R, o, NULL);
    }

    for (int64_t e = 0; e < nst; ++e) dS[e] = t->dhT ? (double)t->dhT[e] : 0.0;

    for (int64_t seg = nseg - 1; seg >= 0; --seg) {
        const int64_t t0 = seg * CKPT, t1 = (t0 + CKPT < T) ? t0 + CKPT : T;
        /* recompute the segment, keeping S', S, u and (v - S'^T k^) per token */
        memcpy(S, ck + seg * nst, sizeof(double) * nst);
        for (int64_t i = t0; i < t1; ++i) {
            const int64_t l = i - t0;
            RQ[l] = l2norm_row(t->q, i * t->sq, dk, t->io_bf16, t->scale, t->eps,
                               QR + l * dk, QN + l * dk);
            RK[l] = l2norm_row(t->k, i * t->sk, dk, t->io_bf16, 1.0, t->eps,
                               KR + l * dk, KN + l * dk);
            token_step(t, i, S, QN + l * dk, KN + l * dk, U + l * dv, R + l * dv, o,
                       Sp + l * nst);
            memcpy(Sn + l * nst, S, sizeof(double) * nst);
        }
        for (int64_t i = t1 - 1; i >= t0; --i) {
            const int64_t l = i - t0;
            const double *qn = QN + l * dk, *kn = KN + l * dk, *u = U + l * dv;
            const double *Spt = Sp + l * nst, *St = Sn + l * nst;
            const double beta = (double)t->beta[i * t->sbeta];
            const float *gi = t->g + i * t->sg;
            for (int j = 0; j < dv; ++j) dov[j] = load_io(t->dO, i * t->sdo + j, t->io_bf16);
            /* o = S^T q^ :  dS += q^ dO^T ; dq^ = S dO */
            for (int c = 0; c < dk; ++c) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) {
                    dS[c * dv + j] += qn[c] * dov[j];
                    acc += St[c * dv + j] * dov[j];
                }
                dqn[c] = acc;
            }
            /* S = S' + k^ u^T :  dk^ = dS u ; du = dS^T k^ ; dS' = dS */
            for (int j = 0; j < dv; ++j) du[j] = 0.0;
            for (int c = 0; c < dk; ++c) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) {
                    acc += dS[c * dv + j] * u[j];
                    du[j] += dS[c * dv + j] * kn[c];
                }
                dkn[c] = acc;
            }
            /* u = beta (v - S'^T k^) */
            double db = 0.0;
            for (int j = 0; j < dv; ++j) db += du[j] * R[l * dv + j];
            for (int c = 0; c < dk; ++c) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) {
                    dSp[c * dv + j] = dS[c * dv + j] - beta * kn[c] * du[j];
                    acc += Spt[c * dv + j] * du[j];
                }
                dkn[c] -= beta * acc;
            }
            /* S' = Diag(exp g) S_prev :  dg_c = sum_j S'_cj dS'_cj ; dS_prev = Diag(exp g) dS' */
            for (int c = 0; c < dk; ++c) {
                double acc = 0.0, dec = exp((double)gi[c]);
                for (int j = 0; j < dv; ++j) {
                    acc += Spt[c * dv + j] * dSp[c * dv + j];
                    dS[c * dv + j] = dec * dSp[c * dv + j];
                }
                if (t->dg) t->dg[i * t->so + c] = acc;
            }
            if (t->dbeta) t->dbeta[i * t->sb] = db;
            if (t->dv_)
                for (int j = 0; j < dv; ++j) t->dv_[i * t->so + j] = beta * du[j];
            /* L2 norm: x^ = s x r, r = (sum x^2 + eps)^(-1/2):
             *   dx = s (r dx^ - r^3 x (x . dx^)) */
            {
                const double *qr = QR + l * dk, *kr = KR + l * dk;
                double rq = RQ[l], rk = RK[l], pq = 0.0, pk = 0.0;
                for (int c = 0; c < dk; ++c) { pq += qr[c] * dqn[c]; pk += kr[c] * dkn[c]; }
                for (int c = 0; c < dk; ++c) {
                    if (t->dq)
                        t->dq[i * t->so + c] = t->scale * (rq * dqn[c] - rq * rq * rq * qr[c] * pq);
                    if (t->dk_)
                        t->dk_[i * t->so + c] = rk * dkn[c] - rk * rk * rk * kr[c] * pk;
                }
            }
        }
    }
    if (t->dh0) memcpy(t->dh0, dS, sizeof(double) * nst);
    free(ck); free(S); free(Sp); free(Sn); free(U); free(R); free(QN); free(KN);
    free(RQ); free(RK); free(QR); free(KR); free(o); free(dS); free(dSp);
    free(dqn); free(dkn); free(du); free(dov);
}

static int pick_threads(int n_threads)
{
#ifdef _OPENMP
    return n_threads > 0 ? n_threads : omp_get_max_threads();
#else
    (void)n_threads;
    return 1;
#endif
}

/* Forward for n independent (sequence, head) tasks, spread over n_threads. */
void kda_oracle_fwd(const kda_oracle_task *tasks, int n, int n_threads)
{
    int nt = pick_threads(n_threads);
    (void)nt;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int i = 0; i < n; ++i) run_forward(&tasks[i], -1);
}

/* Decode / draft-verify: outputs for all T tokens, state committed after accept. */
void kda_oracle_step(const kda_oracle_task *tasks, int n, int n_threads)
{
    int nt = pick_threads(n_threads);
    (void)nt;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int i = 0; i < n; ++i) run_forward(&tasks[i], tasks[i].accept);
}

void kda_oracle_bwd(const kda_oracle_task *tasks, int n, int n_threads)
{
    int nt = pick_threads(n_threads);
    (void)nt;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nt)
    for (int i = 0; i < n; ++i) run_backward(&tasks[i]);
}

int kda_oracle_abi_version(void) { return 1; }
